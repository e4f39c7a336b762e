"""Benchmark: exact integer GEMM throughput (TOPS = 2*M*N*K / s) on GB300.

One step is one GEMM call of the chosen workload through the C-ABI (host plan
+ TMA loads + unpack + tcgen05 MMA + epilogue, and the split-K reduction when
the plan splits K).  Inputs are seeded synthetic operands resident in HBM
before timing.  Between steps no step finds its operands in L2: by default
every step reads its own copy of the operands, rotating over copies worth
three L2 capacities; --l2 flush instead writes 256 MB before every step
(outside the timed events).  Before each timed pass a GPU sleep holds the
stream while the host enqueues every step of the pass, so the device runs the
steps back to back and the events time the device, not the Python launch rate
(the end-to-end leg keeps the host path in its time).  Prints one JSON line.

  python bench.py [--gpus 1] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                  [--l2 rotate|flush] [--seconds S]

--impl reference times the CPU oracle (plain C, int64 accumulation) on the
host cores, each step a bounded row sample of the same workload.
--seconds S adds a sustained leg: steps back to back for about S seconds
under one pair of events, with the SM clock sampled meanwhile.

One GPU only.  The library is a single-GPU library (the GEMM is not sharded;
its cluster kernels share operand tiles between the CTAs of one GPU), so the
benchmark refuses --gpus other than 1 and any launch with WORLD_SIZE above 1
(a torchrun job), with a one-line message and exit status 2.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "int4/W4A8 GEMM TOPS (2*M*N*K/s)"
UNIT = "TOPS"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
E4M3_PER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20  # GB300 L2 (126.5 MiB)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        out = {}
        for k in FALLBACK_PEAKS:
            v = d.get(k)
            if isinstance(v, dict):
                v = v.get("value")
            out[k] = float(v) if v is not None else None
        if all(out[k] for k in ("hbm_gbs", "bf16_tflops")):
            return out, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# CUDA sources without device code (the host-buffer entry points: copies and
# calls of the device entry points), left out of the digest below
HOST_ONLY_SOURCES = ("host.cu",)


def sources_digest():
    """SHA-256 over the CUDA sources that hold device code or launch planning
    (csrc/*.cu, *.cuh by name, HOST_ONLY_SOURCES left out): the DRAM traffic
    recorded in profiles/traffic.json is used only for this exact kernel code."""
    import hashlib
    d = os.path.join(ROOT, "precision_integer_gemm_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh")) and name not in HOST_ONLY_SOURCES:
            h.update(name.encode())
            with open(os.path.join(d, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload):
    """DRAM bytes (read + write) per launch of the workload's GEMM kernel from
    one ncu capture, or None if none was taken for the current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("sources_sha256") != sources_digest():
        return None
    entry = rec.get("workloads", {}).get(workload)
    return None if entry is None else int(entry["dram_bytes_per_launch"])


def workload_bytes(variant, M, N, K):
    if variant in ("fp8", "fp8e5m2"):
        return (M + N) * K + 4 * M * N
    if variant == "fp8bs":
        return (M + N) * K + 4 * M * N + 4 * (M + N) * (-(-K // 128))
    a = M * K if variant == "w4a8" else M * K // 2
    return a + N * K // 2 + 4 * M * N


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        """Start sampling every 20 ms; returns once the first sample arrived."""
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        first = threading.Event()

        def reader():
            for line in self.proc.stdout:
                self.lines.append(line)
                first.set()
            first.set()

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        first.wait(timeout=10.0)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        out = "".join(self.lines)
        sm, smax, power, reasons, mask = [], [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
            try:
                mask |= int(parts[4], 16)  # every clock-event reason seen (NVML bit mask)
            except ValueError:
                pass
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "reasons_mask": hex(mask), "power_w_max": max(power) if power else None}


# variants whose operands are fp8 bytes and whose C is float32
FP8_VARIANTS = ("fp8", "fp8e5m2", "fp8bs")

# the block scales of the fp8bs workload (set in main)
_SCALES = None


def oracle_sample_time(orc, variant, a, b, K, rows, threads):
    """Run the oracle on the first `rows` rows of A; returns seconds."""
    t0 = time.perf_counter()
    if variant in ("fp8", "fp8e5m2"):
        orc.fp8_gemm(np.ascontiguousarray(a[:rows]), b, K, threads=threads,
                     fmt="e5m2" if variant == "fp8e5m2" else "e4m3")
    elif variant == "fp8bs":
        sfa, sfb = _SCALES
        orc.fp8_blockscaled(np.ascontiguousarray(a[:rows]), b, np.ascontiguousarray(sfa[:rows]), sfb, K,
                            threads=threads)
    elif variant == "i4i4":
        orc.i4i4_gemm(orc.pack_int4(a[:rows]), orc.pack_int4(b), K, threads=threads)
    else:
        orc.w4a8_gemm(np.ascontiguousarray(a[:rows]), orc.pack_int4(b), K, threads=threads)
    return time.perf_counter() - t0


def calibrate_rows(orc, variant, a, b, K, threads, target_s):
    M = a.shape[0]
    rows = max(1, min(M, threads))
    t = oracle_sample_time(orc, variant, a, b, K, rows, threads)
    if t < target_s / 8 and rows < M:
        rows = int(min(M, max(rows + 1, rows * target_s / max(t, 1e-3))))
        rows = max(threads, (rows // threads) * threads) if rows >= threads else rows
        rows = min(rows, M)
    return rows


def run_reference(args, variant, M, N, K, a, b):
    import oracle
    orc = oracle.Oracle()
    threads = os.cpu_count() or 1
    step_target = max(0.5, min(4.0, 150.0 / max(1, args.steps + args.warmup)))
    rows = calibrate_rows(orc, variant, a, b, K, threads, step_target)
    for _ in range(args.warmup):
        oracle_sample_time(orc, variant, a, b, K, rows, threads)
    times = [oracle_sample_time(orc, variant, a, b, K, rows, threads) for _ in range(args.steps)]
    ops = 2.0 * rows * N * K
    total = sum(times)
    value = ops * args.steps / total / 1e12
    sample = f"rows 0..{rows - 1} of A against all {N} rows of B, K={K} (each step)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64" if variant in FP8_VARIANTS else "int64",
        "data": "synthetic (SplitMix64-seeded, uniform)",
        "config": {"workload": args.workload, "variant": variant, "M": M, "N": N, "K": K},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, variant, M, N, K, a, b):
    import torch
    import precision_integer_gemm_gb300 as pig

    pig.build_library()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()

    # operands resident in HBM: logical -> packed by the library's pack kernel
    a_dev = torch.from_numpy(a).cuda()
    b_dev = torch.from_numpy(b).cuda()
    if variant in FP8_VARIANTS:
        bp = b_dev  # fp8 bytes as they are
    else:
        bp = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
        pig.pack_int4(b_dev, bp, N, K)
    if variant in ("fp8", "fp8e5m2"):
        a_in = a_dev
        gemm = pig.fp8_gemm if variant == "fp8" else pig.fp8_gemm_e5m2
    elif variant == "fp8bs":
        a_in = a_dev
        sfa_d, sfb_d = (torch.from_numpy(x).cuda() for x in _SCALES)

        def gemm(a_, b_, c_, m_, n_, k_, st):
            pig.fp8_blockscaled_gemm(a_, b_, sfa_d, sfb_d, c_, m_, n_, k_, st)
    elif variant == "i4i4":
        a_in = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
        pig.pack_int4(a_dev, a_in, M, K)
        gemm = pig.i4i4_gemm
    else:
        a_in = a_dev
        gemm = pig.w4a8_gemm
    del b_dev
    C = torch.empty((M, N), dtype=torch.float32 if variant in FP8_VARIANTS else torch.int32, device="cuda")
    # L2 between steps: either every step reads its own copy of the operands,
    # rotating over copies worth three L2 capacities (a step's operands were last
    # touched two or more steps ago, and all later reads evicted them), or a
    # 256 MB write before every step
    op_bytes = a_in.numel() * a_in.element_size() + bp.numel() * bp.element_size()
    if args.l2 == "rotate":
        n_copies = max(2, min(64, -(-3 * L2_BYTES // op_bytes)))
        copies = [(a_in, bp)] + [(a_in.clone(), bp.clone()) for _ in range(n_copies - 1)]
        flush = None
    else:
        n_copies = 1
        copies = [(a_in, bp)]
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    state = {"i": 0}

    def step():
        a_s, b_s = copies[state["i"] % n_copies]
        state["i"] += 1
        gemm(a_s, b_s, C, M, N, K, stream)

    def before_step():
        if flush is not None:
            flush.zero_()

    for _ in range(args.warmup):
        before_step()
        step()
    if pig.igemm_last_status(stream) != 0:
        raise RuntimeError("device status after warm-up is not ok")

    def queue_ahead(n_steps):
        """Keep the GPU busy (a sleep on the stream, before the first event) while
        the host enqueues the next n_steps steps, so the device runs them back to
        back and the events time the device rather than the host's launch rate: a
        call costs the host about 5 us from Python and an event record 2.5 us,
        more than a 256^3 or 1024^3 GEMM takes on the GPU."""
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(int(min(200_000_000, 50_000 * n_steps + 200_000)))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    # events the library records around the GEMM kernel itself (the roofline's
    # dominant kernel); recorded once here so that their handles exist
    k_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    k_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for ev in k_starts + k_ends:
        ev.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    torch.cuda.synchronize()
    sampler.start()
    launched0 = pig.igemm_kernels_launched()
    wall0 = time.perf_counter()
    queue_ahead(args.steps)
    for i in range(args.steps):
        before_step()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    launched = pig.igemm_kernels_launched() - launched0  # this library's kernels in the timed region
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if pig.igemm_last_status(stream) != 0:
        raise RuntimeError("device status after the timed region is not ok")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_s = sum(step_ms) / 1e3
    # the GEMM kernel's own time (the roofline's), from a second pass of the
    # same steps with the library's events armed around that kernel (kept out
    # of the timed steps: events between the kernels of a step change how
    # they overlap)
    queue_ahead(args.steps)
    for i in range(args.steps):
        before_step()
        pig.igemm_time_next_gemm(k_starts[i], k_ends[i])
        step()
    torch.cuda.synchronize()
    gemm_kernel_s = sum(s.elapsed_time(e) for s, e in zip(k_starts, k_ends)) / 1e3 / args.steps

    ops = 2.0 * M * N * K
    value = ops * args.steps / total_s / 1e12
    peaks, peak_src = load_peaks()

    # sustained leg (opt-in): steps back to back for about --seconds, one pair
    # of events around all of them, SM clocks sampled meanwhile
    sustained = None
    if args.seconds > 0:
        n_sus = max(args.steps, int(args.seconds / max(total_s / args.steps, 1e-6)))
        sus_s, sus_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sus_sampler = ClockSampler(0)
        torch.cuda.synchronize()
        sus_sampler.start()
        sus_s.record(stream)
        for _ in range(n_sus):
            before_step()
            step()
        sus_e.record(stream)
        torch.cuda.synchronize()
        sus_clocks = sus_sampler.stop()
        if pig.igemm_last_status(stream) != 0:
            raise RuntimeError("device status after the sustained leg is not ok")
        sus_total = sus_s.elapsed_time(sus_e) / 1e3
        sus_ms = 1e3 * sus_total / n_sus
        sustained = {"value": ops * n_sus / sus_total / 1e12, "unit": UNIT, "steps": n_sus,
                     "seconds": sus_total, "ms_per_step": sus_ms, "clocks": sus_clocks,
                     "kcycles_per_step": (sus_ms * sus_clocks["sm_mhz"]) if sus_clocks.get("sm_mhz") else None,
                     "burst_kcycles_per_step": (1e3 * total_s / args.steps * clocks["sm_mhz"])
                     if clocks.get("sm_mhz") else None}
        if not args.workload.startswith("w4a8_decode") and peaks.get("bf16_tflops_sustained"):
            sus_peak = E4M3_PER_BF16 * peaks["bf16_tflops_sustained"]
            sustained.update({"peak": sus_peak, "frac": sustained["value"] / sus_peak,
                              "peak_source": f"{peak_src} bf16 sustained x {E4M3_PER_BF16}; the step "
                                             f"(preparation pass included) against it"})

    # end to end through the public API with pinned host buffers
    e2e_steps = max(1, min(args.steps, 5))
    a_host = (a_in.cpu() if variant == "i4i4" else torch.from_numpy(a)).pin_memory()
    bp_host = bp.cpu().pin_memory()
    c_host = torch.empty((M, N), dtype=C.dtype).pin_memory()
    # other per-step inputs (the fp8bs scales), pinned host copies
    extra_hosts = [x.cpu().pin_memory() for x in (sfa_d, sfb_d)] if variant == "fp8bs" else []
    e_s = torch.cuda.Event(enable_timing=True)
    e_e = torch.cuda.Event(enable_timing=True)
    # the GEMM's host-buffer entry point: the copies run inside the call,
    # overlapped with the GEMM in row chunks
    host_call = {"i4i4": "i4i4_gemm_host", "w4a8": "w4a8_gemm_host", "fp8": "fp8_gemm_host",
                 "fp8e5m2": "fp8_gemm_e5m2_host", "fp8bs": "fp8_blockscaled_gemm_host"}[variant]
    host_fn = getattr(pig, host_call)

    def e2e_step():
        host_fn(a_host, bp_host, *extra_hosts, c_host, M, N, K, stream)

    e2e_step()  # untimed: the first call sizes the library's memory pool for the call's buffers
    torch.cuda.synchronize()
    e_s.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e_e.record(stream)
    torch.cuda.synchronize()
    e2e_s = e_s.elapsed_time(e_e) / 1e3
    e2e_value = ops * e2e_steps / e2e_s / 1e12
    if not torch.equal(c_host, C.cpu()):
        raise RuntimeError("end-to-end result differs from the device-resident result")

    nbytes = workload_bytes(variant, M, N, K)
    traffic = recorded_traffic(args.workload)
    if args.workload.startswith("w4a8_decode"):
        achieved = nbytes / gemm_kernel_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "kernel": "igemm_skinny_kernel",
                "kernel_ms": 1e3 * gemm_kernel_s, "algorithmic_bytes_per_launch": nbytes,
                "peak_source": f"{peak_src} copy bandwidth"}
    else:
        peak = E4M3_PER_BF16 * peaks["bf16_tflops"]
        achieved = ops / gemm_kernel_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "kernel": ("igemm_bs_kernel" if variant == "fp8bs"
                           else "igemm_small_kernel" if args.workload in ("i4i4_256", "i4i4_1024")
                           else "igemm_ss_kernel"),
                "kernel_ms": 1e3 * gemm_kernel_s, "algorithmic_ops_per_launch": ops,
                "peak_source": f"{peak_src} bf16 burst x {E4M3_PER_BF16} (nominal fp8/bf16 ratio)",
                "mma_macs_per_op": 2 if variant == "w4a8" else 1}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"i4i4": "int4", "w4a8": "int8xint4", "fp8": "e4m3 (float32 accumulate)",
                  "fp8e5m2": "e5m2 (float32 accumulate)",
                  "fp8bs": "e4m3 with float32 block scales (float32 accumulate)"}[variant],
        "data": "synthetic (SplitMix64-seeded, uniform)",
        "config": {"workload": args.workload, "variant": variant, "M": M, "N": N, "K": K,
                   "l2": (f"operands rotate over {n_copies} copies ({n_copies * op_bytes / 1e6:.0f} MB, "
                          f"3x L2 or more): each step's operands were evicted from L2 before it; no flush"
                          if args.l2 == "rotate" else
                          "flushed before every step (256 MB write, outside the timed events)"),
                   "queue": "all steps enqueued behind a GPU sleep before the first event (device time, "
                            "not the host launch rate)",
                   "parallelism": "single"},
        "wall_ms_per_step": 1e3 * wall / args.steps,
        "gpu_launches": launched,
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT,
                "h2d_bytes_per_step": int(a_in.numel() * a_in.element_size() + bp.numel() +
                                          sum(h.numel() * h.element_size() for h in extra_hosts)),
                "d2h_bytes_per_step": int(C.numel() * 4),
                "call": f"{host_call} (host buffers, copies inside the call)"},
        "roofline": roof,
    }
    if sustained is not None:
        line["sustained"] = sustained
    if not args.no_cpu_baseline:
        import oracle
        orc = oracle.Oracle()
        threads = os.cpu_count() or 1
        rows = calibrate_rows(orc, variant, a, b, K, threads, args.cpu_seconds)
        t = oracle_sample_time(orc, variant, a, b, K, rows, threads)
        if t < args.cpu_seconds / 2 and rows < M:
            # the small calibration sample overstates the per-row cost: size once more
            # from this run so that the reported sample is about --cpu-seconds long
            rows = min(M, max(rows + 1, int(rows * args.cpu_seconds / max(t, 1e-3))))
            t = oracle_sample_time(orc, variant, a, b, K, rows, threads)
        line["cpu_baseline"] = {"value": 2.0 * rows * N * K / t / 1e12, "unit": UNIT, "cores": threads,
                                "kind": "oracle",
                                "sample": f"rows 0..{rows - 1} of A against all {N} rows of B, K={K}; {t:.1f} s"}
    print(json.dumps(line), flush=True)


def refuse_multi_gpu(gpus: int) -> str | None:
    """The one-line reason this run is refused, or None for a one-GPU run."""
    world = os.environ.get("WORLD_SIZE", "1")
    try:
        world_n = int(world)
    except ValueError:
        world_n = 2
    if gpus != 1 or world_n > 1:
        return (f"bench.py runs on one GPU only (got --gpus {gpus}, WORLD_SIZE={world}): the library is a "
                f"single-GPU library, its cluster kernels share tiles between CTAs of one GPU")
    return None


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="i4i4_8192", choices=sorted(si.WORKLOADS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--l2", choices=["rotate", "flush"], default="rotate",
                   help="keep operands out of L2 between steps by rotating copies, or by a 256 MB write")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--seconds", type=float, default=0.0,
                   help="add a sustained leg of about this many seconds (0: none)")
    args = p.parse_args()
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    why = refuse_multi_gpu(args.gpus)
    if why:
        print(why, file=sys.stderr, flush=True)
        sys.exit(2)

    variant, M, N, K, a, b = si.workload_operands(args.workload)
    if variant == "fp8bs":
        global _SCALES
        _SCALES = si.block_scales(M, N, K, si.WORKLOADS[args.workload][4])

    if args.impl == "reference":
        run_reference(args, variant, M, N, K, a, b)
        return
    run_ours(args, variant, M, N, K, a, b)


if __name__ == "__main__":
    main()
