"""Benchmark of the tiled GEMM library on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one C = A . B product of the workload (default: bf16 4096^3 with fp32
output), inputs already resident in device memory.  Before every timed step a
256 MiB buffer is written to flush the 129 MB L2; each step is timed with CUDA
events on the launching stream around the single library call, and `value`
is the FLOP rate over the sum of the K step times (max over ranks).

`e2e` measures the same product end to end from pinned host memory through
the C ABI's host-buffer call (tgemm_gemm_host): per step, the host -> device
copies of A and B, the product, and the device -> host copy of C, all inside
the event-timed region (with a fused epilogue: torch copies around
tgemm_gemm_epilogue).

`cpu_baseline` times the CPU oracle (the plain fp64 triple loop, all host
cores) on a bounded sample of rows of the workload, and `cpu_blocked` its
cache-blocked fp64 variant on another; both are reported baselines, not
targets.  `--impl reference` times the oracle alone the same way; it is a
deliberately slow baseline, not a competitor.

Multi-GPU: the product has no exchange step, so N ranks run N independent
replicas of the workload (weak scaling) with no collective on the data path;
the barrier and the max over ranks are the only cross-rank operations.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

# fused epilogues the benchmark can time: (alpha, beta, bias?, activation)
EPILOGUES = {"none": None, "bias_relu": (1.0, 0.0, True, 1), "axpby": (0.5, 1.0, False, 0),
             "all": (2.0, 1.0, True, 1)}

FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "tc_gemm_2sm_swap_bf16_4096x4096x4096_f32out.md")
# sources of the kernel the headline workload runs (the CTA-pair kernel with exchanged operands)
KERNEL_SOURCES = [os.path.join(ROOT, "tiled_dense_gemm_02_gb300", "csrc", f)
                  for f in ("tc_gemm_2sm_swap.cu", "tc_common.cuh", "ptx.cuh", "tgemm_internal.h")]


def _build_library():
    """Build libtgemm.so if stale, through the standalone build script."""
    import importlib.util
    path = os.path.join(ROOT, "tiled_dense_gemm_02_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("tgemm_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=wl.HEADLINE.name,
                   choices=sorted(wl.BY_NAME) + sorted(wl.TRANSPOSE_BY_NAME) + sorted(wl.BATCH_BY_NAME))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads, the FP32 probe and the host-dispatch measurement")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU work of the oracle sample")
    p.add_argument("--options", type=json.loads, default=None,
                   help="tgemm_options fields for the timed call, as a JSON object (e.g. '{\"group_m\": 32}')")
    p.add_argument("--cublas", action="store_true",
                   help="also time torch.matmul (cuBLAS) on the same inputs, as context (outside the timed region)")
    p.add_argument("--workspace", action="store_true",
                   help="time the call through tgemm_gemm_ws with a workspace of tgemm_workspace_size bytes "
                        "(the library may then repack unaligned operands)")
    p.add_argument("--epilogue", default="none", choices=sorted(EPILOGUES),
                   help="fused epilogue C = act(alpha A.B + beta C + bias) timed with the product")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_replicas(local: int, backend: str | None = None):
    """One process per GPU, each an independent replica: the process group
    carries only the start/stop barriers and the max-over-ranks timing (no data
    exchange).  nccl where there are GPUs, gloo where there are none (tests)."""
    import torch
    import torch.distributed as dist
    if backend is None:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return backend


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over all ranks (the slowest replica sets the time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    if workload != wl.HEADLINE.name or not os.path.exists(PROFILE_TRAFFIC):
        return None
    text = open(PROFILE_TRAFFIC).read()
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_bytes or not m_hash or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi sampling (200 ms) while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


def cpu_oracle_sample(w: wl.Workload, A, B, target_seconds: float, rows: int | None = None):
    """Time the oracle (as it stands, all host cores) on the first `rows` rows of
    the product; `rows` is chosen to take about `target_seconds` when None."""
    import oracle
    fin = wl.IN_FORMAT[w.dtype]
    threads = os.cpu_count() or 1
    if rows is None:
        probe = max(1, min(w.M, threads))
        t0 = time.perf_counter()
        oracle.gemm(np.ascontiguousarray(A[:probe]), B, fin, probe, w.N, w.K, threads=threads, with_abs=False)
        per_row = (time.perf_counter() - t0) / probe
        rows = int(max(probe, min(w.M, target_seconds / max(per_row, 1e-9))))
        rows = max(threads, rows // threads * threads) if rows >= threads else rows
    t0 = time.perf_counter()
    oracle.gemm(np.ascontiguousarray(A[:rows]), B, fin, rows, w.N, w.K, threads=threads, with_abs=False)
    dt = time.perf_counter() - t0
    tflops = 2.0 * rows * w.N * w.K / dt / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of the {w.M}x{w.N}x{w.K} product ({rows * w.N} outputs, "
                      f"{dt:.2f} s, fp64 triple loop over the rounded inputs, rows split across threads)"}


def cpu_blocked_sample(w: wl.Workload, A, B, target_seconds: float):
    """Time the cache-blocked fp64 variant of the oracle (all host cores) on
    the first rows of the product, about `target_seconds` of work."""
    import oracle
    fin = wl.IN_FORMAT[w.dtype]
    threads = os.cpu_count() or 1
    # two probes separate the per-call cost (decoding B into doubles) from the per-row cost
    probes, times = (max(1, min(w.M, 2 * threads)), max(1, min(w.M, 6 * threads))), []
    for n in probes:
        t0 = time.perf_counter()
        oracle.gemm_blocked(np.ascontiguousarray(A[:n]), B, fin, n, w.N, w.K, threads=threads)
        times.append(time.perf_counter() - t0)
    per_row = max((times[1] - times[0]) / max(probes[1] - probes[0], 1), times[1] / probes[1] / 8, 1e-9)
    fixed = max(times[0] - per_row * probes[0], 0.0)
    rows = int(max(probes[1], min(w.M, (target_seconds - fixed) / per_row)))
    t0 = time.perf_counter()
    oracle.gemm_blocked(np.ascontiguousarray(A[:rows]), B, fin, rows, w.N, w.K, threads=threads)
    dt = time.perf_counter() - t0
    return {"value": 2.0 * rows * w.N * w.K / dt / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "cache-blocked fp64 variant of the oracle",
            "sample": f"rows 0..{rows - 1} of the {w.M}x{w.N}x{w.K} product ({dt:.2f} s)"}


def run_reference(args, w: wl.Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    A, B = wl.make_inputs(w)
    threads = os.cpu_count() or 1
    rows = max(threads, 2 * threads)
    for _ in range(args.warmup):
        cpu_oracle_sample(w, A, B, 0, rows=rows)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        cpu_oracle_sample(w, A, B, 0, rows=rows)
        times.append(time.perf_counter() - t0)
    per_step = sum(times) / len(times)
    value = 2.0 * rows * w.N * w.K / per_step / 1e12
    line = {
        "impl": "reference", "metric": "GEMM TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} rows of the {w.M}x{w.N}x{w.K} product per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def sampled_check(w: wl.Workload, A, B, got_bits: np.ndarray, n_random: int, seed: int):
    """The oracle at every element of the first and last row and column plus
    `n_random` random positions of the product's output (storage bits), under
    the parity tolerance: (max error/bound, positions checked)."""
    import oracle
    from tests import tolerance
    fin, fout = wl.IN_FORMAT[w.dtype], wl.OUT_FORMAT[w.dtype]
    r = wl.splitmix64(seed, 2 * n_random)
    rows = np.concatenate([np.zeros(w.N, np.int64), np.full(w.N, w.M - 1, np.int64), np.arange(w.M), np.arange(w.M),
                           (r[:n_random] % np.uint64(w.M)).astype(np.int64)])
    cols = np.concatenate([np.arange(w.N), np.arange(w.N), np.zeros(w.M, np.int64), np.full(w.M, w.N - 1, np.int64),
                           (r[n_random:] % np.uint64(w.N)).astype(np.int64)])
    ref, S = oracle.entries(np.ascontiguousarray(A), np.ascontiguousarray(B), fin, w.K, rows, cols)
    got = wl.decode(np.ascontiguousarray(got_bits[rows, cols])[None, :], fout)[0]
    ok, ratio, _ = tolerance.check(got, ref, S, fin, fout)
    return float(ratio), int(rows.size)


def full_check(w: wl.Workload, A, B, got_bits: np.ndarray):
    """Every element against the oracle's full product: (max error/bound, elements)."""
    import oracle
    from tests import tolerance
    fin, fout = wl.IN_FORMAT[w.dtype], wl.OUT_FORMAT[w.dtype]
    ref, S = oracle.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B), fin, w.M, w.N, w.K)
    ok, ratio, _ = tolerance.check(wl.decode(np.ascontiguousarray(got_bits), fout), ref, S, fin, fout)
    return float(ratio), int(w.M * w.N)


def fp32_peak_probe(dev, sms: int):
    """FP32 FMA throughput measured by the probe kernel (libtgemm_probe.so):
    8 independent FMA chains per thread, 8 blocks of 256 threads per SM, best
    of three launches of each of scalar fma.rn.f32 and paired fma.rn.f32x2,
    timed with CUDA events.  None if the probe library is missing."""
    import ctypes
    import torch
    path = os.path.join(ROOT, "tiled_dense_gemm_02_gb300", "libtgemm_probe.so")
    if not os.path.exists(path):
        return None
    lib = ctypes.CDLL(path)
    lib.tgemm_probe_ffma.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                     ctypes.c_void_p]
    lib.tgemm_probe_ffma.restype = ctypes.c_int
    per_iter = lib.tgemm_probe_ffma_per_iter()
    blocks, threads, iters = 8 * sms, 256, 4000
    out = torch.empty(blocks * threads, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    best = {}
    for paired in (0, 1):
        flops = blocks * threads * iters * per_iter * 2 * (2 if paired else 1)
        times = []
        for _ in range(4):
            s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_.record(stream)
            rc = lib.tgemm_probe_ffma(paired, blocks, threads, iters, out.data_ptr(), stream.cuda_stream)
            e_.record(stream)
            if rc != 0:
                raise RuntimeError(f"FFMA probe launch failed: cudaError {rc}")
            torch.cuda.synchronize(dev)
            times.append(s_.elapsed_time(e_))
        best["paired" if paired else "scalar"] = flops / (min(times[1:]) / 1e3) / 1e12
    return {"tflops": max(best.values()), "scalar_tflops": best["scalar"], "paired_tflops": best["paired"],
            "how": f"{blocks} blocks x {threads} threads x {iters} iterations x {per_iter} FMAs "
                   "(8 independent chains), best of 3 after one warm-up, CUDA events"}


def host_dispatch(tg, w: wl.Workload, dev, calls: int = 200):
    """Host microseconds per tgemm_gemm call, measured with the GPU queue kept
    busy (a long device sleep enqueued first), so launches never wait for the
    GPU: the library's validation, planning, cached tensor maps and launch.
    The same loop of calls with M = 0 (validation only, no CUDA call) gives the
    cost of the ctypes call itself."""
    import torch
    fin, fout = wl.IN_FORMAT[w.dtype], wl.OUT_FORMAT[w.dtype]
    tdt = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}
    a = torch.zeros((w.M, w.K), dtype=tdt[fin], device=dev)
    b = torch.zeros((w.K, w.N), dtype=tdt[fin], device=dev)
    c = torch.empty((w.M, w.N), dtype=tdt[fout], device=dev)
    sptr = torch.cuda.current_stream(dev).cuda_stream
    args = (w.K, b.data_ptr(), w.N, c.data_ptr(), w.N, w.dtype, sptr)
    for _ in range(5):
        tg.gemm(w.M, w.N, w.K, a.data_ptr(), *args)
    torch.cuda.synchronize(dev)
    before = tg.host_counters()
    torch.cuda._sleep(int(2e8))  # about 0.1 s of device time ahead of the calls
    t0 = time.perf_counter_ns()
    for _ in range(calls):
        tg.gemm(w.M, w.N, w.K, a.data_ptr(), *args)
    t1 = time.perf_counter_ns()
    for _ in range(calls):
        tg.gemm(0, w.N, w.K, a.data_ptr(), *args)
    t2 = time.perf_counter_ns()
    torch.cuda.synchronize(dev)
    after = tg.host_counters()
    n = after["tc_launches"] - before["tc_launches"]
    return {"us_per_call": (t1 - t0) / calls / 1e3, "ctypes_us_per_call": (t2 - t1) / calls / 1e3,
            "library_prepare_us": (after["ns_prepare"] - before["ns_prepare"]) / max(n, 1) / 1e3,
            "library_launch_us": (after["ns_launch"] - before["ns_launch"]) / max(n, 1) / 1e3,
            "map_encodes": after["map_encodes"] - before["map_encodes"],
            "map_hits": after["map_hits"] - before["map_hits"], "calls": calls, "workload": w.name}


def time_workload(tg, w: wl.Workload, dev, flush, steps: int, peaks: dict, fp32_peak=None, options=None,
                  cublas: bool = False):
    """One workload timed like the headline (L2 flushed before each step,
    CUDA events around the call on its stream), checked against the oracle,
    with its roofline: min(peak FLOP/s, compulsory AI x measured HBM GB/s).
    With `options` the call is tgemm_gemm_ws with those options and a
    workspace of tgemm_workspace_size bytes (allocated before timing).  With
    `cublas`, torch.matmul on the same inputs is timed after it as context."""
    import torch
    fin, fout = wl.IN_FORMAT[w.dtype], wl.OUT_FORMAT[w.dtype]
    A, B = wl.make_inputs(w)
    np_view = {"f32": np.int32, "f16": np.int16, "bf16": np.int16}
    tdt = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}
    a = torch.from_numpy(A.view(np_view[fin])).to(dev)
    b = torch.from_numpy(B.view(np_view[fin])).to(dev)
    c = torch.empty((w.M, w.N), dtype=tdt[fout], device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ws_bytes = 0
    ws = None
    if options is not None:
        st, ws_bytes = tg.workspace_size(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N,
                                         w.dtype, options)
        ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    st, plan = tg.plan(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N, w.dtype, options, sms,
                       workspace_bytes=ws_bytes)

    def call():
        if options is None:
            s_ = tg.gemm(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N, w.dtype, sptr)
        else:
            s_ = tg.gemm_ws(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N, w.dtype, options,
                            ws.data_ptr(), ws_bytes, sptr)
        if s_ != tg.OK:
            raise RuntimeError(tg.status_string(s_))

    for _ in range(3):
        flush.fill_(1)
        call()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i, (s_, e_) in enumerate(ev):
        flush.fill_(i)
        s_.record(stream)
        call()
        e_.record(stream)
    torch.cuda.synchronize(dev)
    if tg.device_status(sptr) != tg.OK:
        raise RuntimeError(f"{w.name}: a kernel gave up a bounded wait")
    step_ms = [s_.elapsed_time(e_) for s_, e_ in ev]
    ms = sum(step_ms) / steps
    achieved = w.flops / (ms / 1e3) / 1e12
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ai = w.flops / w.compulsory_bytes
    if w.dtype == wl.F32:
        flop_peak = fp32_peak["tflops"] if fp32_peak else None
        bound_unit = "fp32 pipe (measured FFMA probe)"
    else:
        flop_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        bound_unit = "tensor (measured bf16 burst)"
    roof = min(flop_peak, ai * hbm / 1e3) if flop_peak else ai * hbm / 1e3
    got = c.cpu().numpy().view(np.uint32 if fout == "f32" else np.uint16).copy()
    entry = {"value": achieved, "unit": "TFLOP/s", "ms_per_step": ms, "step_ms_median": statistics.median(step_ms),
            "step_ms_min": min(step_ms), "steps": steps,
            "roofline": {"achieved": achieved, "peak": roof, "unit": "TFLOP/s", "frac": achieved / roof,
                         "bound": bound_unit if flop_peak and roof == flop_peak else "hbm (measured copy)",
                         "ai_flop_per_byte": ai, "dram_gbs_compulsory": w.compulsory_bytes / (ms / 1e3) / 1e9},
            "kernel": {k: v for k, v in plan.as_dict().items()
                       if k in ("kernel", "tile_m", "tile_n", "tile_k", "ctas", "cta_group", "swap_ab", "tuned",
                                "sk_iters", "workspace_bytes", "packed")},
            "call": "tgemm_gemm" if options is None else f"tgemm_gemm_ws {dict(options)}",
            "launches_per_step": kernel_launches_per_call(tg, plan, False)}
    if cublas:
        entry["context_cublas"] = cublas_context(a, b, w, dev, flush, steps)
    return entry, (A, B, got)


def cublas_context(a_bits, b_bits, w: wl.Workload, dev, flush, steps: int) -> dict:
    """torch.matmul (cuBLAS) on the same device inputs, timed like the
    workload (L2 flush, then CUDA events around the call on the stream):
    context beside the library's number, never part of it.  cuBLAS writes the
    input type, so for bf16 -> fp32 workloads its output is bf16; fp32 runs
    with TF32 off."""
    import torch
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[wl.IN_FORMAT[w.dtype]]
    at, bt = a_bits.view(tdt), b_bits.view(tdt)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        stream = torch.cuda.current_stream(dev)
        for _ in range(3):
            flush.fill_(1)
            torch.matmul(at, bt)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i, (s_, e_) in enumerate(ev):
            flush.fill_(i)
            s_.record(stream)
            torch.matmul(at, bt)
            e_.record(stream)
        torch.cuda.synchronize(dev)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    ms = [s_.elapsed_time(e_) for s_, e_ in ev]
    mean = sum(ms) / len(ms)
    return {"what": "torch.matmul (cuBLAS) on the same inputs, timed the same way; context, not used by the library",
            "out": str(tdt).replace("torch.", ""), "ms_mean": mean, "ms_median": statistics.median(ms),
            "tflops": w.flops / (mean / 1e3) / 1e12, "steps": steps}


def check_output(w: wl.Workload, A, B, got) -> dict:
    """The oracle leg of a timed workload, run on the host after all GPU work:
    every element for products of up to 2^20 outputs, else the borders and
    4096 random positions."""
    if w.M * w.N <= 1 << 20:
        ratio, checked = full_check(w, A, B, got)
    else:
        ratio, checked = sampled_check(w, A, B, got, 4096, seed=77)
    return {"max_err_over_bound": ratio, "elements_checked": checked}


def launch_floor(tg, dev, flush, steps: int = 50):
    """The smallest launch of the library timed like every workload (L2 flush
    first, CUDA events around the call): a 1 x 1 product with K = 0, which is
    one zero-fill kernel writing one float.  What a workload's time has beyond
    this is its own work."""
    import torch
    c = torch.empty(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps + 3)]
    for i, (s_, e_) in enumerate(ev):
        flush.fill_(i)
        s_.record(stream)
        st = tg.gemm(1, 1, 0, 0, 1, 0, 1, c.data_ptr(), 1, tg.F32, sptr)
        e_.record(stream)
        if st != tg.OK:
            raise RuntimeError(tg.status_string(st))
    torch.cuda.synchronize(dev)
    ms = [s_.elapsed_time(e_) for s_, e_ in ev[3:]]
    return {"us_mean": 1e3 * sum(ms) / len(ms), "us_median": 1e3 * statistics.median(ms), "us_min": 1e3 * min(ms),
            "what": "tgemm_gemm(1, 1, 0): one zero-fill kernel, after the same L2 flush, CUDA events"}


def kernel_launches_per_call(tg, plan, epilogue: bool) -> int:
    """Kernels one library call launches for `plan`: a plain fp32 product whose
    last round of tiles is split into K halves first zeroes the rows of C those
    halves add into (two launches); each operand repacked into the workspace
    adds one launch; everything else is one launch."""
    split = plan.kernel == tg.KERNEL_SIMT and plan.ctas != plan.tiles_m * plan.tiles_n
    return (2 if split and not epilogue else 1) + bin(plan.packed).count("1")


def run_ours(args, w: wl.Workload):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        init_replicas(local, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    _build_library()
    import tiled_dense_gemm_02_gb300 as tg

    fin, fout = wl.IN_FORMAT[w.dtype], wl.OUT_FORMAT[w.dtype]
    A, B = wl.make_inputs(w)
    tdt = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}
    np_view = {"f32": np.int32, "f16": np.int16, "bf16": np.int16}
    a_host = torch.from_numpy(A.view(np_view[fin])).pin_memory()
    b_host = torch.from_numpy(B.view(np_view[fin])).pin_memory()
    c_host = torch.empty((w.M, w.N), dtype=tdt[fout]).pin_memory()
    a = a_host.to(dev)
    b = b_host.to(dev)
    c = torch.empty((w.M, w.N), dtype=tdt[fout], device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ws, ws_bytes = None, 0
    opts = args.options
    if args.workspace:
        st, ws_bytes = tg.workspace_size(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N,
                                         w.dtype, opts)
        assert st == tg.OK, tg.status_string(st)
        ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    st, plan = tg.plan(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N, w.dtype, opts, sms,
                       workspace_bytes=ws_bytes)
    assert st == tg.OK, tg.status_string(st)

    epi = EPILOGUES[args.epilogue]
    launches_per_call = kernel_launches_per_call(tg, plan, epi is not None)
    bias = torch.linspace(-1.0, 1.0, w.N, dtype=torch.float32, device=dev) if epi and epi[2] else None
    epi_struct = None if epi is None else tg.Epilogue(alpha=epi[0], beta=epi[1],
                                                     bias=bias.data_ptr() if bias is not None else None,
                                                     activation=epi[3])

    def call():
        if epi_struct is None and ws is None and opts is None:
            s = tg.gemm(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N, w.dtype, sptr)
        elif epi_struct is None and ws is None:
            s = tg.gemm_ex(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N, w.dtype, opts, sptr)
        else:
            s = tg.gemm_epilogue(w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N, c.data_ptr(), w.N, w.dtype,
                                 epi_struct, opts, ws.data_ptr() if ws is not None else 0, ws_bytes, sptr)
        if s != tg.OK:
            raise RuntimeError(tg.status_string(s))

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        call()
    torch.cuda.synchronize(dev)
    assert tg.device_status(sptr) == tg.OK

    # ------------------------------------------------------------- timed region
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i)                  # evict A, B, C from L2 (outside the event pair)
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
    assert tg.device_status(sptr) == tg.OK
    # the output of the last timed step, against the oracle (after the timed region)
    last_c = c.cpu().numpy().view(np.uint32 if fout == "f32" else np.uint16).copy()
    ms_per_step = total_ms / args.steps
    value = world * w.flops * args.steps / (total_ms / 1e3) / 1e12

    # ------------------------------------------------------------- end to end
    e2e_steps = max(3, min(args.steps, 20))
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps + 2):
        j = i - 2
        if j >= 0:
            e_s[j].record(stream)
        if epi_struct is None:
            # the host-buffer entry point: B and row panels of A in, each panel's
            # product, panels of C out, overlapped on the library's copy streams
            s = tg.gemm_host(w.M, w.N, w.K, a_host.data_ptr(), w.K, b_host.data_ptr(), w.N, c_host.data_ptr(), w.N,
                             w.dtype, a.data_ptr(), b.data_ptr(), c.data_ptr(), 0, sptr)
            if s != tg.OK:
                raise RuntimeError(tg.status_string(s))
        else:
            a.copy_(a_host, non_blocking=True)
            b.copy_(b_host, non_blocking=True)
            call()
            c_host.copy_(c, non_blocking=True)
        if j >= 0:
            e_e[j].record(stream)
        torch.cuda.synchronize(dev)
    e2e_ms = sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)) / e2e_steps
    if world > 1:
        e2e_ms = max_over_ranks(e2e_ms, dev)
    e2e_value = world * w.flops / (e2e_ms / 1e3) / 1e12
    headline_cublas = None
    if world == 1 and args.cublas and epi is None:
        try:
            headline_cublas = cublas_context(a, b, w, dev, flush, min(args.steps, 20))
        except Exception as exc:  # context only: the line is printed whatever happens here
            headline_cublas = {"error": repr(exc)}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    errors = {}
    fp32_peak = None
    if world == 1 and (w.dtype == wl.F32 or not args.no_configs):
        try:
            fp32_peak = fp32_peak_probe(dev, sms)
        except Exception as exc:  # the headline line is printed whatever happens here
            errors["fp32_peak_probe"] = repr(exc)
    if w.dtype == wl.F32:
        # the SIMT kernel is bound by the FP32 pipe: the FFMA probe's measured
        # rate, beside SMs x 128 FMA/clk x 2 FLOP x the SM clock
        achieved = w.flops / (ms_per_step / 1e3) / 1e12
        clk = clocks.get("sm_max_mhz") or 2070.0
        derived = sms * 128 * 2 * clk * 1e6 / 1e12
        fp32_peak_value = fp32_peak["tflops"] if fp32_peak else derived
        roofline = {"bound": "alu", "achieved": achieved, "peak": fp32_peak_value, "unit": "TFLOP/s",
                    "frac": achieved / fp32_peak_value, "traffic": None,
                    "peak_source": ("measured: FFMA probe (libtgemm_probe.so), same run" if fp32_peak else
                                    f"derived: {sms} SMs x 128 fp32 FMA/clk x 2 x {clk:.0f} MHz"),
                    "peak_derived": derived, "frac_of_derived": achieved / derived,
                    "algorithmic_flops_per_launch": w.flops}
        if launches_per_call == 2:
            roofline["timed_span"] = "the zero fill of the split tiles' rows plus the SIMT kernel"
    else:
        achieved = w.flops / (ms_per_step / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak,
                    "traffic": profiled_traffic(w.name) if epi is None else None,
                    "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed alone)",
                    "algorithmic_flops_per_launch": w.flops,
                    "compulsory_bytes_per_launch": w.compulsory_bytes}
    # the other configurations, timed the same way (GPU work first, their
    # oracle checks below with the CPU legs)
    configs = dispatch = None
    outputs = {}
    if world == 1 and not args.no_configs and epi is None:
        configs = {}
        for name, steps in (("f32_64x64x64", 50), ("f16_1024x1024x1024", 50), ("bf16_2048x2048x2048", 50),
                            ("bf16_1000x1500x4096_ragged", 50), ("f32_4096x4096x4096", 10)):
            if name == w.name:
                continue
            try:
                configs[name], outputs[name] = time_workload(tg, wl.BY_NAME[name], dev, flush, steps, peaks,
                                                             fp32_peak, cublas=args.cublas)
            except Exception as exc:
                errors[name] = repr(exc)
        # the ragged shape again through tgemm_gemm_ws: with a workspace the
        # library repacks B (3000-byte rows) for the bulk-tensor kernels; and
        # the per-thread copy pairs with the stream-K split over every pair
        name = "bf16_1000x1500x4096_ragged"
        for tag, opts in (("+workspace", {}), ("+stream_k", {"stream_k": 2, "repack": 1})):
            try:
                configs[name + tag], outputs[name + tag] = time_workload(
                    tg, wl.BY_NAME[name], dev, flush, 50, peaks, fp32_peak, options=opts)
            except Exception as exc:
                errors[name + tag] = repr(exc)
        if fp32_peak:
            configs["fp32_peak_probe"] = fp32_peak
        try:
            configs["launch_floor"] = launch_floor(tg, dev, flush)
        except Exception as exc:
            errors["launch_floor"] = repr(exc)
        try:
            dispatch = {n: host_dispatch(tg, wl.BY_NAME[n], dev)
                        for n in ("f16_1024x1024x1024", "bf16_4096x4096x4096_f32out")}
        except Exception as exc:
            errors["host_dispatch"] = repr(exc)

    # ---------------------------------------------- CPU legs (oracle), no GPU work
    check = None
    if epi is None:
        ratio, checked = sampled_check(w, A, B, last_c, 4096, seed=78)
        check = {"max_err_over_bound": ratio, "elements_checked": checked,
                 "what": "the last timed step's C at every element of the first and last row and column and 4096 "
                         "random positions, against the oracle under the parity tolerance"}
    for name, (a_bits, b_bits, got) in outputs.items():
        configs[name].update(check_output(wl.BY_NAME[name.split("+")[0]], a_bits, b_bits, got))
    cpu = cpu_blocked = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_oracle_sample(w, A, B, args.cpu_seconds)
        cpu_blocked = cpu_blocked_sample(w, A, B, args.cpu_seconds / 2)
    line = {
        "metric": "GEMM TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": fin, "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in": fin, "out": fout, "accumulate": "f32",
                   "l2": "flushed before every timed step (256 MiB write)", "parallelism": f"replicas{world}",
                   "kernel": plan.as_dict(), "sms": sms, "epilogue": args.epilogue, "workspace_bytes": ws_bytes,
                   "options": opts,
                   "step_ms_min": min(step_ms),
                   "step_ms_median": statistics.median(step_ms), "wall_s": wall,
                   "host_dispatch_us": dispatch[w.name]["us_per_call"] if dispatch and w.name in dispatch else None},
        "roofline": roofline,
        "check": check,
        "context_cublas": headline_cublas,
        "configs": configs,
        "host_dispatch": dispatch,
        "cpu_baseline": cpu,
        "cpu_blocked": cpu_blocked,
        "errors": errors or None,
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(A.nbytes + B.nbytes), "d2h_bytes_per_step": int(c.numel() * c.element_size())},
        "gpu_launches": args.steps * launches_per_call,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def transpose_oracle_sample(w, target_seconds: float):
    """The oracle's transpose on host cores over a bounded slice of the
    workload's rows (grown until about target_seconds of work): GB/s of the
    same traffic measure (each element read and written once)."""
    import numpy as np
    from oracle import transpose as ot
    rng = np.random.default_rng(w.seed)
    bits = np.uint32 if w.elem_bytes == 4 else np.uint16
    rows = 256
    while True:
        src = rng.integers(0, 2 ** 16, size=(rows, w.cols), dtype=np.uint64).astype(bits)
        t0 = time.perf_counter()
        ot.transpose(src, rows, w.cols)
        dt = time.perf_counter() - t0
        if dt >= target_seconds or rows >= w.rows:
            break
        rows = min(w.rows, rows * 2 if dt < target_seconds / 4 else int(rows * target_seconds / max(dt, 1e-6)) + 1)
    moved = 2 * rows * w.cols * w.elem_bytes
    return {"value": moved / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of the {w.rows}x{w.cols} transpose ({dt:.2f} s, numpy column copies, "
                      f"one thread)"}


def run_transpose_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    per = max(0.5, min(args.cpu_seconds, 60.0) / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        transpose_oracle_sample(w, per)
    vals = [transpose_oracle_sample(w, per) for _ in range(args.steps)]
    value = statistics.median(v["value"] for v in vals)
    print(json.dumps({
        "impl": "reference", "metric": "transpose GB/s", "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u32" if w.elem_bytes == 4 else "u16", "data": "synthetic",
        "config": {"workload": w.name, "rows": w.rows, "cols": w.cols, "elem_bytes": w.elem_bytes},
        "cpu_baseline": {**vals[-1], "value": value},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)


def run_transpose(args, w):
    """The tiled transpose: GB/s of HBM traffic (each element read once and
    written once), against the measured copy bandwidth."""
    import torch
    world, rank, local = dist_env()
    if world > 1:
        init_replicas(local, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build_library()
    import tiled_dense_gemm_02_gb300 as tg
    tdt = torch.int32 if w.elem_bytes == 4 else torch.int16
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    src_host = torch.randint(-2 ** 15, 2 ** 15, (w.rows, w.cols), generator=gen, dtype=torch.int32).to(tdt).pin_memory()
    dst_host = torch.empty((w.cols, w.rows), dtype=tdt).pin_memory()
    src = src_host.to(dev)
    dst = torch.empty((w.cols, w.rows), dtype=tdt, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    def call():
        st = tg.transpose(w.rows, w.cols, src.data_ptr(), w.cols, dst.data_ptr(), w.rows, w.elem_bytes, sptr)
        if st != tg.OK:
            raise RuntimeError(tg.status_string(st))

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):   # 2 GiB (fp32) per step: inputs far larger than L2
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    total_ms = sum(step_ms)
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
    ms = total_ms / args.steps
    value = world * w.bytes_moved * args.steps / (total_ms / 1e3) / 1e9
    # end to end: host -> device copy of the input, the transpose, device -> host copy of the result
    e2e = []
    for i in range(5):
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record(stream)
        src.copy_(src_host, non_blocking=True)
        call()
        dst_host.copy_(dst, non_blocking=True)
        e_.record(stream)
        torch.cuda.synchronize(dev)
        if i >= 2:
            e2e.append(s_.elapsed_time(e_))
    e2e_ms = sum(e2e) / len(e2e)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = w.bytes_moved / (ms / 1e3) / 1e9
    line = {
        "metric": "transpose GB/s", "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u32" if w.elem_bytes == 4 else "u16", "data": "synthetic",
        "config": {"workload": w.name, "rows": w.rows, "cols": w.cols, "elem_bytes": w.elem_bytes,
                   "l2": f"inputs {w.rows * w.cols * w.elem_bytes >> 20} MiB, far larger than L2 (no flush)",
                   "parallelism": f"replicas{world}", "step_ms_min": min(step_ms),
                   "step_ms_median": statistics.median(step_ms), "wall_s": wall},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": None, "peak_source": f"{peak_src} hbm_gbs (copy)",
                     "algorithmic_bytes_per_launch": w.bytes_moved},
        "cpu_baseline": None if (args.no_cpu_baseline or world > 1) else transpose_oracle_sample(w, args.cpu_seconds),
        "clocks": clocks,
        "e2e": {"value": world * w.bytes_moved / (e2e_ms / 1e3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": w.rows * w.cols * w.elem_bytes,
                "d2h_bytes_per_step": w.rows * w.cols * w.elem_bytes},
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_batched(args, w):
    """A strided batch in one tgemm_gemm_batched call: TFLOP/s of the whole
    batch, timed like the product workloads (L2 flushed before each step, CUDA
    events around the call), with three of its products checked in full
    against the oracle after the timed region."""
    import torch
    world, rank, local = dist_env()
    if world > 1:
        init_replicas(local, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build_library()
    import tiled_dense_gemm_02_gb300 as tg
    fin, fout = wl.IN_FORMAT[w.dtype], wl.OUT_FORMAT[w.dtype]
    A, B = wl.make_batch_inputs(w)
    tdt = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}
    npv = {"f32": np.int32, "f16": np.int16, "bf16": np.int16}
    a_host = torch.from_numpy(A.view(npv[fin])).pin_memory()
    b_host = torch.from_numpy(B.view(npv[fin])).pin_memory()
    c_host = torch.empty((w.batch * w.M, w.N), dtype=tdt[fout]).pin_memory()
    a, b = a_host.to(dev), b_host.to(dev)
    c = torch.empty((w.batch * w.M, w.N), dtype=tdt[fout], device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sa, sb, sc = w.M * w.K, w.K * w.N, w.M * w.N
    st, plan, launches = tg.plan_batched(w.batch, w.M, w.N, w.K, a.data_ptr(), w.K, sa, b.data_ptr(), w.N, sb,
                                         c.data_ptr(), w.N, sc, w.dtype, args.options, sms)
    assert st == tg.OK, tg.status_string(st)

    def call():
        s_ = tg.gemm_batched(w.batch, w.M, w.N, w.K, a.data_ptr(), w.K, sa, b.data_ptr(), w.N, sb, c.data_ptr(), w.N,
                             sc, w.dtype, None, args.options, sptr)
        if s_ != tg.OK:
            raise RuntimeError(tg.status_string(s_))

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        call()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.fill_(i)
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    assert tg.device_status(sptr) == tg.OK
    step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    total_ms = sum(step_ms)
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
    ms = total_ms / args.steps
    value = world * w.flops * args.steps / (total_ms / 1e3) / 1e12
    got = c.cpu().numpy().view(np.uint32 if fout == "f32" else np.uint16).copy()
    # end to end: inputs in from pinned host memory, the batch, C back
    e2e = []
    for i in range(5):
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record(stream)
        a.copy_(a_host, non_blocking=True)
        b.copy_(b_host, non_blocking=True)
        call()
        c_host.copy_(c, non_blocking=True)
        e_.record(stream)
        torch.cuda.synchronize(dev)
        if i >= 2:
            e2e.append(s_.elapsed_time(e_))
    e2e_ms = sum(e2e) / len(e2e)
    cublas = None
    if args.cublas and world == 1:
        tt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[fin]
        at = a.view(tt).view(w.batch, w.M, w.K)
        bt = b.view(tt).view(w.batch, w.K, w.N)
        for _ in range(3):
            flush.fill_(1)
            torch.bmm(at, bt)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i, (s_, e_) in enumerate(ev):
            flush.fill_(i)
            s_.record(stream)
            torch.bmm(at, bt)
            e_.record(stream)
        torch.cuda.synchronize(dev)
        cms = sum(s_.elapsed_time(e_) for s_, e_ in ev) / len(ev)
        cublas = {"what": "torch.bmm (cuBLAS) on the same inputs, timed the same way; context, not used by the library",
                  "ms_mean": cms, "tflops": w.flops / (cms / 1e3) / 1e12}
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    # three products of the batch, every element, against the oracle
    one = w.one()
    worst, checked = 0.0, 0
    for bi in (0, w.batch // 2, w.batch - 1):
        ratio, n = full_check(one, A[bi * w.M:(bi + 1) * w.M], B[bi * w.K:(bi + 1) * w.K],
                              got[bi * w.M:(bi + 1) * w.M])
        worst, checked = max(worst, ratio), checked + n
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = w.flops / (ms / 1e3) / 1e12
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_oracle_sample(one, A[:w.M], B[:w.K], args.cpu_seconds)
        cpu["sample"] = "one product of the batch: " + cpu["sample"]
    line = {
        "metric": "GEMM TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": fin, "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "M": w.M, "N": w.N, "K": w.K, "in": fin, "out": fout,
                   "l2": "flushed before every timed step (256 MiB write)", "parallelism": f"replicas{world}",
                   "kernel": plan.as_dict(), "launches_per_call": launches, "options": args.options,
                   "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms)},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": None, "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed alone)",
                     "algorithmic_flops_per_launch": w.flops},
        "check": {"max_err_over_bound": worst, "elements_checked": checked,
                  "what": "products 0, batch/2 and batch-1 of the last timed step, every element, against the oracle"},
        "context_cublas": cublas,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "e2e": {"value": world * w.flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(A.nbytes + B.nbytes), "d2h_bytes_per_step": int(c.numel() * c.element_size())},
        "gpu_launches": args.steps * launches,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse_args()
    if args.workload in wl.BATCH_BY_NAME:
        if args.impl == "reference":
            bw = wl.BATCH_BY_NAME[args.workload]
            run_reference(args, bw.one())
        else:
            run_batched(args, wl.BATCH_BY_NAME[args.workload])
        return
    if args.workload in wl.TRANSPOSE_BY_NAME:
        if args.impl == "reference":
            run_transpose_reference(args, wl.TRANSPOSE_BY_NAME[args.workload])
        else:
            run_transpose(args, wl.TRANSPOSE_BY_NAME[args.workload])
        return
    w = wl.BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
