"""Offline tile-configuration selection: measure candidate launch options for a
list of shapes on the GPU at hand and write the fastest into a table that the
library compiles in (``csrc/tuned_shapes.inc``).

"Tiling 策略与内存层次优化" (its autotune step) and "GPU Kernel 的 Tile、Grid、
Wave 与 Launch Overhead" pick block sizes per problem shape by measurement; this
is that step done ahead of time, with the choice committed as a table rather
than searched at run time.  A call whose shape and dtype match an entry
exactly, and which leaves every tuned option at 0 (auto), is planned with the
entry's options; any other call keeps the library's own heuristics.

    python -m tiled_dense_gemm_02_gb300.tune [--out PATH] [--reps N] [SHAPE ...]

SHAPE is MxNxK:dtype with dtype one of f16, bf16, bf16f32, f16f32 (the default
list is the shapes the benchmark and tests name).  Needs a GPU and the built
library; it only times the library's own kernels through its C ABI.
"""
from __future__ import annotations

import argparse
import datetime
import itertools
import json
import os
import statistics
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
DEFAULT_OUT = os.path.join(HERE, "csrc", "tuned_shapes.inc")
DTYPES = {"f16": 1, "bf16": 2, "bf16f32": 3, "f16f32": 4}
DEFAULT_SHAPES = ["512x512x512:f16", "1024x1024x1024:f16", "2048x2048x2048:bf16", "4096x4096x4096:bf16f32",
                  "4096x4096x4096:bf16", "8192x8192x8192:f16", "8192x8192x8192:bf16"]
# the option fields a table entry sets, in the order of the C struct
FIELDS = ("kernel", "cta_group", "tile_n", "tile_m", "swap_ab", "tile_k", "group_m")


def candidates():
    """Option sets tried for every shape (invalid ones for a shape are skipped)."""
    out = [{}]
    for tm, tk, g in itertools.product((128, 192, 224, 256), (64, 128), (1, 2, 4, 8)):
        out.append({"swap_ab": 2, "tile_m": tm, "tile_n": 256, "tile_k": tk, "group_m": g})
    for bn, tk, g in itertools.product((128, 192, 224, 256), (64, 128), (4, 8)):
        out.append({"cta_group": 2, "swap_ab": 1, "tile_n": bn, "tile_k": tk, "group_m": g})
    for bn, g in itertools.product((64, 128, 192, 256), (4, 8)):
        out.append({"cta_group": 1, "tile_n": bn, "group_m": g})
    return out


def measure(shapes, reps):
    """Time every valid candidate of each shape.  The candidates are timed
    interleaved: each round calls all of them once, in an order rotated by one
    from the previous round, each call after an L2 flush; the ranking is by the
    mean over rounds.  (The median of back-to-back calls of one candidate moves
    in the steps of the event clock, about 2 us on GB300, and the first call
    of a round runs slower; rotating spreads that over all candidates.)"""
    import torch
    sys.path.insert(0, os.path.dirname(HERE))
    import tiled_dense_gemm_02_gb300 as tg
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    results = []
    for spec in shapes:
        dims, dname = spec.split(":")
        M, N, K = (int(x) for x in dims.split("x"))
        dtype = DTYPES[dname]
        a = torch.randn(M, K, device=dev).to(torch.bfloat16 if dname.startswith("bf16") else torch.float16)
        b = torch.randn(K, N, device=dev).to(a.dtype)
        c = torch.empty(M, N, device=dev, dtype=torch.float32 if dname.endswith("f32") else a.dtype)
        # "auto": the heuristics alone (a CTA cap of one per SM changes nothing
        # but keeps the compiled-in table out of the plan)
        cands = [{"max_ctas": sms}] + candidates()[1:]
        calls = []
        for opts in cands:
            st, _ = tg.plan(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, dtype, opts, sm_count=sms)
            if st != tg.OK:
                continue
            call = (lambda o: lambda: tg.gemm_ex(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, dtype,
                                                 o, sp))(opts)
            if call() != tg.OK:
                continue
            calls.append((opts, call, []))
        torch.cuda.synchronize()
        for r in range(reps + 2):
            for i in range(len(calls)):
                opts, call, ts = calls[(i + r) % len(calls)]
                flush.fill_(1)
                s = torch.cuda.Event(enable_timing=True)
                e = torch.cuda.Event(enable_timing=True)
                s.record()
                call()
                e.record()
                torch.cuda.synchronize()
                if r >= 2:  # two warm-up rounds
                    ts.append(s.elapsed_time(e) * 1000.0)
        assert tg.device_status(sp) == tg.OK
        means = [(statistics.mean(ts), opts) for opts, _, ts in calls]
        best_us, best_opts = min(means, key=lambda x: x[0])
        auto_us = means[0][0]
        if "max_ctas" in best_opts:  # the heuristics won: the entry leaves every option at 0
            best_opts = {}
        results.append({"shape": spec, "M": M, "N": N, "K": K, "dtype": dtype, "best_us": round(best_us, 2),
                        "auto_us": round(auto_us, 2), "options": best_opts,
                        "tflops": round(2.0 * M * N * K / (best_us * 1e-6) / 1e12, 1)})
        print(json.dumps(results[-1]), flush=True)
    return results, torch.cuda.get_device_name(dev)


def write_table(results, device, path):
    lines = [
        "// Tuned launch options per shape, written by tiled_dense_gemm_02_gb300/tune.py",
        f"// on {device}, {datetime.date.today().isoformat()}: the fastest of the candidate option sets",
        "// (mean over rounds of interleaved calls in rotating order, each after an L2",
        "// flush; auto = the heuristics alone).  Entry: M, N, K, dtype, then the",
        "// tgemm_options fields " + ", ".join(FIELDS) + " (0 = auto).",
    ]
    for r in results:
        o = r["options"]
        vals = [r["M"], r["N"], r["K"], r["dtype"]] + [int(o.get(f, 0)) for f in FIELDS]
        lines.append("{" + ", ".join(str(v) for v in vals) + "},  "
                     f"// {r['shape']}: {r['best_us']} us ({r['tflops']} TFLOP/s), auto {r['auto_us']} us")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("shapes", nargs="*", default=DEFAULT_SHAPES)
    ap.add_argument("--out", default=DEFAULT_OUT)
    ap.add_argument("--reps", type=int, default=30)
    args = ap.parse_args()
    results, device = measure(args.shapes, args.reps)
    write_table(results, device, args.out)
    print(f"wrote {args.out}")


if __name__ == "__main__":
    main()
