"""Several host threads calling the library at once, each on its own CUDA
stream, with different shapes, dtypes and kernels: the host caches (device
attributes, occupancy, kernel attributes) are shared under a mutex, and
every result must still match the oracle."""
import threading

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import gpu_harness as H
from tests import tolerance

pytestmark = pytest.mark.gpu

CASES = [(300, 520, 200, wl.BF16, None), (257, 264, 136, wl.F16, {"swap_ab": 2}),
         (129, 257, 33, wl.F32, None), (600, 264, 448, wl.BF16_F32OUT, {"cta_group": 2, "swap_ab": 1}),
         (500, 300, 96, wl.F16, {"cta_group": 1}), (256, 256, 1024, wl.BF16, {"cta_group": 2, "tile_k": 128, "swap_ab": 1})]


def test_concurrent_host_threads_on_separate_streams():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lib = H.tg()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    results, errors = {}, []

    def worker(tid):
        try:
            torch.cuda.set_device(dev)
            stream = torch.cuda.Stream(device=dev)
            with torch.cuda.stream(stream):
                for rep in range(3):
                    for ci, (M, N, K, dtype, opts) in enumerate(CASES):
                        fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
                        w = wl.Workload("thr", M, N, K, dtype, "uniform", 700 + 10 * tid + ci)
                        A, B = wl.make_inputs(w)
                        vi = {"f32": np.int32, "f16": np.int16, "bf16": np.int16}
                        a = torch.from_numpy(A.view(vi[fin])).to(dev, non_blocking=False)
                        b = torch.from_numpy(B.view(vi[fin])).to(dev, non_blocking=False)
                        c = torch.empty((M, N), dtype=torch.int32 if fout == "f32" else torch.int16, device=dev)
                        st = lib.gemm_ex(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, dtype, opts,
                                         stream.cuda_stream)
                        assert st == lib.OK, lib.status_string(st)
                        stream.synchronize()
                        results[(tid, rep, ci)] = (A, B, c.cpu().numpy())
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert lib.device_status(torch.cuda.current_stream(dev).cuda_stream) == lib.OK
    for (tid, rep, ci), (A, B, raw) in results.items():
        M, N, K, dtype, _ = CASES[ci]
        fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
        got = wl.decode(raw.view(np.uint32 if fout == "f32" else np.uint16), fout)
        ref, S = oracle.gemm(A, B, fin, M, N, K)
        ok, ratio, where = tolerance.check(got, ref, S, fin, fout)
        assert ok, f"thread {tid} rep {rep} case {ci}: error/bound {ratio:.3g} at {where}"
    assert len(results) == 4 * 3 * len(CASES)
