"""tgemm_gemm_noalloc: the multiply for callers that cannot allocate device
memory (hosts that hand out all device memory from their own pool, services
with a memory budget fixed after start-up).  It runs the stream-K split with
the scratch array built into the library instead of a caller workspace.

Its output is compared with the existing workspace entry point,
tgemm_gemm_ws, on the same inputs and split, within the parity tolerance
(tests/tolerance.py), on two calls in a row: the second call reuses the
scratch the first one left behind.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import gpu_harness as H
from tests import tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    torch.cuda.set_device(0)
    return H.tg()


@pytest.mark.parametrize("M,N,K,dtype,opts", [
    (1100, 1304, 1024, wl.BF16, {"cta_group": 2, "tile_n": 256, "max_ctas": 16}),
    (2048, 2048, 2048, wl.BF16_F32OUT, {"cta_group": 2, "tile_n": 256}),
], ids=["eight_pairs_bf16", "all_pairs_f32out"])
def test_noalloc_matches_workspace_entry_point_twice(lib, M, N, K, dtype, opts):
    dev = torch.device("cuda:0")
    fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
    w = wl.Workload("noalloc", M, N, K, dtype, "uniform", 90)
    A, B = wl.make_inputs(w)
    view = {"f32": np.int32, "f16": np.int16, "bf16": np.int16}
    a = torch.from_numpy(A.view(view[fin])).to(dev)
    b = torch.from_numpy(B.view(view[fin])).to(dev)
    cdt = torch.int32 if fout == "f32" else torch.int16
    stream = torch.cuda.current_stream(dev).cuda_stream
    sk = dict(opts, stream_k=2)

    # the existing entry point with a caller workspace, same split
    c_ref = torch.zeros((M, N), dtype=cdt, device=dev)
    st, need = lib.workspace_size(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c_ref.data_ptr(), N, dtype, sk)
    assert st == lib.OK and 0 < need <= lib.NOALLOC_SCRATCH_BYTES
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    st = lib.gemm_ws(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c_ref.data_ptr(), N, dtype, sk, ws.data_ptr(), need,
                     stream)
    assert st == lib.OK, lib.status_string(st)
    assert lib.device_status(stream) == lib.OK

    bits = np.uint32 if fout == "f32" else np.uint16
    ref = wl.decode(c_ref.cpu().numpy().view(bits), fout)
    _, S = oracle.gemm(A, B, fin, M, N, K)

    for call in range(2):
        c = torch.full((M, N), -1, dtype=cdt, device=dev)
        st = lib.gemm_noalloc(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, dtype, opts, stream)
        assert st == lib.OK, lib.status_string(st)
        assert lib.device_status(stream) == lib.OK
        got = wl.decode(c.cpu().numpy().view(bits), fout)
        ok, ratio, where = tolerance.check(got, ref, S, fin, fout)
        assert ok, f"call {call}: error/bound {ratio:.3g} at {where}"
