"""tgemm_gemm_noalloc: the multiply for callers that cannot allocate device
memory (hosts that hand out all device memory from their own pool, services
with a memory budget fixed after start-up).  It runs the stream-K split with
the scratch array built into the library instead of a caller workspace.

Each call's output is compared element by element with the oracle's product
of the same inputs, within the parity tolerance (tests/tolerance.py), and
with the existing workspace entry point, tgemm_gemm_ws, on the same split.
Two calls run in a row: the second reuses the scratch the first one left
behind.  The plan is checked first, so a call that silently ran without the
split (and so never touched the scratch array) would fail.
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
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(lib, M, N, K, dtype, opts):
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
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    # the split this call takes on this device: a nonzero scratch need means
    # some k-stages are spread over the pairs; it must fit the built-in array
    c_ref = torch.zeros((M, N), dtype=cdt, device=dev)
    st, need = lib.workspace_size(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c_ref.data_ptr(), N, dtype, sk)
    assert st == lib.OK and 0 < need <= lib.NOALLOC_SCRATCH_BYTES
    # the device-free plan (pairs modelled as SMs / 2) takes the split too; with
    # a CTA cap both count the same pairs, so the scratch sizes agree
    st, plan = lib.plan(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c_ref.data_ptr(), N, dtype, sk, sm_count=sms,
                        workspace_bytes=lib.NOALLOC_SCRATCH_BYTES)
    assert st == lib.OK and plan.sk_iters > 0
    if "max_ctas" in opts:
        assert plan.workspace_bytes == need

    # the oracle's product of the same inputs
    C64, S = oracle.gemm(A, B, fin, M, N, K)

    # the existing entry point with a caller workspace, same split
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    st = lib.gemm_ws(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c_ref.data_ptr(), N, dtype, sk, ws.data_ptr(), need,
                     stream)
    assert st == lib.OK, lib.status_string(st)
    assert lib.device_status(stream) == lib.OK
    bits = np.uint32 if fout == "f32" else np.uint16
    ws_out = wl.decode(c_ref.cpu().numpy().view(bits), fout)
    ok, ratio, where = tolerance.check(ws_out, C64, S, fin, fout)
    assert ok, f"workspace entry point: error/bound {ratio:.3g} at {where}"

    for call in range(2):
        c = torch.full((M, N), -1, dtype=cdt, device=dev)
        st = lib.gemm_noalloc(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, dtype, opts, stream)
        assert st == lib.OK, lib.status_string(st)
        assert lib.device_status(stream) == lib.OK
        got = wl.decode(c.cpu().numpy().view(bits), fout)
        ok, ratio, where = tolerance.check(got, C64, S, fin, fout)
        assert ok, f"call {call}: error/bound {ratio:.3g} at {where} against the oracle"
        ok, ratio, where = tolerance.check(got, ws_out, S, fin, fout)
        assert ok, f"call {call}: error/bound {ratio:.3g} at {where} against tgemm_gemm_ws"
