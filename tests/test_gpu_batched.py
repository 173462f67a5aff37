"""GPU parity of the strided batch, tgemm_gemm_batched: every product of the
batch against the oracle, with one launch of the swapped-operand kernel over
all matrices (checked through tgemm_plan_batched) or one launch per product;
shared operands (stride 0), the fused epilogue, per-thread stores of C, and
canaries in every gap between the C windows.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import epilogue as oepi
import workloads as wl
from tests import gpu_harness as H
from tests import tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    H.tg()
    torch.cuda.set_device(0)


def run_batch(batch, M, N, K, dtype, sa, sb, sc, seed, epi=None, options=None, ldc=None):
    lib = H.tg()
    dev = torch.device("cuda:0")
    fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
    ldc = N if ldc is None else ldc
    bits_in = H.NP_BITS[fin]
    nA, nB = max(sa * (batch - 1), 0) + M * K, max(sb * (batch - 1), 0) + K * N
    A_all = np.zeros(nA, dtype=bits_in)
    B_all = np.zeros(nB, dtype=bits_in)
    mats = []
    for b in range(batch):
        w = wl.Workload("batch", M, N, K, dtype, "uniform", seed + b)
        A, B = wl.make_inputs(w)
        if sa or b == 0:
            A_all[b * sa: b * sa + M * K] = A.reshape(-1)
        if sb or b == 0:
            B_all[b * sb: b * sb + K * N] = B.reshape(-1)
        mats.append((A_all[b * sa: b * sa + M * K].reshape(M, K), B_all[b * sb: b * sb + K * N].reshape(K, N)))
    c_elems = H.GUARD + sc * (batch - 1) + (M - 1) * ldc + N + H.GUARD
    prior_vals = wl.round_to_format(wl.uniform_pm1(seed + 99, c_elems), fout)
    c_init = np.full(c_elems, H.CANARY[fout], dtype=H.NP_BITS[fout])
    windows = np.zeros(c_elems, dtype=bool)
    for b in range(batch):
        for i in range(M):
            start = H.GUARD + b * sc + i * ldc
            windows[start:start + N] = True
    if epi is not None and epi.get("beta", 0.0) != 0.0:
        c_init[windows] = wl.encode(prior_vals[windows], fout)
    a_buf, a_ptr = H.upload(A_all, 0, dev)
    b_buf, b_ptr = H.upload(B_all, 0, dev)
    c_buf, c_base = H.upload(c_init, 0, dev)
    c_ptr = c_base + H.GUARD * wl.FORMATS[fout][3]
    bias_buf, ep = None, None
    if epi is not None:
        ep = {k: v for k, v in epi.items() if k != "bias"}
        if epi.get("bias") is not None:
            bias_buf = torch.from_numpy(np.asarray(epi["bias"], dtype=np.float32)).to(dev)
            ep["bias"] = bias_buf.data_ptr()
    stream = torch.cuda.current_stream(dev).cuda_stream
    st = lib.gemm_batched(batch, M, N, K, a_ptr, K, sa, b_ptr, N, sb, c_ptr, ldc, sc, dtype, ep, options, stream)
    assert st == lib.OK, lib.status_string(st)
    assert lib.device_status(stream) == lib.OK
    pst, plan, launches = lib.plan_batched(batch, M, N, K, a_ptr, K, sa, b_ptr, N, sb, c_ptr, ldc, sc, dtype, options,
                                           sm_count=torch.cuda.get_device_properties(dev).multi_processor_count)
    raw = c_buf[c_base - c_buf.data_ptr():][: c_elems * wl.FORMATS[fout][3]].cpu().numpy().view(H.NP_BITS[fout])
    assert np.all(raw[~windows] == H.CANARY[fout]), "an element outside every C window was written"
    for b, (A, B) in enumerate(mats):
        D, S = oracle.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B), fin, M, N, K)
        win = np.stack([raw[H.GUARD + b * sc + i * ldc: H.GUARD + b * sc + i * ldc + N] for i in range(M)])
        got = wl.decode(np.ascontiguousarray(win), fout)
        if epi is None:
            ok, ratio, where = tolerance.check(got, D, S, fin, fout)
        else:
            prior = np.stack([prior_vals[H.GUARD + b * sc + i * ldc: H.GUARD + b * sc + i * ldc + N]
                              for i in range(M)])
            bias = None if epi.get("bias") is None else np.asarray(epi["bias"], dtype=np.float64)
            act = "relu" if epi.get("activation", 0) == 1 else "none"
            Z = oepi.apply(D, prior, epi["alpha"], epi["beta"], bias, act)
            T = oepi.magnitude(S, prior, epi["alpha"], epi["beta"], bias)
            ok, ratio, where = tolerance.check(got, Z, S, fin, fout,
                                               tol=tolerance.bound_epilogue(Z, S, T, epi["alpha"], fin, fout))
        assert ok, f"product {b}: error/bound {ratio:.3g} at {where}"
    return plan, launches


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16, wl.BF16_F32OUT], ids=lambda d: wl.DTYPE_NAMES[d])
def test_batch_in_one_launch(dtype):
    """Six ragged products (300 x 520 x 200), matrices padded apart."""
    M, N, K = 300, 520, 200
    plan, launches = run_batch(6, M, N, K, dtype, M * K + 64, K * N + 8, M * N + 40, seed=500)
    assert launches == 1 and plan.swap_ab == 1


@pytest.mark.parametrize("shared", ["a", "b"])
def test_batch_with_a_shared_operand(shared):
    M, N, K = 257, 264, 136
    sa, sb = (0, K * N) if shared == "a" else (M * K, 0)
    plan, launches = run_batch(5, M, N, K, wl.BF16, sa, sb, M * N, seed=510)
    assert launches == 1


def test_batch_with_epilogue():
    M, N, K = 300, 520, 200
    bias = wl.round_to_format(wl.uniform_pm1(520, N), "bf16")
    epi = {"alpha": 2.0, "beta": 1.0, "activation": 1, "bias": bias}
    plan, launches = run_batch(4, M, N, K, wl.BF16_F32OUT, M * K, K * N, M * N, seed=530, epi=epi)
    assert launches == 1


def test_batch_per_thread_stores():
    """C windows whose starts break 16-byte alignment: the one launch stores C
    per thread."""
    M, N, K = 130, 264, 64
    plan, launches = run_batch(4, M, N, K, wl.BF16, M * K, K * N, M * N + 3, seed=540)
    assert launches == 1


def test_batch_falls_back_to_one_launch_per_product():
    """A stride that breaks 16-byte alignment of the operands: one launch per
    product (any kernel)."""
    M, N, K = 200, 136, 96
    plan, launches = run_batch(3, M, N, K, wl.BF16, M * K + 4, K * N, M * N, seed=550)
    assert launches == 3


def test_batch_fp32_simt():
    M, N, K = 100, 70, 50
    plan, launches = run_batch(3, M, N, K, wl.F32, M * K, K * N, M * N, seed=560)
    assert launches == 3


def test_many_small_products():
    """64 products of 128 x 256 x 512: one launch keeps all pairs busy where one
    product alone fills 1 of 76."""
    M, N, K = 128, 256, 512
    plan, launches = run_batch(64, M, N, K, wl.BF16, M * K, K * N, M * N, seed=570)
    assert launches == 1 and plan.ctas == 2 * min(plan.dp_tiles, 76)


def test_benchmark_batch_every_product():
    """The benchmark's batch (64 products of bf16 512 x 512 x 512, inputs of
    workloads.make_batch_inputs, one launch in the default plan): every element
    of every product against the oracle."""
    lib = H.tg()
    dev = torch.device("cuda:0")
    bw = wl.BATCH_BY_NAME["batch64_bf16_512x512x512"]
    A, B = wl.make_batch_inputs(bw)
    M, N, K, batch = bw.M, bw.N, bw.K, bw.batch
    a = torch.from_numpy(A.view(np.int16)).to(dev)
    b = torch.from_numpy(B.view(np.int16)).to(dev)
    c = torch.zeros((batch * M, N), dtype=torch.int16, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    st = lib.gemm_batched(batch, M, N, K, a.data_ptr(), K, M * K, b.data_ptr(), N, K * N, c.data_ptr(), N, M * N,
                          bw.dtype, None, None, stream)
    assert st == lib.OK, lib.status_string(st)
    assert lib.device_status(stream) == lib.OK
    pst, plan, launches = lib.plan_batched(batch, M, N, K, a.data_ptr(), K, M * K, b.data_ptr(), N, K * N,
                                           c.data_ptr(), N, M * N, bw.dtype, None, 152)
    assert pst == lib.OK and launches == 1
    got_all = wl.decode(c.cpu().numpy().view(np.uint16), "bf16")
    for bi in range(batch):
        Ab, Bb = A[bi * M:(bi + 1) * M], B[bi * K:(bi + 1) * K]
        D, S = oracle.gemm(np.ascontiguousarray(Ab), np.ascontiguousarray(Bb), "bf16", M, N, K)
        ok, ratio, where = tolerance.check(got_all[bi * M:(bi + 1) * M], D, S, "bf16", "bf16")
        assert ok, f"product {bi}: error/bound {ratio:.3g} at {where}"
