"""GPU parity of tgemm_gemm_host: A, B and C in host memory (page-locked or
pageable), copied in row panels through caller-owned device buffers, against
the oracle.  Padding columns of C's host rows (ldc > N) must keep their
canary, and a second call that reuses the device buffers must see its own
inputs (the call's copies follow the work already on the stream).
"""
import numpy as np
import pytest
import torch

import oracle
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


def host_buffer(bits: np.ndarray, pinned: bool):
    """A host copy of `bits` (pinned torch tensor or plain numpy array) and its address."""
    if pinned:
        t = torch.from_numpy(np.ascontiguousarray(bits)).pin_memory()
        return t, t.data_ptr()
    a = np.ascontiguousarray(bits).copy()
    return a, a.ctypes.data


def run_host(M, N, K, dtype, seed, lda=None, ldb=None, ldc=None, panels=0, pinned=True, dev_bufs=None):
    lib = H.tg()
    dev = torch.device("cuda:0")
    fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
    ldc = N if ldc is None else ldc
    if K > 0:
        A, B = wl.make_inputs(wl.Workload("host", M, N, K, dtype, "uniform", seed), lda=lda, ldb=ldb)
    else:
        A = np.zeros((M, 1), dtype=H.NP_BITS[fin])
        B = np.zeros((1, N), dtype=H.NP_BITS[fin])
    a_h, a_ptr = host_buffer(A, pinned)
    b_h, b_ptr = host_buffer(B, pinned)
    c_init = np.full((M, ldc), H.CANARY[fout], dtype=H.NP_BITS[fout])
    c_h, c_ptr = host_buffer(c_init, pinned)
    ei, eo = wl.FORMATS[fin][3], wl.FORMATS[fout][3]
    if dev_bufs is None:
        dev_bufs = [torch.empty(max(n, 1) * e, dtype=torch.uint8, device=dev)
                    for n, e in ((M * K, ei), (K * N, ei), (M * N, eo))]
    dA, dB, dC = dev_bufs
    stream = torch.cuda.current_stream(dev).cuda_stream
    st = lib.gemm_host(M, N, K, a_ptr, A.shape[1], b_ptr, B.shape[1], c_ptr, ldc, dtype,
                       dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), panels, stream)
    assert st == lib.OK, lib.status_string(st)
    torch.cuda.synchronize()
    assert lib.device_status(stream) == lib.OK
    raw = (c_h.numpy() if pinned else c_h).view(H.NP_BITS[fout]).reshape(M, ldc)
    assert np.all(raw[:, N:] == H.CANARY[fout]), "a padding element of C's host rows was written"
    got = wl.decode(np.ascontiguousarray(raw[:, :N]), fout)
    if K > 0:
        D, S = oracle.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B), fin, M, N, K)
    else:
        D, S = np.zeros((M, N)), np.zeros((M, N))
    ok, ratio, where = tolerance.check(got, D, S, fin, fout)
    assert ok, f"{M}x{N}x{K} {wl.DTYPE_NAMES[dtype]} panels {panels}: error/bound {ratio:.3g} at {where}"
    return dev_bufs


@pytest.mark.parametrize("panels", [0, 1, 3])
def test_ragged_product_from_host(panels):
    """The ragged 1000 x 1500 x 4096 bf16 product (3000-byte rows) from pinned memory."""
    run_host(1000, 1500, 4096, wl.BF16, seed=90, panels=panels)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16_F32OUT, wl.F32], ids=lambda d: wl.DTYPE_NAMES[d])
def test_padded_host_rows(dtype):
    """Leading dimensions above the extents on the host side; the device copies are dense."""
    run_host(300, 520, 200, dtype, seed=91, lda=208, ldb=530, ldc=533, panels=3)


def test_pageable_host_memory():
    run_host(513, 300, 1000, wl.BF16, seed=92, pinned=False, panels=2)


def test_k_zero_from_host():
    run_host(130, 70, 0, wl.BF16, seed=93)


def test_reused_device_buffers_see_each_calls_inputs():
    bufs = run_host(700, 400, 300, wl.BF16, seed=94, panels=2)
    run_host(700, 400, 300, wl.BF16, seed=95, panels=4, dev_bufs=bufs)


def test_graduated_panels_from_host():
    """C of 8 MB (fp32 2048 x 1024): the automatic schedule takes graduated
    panels of 128, 128, 256, 512, 512 and 512 rows; the product is checked
    against the oracle like every other schedule."""
    run_host(2048, 1024, 512, wl.BF16_F32OUT, seed=96)


@pytest.mark.parametrize("dtype,panels", [(wl.F16_F32OUT, 3), (wl.BF16_F32OUT, 0), (wl.BF16, 3)],
                         ids=["f16_f32out_3", "bf16_f32out_auto", "bf16_3"])
def test_first_panel_in_two_k_halves(dtype, panels):
    """fp32 output with several panels and K >= 256: the first panel's product
    runs in two K halves (the second added onto the first as B's second half
    arrives); with padded host rows, a K that is not a multiple of the 64-deep
    split point's step, and a 16-bit output for contrast (one pass)."""
    run_host(1300, 1300, 700, dtype, seed=97, lda=712, ldb=1308, ldc=1303, panels=panels)  # fp32 C: 6.8 MB


def test_host_calls_from_several_threads():
    """Three host threads, each on its own stream with its own buffers, call
    tgemm_gemm_host three times in a row (fp32 output in three panels, so the
    first panel runs in two K halves).  The calls share the library's copy
    streams and its pool of events; every product is checked against the
    oracle and every padding element of C's host rows keeps its canary."""
    import threading
    lib = H.tg()
    dev = torch.device("cuda:0")
    M, N, K, dtype = 700, 900, 512, wl.BF16_F32OUT
    fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
    ldc = N + 4
    errors = []

    def worker(w):
        try:
            torch.cuda.set_device(0)
            stream = torch.cuda.Stream(device=dev)
            dA = torch.empty(M * K * 2, dtype=torch.uint8, device=dev)
            dB = torch.empty(K * N * 2, dtype=torch.uint8, device=dev)
            dC = torch.empty(M * N * 4, dtype=torch.uint8, device=dev)
            for call in range(3):
                A, B = wl.make_inputs(wl.Workload("host_threads", M, N, K, dtype, "uniform", 200 + 10 * w + call))
                a_h, a_ptr = host_buffer(A, True)
                b_h, b_ptr = host_buffer(B, True)
                c_h, c_ptr = host_buffer(np.full((M, ldc), H.CANARY[fout], dtype=H.NP_BITS[fout]), True)
                st = lib.gemm_host(M, N, K, a_ptr, K, b_ptr, N, c_ptr, ldc, dtype, dA.data_ptr(), dB.data_ptr(),
                                   dC.data_ptr(), 3, stream.cuda_stream)
                assert st == lib.OK, lib.status_string(st)
                stream.synchronize()
                assert lib.device_status(stream.cuda_stream) == lib.OK
                raw = c_h.numpy().view(H.NP_BITS[fout]).reshape(M, ldc)
                assert np.all(raw[:, N:] == H.CANARY[fout]), "a padding element of C's host rows was written"
                got = wl.decode(np.ascontiguousarray(raw[:, :N]), fout)
                D, S = oracle.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B), fin, M, N, K)
                ok, ratio, where = tolerance.check(got, D, S, fin, fout)
                assert ok, f"thread {w} call {call}: error/bound {ratio:.3g} at {where}"
        except Exception as exc:  # reported by the main thread
            errors.append(repr(exc))

    threads = [threading.Thread(target=worker, args=(w,)) for w in range(3)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
