"""Helpers of the GPU parity tests: place seeded storage bits in device memory
(optionally at a misaligned offset, with guard bands), call the C ABI, and
compare the result with the oracle under the parity tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl
from tests import tolerance

# NaN patterns no kernel writes; a guard element that changes was overwritten
CANARY = {"f32": 0x7FA1B2C3, "f16": 0x7E5A, "bf16": 0x7FDA}
NP_BITS = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16}
GUARD = 256  # guard elements before and after C


def tg():
    from tests.conftest import build_library
    build_library()
    import tiled_dense_gemm_02_gb300 as lib
    return lib


def device_bytes(nbytes: int, offset: int, dev) -> tuple[torch.Tensor, int]:
    """A byte buffer and a pointer `offset` bytes past a 256-byte boundary."""
    buf = torch.empty(nbytes + offset + 512, dtype=torch.uint8, device=dev)
    base = (buf.data_ptr() + 255) // 256 * 256
    return buf, base + offset


def upload(bits: np.ndarray, offset: int, dev) -> tuple[torch.Tensor, int]:
    raw = np.ascontiguousarray(bits).view(np.uint8).reshape(-1)
    buf, ptr = device_bytes(raw.size, offset, dev)
    start = ptr - buf.data_ptr()
    buf[start:start + raw.size].copy_(torch.from_numpy(raw))
    return buf, ptr


class Result:
    def __init__(self, got, status, plan, guard_ok, pad_ok):
        self.got, self.status, self.plan, self.guard_ok, self.pad_ok = got, status, plan, guard_ok, pad_ok


def run_gpu(A_bits: np.ndarray, B_bits: np.ndarray, M: int, N: int, K: int, dtype: int,
            ldc: int | None = None, a_off: int = 0, b_off: int = 0, c_off: int = 0,
            options=None, dev=None, check_status: bool = True, workspace=None,
            epilogue=None, c_prior: np.ndarray | None = None, bias: np.ndarray | None = None) -> Result:
    """C = A . B on the GPU through the C ABI; A/B given as [rows, ld] bit arrays.

    workspace: None (tgemm_gemm_ex), True (a fresh zeroed workspace of
    tgemm_workspace_size bytes, tgemm_gemm_ws) or a torch uint8 tensor to reuse.
    epilogue: a dict of tgemm_epilogue fields (alpha, beta, activation) for
    tgemm_gemm_epilogue; c_prior (M x N storage bits of C's output format) is
    C's content before the call, bias (N float32 values) goes to the device."""
    lib = tg()
    dev = dev or torch.device("cuda:0")
    fout = wl.OUT_FORMAT[dtype]
    eo = wl.FORMATS[fout][3]
    ldc = N if ldc is None else ldc
    lda, ldb = A_bits.shape[1], B_bits.shape[1]
    a_buf, a_ptr = upload(A_bits, a_off, dev)
    b_buf, b_ptr = upload(B_bits, b_off, dev)
    c_elems = GUARD + M * ldc + GUARD
    c_init = np.full(c_elems, CANARY[fout], dtype=NP_BITS[fout])
    if c_prior is not None:
        window = c_init[GUARD:GUARD + M * ldc].reshape(M, ldc)
        window[:, :N] = c_prior
    c_buf, c_base = upload(c_init, c_off, dev)
    c_ptr = c_base + GUARD * eo
    stream = torch.cuda.current_stream(dev).cuda_stream
    st_plan, plan = lib.plan(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, dtype, options,
                             sm_count=torch.cuda.get_device_properties(dev).multi_processor_count)
    ws_tensor = None
    bias_buf = None
    if epilogue is not None:
        ep = dict(epilogue)
        if bias is not None:
            bias_buf = torch.from_numpy(np.ascontiguousarray(bias, dtype=np.float32)).to(dev)
            ep["bias"] = bias_buf.data_ptr()
        ws_ptr, ws_n = 0, 0
        if workspace is not None:
            st_ws, nbytes = lib.workspace_size(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, dtype, options)
            assert st_ws == lib.OK, lib.status_string(st_ws)
            ws_tensor = torch.zeros(max(nbytes, 1), dtype=torch.uint8, device=dev)
            ws_ptr, ws_n = ws_tensor.data_ptr(), ws_tensor.numel()
            st_plan, plan = lib.plan(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, dtype, options,
                                     sm_count=torch.cuda.get_device_properties(dev).multi_processor_count,
                                     workspace_bytes=ws_n)
        status = lib.gemm_epilogue(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, dtype, ep, options, ws_ptr, ws_n,
                                   stream)
    elif workspace is None:
        status = lib.gemm_ex(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, dtype, options, stream)
    else:
        st_ws, nbytes = lib.workspace_size(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, dtype, options)
        assert st_ws == lib.OK, lib.status_string(st_ws)
        ws_tensor = workspace if isinstance(workspace, torch.Tensor) else torch.zeros(max(nbytes, 1), dtype=torch.uint8,
                                                                                    device=dev)
        assert ws_tensor.data_ptr() % 256 == 0
        if workspace is True:
            assert ws_tensor.numel() >= nbytes
        st_plan, plan = lib.plan(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, dtype, options,
                                 sm_count=torch.cuda.get_device_properties(dev).multi_processor_count,
                                 workspace_bytes=ws_tensor.numel())
        status = lib.gemm_ws(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, dtype, options, ws_tensor.data_ptr(),
                             ws_tensor.numel(), stream)
    dstat = lib.device_status(stream)
    if check_status:
        assert status == lib.OK, lib.status_string(status)
        assert dstat == lib.OK, lib.status_string(dstat)
    start = c_base - c_buf.data_ptr()
    raw = c_buf[start:start + c_elems * eo].cpu().numpy().view(NP_BITS[fout])
    guard_ok = bool(np.all(raw[:GUARD] == CANARY[fout]) and np.all(raw[GUARD + M * ldc:] == CANARY[fout]))
    body = raw[GUARD:GUARD + M * ldc].reshape(M, ldc) if M > 0 else np.zeros((0, ldc), NP_BITS[fout])
    pad_ok = bool(np.all(body[:, N:] == CANARY[fout]))
    got = wl.decode(np.ascontiguousarray(body[:, :N]), fout)
    res = Result(got, (status, dstat), plan, guard_ok, pad_ok)
    res.raw = body[:, :N].copy()
    res.workspace = ws_tensor
    return res


# full oracle products of named workloads, kept for the tests of one process
# that compare several launches of the same workload (at most three: 4096^2
# doubles are 128 MB per array)
_WORKLOAD_REF: dict = {}


def workload_reference(name: str):
    """(A bits, B bits, C_ref, S) of a named workload: the oracle's full product,
    computed once per process."""
    if name not in _WORKLOAD_REF:
        if len(_WORKLOAD_REF) >= 3:
            _WORKLOAD_REF.pop(next(iter(_WORKLOAD_REF)))
        w = wl.BY_NAME[name]
        A, B = wl.make_inputs(w)
        ref, S = oracle.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B), wl.IN_FORMAT[w.dtype], w.M, w.N, w.K)
        _WORKLOAD_REF[name] = (A, B, ref, S)
    return _WORKLOAD_REF[name]


def check_full(res: Result, A_bits, B_bits, M, N, K, dtype, label="", reference=None):
    """Every element of C against the oracle; `reference` = (C_ref, S) when the
    caller already holds the oracle's product of these inputs."""
    fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
    if reference is None:
        ref, S = oracle.gemm(np.ascontiguousarray(A_bits), np.ascontiguousarray(B_bits), fin, M, N, K)
    else:
        ref, S = reference
    ok, ratio, where = tolerance.check(res.got, ref, S, fin, fout)
    assert res.guard_ok, f"{label}: guard band around C overwritten"
    assert res.pad_ok, f"{label}: ldc padding of C overwritten"
    assert ok, (f"{label}: error/bound {ratio:.3g} at {where}: got {res.got[where]} want {ref[where]} "
                f"S {S[where]} plan {res.plan.as_dict()}")
    return ratio


def check_sampled(res: Result, A_bits, B_bits, K, dtype, rows, cols, label=""):
    fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
    ref, S = oracle.entries(np.ascontiguousarray(A_bits), np.ascontiguousarray(B_bits), fin, K, rows, cols)
    ok, ratio, where = tolerance.check(res.got[rows, cols], ref, S, fin, fout)
    assert res.guard_ok and res.pad_ok, f"{label}: guard band or padding overwritten"
    assert ok, f"{label}: error/bound {ratio:.3g} at sample {where} (row {rows[where]}, col {cols[where]})"
    return ratio


def check_block(res: Result, A_bits, B_bits, K, dtype, r0, r1, c0, c1, label=""):
    """Every element of the block C[r0:r1, c0:c1] against the oracle's product
    of those rows of A and columns of B."""
    fin, fout = wl.IN_FORMAT[dtype], wl.OUT_FORMAT[dtype]
    ref, S = oracle.gemm(np.ascontiguousarray(A_bits[r0:r1]), np.ascontiguousarray(B_bits[:, c0:c1]), fin,
                         r1 - r0, c1 - c0, K)
    ok, ratio, where = tolerance.check(res.got[r0:r1, c0:c1], ref, S, fin, fout)
    assert res.guard_ok and res.pad_ok, f"{label}: guard band or padding overwritten"
    assert ok, f"{label}: error/bound {ratio:.3g} at block offset {where} of rows {r0}.. cols {c0}.."
    return ratio


def sample_positions(M: int, N: int, n_random: int, seed: int):
    """Every element of the first and last row and column, the corners of
    every 128-row band, plus `n_random` uniformly drawn positions."""
    r = wl.splitmix64(seed, 2 * n_random)
    rows = [np.zeros(N, np.int64), np.full(N, M - 1, np.int64), np.arange(M), np.arange(M),
            (r[:n_random] % np.uint64(M)).astype(np.int64)]
    cols = [np.arange(N), np.arange(N), np.zeros(M, np.int64), np.full(M, N - 1, np.int64),
            (r[n_random:] % np.uint64(N)).astype(np.int64)]
    return np.concatenate(rows), np.concatenate(cols)
