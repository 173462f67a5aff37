"""Python binding of libtgemm.so, the tiled dense GEMM for GB300 (sm_103a).

The functions below carry the names of the C ABI in ``include/tgemm.h`` and
only marshal arguments; every step of the product runs in the library's CUDA
kernels.  There is no CPU fallback: importing this package raises if the
library has not been built (``python tiled_dense_gemm_02_gb300/build.py``).

``matmul`` is a convenience for torch tensors (torch is used for device memory
and streams only).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libtgemm.so")

# enum tgemm_dtype
F32, F16, BF16, BF16_F32OUT, F16_F32OUT = 0, 1, 2, 3, 4
# enum tgemm_status
OK, ERR_INVALID_VALUE, ERR_UNSUPPORTED_DTYPE, ERR_MISALIGNED, ERR_ALIAS = 0, 1, 2, 3, 4
ERR_UNSUPPORTED_DEVICE, ERR_LAUNCH, ERR_DEVICE_TIMEOUT, ERR_TOO_LARGE = 5, 6, 7, 8
# enum tgemm_kernel
KERNEL_AUTO, KERNEL_TC_TMA, KERNEL_TC_COPY, KERNEL_SIMT = 0, 1, 2, 3
# enum tgemm_activation
ACT_NONE, ACT_RELU = 0, 1

EXPORTS = ("tgemm_gemm", "tgemm_gemm_ex", "tgemm_gemm_ws", "tgemm_workspace_size", "tgemm_plan",
           "tgemm_gemm_noalloc", "tgemm_gemm_epilogue", "tgemm_gemm_batched", "tgemm_plan_batched",
           "tgemm_transpose", "tgemm_gemm_host", "tgemm_device_status", "tgemm_status_string", "tgemm_version",
           "tgemm_host_counters")
# bytes of the scratch array built into the library (TGEMM_NOALLOC_SCRATCH_BYTES)
NOALLOC_SCRATCH_BYTES = 20 * 1024 * 1024 + 4096


class Options(ctypes.Structure):
    """struct tgemm_options"""
    _fields_ = [("kernel", ctypes.c_int), ("tile_n", ctypes.c_int), ("group_m", ctypes.c_int),
                ("max_ctas", ctypes.c_int), ("store_mode", ctypes.c_int), ("wait_timeout_us", ctypes.c_int),
                ("inject_fault", ctypes.c_int), ("cta_group", ctypes.c_int), ("tile_k", ctypes.c_int),
                ("stream_k", ctypes.c_int), ("reserved0", ctypes.c_int),
                ("swap_ab", ctypes.c_int), ("tile_m", ctypes.c_int), ("simt_split", ctypes.c_int),
                ("repack", ctypes.c_int), ("reserved", ctypes.c_int * 1)]


class Epilogue(ctypes.Structure):
    """struct tgemm_epilogue"""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("activation", ctypes.c_int), ("reserved", ctypes.c_int * 3)]


class PlanInfo(ctypes.Structure):
    """struct tgemm_plan_info"""
    _fields_ = [("kernel", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("tile_k", ctypes.c_int), ("stages", ctypes.c_int), ("tiles_m", ctypes.c_int),
                ("tiles_n", ctypes.c_int), ("ctas", ctypes.c_int), ("group_m", ctypes.c_int),
                ("a_copy_bytes", ctypes.c_int), ("b_copy_bytes", ctypes.c_int), ("store_bytes", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("cta_group", ctypes.c_int), ("dp_tiles", ctypes.c_int),
                ("sk_iters", ctypes.c_int), ("workspace_bytes", ctypes.c_int),
                ("cluster_ctas", ctypes.c_int), ("swap_ab", ctypes.c_int), ("tuned", ctypes.c_int),
                ("packed", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_ if name != "reserved"}


class Counters(ctypes.Structure):
    """struct tgemm_counters"""
    _fields_ = [("tc_launches", ctypes.c_uint64), ("map_hits", ctypes.c_uint64), ("map_encodes", ctypes.c_uint64),
                ("ns_prepare", ctypes.c_uint64), ("ns_launch", ctypes.c_uint64)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class TgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


def _load():
    if not os.path.exists(LIBRARY):
        raise ImportError(f"{LIBRARY} is missing: build it with `python tiled_dense_gemm_02_gb300/build.py` "
                          "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIBRARY)
    i64, vp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.tgemm_gemm.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ip, vp]
    lib.tgemm_gemm.restype = ip
    lib.tgemm_gemm_ex.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ip, ctypes.POINTER(Options), vp]
    lib.tgemm_gemm_ex.restype = ip
    lib.tgemm_plan.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ip, ctypes.POINTER(Options),
                               ctypes.c_size_t, ip, ctypes.POINTER(PlanInfo)]
    lib.tgemm_gemm_ws.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ip, ctypes.POINTER(Options), vp,
                                  ctypes.c_size_t, vp]
    lib.tgemm_gemm_ws.restype = ip
    lib.tgemm_workspace_size.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ip, ctypes.POINTER(Options),
                                         ctypes.POINTER(ctypes.c_size_t)]
    lib.tgemm_workspace_size.restype = ip
    lib.tgemm_plan.restype = ip
    lib.tgemm_gemm_noalloc.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ip, ctypes.POINTER(Options), vp]
    lib.tgemm_gemm_noalloc.restype = ip
    lib.tgemm_gemm_epilogue.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ip, ctypes.POINTER(Epilogue),
                                        ctypes.POINTER(Options), vp, ctypes.c_size_t, vp]
    lib.tgemm_gemm_epilogue.restype = ip
    lib.tgemm_gemm_batched.argtypes = [i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64, ip,
                                       ctypes.POINTER(Epilogue), ctypes.POINTER(Options), vp]
    lib.tgemm_gemm_batched.restype = ip
    lib.tgemm_plan_batched.argtypes = [i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64, ip,
                                       ctypes.POINTER(Options), ip, ctypes.POINTER(PlanInfo),
                                       ctypes.POINTER(ctypes.c_int)]
    lib.tgemm_plan_batched.restype = ip
    lib.tgemm_transpose.argtypes = [i64, i64, vp, i64, vp, i64, ip, vp]
    lib.tgemm_transpose.restype = ip
    lib.tgemm_gemm_host.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ip, vp, vp, vp, ip, vp]
    lib.tgemm_gemm_host.restype = ip
    lib.tgemm_device_status.argtypes = [vp]
    lib.tgemm_device_status.restype = ip
    lib.tgemm_status_string.argtypes = [ip]
    lib.tgemm_status_string.restype = ctypes.c_char_p
    lib.tgemm_version.argtypes = []
    lib.tgemm_version.restype = ip
    lib.tgemm_host_counters.argtypes = [ctypes.POINTER(Counters)]
    lib.tgemm_host_counters.restype = ip
    return lib


_lib = _load()


def library():
    """The ctypes handle of libtgemm.so."""
    return _lib


def _opts(options):
    if options is None:
        return None
    if isinstance(options, Options):
        return ctypes.byref(options)
    o = Options()
    for k, v in dict(options).items():
        setattr(o, k, int(v))
    return ctypes.byref(o)


def gemm(M, N, K, A, lda, B, ldb, C, ldc, dtype, stream=0) -> int:
    """tgemm_gemm: raw device pointers (ints) and sizes; returns the status."""
    return _lib.tgemm_gemm(M, N, K, A, lda, B, ldb, C, ldc, dtype, stream)


def gemm_ex(M, N, K, A, lda, B, ldb, C, ldc, dtype, options=None, stream=0) -> int:
    """tgemm_gemm_ex with an Options struct or a dict of its fields."""
    return _lib.tgemm_gemm_ex(M, N, K, A, lda, B, ldb, C, ldc, dtype, _opts(options), stream)


def gemm_ws(M, N, K, A, lda, B, ldb, C, ldc, dtype, options=None, workspace=0, workspace_bytes=0, stream=0) -> int:
    """tgemm_gemm_ws: tgemm_gemm_ex with a caller-owned device workspace."""
    return _lib.tgemm_gemm_ws(M, N, K, A, lda, B, ldb, C, ldc, dtype, _opts(options), workspace, workspace_bytes,
                              stream)


def gemm_noalloc(M, N, K, A, lda, B, ldb, C, ldc, dtype, options=None, stream=0) -> int:
    """tgemm_gemm_noalloc: the stream-K variant with the library's built-in
    scratch array, for callers that cannot allocate device memory."""
    return _lib.tgemm_gemm_noalloc(M, N, K, A, lda, B, ldb, C, ldc, dtype, _opts(options), stream)


def _epi(epilogue):
    if epilogue is None:
        return None
    if isinstance(epilogue, Epilogue):
        return ctypes.byref(epilogue)
    e = Epilogue(alpha=1.0, beta=0.0, bias=None, activation=ACT_NONE)
    for k, v in dict(epilogue).items():
        setattr(e, k, v)
    return ctypes.byref(e)


def gemm_epilogue(M, N, K, A, lda, B, ldb, C, ldc, dtype, epilogue=None, options=None, workspace=0,
                  workspace_bytes=0, stream=0) -> int:
    """tgemm_gemm_epilogue: C = act(alpha A.B + beta C + bias) with an Epilogue
    struct or a dict of its fields (alpha, beta, bias as a device pointer int,
    activation); workspace as in gemm_ws."""
    return _lib.tgemm_gemm_epilogue(M, N, K, A, lda, B, ldb, C, ldc, dtype, _epi(epilogue), _opts(options),
                                    workspace, workspace_bytes, stream)


def gemm_batched(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, C, ldc, stride_c, dtype, epilogue=None,
                 options=None, stream=0) -> int:
    """tgemm_gemm_batched: `batch` products with element strides between matrices."""
    return _lib.tgemm_gemm_batched(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, C, ldc, stride_c, dtype,
                                   _epi(epilogue), _opts(options), stream)


def plan_batched(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, C, ldc, stride_c, dtype, options=None,
                 sm_count=148):
    """tgemm_plan_batched: (status, PlanInfo of one launch, kernel launches of the call)."""
    info = PlanInfo()
    n = ctypes.c_int(0)
    st = _lib.tgemm_plan_batched(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, C, ldc, stride_c, dtype,
                                 _opts(options), sm_count, ctypes.byref(info), ctypes.byref(n))
    return st, info, n.value


def transpose(rows, cols, src, ld_src, dst, ld_dst, elem_bytes, stream=0) -> int:
    """tgemm_transpose: dst (cols x rows) = src (rows x cols) transposed."""
    return _lib.tgemm_transpose(rows, cols, src, ld_src, dst, ld_dst, elem_bytes, stream)


def gemm_host(M, N, K, A_host, lda, B_host, ldb, C_host, ldc, dtype, dA, dB, dC, panels=0, stream=0) -> int:
    """tgemm_gemm_host: A, B, C in host memory (pointers as ints), staged through
    the caller's device buffers dA, dB, dC; returns the status."""
    return _lib.tgemm_gemm_host(M, N, K, A_host, lda, B_host, ldb, C_host, ldc, dtype, dA, dB, dC, panels, stream)


def workspace_size(M, N, K, A, lda, B, ldb, C, ldc, dtype, options=None):
    """tgemm_workspace_size: (status, bytes) on the current device."""
    n = ctypes.c_size_t(0)
    st = _lib.tgemm_workspace_size(M, N, K, A, lda, B, ldb, C, ldc, dtype, _opts(options), ctypes.byref(n))
    return st, n.value


def plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, options=None, sm_count=148, workspace_bytes=0):
    """tgemm_plan: (status, PlanInfo) of the dispatch decision; no GPU needed."""
    info = PlanInfo()
    st = _lib.tgemm_plan(M, N, K, A, lda, B, ldb, C, ldc, dtype, _opts(options), workspace_bytes, sm_count,
                         ctypes.byref(info))
    return st, info


def device_status(stream=0) -> int:
    """tgemm_device_status: synchronise `stream`, return and clear the device status."""
    return _lib.tgemm_device_status(stream)


def status_string(status: int) -> str:
    return _lib.tgemm_status_string(status).decode()


def version() -> int:
    return _lib.tgemm_version()


def host_counters() -> dict:
    """tgemm_host_counters: cumulative tensor-core launches, tensor-map cache
    hits and encodes, and host nanoseconds before and inside the launches."""
    c = Counters()
    st = _lib.tgemm_host_counters(ctypes.byref(c))
    if st != OK:
        raise TgemmError(st, "tgemm_host_counters")
    return c.as_dict()


# ------------------------------------------------------------ torch helpers

def _torch_dtype_code(a_dtype, out_dtype):
    import torch
    table = {
        (torch.float32, torch.float32): F32,
        (torch.float16, torch.float16): F16,
        (torch.bfloat16, torch.bfloat16): BF16,
        (torch.bfloat16, torch.float32): BF16_F32OUT,
        (torch.float16, torch.float32): F16_F32OUT,
    }
    if (a_dtype, out_dtype) not in table:
        raise ValueError(f"unsupported (input, output) dtypes: {a_dtype}, {out_dtype}")
    return table[(a_dtype, out_dtype)]


def matmul(a, b, out=None, out_dtype=None, options=None, stream=None):
    """C = a @ b for 2-D CUDA tensors with unit column stride (row-major rows,
    any row stride).  Returns ``out`` (allocated by torch if None)."""
    import torch
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError("expected a [M, K] and b [K, N]")
    if a.dtype != b.dtype:
        raise ValueError("a and b must have the same dtype")
    M, K = a.shape
    N = b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or a.dtype, device=a.device)
    for name, t in (("a", a), ("b", b), ("out", out)):
        if t.numel() and t.stride(1) != 1:
            raise ValueError(f"{name} must have unit column stride")
    code = _torch_dtype_code(a.dtype, out.dtype)
    s = stream if stream is not None else torch.cuda.current_stream(a.device).cuda_stream
    lda = max(a.stride(0), 1) if M > 1 else max(K, 1)
    ldb = max(b.stride(0), 1) if K > 1 else max(N, 1)
    ldc = max(out.stride(0), 1) if M > 1 else max(N, 1)
    with torch.cuda.device(a.device):
        st = gemm_ex(M, N, K, a.data_ptr(), lda, b.data_ptr(), ldb, out.data_ptr(), ldc, code, options, s)
    if st != OK:
        raise TgemmError(st, "tgemm_gemm_ex")
    return out
