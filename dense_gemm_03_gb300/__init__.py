"""Python binding of libgemm.so, the GB300 dense GEMM library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI (include/gemm.h).  Loading fails loudly when the
compiled library is missing -- there is no Python or CPU fallback.

Operands may be given as torch tensors (device memory for the device forms,
host memory for the ``*_host`` forms) or as raw integer addresses.  Leading
dimensions default to the natural row-major ones (lda=K, ldb=N, ldc=N).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "GemmError", "lib", "library_path", "gemm_f16", "gemm_f16_f32out", "f32_to_f16",
    "sgemm_f32", "gemm_f16_host",
    "sgemm_f32_host", "gemm_f16_splitk_noalloc", "l2_flush", "force_path", "force_splits", "stage_kblocks",
    "set_wait_limit_ns",
    "debug_status", "last_path", "launch_count", "plan_stream_k", "release", "EXPORTS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libgemm.so")
_lock = threading.Lock()
_lib = None

# Every symbol include/gemm.h declares.
EXPORTS = (
    "gemm_f16", "gemm_f16_ld", "sgemm_f32", "sgemm_f32_ld", "gemm_f16_host", "sgemm_f32_host",
    "gemm_l2_flush", "gemm_force_path", "gemm_force_splits", "gemm_set_wait_limit_ns",
    "gemm_debug_status", "gemm_last_path", "gemm_strerror", "gemm_release",
    "gemm_f16_splitk_noalloc", "gemm_launch_count", "gemm_plan_stream_k", "gemm_f16_f32out",
    "gemm_f32_to_f16", "gemm_debug_wait_probe", "gemm_plan_tf32_slices", "gemm_stage_kblocks",
)

PATH_AUTO, PATH_TMA, PATH_MANUAL, PATH_SPLITK, PATH_F32_SCALAR = 0, 1, 2, 3, 4


class GemmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib().gemm_strerror(code).decode() if _lib is not None else str(code)
        super().__init__("%s failed: %s (%d)" % (where, msg, code))


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded library (ctypes.CDLL).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError("libgemm.so is not built (run __graft_entry__.build() or "
                                  "python dense_gemm_03_gb300/build.py)")
            L = ctypes.CDLL(_LIB_PATH)
            vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            for name in ("gemm_f16", "sgemm_f32"):
                fn = getattr(L, name)
                fn.restype = i
                fn.argtypes = [vp, vp, vp, i, i, i, f, f, vp]
            for name in ("gemm_f16_ld", "sgemm_f32_ld", "gemm_f16_host", "sgemm_f32_host"):
                fn = getattr(L, name)
                fn.restype = i
                fn.argtypes = [vp, vp, vp, i, i, i, i, i, i, f, f, vp]
            L.gemm_debug_wait_probe.restype = i
            L.gemm_debug_wait_probe.argtypes = [ctypes.c_longlong, vp]
            L.gemm_f16_f32out.restype = i
            L.gemm_f16_f32out.argtypes = [vp, vp, vp, i, i, i, i, i, i, f, f, vp]
            L.gemm_f32_to_f16.restype = i
            L.gemm_f32_to_f16.argtypes = [vp, vp, ctypes.c_longlong, vp]
            L.gemm_f16_splitk_noalloc.restype = i
            L.gemm_f16_splitk_noalloc.argtypes = [vp, vp, vp, i, i, i, i, i, i, f, f, i, vp]
            L.gemm_l2_flush.restype = i
            L.gemm_l2_flush.argtypes = [ctypes.c_size_t, vp]
            L.gemm_force_path.restype = i
            L.gemm_force_path.argtypes = [i]
            L.gemm_force_splits.restype = i
            L.gemm_force_splits.argtypes = [i]
            L.gemm_stage_kblocks.restype = i
            L.gemm_stage_kblocks.argtypes = [i]
            L.gemm_set_wait_limit_ns.restype = ctypes.c_longlong
            L.gemm_set_wait_limit_ns.argtypes = [ctypes.c_longlong]
            L.gemm_debug_status.restype = i
            L.gemm_debug_status.argtypes = []
            L.gemm_plan_stream_k.restype = i
            L.gemm_plan_stream_k.argtypes = [ctypes.c_longlong, ctypes.c_longlong, i, i,
                                             ctypes.POINTER(ctypes.c_longlong)]
            L.gemm_plan_tf32_slices.restype = i
            L.gemm_plan_tf32_slices.argtypes = [ctypes.c_longlong, ctypes.c_longlong, i, i,
                                                ctypes.POINTER(ctypes.c_longlong)]
            L.gemm_launch_count.restype = ctypes.c_longlong
            L.gemm_launch_count.argtypes = []
            L.gemm_last_path.restype = ctypes.c_char_p
            L.gemm_last_path.argtypes = []
            L.gemm_strerror.restype = ctypes.c_char_p
            L.gemm_strerror.argtypes = [i]
            L.gemm_release.restype = i
            L.gemm_release.argtypes = []
            _lib = L
    return _lib


def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):                      # numpy array
        return x.ctypes.data
    raise TypeError("expected a tensor, an array or an address, got %r" % type(x))


_current_stream = None


def _current_stream_fn():
    """A cheap getter of the current CUDA stream's handle (None without CUDA)."""
    global _current_stream
    if _current_stream is None:
        fn = lambda: None
        try:
            import torch
            if torch.cuda.is_available():
                raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
                dev = getattr(torch._C, "_cuda_getDevice", None)
                if raw is not None and dev is not None:
                    fn = lambda: raw(dev())
                else:
                    fn = lambda: torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        _current_stream = fn
    return _current_stream


def _stream(stream):
    if stream is None:
        return _current_stream_fn()()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dims(A, B, M, N, K):
    if M is None:
        M = A.shape[0]
    if K is None:
        K = A.shape[1]
    if N is None:
        N = B.shape[1]
    return int(M), int(N), int(K)


def _check(rc: int, where: str):
    if rc != 0:
        raise GemmError(rc, where)


def gemm_f16(A, B, C, alpha=1.0, beta=0.0, M=None, N=None, K=None, lda=None, ldb=None, ldc=None,
             stream=None):
    """C := alpha*A*B + beta*C on device fp16 operands (fp32 accumulation)."""
    M, N, K = _dims(A, B, M, N, K)
    L = lib()
    s = _stream(stream)
    if lda is None and ldb is None and ldc is None:
        rc = L.gemm_f16(_addr(A), _addr(B), _addr(C), M, N, K, float(alpha), float(beta), s)
    else:
        rc = L.gemm_f16_ld(_addr(A), _addr(B), _addr(C), M, N, K,
                           int(K if lda is None else lda), int(N if ldb is None else ldb),
                           int(N if ldc is None else ldc), float(alpha), float(beta), s)
    _check(rc, "gemm_f16")


def gemm_f16_f32out(A, B, C, alpha=1.0, beta=0.0, M=None, N=None, K=None, lda=None, ldb=None,
                    ldc=None, stream=None):
    """C := alpha*A*B + beta*C with device fp16 A, B and an fp32 C."""
    M, N, K = _dims(A, B, M, N, K)
    rc = lib().gemm_f16_f32out(_addr(A), _addr(B), _addr(C), M, N, K,
                               int(K if lda is None else lda), int(N if ldb is None else ldb),
                               int(N if ldc is None else ldc), float(alpha), float(beta),
                               _stream(stream))
    _check(rc, "gemm_f16_f32out")


def f32_to_f16(src, dst, n=None, stream=None):
    """dst := src rounded to half (nearest, ties to even), n elements."""
    if n is None:
        n = src.numel() if hasattr(src, "numel") else src.size
    _check(lib().gemm_f32_to_f16(_addr(src), _addr(dst), int(n), _stream(stream)),
           "gemm_f32_to_f16")


def sgemm_f32(A, B, C, alpha=1.0, beta=0.0, M=None, N=None, K=None, lda=None, ldb=None, ldc=None,
              stream=None):
    """C := alpha*A*B + beta*C on device fp32 operands."""
    M, N, K = _dims(A, B, M, N, K)
    L = lib()
    s = _stream(stream)
    if lda is None and ldb is None and ldc is None:
        rc = L.sgemm_f32(_addr(A), _addr(B), _addr(C), M, N, K, float(alpha), float(beta), s)
    else:
        rc = L.sgemm_f32_ld(_addr(A), _addr(B), _addr(C), M, N, K,
                            int(K if lda is None else lda), int(N if ldb is None else ldb),
                            int(N if ldc is None else ldc), float(alpha), float(beta), s)
    _check(rc, "sgemm_f32")


def gemm_f16_host(A, B, C, alpha=1.0, beta=0.0, M=None, N=None, K=None, lda=None, ldb=None,
                  ldc=None, stream=None):
    """Host-buffer form: copies in, computes, copies C back, synchronises."""
    M, N, K = _dims(A, B, M, N, K)
    rc = lib().gemm_f16_host(_addr(A), _addr(B), _addr(C), M, N, K,
                             int(K if lda is None else lda), int(N if ldb is None else ldb),
                             int(N if ldc is None else ldc), float(alpha), float(beta),
                             _stream(stream))
    _check(rc, "gemm_f16_host")


def sgemm_f32_host(A, B, C, alpha=1.0, beta=0.0, M=None, N=None, K=None, lda=None, ldb=None,
                   ldc=None, stream=None):
    """Host-buffer fp32 form: copies in, computes, copies C back, synchronises."""
    M, N, K = _dims(A, B, M, N, K)
    rc = lib().sgemm_f32_host(_addr(A), _addr(B), _addr(C), M, N, K,
                              int(K if lda is None else lda), int(N if ldb is None else ldb),
                              int(N if ldc is None else ldc), float(alpha), float(beta),
                              _stream(stream))
    _check(rc, "sgemm_f32_host")


def gemm_f16_splitk_noalloc(A, B, C, alpha=1.0, beta=0.0, M=None, N=None, K=None, lda=None,
                            ldb=None, ldc=None, splits=0, stream=None):
    """Split-K fp16 GEMM on the library's fixed static scratch array: never
    allocates device memory (for callers that must not).  Raises GemmError
    (GEMM_ERR_ARG) when the partial sums would not fit the array."""
    M, N, K = _dims(A, B, M, N, K)
    rc = lib().gemm_f16_splitk_noalloc(_addr(A), _addr(B), _addr(C), M, N, K,
                                       int(K if lda is None else lda), int(N if ldb is None else ldb),
                                       int(N if ldc is None else ldc), float(alpha), float(beta),
                                       int(splits), _stream(stream))
    _check(rc, "gemm_f16_splitk_noalloc")


def l2_flush(nbytes: int = 0, stream=None):
    _check(lib().gemm_l2_flush(int(nbytes), _stream(stream)), "gemm_l2_flush")


def force_path(path: int) -> int:
    prev = lib().gemm_force_path(int(path))
    if prev < 0:
        raise GemmError(prev, "gemm_force_path")
    return prev


def force_splits(splits: int) -> int:
    prev = lib().gemm_force_splits(int(splits))
    if prev < 0:
        raise GemmError(prev, "gemm_force_splits")
    return prev


def stage_kblocks(kblocks: int) -> int:
    prev = lib().gemm_stage_kblocks(int(kblocks))
    if prev < 0:
        raise GemmError(prev, "gemm_stage_kblocks")
    return prev


def set_wait_limit_ns(ns: int) -> int:
    return int(lib().gemm_set_wait_limit_ns(int(ns)))


def debug_status() -> int:
    return int(lib().gemm_debug_status())


def last_path() -> str:
    return lib().gemm_last_path().decode()


def plan_stream_k(tiles: int, slots: int, kb: int, all_tiles: bool = False,
                  tail: bool = False) -> dict:
    """The stream-K plan of the half-precision path (host-side query):
    the last two waves, all tiles (``all_tiles``) or the last partial wave
    (``tail``)."""
    out = (ctypes.c_longlong * 4)()
    mode = 2 if tail else int(bool(all_tiles))
    _check(lib().gemm_plan_stream_k(tiles, slots, kb, mode, out), "gemm_plan_stream_k")
    return {"dp_tiles": out[0], "sk_tiles": out[1], "workers": out[2], "max_pieces": out[3]}


def plan_tf32_slices(tiles: int, pairs: int, kb: int, forced_slices: int = 0) -> dict:
    """The K-slice plan of the fp32 tensor-core path (host-side query)."""
    out = (ctypes.c_longlong * 2)()
    _check(lib().gemm_plan_tf32_slices(tiles, pairs, kb, forced_slices, out),
           "gemm_plan_tf32_slices")
    return {"splits": out[0], "kb_per_split": out[1]}


def debug_wait_probe(limit_ns: int, stream=None):
    """Launches a wait on a barrier that nothing releases; it gives up after
    limit_ns and the next debug_status() returns GEMM_ERR_TIMEOUT (-6)."""
    _check(lib().gemm_debug_wait_probe(int(limit_ns), _stream(stream)), "gemm_debug_wait_probe")


def launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(lib().gemm_launch_count())


def release():
    _check(lib().gemm_release(), "gemm_release")
