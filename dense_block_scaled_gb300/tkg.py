"""ctypes binding of libtkg.so (C ABI in include/tkg_gemm.h).

Argument marshalling only: every entry point forwards device pointers, sizes
and a CUDA stream handle to the library; all arithmetic runs in the library's
CUDA kernels.  The library is built in-tree (``python -m
dense_block_scaled_gb300.build``); if it is missing or fails to load, every
call raises -- there is no fallback path.

Helpers accept torch tensors only as carriers of device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
# TKG_LIBRARY selects another build of the library, e.g. libtkg_check.so
LIB_PATH = os.environ.get("TKG_LIBRARY") or os.path.join(PKG, "libtkg.so")

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_CHECK = range(7)
OPT_CTA_GROUP, OPT_SINGLE_STAGE, OPT_TIMEOUT_MS, OPT_INJECT_STALL, OPT_MAX_CLUSTERS, OPT_ACC_STAGES = 1, 2, 3, 4, 5, 6
OPT_SCHEDULER = 7
OPT_SPLIT_K = 8
OPT_RASTER_GROUP = 9
OPT_BF16_TILE_N = 10
OPT_TAIL_SPLIT = 11
OPT_EPILOGUE_STORE = 12

EXPORTS = [
    "tkg_gemm_bf16", "tkg_gemm_mxfp8", "tkg_gemm_nvfp4", "tkg_get_device_status", "tkg_status_string",
    "tkg_scale_bytes", "tkg_scales_to_tiled", "tkg_quantize_mxfp8", "tkg_quantize_nvfp4",
    "tkg_set_option", "tkg_get_option", "tkg_gemm_bf16_noalloc",
    "tkg_gemm_grouped_bf16", "tkg_gemm_grouped_mxfp8", "tkg_gemm_grouped_nvfp4", "tkg_grouped_scale_bytes",
    "tkg_gemm_bf16_from_host", "tkg_gemm_grouped_dev_bf16", "tkg_gemm_grouped_dev_mxfp8",
    "tkg_gemm_grouped_dev_nvfp4", "tkg_grouped_dev_scale_bytes", "tkg_quantize_nvfp4_scaled",
    "tkg_gemm_list_bf16", "tkg_gemm_list_mxfp8", "tkg_gemm_list_nvfp4",
    "tkg_gemm_bf16_strided", "tkg_gemm_mxfp8_strided", "tkg_gemm_nvfp4_strided",
]

MAX_LIST = 16


class GemmDesc(ctypes.Structure):
    """tkg_gemm_desc: one GEMM of a list (device pointers, sizes, alpha)."""
    _fields_ = [("m", ctypes.c_int), ("n", ctypes.c_int), ("k", ctypes.c_int),
                ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("sfa", ctypes.c_void_p), ("sfb", ctypes.c_void_p),
                ("tensor_scale_a", ctypes.c_void_p), ("tensor_scale_b", ctypes.c_void_p),
                ("D", ctypes.c_void_p), ("alpha", ctypes.c_float)]

_lock = threading.Lock()
_lib = None


class TkgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Load libtkg.so (raises if it has not been built)."""
    global _lib
    lib = _lib
    if lib is not None:   # loaded: no lock on the per-call path
        return lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m dense_block_scaled_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            i, vp, f, st = ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
            lib.tkg_gemm_bf16.argtypes = [i, i, i, vp, vp, vp, f, vp]
            lib.tkg_gemm_bf16_noalloc.argtypes = [i, i, i, vp, vp, vp, f, vp]
            lib.tkg_gemm_mxfp8.argtypes = [i, i, i, vp, vp, vp, vp, vp, f, vp]
            lib.tkg_gemm_nvfp4.argtypes = [i, i, i, vp, vp, vp, vp, vp, vp, vp, f, vp]
            lib.tkg_gemm_grouped_bf16.argtypes = [i, vp, i, i, vp, vp, vp, f, vp]
            lib.tkg_gemm_grouped_mxfp8.argtypes = [i, vp, i, i, vp, vp, vp, vp, vp, f, vp]
            lib.tkg_gemm_grouped_nvfp4.argtypes = [i, vp, i, i, vp, vp, vp, vp, vp, vp, vp, f, vp]
            lib.tkg_grouped_scale_bytes.argtypes = [i, vp, i, i]
            lib.tkg_grouped_scale_bytes.restype = ctypes.c_size_t
            lib.tkg_gemm_bf16_from_host.argtypes = [i, i, i, vp, vp, vp, vp, vp, vp, f, vp]
            lib.tkg_gemm_grouped_dev_bf16.argtypes = [i, vp, i, i, i, vp, vp, vp, f, vp]
            lib.tkg_gemm_grouped_dev_mxfp8.argtypes = [i, vp, i, i, i, vp, vp, vp, vp, vp, f, vp]
            lib.tkg_gemm_grouped_dev_nvfp4.argtypes = [i, vp, i, i, i, vp, vp, vp, vp, vp, vp, vp, f, vp]
            lib.tkg_grouped_dev_scale_bytes.argtypes = [i, i, i, i]
            lib.tkg_grouped_dev_scale_bytes.restype = ctypes.c_size_t
            for name in ("tkg_gemm_list_bf16", "tkg_gemm_list_mxfp8", "tkg_gemm_list_nvfp4"):
                getattr(lib, name).argtypes = [i, ctypes.POINTER(GemmDesc), vp]
                getattr(lib, name).restype = ctypes.c_int
            lib.tkg_gemm_bf16_strided.argtypes = [i, i, i, vp, i, vp, i, vp, i, f, vp]
            lib.tkg_gemm_mxfp8_strided.argtypes = [i, i, i, vp, i, vp, i, vp, vp, vp, i, f, vp]
            lib.tkg_gemm_nvfp4_strided.argtypes = [i, i, i, vp, i, vp, i, vp, vp, vp, vp, vp, i, f, vp]
            for name in ("tkg_gemm_bf16_strided", "tkg_gemm_mxfp8_strided", "tkg_gemm_nvfp4_strided"):
                getattr(lib, name).restype = ctypes.c_int
            lib.tkg_get_device_status.argtypes = [vp]
            lib.tkg_status_string.argtypes = [st]
            lib.tkg_status_string.restype = ctypes.c_char_p
            lib.tkg_scale_bytes.argtypes = [i, i, i]
            lib.tkg_scale_bytes.restype = ctypes.c_size_t
            lib.tkg_scales_to_tiled.argtypes = [i, i, vp, i, vp, vp]
            lib.tkg_quantize_mxfp8.argtypes = [i, i, vp, vp, vp, vp]
            lib.tkg_quantize_nvfp4.argtypes = [i, i, vp, vp, vp, vp, vp]
            lib.tkg_quantize_nvfp4_scaled.argtypes = [i, i, vp, vp, vp, vp, vp]
            lib.tkg_set_option.argtypes = [i, i]
            lib.tkg_get_option.argtypes = [i]
            for name in ("tkg_gemm_bf16", "tkg_gemm_bf16_noalloc", "tkg_gemm_mxfp8", "tkg_gemm_nvfp4", "tkg_get_device_status",
                         "tkg_scales_to_tiled", "tkg_quantize_mxfp8", "tkg_quantize_nvfp4",
                         "tkg_quantize_nvfp4_scaled", "tkg_set_option",
                         "tkg_get_option"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().tkg_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise TkgError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- raw C calls (pointers)

def gemm_bf16_raw(m, n, k, A, B, D, alpha, stream) -> int:
    return load().tkg_gemm_bf16(m, n, k, A, B, D, ctypes.c_float(alpha), stream)


def gemm_bf16_noalloc_raw(m, n, k, A, B, D, alpha, stream) -> int:
    return load().tkg_gemm_bf16_noalloc(m, n, k, A, B, D, ctypes.c_float(alpha), stream)


def gemm_mxfp8_raw(m, n, k, A, B, sfa, sfb, D, alpha, stream) -> int:
    return load().tkg_gemm_mxfp8(m, n, k, A, B, sfa, sfb, D, ctypes.c_float(alpha), stream)


def gemm_nvfp4_raw(m, n, k, A, B, sfa, sfb, ta, tb, D, alpha, stream) -> int:
    return load().tkg_gemm_nvfp4(m, n, k, A, B, sfa, sfb, ta, tb, D, ctypes.c_float(alpha), stream)


def _sizes(m_sizes):
    """Host int32 array of group sizes (kept alive by the caller's reference)."""
    arr = (ctypes.c_int * len(m_sizes))(*[int(x) for x in m_sizes])
    return arr, len(m_sizes)


def gemm_grouped_bf16_raw(groups, m_sizes, n, k, A, B, D, alpha, stream) -> int:
    return load().tkg_gemm_grouped_bf16(groups, m_sizes, n, k, A, B, D, ctypes.c_float(alpha), stream)


def gemm_grouped_mxfp8_raw(groups, m_sizes, n, k, A, B, sfa, sfb, D, alpha, stream) -> int:
    return load().tkg_gemm_grouped_mxfp8(groups, m_sizes, n, k, A, B, sfa, sfb, D, ctypes.c_float(alpha), stream)


def gemm_grouped_nvfp4_raw(groups, m_sizes, n, k, A, B, sfa, sfb, ta, tb, D, alpha, stream) -> int:
    return load().tkg_gemm_grouped_nvfp4(groups, m_sizes, n, k, A, B, sfa, sfb, ta, tb, D, ctypes.c_float(alpha),
                                         stream)


# ---------------------------------------------------------------- tensor helpers

def gemm_bf16(A, B, D, alpha: float = 1.0, stream=None) -> None:
    """D (m x n bf16) = alpha * A (m x k bf16) @ B (n x k bf16)^T."""
    m, k = A.shape
    n = B.shape[0]
    _check(gemm_bf16_raw(m, n, k, _ptr(A), _ptr(B), _ptr(D), alpha, _stream(stream)), "tkg_gemm_bf16")


def gemm_bf16_noalloc(A, B, D, alpha: float = 1.0, stream=None) -> None:
    """As gemm_bf16, through the entry point that allocates no device memory."""
    m, k = A.shape
    n = B.shape[0]
    _check(gemm_bf16_noalloc_raw(m, n, k, _ptr(A), _ptr(B), _ptr(D), alpha, _stream(stream)),
           "tkg_gemm_bf16_noalloc")


def gemm_mxfp8(A, B, sfa, sfb, D, alpha: float = 1.0, stream=None) -> None:
    """A (m x k uint8 E4M3), B (n x k), tiled E8M0 scales sfa / sfb (uint8)."""
    m, k = A.shape
    n = B.shape[0]
    _check(gemm_mxfp8_raw(m, n, k, _ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(D), alpha, _stream(stream)),
           "tkg_gemm_mxfp8")


def gemm_nvfp4(A, B, sfa, sfb, D, alpha: float = 1.0, ta=None, tb=None, stream=None) -> None:
    """A (m x k/2 uint8, packed E2M1), B (n x k/2), tiled UE4M3 scales, FP32 per-tensor scales ta / tb (device)."""
    m, kh = A.shape
    n = B.shape[0]
    _check(gemm_nvfp4_raw(m, n, 2 * kh, _ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(ta), _ptr(tb), _ptr(D),
                          alpha, _stream(stream)), "tkg_gemm_nvfp4")


def gemm_strided(fmt: str, m: int, n: int, k: int, A, lda: int, B, ldb: int, D, ldd: int, alpha: float = 1.0,
                 sfa=None, sfb=None, ta=None, tb=None, stream=None) -> None:
    """The GEMM on row-pitched views: lda / ldb in storage units (bf16 elements, or bytes of E4M3 / packed E2M1
    codes), ldd in bf16 elements; A, B, D are the first elements of the views."""
    lib = load()
    s = _stream(stream)
    if fmt == "bf16":
        st = lib.tkg_gemm_bf16_strided(m, n, k, _ptr(A), lda, _ptr(B), ldb, _ptr(D), ldd, ctypes.c_float(alpha), s)
    elif fmt == "mxfp8":
        st = lib.tkg_gemm_mxfp8_strided(m, n, k, _ptr(A), lda, _ptr(B), ldb, _ptr(sfa), _ptr(sfb), _ptr(D), ldd,
                                        ctypes.c_float(alpha), s)
    else:
        st = lib.tkg_gemm_nvfp4_strided(m, n, k, _ptr(A), lda, _ptr(B), ldb, _ptr(sfa), _ptr(sfb), _ptr(ta), _ptr(tb),
                                        _ptr(D), ldd, ctypes.c_float(alpha), s)
    _check(st, f"tkg_gemm_{fmt}_strided")


def gemm_grouped_bf16(m_sizes, A, B, D, alpha: float = 1.0, stream=None) -> None:
    """Grouped: rows of A (sum(m_sizes) x k bf16) in consecutive groups, B (groups x n x k), D (sum x n)."""
    arr, g = _sizes(m_sizes)
    k = A.shape[-1]
    n = B.shape[-2]
    _check(gemm_grouped_bf16_raw(g, arr, n, k, _ptr(A), _ptr(B), _ptr(D), alpha, _stream(stream)),
           "tkg_gemm_grouped_bf16")


def gemm_grouped_mxfp8(m_sizes, A, B, sfa, sfb, D, alpha: float = 1.0, stream=None) -> None:
    """Grouped MXFP8: per-group tiled SFA buffers back to back, SFB one tiled buffer per group."""
    arr, g = _sizes(m_sizes)
    k = A.shape[-1]
    n = B.shape[-2]
    _check(gemm_grouped_mxfp8_raw(g, arr, n, k, _ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(D), alpha,
                                  _stream(stream)), "tkg_gemm_grouped_mxfp8")


def gemm_grouped_nvfp4(m_sizes, A, B, sfa, sfb, D, alpha: float = 1.0, ta=None, tb=None, stream=None) -> None:
    """Grouped NVFP4: ta one FP32 (device) for A, tb one FP32 per group (device)."""
    arr, g = _sizes(m_sizes)
    k = 2 * A.shape[-1]
    n = B.shape[-2]
    _check(gemm_grouped_nvfp4_raw(g, arr, n, k, _ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(ta), _ptr(tb),
                                  _ptr(D), alpha, _stream(stream)), "tkg_gemm_grouped_nvfp4")


def gemm_bf16_from_host(A_host, B_host, D_host, A_dev, B_dev, D_dev, alpha: float = 1.0, stream=None) -> None:
    """D_host = alpha * A_host @ B_host^T with host (pinned) operands; *_dev are device staging buffers."""
    m, k = A_host.shape
    n = B_host.shape[0]
    _check(load().tkg_gemm_bf16_from_host(m, n, k, _ptr(A_host), _ptr(B_host), _ptr(D_host), _ptr(A_dev),
                                          _ptr(B_dev), _ptr(D_dev), ctypes.c_float(alpha), _stream(stream)),
           "tkg_gemm_bf16_from_host")


def gemm_grouped_dev_bf16(sizes_dev, A, B, D, alpha: float = 1.0, stream=None) -> None:
    """Grouped BF16 GEMM with the group sizes in a device int32 tensor; A, D hold up to A.shape[0] rows."""
    g = sizes_dev.numel()
    _check(load().tkg_gemm_grouped_dev_bf16(g, _ptr(sizes_dev), A.shape[0], B.shape[-2], A.shape[-1], _ptr(A),
                                            _ptr(B), _ptr(D), ctypes.c_float(alpha), _stream(stream)),
           "tkg_gemm_grouped_dev_bf16")


def gemm_grouped_dev_mxfp8(sizes_dev, A, B, sfa, sfb, D, alpha: float = 1.0, stream=None) -> None:
    g = sizes_dev.numel()
    _check(load().tkg_gemm_grouped_dev_mxfp8(g, _ptr(sizes_dev), A.shape[0], B.shape[-2], A.shape[-1], _ptr(A),
                                             _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(D), ctypes.c_float(alpha),
                                             _stream(stream)), "tkg_gemm_grouped_dev_mxfp8")


def gemm_grouped_dev_nvfp4(sizes_dev, A, B, sfa, sfb, D, alpha: float = 1.0, ta=None, tb=None, stream=None) -> None:
    g = sizes_dev.numel()
    _check(load().tkg_gemm_grouped_dev_nvfp4(g, _ptr(sizes_dev), A.shape[0], B.shape[-2], 2 * A.shape[-1], _ptr(A),
                                             _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(ta), _ptr(tb), _ptr(D),
                                             ctypes.c_float(alpha), _stream(stream)), "tkg_gemm_grouped_dev_nvfp4")


def gemm_list_raw(fmt: str, descs, stream) -> int:
    """tkg_gemm_list_<fmt> on a sequence of GemmDesc."""
    arr = (GemmDesc * max(len(descs), 1))(*descs)
    return getattr(load(), f"tkg_gemm_list_{fmt}")(len(descs), arr, stream)


def gemm_desc(fmt: str, A, B, D, alpha: float = 1.0, sfa=None, sfb=None, ta=None, tb=None) -> GemmDesc:
    """Descriptor of one GEMM from its device tensors (A: m x k, or m x k/2 bytes for NVFP4)."""
    m = A.shape[0]
    k = 2 * A.shape[1] if fmt == "nvfp4" else A.shape[1]
    return GemmDesc(m, B.shape[0], k, _ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), _ptr(ta), _ptr(tb), _ptr(D),
                    float(alpha))


def gemm_list(fmt: str, descs, stream=None) -> None:
    """Several independent GEMMs (GemmDesc each, at most MAX_LIST) in one launch."""
    _check(gemm_list_raw(fmt, descs, _stream(stream)), f"tkg_gemm_list_{fmt}")


def grouped_dev_scale_bytes(groups: int, m_capacity: int, k: int, block: int) -> int:
    return int(load().tkg_grouped_dev_scale_bytes(groups, m_capacity, k, block))


def grouped_scale_bytes(m_sizes, k: int, block: int) -> int:
    arr, g = _sizes(m_sizes)
    return int(load().tkg_grouped_scale_bytes(g, arr, k, block))


def scale_bytes(rows: int, k: int, block: int) -> int:
    return int(load().tkg_scale_bytes(rows, k, block))


def scales_to_tiled(src, dst, kblocks: int | None = None, stream=None) -> None:
    rows, ld = src.shape
    kb = ld if kblocks is None else kblocks
    _check(load().tkg_scales_to_tiled(rows, kb, _ptr(src), ld, _ptr(dst), _stream(stream)), "tkg_scales_to_tiled")


def quantize_mxfp8(X, Q, sf, stream=None) -> None:
    rows, k = X.shape
    _check(load().tkg_quantize_mxfp8(rows, k, _ptr(X), _ptr(Q), _ptr(sf), _stream(stream)), "tkg_quantize_mxfp8")


def quantize_nvfp4(X, Q, sf, tensor_scale, stream=None) -> None:
    rows, k = X.shape
    _check(load().tkg_quantize_nvfp4(rows, k, _ptr(X), _ptr(Q), _ptr(sf), _ptr(tensor_scale), _stream(stream)),
           "tkg_quantize_nvfp4")


def quantize_nvfp4_scaled(X, Q, sf, tensor_scale, stream=None) -> None:
    """NVFP4 codes and tiled scales of X with the given FP32 tensor scale (device, one element, read only)."""
    rows, k = X.shape
    _check(load().tkg_quantize_nvfp4_scaled(rows, k, _ptr(X), _ptr(Q), _ptr(sf), _ptr(tensor_scale),
                                            _stream(stream)), "tkg_quantize_nvfp4_scaled")


def device_status(stream=None) -> int:
    return int(load().tkg_get_device_status(_stream(stream)))


def set_option(option: int, value: int) -> None:
    _check(load().tkg_set_option(option, value), "tkg_set_option")


def get_option(option: int) -> int:
    return int(load().tkg_get_option(option))
