"""CPU oracle for the dense / block-scaled GEMM  D = alpha * A * B^T.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the bench's
CPU-baseline leg are the only callers.  Nothing in the CUDA library imports
this package, and this package imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, FP64 accumulation, table
decoders, FP32 quantisers); this module compiles it with gcc on first use and
exposes numpy-level wrappers.

Formats (names from "ThunderKittens 2.0 GPU Kernel优化", opening section; bit
layouts are the standard ones for the type names listed in "剖析
ThunderKittens", section "Tile 抽象"):

* ``bf16``  : A, B are uint16 codes, shape (rows, K).
* ``mxfp8`` : A, B are uint8 E4M3 codes (rows, K); scales are uint8 E8M0
  codes, row-major (rows, ld_sf), one per 1x32 block along K.
* ``nvfp4`` : A, B are uint8, two E2M1 codes per byte (rows, K/2), element 2j
  in the low nibble of byte j; scales are uint8 E4M3 codes, row-major
  (rows, ld_sf), one per 1x16 block along K.  The FP32 per-tensor scales
  enter through ``alpha`` (alpha_eff = fp32(fp32(alpha * tA) * tB)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FORMATS = {"bf16": 0, "mxfp8": 1, "nvfp4": 2}
BLOCK = {"mxfp8": 32, "nvfp4": 16}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP, no FMA
    contraction so that results do not depend on the host ISA)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            vp = ctypes.c_void_p
            lib.orc_gemm_rows.argtypes = [i32, i64, i64, i64, vp, vp, vp, vp, i64, dbl, i64, i64, vp, vp]
            lib.orc_gemm_rows.restype = i32
            lib.orc_gemm_elems.argtypes = [i32, i64, i64, i64, vp, vp, vp, vp, i64, dbl, i64, vp, vp, vp, vp]
            lib.orc_gemm_elems.restype = i32
            lib.orc_decode_table.argtypes = [i32, vp]
            lib.orc_decode_table.restype = None
            lib.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
            lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
            lib.orc_f32_to_e2m1.argtypes = [ctypes.c_float]
            lib.orc_f32_to_e2m1.restype = ctypes.c_uint8
            lib.orc_quant_mxfp8.argtypes = [i64, i64, vp, vp, vp, i64]
            lib.orc_quant_mxfp8.restype = i32
            lib.orc_quant_nvfp4.argtypes = [i64, i64, vp, vp, vp, i64]
            lib.orc_quant_nvfp4.restype = ctypes.c_float
            lib.orc_quant_nvfp4_given.argtypes = [i64, i64, vp, vp, vp, i64, ctypes.c_float]
            lib.orc_quant_nvfp4_given.restype = i32
            lib.orc_num_threads.argtypes = []
            lib.orc_num_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def ld_sf(k: int, fmt: str) -> int:
    """Row pitch (bytes) of a row-major scale matrix: K/bs rounded up to 16."""
    kb = -(-k // BLOCK[fmt])
    return -(-kb // 16) * 16


def decode_table(name: str) -> np.ndarray:
    """FP64 value of every code: 'bf16' (65536), 'e4m3' (256), 'e2m1' (16), 'e8m0' (256)."""
    which, size = {"bf16": (0, 65536), "e4m3": (1, 256), "e2m1": (2, 16), "e8m0": (3, 256)}[name]
    out = np.empty(size, dtype=np.float64)
    _load().orc_decode_table(which, _ptr(out))
    return out


def f32_to_e4m3(v: float) -> int:
    return int(_load().orc_f32_to_e4m3(float(v)))


def f32_to_e2m1(v: float) -> int:
    return int(_load().orc_f32_to_e2m1(float(v)))


def _check_operand(fmt, X, k):
    X = np.ascontiguousarray(X)
    if fmt == "bf16":
        assert X.dtype == np.uint16 and X.shape[1] == k
    elif fmt == "mxfp8":
        assert X.dtype == np.uint8 and X.shape[1] == k
    else:
        assert X.dtype == np.uint8 and X.shape[1] * 2 == k
    return X


def _k_of(fmt, A):
    return A.shape[1] * 2 if fmt == "nvfp4" else A.shape[1]


def _check_sf(fmt, sf, rows, k):
    if fmt == "bf16":
        return None, 0
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    assert sf.shape[0] == rows and sf.shape[1] >= -(-k // BLOCK[fmt])
    return sf, sf.shape[1]


def gemm(fmt: str, A, B, sfa=None, sfb=None, alpha: float = 1.0, rows=None):
    """Returns (ref, S), float64 arrays of shape (nrows, N).

    ``rows`` = (row0, nrows) restricts the evaluation to a band of rows."""
    lib = _load()
    k = _k_of(fmt, A)
    A = _check_operand(fmt, A, k)
    B = _check_operand(fmt, B, k)
    m, n = A.shape[0], B.shape[0]
    sfa, lda = _check_sf(fmt, sfa, m, k)
    sfb, ldb = _check_sf(fmt, sfb, n, k)
    if fmt != "bf16":
        assert lda == ldb, "A and B scales must share one row pitch"
    row0, nrows = (0, m) if rows is None else rows
    ref = np.empty((nrows, n), dtype=np.float64)
    S = np.empty((nrows, n), dtype=np.float64)
    rc = lib.orc_gemm_rows(FORMATS[fmt], m, n, k, _ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb),
                           lda, float(alpha), row0, nrows, _ptr(ref), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"orc_gemm_rows failed ({rc})")
    return ref, S


def gemm_elems(fmt: str, A, B, sfa, sfb, alpha: float, ii, jj):
    """(ref, S) at the listed output coordinates only."""
    lib = _load()
    k = _k_of(fmt, A)
    A = _check_operand(fmt, A, k)
    B = _check_operand(fmt, B, k)
    m, n = A.shape[0], B.shape[0]
    sfa, lda = _check_sf(fmt, sfa, m, k)
    sfb, _ = _check_sf(fmt, sfb, n, k)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    ref = np.empty(ii.shape[0], dtype=np.float64)
    S = np.empty(ii.shape[0], dtype=np.float64)
    rc = lib.orc_gemm_elems(FORMATS[fmt], m, n, k, _ptr(A), _ptr(B), _ptr(sfa), _ptr(sfb), lda,
                            float(alpha), ii.shape[0], _ptr(ii), _ptr(jj), _ptr(ref), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"orc_gemm_elems failed ({rc})")
    return ref, S


def gemm_grouped(fmt: str, m_sizes, A, B, sfa=None, sfb=None, alpha=1.0):
    """Grouped GEMM by its definition: group g takes the m_sizes[g] rows of A
    that follow the earlier groups' rows and multiplies them by B[g]^T.

    A: (sum m_sizes, K or K/2); B: (groups, N, K or K/2); sfa: row-major scales
    of all rows of A (sum m_sizes, ld_sf); sfb: (groups, N, ld_sf); alpha: one
    value or one per group.  Returns (ref, S) of shape (sum m_sizes, N)."""
    m_sizes = [int(x) for x in m_sizes]
    groups = len(m_sizes)
    assert B.shape[0] == groups
    alphas = list(alpha) if np.ndim(alpha) else [float(alpha)] * groups
    total = sum(m_sizes)
    n = B.shape[1]
    ref = np.zeros((total, n), dtype=np.float64)
    S = np.zeros((total, n), dtype=np.float64)
    row = 0
    for g, mg in enumerate(m_sizes):
        if mg > 0:
            r, s = gemm(fmt, A[row:row + mg], B[g],
                        None if sfa is None else sfa[row:row + mg], None if sfb is None else sfb[g],
                        float(alphas[g]))
            ref[row:row + mg] = r
            S[row:row + mg] = s
        row += mg
    return ref, S


def quant_mxfp8(X):
    """FP32 (rows, K) -> (E4M3 codes (rows, K), E8M0 scales (rows, ld_sf))."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    rows, k = X.shape
    ld = ld_sf(k, "mxfp8")
    Q = np.empty((rows, k), dtype=np.uint8)
    SF = np.zeros((rows, ld), dtype=np.uint8)
    if _load().orc_quant_mxfp8(rows, k, _ptr(X), _ptr(Q), _ptr(SF), ld) != 0:
        raise ValueError("K must be a multiple of 32")
    return Q, SF


def quant_nvfp4(X, t=None):
    """FP32 (rows, K) -> (packed E2M1 (rows, K/2), E4M3 scales (rows, ld_sf), FP32 tensor scale).

    With t given, that FP32 tensor scale is used instead of amax / 2688 (values
    above 6 * 448 * t saturate) and returned as is."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    rows, k = X.shape
    ld = ld_sf(k, "nvfp4")
    Q = np.empty((rows, k // 2), dtype=np.uint8)
    SF = np.zeros((rows, ld), dtype=np.uint8)
    if t is None:
        t = _load().orc_quant_nvfp4(rows, k, _ptr(X), _ptr(Q), _ptr(SF), ld)
        if t < 0:
            raise ValueError("K must be a multiple of 16")
    elif _load().orc_quant_nvfp4_given(rows, k, _ptr(X), _ptr(Q), _ptr(SF), ld, float(np.float32(t))) != 0:
        raise ValueError("K must be a multiple of 16")
    return Q, SF, np.float32(t)


def alpha_eff(alpha: float, ta: float = 1.0, tb: float = 1.0) -> float:
    """fp32(fp32(alpha * tA) * tB): how the NVFP4 per-tensor scales join alpha."""
    a = np.float32(np.float32(alpha) * np.float32(ta))
    return float(np.float32(a * np.float32(tb)))
