"""The GEMMs on row-pitched views (tkg_gemm_*_strided): A and B rows padded
with garbage past their K elements, D rows wider than N with guard values in
the padding.  Outputs are compared with the oracle on the unpadded matrices,
element by element at the acceptance tolerance, and the padding of D must be
untouched.  Covers the persistent kernel (CTA pairs, single CTA, dual
accumulate), split-K and k == 0."""
import numpy as np
import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64

pytestmark = pytest.mark.gpu

GUARD = 0x7F7F


def _padded(codes: np.ndarray, ld: int, seed: int):
    """codes (rows x width) placed in rows of ld units, garbage after each row."""
    rows, width = codes.shape
    rng = np.random.default_rng(seed)
    if codes.dtype == np.uint16:
        # finite BF16 garbage so a stray read would show up as a wrong value, not a NaN
        pad = (rng.standard_normal((rows, ld)) * 100).astype(np.float32).view(np.uint32) >> 16
        buf = pad.astype(np.uint16)
    else:
        buf = rng.integers(0, 256, size=(rows, ld), dtype=np.uint8)
    buf[:, :width] = codes
    return torch.from_numpy(buf).cuda()


@pytest.fixture
def options():
    yield
    for o in (tkg.OPT_SPLIT_K, tkg.OPT_CTA_GROUP, tkg.OPT_BF16_TILE_N):
        tkg.set_option(o, 0)


# pads of A and B in 16-byte units (odd counts give pitches 16 bytes off a 32-byte multiple), of D in elements
CASES = [(300, 264, 512, 1, 2, 24, {}), (1000, 1032, 640, 4, 3, 8, {}), (16, 2048, 1024, 2, 5, 40, {}),
         (512, 2048, 512, 3, 1, 16, {"tile": 512}), (777, 136, 320, 1, 1, 8, {"cg": 1})]


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
@pytest.mark.parametrize("m,n,k,pad_a,pad_b,pad_d,opts", CASES)
def test_strided_matches_oracle(fmt, m, n, k, pad_a, pad_b, pad_d, opts, options):
    if opts.get("tile"):
        tkg.set_option(tkg.OPT_BF16_TILE_N, opts["tile"])
    if opts.get("cg"):
        tkg.set_option(tkg.OPT_CTA_GROUP, opts["cg"])
    ops = Operands(fmt, m, n, k, seed=700 + m, alpha=0.75)
    _, _, sfa, sfb, ta, tb = ops.upload()
    row = ops.A.shape[1]                       # storage units per row: k, or k/2 bytes for NVFP4
    unit16 = 8 if fmt == "bf16" else 16        # storage units in 16 bytes
    lda, ldb, ldd = row + pad_a * unit16, row + pad_b * unit16, n + pad_d
    A = _padded(ops.A, lda, 1)
    B = _padded(ops.B, ldb, 2)
    Dbuf = torch.full((m, ldd), GUARD, dtype=torch.int16, device="cuda")
    tkg.gemm_strided(fmt, m, n, k, A, lda, B, ldb, Dbuf, ldd, 0.75, sfa=sfa, sfb=sfb, ta=ta, tb=tb)
    assert tkg.device_status() == tkg.OK
    out = Dbuf.cpu()
    assert (out[:, n:] == GUARD).all(), "padding of D written"
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(out[:, :n]), ref, S, f"strided {fmt} {m}x{n}x{k} lda {lda} ldb {ldb} ldd {ldd}")


def test_strided_k0_zeroes_the_block():
    Dbuf = torch.full((40, 64), GUARD, dtype=torch.int16, device="cuda")
    tkg.gemm_strided("bf16", 40, 48, 0, None, 0, None, 0, Dbuf, 64, 1.0)
    torch.cuda.synchronize()
    out = Dbuf.cpu()
    assert (out[:, :48] == 0).all() and (out[:, 48:] == GUARD).all()


def test_strided_views_of_a_fused_weight():
    # three projections stored as one (3n x k) weight: each is a row range of
    # it, and D can be a column range of a wider output
    m, n, k = 64, 256, 512
    ops = Operands("bf16", m, 3 * n, k, seed=790)
    A = torch.from_numpy(ops.A).cuda()
    W = torch.from_numpy(ops.B).cuda()
    out = torch.full((m, 3 * n), GUARD, dtype=torch.int16, device="cuda")
    for p in range(3):
        tkg.gemm_strided("bf16", m, n, k, A, k, W[p * n:(p + 1) * n], k, out[:, p * n:], 3 * n, 1.0)
    assert tkg.device_status() == tkg.OK
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(out.cpu()), ref, S, "fused weight in three views")
