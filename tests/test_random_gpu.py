"""Seeded random parity cases mixing what the other tests vary one at a time:
shape (ragged M, N, K, from one row up), format, entry point (plain, strided
views with padded rows, a list of GEMMs) and options (CTA grouping, split-K,
schedule, BF16 tile width, tail split, epilogue stores).  Every output is
compared with the oracle element by element at the acceptance tolerance."""
import numpy as np
import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64

pytestmark = pytest.mark.gpu

OPTIONS = {
    tkg.OPT_CTA_GROUP: (0, 0, 1, 2),
    tkg.OPT_SPLIT_K: (0, 0, 1),
    tkg.OPT_SCHEDULER: (0, 0, 1),
    tkg.OPT_BF16_TILE_N: (0, 0, 256, 512),
    tkg.OPT_TAIL_SPLIT: (0, 0, 1, 2),
    tkg.OPT_EPILOGUE_STORE: (0, 0, 1, 2),
}
K_STEP = {"bf16": 8, "mxfp8": 32, "nvfp4": 32}


def _case(i):
    rng = np.random.default_rng(9000 + i)
    fmt = ("bf16", "mxfp8", "nvfp4")[i % 3]
    m = int(rng.choice([int(rng.integers(1, 40)), int(rng.integers(1, 1300))]))
    n = 8 * int(rng.integers(1, 160))
    k = K_STEP[fmt] * int(rng.integers(1, 2048 // K_STEP[fmt] + 1))
    opts = {o: int(rng.choice(v)) for o, v in OPTIONS.items()}
    entry = ("plain", "strided", "list")[int(rng.integers(0, 3))]
    return fmt, m, n, k, opts, entry, rng


@pytest.fixture
def reset_options():
    yield
    for o in OPTIONS:
        tkg.set_option(o, 0)


@pytest.mark.parametrize("i", range(48))
def test_random_case(i, reset_options):
    fmt, m, n, k, opts, entry, rng = _case(i)
    for o, v in opts.items():
        tkg.set_option(o, v)
    alpha = float(rng.choice([1.0, 0.5, 1.25]))
    ops = Operands(fmt, m, n, k, seed=9100 + i, alpha=alpha)
    A, B, sfa, sfb, ta, tb = ops.upload()
    what = f"case {i}: {fmt} {m}x{n}x{k} {entry} {opts}"
    if entry == "plain":
        D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        if fmt == "bf16":
            tkg.gemm_bf16(A, B, D, alpha)
        elif fmt == "mxfp8":
            tkg.gemm_mxfp8(A, B, sfa, sfb, D, alpha)
        else:
            tkg.gemm_nvfp4(A, B, sfa, sfb, D, alpha, ta=ta, tb=tb)
        got = bf16_to_f64(D)
    elif entry == "strided":
        unit16 = 8 if fmt == "bf16" else 16
        row = A.shape[1]
        lda, ldb, ldd = row + unit16 * int(rng.integers(0, 4)), row + unit16 * int(rng.integers(0, 4)), n + 8
        dt = torch.int16 if fmt == "bf16" else torch.uint8
        Ap = torch.zeros((m, lda), dtype=dt, device="cuda")
        Ap[:, :row] = A.view(dt)
        Bp = torch.zeros((n, ldb), dtype=dt, device="cuda")
        Bp[:, :row] = B.view(dt)
        Dbuf = torch.full((m, ldd), 0x7F7F, dtype=torch.int16, device="cuda")
        tkg.gemm_strided(fmt, m, n, k, Ap, lda, Bp, ldb, Dbuf, ldd, alpha, sfa=sfa, sfb=sfb, ta=ta, tb=tb)
        out = Dbuf.cpu()
        assert (out[:, n:] == 0x7F7F).all(), what + ": padding of D written"
        got = bf16_to_f64(out[:, :n])
    else:
        # the case's GEMM in a list beside a second, fixed one
        D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        other = Operands(fmt, 64, 136, K_STEP[fmt] * 16, seed=9200 + i)
        A2, B2, sfa2, sfb2, ta2, tb2 = other.upload()
        D2 = torch.empty((64, 136), dtype=torch.bfloat16, device="cuda")
        tkg.gemm_list(fmt, [tkg.gemm_desc(fmt, A, B, D, alpha, sfa=sfa, sfb=sfb, ta=ta, tb=tb),
                            tkg.gemm_desc(fmt, A2, B2, D2, 1.0, sfa=sfa2, sfb=sfb2, ta=ta2, tb=tb2)])
        ref2, S2 = other.reference()
        assert_within_tolerance(bf16_to_f64(D2), ref2, S2, what + " (second GEMM of the list)")
        got = bf16_to_f64(D)
    assert tkg.device_status() == tkg.OK, what
    ref, S = ops.reference()
    assert_within_tolerance(got, ref, S, what)
