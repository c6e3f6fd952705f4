"""The epilogue's two ways of writing D on the persistent kernel: TMA stores of
32 x 32 boxes staged in shared memory, and 16-byte stores straight from
registers masked at m and n (TKG_OPT_EPILOGUE_STORE 1 / 2; automatic: direct
stores for dual accumulate).  Both are compared
with the oracle element by element and with each other bit for bit, over
ragged edges, short A, narrow B, dual accumulate and the split tail; guard
bands around D must stay untouched."""
import numpy as np
import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64, run_gemm

pytestmark = pytest.mark.gpu

GUARD = 0x7F7F


@pytest.fixture
def options():
    yield
    for o in (tkg.OPT_EPILOGUE_STORE, tkg.OPT_SPLIT_K, tkg.OPT_BF16_TILE_N, tkg.OPT_TAIL_SPLIT, tkg.OPT_CTA_GROUP):
        tkg.set_option(o, 0)


def _run(fmt, ops, dev, store):
    m, n = ops.m, ops.n
    buf = torch.full((m + 2, n), GUARD, dtype=torch.int16, device="cuda")
    D = buf[1:m + 1].view(torch.bfloat16)
    tkg.set_option(tkg.OPT_EPILOGUE_STORE, store)
    run_gemm(fmt, dev, m, n, ops.k, ops.alpha, D=D)
    assert tkg.device_status() == tkg.OK
    out = buf.cpu()
    assert (out[0] == GUARD).all() and (out[m + 1] == GUARD).all(), "guard rows written"
    return bf16_to_f64(out[1:m + 1])


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
@pytest.mark.parametrize("m,n,k,opts", [
    (300, 520, 512, {}), (1000, 1032, 640, {}), (100, 264, 4096, {}), (1, 2048, 256, {}),
    (777, 136, 320, {}), (512, 1024, 512, {tkg.OPT_TAIL_SPLIT: 2}), (640, 1536, 256, {tkg.OPT_CTA_GROUP: 1}),
    (512, 2048, 512, {tkg.OPT_BF16_TILE_N: 512}), (300, 1544, 320, {tkg.OPT_BF16_TILE_N: 512, tkg.OPT_TAIL_SPLIT: 2})])
def test_direct_stores_match_tma_stores(fmt, m, n, k, opts, options):
    tkg.set_option(tkg.OPT_SPLIT_K, 1)
    for o, v in opts.items():
        tkg.set_option(o, v)
    ops = Operands(fmt, m, n, k, seed=500 + m + n, alpha=0.5)
    dev = ops.upload()
    via_tma = _run(fmt, ops, dev, 1)
    direct = _run(fmt, ops, dev, 2)
    ref, S = ops.reference()
    assert_within_tolerance(direct, ref, S, f"direct stores {fmt} {m}x{n}x{k} {opts}")
    assert np.array_equal(direct, via_tma)
