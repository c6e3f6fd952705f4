"""GPU parity: the CUDA GEMMs (through the C ABI) against the CPU oracle.

Acceptance bound per element: |D - ref| <= 2^-7 |ref| + 1e-5 * sum_k |alpha a_k b_k|;
exact equality for the format-decode and scale-index cases."""
import numpy as np
import pytest
import torch

import oracle
from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64, run_gemm, tiled_scales, to_dev

pytestmark = pytest.mark.gpu

FMTS = ["bf16", "mxfp8", "nvfp4"]


ALL_OPTIONS = (tkg.OPT_CTA_GROUP, tkg.OPT_SINGLE_STAGE, tkg.OPT_TIMEOUT_MS, tkg.OPT_INJECT_STALL,
               tkg.OPT_MAX_CLUSTERS, tkg.OPT_ACC_STAGES, tkg.OPT_SCHEDULER, tkg.OPT_SPLIT_K,
               tkg.OPT_RASTER_GROUP, tkg.OPT_BF16_TILE_N)


@pytest.fixture(autouse=True)
def _reset_options():
    for o in ALL_OPTIONS:
        tkg.set_option(o, 0)
    yield
    for o in ALL_OPTIONS:
        tkg.set_option(o, 0)


def _check(fmt, m, n, k, seed, alpha=1.0, cta_group=0, split=0):
    tkg.set_option(tkg.OPT_CTA_GROUP, cta_group)
    tkg.set_option(tkg.OPT_SPLIT_K, split)
    ops = Operands(fmt, m, n, k, seed, alpha)
    D = run_gemm(fmt, ops.upload(), m, n, k, alpha)
    assert tkg.device_status() == tkg.OK
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(D), ref, S, f"{fmt} {m}x{n}x{k} cg={cta_group}")
    return D


# 512^3 (the small square workload), several tiles with ragged M/N/K tails
SHAPES = [(512, 512, 512), (300, 264, 320), (129, 136, 96), (1, 8, 32), (257, 520, 1056)]


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", SHAPES)
def test_gemm_matches_oracle(fmt, shape, cta_group):
    # persistent kernel (split-K disabled)
    m, n, k = shape
    _check(fmt, m, n, k, seed=1000 + m + n + k, alpha=1.0, cta_group=cta_group, split=1)


@pytest.mark.parametrize("shape", SHAPES + [(1024, 1536, 768), (600, 1000, 4000)])
def test_bf16_dual_accumulate_matches_oracle(shape):
    # 256 x 512 pair tiles: two N=256 MMAs per K step into the two halves of
    # tensor memory, sharing the A tile
    m, n, k = shape
    tkg.set_option(tkg.OPT_BF16_TILE_N, 512)
    _check("bf16", m, n, k, seed=1700 + m + n + k, alpha=0.5, split=1)


SPLIT_SHAPES = [(512, 512, 512), (300, 264, 320), (16, 1024, 2048), (5, 136, 4000), (128, 256, 96), (33, 256, 512)]


@pytest.mark.parametrize("split", [0, 2, 3])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", SPLIT_SHAPES)
def test_split_k_matches_oracle(fmt, shape, split):
    # split-K kernel: automatic choice, or forced to 2 / 3 CTAs per tile
    m, n, k = shape
    _check(fmt, m, n, k, seed=2000 + m + n + k, alpha=0.5, split=split)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n", [4864, 6400])
def test_split_choice_by_resident_clusters(fmt, n):
    # 38 and 50 tiles of 128 columns: 3 CTAs per tile would fit the SMs, but
    # the automatic choice takes the split only if all its clusters can be
    # resident at once (50 clusters of 3 cannot); both must match the oracle
    _check(fmt, 16, n, 2048, seed=2100 + n, alpha=0.5, split=0)


@pytest.mark.parametrize("split", [0, 1])
@pytest.mark.parametrize("m", [1, 2, 7, 8, 9, 31, 100])
@pytest.mark.parametrize("fmt", FMTS)
def test_short_a_box(fmt, m, split):
    # M below the tile height: the A box is exactly M rows (no box partly past
    # the last row), on the persistent kernel (split=1) and on split-K where it
    # is chosen; ragged N and K
    _check(fmt, m, 520, 640, seed=2600 + m, alpha=0.5, split=split)


@pytest.mark.parametrize("path", ["auto", "pair", "splitk"])
@pytest.mark.parametrize("n", [8, 16, 56, 64, 120, 128, 136])
@pytest.mark.parametrize("fmt", FMTS)
def test_narrow_b(fmt, n, path):
    # N at most half the MMA width runs a half-width MMA (N=128 on CTA pairs and
    # single-CTA tiles, 64 on split-K tiles) with the B box clipped to N rows; 136
    # stays full width.  "auto" picks single-CTA tiles for N <= 256; "pair" forces
    # CTA pairs.  M = 1000 (ragged tiles) on the persistent kernel, 40 for split-K.
    if path == "splitk":
        _check(fmt, 40, n, 640, seed=2700 + n, alpha=0.5, split=0)
    else:
        _check(fmt, 1000, n, 640, seed=2700 + n, alpha=0.5, split=1, cta_group=2 if path == "pair" else 0)


@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_alpha_and_k_tail(fmt):
    # K = 4000: not a multiple of any stage depth; alpha != 1
    _check(fmt, 200, 136, 4000, seed=7, alpha=-0.375)


def test_bf16_odd_k():
    _check("bf16", 130, 24, 40, seed=8)


@pytest.mark.parametrize("fmt", FMTS)
def test_many_tiles_per_cta(fmt):
    # static schedule on few persistent clusters: every CTA walks many tiles,
    # the stage and accumulator phases wrap many times
    tkg.set_option(tkg.OPT_SCHEDULER, 1)
    tkg.set_option(tkg.OPT_MAX_CLUSTERS, 3)
    _check(fmt, 1024, 1024, 512, seed=9)


@pytest.mark.parametrize("fmt", FMTS)
def test_launch_control_equals_static_schedule(fmt):
    # cluster launch control and the static schedule compute every tile the
    # same way: identical bits; many more tiles than resident clusters
    m, n, k = 4096, 2048, 512
    ops = Operands(fmt, m, n, k, seed=14)
    dev = ops.upload()
    D_clc = run_gemm(fmt, dev, m, n, k, 1.0)
    tkg.set_option(tkg.OPT_SCHEDULER, 1)
    D_static = run_gemm(fmt, dev, m, n, k, 1.0)
    assert tkg.device_status() == tkg.OK
    assert torch.equal(D_clc.view(torch.int16), D_static.view(torch.int16))
    ref, S = ops.reference(rows=(m - 300, 300))
    assert_within_tolerance(bf16_to_f64(D_clc[m - 300:]), ref, S, "launch control")


@pytest.mark.parametrize("fmt", FMTS)
def test_single_stage_equals_deep_pipeline(fmt):
    # pipeline depth 1 and the deep ring must give identical bits ("异步Tensor Core原理与实战", §5.2)
    m, n, k = 384, 512, 1024
    tkg.set_option(tkg.OPT_SPLIT_K, 1)   # the persistent kernel, whose ring depth is under test
    ops = Operands(fmt, m, n, k, seed=11)
    dev = ops.upload()
    D_deep = run_gemm(fmt, dev, m, n, k, 1.0)
    tkg.set_option(tkg.OPT_SINGLE_STAGE, 1)
    D_one = run_gemm(fmt, dev, m, n, k, 1.0)
    tkg.set_option(tkg.OPT_SINGLE_STAGE, 0)
    assert tkg.device_status() == tkg.OK
    assert torch.equal(D_deep.view(torch.int16), D_one.view(torch.int16))


@pytest.mark.parametrize("fmt", FMTS)
def test_repeatable_bits(fmt):
    m, n, k = 512, 256, 768
    ops = Operands(fmt, m, n, k, seed=12)
    dev = ops.upload()
    D1 = run_gemm(fmt, dev, m, n, k, 1.0)
    D2 = run_gemm(fmt, dev, m, n, k, 1.0)
    assert torch.equal(D1.view(torch.int16), D2.view(torch.int16))


@pytest.mark.parametrize("fmt", FMTS)
def test_guard_bands_untouched(fmt):
    m, n, k = 200, 136, 256
    ops = Operands(fmt, m, n, k, seed=13)
    pad = 4096
    buf = torch.full((pad + m * n + pad,), 0x5A5A, dtype=torch.int16, device="cuda")
    D = buf[pad:pad + m * n].view(torch.bfloat16).view(m, n)
    run_gemm(fmt, ops.upload(), m, n, k, 1.0, D=D)
    assert tkg.device_status() == tkg.OK
    host = buf.cpu()
    assert bool((host[:pad] == 0x5A5A).all()) and bool((host[pad + m * n:] == 0x5A5A).all())
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(D), ref, S, "guarded")


def test_empty_and_k0():
    from dense_block_scaled_gb300 import tkg as t
    D = torch.full((4, 8), 3.0, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((4, 8), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((8, 8), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert t.gemm_bf16_raw(0, 8, 8, A.data_ptr(), B.data_ptr(), D.data_ptr(), 1.0, s) == t.OK
    assert bool((D == 3.0).all())
    assert t.gemm_bf16_raw(4, 8, 0, A.data_ptr(), B.data_ptr(), D.data_ptr(), 1.0, s) == t.OK
    torch.cuda.synchronize()
    assert bool((D == 0).all())
    assert t.gemm_bf16_raw(4, 8, 12, A.data_ptr(), B.data_ptr(), D.data_ptr(), 1.0, s) == t.ERR_ALIGNMENT
    assert t.gemm_bf16_raw(4, 8, 8, A.data_ptr() + 2, B.data_ptr(), D.data_ptr(), 1.0, s) == t.ERR_ALIGNMENT


# --------------------------------------------------------------------------- exact cases

def test_bf16_every_code_exact():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ex = (codes >> 7) & 0xFF
    keep = codes[(ex != 0xFF) & ((ex != 0) | ((codes & 0x7F) == 0))]   # no Inf/NaN, no subnormals
    m = keep.size
    k, n = 8, 8
    A = np.zeros((m, k), np.uint16)
    A[:, 0] = keep
    B = np.zeros((n, k), np.uint16)
    B[0, 0] = 0x3F80          # 1.0
    D = run_gemm("bf16", (to_dev(A), to_dev(B), None, None, None, None), m, n, k, 1.0)
    ref, _ = oracle.gemm("bf16", A, B)
    got = bf16_to_f64(D)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_every_code_pair_exact(fmt, cta_group):
    tkg.set_option(tkg.OPT_CTA_GROUP, cta_group)
    k = 32
    if fmt == "mxfp8":
        codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
        rows = 256
        A = np.zeros((rows, k), np.uint8)
        A[:len(codes), 0] = codes
        unit = 127
    else:
        codes = list(range(16))
        rows = 16
        A = np.zeros((rows, k // 2), np.uint8)
        A[:, 0] = codes
        unit = 0x38
    B = A.copy()
    ld = oracle.ld_sf(k, fmt)
    sf = np.full((rows, ld), unit, np.uint8)
    kb = k // oracle.BLOCK[fmt]
    dev = (to_dev(A), to_dev(B), to_dev(tiled_scales(sf, kb)), to_dev(tiled_scales(sf, kb)), None, None)
    D = run_gemm(fmt, dev, rows, rows, k, 1.0)
    ref, _ = oracle.gemm(fmt, A, B, sf, sf, 1.0)
    assert np.array_equal(bf16_to_f64(D), ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("cta_group,split", [(1, 1), (2, 1), (0, 3)])
def test_scale_index_exact(fmt, cta_group, split):
    # one nonzero block per row; distinct scale codes per (row, block); rows
    # cross 128-row tiles and the CTA pair, blocks cross stages, atoms and the
    # K stretches of a split-K cluster
    tkg.set_option(tkg.OPT_CTA_GROUP, cta_group)
    tkg.set_option(tkg.OPT_SPLIT_K, split)
    bs = oracle.BLOCK[fmt]
    m, n, k = 520, 264, 1536
    kb = k // bs
    rng = np.random.default_rng(31)
    lo, hi = (110, 145) if fmt == "mxfp8" else (0x28, 0x50)
    ld = oracle.ld_sf(k, fmt)
    sfa = rng.integers(lo, hi, size=(m, ld)).astype(np.uint8)
    sfb = rng.integers(lo, hi, size=(n, ld)).astype(np.uint8)
    blk_a = rng.integers(0, kb, size=m)
    blk_b = blk_a[rng.integers(0, m, size=n)]      # many (i, j) share a block
    one = 0x38 if fmt == "mxfp8" else 0x2

    def fill(rows, blk):
        if fmt == "mxfp8":
            X = np.zeros((rows, k), np.uint8)
            for r in range(rows):
                X[r, blk[r] * bs] = one
        else:
            X = np.zeros((rows, k // 2), np.uint8)
            for r in range(rows):
                X[r, blk[r] * bs // 2] = one
        return X

    A, B = fill(m, blk_a), fill(n, blk_b)
    dev = (to_dev(A), to_dev(B), to_dev(tiled_scales(sfa, kb)), to_dev(tiled_scales(sfb, kb)), None, None)
    D = run_gemm(fmt, dev, m, n, k, 1.0)
    ref, _ = oracle.gemm(fmt, A, B, sfa, sfb, 1.0)
    assert np.count_nonzero(ref) > 1000
    assert np.array_equal(bf16_to_f64(D), ref)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_every_scale_code_against_unit(fmt):
    # each scale code on A's side times a unit scale on B's side
    if fmt == "mxfp8":
        codes, unit, k = list(range(1, 255)), 127, 32
    else:
        codes, unit, k = list(range(0x01, 0x7F)), 0x38, 32
    m = 256
    bs = oracle.BLOCK[fmt]
    ld = oracle.ld_sf(k, fmt)
    sfa = np.full((m, ld), unit, np.uint8)
    sfa[:len(codes), 0] = codes
    sfb = np.full((8, ld), unit, np.uint8)
    if fmt == "mxfp8":
        A = np.zeros((m, k), np.uint8)
        A[:, 0] = 0x38
        B = np.zeros((8, k), np.uint8)
        B[0, 0] = 0x38
    else:
        A = np.zeros((m, k // 2), np.uint8)
        A[:, 0] = 0x2
        B = np.zeros((8, k // 2), np.uint8)
        B[0, 0] = 0x2
    kb = k // bs
    dev = (to_dev(A), to_dev(B), to_dev(tiled_scales(sfa, kb)), to_dev(tiled_scales(sfb, kb)), None, None)
    D = run_gemm(fmt, dev, m, 8, k, 1.0)
    ref, _ = oracle.gemm(fmt, A, B, sfa, sfb, 1.0)
    assert np.array_equal(bf16_to_f64(D), ref)


# --------------------------------------------------------------------------- full size, sampled

FULL = [("bf16", 16384), ("mxfp8", 16384), ("nvfp4", 16384), ("bf16", 4000), ("nvfp4", 4000)]


@pytest.mark.parametrize("fmt,size", FULL)
def test_full_size_sampled(fmt, size):
    m = n = k = size
    ops = Operands(fmt, m, n, k, seed=1000 + size)
    dev = ops.upload()
    D = run_gemm(fmt, dev, m, n, k, 1.0)
    assert tkg.device_status() == tkg.OK
    # 2^16 random outputs, plus every output of the first and last rows and
    # columns and of the rows / columns on tile seams (128, 256, 512)
    rng = np.random.default_rng(size)
    edge_r = np.array([0, m - 1, 127, 128, 255, 256, 511, 512])
    edge_c = np.array([0, n - 1, 127, 128, 255, 256, 511, 512])
    cols, rows = np.arange(n), np.arange(m)
    ii = np.concatenate([rng.integers(0, m, 1 << 16), np.repeat(edge_r, n), np.tile(rows, edge_c.size)])
    jj = np.concatenate([rng.integers(0, n, 1 << 16), np.tile(cols, edge_r.size), np.repeat(edge_c, m)])
    ref, S = ops.reference_elems(ii, jj)
    got = bf16_to_f64(D[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()])
    assert_within_tolerance(got, ref, S, f"{fmt} {size}^3 sampled")


@pytest.mark.parametrize("fmt", ["bf16", "nvfp4"])
@pytest.mark.parametrize("m", [1, 16, 128, 1024])
def test_skinny_full_size(fmt, m):
    n = k = 8192
    ops = Operands(fmt, m, n, k, seed=1004)
    D = run_gemm(fmt, ops.upload(), m, n, k, 1.0)
    assert tkg.device_status() == tkg.OK
    rows = min(m, 16)
    ref, S = ops.reference(rows=(m - rows, rows))
    assert_within_tolerance(bf16_to_f64(D[m - rows:]), ref, S, f"{fmt} skinny m={m}")


@pytest.mark.parametrize("n", [16, 128])
def test_tall_narrow_full_size(n):
    # a router-shaped GEMM at full size (single-CTA tiles, half-width MMA, B box
    # clipped to N): rows sampled across the M range, all columns
    m, k = 16384, 4096
    ops = Operands("bf16", m, n, k, seed=1008)
    D = run_gemm("bf16", ops.upload(), m, n, k, 1.0)
    assert tkg.device_status() == tkg.OK
    for r0 in (0, 8000, m - 64):
        ref, S = ops.reference(rows=(r0, 64))
        assert_within_tolerance(bf16_to_f64(D[r0:r0 + 64]), ref, S, f"tall narrow n={n} rows {r0}..")


@pytest.mark.parametrize("fmt", FMTS)
def test_long_k_single_tile(fmt):
    # K = 65536 on one 256 x 256 tile: over a thousand ring stages (BF16) through
    # one accumulation, the stage phases wrapping hundreds of times
    m, n, k = 256, 256, 65536
    tkg.set_option(tkg.OPT_SPLIT_K, 1)
    ops = Operands(fmt, m, n, k, seed=2900)
    D = run_gemm(fmt, ops.upload(), m, n, k, 1.0)
    assert tkg.device_status() == tkg.OK
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(D), ref, S, f"{fmt} K={k}")
