"""Sizes whose byte or element offsets pass 2^32 / 2^31, where any 32-bit
offset arithmetic would wrap:

* a ragged BF16 output of 49200 x 49160 (4.8 GB), through TMA-box and
  register (16-byte) stores, the ragged edge tiles always through the latter;
* an NVFP4 GEMM whose A holds 4.3 GB of codes (524388 rows, K = 16384) and
  537 MB of tiled scales;
* both quantisers on an X of 65600 x 32768 FP32 (2^31 + 2^21 elements), the
  NVFP4 tensor amax planted in the very last element.

Inputs are drawn on the device by torch's seeded generator (input generation
only); the sampled rows are copied back and the oracle evaluates exactly those
outputs -- random samples plus the last rows and columns -- at the acceptance
tolerance (GEMMs) or bit for bit (quantiser codes, scales, tensor scale)."""
import numpy as np
import pytest
import torch

import oracle
from dense_block_scaled_gb300 import tkg
from helpers import assert_within_tolerance, bf16_to_f64

pytestmark = pytest.mark.gpu


def _gen(seed):
    return torch.Generator(device="cuda").manual_seed(seed)


def _samples(m, n, count, seed):
    rng = np.random.default_rng(seed)
    ii = np.concatenate([rng.integers(0, m, count), np.full(64, m - 1), np.arange(m - 64, m), [0]])
    jj = np.concatenate([rng.integers(0, n, count), np.arange(n - 64, n), np.full(64, n - 1), [0]])
    return ii.astype(np.int64), jj.astype(np.int64)


def _rows_of(ii):
    """Unique rows and each sample's index into them."""
    rows, local = np.unique(ii, return_inverse=True)
    return rows, local.astype(np.int64)


def _tiled_offsets(r, kb, ka):
    """Byte offset of scale (r, kb) in the tiled layout (the formula the ABI states)."""
    return ((r // 128) * ka + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4


@pytest.fixture
def reset_options():
    yield
    tkg.set_option(tkg.OPT_EPILOGUE_STORE, 0)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("store", [1, 2])
def test_bf16_output_past_4gb(store, reset_options):
    m, n, k = 49200, 49160, 64
    g = _gen(5)
    A = torch.randn((m, k), device="cuda", generator=g).bfloat16()
    B = torch.randn((n, k), device="cuda", generator=g).bfloat16()
    D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    assert D.numel() * 2 > 2 ** 32
    tkg.set_option(tkg.OPT_EPILOGUE_STORE, store)
    tkg.gemm_bf16(A, B, D, 0.5)
    assert tkg.device_status() == tkg.OK
    ii, jj = _samples(m, n, 4096, 6)
    got = bf16_to_f64(D[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()])
    del D
    ra, la = _rows_of(ii)
    rb, lb = _rows_of(jj)
    Ah = A[torch.from_numpy(ra).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    Bh = B[torch.from_numpy(rb).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    ref, S = oracle.gemm_elems("bf16", Ah, Bh, None, None, 0.5, la, lb)
    assert_within_tolerance(got, ref, S, f"BF16 {m}x{n}x{k}, store mode {store}, sampled")


def _tiled_on_device(sf, kblocks):
    """Row-major scale codes (rows, >= kblocks) on the device -> tiled buffer, by torch indexing."""
    rows = sf.shape[0]
    ka = -(-kblocks // 4)
    out = torch.zeros(-(-rows // 128) * 128 * ka * 4, dtype=torch.uint8, device="cuda")
    r = torch.arange(rows, device="cuda", dtype=torch.int64)[:, None]
    kb = torch.arange(kblocks, device="cuda", dtype=torch.int64)[None, :]
    out[_tiled_offsets(r, kb, ka).reshape(-1)] = sf[:, :kblocks].reshape(-1)
    return out


def test_nvfp4_operand_past_4gb(reset_options):
    m, n, k = 524388, 256, 16384
    kb = k // 16
    g = _gen(7)
    A = torch.randint(0, 256, (m, k // 2), dtype=torch.uint8, device="cuda", generator=g)   # any E2M1 pair is finite
    B = torch.randint(0, 256, (n, k // 2), dtype=torch.uint8, device="cuda", generator=g)
    assert A.numel() > 2 ** 32

    def ue4m3(rows):
        # finite UE4M3 block scales in [2^-3, 15]: exponent field 4..10, any mantissa
        e = torch.randint(4, 11, (rows, kb), dtype=torch.uint8, device="cuda", generator=g)
        f = torch.randint(0, 8, (rows, kb), dtype=torch.uint8, device="cuda", generator=g)
        return (e << 3) | f

    sa, sb = ue4m3(m), ue4m3(n)
    sfa, sfb = _tiled_on_device(sa, kb), _tiled_on_device(sb, kb)
    ta = torch.tensor([0.5], device="cuda")
    tb = torch.tensor([0.75], device="cuda")
    D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    tkg.gemm_nvfp4(A, B, sfa, sfb, D, 0.25, ta=ta, tb=tb)
    assert tkg.device_status() == tkg.OK
    ii, jj = _samples(m, n, 2048, 8)
    got = bf16_to_f64(D[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()])
    ra, la = _rows_of(ii)
    rb, lb = _rows_of(jj)
    pick = lambda t, rows: t[torch.from_numpy(rows).cuda()].cpu().numpy()
    ld = oracle.ld_sf(k, "nvfp4")
    sah = np.zeros((len(ra), ld), dtype=np.uint8)
    sbh = np.zeros((len(rb), ld), dtype=np.uint8)
    sah[:, :kb] = pick(sa, ra)
    sbh[:, :kb] = pick(sb, rb)
    ref, S = oracle.gemm_elems("nvfp4", pick(A, ra), pick(B, rb), sah, sbh,
                               oracle.alpha_eff(0.25, 0.5, 0.75), la, lb)
    assert_within_tolerance(got, ref, S, f"NVFP4 {m}x{n}x{k}, sampled")


QUANT_ROWS, QUANT_K = 65600, 32768


@pytest.fixture(scope="module")
def big_x():
    g = _gen(11)
    X = torch.randn((QUANT_ROWS, QUANT_K), device="cuda", generator=g).clamp_(-4.0, 4.0)
    X[-1, -1] = 10.0           # the tensor's largest magnitude, at element 2^31 + 2^21 - 1
    rng = np.random.default_rng(12)
    rows = np.unique(np.concatenate([rng.integers(0, QUANT_ROWS, 96), np.arange(QUANT_ROWS - 70, QUANT_ROWS),
                                     [0, 127, 128, 65535, 65536]]))
    Xh = X[torch.from_numpy(rows).cuda()].cpu().numpy()
    yield X, rows, Xh
    del X
    torch.cuda.empty_cache()


def _check_scales(sf_dev, rows, sf_ref, kblocks, what):
    ka = -(-kblocks // 4)
    sf = sf_dev.cpu().numpy()
    got = sf[_tiled_offsets(rows[:, None], np.arange(kblocks)[None, :], ka)]
    bad = np.argwhere(got != sf_ref[:, :kblocks])
    assert bad.size == 0, f"{what}: {len(bad)} scale codes differ, first at (row {rows[bad[0][0]]}, block {bad[0][1]})"


def _check_codes(q_dev, rows, q_ref, what):
    got = q_dev[torch.from_numpy(rows).cuda()].cpu().numpy()
    bad = np.argwhere(got != q_ref)
    assert bad.size == 0, f"{what}: {len(bad)} code bytes differ, first at (row {rows[bad[0][0]]}, byte {bad[0][1]})"


def test_quantize_mxfp8_past_2g_elements(big_x):
    X, rows, Xh = big_x
    assert X.numel() > 2 ** 31
    Q = torch.empty((QUANT_ROWS, QUANT_K), dtype=torch.uint8, device="cuda")
    SF = torch.empty(tkg.scale_bytes(QUANT_ROWS, QUANT_K, 32), dtype=torch.uint8, device="cuda")
    tkg.quantize_mxfp8(X, Q, SF)
    torch.cuda.synchronize()
    q_ref, sf_ref = oracle.quant_mxfp8(Xh)
    _check_codes(Q, rows, q_ref, "MXFP8 codes")
    _check_scales(SF, rows, sf_ref, QUANT_K // 32, "MXFP8 scales")


def test_quantize_nvfp4_past_2g_elements(big_x):
    X, rows, Xh = big_x
    Q = torch.empty((QUANT_ROWS, QUANT_K // 2), dtype=torch.uint8, device="cuda")
    SF = torch.empty(tkg.scale_bytes(QUANT_ROWS, QUANT_K, 16), dtype=torch.uint8, device="cuda")
    T = torch.empty(1, device="cuda")
    tkg.quantize_nvfp4(X, Q, SF, T)
    torch.cuda.synchronize()
    # the tensor scale follows from amax alone; the last sampled row holds the planted maximum
    _, _, t_ref = oracle.quant_nvfp4(Xh[-1:])
    assert T.cpu().numpy()[0] == t_ref, f"tensor scale {T.item()!r} != {t_ref!r}"
    q_ref, sf_ref, _ = oracle.quant_nvfp4(Xh, t=t_ref)
    _check_codes(Q, rows, q_ref, "NVFP4 codes")
    _check_scales(SF, rows, sf_ref, QUANT_K // 16, "NVFP4 scales")
