"""GPU quantisers and scale-layout conversion against the CPU oracle: bit-exact
(every code and scale byte, and the FP32 tensor scale)."""
import numpy as np
import pytest
import torch

import oracle
from dense_block_scaled_gb300 import synth, tkg
from helpers import tiled_scales, to_dev

pytestmark = pytest.mark.gpu

# k/bs both a multiple of 4 (packed scale stores) and not; sizes spanning
# several grid-stride trips with a ragged last one
SHAPES = [(1, 32), (130, 96), (257, 4000), (1024, 2048), (333, 2080), (4099, 8192)]


@pytest.mark.parametrize("rows,k", SHAPES)
def test_quantize_mxfp8_bit_exact(rows, k):
    x, _ = synth.gemm_inputs_f32(rows, 1, k, seed=rows + k)
    x[0, :32] = 0.0                                   # a zero block
    if rows > 1:
        x[1, 32:64] *= np.float32(1e-30)             # tiny block (clamped exponent)
    Q_ref, SF_ref = oracle.quant_mxfp8(x)
    X = to_dev(x)
    Q = torch.empty((rows, k), dtype=torch.uint8, device="cuda")
    SF = torch.full((tkg.scale_bytes(rows, k, 32),), 0xEE, dtype=torch.uint8, device="cuda")
    tkg.quantize_mxfp8(X, Q, SF)
    assert np.array_equal(Q.cpu().numpy(), Q_ref)
    assert np.array_equal(SF.cpu().numpy(), tiled_scales(SF_ref, k // 32))


@pytest.mark.parametrize("rows,k", SHAPES)
def test_quantize_nvfp4_bit_exact(rows, k):
    x, _ = synth.gemm_inputs_f32(rows, 1, k, seed=2 * rows + k)
    x[0, 16:32] = 0.0
    Q_ref, SF_ref, t_ref = oracle.quant_nvfp4(x)
    X = to_dev(x)
    Q = torch.empty((rows, k // 2), dtype=torch.uint8, device="cuda")
    SF = torch.full((tkg.scale_bytes(rows, k, 16),), 0xEE, dtype=torch.uint8, device="cuda")
    t = torch.empty(1, dtype=torch.float32, device="cuda")
    tkg.quantize_nvfp4(X, Q, SF, t)
    assert t.item() == float(t_ref)
    assert np.array_equal(Q.cpu().numpy(), Q_ref)
    assert np.array_equal(SF.cpu().numpy(), tiled_scales(SF_ref, k // 16))


def test_quantize_nvfp4_zero_tensor():
    X = torch.zeros((4, 64), dtype=torch.float32, device="cuda")
    Q = torch.full((4, 32), 0x77, dtype=torch.uint8, device="cuda")
    SF = torch.full((tkg.scale_bytes(4, 64, 16),), 0x77, dtype=torch.uint8, device="cuda")
    t = torch.full((1,), 5.0, dtype=torch.float32, device="cuda")
    tkg.quantize_nvfp4(X, Q, SF, t)
    assert t.item() == 0.0 and not Q.any() and not SF.any()


@pytest.mark.parametrize("factor", [1.0, 0.25, 3.0])
@pytest.mark.parametrize("rows,k", [(130, 96), (1024, 2048), (333, 2080)])
def test_quantize_nvfp4_scaled_bit_exact(rows, k, factor):
    # supplied tensor scale: the tensor's own (the codes of tkg_quantize_nvfp4),
    # a quarter of it (the largest blocks saturate) and three times it
    x, _ = synth.gemm_inputs_f32(rows, 1, k, seed=3 * rows + k)
    x[0, 16:32] = 0.0
    t_own = np.float32(np.float32(np.abs(x).max()) / np.float32(2688))
    tg = np.float32(t_own * np.float32(factor))
    Q_ref, SF_ref, _ = oracle.quant_nvfp4(x, t=tg)
    X = to_dev(x)
    Q = torch.empty((rows, k // 2), dtype=torch.uint8, device="cuda")
    SF = torch.full((tkg.scale_bytes(rows, k, 16),), 0xEE, dtype=torch.uint8, device="cuda")
    T = torch.tensor([float(tg)], dtype=torch.float32, device="cuda")
    tkg.quantize_nvfp4_scaled(X, Q, SF, T)
    assert T.item() == float(tg)                      # read, not written
    assert np.array_equal(Q.cpu().numpy(), Q_ref)
    assert np.array_equal(SF.cpu().numpy(), tiled_scales(SF_ref, k // 16))


def test_quantize_nvfp4_scaled_slices_share_the_scale():
    # slices of rows quantised with the whole tensor's scale: each slice's codes
    # are its rows of the whole tensor's codes; a zero scale gives zeros
    rows, k = 96, 256
    x, _ = synth.gemm_inputs_f32(rows, 1, k, seed=77)
    X = to_dev(x)
    Q = torch.empty((rows, k // 2), dtype=torch.uint8, device="cuda")
    SF = torch.empty((tkg.scale_bytes(rows, k, 16),), dtype=torch.uint8, device="cuda")
    T = torch.empty(1, dtype=torch.float32, device="cuda")
    tkg.quantize_nvfp4(X, Q, SF, T)
    for r0, r1 in ((0, 16), (16, 48), (48, 96)):
        Qs = torch.empty((r1 - r0, k // 2), dtype=torch.uint8, device="cuda")
        SFs = torch.full((tkg.scale_bytes(r1 - r0, k, 16),), 0xEE, dtype=torch.uint8, device="cuda")
        tkg.quantize_nvfp4_scaled(X[r0:r1], Qs, SFs, T)
        assert torch.equal(Qs, Q[r0:r1])
        _, SF_ref, _ = oracle.quant_nvfp4(x[r0:r1], t=np.float32(T.item()))
        assert np.array_equal(SFs.cpu().numpy(), tiled_scales(SF_ref, k // 16))
    Z = torch.zeros(1, dtype=torch.float32, device="cuda")
    Qz = torch.full((rows, k // 2), 0x77, dtype=torch.uint8, device="cuda")
    SFz = torch.full((tkg.scale_bytes(rows, k, 16),), 0x77, dtype=torch.uint8, device="cuda")
    tkg.quantize_nvfp4_scaled(X, Qz, SFz, Z)
    assert not Qz.any() and not SFz.any()


@pytest.mark.parametrize("rows,kb", [(1, 1), (130, 7), (300, 125)])
def test_scales_to_tiled_bit_exact(rows, kb):
    rng = np.random.default_rng(rows)
    ld = -(-kb // 16) * 16
    src = rng.integers(0, 256, size=(rows, ld)).astype(np.uint8)
    dst = torch.full((-(-rows // 128) * 128 * (-(-kb // 4)) * 4,), 0x33, dtype=torch.uint8, device="cuda")
    tkg.scales_to_tiled(to_dev(src), dst, kblocks=kb)
    assert np.array_equal(dst.cpu().numpy(), tiled_scales(src, kb))


def _boundary_blocks(rows, k, seed):
    """FP32 input whose element quotients x / den fall exactly on, and a few ulps
    either side of, every E2M1 rounding boundary (0.25, 0.75, ..., 5).

    t = 2^-10 and block 0 holds 6 * 448 * t, so the tensor scale is exactly t;
    each block's maximum is 6 * dec(s) * t for a chosen E4M3 code s, so the block
    scale decodes to dec(s) and den = dec(s) * t, all exact in FP32."""
    rng = np.random.default_rng(seed)
    e4m3 = oracle.decode_table("e4m3")
    t = np.float32(2.0 ** -10)
    bounds = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    nb = rows * k // 16
    codes = rng.integers(8, 108, size=nb)
    codes[0] = 0x7E                                          # 448: the tensor maximum
    den = (e4m3[codes] * float(t)).astype(np.float32)
    x = np.empty((nb, 16), dtype=np.float32)
    x[:, 0] = np.float32(6.0) * den
    base = bounds[rng.integers(0, 7, size=(nb, 15))] * den[:, None]
    ulps = rng.integers(-4, 5, size=(nb, 15)).astype(np.int32)
    x[:, 1:] = (base.view(np.int32) + ulps).view(np.float32)
    x[:, 1:] *= np.where(rng.integers(0, 2, size=(nb, 15)) == 1, np.float32(-1), np.float32(1))
    return x.reshape(rows, k)


@pytest.mark.parametrize("rows,k", [(64, 1024), (40, 96)])
def test_quantize_nvfp4_rounding_boundaries(rows, k):
    # quotients on and next to every E2M1 tie, each side of zero: the kernel's
    # fast quotient must fall back to the IEEE division exactly where needed
    x = _boundary_blocks(rows, k, seed=rows * k)
    Q_ref, SF_ref, t_ref = oracle.quant_nvfp4(x)
    assert float(t_ref) == 2.0 ** -10
    X = to_dev(x)
    Q = torch.empty((rows, k // 2), dtype=torch.uint8, device="cuda")
    SF = torch.full((tkg.scale_bytes(rows, k, 16),), 0xEE, dtype=torch.uint8, device="cuda")
    t = torch.empty(1, dtype=torch.float32, device="cuda")
    tkg.quantize_nvfp4(X, Q, SF, t)
    assert t.item() == float(t_ref)
    assert np.array_equal(Q.cpu().numpy(), Q_ref)
    assert np.array_equal(SF.cpu().numpy(), tiled_scales(SF_ref, k // 16))
