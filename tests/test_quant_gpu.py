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


@pytest.mark.parametrize("rows,kb", [(1, 1), (130, 7), (300, 125)])
def test_scales_to_tiled_bit_exact(rows, kb):
    rng = np.random.default_rng(rows)
    ld = -(-kb // 16) * 16
    src = rng.integers(0, 256, size=(rows, ld)).astype(np.uint8)
    dst = torch.full((-(-rows // 128) * 128 * (-(-kb // 4)) * 4,), 0x33, dtype=torch.uint8, device="cuda")
    tkg.scales_to_tiled(to_dev(src), dst, kblocks=kb)
    assert np.array_equal(dst.cpu().numpy(), tiled_scales(src, kb))
