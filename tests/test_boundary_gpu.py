"""The boundary as a caller without the tiled layout uses it: the oracle's
row-major scale matrices (rows x ld_sf bytes, ld_sf = K/bs rounded up to 16)
go to the device as they are, tkg_scales_to_tiled converts them, and the
block-scaled GEMM consumes the result -- all through the C ABI, with no
test-side layout code on the path.  NVFP4 runs both ways the per-tensor scales
can enter: as device pointers, and as NULL with the caller folding them into
alpha on the host (fp32(fp32(alpha * tA) * tB)).  Outputs are compared with the
oracle element by element at the acceptance tolerance.

Formats from "ThunderKittens 2.0 GPU Kernel优化" (table of updates: MXFP8 /
NVFP4 support)."""
import numpy as np
import pytest
import torch

import oracle
from dense_block_scaled_gb300 import synth, tkg
from helpers import assert_within_tolerance, bf16_to_f64

pytestmark = pytest.mark.gpu


def _tiled_on_device(sf_rowmajor, rows, k, bs):
    """Row-major codes uploaded unchanged, converted by the library."""
    src = torch.from_numpy(np.ascontiguousarray(sf_rowmajor)).cuda()
    dst = torch.full((tkg.scale_bytes(rows, k, bs),), 0xAB, dtype=torch.uint8, device="cuda")
    tkg.scales_to_tiled(src, dst, kblocks=k // bs)
    return dst


@pytest.mark.parametrize("m,n,k", [(300, 264, 512), (1000, 520, 4096), (16, 8192, 1024)])
def test_mxfp8_rowmajor_scales_through_the_abi(m, n, k):
    a, b = synth.gemm_inputs_f32(m, n, k, seed=90 + m)
    A, sa = oracle.quant_mxfp8(a)
    B, sb = oracle.quant_mxfp8(b)
    assert sa.shape == (m, oracle.ld_sf(k, "mxfp8"))
    alpha = 0.75
    D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    tkg.gemm_mxfp8(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), _tiled_on_device(sa, m, k, 32),
                   _tiled_on_device(sb, n, k, 32), D, alpha)
    assert tkg.device_status() == tkg.OK
    ref, S = oracle.gemm("mxfp8", A, B, sa, sb, alpha)
    assert_within_tolerance(bf16_to_f64(D), ref, S, f"mxfp8 {m}x{n}x{k} row-major scales")


@pytest.mark.parametrize("m,n,k", [(300, 264, 512), (1000, 520, 4096), (16, 8192, 1024)])
def test_nvfp4_rowmajor_scales_through_the_abi(m, n, k):
    a, b = synth.gemm_inputs_f32(m, n, k, seed=95 + m)
    A, sa, ta = oracle.quant_nvfp4(a)
    B, sb, tb = oracle.quant_nvfp4(b)
    assert sa.shape == (m, oracle.ld_sf(k, "nvfp4"))
    alpha = 1.25
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    sfa, sfb = _tiled_on_device(sa, m, k, 16), _tiled_on_device(sb, n, k, 16)
    ref, S = oracle.gemm("nvfp4", A, B, sa, sb, oracle.alpha_eff(alpha, ta, tb))

    # per-tensor scales as device pointers
    D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    tat = torch.tensor([float(ta)], dtype=torch.float32, device="cuda")
    tbt = torch.tensor([float(tb)], dtype=torch.float32, device="cuda")
    tkg.gemm_nvfp4(Ad, Bd, sfa, sfb, D, alpha, ta=tat, tb=tbt)
    assert tkg.device_status() == tkg.OK
    got_ptr = bf16_to_f64(D)
    assert_within_tolerance(got_ptr, ref, S, f"nvfp4 {m}x{n}x{k} tensor scales on the device")

    # per-tensor scales folded into alpha by the caller, NULL pointers
    D2 = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    tkg.gemm_nvfp4(Ad, Bd, sfa, sfb, D2, oracle.alpha_eff(alpha, ta, tb), ta=None, tb=None)
    assert tkg.device_status() == tkg.OK
    got_fold = bf16_to_f64(D2)
    assert_within_tolerance(got_fold, ref, S, f"nvfp4 {m}x{n}x{k} tensor scales folded into alpha")
    # the two routes form the same FP32 alpha, so they agree bit for bit
    assert np.array_equal(got_ptr, got_fold)
