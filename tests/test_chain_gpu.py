"""Back-to-back launches on one stream with no host synchronisation between
them.  Every GEMM launch may start (set-up, L2 prefetches, the producer's own
set-up) before the previous kernel has finished; only its loads, its reads of
tensor scales and its stores of D must wait for that kernel.  Each test makes a
launch depend on what the previous one writes or reads and checks the result:
against the oracle on host-made inputs, or bit for bit against the same launch
repeated after a synchronisation (the kernels are deterministic)."""
import numpy as np
import pytest
import torch

import oracle
from dense_block_scaled_gb300 import synth, tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64, tiled_scales, to_dev

pytestmark = pytest.mark.gpu

# (M, N, K) of the first GEMM, and N of the GEMM that reads its D: shapes with
# enough output tiles for the persistent kernel (CTA pairs, cluster launch
# control), and skinny ones for the split-K kernel
SHAPES = {"persistent": (1024, 2048, 2048), "split_k": (16, 2048, 2048)}
READER_N = {"persistent": 1536, "split_k": 96}


def _bits(t):
    return t.cpu().view(torch.int16).numpy().copy()


@pytest.mark.parametrize("path", sorted(SHAPES))
def test_read_after_write(path):
    """GEMM 2 reads as A the D that GEMM 1 writes."""
    m, n, k = SHAPES[path]
    ops = Operands("bf16", m, n, k, seed=80)
    A, B, *_ = ops.upload()
    n2 = READER_N[path]
    b2 = synth.bf16_codes(np.random.default_rng(82).standard_normal((n2, n)).astype(np.float32))
    B2 = to_dev(b2, torch.bfloat16)
    D1 = torch.full((m, n), 7.0, dtype=torch.bfloat16, device="cuda")   # stale contents GEMM 2 must not see
    D2 = torch.empty((m, n2), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):   # a few rounds, so the second launch also follows a warm first one
        D1.fill_(7.0)
        torch.cuda.synchronize()
        tkg.gemm_bf16(A, B, D1)
        tkg.gemm_bf16(D1, B2, D2)
        assert tkg.device_status() == tkg.OK
        chained = _bits(D2)
        ref1, S1 = ops.reference()
        assert_within_tolerance(bf16_to_f64(D1), ref1, S1, f"{path}: first launch")
        D2r = torch.empty_like(D2)
        tkg.gemm_bf16(D1, B2, D2r)
        assert tkg.device_status() == tkg.OK
        assert np.array_equal(chained, _bits(D2r)), f"{path}: the chained launch read a stale D"


@pytest.mark.parametrize("path", sorted(SHAPES))
def test_write_after_read(path):
    """GEMM 2 overwrites the A that GEMM 1 reads: GEMM 1 must see the old A."""
    m, n, k = SHAPES[path]
    ops = Operands("bf16", m, n, k, seed=83)
    A, B, *_ = ops.upload()
    # GEMM 2: A (m x k) := A2 (m x 64) . B2 (k x 64)^T
    rng = np.random.default_rng(84)
    A2 = to_dev(synth.bf16_codes(rng.standard_normal((m, 64)).astype(np.float32)), torch.bfloat16)
    B2 = to_dev(synth.bf16_codes(rng.standard_normal((k, 64)).astype(np.float32)), torch.bfloat16)
    D1 = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    tkg.gemm_bf16(A, B, D1)
    tkg.gemm_bf16(A2, B2, A)
    assert tkg.device_status() == tkg.OK
    ref1, S1 = ops.reference()
    assert_within_tolerance(bf16_to_f64(D1), ref1, S1, f"{path}: the first launch read an overwritten A")


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("path", sorted(SHAPES))
def test_quantize_then_gemm(fmt, path):
    """The quantiser writes A's codes, scales and (NVFP4) tensor scale; the GEMM
    right behind it reads them (the tensor scale in its epilogue)."""
    m, n, k = SHAPES[path]
    a, b = synth.gemm_inputs_f32(m, n, k, 85)
    bs = 32 if fmt == "mxfp8" else 16
    cols = k if fmt == "mxfp8" else k // 2
    X = torch.from_numpy(a).cuda()
    Q = torch.full((m, cols), 0x55, dtype=torch.uint8, device="cuda")
    S = torch.full((tkg.scale_bytes(m, k, bs),), 0x7F, dtype=torch.uint8, device="cuda")
    T = torch.full((1,), float("nan"), device="cuda")
    if fmt == "mxfp8":
        qb, sb = oracle.quant_mxfp8(b)
        tb = None
    else:
        qb, sb, tb_host = oracle.quant_nvfp4(b)
        tb = torch.tensor([float(tb_host)], device="cuda")
    Bd = to_dev(qb)
    SBd = to_dev(tiled_scales(sb, k // bs))
    D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    if fmt == "mxfp8":
        tkg.quantize_mxfp8(X, Q, S)
        tkg.gemm_mxfp8(Q, Bd, S, SBd, D, 0.5)
        qa, sa = oracle.quant_mxfp8(a)
        alpha = 0.5
    else:
        tkg.quantize_nvfp4(X, Q, S, T)
        tkg.gemm_nvfp4(Q, Bd, S, SBd, D, 0.5, ta=T, tb=tb)
        qa, sa, ta_host = oracle.quant_nvfp4(a)
        alpha = oracle.alpha_eff(0.5, ta_host, tb_host)
    assert tkg.device_status() == tkg.OK
    ref, Sr = oracle.gemm(fmt, qa, qb, sa, sb, alpha)
    assert_within_tolerance(bf16_to_f64(D), ref, Sr, f"{fmt} {path}: GEMM right behind the quantiser")
