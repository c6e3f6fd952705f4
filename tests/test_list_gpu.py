"""A list of independent GEMMs in one launch (tkg_gemm_list_*): every GEMM of
the list is compared element by element with the oracle at the acceptance
tolerance, over mixed shapes (ragged, short A, narrow B, long K), both CTA
groupings, both schedules, the maximum list length, skipped and k == 0
entries, and the skinny decode shapes the list exists for.

The pages name cluster-launch-control scheduling and programmatic dependent
launch as the means for back-to-back small GEMMs ("ThunderKittens 2.0 GPU
Kernel优化", table of updates); the list puts such GEMMs in one launch."""
import numpy as np
import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64

pytestmark = pytest.mark.gpu

MIXED = [(512, 512, 512), (300, 264, 320), (16, 1024, 1024), (100, 136, 4096), (1, 8, 64), (257, 128, 96)]


def _entries(fmt, shapes, seed0):
    out = []
    for i, (m, n, k) in enumerate(shapes):
        alpha = [1.0, 0.5, 1.5, 0.25, 2.0, 0.75][i % 6]
        ops = Operands(fmt, m, n, k, seed0 + i, alpha=alpha)
        dev = ops.upload()
        D = torch.full((m, n), 3.0, dtype=torch.bfloat16, device="cuda")
        A, B, sfa, sfb, ta, tb = dev
        desc = tkg.gemm_desc(fmt, A, B, D, alpha, sfa=sfa, sfb=sfb, ta=ta, tb=tb)
        out.append((ops, dev, D, desc))
    return out


def _check(fmt, entries, what):
    for i, (ops, _, D, _) in enumerate(entries):
        ref, S = ops.reference()
        assert_within_tolerance(bf16_to_f64(D), ref, S, f"{what}: {fmt} GEMM {i} {ops.m}x{ops.n}x{ops.k}")


@pytest.fixture
def options():
    yield
    for o in (tkg.OPT_CTA_GROUP, tkg.OPT_SCHEDULER):
        tkg.set_option(o, 0)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
@pytest.mark.parametrize("cta_group,scheduler", [(0, 0), (1, 0), (2, 0), (2, 1), (1, 1)])
def test_list_mixed_shapes(fmt, cta_group, scheduler, options):
    tkg.set_option(tkg.OPT_CTA_GROUP, cta_group)
    tkg.set_option(tkg.OPT_SCHEDULER, scheduler)
    entries = _entries(fmt, MIXED, seed0=400)
    tkg.gemm_list(fmt, [e[3] for e in entries])
    assert tkg.device_status() == tkg.OK
    _check(fmt, entries, f"cta_group {cta_group} scheduler {scheduler}")


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
def test_list_of_sixteen_random_shapes(fmt):
    rng = np.random.default_rng(17)
    shapes = [(int(rng.integers(1, 600)), 8 * int(rng.integers(1, 75)), 32 * int(rng.integers(1, 33)))
              for _ in range(tkg.MAX_LIST)]
    entries = _entries(fmt, shapes, seed0=500)
    tkg.gemm_list(fmt, [e[3] for e in entries])
    assert tkg.device_status() == tkg.OK
    _check(fmt, entries, "16 random shapes")


@pytest.mark.parametrize("fmt", ["bf16", "nvfp4"])
def test_list_skinny_decode_shapes(fmt):
    # four M=16 GEMMs with N = K = 8192 (the skinny workload), distinct weights
    entries = _entries(fmt, [(16, 8192, 8192)] * 4, seed0=600)
    tkg.gemm_list(fmt, [e[3] for e in entries])
    assert tkg.device_status() == tkg.OK
    _check(fmt, entries, "skinny decode list")


def test_list_skips_empty_and_zeroes_k0():
    fmt = "bf16"
    entries = _entries(fmt, [(300, 264, 320), (64, 128, 256)], seed0=700)
    D_empty = torch.full((8, 16), 5.0, dtype=torch.bfloat16, device="cuda")
    empty = tkg.GemmDesc(0, 16, 64, None, None, None, None, None, None, D_empty.data_ptr(), 1.0)
    D_k0 = torch.full((40, 24), 5.0, dtype=torch.bfloat16, device="cuda")
    k0 = tkg.GemmDesc(40, 24, 0, None, None, None, None, None, None, D_k0.data_ptr(), 1.0)
    tkg.gemm_list(fmt, [entries[0][3], empty, k0, entries[1][3]])
    assert tkg.device_status() == tkg.OK
    _check(fmt, entries, "with empty and k=0 entries")
    assert bool((D_empty.float() == 5.0).all())
    assert bool((D_k0.float() == 0.0).all())


def test_list_rejected_entry_launches_nothing():
    fmt = "bf16"
    entries = _entries(fmt, [(128, 128, 128)], seed0=800)
    D = entries[0][2]
    bad = tkg.GemmDesc(64, 64, 60, 16, 16, None, None, None, None, 16, 1.0)   # k % 8 != 0
    s = torch.cuda.current_stream().cuda_stream
    assert tkg.gemm_list_raw(fmt, [entries[0][3], bad], s) == tkg.ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert bool((D.float() == 3.0).all())


def test_list_outputs_match_single_gemm_launches():
    # the same GEMMs one launch each: both within tolerance of the oracle
    fmt = "nvfp4"
    entries = _entries(fmt, MIXED, seed0=900)
    tkg.gemm_list(fmt, [e[3] for e in entries])
    assert tkg.device_status() == tkg.OK
    _check(fmt, entries, "list")
    for ops, (A, B, sfa, sfb, ta, tb), D, _ in entries:
        D1 = torch.empty_like(D)
        tkg.gemm_nvfp4(A, B, sfa, sfb, D1, ops.alpha, ta=ta, tb=tb)
        ref, S = ops.reference()
        assert_within_tolerance(bf16_to_f64(D1), ref, S, f"single launch {ops.m}x{ops.n}x{ops.k}")
    assert tkg.device_status() == tkg.OK
