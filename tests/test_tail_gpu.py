"""Half-width tiles for the last partial wave of the persistent GEMM: with T
output tiles on P resident clusters the last round holds T mod P tiles; when
twice that many half-width tiles still fit one round, those tiles run as
halves (half-width MMAs, or one of dual accumulate's two MMAs).  Compared with
the oracle element by element: every tile split (each kernel variant), and the
automatic split under both schedules.

Tile scheduling follows "ThunderKittens 2.0 GPU Kernel优化" (table of updates:
cluster-launch-control scheduling)."""
import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64, run_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture
def options():
    yield
    for o in (tkg.OPT_TAIL_SPLIT, tkg.OPT_CTA_GROUP, tkg.OPT_BF16_TILE_N, tkg.OPT_SPLIT_K, tkg.OPT_SCHEDULER,
              tkg.OPT_MAX_CLUSTERS):
        tkg.set_option(o, 0)


def _check(fmt, m, n, k, seed, what):
    ops = Operands(fmt, m, n, k, seed, alpha=0.75)
    dev = ops.upload()
    D = run_gemm(fmt, dev, m, n, k, 0.75)
    assert tkg.device_status() == tkg.OK
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(D), ref, S, f"{what}: {fmt} {m}x{n}x{k}")
    return bf16_to_f64(D)


VARIANTS = [("bf16", {tkg.OPT_BF16_TILE_N: 512}), ("bf16", {tkg.OPT_BF16_TILE_N: 256}),
            ("bf16", {tkg.OPT_CTA_GROUP: 1}), ("mxfp8", {}), ("mxfp8", {tkg.OPT_CTA_GROUP: 1}),
            ("nvfp4", {}), ("nvfp4", {tkg.OPT_CTA_GROUP: 1})]


@pytest.mark.parametrize("fmt,opts", VARIANTS)
@pytest.mark.parametrize("m,n,k", [(300, 520, 512), (1000, 1032, 640), (512, 1024, 4096)])
def test_every_tile_split(fmt, opts, m, n, k, options):
    tkg.set_option(tkg.OPT_SPLIT_K, 1)
    for o, v in opts.items():
        tkg.set_option(o, v)
    tkg.set_option(tkg.OPT_TAIL_SPLIT, 2)
    _check(fmt, m, n, k, seed=300 + m, what=f"all tiles halved {opts}")


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
def test_automatic_split_static_schedule(fmt, options):
    # 1024 x 2048 on CTA pairs of 256 x 256: 32 tiles on 10 resident clusters
    # leaves 2 for the last round, which run as 4 halves
    tkg.set_option(tkg.OPT_SPLIT_K, 1)
    tkg.set_option(tkg.OPT_BF16_TILE_N, 256)
    tkg.set_option(tkg.OPT_SCHEDULER, 1)
    tkg.set_option(tkg.OPT_MAX_CLUSTERS, 10)
    split = _check(fmt, 1024, 2048, 512, seed=310, what="automatic split, static")
    tkg.set_option(tkg.OPT_TAIL_SPLIT, 1)
    whole = _check(fmt, 1024, 2048, 512, seed=310, what="no split, static")
    # the same products, summed in the same K order: identical bits
    assert (split == whole).all()


@pytest.mark.parametrize("fmt", ["bf16", "nvfp4"])
def test_automatic_split_launch_control(fmt, options):
    # 2560 x 2048 (BF16 256-wide) / 2560 x 2048 (NVFP4): 80 pair tiles on the
    # device's resident clusters, the few left over run as halves
    tkg.set_option(tkg.OPT_BF16_TILE_N, 256)
    split = _check(fmt, 2560, 2048, 256, seed=320, what="automatic split, launch control")
    tkg.set_option(tkg.OPT_TAIL_SPLIT, 1)
    whole = _check(fmt, 2560, 2048, 256, seed=320, what="no split, launch control")
    assert (split == whole).all()
