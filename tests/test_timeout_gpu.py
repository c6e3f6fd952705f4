"""Bounded waits: a GEMM whose MMA role waits on a barrier that nothing ever
arrives on must return within the wait limit, report TKG_ERR_TIMEOUT through
tkg_get_device_status, and leave the context usable for the next GEMM.
No fault, trap or hang is involved: the kernel gives up on its own."""
import time

import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64, run_gemm

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["bf16", "nvfp4"])
@pytest.mark.parametrize("cta_group,split", [(1, 1), (2, 1), (0, 2)])
def test_stalled_wait_times_out_and_recovers(fmt, cta_group, split):
    m, n, k = 512, 512, 1024
    ops = Operands(fmt, m, n, k, seed=77)
    dev = ops.upload()
    tkg.set_option(tkg.OPT_CTA_GROUP, cta_group)
    tkg.set_option(tkg.OPT_SPLIT_K, split)
    try:
        tkg.set_option(tkg.OPT_TIMEOUT_MS, 100)
        tkg.set_option(tkg.OPT_INJECT_STALL, 1)
        t0 = time.time()
        run_gemm(fmt, dev, m, n, k, 1.0)
        st = tkg.device_status()
        elapsed = time.time() - t0
        assert st == tkg.ERR_TIMEOUT
        assert elapsed < 10.0
    finally:
        tkg.set_option(tkg.OPT_INJECT_STALL, 0)
        tkg.set_option(tkg.OPT_TIMEOUT_MS, 0)
    # the status word was cleared and the next launch is healthy
    D = run_gemm(fmt, dev, m, n, k, 1.0)
    assert tkg.device_status() == tkg.OK
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(D), ref, S, "after recovery")
    tkg.set_option(tkg.OPT_CTA_GROUP, 0)
    tkg.set_option(tkg.OPT_SPLIT_K, 0)
    torch.cuda.synchronize()


def test_grouped_stall_times_out_and_recovers():
    # the grouped instantiation shares the bounded waits
    from test_grouped_gpu import GroupedOperands, run_grouped
    sizes = [300, 0, 257]
    ops = GroupedOperands("mxfp8", sizes, 264, 512, seed=78)
    dev = ops.upload()
    D = torch.empty((sum(sizes), 264), dtype=torch.bfloat16, device="cuda")
    try:
        tkg.set_option(tkg.OPT_TIMEOUT_MS, 100)
        tkg.set_option(tkg.OPT_INJECT_STALL, 1)
        t0 = time.time()
        run_grouped("mxfp8", sizes, dev, D)
        assert tkg.device_status() == tkg.ERR_TIMEOUT
        assert time.time() - t0 < 10.0
    finally:
        tkg.set_option(tkg.OPT_INJECT_STALL, 0)
        tkg.set_option(tkg.OPT_TIMEOUT_MS, 0)
    run_grouped("mxfp8", sizes, dev, D)
    assert tkg.device_status() == tkg.OK
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(D), ref, S, "grouped after recovery")


def test_dual_accumulate_stall_times_out_and_recovers():
    # the 256 x 512 BF16 tile variant shares the bounded waits
    m, n, k = 512, 1024, 1024
    ops = Operands("bf16", m, n, k, seed=79)
    dev = ops.upload()
    tkg.set_option(tkg.OPT_BF16_TILE_N, 512)
    tkg.set_option(tkg.OPT_SPLIT_K, 1)
    try:
        tkg.set_option(tkg.OPT_TIMEOUT_MS, 100)
        tkg.set_option(tkg.OPT_INJECT_STALL, 1)
        t0 = time.time()
        run_gemm("bf16", dev, m, n, k, 1.0)
        assert tkg.device_status() == tkg.ERR_TIMEOUT
        assert time.time() - t0 < 10.0
    finally:
        tkg.set_option(tkg.OPT_INJECT_STALL, 0)
        tkg.set_option(tkg.OPT_TIMEOUT_MS, 0)
    D = run_gemm("bf16", dev, m, n, k, 1.0)
    assert tkg.device_status() == tkg.OK
    tkg.set_option(tkg.OPT_BF16_TILE_N, 0)
    tkg.set_option(tkg.OPT_SPLIT_K, 0)
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(D), ref, S, "dual after recovery")
