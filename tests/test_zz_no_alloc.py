"""The allocation-free BF16 entry point (tkg_gemm_bf16_noalloc), for callers
that cannot call cudaMalloc -- runtimes that reserve all device memory at
start-up, or code under a memory budget where a hidden allocation inside a
library call must not happen.  Its output must match tkg_gemm_bf16's, within
the tolerance the parity tests use, on two calls in a row (the second one
reuses the fixed scratch array the first one left behind), and a bounded wait
that runs out there must show up in tkg_get_device_status.

Collected last on purpose, so a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process."""
import time

import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64

pytestmark = pytest.mark.gpu


def _both(m, n, k, seed, alpha=0.5):
    s = torch.cuda.current_stream().cuda_stream
    ops = Operands("bf16", m, n, k, seed, alpha=alpha)
    A, B, _, _, _, _ = ops.upload()
    D_ref = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    D_new = torch.full((m, n), 7.0, dtype=torch.bfloat16, device="cuda")
    assert tkg.gemm_bf16_raw(m, n, k, A.data_ptr(), B.data_ptr(), D_ref.data_ptr(), alpha, s) == tkg.OK
    assert tkg.gemm_bf16_noalloc_raw(m, n, k, A.data_ptr(), B.data_ptr(), D_new.data_ptr(), alpha, s) == tkg.OK
    torch.cuda.synchronize()
    assert tkg.device_status() == tkg.OK
    return ops, D_ref, D_new


def test_noalloc_matches_allocating_entry_point_twice():
    for call, (m, n, k, seed) in enumerate([(300, 264, 320, 51), (512, 512, 1024, 52)]):
        ops, D_ref, D_new = _both(m, n, k, seed)
        ref, S = ops.reference()
        got = bf16_to_f64(D_new)
        assert_within_tolerance(got, bf16_to_f64(D_ref), S, f"noalloc vs tkg_gemm_bf16, call {call + 1}")
        assert_within_tolerance(got, ref, S, f"noalloc vs oracle, call {call + 1}")


@pytest.mark.parametrize("m,n,k", [(16, 8, 64), (100, 128, 320), (1, 136, 64), (257, 8, 4096)])
def test_noalloc_short_and_narrow(m, n, k):
    # A boxes shorter than the 128-row tile, B narrower than half the MMA
    ops, D_ref, D_new = _both(m, n, k, seed=53 + m)
    ref, S = ops.reference()
    got = bf16_to_f64(D_new)
    assert_within_tolerance(got, bf16_to_f64(D_ref), S, f"noalloc vs tkg_gemm_bf16 {m}x{n}x{k}")
    assert_within_tolerance(got, ref, S, f"noalloc vs oracle {m}x{n}x{k}")


def test_noalloc_timeout_is_reported_and_recovers():
    # A wait that nothing ever completes (the stall test option): the kernel
    # gives up after the wait limit, sets the status word in the fixed array,
    # and tkg_get_device_status reports and clears it.  No fault, trap or hang.
    m, n, k = 512, 512, 1024
    s = torch.cuda.current_stream().cuda_stream
    ops = Operands("bf16", m, n, k, seed=60)
    A, B, _, _, _, _ = ops.upload()
    D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    try:
        tkg.set_option(tkg.OPT_TIMEOUT_MS, 100)
        tkg.set_option(tkg.OPT_INJECT_STALL, 1)
        t0 = time.time()
        assert tkg.gemm_bf16_noalloc_raw(m, n, k, A.data_ptr(), B.data_ptr(), D.data_ptr(), 1.0, s) == tkg.OK
        assert tkg.device_status() == tkg.ERR_TIMEOUT
        assert time.time() - t0 < 10.0
    finally:
        tkg.set_option(tkg.OPT_INJECT_STALL, 0)
        tkg.set_option(tkg.OPT_TIMEOUT_MS, 0)
    assert tkg.device_status() == tkg.OK   # read once, cleared
    assert tkg.gemm_bf16_noalloc_raw(m, n, k, A.data_ptr(), B.data_ptr(), D.data_ptr(), 1.0, s) == tkg.OK
    assert tkg.device_status() == tkg.OK
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(D), ref, S, "noalloc after a timed-out call")


def test_noalloc_argument_checks():
    s = torch.cuda.current_stream().cuda_stream
    assert tkg.gemm_bf16_noalloc_raw(-1, 8, 8, 16, 16, 16, 1.0, s) == tkg.ERR_INVALID_ARG
    assert tkg.gemm_bf16_noalloc_raw(8, 12, 8, 16, 16, 16, 1.0, s) == tkg.ERR_ALIGNMENT
    assert tkg.gemm_bf16_noalloc_raw(0, 8, 8, None, None, None, 1.0, s) == tkg.OK
