"""The allocation-free BF16 entry point (tkg_gemm_bf16_noalloc), for callers
that cannot call cudaMalloc: its output must match tkg_gemm_bf16's, within
the tolerance the parity tests use, on two calls in a row (the second one
reuses the fixed scratch array the first one left behind).

Collected last on purpose, so a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64

pytestmark = pytest.mark.gpu


def test_noalloc_matches_allocating_entry_point_twice():
    s = torch.cuda.current_stream().cuda_stream
    for call, (m, n, k, seed) in enumerate([(300, 264, 320, 51), (512, 512, 1024, 52)]):
        ops = Operands("bf16", m, n, k, seed, alpha=0.5)
        A, B, _, _, _, _ = ops.upload()
        D_ref = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        D_new = torch.full((m, n), 7.0, dtype=torch.bfloat16, device="cuda")
        assert tkg.gemm_bf16_raw(m, n, k, A.data_ptr(), B.data_ptr(), D_ref.data_ptr(), 0.5, s) == tkg.OK
        assert tkg.gemm_bf16_noalloc_raw(m, n, k, A.data_ptr(), B.data_ptr(), D_new.data_ptr(), 0.5, s) == tkg.OK
        torch.cuda.synchronize()
        assert tkg.device_status() == tkg.OK
        ref, S = ops.reference()
        got = bf16_to_f64(D_new)
        assert_within_tolerance(got, bf16_to_f64(D_ref), S, f"noalloc vs tkg_gemm_bf16, call {call + 1}")
        assert_within_tolerance(got, ref, S, f"noalloc vs oracle, call {call + 1}")


def test_noalloc_argument_checks():
    s = torch.cuda.current_stream().cuda_stream
    assert tkg.gemm_bf16_noalloc_raw(-1, 8, 8, 16, 16, 16, 1.0, s) == tkg.ERR_INVALID_ARG
    assert tkg.gemm_bf16_noalloc_raw(8, 12, 8, 16, 16, 16, 1.0, s) == tkg.ERR_ALIGNMENT
    assert tkg.gemm_bf16_noalloc_raw(0, 8, 8, None, None, None, 1.0, s) == tkg.OK
