"""tkg_gemm_bf16_from_host: operands in pinned host memory, copies overlapped
with the GEMM inside the library.  Its result matches the device-resident GEMM
and the oracle within tolerance; back-to-back calls on shared staging buffers
stay ordered."""
import numpy as np
import pytest
import torch

from dense_block_scaled_gb300 import tkg
from helpers import Operands, assert_within_tolerance, bf16_to_f64

pytestmark = pytest.mark.gpu


def _host(codes):
    return torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).view(torch.bfloat16).pin_memory()


def _run(ops, m, n, k, alpha=1.0):
    Ah, Bh = _host(ops.A), _host(ops.B)
    Dh = torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
    Ad = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    Bd = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
    Dd = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    tkg.gemm_bf16_from_host(Ah, Bh, Dh, Ad, Bd, Dd, alpha)
    torch.cuda.current_stream().synchronize()   # Ah, Bh stay referenced until here
    assert tkg.device_status() == tkg.OK
    return Dh


def test_from_host_equals_device_gemm():
    # four bands of A and two of B (eight rectangles of D, launched separately)
    # against the whole GEMM on device-resident operands: the same products,
    # summed in a K order that may run either way per tile (serpentine order),
    # so equal within the tolerance, band edges included
    m, n, k = 8192, 4096, 512
    ops = Operands("bf16", m, n, k, seed=41)
    Dh = _run(ops, m, n, k)
    A = torch.from_numpy(ops.A.view(np.int16)).view(torch.bfloat16).cuda()
    B = torch.from_numpy(ops.B.view(np.int16)).view(torch.bfloat16).cuda()
    D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    tkg.gemm_bf16(A, B, D)
    got, dev = bf16_to_f64(Dh), bf16_to_f64(D)
    for r0 in (0, 2040, 4088, m - 64):
        ref, S = ops.reference(rows=(r0, 64))
        assert_within_tolerance(got[r0:r0 + 64], ref, S, f"from_host rows {r0}..")
        assert_within_tolerance(got[r0:r0 + 64], dev[r0:r0 + 64], S, f"from_host vs device rows {r0}..")


# (5000, 4104, 96): two ragged bands of each operand, so rectangles of D with
# ragged rows and columns, stored with D's full row stride
@pytest.mark.parametrize("shape", [(5000, 264, 320), (100, 64, 64), (2049, 136, 96), (5000, 4104, 96)])
def test_from_host_matches_oracle(shape):
    m, n, k = shape
    ops = Operands("bf16", m, n, k, seed=43 + m, alpha=0.5)
    Dh = _run(ops, m, n, k, alpha=0.5)
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(Dh), ref, S, f"from_host {m}x{n}x{k}")


def test_from_host_k0_and_ordering():
    # K = 0 gives zeros; two calls on the same staging buffers, queued back to
    # back without a host sync, each see their own inputs
    Dh = torch.full((8, 16), 3.0, dtype=torch.bfloat16).pin_memory()
    Ad = torch.empty((8, 8), dtype=torch.bfloat16, device="cuda")
    Dd = torch.empty((8, 16), dtype=torch.bfloat16, device="cuda")
    Ah = torch.empty((8, 0), dtype=torch.bfloat16).pin_memory()
    Bh = torch.empty((16, 0), dtype=torch.bfloat16).pin_memory()
    tkg.gemm_bf16_from_host(Ah, Bh, Dh, Ad, Ad, Dd)
    torch.cuda.current_stream().synchronize()
    assert not Dh.float().any()

    m, n, k = 4096, 512, 256
    o1 = Operands("bf16", m, n, k, seed=51)
    o2 = Operands("bf16", m, n, k, seed=52)
    Ad = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    Bd = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
    Dd = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    outs, keep = [], []   # host buffers must outlive the asynchronous copies
    for o in (o1, o2):
        Dh = torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
        Ah, Bh = _host(o.A), _host(o.B)
        keep += [Ah, Bh]
        tkg.gemm_bf16_from_host(Ah, Bh, Dh, Ad, Bd, Dd)
        outs.append(Dh)
    torch.cuda.current_stream().synchronize()
    for o, Dh in zip((o1, o2), outs):
        ref, S = o.reference(rows=(0, 256))
        assert_within_tolerance(bf16_to_f64(Dh)[:256], ref, S, "ordered calls")


def test_from_host_full_size_sampled():
    # the e2e configuration of the bench: M=N=K=16384 from pinned host buffers
    # (eight bands of each operand, fifteen rectangles of D); rows sampled in
    # the first and last bands of A, all columns (every band of B)
    m = n = k = 16384
    ops = Operands("bf16", m, n, k, seed=1001)
    Dh = _run(ops, m, n, k)
    got = bf16_to_f64(Dh)
    for r0 in (0, 2040, m - 48):
        ref, S = ops.reference(rows=(r0, 48))
        assert_within_tolerance(got[r0:r0 + 48], ref, S, f"from_host 16384^3 rows {r0}..")
