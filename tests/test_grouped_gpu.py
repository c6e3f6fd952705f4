"""Grouped GEMM (groups of rows of A, each against its own B) against the CPU
oracle's grouped definition, through the C ABI: ragged and empty groups,
group ends inside a 32-row store box, N tails, both CTA-group sizes, and the
rows of D outside the groups left alone."""
import numpy as np
import pytest
import torch

import oracle
from dense_block_scaled_gb300 import synth, tkg
from helpers import assert_within_tolerance, bf16_to_f64, tiled_scales, to_dev

pytestmark = pytest.mark.gpu

FMTS = ["bf16", "mxfp8", "nvfp4"]


@pytest.fixture(autouse=True)
def _reset_options():
    yield
    tkg.set_option(tkg.OPT_CTA_GROUP, 0)


class GroupedOperands:
    """Seeded grouped operands: A (sum of sizes rows), B (groups x n x k); A is
    quantised as one tensor, each B_g as its own tensor (NVFP4: one tensor
    scale per group)."""

    def __init__(self, fmt, sizes, n, k, seed, alpha=1.0):
        self.fmt, self.sizes, self.n, self.k = fmt, list(sizes), n, k
        groups, total = len(sizes), sum(sizes)
        a, b = synth.gemm_inputs_f32(max(total, 1), groups * n, k, seed)
        a = a[:total]
        b = b.reshape(groups, n, k)
        self.alphas = [alpha] * groups
        self.sfa = self.sfb = None
        self.ta, self.tb = None, None
        if fmt == "bf16":
            self.A = synth.bf16_codes(a)
            self.B = synth.bf16_codes(b.reshape(groups * n, k)).reshape(groups, n, k)
        elif fmt == "mxfp8":
            self.A, self.sfa = oracle.quant_mxfp8(a)
            qb = [oracle.quant_mxfp8(b[g]) for g in range(groups)]
            self.B = np.stack([q for q, _ in qb])
            self.sfb = np.stack([s for _, s in qb])
        else:
            self.A, self.sfa, self.ta = oracle.quant_nvfp4(a)
            qb = [oracle.quant_nvfp4(b[g]) for g in range(groups)]
            self.B = np.stack([q for q, _, _ in qb])
            self.sfb = np.stack([s for _, s, _ in qb])
            self.tb = [t for _, _, t in qb]
            self.alphas = [oracle.alpha_eff(alpha, self.ta, t) for t in self.tb]

    def reference(self):
        return oracle.gemm_grouped(self.fmt, self.sizes, self.A, self.B, self.sfa, self.sfb, self.alphas)

    def upload(self):
        """Device tensors (A, B, sfa, sfb, ta, tb) in the grouped layouts."""
        A, B = to_dev(self.A), to_dev(self.B)
        if self.fmt == "bf16":
            return A, B, None, None, None, None
        kb = self.k // oracle.BLOCK[self.fmt]
        parts, row = [], 0
        for mg in self.sizes:
            if mg:
                parts.append(tiled_scales(self.sfa[row:row + mg], kb))
            row += mg
        sfa = to_dev(np.concatenate(parts) if parts else np.zeros(16, np.uint8))
        sfb = to_dev(np.concatenate([tiled_scales(self.sfb[g], kb) for g in range(len(self.sizes))]))
        ta = tb = None
        if self.fmt == "nvfp4":
            ta = torch.tensor([float(self.ta)], dtype=torch.float32, device="cuda")
            tb = torch.tensor([float(t) for t in self.tb], dtype=torch.float32, device="cuda")
        return A, B, sfa, sfb, ta, tb


def run_grouped(fmt, sizes, dev, D, alpha=1.0):
    A, B, sfa, sfb, ta, tb = dev
    if fmt == "bf16":
        tkg.gemm_grouped_bf16(sizes, A, B, D, alpha)
    elif fmt == "mxfp8":
        tkg.gemm_grouped_mxfp8(sizes, A, B, sfa, sfb, D, alpha)
    else:
        tkg.gemm_grouped_nvfp4(sizes, A, B, sfa, sfb, D, alpha, ta=ta, tb=tb)


GUARD = 0x7F7F   # a BF16 NaN pattern no GEMM result takes


def _check(fmt, sizes, n, k, seed, cta_group=0, alpha=1.0):
    tkg.set_option(tkg.OPT_CTA_GROUP, cta_group)
    ops = GroupedOperands(fmt, sizes, n, k, seed, alpha)
    dev = ops.upload()
    total = sum(sizes)
    # D with 40 guard rows after the groups' rows: never written
    Dfull = torch.full((total + 40, n), GUARD, dtype=torch.int16, device="cuda")
    run_grouped(fmt, sizes, dev, Dfull.view(torch.bfloat16), alpha)
    assert tkg.device_status() == tkg.OK
    out = Dfull.cpu().numpy()
    assert (out[total:] == GUARD).all(), "rows past the groups were written"
    if total:
        ref, S = ops.reference()
        assert_within_tolerance(bf16_to_f64(out[:total].view(np.uint16)), ref, S,
                                f"{fmt} sizes={sizes} n={n} k={k} cg={cta_group}")


SIZES = [
    [128, 256, 384],                 # whole tiles
    [1, 0, 300, 129, 7],             # ragged, one empty group, ends inside store boxes
    [0, 0, 5],                       # leading empty groups
    [500],                           # one group
]


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("sizes", SIZES, ids=lambda s: "-".join(map(str, s)))
def test_grouped_matches_oracle(fmt, sizes, cta_group):
    _check(fmt, sizes, 264, 512, seed=3000 + sum(sizes), cta_group=cta_group, alpha=0.5)


@pytest.mark.parametrize("cta_group", [1, 2])
@pytest.mark.parametrize("n", [8, 16, 72])
@pytest.mark.parametrize("fmt", FMTS)
def test_grouped_narrow_experts(fmt, n, cta_group):
    # N far below the tile: each expert's B box runs into the next expert's rows
    # (and past the end of B for the last one); single-row and ragged groups,
    # the decode regime's shapes
    _check(fmt, [1, 1, 0, 17, 1, 130], n, 640, seed=3200 + n, cta_group=cta_group, alpha=0.5)


@pytest.mark.parametrize("fmt", FMTS)
def test_grouped_many_groups(fmt):
    # 40 groups of 0..200 rows, N a multiple of the tile, K with a ragged last stage
    rng = np.random.default_rng(17)
    sizes = [int(x) for x in rng.integers(0, 201, size=40)]
    sizes[3] = 0
    _check(fmt, sizes, 512, 1056 if fmt == "bf16" else 1088, seed=3100)


@pytest.mark.parametrize("fmt", FMTS)
def test_grouped_all_empty_and_k0(fmt):
    # every group empty: nothing is read or written
    D = torch.full((8, 64), GUARD, dtype=torch.int16, device="cuda")
    X = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    if fmt == "bf16":
        tkg.gemm_grouped_bf16([0, 0], X, X.view(1, 64, 64), D.view(torch.bfloat16))
    elif fmt == "mxfp8":
        tkg.gemm_grouped_mxfp8([0, 0], X.view(64, 64), X.view(1, 64, 64), X, X, D.view(torch.bfloat16))
    else:
        tkg.gemm_grouped_nvfp4([0, 0], X.view(128, 32), X.view(2, 64, 32), X, X, D.view(torch.bfloat16))
    torch.cuda.synchronize()
    assert (D.cpu().numpy() == GUARD).all()
    # K = 0: the groups' rows of D become zero, the rest untouched
    A = torch.zeros((6, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((2, 64, 0), dtype=torch.bfloat16, device="cuda")
    tkg.gemm_grouped_bf16([2, 4], A, B, D.view(torch.bfloat16))
    torch.cuda.synchronize()
    out = D.cpu().numpy()
    assert (out[:6] == 0).all() and (out[6:] == GUARD).all()


def run_grouped_dev(fmt, sizes_dev, dev, D, alpha=1.0):
    A, B, sfa, sfb, ta, tb = dev
    if fmt == "bf16":
        tkg.gemm_grouped_dev_bf16(sizes_dev, A, B, D, alpha)
    elif fmt == "mxfp8":
        tkg.gemm_grouped_dev_mxfp8(sizes_dev, A, B, sfa, sfb, D, alpha)
    else:
        tkg.gemm_grouped_dev_nvfp4(sizes_dev, A, B, sfa, sfb, D, alpha, ta=ta, tb=tb)


def _with_capacity(fmt, ops, dev, capacity):
    """Operands padded to `capacity` rows of A (garbage past the groups) and an
    SFA buffer of the size the device-size entry points require."""
    A, B, sfa, sfb, ta, tb = dev
    extra = capacity - A.shape[0]
    if extra > 0:   # garbage rows past the groups, of A's own dtype
        if A.dtype == torch.uint8:
            pad = torch.randint(0, 256, (extra, A.shape[1]), dtype=torch.int32, device="cuda").to(torch.uint8)
        else:
            pad = torch.randn(extra, A.shape[1], device="cuda").to(A.dtype)
        A = torch.cat([A, pad])
    if fmt != "bf16":
        need = tkg.grouped_dev_scale_bytes(len(ops.sizes), capacity, ops.k, oracle.BLOCK[fmt])
        sfa = torch.cat([sfa, torch.zeros(need - sfa.numel(), dtype=torch.uint8, device="cuda")])
    return A, B, sfa, sfb, ta, tb


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("sizes", [[1, 0, 300, 129, 7], [128, 256, 384], [0, 0, 5]],
                         ids=lambda s: "-".join(map(str, s)))
def test_grouped_device_sizes_equal_host_sizes(fmt, sizes):
    # the same groups with sizes read on the device: identical bits to the
    # host-table launch, and no row past the groups written
    n, k = 264, 512
    ops = GroupedOperands(fmt, sizes, n, k, seed=3300 + sum(sizes))
    dev = ops.upload()
    total = sum(sizes)
    D_host = torch.empty((total, n), dtype=torch.bfloat16, device="cuda")
    run_grouped(fmt, sizes, dev, D_host)
    capacity = total + 100
    dev_c = _with_capacity(fmt, ops, dev, capacity)
    D = torch.full((capacity, n), GUARD, dtype=torch.int16, device="cuda")
    sizes_dev = torch.tensor(sizes, dtype=torch.int32, device="cuda")
    run_grouped_dev(fmt, sizes_dev, dev_c, D.view(torch.bfloat16))
    assert tkg.device_status() == tkg.OK
    out = D.cpu()
    assert torch.equal(out[:total], D_host.cpu().view(torch.int16))
    assert (out[total:] == GUARD).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_grouped_device_sizes_decode_capacity(fmt):
    # the decode regime with device sizes: 8 groups of 16 rows in a capacity of
    # 128 rows (single-CTA tiles), bit for bit the host-table launch
    sizes = [16] * 8
    n, k = 520, 1024
    ops = GroupedOperands(fmt, sizes, n, k, seed=3350)
    dev = ops.upload()
    D_host = torch.empty((128, n), dtype=torch.bfloat16, device="cuda")
    run_grouped(fmt, sizes, dev, D_host)
    dev_c = _with_capacity(fmt, ops, dev, 128)
    D = torch.full((128, n), GUARD, dtype=torch.int16, device="cuda")
    run_grouped_dev(fmt, torch.tensor(sizes, dtype=torch.int32, device="cuda"), dev_c, D.view(torch.bfloat16))
    assert tkg.device_status() == tkg.OK
    assert torch.equal(D.cpu(), D_host.cpu().view(torch.int16))
    ref, S = ops.reference()
    assert_within_tolerance(bf16_to_f64(D_host), ref, S, f"{fmt} decode groups")


def test_grouped_device_sizes_negative_and_over_capacity():
    n, k = 136, 256
    ops = GroupedOperands("bf16", [5, 0, 7], n, k, seed=3400)
    dev = ops.upload()
    D_ref = torch.empty((12, n), dtype=torch.bfloat16, device="cuda")
    run_grouped("bf16", [5, 0, 7], dev, D_ref)
    # a negative size counts as 0
    D = torch.full((12, n), GUARD, dtype=torch.int16, device="cuda")
    run_grouped_dev("bf16", torch.tensor([5, -3, 7], dtype=torch.int32, device="cuda"), dev, D.view(torch.bfloat16))
    assert tkg.device_status() == tkg.OK
    assert torch.equal(D.cpu(), D_ref.cpu().view(torch.int16))
    # sizes past the capacity: rows up to the capacity are right, nothing beyond is touched
    big = torch.full((12 + 64, n), GUARD, dtype=torch.int16, device="cuda")
    Dcap = big[:12]
    run_grouped_dev("bf16", torch.tensor([5, 0, 500], dtype=torch.int32, device="cuda"), dev, Dcap.view(torch.bfloat16))
    assert tkg.device_status() == tkg.OK
    out = big.cpu()
    assert torch.equal(out[:12], D_ref.cpu().view(torch.int16))
    assert (out[12:] == GUARD).all()


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
def test_grouped_decode_full_size(fmt):
    # the bench's decode-regime grouped GEMM: 8 experts x 16 rows, N=4096, K=7168
    _check(fmt, [16] * 8, 4096, 7168, seed=3300)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
def test_grouped_prefill_full_size_sampled(fmt):
    # the bench's prefill grouped GEMM (8 experts, 16384 rows in the seeded
    # 128-row-multiple sizes, N=4096, K=7168): the first and last 32 rows of
    # every other group against the oracle on that group's own slices
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    sizes = bench.grouped_sizes(8, 16384)
    n, k = 4096, 7168
    ops = GroupedOperands(fmt, sizes, n, k, seed=3400)
    dev = ops.upload()
    D = torch.empty((sum(sizes), n), dtype=torch.bfloat16, device="cuda")
    run_grouped(fmt, sizes, dev, D)
    assert tkg.device_status() == tkg.OK
    got = bf16_to_f64(D)
    row0 = np.concatenate([[0], np.cumsum(sizes)])
    for g in range(0, len(sizes), 2):
        for r in (0, sizes[g] - 32):
            a0 = int(row0[g]) + r
            sfa = ops.sfa[a0:a0 + 32] if ops.sfa is not None else None
            sfb = ops.sfb[g] if ops.sfb is not None else None
            ref, S = oracle.gemm(fmt, ops.A[a0:a0 + 32], ops.B[g], sfa, sfb, ops.alphas[g])
            assert_within_tolerance(got[a0:a0 + 32], ref, S, f"{fmt} group {g} rows {r}..")
