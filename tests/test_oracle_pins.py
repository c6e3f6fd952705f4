"""Pins for the CPU oracle, each against something other than the oracle itself:
library decoders (torch's float8 / bfloat16 casts), exhaustive nearest-value
searches, exact rational arithmetic (fractions.Fraction) and closed forms.

Format names come from "ThunderKittens 2.0 GPU Kernel优化" (opening section:
BF16/MXFP8/NVFP4 GEMMs); the quantisation rules are those of the workload
definition (MXFP8 scale 2^ceil(log2(amax/448)); NVFP4 tensor scale
amax/(6*448), block scale blockamax/(6*tensor scale))."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dense_block_scaled_gb300 import synth

E4M3_NAN = (0x7F, 0xFF)


# --------------------------------------------------------------------------- decoders

def test_decode_bf16_matches_torch():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    lib = codes.view(torch.bfloat16).to(torch.float64).numpy()
    ours = oracle.decode_table("bf16")
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], ours[ok])


def test_decode_e4m3_matches_torch():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.decode_table("e4m3")
    assert sorted(np.flatnonzero(np.isnan(ours)).tolist()) == list(E4M3_NAN)
    ok = ~np.isnan(lib)
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    assert np.array_equal(lib[ok], ours[ok])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_decode_e8m0_matches_torch():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    ours = oracle.decode_table("e8m0")
    assert np.isnan(ours[255]) and np.isnan(lib[255])
    assert np.array_equal(lib[:255], ours[:255])
    assert ours[127] == 1.0


def test_decode_e2m1_closed_form():
    # E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign.
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    ours = oracle.decode_table("e2m1")
    assert ours[:8].tolist() == mags
    assert ours[8:].tolist() == [-v for v in mags]


# --------------------------------------------------------------------------- rounding

def _nearest_even_code(v: float, table: np.ndarray, codes, vmax: float, mant_mask: int):
    """Exhaustive search: the code whose value is nearest to v; a tie goes to the
    code with an even mantissa; |v| beyond the largest finite clamps to it."""
    a = min(abs(v), vmax)
    best, bestd = None, None
    for c in codes:
        d = abs(table[c] - a)
        if bestd is None or d < bestd or (d == bestd and (c & mant_mask) % 2 == 0):
            best, bestd = c, d
    return best


def _fp32_samples(seed, n):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n).astype(np.float32) * np.float32(60.0)
    return x


def test_round_e4m3_bruteforce():
    table = oracle.decode_table("e4m3")
    pos = [c for c in range(0x7F)]  # non-negative finite codes
    vals = list(_fp32_samples(1, 400))
    # every midpoint between neighbours (exact ties) and both its float neighbours
    grid = sorted(set(table[c] for c in pos))
    for lo, hi in zip(grid[:-1], grid[1:]):
        mid = np.float32((lo + hi) / 2)
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))]
    vals += [448.0, 449.0, 463.9, 464.0, 1e6, 2.0 ** -10, 2.0 ** -11, 0.0]
    for v in vals:
        v = np.float32(v)
        want = _nearest_even_code(float(v), table, pos, 448.0, 0x1)
        got = oracle.f32_to_e4m3(v)
        assert got & 0x7F == want, (float(v), got, want)
        assert (got >> 7) == (1 if np.signbit(v) else 0)
        assert oracle.f32_to_e4m3(np.float32(-abs(v))) == (want | 0x80)
        assert oracle.f32_to_e4m3(np.float32(abs(v))) == want


def test_round_e4m3_matches_torch_in_range():
    v = _fp32_samples(2, 20000)
    v = v[np.abs(v) <= 448.0]
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.f32_to_e4m3(x) for x in v], dtype=np.uint8)
    assert np.array_equal(lib, ours)


def test_round_e2m1_ties_and_saturation():
    cases = {0.25: 0x0, 0.75: 0x2, 1.25: 0x2, 1.75: 0x4, 2.5: 0x4, 3.5: 0x6, 5.0: 0x6,
             6.0: 0x7, 6.9: 0x7, 7.0: 0x7, 100.0: 0x7, 0.2: 0x0, 0.3: 0x1, 5.1: 0x7}
    for v, code in cases.items():
        assert oracle.f32_to_e2m1(v) == code, v
        assert oracle.f32_to_e2m1(-v) == code | 0x8, v


def test_round_e2m1_bruteforce():
    table = oracle.decode_table("e2m1")
    pos = list(range(8))
    for v in _fp32_samples(3, 2000) / np.float32(8.0):
        want = _nearest_even_code(float(v), table, pos, 6.0, 0x1)
        got = oracle.f32_to_e2m1(v)
        assert got & 0x7 == want, (float(v), got, want)


# --------------------------------------------------------------------------- quantisers

def _smallest_e(amax: float) -> int:
    """Brute force: smallest integer e in [-127, 127] with 448 * 2^e >= amax."""
    for e in range(-127, 128):
        if Fraction(448) * Fraction(2) ** e >= Fraction(float(amax)):
            return e
    return 127


def test_quant_mxfp8_scale_rule():
    rng = np.random.default_rng(5)
    rows = []
    for e in (-20, -3, 0, 1, 7, 30):
        base = np.float32(448.0 * 2.0 ** e)
        blk = rng.standard_normal(32).astype(np.float32) * np.float32(2.0 ** e)
        blk[0] = base                      # amax exactly 448 * 2^e -> code e + 127
        rows.append(blk)
        blk2 = blk.copy()
        blk2[0] = np.nextafter(base, np.float32(np.inf))   # just above -> e + 1
        rows.append(blk2)
    rows.append(np.zeros(32, np.float32))                  # zero block -> code 0
    rows.append(np.full(32, np.float32(2.0 ** -140)))       # tiny -> clamped to -127
    X = np.stack(rows)
    Q, SF = oracle.quant_mxfp8(X)
    for r in range(X.shape[0]):
        amax = float(np.max(np.abs(X[r])))
        e = -127 if amax == 0.0 else _smallest_e(amax)
        assert SF[r, 0] == e + 127, (r, amax, SF[r, 0], e)
    assert np.all(Q[-2] == 0)
    assert SF[0, 0] == -20 + 127 and SF[1, 0] == -19 + 127


def test_quant_mxfp8_values_are_nearest():
    a, _ = synth.gemm_inputs_f32(8, 1, 256, seed=11)
    Q, SF = oracle.quant_mxfp8(a)
    table = oracle.decode_table("e4m3")
    finite = [c for c in range(0x7F)]
    for r in range(a.shape[0]):
        for b in range(256 // 32):
            e = int(SF[r, b]) - 127
            assert _smallest_e(np.max(np.abs(a[r, b * 32:(b + 1) * 32]))) == e
            for i in range(b * 32, b * 32 + 32, 7):
                scaled = np.float32(a[r, i]) * np.float32(2.0 ** -e)   # exact power-of-two scaling
                want = _nearest_even_code(float(scaled), table, finite, 448.0, 0x1)
                assert Q[r, i] & 0x7F == want


def test_quant_nvfp4_rules():
    a, _ = synth.gemm_inputs_f32(6, 1, 128, seed=12)
    a[3, 16:32] = 0.0                      # one all-zero block
    Q, SF, t = oracle.quant_nvfp4(a)
    amax = np.float32(np.max(np.abs(a)))
    assert t == np.float32(amax) / np.float32(2688.0)      # IEEE FP32 division (numpy)
    e4 = oracle.decode_table("e4m3")
    e2 = oracle.decode_table("e2m1")
    for r in range(a.shape[0]):
        for b in range(128 // 16):
            blk = a[r, b * 16:(b + 1) * 16]
            ratio = np.float32(np.max(np.abs(blk))) / (np.float32(6.0) * t)
            want_s = _nearest_even_code(float(ratio), e4, list(range(0x7F)), 448.0, 0x1)
            assert SF[r, b] == want_s
            den = np.float32(np.float32(e4[SF[r, b]]) * t)
            for i in range(16):
                nib = (Q[r, (b * 16 + i) // 2] >> (4 * (i % 2))) & 0xF
                if den == 0:
                    assert nib == 0
                    continue
                q = np.float32(blk[i]) / den
                want = _nearest_even_code(float(q), e2, list(range(8)), 6.0, 0x1)
                assert nib & 0x7 == want
                # reconstruction stays within half an E2M1 step (or saturates at 6)
                rec = e2[nib] * float(den)
                step = {0: 0.5, 1: 0.5, 2: 1.0, 3: 2.0}
                mag = min(abs(float(q)), 6.0)
                half = 0.5 * (0.5 if mag < 2 else (1.0 if mag < 4 else 2.0))
                assert abs(abs(rec) - mag * float(den)) <= half * float(den) * (1 + 1e-6)
    assert np.all(SF[3, 1] == 0)


def test_quant_nvfp4_given_scale_closed_forms():
    # the NVFP4 rule with the tensor scale supplied, t = 2^-10, every step exact:
    #   block 0: max 12t -> s = E4M3(12t / 6t) = 2.0 (0x40), den = 2t; 12t -> 6 (0x7),
    #            3t -> 1.5 (0x3), -t -> -0.5 (0x9)
    #   block 1: max 10000t is above 6 * 448 * t: s saturates at 448 (0x7E), den = 448t;
    #            10000t / den = 22.3 saturates to 6 (0x7); 448t -> 1.0 (0x2)
    #   block 2: all zero -> s = 0, codes 0
    #   block 3: max 6 * 2^-9 * t -> s = 2^-9, the smallest E4M3 subnormal (0x01); that max -> 6
    t = np.float32(2.0 ** -10)
    x = np.zeros((1, 64), np.float32)
    x[0, 0], x[0, 1], x[0, 2] = 12 * t, 3 * t, -t
    x[0, 16], x[0, 17] = 10000 * t, 448 * t
    x[0, 48] = 6 * t * np.float32(2.0 ** -9)
    Q, SF, tt = oracle.quant_nvfp4(x, t=t)
    assert tt == t
    assert list(SF[0, :4]) == [0x40, 0x7E, 0x00, 0x01]
    want = np.zeros(32, np.uint8)
    want[0], want[1], want[8], want[24] = 0x37, 0x09, 0x27, 0x07
    assert np.array_equal(Q[0], want)
    # decoded, the saturated element sits at the ceiling 6 * 448 * t
    e2m1, e4m3 = oracle.decode_table("e2m1"), oracle.decode_table("e4m3")
    assert e2m1[Q[0, 8] & 0xF] * e4m3[SF[0, 1]] * float(t) == 2688 * float(t)


def test_quant_nvfp4_given_scale_agrees_with_amax_rule():
    # given its own amax / 2688, the given-scale path reproduces the full rule;
    # t <= 0 gives all-zero codes and scales
    a, _ = synth.gemm_inputs_f32(9, 1, 160, seed=13)
    Q0, SF0, t0 = oracle.quant_nvfp4(a)
    assert t0 == np.float32(np.float32(np.abs(a).max()) / np.float32(2688))
    Q1, SF1, _ = oracle.quant_nvfp4(a, t=t0)
    assert np.array_equal(Q0, Q1) and np.array_equal(SF0, SF1)
    for bad in (0.0, -1.0):
        Q2, SF2, _ = oracle.quant_nvfp4(a, t=bad)
        assert not Q2.any() and not SF2.any()


def test_quant_nvfp4_zero_tensor():
    Q, SF, t = oracle.quant_nvfp4(np.zeros((4, 64), np.float32))
    assert t == 0.0 and not Q.any() and not SF.any()


# --------------------------------------------------------------------------- GEMM

def _exact_gemm(fmt, A, B, sfa, sfb, alpha):
    """Exact rational GEMM from torch-decoded values (an independent decoder)."""
    def dec_vals(X):
        if fmt == "bf16":
            return torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).double().numpy()
        if fmt == "mxfp8":
            return torch.from_numpy(X).view(torch.float8_e4m3fn).double().numpy()
        lo = X & 0xF
        hi = X >> 4
        nib = np.stack([lo, hi], axis=-1).reshape(X.shape[0], -1)
        mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
        return np.where(nib & 8, -1.0, 1.0) * mags[nib & 7]

    def dec_sf(s):
        if fmt == "mxfp8":
            return torch.from_numpy(s).view(torch.float8_e8m0fnu).double().numpy()
        return torch.from_numpy(s).view(torch.float8_e4m3fn).double().numpy()

    a, b = dec_vals(A), dec_vals(B)
    k = a.shape[1]
    if fmt != "bf16":
        bs = oracle.BLOCK[fmt]
        a = a * np.repeat(dec_sf(sfa)[:, : k // bs], bs, axis=1)
        b = b * np.repeat(dec_sf(sfb)[:, : k // bs], bs, axis=1)
    al = Fraction(alpha)
    ref = [[al * sum(Fraction(a[i, kk]) * Fraction(b[j, kk]) for kk in range(k))
            for j in range(b.shape[0])] for i in range(a.shape[0])]
    S = [[sum(abs(al * Fraction(a[i, kk]) * Fraction(b[j, kk])) for kk in range(k))
          for j in range(b.shape[0])] for i in range(a.shape[0])]
    return ref, S


def _rand_operands(fmt, m, n, k, seed, sf_lo, sf_hi):
    rng = np.random.default_rng(seed)
    if fmt == "bf16":
        A = synth.bf16_codes(rng.standard_normal((m, k)).astype(np.float32))
        B = synth.bf16_codes(rng.standard_normal((n, k)).astype(np.float32))
        return A, B, None, None
    if fmt == "mxfp8":
        A = synth.random_codes((m, k), 256, seed, E4M3_NAN).astype(np.uint8)
        B = synth.random_codes((n, k), 256, seed + 1, E4M3_NAN).astype(np.uint8)
    else:
        A = synth.random_codes((m, k // 2), 256, seed).astype(np.uint8)
        B = synth.random_codes((n, k // 2), 256, seed + 1).astype(np.uint8)
    ld = oracle.ld_sf(k, fmt)
    sfa = np.zeros((m, ld), np.uint8)
    sfb = np.zeros((n, ld), np.uint8)
    kb = k // oracle.BLOCK[fmt]
    sfa[:, :kb] = rng.integers(sf_lo, sf_hi, size=(m, kb))
    sfb[:, :kb] = rng.integers(sf_lo, sf_hi, size=(n, kb))
    return A, B, sfa, sfb


@pytest.mark.parametrize("fmt,m,n", [("bf16", 16, 16), ("mxfp8", 16, 16), ("nvfp4", 16, 16),
                                     ("mxfp8", 12, 5), ("nvfp4", 5, 12), ("bf16", 3, 9)])
def test_gemm_bruteforce_fraction(fmt, m, n):
    k = 64
    # Scale codes bounded so every FP8/FP4 sum is exact in FP64: MXFP8 products
    # are multiples of 2^-22 below 2^21.6 (scales 2^-2..2^2), so 64 of them need
    # < 50 bits; NVFP4 products are multiples of 2^-14 below 2^13.
    lo, hi = {"bf16": (0, 1), "mxfp8": (125, 130), "nvfp4": (0x20, 0x50)}[fmt]
    A, B, sfa, sfb = _rand_operands(fmt, m, n, k, seed=100 + m * 7 + n, sf_lo=lo, sf_hi=hi)
    alpha = 0.75
    ref, S = oracle.gemm(fmt, A, B, sfa, sfb, alpha)
    eref, eS = _exact_gemm(fmt, A, B, sfa, sfb, alpha)
    for i in range(m):
        for j in range(n):
            if fmt == "bf16":
                assert abs(Fraction(ref[i, j]) - eref[i][j]) <= Fraction(2) ** -52 * eS[i][j]
            else:
                assert Fraction(ref[i, j]) == eref[i][j], (i, j)
            assert abs(Fraction(S[i, j]) - eS[i][j]) <= Fraction(2) ** -50 * eS[i][j]


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
def test_gemm_identity_closed_form(fmt):
    # A = I (M = K):  D[i][j] = sA(i, i/bs) * dec(B[j][i]) * sB(j, i/bs)
    k = 64
    n = 24
    _, B, _, sfb = _rand_operands(fmt, 1, n, k, seed=7, sf_lo=120, sf_hi=134) if fmt == "mxfp8" else \
        _rand_operands(fmt, 1, n, k, seed=7, sf_lo=0x30, sf_hi=0x48)
    if fmt == "bf16":
        A = np.zeros((k, k), np.uint16)
        A[np.arange(k), np.arange(k)] = 0x3F80
        sfa = None
    elif fmt == "mxfp8":
        A = np.zeros((k, k), np.uint8)
        A[np.arange(k), np.arange(k)] = 0x38          # E4M3 1.0
        sfa = np.full((k, oracle.ld_sf(k, fmt)), 127, np.uint8)
    else:
        A = np.zeros((k, k // 2), np.uint8)
        for i in range(k):
            A[i, i // 2] |= (0x2 << (4 * (i % 2)))     # E2M1 1.0
        sfa = np.full((k, oracle.ld_sf(k, fmt)), 0x38, np.uint8)   # E4M3 1.0
    ref, _ = oracle.gemm(fmt, A, B, sfa, sfb, 1.0)
    eref, _ = _exact_gemm(fmt, np.ascontiguousarray(A), B, sfa, sfb, 1.0)
    # closed form, element by element: the decoded (scaled) B transposed
    for i in range(k):
        for j in range(n):
            assert Fraction(ref[i, j]) == eref[i][j]
    bdec = np.array(eref, dtype=object)
    assert bdec.shape == (k, n)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
def test_gemm_all_ones_closed_form(fmt):
    # all-ones A with unit scales: D[i][j] = sum_k dec(b_jk) * sB(j, k/bs)
    m, n, k = 3, 10, 96
    lo, hi = {"bf16": (0, 1), "mxfp8": (120, 134), "nvfp4": (0x30, 0x48)}[fmt]
    _, B, _, sfb = _rand_operands(fmt, 1, n, k, seed=9, sf_lo=lo, sf_hi=hi)
    if fmt == "bf16":
        A = np.full((m, k), 0x3F80, np.uint16)
        sfa = None
    elif fmt == "mxfp8":
        A = np.full((m, k), 0x38, np.uint8)
        sfa = np.full((m, oracle.ld_sf(k, fmt)), 127, np.uint8)
    else:
        A = np.full((m, k // 2), 0x22, np.uint8)
        sfa = np.full((m, oracle.ld_sf(k, fmt)), 0x38, np.uint8)
    ref, _ = oracle.gemm(fmt, A, B, sfa, sfb, 1.0)
    if fmt == "bf16":
        bvals = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).double().numpy()
    elif fmt == "mxfp8":
        bvals = torch.from_numpy(B).view(torch.float8_e4m3fn).double().numpy() * \
            np.repeat(torch.from_numpy(sfb).view(torch.float8_e8m0fnu).double().numpy()[:, :k // 32], 32, 1)
    else:
        nib = np.stack([B & 0xF, B >> 4], -1).reshape(n, k)
        mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
        bvals = np.where(nib & 8, -1.0, 1.0) * mags[nib & 7] * \
            np.repeat(torch.from_numpy(sfb).view(torch.float8_e4m3fn).double().numpy()[:, :k // 16], 16, 1)
    for j in range(n):
        want = sum(Fraction(v) for v in bvals[j])
        for i in range(m):
            if fmt == "bf16":
                assert abs(Fraction(ref[i, j]) - want) <= Fraction(2) ** -50 * sum(abs(Fraction(v)) for v in bvals[j])
            else:
                assert Fraction(ref[i, j]) == want


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_gemm_every_code_pair(fmt):
    # one-hot: A[i][0] = code i, B[j][0] = code j, all else 0, unit scales
    if fmt == "mxfp8":
        codes = [c for c in range(256) if c not in E4M3_NAN]
        k = 32
        A = np.zeros((len(codes), k), np.uint8)
        A[:, 0] = codes
        B = A.copy()
        unit = 127
        dec = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    else:
        codes = list(range(16))
        k = 32
        A = np.zeros((16, k // 2), np.uint8)
        A[:, 0] = codes
        B = A.copy()
        unit = 0x38
        mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
        dec = np.array([(-1.0 if c & 8 else 1.0) * mags[c & 7] for c in codes])
    ld = oracle.ld_sf(k, fmt)
    sfa = np.full((A.shape[0], ld), unit, np.uint8)
    ref, _ = oracle.gemm(fmt, A, B, sfa, sfa, 1.0)
    assert np.array_equal(ref, np.outer(dec, dec))


def test_gemm_bf16_every_code_onehot():
    # one-hot B = e_0: D[i][0] reproduces every finite BF16 code of A exactly
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = codes[((codes >> 7) & 0xFF) != 0xFF]
    A = np.zeros((finite.size, 8), np.uint16)
    A[:, 0] = finite
    B = np.zeros((2, 8), np.uint16)
    B[0, 0] = 0x3F80
    ref, _ = oracle.gemm("bf16", A, B)
    want = torch.from_numpy(finite.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(ref[:, 0], want)
    assert not ref[:, 1].any()


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_gemm_scale_index(fmt):
    # values 1.0 in the single block b of row i; distinct scale codes per
    # (row, block): D[i][j] = dec(sA[i][b]) * dec(sB[j][b])
    bs = oracle.BLOCK[fmt]
    m, n, k = 9, 7, bs * 6
    one = 0x38 if fmt == "mxfp8" else 0x2
    ld = oracle.ld_sf(k, fmt)
    rng = np.random.default_rng(3)
    lo, hi = (100, 150) if fmt == "mxfp8" else (0x20, 0x58)
    sfa = rng.integers(lo, hi, size=(m, ld)).astype(np.uint8)
    sfb = rng.integers(lo, hi, size=(n, ld)).astype(np.uint8)
    blk_a = rng.integers(0, k // bs, size=m)
    blk_b = rng.integers(0, k // bs, size=n)

    def fill(rows, blk):
        if fmt == "mxfp8":
            X = np.zeros((rows, k), np.uint8)
            for r in range(rows):
                X[r, blk[r] * bs:(blk[r] + 1) * bs] = one
        else:
            X = np.zeros((rows, k // 2), np.uint8)
            for r in range(rows):
                X[r, blk[r] * bs // 2:(blk[r] + 1) * bs // 2] = one | (one << 4)
        return X

    A, B = fill(m, blk_a), fill(n, blk_b)
    ref, _ = oracle.gemm(fmt, A, B, sfa, sfb, 1.0)
    sdec = oracle.decode_table("e8m0" if fmt == "mxfp8" else "e4m3")
    for i in range(m):
        for j in range(n):
            want = 0.0 if blk_a[i] != blk_b[j] else bs * sdec[sfa[i, blk_a[i]]] * sdec[sfb[j, blk_b[j]]]
            assert ref[i, j] == want


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
def test_gemm_elems_equal_rows(fmt):
    lo, hi = {"bf16": (0, 1), "mxfp8": (110, 140), "nvfp4": (0x20, 0x50)}[fmt]
    A, B, sfa, sfb = _rand_operands(fmt, 20, 17, 128, seed=21, sf_lo=lo, sf_hi=hi)
    ref, S = oracle.gemm(fmt, A, B, sfa, sfb, 1.5)
    ii = np.array([0, 5, 19, 7, 13])
    jj = np.array([16, 0, 3, 9, 11])
    r2, s2 = oracle.gemm_elems(fmt, A, B, sfa, sfb, 1.5, ii, jj)
    assert np.array_equal(r2, ref[ii, jj]) and np.array_equal(s2, S[ii, jj])
    r3, s3 = oracle.gemm(fmt, A, B, sfa, sfb, 1.5, rows=(5, 7))
    assert np.array_equal(r3, ref[5:12]) and np.array_equal(s3, S[5:12])


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "nvfp4"])
def test_gemm_grouped_bruteforce_fraction(fmt):
    # grouped GEMM: each group's rows against its own B, per-group alpha;
    # checked against the exact rational product of the group's slice
    sizes = [3, 0, 5, 1]
    n, k = 6, 64
    lo, hi = {"bf16": (0, 1), "mxfp8": (125, 130), "nvfp4": (0x20, 0x50)}[fmt]
    A, _, sfa, _ = _rand_operands(fmt, sum(sizes), 1, k, seed=31, sf_lo=lo, sf_hi=hi)
    Bs, sfbs = [], []
    for g in range(len(sizes)):
        _, Bg, _, sfbg = _rand_operands(fmt, 1, n, k, seed=40 + g, sf_lo=lo, sf_hi=hi)
        Bs.append(Bg)
        sfbs.append(sfbg)
    B = np.stack(Bs)
    sfb = None if fmt == "bf16" else np.stack(sfbs)
    alphas = [0.5, 2.0, -1.0, 0.25]
    ref, S = oracle.gemm_grouped(fmt, sizes, A, B, sfa, sfb, alphas)
    assert ref.shape == (sum(sizes), n)
    row = 0
    for g, mg in enumerate(sizes):
        if mg == 0:
            continue
        sl = slice(row, row + mg)
        eref, eS = _exact_gemm(fmt, A[sl], B[g], None if sfa is None else sfa[sl],
                               None if sfb is None else sfb[g], alphas[g])
        for i in range(mg):
            for j in range(n):
                if fmt == "bf16":
                    assert abs(Fraction(ref[row + i, j]) - eref[i][j]) <= Fraction(2) ** -52 * eS[i][j]
                else:
                    assert Fraction(ref[row + i, j]) == eref[i][j], (g, i, j)
        row += mg


# --------------------------------------------------------------------------- NVFP4 per-tensor scales

def _round_f32(x: Fraction) -> Fraction:
    """x > 0 rounded to the nearest FP32 value, ties to even (normal range),
    written from the definition: 24 significant bits at x's binade."""
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    q = x / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n * ulp


def test_alpha_eff_double_rounding_in_fp32():
    # The NVFP4 per-tensor scales join alpha as fp32(fp32(alpha * tA) * tB): two
    # FP32 products in that order ("ThunderKittens 2.0 GPU Kernel优化", table of
    # updates: NVFP4 with its FP32 per-tensor scale).  These operands are exact
    # FP32 values chosen so that every plausible slip -- one rounding of the
    # exact product, the other multiplication order, an FP64 product -- gives a
    # different FP32 result.
    alpha = 1 + Fraction(1025, 2 ** 23)
    ta = (1 + Fraction(1, 4096)) * Fraction(1, 2 ** 9)
    tb = (1 + Fraction(3, 4096)) * Fraction(1, 2 ** 10)
    for v in (alpha, ta, tb):
        assert _round_f32(v) == v
    want = _round_f32(_round_f32(alpha * ta) * tb)
    slips = {
        "single rounding": _round_f32(alpha * ta * tb),
        "tA*tB first": _round_f32(alpha * _round_f32(ta * tb)),
        "alpha*tB first": _round_f32(_round_f32(alpha * tb) * ta),
        "fp64 product": Fraction(float(np.float32(float(alpha) * float(ta) * float(tb)))),
    }
    for name, v in slips.items():
        assert v != want, name
    got = oracle.alpha_eff(float(alpha), float(ta), float(tb))
    assert Fraction(got) == want
    # a scale of 1.0 leaves alpha as is, and the default arguments are 1.0
    assert oracle.alpha_eff(float(alpha)) == float(alpha)
    assert oracle.alpha_eff(0.75, 1.0, 1.0) == 0.75
