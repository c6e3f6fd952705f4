"""Test-side helpers: layout conversion written from the ABI's description of
the tiled scale layout, BF16 decoding through torch, and the tolerance check.
Nothing here is shared with the CUDA library."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def tiled_scales(sf_rowmajor: np.ndarray, kblocks: int) -> np.ndarray:
    """Row-major (rows, >= kblocks) scale codes -> tiled byte buffer.

    Scale (r, kb) sits at ((r//128)*KA + kb//4)*512 + (r%32)*16 + ((r%128)//32)*4 + kb%4,
    KA = ceil(kblocks/4); padding bytes are zero."""
    rows = sf_rowmajor.shape[0]
    ka = -(-kblocks // 4)
    rb = -(-rows // 128)
    out = np.zeros(rb * 128 * ka * 4, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    kb = np.arange(kblocks)[None, :]
    off = ((r // 128) * ka + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4
    out[off.ravel()] = sf_rowmajor[:, :kblocks].ravel()
    return out


def bf16_to_f64(codes) -> np.ndarray:
    if isinstance(codes, torch.Tensor):
        codes = codes.cpu()
        if codes.dtype == torch.bfloat16:
            return codes.double().numpy()
        return codes.view(torch.bfloat16).double().numpy()
    return torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).view(torch.bfloat16).double().numpy()


def tolerance_violations(d: np.ndarray, ref: np.ndarray, S: np.ndarray):
    """Elements breaking |D - ref| <= 2^-7 |ref| + 1e-5 * S (the acceptance bound)."""
    err = np.abs(d - ref)
    bound = 2.0 ** -7 * np.abs(ref) + 1e-5 * S
    bad = ~(err <= bound)
    return bad, err, bound


def assert_within_tolerance(d, ref, S, what=""):
    bad, err, bound = tolerance_violations(d, ref, S)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: got {d[tuple(i)]!r} ref {ref[tuple(i)]!r} bound {bound[tuple(i)]:.3g}"
                           for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; {detail}")


def to_dev(a: np.ndarray, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


class Operands:
    """Seeded operands of one GEMM in every representation the tests need."""

    def __init__(self, fmt, m, n, k, seed, alpha=1.0):
        from dense_block_scaled_gb300 import synth
        self.fmt, self.m, self.n, self.k, self.alpha = fmt, m, n, k, alpha
        a, b = synth.gemm_inputs_f32(m, n, k, seed)
        self.ta = self.tb = None
        if fmt == "bf16":
            self.A, self.B = synth.bf16_codes(a), synth.bf16_codes(b)
            self.sfa = self.sfb = None
            self.alpha_eff = alpha
        elif fmt == "mxfp8":
            self.A, self.sfa = oracle.quant_mxfp8(a)
            self.B, self.sfb = oracle.quant_mxfp8(b)
            self.alpha_eff = alpha
        else:
            self.A, self.sfa, self.ta = oracle.quant_nvfp4(a)
            self.B, self.sfb, self.tb = oracle.quant_nvfp4(b)
            self.alpha_eff = oracle.alpha_eff(alpha, self.ta, self.tb)

    def reference(self, rows=None):
        return oracle.gemm(self.fmt, self.A, self.B, self.sfa, self.sfb, self.alpha_eff, rows=rows)

    def reference_elems(self, ii, jj):
        return oracle.gemm_elems(self.fmt, self.A, self.B, self.sfa, self.sfb, self.alpha_eff, ii, jj)

    def upload(self):
        """Device tensors (A, B, sfa_tiled, sfb_tiled, ta, tb)."""
        bs = oracle.BLOCK.get(self.fmt)
        A = to_dev(self.A)
        B = to_dev(self.B)
        if self.fmt == "bf16":
            return A, B, None, None, None, None
        kb = self.k // bs
        sfa = to_dev(tiled_scales(self.sfa, kb))
        sfb = to_dev(tiled_scales(self.sfb, kb))
        ta = tb = None
        if self.fmt == "nvfp4":
            ta = torch.tensor([float(self.ta)], dtype=torch.float32, device="cuda")
            tb = torch.tensor([float(self.tb)], dtype=torch.float32, device="cuda")
        return A, B, sfa, sfb, ta, tb


def run_gemm(fmt, dev_ops, m, n, k, alpha, D=None, stream=None):
    from dense_block_scaled_gb300 import tkg
    A, B, sfa, sfb, ta, tb = dev_ops
    if D is None:
        D = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    if fmt == "bf16":
        tkg.gemm_bf16(A, B, D, alpha, stream=stream)
    elif fmt == "mxfp8":
        tkg.gemm_mxfp8(A, B, sfa, sfb, D, alpha, stream=stream)
    else:
        tkg.gemm_nvfp4(A, B, sfa, sfb, D, alpha, ta=ta, tb=tb, stream=stream)
    return D
