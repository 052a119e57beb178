"""Shared helpers for the GPU parity tests: run a Case through the C ABI with
a guarded, NaN-prefilled output buffer, run the same Case through the CPU
oracle, and compare."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import workloads as W

GUARD = 256                      # elements of canary on each side of Y
SENTINEL = 0x7FDA                # a NaN bit pattern in both fp16 and bf16

TOL = {None: (1e-2, 1e-3), "fp8": (3e-2, 3e-3), "int8": (3e-2, 3e-3)}

# Allowance for quantised codes that may legitimately round either way.  The
# kernel decides each code from x = 2^(S*c - lam) in fp32: S is the tensor
# core's fp32 dot product of 16-bit values, c = scale*log2(e), lam = m +
# log2(l) + log2(s_q) with l an fp32 sum of exponentials.  Its relative error
# is ln2 * |error of S*c - lam| plus the error of the hardware exp2 (about
# 2^-22).  Emulating that arithmetic on the CPU (fp32 dot products, fp32 sums
# in the kernel's order) over 1.1 M codes of the 4 x 16 x 4096 quantized
# workload gave at most 2.7e-6 (2^-18.5).  AMBIGUITY_EPS = 2^-16 is about six
# times that, for the tensor core's own accumulation order and the exp2.  It
# is relative, with no absolute floor: the oracle marks a code only when x
# lies within AMBIGUITY_EPS * x of a rounding midpoint.  test_gpu_code_flips
# reads the kernel's codes directly and checks that every code that differs
# from the oracle's is one of those.  Tests assert the raw error (no
# allowance) against the tolerance too.
AMBIGUITY_EPS = 2.0 ** -16


def guarded_output(q):
    """Y as a view into a bigger buffer prefilled with SENTINEL."""
    n = q.numel()
    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.int16, device=q.device)
    y = buf[GUARD:GUARD + n].view(q.dtype).view(q.shape)
    return buf, y


def run_gpu(case: W.Case, *, status=None):
    """Returns (y_gpu as float64 numpy, raw int16 buffer, status tensor)."""
    dc = W.to_device(case, "cuda")
    buf, y = guarded_output(dc.q)
    kw = dict(q_form=dc.q_form, kv_form=dc.kv_form, query_lengths=dc.query_lengths,
              kv_lengths=dc.kv_lengths, mask=dc.mask, scale=dc.scale, causal=dc.causal,
              norm=dc.norm, out=y, status=status, return_status=True)
    if dc.kv_form == W.PAGED:
        ks, vs = dc.kv_scales if dc.kv_scales is not None else (None, None)
        _, st = binding.trt_attention_paged_kv(
            dc.q, dc.k, dc.v, dc.page_table, dc.kv_lengths, k_scale=ks, v_scale=vs,
            q_form=dc.q_form, query_lengths=dc.query_lengths, mask=dc.mask, scale=dc.scale,
            causal=dc.causal, norm=dc.norm, out=y, status=status, return_status=True)
    elif dc.kv_scales is not None:
        _, st = binding.trt_attention_fp8_kv(dc.q, dc.k, dc.v, k_scale=dc.kv_scales[0],
                                             v_scale=dc.kv_scales[1], **kw)
    elif dc.quant is None:
        _, st = binding.trt_attention(dc.q, dc.k, dc.v, **kw)
    else:
        _, st = binding.trt_quantized_attention(dc.q, dc.k, dc.v, quant=dc.quant,
                                                quant_scale=dc.quant_scale, **kw)
    torch.cuda.synchronize()
    return y.double().cpu().numpy(), buf.cpu().numpy(), st


def run_oracle(case: W.Case):
    """Oracle output, or (output, ambiguity bound) for the quantized op.  A
    paged cache is first gathered into the linear padded cache."""
    k, v, kv_form = case.k, case.v, case.kv_form
    if kv_form == W.PAGED:
        k = oracle.gather_pages(case.k, case.page_table, 0, case.kv_lens)
        v = oracle.gather_pages(case.v, case.page_table, 1, case.kv_lens)
        kv_form = W.PADDED
    return oracle.attention(
        case.q, k, v, q_form=case.q_form, kv_form=kv_form,
        query_lengths=case.query_lengths, kv_lengths=case.kv_lengths, mask=case.mask,
        scale=case.scale, causal=case.causal, norm=case.norm, quant=case.quant,
        quant_scale=case.quant_scale,
        ambiguity_eps=AMBIGUITY_EPS if case.quant else None, kv_fp8_scales=case.kv_scales)


def valid_row_mask(case: W.Case):
    """Boolean array over Y's rows (all but the last dim): True where the
    row belongs to a sequence and must be written."""
    if case.q_form == W.PACKED:
        m = np.zeros(case.q.shape[:-1], dtype=bool)
        m[:sum(case.q_lens)] = True
        return m
    B, H, N = case.q.shape[:3]
    m = np.zeros((B, H, N), dtype=bool)
    for b, n in enumerate(case.q_lens):
        m[b, :, :n] = True
    return m


def check(case: W.Case, y_gpu, raw, y_ref, tol=None):
    """Element-wise parity on valid rows; bit-exact sentinel elsewhere.

    For the quantized op the raw error (no allowance) must meet the
    tolerance, and so must the error less the oracle's ambiguity bound.
    Returns the raw max-abs error."""
    atol_max, atol_mean = tol or TOL[case.quant]
    amb = None
    if isinstance(y_ref, tuple):
        y_ref, amb = y_ref
    rows = valid_row_mask(case)
    g, r = y_gpu[rows], y_ref[rows]
    assert np.isfinite(g).all(), "non-finite output in a valid row"
    err = np.abs(g - r)
    if err.size:
        note = ""
        if amb is not None:   # allowed rounding flips of ambiguous codes
            a = amb[rows]
            adj = np.maximum(err - a, 0.0)
            note = f" (allowance max {a.max():.3e}, error less allowance {adj.max():.3e})"
            assert adj.max() <= atol_max, f"max abs err less allowance {adj.max():.3e}{note}"
        assert err.max() <= atol_max, f"raw max abs err {err.max():.3e} > {atol_max}{note}"
        assert err.mean() <= atol_mean, f"mean abs err {err.mean():.3e} > {atol_mean}"
    # untouched: invalid rows and the guard bands keep the sentinel bits
    body = raw[GUARD:GUARD + case.q.numel()].reshape(case.q.shape)
    assert (body[~rows] == np.int16(SENTINEL)).all(), "a row outside the sequences was written"
    assert (raw[:GUARD] == np.int16(SENTINEL)).all() and \
        (raw[GUARD + case.q.numel():] == np.int16(SENTINEL)).all(), "guard band overwritten"
    return float(err.max()) if err.size else 0.0


def tree_mask(B, T, N, cache):
    """A mask(gen) callable for W.make_case: speculative-decoding tree masks
    [B, 1, T, N] where draft token i of sequence b sees every cached key
    (cache[b] of them) and, of the T drafts stored right after them, itself
    and its ancestors in a seeded random tree."""
    def draw(gen):
        keep = torch.zeros(B, 1, T, N, dtype=torch.bool)
        for b in range(B):
            parent = [-1] + [int(torch.randint(0, i, (1,), generator=gen)) for i in range(1, T)]
            keep[b, 0, :, :cache[b]] = True
            for i in range(T):
                j = i
                while j >= 0:
                    keep[b, 0, i, cache[b] + j] = True
                    j = parent[j]
        return keep
    return draw

