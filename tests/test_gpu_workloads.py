"""The named workloads (2 to 10) at full size, run on the GPU exactly as the
benchmark launches them; the oracle checks sampled (batch, KV head) pairs
(each one a complete sub-problem it can finish in seconds), and every row
outside the sequences is checked for its sentinel bits."""
import numpy as np
import pytest
import torch

import oracle
from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import workloads as W

from helpers import AMBIGUITY_EPS, GUARD, SENTINEL, TOL, run_gpu, valid_row_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load(build_if_missing=True)


def sub_problem(c: W.Case, b: int, g: int):
    """Oracle inputs for sequence b and KV head g alone (layout slicing only)."""
    G = c.q_heads // c.kv_heads
    hs = slice(g * G, (g + 1) * G)
    ql, kl = c.q_lens[b], c.kv_lens[b]
    if c.q_form == W.PACKED:
        qo = int(c.query_lengths[b])
        q = c.q[qo:qo + ql, hs]
        qlen = torch.tensor([0, ql], dtype=torch.int32)
    else:
        q = c.q[b:b + 1, hs]
        qlen = torch.tensor([0, ql], dtype=torch.int32)
    kv_form = c.kv_form
    if c.kv_form == W.PACKED:
        ko = int(c.kv_lengths[b])
        k, v = c.k[ko:ko + kl, g:g + 1], c.v[ko:ko + kl, g:g + 1]
        klen = torch.tensor([0, kl], dtype=torch.int32)
    elif c.kv_form == W.PAGED:   # sequence b's pages gathered into a linear cache
        t = c.page_table[b:b + 1]
        k = oracle.gather_pages(c.k, t, 0, [kl])[:, g:g + 1]
        v = oracle.gather_pages(c.v, t, 1, [kl])[:, g:g + 1]
        klen = torch.tensor([kl], dtype=torch.int32)
        kv_form = W.PADDED
    else:
        k, v = c.k[b:b + 1, g:g + 1], c.v[b:b + 1, g:g + 1]
        klen = torch.tensor([kl], dtype=torch.int32)
    mask = c.mask
    if mask is not None:
        m = mask.reshape((1,) * (4 - mask.dim()) + tuple(mask.shape))
        m = m[b:b + 1] if m.shape[0] > 1 else m
        m = m[:, hs] if m.shape[1] > 1 else m
        mask = m
    return oracle.attention(q, k, v, q_form=c.q_form, kv_form=kv_form, query_lengths=qlen,
                            kv_lengths=klen, mask=mask, scale=c.scale, causal=c.causal,
                            norm=c.norm, quant=c.quant, quant_scale=c.quant_scale,
                            ambiguity_eps=AMBIGUITY_EPS if c.quant else None,
                            kv_fp8_scales=c.kv_scales)


def gpu_rows(c: W.Case, y, b, g):
    G = c.q_heads // c.kv_heads
    hs = slice(g * G, (g + 1) * G)
    ql = c.q_lens[b]
    if c.q_form == W.PACKED:
        qo = int(c.query_lengths[b])
        return y[qo:qo + ql, hs]
    return y[b:b + 1, hs, :ql]


def ref_rows(c: W.Case, yref, b):
    if c.q_form == W.PACKED:
        return yref
    return yref[:, :, :c.q_lens[b]]


CASES = [(2, None), (3, None), (4, None), (5, "fp8"), (5, "int8"), (6, None), (7, None), (8, None),
         (9, None), (10, None)]


@pytest.mark.parametrize("index,quant", CASES, ids=[f"w{i}-{q}" for i, q in CASES])
def test_workload_full_size_sampled(index, quant):
    c = W.workload(index, quant=quant or "fp8")
    y, raw, st = run_gpu(c)
    assert binding.device_status(st) == 0
    rows = valid_row_mask(c)
    assert np.isfinite(y[rows]).all()
    body = raw[GUARD:GUARD + c.q.numel()].reshape(c.q.shape)
    assert (body[~rows] == np.int16(SENTINEL)).all()
    rng = np.random.default_rng(index)
    # the longest and the shortest sequence, plus a random one
    order = np.argsort(c.q_lens)
    picks = {int(order[0]), int(order[-1]), int(rng.integers(c.batch))}
    amax, amean = TOL[c.quant]
    errs = []
    for b in sorted(picks):
        g = int(rng.integers(c.kv_heads))
        yref = sub_problem(c, b, g)
        amb = None
        if isinstance(yref, tuple):
            yref, amb = yref
        got = gpu_rows(c, y, b, g)
        err = np.abs(got - ref_rows(c, yref, b))
        note = ""
        if amb is not None:
            # quantized P: the error less the allowance for codes within
            # AMBIGUITY_EPS of a rounding midpoint meets the bar, and so does
            # the raw error with no allowance
            a = ref_rows(c, amb, b)
            adj = np.maximum(err - a, 0.0)
            note = f"allowance max {a.max():.3e}, error less allowance {adj.max():.3e}"
            assert adj.max() <= amax, (b, g, note)
        errs.append(err)
        assert err.max() <= amax, (b, g, f"raw max abs err {err.max():.3e}", note)
    allerr = np.concatenate([e.ravel() for e in errs])
    assert allerr.mean() <= amean
