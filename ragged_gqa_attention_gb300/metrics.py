"""Algorithmic work of one attention call, for throughput and roofline
numbers: FLOPs = 4 * D * (attendable (query, key) pairs), counting causal,
length and bool-mask exclusions exactly (an additive mask counts every
in-length pair); decode bytes = K and V over the valid rows plus Q and Y.
"""
from __future__ import annotations

import numpy as np

from .workloads import PACKED, Case


def _allowed_per_row(case: Case, b: int) -> np.ndarray:
    """Number of keys each query row of sequence b may attend (int64 [q_len])."""
    ql, kl = case.q_lens[b], case.kv_lens[b]
    i = np.arange(ql, dtype=np.int64)
    if case.causal == "upper_left":
        lim = i + 1
    elif case.causal == "lower_right":
        lim = i + 1 + kl - ql
    else:
        lim = np.full(ql, kl, dtype=np.int64)
    return np.clip(lim, 0, kl)


def attendable_pairs(case: Case) -> int:
    """Sum over batches, query heads and rows of the attendable keys."""
    H = case.q_heads
    total = 0
    m = None
    if case.mask is not None and case.mask.dtype.is_floating_point is False:
        m = case.mask.cpu().numpy()
        m = m.reshape((1,) * (4 - m.ndim) + m.shape)
    for b in range(case.batch):
        ql, kl = case.q_lens[b], case.kv_lens[b]
        if ql == 0 or kl == 0:
            continue
        lim = _allowed_per_row(case, b)
        if m is None:
            total += H * int(lim.sum())
            continue
        mb = m[b if m.shape[0] > 1 else 0]
        keys = np.arange(kl)
        causal_ok = keys[None, :] < lim[:, None]                      # [ql, kl]
        for h in range(H):
            mh = mb[h if mb.shape[0] > 1 else 0]
            mq = mh[:ql] if mh.shape[0] > 1 else np.broadcast_to(mh, (ql, mh.shape[1]))
            mk = mq[:, :kl] if mq.shape[1] > 1 else np.broadcast_to(mq, (ql, kl))
            total += int((causal_ok & mk.astype(bool)).sum())
    return total


def flops(case: Case) -> float:
    return 4.0 * case.head_dim * attendable_pairs(case)


def decode_bytes(case: Case) -> float:
    """K and V bytes over the valid key rows (one byte per element for an
    fp8 KV cache), plus Q and Y."""
    kv = 2 * sum(case.kv_lens) * case.kv_heads * case.head_dim * case.k.element_size()
    rows = sum(case.q_lens) * case.q_heads * case.head_dim * case.q.element_size()
    return float(kv + 2 * rows)


def input_bytes(case: Case):
    """Host->device bytes of one call's inputs (Q, K, V, lengths, mask, scale)."""
    n = 0
    for t in (case.q, case.k, case.v, case.query_lengths, case.kv_lengths, case.mask,
              case.quant_scale, case.page_table, *(case.kv_scales or ())):
        if t is not None:
            n += t.numel() * t.element_size()
    return n


def is_decode(case: Case) -> bool:
    """Short query rows per sequence (at most 16 tokens on average, as in
    vanilla and tree decoding): the work is bound by reading K and V, and
    is reported in GB/s of decode_bytes."""
    return case.q_form == PACKED and case.q.shape[0] <= 16 * case.batch
