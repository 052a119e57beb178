"""Oracle of the KV cache update op (test infrastructure only; the product
path never imports it).

"TensorRT Custom Operator Schemas", TRT_KVCacheUpdate: a TensorScatter
update of past_cache [B, H, N, D] along axis -2 in "linear" mode.  For every
batch b, the first len_b tokens of b's update are written into the cache at
sequence positions write_indices[b], write_indices[b] + 1, ..., for every
head; Y is the cache after the writes (every other element as in
past_cache).  The update is padded [B, H, N_u, D] or packed [T, H, D] with
cumulative update_lengths [B + 1].

Readings where the section leaves a step open (listed in the design notes):
  - write_indices absent: every batch writes at position 0;
  - padded update without update_lengths: every batch writes all N_u tokens;
    with update_lengths, len_b = update_lengths[b+1] - update_lengths[b];
  - packed update: update_lengths is required; batch b's tokens are rows
    update_lengths[b] .. update_lengths[b+1] - 1 of the update;
  - a window [w_b, w_b + len_b) outside [0, N), negative lengths, or
    lengths that do not fit the update tensor make the call invalid
    (TensorScatter's linear mode requires the window inside the cache).

The op moves values without arithmetic, so this oracle works on the raw
element bits (any element type) and is the definition written out as loops.
"""
from __future__ import annotations

import numpy as np


def _bits(t):
    """numpy view of a tensor's raw element bits (torch or numpy input)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu()
            view = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[t.element_size()]
            return t.contiguous().view(view).numpy()
    except ImportError:
        pass
    return np.asarray(t)


def kv_cache_update(past_cache, update, *, update_form="padded", write_indices=None,
                    update_lengths=None):
    """Y of TRT_KVCacheUpdate as raw element bits (numpy, same shape as
    past_cache).  Raises ValueError for an invalid call."""
    cache = np.array(_bits(past_cache), copy=True)
    upd = _bits(update)
    if cache.ndim != 4:
        raise ValueError("past_cache must be [B, H, N, D]")
    B, H, N, D = cache.shape
    if update_form == "padded":
        if upd.ndim != 4 or upd.shape[0] != B or upd.shape[1] != H or upd.shape[3] != D:
            raise ValueError("padded update must be [B, H, N_u, D]")
        n_u = upd.shape[2]
    elif update_form == "packed":
        if upd.ndim != 3 or upd.shape[1] != H or upd.shape[2] != D:
            raise ValueError("packed update must be [T, H, D]")
        if update_lengths is None:
            raise ValueError("the packed form needs update_lengths")
        n_u = upd.shape[0]
    else:
        raise ValueError(update_form)

    cu = None if update_lengths is None else [int(x) for x in _bits(update_lengths).reshape(-1)]
    if cu is not None:
        if len(cu) != B + 1 or cu[0] != 0:
            raise ValueError("update_lengths must be cumulative [B + 1] from 0")
    w = [0] * B if write_indices is None else [int(x) for x in _bits(write_indices).reshape(-1)]
    if len(w) != B:
        raise ValueError("write_indices must be [B]")

    # lengths and the first update row of every batch
    lens, first = [], []
    for b in range(B):
        n = n_u if cu is None else cu[b + 1] - cu[b]
        if n < 0:
            raise ValueError(f"batch {b}: negative update length")
        if update_form == "padded" and n > n_u:
            raise ValueError(f"batch {b}: {n} tokens in a padded update of {n_u}")
        if update_form == "packed" and cu[b + 1] > n_u:
            raise ValueError(f"batch {b}: update rows past the packed update")
        if w[b] < 0 or w[b] + n > N:
            raise ValueError(f"batch {b}: window [{w[b]}, {w[b] + n}) outside the cache")
        lens.append(n)
        first.append(0 if cu is None or update_form == "padded" else cu[b])

    for b in range(B):
        for t in range(lens[b]):
            for h in range(H):
                if update_form == "padded":
                    cache[b, h, w[b] + t, :] = upd[b, h, t, :]
                else:
                    cache[b, h, w[b] + t, :] = upd[first[b] + t, h, :]
    return cache
