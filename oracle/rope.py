"""Oracle of the rotary position embedding (test infrastructure only; the
product path never imports it).

"TensorRT Plugins Guide", AttentionPlugin: the plugin handles rotary
positional encoding; its decoder contract passes RopeCosSin token-aligned
with the physical rows and marks padding rows with position -1.  Reading
taken (the pages give neither the pairing nor the table layout): row t of
the table holds the cosines of the R/2 rotary angles, then their sines
(R = rotary_dim); element i < R/2 of a head vector pairs with i + R/2 and
the pair turns by the angle:

    x'[i]       = x[i] cos - x[i + R/2] sin
    x'[i + R/2] = x[i + R/2] cos + x[i] sin

Dims R..D-1 and rows with a negative position stay as they are.  Computed in
fp64 from the stored element values and the stored fp32 table.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.array(x, dtype=np.float64)


def rope(x, cos_sin, positions=None):
    """fp64 rotated copy of packed rows x [T, H, D] with table cos_sin [T, R]."""
    X = _f64(x)
    CS = _f64(cos_sin)
    T, H, D = X.shape
    R = CS.shape[1]
    assert CS.shape[0] == T and R % 2 == 0 and R <= D
    h = R // 2
    pos = None if positions is None else [int(p) for p in _f64(positions).reshape(-1)]
    Y = X.copy()
    for t in range(T):
        if pos is not None and pos[t] < 0:
            continue
        c, s = CS[t, :h], CS[t, h:]
        a, b = X[t, :, :h], X[t, :, h:R]
        Y[t, :, :h] = a * c - b * s
        Y[t, :, h:R] = b * c + a * s
    return Y
