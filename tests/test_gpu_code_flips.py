"""The quantised codes of P read straight out of the prefill kernel.

TRT_QuantizedAttention ("TensorRT Custom Operator Schemas":
normalization_quantize_to_type, normalization_quantize_scale) quantises the
normalised probabilities before BMM2.  With V equal to the identity on the
first D keys and zero after them, output element (i, d) is s_q times the code
of p[i, d] alone, so the test recovers every code the kernel decided for those
keys (the row's other keys still enter its softmax sum).  The kernel decides
in fp32 and the oracle in fp64, so a code may differ only where the exact
value lies within AMBIGUITY_EPS (relative) of a rounding midpoint: every
differing code must be one the oracle flags, and must differ by exactly one
quantisation step.  The counts are printed (pytest -s) and kept in the
assertion messages.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import workloads as W

from helpers import run_gpu, run_oracle, valid_row_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load(build_if_missing=True)


def _grid_step(x, quant):
    """Quantisation step at the code value x (E4M3FN: 3 mantissa bits,
    subnormal spacing 2^-9; int8: 1)."""
    if quant == "int8":
        return np.ones_like(x)
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -6)))
    return 2.0 ** (e - 3)


@pytest.mark.parametrize("quant", ["fp8", "int8"])
def test_quantized_codes_differ_only_where_ambiguous(quant):
    N, D, H = 4096, 128, 2
    # the quantized workload's form: padded fp16, upper_left, a key-suffix
    # bool mask (here 400 keys), rows of up to 3696 attendable keys
    keep = (torch.arange(N) < N - 400).reshape(1, 1, 1, N)
    c = W.make_case(f"codes_{quant}", 41, batch=1, q_heads=H, kv_heads=H, head_dim=D,
                    q_lens=[N], kv_lens=[N], dtype=torch.float16, causal="upper_left",
                    mask=keep, quant=quant, pass_kv_lengths=False)
    v = torch.zeros_like(c.v)
    v[0, :, :D, :] = torch.eye(D, dtype=v.dtype)
    c = replace(c, v=v)
    y, _, st = run_gpu(c)
    assert binding.device_status(st) == 0
    yref, amb = run_oracle(c)
    sq = float(c.quant_scale)
    rows = valid_row_mask(c)
    # codes: exact from the oracle (one product per element); from the GPU by
    # rounding y / s_q (y holds the code times s_q to 16-bit precision) to
    # the code grid, which recovers it exactly
    ref_codes = yref[rows] / sq
    x = y[rows] / sq
    if quant == "int8":
        gpu_codes = np.rint(x)
    else:
        gpu_codes = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    assert np.isfinite(gpu_codes).all()
    flagged = amb[rows] > 0
    flips = gpu_codes != ref_codes
    msg = (f"{quant}: {int(flips.sum())} codes differ of {ref_codes.size} read "
           f"({int(np.count_nonzero(ref_codes))} nonzero in the oracle); "
           f"{int(flagged.sum())} flagged as ambiguous")
    print(msg)
    assert (~flips | flagged).all(), "a code differs where the oracle saw no ambiguity: " + msg
    diff = np.abs(gpu_codes - ref_codes)[flips]
    lo = np.minimum(np.abs(gpu_codes), np.abs(ref_codes))[flips]
    assert np.allclose(diff, _grid_step(lo, quant)), "a code moved by more than one step: " + msg
