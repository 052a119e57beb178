"""trt_attention_static_scratch: the entry point for callers that cannot
allocate device memory (it uses a scratch array inside the library instead
of a caller-provided workspace).  Called through the C ABI, twice in a row,
and compared with trt_attention on the same inputs.

This file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import workloads as W

from helpers import TOL

pytestmark = pytest.mark.gpu

CASES = {
    # split-KV decode: uses the scratch for split partials and tickets
    "decode": dict(batch=8, q_heads=32, kv_heads=4, head_dim=128, q_lens=[1] * 8,
                   kv_lens=[1, 40, 600, 1500, 2100, 3000, 64, 999], q_form="packed",
                   kv_form="padded", kv_seq=3000, dtype=torch.bfloat16, causal="lower_right"),
    # prefill: uses the scratch for the scheduler's work list
    "prefill": dict(batch=3, q_heads=8, kv_heads=2, head_dim=128, q_lens=[300, 17, 129],
                    kv_lens=[300, 17, 129], q_form="packed", kv_form="packed",
                    dtype=torch.float16, causal="upper_left"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_scratch_matches_trt_attention(name):
    lib = binding.load(build_if_missing=True)
    c = W.to_device(W.make_case(name, 31, **CASES[name]), "cuda")
    kw = dict(q_form=c.q_form, kv_form=c.kv_form, query_lengths=c.query_lengths,
              kv_lengths=c.kv_lengths, scale=c.scale, causal=c.causal)
    ref = binding.trt_attention(c.q, c.k, c.v, **kw)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    for call in range(2):
        y = torch.full_like(c.q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        a = binding.make_args(c.q, c.k, c.v, y, status=status, **kw)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = lib.trt_attention_static_scratch(ctypes.byref(a),
                                              ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, binding.STATUS_NAMES.get(rc, rc)
        torch.cuda.synchronize()
        if call == 1:
            # the first call may load the library's modules on this device;
            # after that a call takes no device memory at all
            assert torch.cuda.mem_get_info()[0] == free_before, "the call allocated device memory"
        assert int(status.item()) == 0
        rows = torch.isfinite(ref)
        assert torch.equal(torch.isfinite(y), rows), f"call {call}: written rows differ"
        err = (y[rows].double() - ref[rows].double()).abs().max().item()
        assert err <= TOL[None][0], f"call {call}: max abs err {err}"


def test_static_scratch_rejects_oversized_problems():
    lib = binding.load(build_if_missing=True)
    # prefill over 50000 packed sequences x 64 KV heads: the work list has room
    # for 64 * (1 + 50000) items of 16 bytes (51 MB), more than the 40 MiB
    # scratch; the sequences are empty, so the tensors stay tiny
    B, H, D = 50000, 64, 64
    q = torch.zeros(64, H, D, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(1, H, D, dtype=torch.bfloat16, device="cuda")
    y = torch.full_like(q, float("nan"))
    lens = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = binding.make_args(q, kv, kv, y, q_form="packed", kv_form="packed",
                          query_lengths=lens, kv_lengths=lens, status=status)
    assert lib.rga_attention_workspace_size(ctypes.byref(a)) > (40 << 20)
    rc = lib.trt_attention_static_scratch(ctypes.byref(a), None)
    assert rc == 6
    torch.cuda.synchronize()
    assert torch.isnan(y).all()   # nothing ran
