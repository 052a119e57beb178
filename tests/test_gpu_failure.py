"""The failure path of the bounded waits on the GPU, without a fault: a wait
that nothing completes gives up after its limit and reports RGA_ERR_TIMEOUT
through the device status word, and the context keeps working."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_timed_out_wait_sets_status_and_context_survives():
    lib = binding.load(build_if_missing=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # about a millisecond of clock cycles: the wait runs out and returns
    rc = lib.rga_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()), 2_000_000, stream)
    assert rc == 0
    assert binding.device_status(status) == 5
    # the same context still computes attention correctly afterwards
    c = W.make_case("after_timeout", 40, batch=2, q_heads=8, kv_heads=2, head_dim=128,
                    q_lens=[70, 33], kv_lens=[70, 33], q_form="packed", kv_form="packed",
                    dtype=torch.bfloat16, causal="upper_left")
    dc = W.to_device(c, "cuda")
    y, st = binding.trt_attention(dc.q, dc.k, dc.v, q_form=dc.q_form, kv_form=dc.kv_form,
                                  query_lengths=dc.query_lengths, kv_lengths=dc.kv_lengths,
                                  scale=dc.scale, causal=dc.causal, return_status=True)
    torch.cuda.synchronize()
    assert binding.device_status(st) == 0
    ref = oracle.attention(c.q, c.k, c.v, q_form=c.q_form, kv_form=c.kv_form,
                           query_lengths=c.query_lengths, kv_lengths=c.kv_lengths,
                           scale=c.scale, causal=c.causal)
    assert np.abs(y.double().cpu().numpy() - ref).max() <= 1e-2
