"""The debug-checks build (librga_debug.so, selected by RGA_DEBUG_CHECKS=1):
its kernels check every TMA start coordinate and direct global access
against its tensor, skip an access outside and record status 7.

Run the whole GPU suite with RGA_DEBUG_CHECKS=1 to check that no kernel
makes such an access on any of its cases: every parity test asserts device
status 0.  This file checks the mechanism itself with one guarded store, in
bounds and out of bounds (the out-of-bounds store is skipped by the check,
so nothing outside the buffer is touched), and that the ordinary build
refuses the self-test."""
import pytest
import torch

from ragged_gqa_attention_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load(build_if_missing=True)


def test_bounds_check_selftest():
    buf = torch.zeros(8, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if not binding.debug_checks():
        assert binding.selftest_bounds_check(buf, 3, st) == 2   # RGA_ERR_UNSUPPORTED
        return
    assert binding.selftest_bounds_check(buf, 3, st) == 0
    assert binding.device_status(st) == 0
    assert buf.cpu().tolist() == [0, 0, 0, 1, 0, 0, 0, 0]
    for bad in (8, 1 << 20, -1):
        st.zero_()
        assert binding.selftest_bounds_check(buf, bad, st) == 0
        assert binding.device_status(st) == 7                  # RGA_ERR_DEBUG_BOUNDS
    assert buf.cpu().tolist() == [0, 0, 0, 1, 0, 0, 0, 0]
