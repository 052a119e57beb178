"""Pins of the TRT_KVCacheUpdate oracle ("TensorRT Custom Operator Schemas",
TRT_KVCacheUpdate) against hand-derived cases and properties the section
fixes, independent of the oracle's own loops."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_update_cases.json")


def rule_cache(shape):
    B, H, N, D = shape
    b, h, n, d = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), np.arange(D), indexing="ij")
    return (1000 * b + 100 * h + 10 * n + d).astype(np.int16)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_golden(case):
    cache = rule_cache(case["shape"])
    upd = np.array(case["update"], dtype=np.int16)
    lens = None if case["update_lengths"] is None else np.array(case["update_lengths"], np.int32)
    wi = None if case["write_indices"] is None else np.array(case["write_indices"], np.int32)
    if case.get("invalid"):
        with pytest.raises(ValueError):
            oracle.kv_cache_update(cache, upd, update_form=case["update_form"], write_indices=wi,
                                   update_lengths=lens)
        return
    y = oracle.kv_cache_update(cache, upd, update_form=case["update_form"], write_indices=wi,
                               update_lengths=lens)
    touched = np.zeros(cache.shape[:3], dtype=bool)
    for b, h, n, row in case["expected_rows"]:
        assert y[b, h, n].tolist() == row
        touched[b, h, n] = True
    assert np.array_equal(y[~touched], cache[~touched])


def _random(seed, B=3, H=2, N=9, D=4, n_u=4):
    g = np.random.default_rng(seed)
    cache = g.integers(-30000, 30000, (B, H, N, D), dtype=np.int16)
    upd = g.integers(-30000, 30000, (B, H, n_u, D), dtype=np.int16)
    lens = g.integers(0, n_u + 1, B)
    wi = np.array([g.integers(0, N - l + 1) for l in lens], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return cache, upd, lens, wi, cu


def test_zero_lengths_leave_the_cache_unchanged():
    cache, upd, _, wi, _ = _random(1)
    cu = np.zeros(cache.shape[0] + 1, np.int32)
    y = oracle.kv_cache_update(cache, upd, write_indices=wi, update_lengths=cu)
    assert np.array_equal(y, cache)


@pytest.mark.parametrize("seed", range(5))
def test_padded_equals_packed(seed):
    cache, upd, lens, wi, cu = _random(seed)
    packed = np.concatenate([upd[b, :, :lens[b]].transpose(1, 0, 2) for b in range(len(lens))], 0)
    y_pad = oracle.kv_cache_update(cache, upd, write_indices=wi, update_lengths=cu)
    y_pck = oracle.kv_cache_update(cache, packed, update_form="packed", write_indices=wi,
                                   update_lengths=cu)
    assert np.array_equal(y_pad, y_pck)


@pytest.mark.parametrize("seed", range(5))
def test_windows_hold_the_update_and_the_rest_is_untouched(seed):
    cache, upd, lens, wi, cu = _random(seed)
    y = oracle.kv_cache_update(cache, upd, write_indices=wi, update_lengths=cu)
    for b in range(len(lens)):
        sl = slice(wi[b], wi[b] + lens[b])
        assert np.array_equal(y[b, :, sl], upd[b, :, :lens[b]])
        keep = np.ones(cache.shape[2], bool)
        keep[sl] = False
        assert np.array_equal(y[b, :, keep], cache[b, :, keep])


def test_disjoint_updates_commute():
    cache, upd, _, _, _ = _random(7, B=1, N=12, n_u=3)
    a = dict(write_indices=np.array([0], np.int32), update_lengths=np.array([0, 3], np.int32))
    b = dict(write_indices=np.array([6], np.int32), update_lengths=np.array([0, 2], np.int32))
    ab = oracle.kv_cache_update(oracle.kv_cache_update(cache, upd, **a), upd[:, :, ::-1], **b)
    ba = oracle.kv_cache_update(oracle.kv_cache_update(cache, upd[:, :, ::-1], **b), upd, **a)
    assert np.array_equal(ab, ba)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_moves_bits_for_every_element_width(dtype):
    g = torch.Generator().manual_seed(3)
    cache = torch.randn(2, 2, 5, 8, generator=g).to(dtype)
    upd = torch.randn(3, 2, 8, generator=g).to(dtype)
    cu = torch.tensor([0, 1, 3], dtype=torch.int32)
    wi = torch.tensor([4, 1], dtype=torch.int32)
    y = oracle.kv_cache_update(cache, upd, update_form="packed", write_indices=wi, update_lengths=cu)
    want = cache.clone()
    want[0, :, 4] = upd[0]
    want[1, :, 1] = upd[1]
    want[1, :, 2] = upd[2]
    view = {2: torch.int16, 4: torch.int32}[cache.element_size()]
    assert np.array_equal(y, want.view(view).numpy())


@pytest.mark.parametrize("bad", ["negative_index", "past_end", "lengths_past_update", "not_from_zero"])
def test_invalid_calls_raise(bad):
    cache = np.zeros((2, 1, 4, 2), np.int16)
    upd = np.zeros((3, 1, 2), np.int16)
    cu, wi = np.array([0, 1, 3], np.int32), np.array([0, 0], np.int32)
    if bad == "negative_index":
        wi = np.array([-1, 0], np.int32)
    elif bad == "past_end":
        wi = np.array([0, 3], np.int32)
    elif bad == "lengths_past_update":
        cu = np.array([0, 2, 4], np.int32)
    else:
        cu = np.array([1, 2, 3], np.int32)
    with pytest.raises(ValueError):
        oracle.kv_cache_update(cache, upd, update_form="packed", write_indices=wi, update_lengths=cu)
