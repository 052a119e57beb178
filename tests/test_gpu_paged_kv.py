"""Attention over a paged KV cache on the GPU against the oracle
("TensorRT Plugins Guide", AttentionPlugin: the decoder contract's
kv_page_table [N, 2, max_pages_per_sequence] into resident paged pools).

Pages are placed at random positions of pools that hold spare pages and
NaN everywhere no sequence's key lives, K and V with different page lists;
page-table entries past a sequence's last page are -1.  Covers page sizes 32
to 256, both dtypes and head dims, fp8 (E4M3) pools, tree decoding, empty
sequences, identity paging against the linear cache (bit for bit: the same
tiles in the same order), and a page index outside the pools (device status
4, Y untouched)."""
import dataclasses

import numpy as np
import pytest
import torch

from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import workloads as W

from helpers import GUARD, SENTINEL, check, run_gpu, run_oracle, tree_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load(build_if_missing=True)


def _decode(seed, *, D=128, dtype=torch.bfloat16, kv_lens=(0, 1, 63, 64, 65, 700), G=4,
            fp8=False, N=None):
    B = len(kv_lens)
    return W.make_case(f"paged_{seed}", seed, batch=B, q_heads=2 * G, kv_heads=2, head_dim=D,
                       q_lens=[1] * B, kv_lens=list(kv_lens), q_form="packed",
                       kv_form="padded", kv_seq=N or max(kv_lens) + 9, dtype=dtype,
                       causal="lower_right", kv_fp8=W.FP8_KV_SCALES if fp8 else None)


def _parity(case):
    y, raw, st = run_gpu(case)
    assert binding.device_status(st) == 0
    check(case, y, raw, run_oracle(case))


@pytest.mark.parametrize("page_size", [32, 64, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [64, 128])
def test_paged_decode(page_size, dtype, D):
    c = _decode(200 + page_size + D, D=D, dtype=dtype)
    _parity(W.paged(c, page_size, seed=7))


@pytest.mark.parametrize("page_size", [32, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_paged_fp8_pools(page_size, dtype):
    c = _decode(210 + page_size, dtype=dtype, fp8=True, kv_lens=(5, 300, 0, 1024, 97))
    _parity(W.paged(c, page_size, seed=8))


def test_paged_tree_decoding():
    B, T = 3, 8
    cache = [40, 500, 129]
    N = max(cache) + T + 5
    for fp8 in (False, True):
        c = W.make_case("paged_tree", 220, batch=B, q_heads=16, kv_heads=2, head_dim=128,
                        q_lens=[T] * B, kv_lens=[x + T for x in cache], q_form="packed",
                        kv_form="padded", kv_seq=N, dtype=torch.bfloat16,
                        mask=tree_mask(B, T, N, cache),
                        kv_fp8=W.FP8_KV_SCALES if fp8 else None)
        _parity(W.paged(c, 64, seed=9))


def test_long_sequences_split_across_warps():
    c = _decode(230, kv_lens=(4000, 2100, 3333), G=8)
    _parity(W.paged(c, 128, seed=10))


def test_identity_pages_match_the_linear_cache_bit_for_bit():
    ps = 64
    c = _decode(240, kv_lens=(640, 64, 333, 1), N=640)
    B, H, N, D = c.k.shape
    pools = [t.reshape(B, H, N // ps, ps, D).permute(0, 2, 1, 3, 4).reshape(B * N // ps, H, ps, D)
             .contiguous() for t in (c.k, c.v)]
    table = torch.arange(B * N // ps, dtype=torch.int32).reshape(B, 1, N // ps).repeat(1, 2, 1)
    pc = dataclasses.replace(c, k=pools[0], v=pools[1], kv_form=W.PAGED, page_table=table)
    y_lin, _, st1 = run_gpu(c)
    y_pag, _, st2 = run_gpu(pc)
    assert binding.device_status(st1) == 0 and binding.device_status(st2) == 0
    assert np.array_equal(y_lin.view(np.int64), y_pag.view(np.int64))


def test_page_outside_the_pools_sets_status_and_leaves_y_untouched():
    c = W.paged(_decode(250, kv_lens=(100, 200, 50)), 64, seed=11)
    for bad in (-5, c.k.shape[0]):
        t = c.page_table.clone()
        t[1, 1, 2] = bad          # V page of keys 128..191 of sequence 1
        y, raw, st = run_gpu(dataclasses.replace(c, page_table=t))
        assert binding.device_status(st) == 4
        assert (raw == np.int16(SENTINEL)).all()


def test_prefill_shapes_are_unsupported():
    c = W.make_case("paged_prefill", 260, batch=2, q_heads=8, kv_heads=2, head_dim=128,
                    q_lens=[64, 64], kv_lens=[64, 64], dtype=torch.bfloat16,
                    causal="upper_left", kv_seq=64)
    with pytest.raises(binding.RgaError) as e:
        run_gpu(W.paged(c, 64, seed=12))
    assert e.value.code == 2
