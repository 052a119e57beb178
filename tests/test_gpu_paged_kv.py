"""Attention over a paged KV cache on the GPU against the oracle
("TensorRT Plugins Guide", AttentionPlugin: the decoder contract's
kv_page_table [N, 2, max_pages_per_sequence] into resident paged pools).

Pages are placed at random positions of pools that hold spare pages and
NaN everywhere no sequence's key lives, K and V with different page lists;
page-table entries past a sequence's last page are -1.  Covers page sizes 32
to 256, both dtypes and head dims, fp8 (E4M3) pools, tree decoding, empty
sequences, identity paging against the linear cache (bit for bit: the same
tiles in the same order), and a page index outside the pools (device status
4, Y untouched).  Chunked-prefill shapes run on the prefill kernel with page
sizes 32 to 256 (96 included: tiles that straddle pages), 16-bit and fp8
pools, and the same identity and bad-page checks."""
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


# --------------------------------------------------------------------------
# prefill and chunked-prefill shapes: the prefill kernel loads each 128-key
# tile as boxes of pf_page_rows(page_size) rows, one page each
# --------------------------------------------------------------------------
# Chunks of a longer context (every row attends at least 64 keys), as the
# prefill of a paged cache sees them.  (Rows that attend one or two keys
# return about one V row, |y| up to ~3.5, where bf16 output rounding alone
# reaches 7.8e-3 of the 1e-2 bar; the linear-cache tests and the
# self-attention case below cover such rows.)
def _chunked(seed, *, D=128, dtype=torch.bfloat16, fp8=False, G=4,
             q_lens=(100, 257, 1, 64, 130), kv_lens=(612, 321, 300, 128, 1000), causal="lower_right",
             kv_seq=None):
    B = len(q_lens)
    return W.make_case(f"paged_prefill_{seed}", seed, batch=B, q_heads=2 * G, kv_heads=2,
                       head_dim=D, q_lens=list(q_lens), kv_lens=list(kv_lens), q_form="packed",
                       kv_form="padded", kv_seq=kv_seq or max(kv_lens) + 40, dtype=dtype,
                       causal=causal,
                       kv_fp8=W.FP8_KV_SCALES if fp8 else None)


@pytest.mark.parametrize("page_size", [32, 64, 96, 128, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_paged_chunked_prefill(page_size, dtype):
    _parity(W.paged(_chunked(270 + page_size, dtype=dtype), page_size, seed=13))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("page_size", [64, 128])
def test_paged_prefill_fp8_pools(D, page_size):
    _parity(W.paged(_chunked(280 + D + page_size, D=D, fp8=True), page_size, seed=14))


def test_paged_prefill_self_attention():
    c = _chunked(290, q_lens=(300, 77, 129), kv_lens=(300, 77, 129), causal="upper_left", G=8)
    _parity(W.paged(c, 64, seed=15))


def test_paged_prefill_identity_pages_match_the_linear_cache_bit_for_bit():
    ps = 64
    c = _chunked(295, q_lens=(100, 64, 300), kv_lens=(640, 64, 333), kv_seq=640)
    B, H, N, D = c.k.shape
    assert N % ps == 0
    pools = [t.reshape(B, H, N // ps, ps, D).permute(0, 2, 1, 3, 4).reshape(B * N // ps, H, ps, D)
             .contiguous() for t in (c.k, c.v)]
    table = torch.arange(B * N // ps, dtype=torch.int32).reshape(B, 1, N // ps).repeat(1, 2, 1)
    pc = dataclasses.replace(c, k=pools[0], v=pools[1], kv_form=W.PAGED, page_table=table)
    y_lin, _, st1 = run_gpu(c)
    y_pag, _, st2 = run_gpu(pc)
    assert binding.device_status(st1) == 0 and binding.device_status(st2) == 0
    assert np.array_equal(y_lin.view(np.int64), y_pag.view(np.int64))


def test_paged_prefill_page_outside_the_pools_sets_status():
    c = W.paged(_chunked(297), 64, seed=16)
    for bad in (-1, c.k.shape[0]):
        t = c.page_table.clone()
        t[4, 0, 9] = bad          # K page of keys 576..639 of sequence 4 (1000 keys)
        y, raw, st = run_gpu(dataclasses.replace(c, page_table=t))
        assert binding.device_status(st) == 4
        assert (raw == np.int16(SENTINEL)).all()
