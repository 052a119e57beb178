"""Attention over an FP8 (E4M3) KV cache on the GPU against the oracle
("TensorRT Plugins Guide", AttentionPlugin: kv_cache_type FP8).

Covers the decode kernel's in-register E4M3 conversion for all 256 codes;
vanilla decoding in both KV forms, both Q forms, both dtypes, both head dims
and both normalisations, with empty, one-key and ragged key ranges and NaN
codes in every padding row; GQA group sizes 1, 4 and 16; long key ranges
that the stream-K split cuts across warps; tree decoding with a bool mask;
agreement with the 16-bit path on a cache whose dequantised values are
exactly bf16.  Prefill and chunked-prefill shapes run on the prefill kernel:
both Q and KV forms, every causal kind, masks, 'none', GQA group sizes 1 to
16, and bit-for-bit agreement with the 16-bit prefill on exact values."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import workloads as W

from helpers import TOL, check, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load(build_if_missing=True)


def test_e4m3_conversion_all_codes():
    f16, bf16 = binding.selftest_e4m3_decode()
    torch.cuda.synchronize()
    f = f16.cpu().view(torch.float16).double().numpy()
    b = bf16.cpu().view(torch.bfloat16).double().numpy()
    for c in range(256):
        want = oracle.e4m3_decode(c)
        if math.isnan(want):     # NaN codes: NaN as f16; the bf16 form is never used
            assert math.isnan(f[c]), c
            continue
        assert f[c] == want and np.signbit(f[c]) == np.signbit(want), (c, f[c], want)
        assert b[c] == want and np.signbit(b[c]) == np.signbit(want), (c, b[c], want)


def _decode_case(seed, *, B=5, Hq=8, Hkv=2, D=128, kv_lens=(0, 1, 31, 33, 200),
                 q_form="packed", kv_form="padded", dtype=torch.bfloat16, norm="softmax",
                 causal="lower_right", kv_seq=None, scales=W.FP8_KV_SCALES):
    kv_lens = list(kv_lens)
    kw = dict(q_seq=1) if q_form == "padded" else {}
    if kv_form == "padded":
        kw["kv_seq"] = kv_seq or max(kv_lens) + 17
    else:
        kw["tail"] = 5
    # 'none' keeps the unnormalised sums: a small score scale keeps them
    # O(1), where the output dtype's rounding stays inside the tolerance
    return W.make_case(f"fp8kv_{seed}", seed, batch=B, q_heads=Hq, kv_heads=Hkv, head_dim=D,
                       q_lens=[1] * B, kv_lens=kv_lens, q_form=q_form, kv_form=kv_form,
                       dtype=dtype, norm=norm, causal=causal, kv_fp8=scales,
                       scale=0.005 if norm == "none" else None, **kw)


def _parity(case):
    y, raw, st = run_gpu(case)
    assert binding.device_status(st) == 0
    check(case, y, raw, run_oracle(case))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("kv_form", ["padded", "packed"])
@pytest.mark.parametrize("norm", ["softmax", "none"])
def test_vanilla_decode(D, dtype, kv_form, norm):
    seed = 100 + D + (dtype == torch.bfloat16) * 3 + (kv_form == "packed") * 5 + (norm == "none")
    _parity(_decode_case(seed, D=D, dtype=dtype, kv_form=kv_form, norm=norm))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_padded_query(dtype):
    _parity(_decode_case(120, q_form="padded", dtype=dtype, kv_lens=(7, 64, 129, 0, 1)))


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (32, 2)])
def test_group_sizes(Hq, Hkv):
    _parity(_decode_case(130 + Hq, Hq=Hq, Hkv=Hkv, kv_lens=(95, 3, 160, 32, 250)))


@pytest.mark.parametrize("D", [64, 128])
def test_long_ranges_split_across_warps(D):
    # few pairs with many key tiles: the stream-K ranges cut every pair
    _parity(_decode_case(140 + D, B=3, D=D, kv_lens=(3000, 1111, 2049), kv_form="padded"))


def test_tree_decoding_mask():
    from helpers import tree_mask
    B, T = 3, 8
    cache = [40, 257, 100]
    N = max(cache) + T + 3
    for dtype in (torch.float16, torch.bfloat16):
        c = W.make_case("fp8kv_tree", 150, batch=B, q_heads=16, kv_heads=2, head_dim=128,
                        q_lens=[T] * B, kv_lens=[x + T for x in cache], q_form="packed",
                        kv_form="padded", kv_seq=N, dtype=dtype, mask=tree_mask(B, T, N, cache),
                        kv_fp8=W.FP8_KV_SCALES)
        _parity(c)


def test_scales_of_other_magnitudes():
    # tiny and large scales: the dequantised keys and values span a wide range
    _parity(_decode_case(160, scales=(1.0 / 448.0, 3.0), kv_lens=(50, 90, 1, 130, 64)))
    _parity(_decode_case(161, scales=(0.25, 1.0 / 1000.0), kv_lens=(50, 90, 1, 130, 64)))


def test_matches_16bit_path_on_exact_values():
    # scales that are powers of two make every dequantised value a bf16
    # value: the 16-bit kernel on those values computes the same attention
    c = _decode_case(170, scales=(1.0 / 64.0, 1.0 / 32.0), kv_lens=(300, 77, 1, 512, 33))
    y8, _, st = run_gpu(c)
    assert binding.device_status(st) == 0
    kd = torch.from_numpy(oracle.dequant_e4m3(c.k, c.kv_scales[0])).to(torch.bfloat16)
    vd = torch.from_numpy(oracle.dequant_e4m3(c.v, c.kv_scales[1])).to(torch.bfloat16)
    c16 = dataclasses.replace(c, k=torch.nan_to_num(kd), v=torch.nan_to_num(vd), kv_scales=None)
    y16, _, st = run_gpu(c16)
    assert binding.device_status(st) == 0
    assert np.abs(y8 - y16).max() <= 4e-3


# --------------------------------------------------------------------------
# prefill and chunked-prefill shapes: the tcgen05 prefill kernel, whose
# converter warps expand each landed tile of codes into 16-bit values
# --------------------------------------------------------------------------
def _prefill_case(seed, *, D=128, dtype=torch.bfloat16, q_form="packed", kv_form="padded",
                  causal="lower_right", norm="softmax", G=4, q_lens=(100, 257, 1, 64, 130),
                  kv_lens=(612, 257, 300, 64, 1000), mask=None, scales=W.FP8_KV_SCALES):
    B = len(q_lens)
    kw = {"kv_seq": max(kv_lens) + 40} if kv_form == "padded" else {"tail": 7}
    return W.make_case(f"fp8kv_prefill_{seed}", seed, batch=B, q_heads=2 * G, kv_heads=2,
                       head_dim=D, q_lens=list(q_lens), kv_lens=list(kv_lens), q_form=q_form,
                       kv_form=kv_form, dtype=dtype, causal=causal, norm=norm, mask=mask,
                       # 'none' sums s * v over up to 1000 keys unnormalised: a small
                       # score scale keeps |y| below 4, where bf16 output rounding
                       # stays inside the tolerance
                       kv_fp8=scales, scale=0.002 if norm == "none" else None,
                       pass_query_lengths=True, **kw)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("kv_form", ["padded", "packed"])
def test_chunked_prefill(D, dtype, kv_form):
    seed = 300 + D + (dtype == torch.bfloat16) * 3 + (kv_form == "packed") * 5
    _parity(_prefill_case(seed, D=D, dtype=dtype, kv_form=kv_form))


@pytest.mark.parametrize("causal", ["none", "upper_left"])
@pytest.mark.parametrize("q_form", ["packed", "padded"])
def test_prefill_causal_kinds_and_forms(causal, q_form):
    q_lens = (130, 64, 300) if causal == "upper_left" else (100, 17, 300)
    kv_lens = (130, 64, 300) if causal == "upper_left" else (50, 400, 129)
    _parity(_prefill_case(320 + len(causal) + len(q_form), q_form=q_form, causal=causal,
                          q_lens=q_lens, kv_lens=kv_lens))


@pytest.mark.parametrize("G", [1, 8, 16])
def test_prefill_group_sizes(G):
    _parity(_prefill_case(340 + G, G=G, q_lens=(70, 200), kv_lens=(333, 200)))


def test_prefill_none_and_masks():
    _parity(_prefill_case(350, norm="none", causal="none", q_lens=(90, 140), kv_lens=(300, 140)))
    B, N = 2, 340   # the mask's key dim is the padded cache's extent (300 + 40)
    _parity(_prefill_case(351, causal="none", q_lens=(90, 140), kv_lens=(300, 140),
                          mask=lambda g: torch.rand((B, 1, 140, N), generator=g) > 0.3))
    _parity(_prefill_case(352, causal="none", q_lens=(90, 140), kv_lens=(300, 140),
                          mask=lambda g: torch.randn((B, 8, 140, N), generator=g)))


def test_prefill_scales_of_other_magnitudes():
    _parity(_prefill_case(360, scales=(1.0 / 448.0, 3.0)))
    _parity(_prefill_case(361, scales=(0.25, 1.0 / 1000.0)))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_prefill_matches_16bit_path_on_exact_values(dtype):
    """Power-of-two scales make every dequantised value a 16-bit value, and
    scaling by a power of two commutes with every rounding on the way.  With
    f16 queries the prefill kernel over the codes computes exactly what it
    computes over the dequantised 16-bit cache (bit for bit).  With bf16
    queries the softmax's products run in f16 over a cache of codes (Q
    scaled by a power of two, P rounded to f16 rather than bf16), so the two
    agree to P's rounding."""
    c = _prefill_case(370, dtype=dtype, scales=(1.0 / 64.0, 1.0 / 32.0))
    y8, _, st = run_gpu(c)
    assert binding.device_status(st) == 0
    kd = torch.from_numpy(oracle.dequant_e4m3(c.k, c.kv_scales[0])).to(dtype)
    vd = torch.from_numpy(oracle.dequant_e4m3(c.v, c.kv_scales[1])).to(dtype)
    c16 = dataclasses.replace(c, k=torch.nan_to_num(kd), v=torch.nan_to_num(vd), kv_scales=None)
    y16, _, st = run_gpu(c16)
    assert binding.device_status(st) == 0
    rows = np.isfinite(y16)
    assert np.array_equal(np.isfinite(y8), rows)
    if dtype == torch.float16:
        assert np.array_equal(y8[rows], y16[rows])
    else:   # P's rounding, and one bf16 ulp of the output where it falls differently
        d = np.abs(y8[rows] - y16[rows])
        assert (d <= 4e-3 + 2.0 ** -7 * np.abs(y16[rows])).all(), d.max()
