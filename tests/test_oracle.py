"""Pins for the CPU oracle against facts that do not come from the oracle.

Each test ties one part of the oracle to something fixed outside it: hand
derivations (tests/golden), a library routine on a special case (PyTorch's
scaled_dot_product_attention in fp64, PyTorch's float8_e4m3fn cast), closed
forms and invariants of the definition on the "TensorRT Custom Operator
Schemas" page (TRT_Attention / TRT_QuantizedAttention).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from ragged_gqa_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# Quantisers
# ----------------------------------------------------------------------------
def test_e4m3_decode_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])


def test_e4m3_encode_decode_roundtrip():
    for c in range(256):
        x = oracle.e4m3_decode(c)
        if math.isnan(x):
            continue
        e = oracle.e4m3_encode(x)
        if x == 0:
            assert e in (0x00, 0x80)
        else:
            assert e == c, (c, x, e)


def test_e4m3_round_matches_torch_cast_in_range():
    # dense sweep including every midpoint between neighbouring codes
    vals = [oracle.e4m3_decode(c) for c in range(127)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    rng = np.random.default_rng(0)
    xs = np.concatenate([vals, mids, rng.uniform(0, 448, 20000),
                         rng.uniform(0, 0.05, 5000)])
    xs = np.concatenate([xs, -xs])
    ref = torch.tensor(xs, dtype=torch.float64).to(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_round(x) for x in xs])
    assert np.array_equal(got, ref)


def test_e4m3_midpoints_and_saturation():
    assert oracle.e4m3_round(1.0625) == 1.0      # tie -> even mantissa 0
    assert oracle.e4m3_round(1.1875) == 1.25     # tie -> even mantissa 2
    assert oracle.e4m3_round(2.0 ** -10) == 0.0  # half the smallest subnormal
    assert oracle.e4m3_round(3 * 2.0 ** -10) == 2.0 ** -8
    assert oracle.e4m3_round(464.0) == 448.0     # saturating, no inf
    assert oracle.e4m3_round(1e9) == 448.0
    assert oracle.e4m3_round(-1e9) == -448.0


def test_int8_round_half_even_and_clamp():
    cases = {2.5: 2, 3.5: 4, -2.5: -2, 0.5: 0, 1.5: 2, 127.6: 127,
             126.5: 126, -128.4: -128, -200.0: -128, 1000.0: 127, 41.4999: 41}
    for x, want in cases.items():
        assert oracle.int8_round(x) == want, x


# ----------------------------------------------------------------------------
# Hand-derived golden cases
# ----------------------------------------------------------------------------
def _golden_cases():
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        g = json.load(f)
    return g["common"], g["cases"]


@pytest.mark.parametrize("case", _golden_cases()[1], ids=lambda c: c["name"])
def test_hand_golden(case):
    common, _ = _golden_cases()
    nq = case["nq"]
    q = np.array([common["q_row"]] * nq, dtype=np.float64)[None, None]
    k = np.array(common["k"], dtype=np.float64)[None, None]
    v = np.array(common["v"], dtype=np.float64)[None, None]
    mask = None
    if "bool_mask" in case:
        mask = np.array(case["bool_mask"], dtype=bool)
    if "add_mask" in case:
        mask = np.array(case["add_mask"], dtype=np.float64)
    y = oracle.attention(q, k, v, scale=math.log(2.0), causal=case["causal"],
                         norm=case["norm"], mask=mask, quant=case.get("quant"),
                         quant_scale=case.get("quant_scale"))
    np.testing.assert_allclose(y[0, 0], np.array(case["y"]), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# Library routine on the special cases it covers: PyTorch SDPA in fp64
# (padded MHA, no lengths; upper_left causal = SDPA's is_causal)
# ----------------------------------------------------------------------------
def _rand(shape, seed, dtype=torch.float16):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(dtype)


@pytest.mark.parametrize("causal", ["none", "upper_left"])
@pytest.mark.parametrize("maskkind", [None, "bool", "add"])
def test_matches_torch_sdpa_fp64(causal, maskkind):
    if causal != "none" and maskkind is not None:
        pytest.skip("SDPA takes either a mask or is_causal")
    B, H, N, D = 2, 3, 37, 16
    q, k, v = (_rand((B, H, N, D), s) for s in (1, 2, 3))
    scale = 0.3
    mask = None
    if maskkind == "bool":
        g = torch.Generator().manual_seed(9)
        mask = torch.rand((B, 1, N, N), generator=g) > 0.3
        mask[..., 0] = True   # keep every row non-empty (SDPA gives NaN)
    elif maskkind == "add":
        mask = _rand((1, H, N, N), 10, torch.float32)
    y = oracle.attention(q, k, v, scale=scale, causal=causal, mask=mask)
    ref = F.scaled_dot_product_attention(
        q.double(), k.double(), v.double(),
        attn_mask=None if mask is None else (mask if mask.dtype == torch.bool else mask.double()),
        is_causal=(causal == "upper_left"), scale=scale)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_quantized_matches_library_qdq_path():
    """Q/DQ of the normalised P: torch softmax (fp64) -> torch float8 cast /
    round-half-even int8 -> matmul, against the oracle."""
    B, H, N, D = 1, 2, 40, 8
    q, k, v = (_rand((B, H, N, D), s) for s in (4, 5, 6))
    scale = 0.7
    s = q.double() @ k.double().transpose(-1, -2) * scale
    p = torch.softmax(s, dim=-1)
    for quant, sq in (("fp8", 1 / 448), ("int8", 1 / 127)):
        if quant == "fp8":
            pq = (p / sq).clamp(-448, 448).to(torch.float8_e4m3fn).double() * sq
        else:
            pq = torch.round(p / sq).clamp(-128, 127) * sq
        ref = pq @ v.double()
        y = oracle.attention(q, k, v, scale=scale, quant=quant, quant_scale=sq)
        np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_none_normalization_is_two_matmuls():
    B, H, N, D = 1, 2, 20, 8
    q, k, v = (_rand((B, H, N, D), s) for s in (7, 8, 9))
    ref = (q.double() @ k.double().transpose(-1, -2) * 0.5) @ v.double()
    y = oracle.attention(q, k, v, scale=0.5, norm="none")
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# Invariants and closed forms of the definition
# ----------------------------------------------------------------------------
def _case(**kw):
    base = dict(batch=3, q_heads=4, kv_heads=2, head_dim=8,
                q_lens=[5, 1, 7], kv_lens=[9, 4, 7], dtype=torch.float16,
                pass_query_lengths=True)
    base.update(kw)
    return W.make_case("t", kw.pop("seed", 11), **base)


def _run(c, **over):
    kw = dict(q_form=c.q_form, kv_form=c.kv_form, query_lengths=c.query_lengths,
              kv_lengths=c.kv_lengths, mask=c.mask, scale=c.scale,
              causal=c.causal, norm=c.norm, quant=c.quant,
              quant_scale=c.quant_scale)
    kw.update(over)
    return oracle.attention(c.q, c.k, c.v, **kw)


def _padded_to_packed(x, lens):
    """[B,H,N,D] -> [sum(lens),H,D] (layout only)."""
    return torch.cat([x[b, :, :n].transpose(0, 1) for b, n in enumerate(lens)], 0)


def _packed_rows(y, lens):
    """Split a packed [T,H,D] result into per-batch [H,n,D] arrays."""
    out, o = [], 0
    for n in lens:
        out.append(np.transpose(y[o:o + n], (1, 0, 2)))
        o += n
    return out


@pytest.mark.parametrize("causal", ["none", "upper_left", "lower_right"])
def test_packed_equals_padded(causal):
    # padded Q passes query_lengths, so lower_right sees the true q_len
    c = _case(causal=causal, kv_pad=0.0, pass_query_lengths=True)
    y_pad = _run(c)
    qp = _padded_to_packed(c.q, c.q_lens)
    kp = _padded_to_packed(c.k, c.kv_lens)
    vp = _padded_to_packed(c.v, c.kv_lens)
    ql = torch.tensor(np.cumsum([0] + c.q_lens), dtype=torch.int32)
    kl = torch.tensor(np.cumsum([0] + c.kv_lens), dtype=torch.int32)
    for qf, kf in (("packed", "packed"), ("packed", "padded"), ("padded", "packed")):
        y = oracle.attention(
            qp if qf == "packed" else c.q, kp if kf == "packed" else c.k,
            vp if kf == "packed" else c.v, q_form=qf, kv_form=kf,
            query_lengths=ql,
            kv_lengths=kl if kf == "packed" else c.kv_lengths,
            scale=c.scale, causal=causal)
        rows = _packed_rows(y, c.q_lens) if qf == "packed" else [
            y[b, :, :n] for b, n in enumerate(c.q_lens)]
        for b, n in enumerate(c.q_lens):
            np.testing.assert_allclose(rows[b], y_pad[b, :, :n], rtol=1e-13, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv():
    c = _case(causal="upper_left")
    G = c.q_heads // c.kv_heads
    y = _run(c)
    k2 = c.k.repeat_interleave(G, dim=1)
    v2 = c.v.repeat_interleave(G, dim=1)
    y2 = oracle.attention(c.q, k2, v2, query_lengths=c.query_lengths,
                          kv_lengths=c.kv_lengths, scale=c.scale,
                          causal="upper_left")
    np.testing.assert_array_equal(y, y2)


def test_upper_left_equals_lower_right_when_lengths_match():
    c = _case(q_lens=[6, 3, 8], kv_lens=[6, 3, 8])
    a = _run(c, causal="upper_left")
    b = _run(c, causal="lower_right")
    np.testing.assert_array_equal(a, b)


def test_single_query_lower_right_is_full_attention():
    c = _case(q_lens=[1, 1, 1], kv_lens=[9, 4, 7])
    np.testing.assert_array_equal(_run(c, causal="lower_right"), _run(c, causal="none"))


def test_scale_zero_is_mean_of_allowed_values():
    c = _case(causal="upper_left", q_lens=[5, 4, 7], kv_lens=[9, 4, 7], kv_pad=0.0)
    y = _run(c, scale=0.0)
    v = c.v.double().numpy()
    for b in range(c.batch):
        for h in range(c.q_heads):
            g = h // 2
            for i in range(c.q_lens[b]):
                want = v[b, g, :min(i + 1, c.kv_lens[b])].mean(axis=0)
                np.testing.assert_allclose(y[b, h, i], want, rtol=1e-13, atol=1e-13)


def test_constant_v_returns_v():
    c = _case(causal="lower_right")
    c.v[:] = 0.75
    y = _run(c)
    for b, n in enumerate(c.q_lens):
        np.testing.assert_allclose(y[b, :, :n], 0.75, rtol=1e-13)


def test_rows_sum_to_one_with_identity_values():
    # D >= kv_len and v_j = e_j: y_i[j] = p_ij, so each row sums to 1
    D = 16
    c = _case(head_dim=D, q_lens=[5, 2, 9], kv_lens=[16, 3, 11], causal="upper_left")
    for b in range(c.batch):
        c.v[b] = 0
        for j in range(c.kv_lens[b]):
            c.v[b, :, j, j] = 1
    y = _run(c)
    for b, n in enumerate(c.q_lens):
        rows = y[b, :, :n].sum(-1)
        np.testing.assert_allclose(rows, 1.0, rtol=1e-13)
        assert (y[b, :, :n] >= 0).all()


def test_single_allowed_key_returns_its_value():
    c = _case(causal="upper_left", q_lens=[5, 4, 7], kv_pad=0.0)
    y = _run(c)
    v = c.v.double().numpy()
    for b in range(c.batch):
        for h in range(c.q_heads):
            np.testing.assert_array_equal(y[b, h, 0], v[b, h // 2, 0])


def test_bool_key_suffix_mask_equals_kv_lengths():
    B, N = 3, 12
    m = [0, 3, 5]
    c = _case(q_lens=[N] * B, kv_lens=[N] * B, causal="upper_left")
    keep = torch.arange(N)[None, :] < (N - torch.tensor(m))[:, None]
    a = _run(c, mask=keep.reshape(B, 1, 1, N), kv_lengths=None)
    b = _run(c, kv_lengths=torch.tensor([N - x for x in m], dtype=torch.int32))
    np.testing.assert_array_equal(a, b)


def test_trivial_masks_equal_no_mask():
    c = _case(q_lens=[6, 6, 6], kv_lens=[9, 9, 9])
    base = _run(c)
    np.testing.assert_array_equal(_run(c, mask=np.ones((6, 9), bool)), base)
    np.testing.assert_array_equal(_run(c, mask=np.zeros((1, 1, 6, 9))), base)


def test_additive_minus_inf_equals_bool_false():
    c = _case(q_lens=[6, 6, 6], kv_lens=[9, 9, 9])
    g = np.random.default_rng(3)
    keep = g.random((3, 4, 6, 9)) > 0.4
    keep[..., 0] = True
    add = np.where(keep, 0.0, -np.inf)
    np.testing.assert_array_equal(_run(c, mask=keep), _run(c, mask=add))


def test_empty_rows_are_zero_and_padding_untouched():
    # kv_len 0, lower_right with q_len > kv_len, q_len 0
    c = _case(q_lens=[4, 0, 6], kv_lens=[0, 3, 2], q_seq=6, causal="lower_right",
              pass_query_lengths=True)
    y = _run(c)
    assert (y[0, :, :4] == 0).all()                 # no keys at all
    assert np.isnan(y[0, :, 4:]).all()              # padded rows untouched
    assert np.isnan(y[1]).all()                     # q_len 0: nothing written
    assert (y[2, :, :4] == 0).all()                 # i + 2 - 6 < 0: no key
    assert np.isfinite(y[2, :, 4:]).all()


def test_bad_lengths_rejected():
    c = _case(q_form="packed", kv_form="packed")
    ql = c.query_lengths.clone()
    ql[2] = ql[1] - 1   # non-monotonic
    with pytest.raises(oracle.OracleError) as e:
        _run(c, query_lengths=ql)
    assert e.value.code == 4
    kl = torch.tensor([10, 10, 10], dtype=torch.int32)   # > kv_seq (padded)
    with pytest.raises(oracle.OracleError):
        _run(_case(), kv_lengths=kl)


# ----------------------------------------------------------------------------
# Brute force on 1-4 token inputs, every flag combination, against a direct
# matrix formulation (numpy, whole score matrix at once) written here.
# ----------------------------------------------------------------------------
def _direct(q, k, v, ql, kl, scale, causal, norm, mask, quant, sq):
    """q [Hq,ql,D], k/v [Hkv,kl,D] float64; mask broadcastable to [Hq,ql,kl]."""
    Hq, Hkv = q.shape[0], k.shape[0]
    kk = np.repeat(k, Hq // Hkv, axis=0)
    vv = np.repeat(v, Hq // Hkv, axis=0)
    s = np.einsum("hid,hjd->hij", q, kk) * scale
    i = np.arange(ql)[:, None]
    j = np.arange(kl)[None, :]
    allow = np.ones((ql, kl), bool)
    if causal == "upper_left":
        allow = j - i <= 0
    elif causal == "lower_right":
        allow = j - i <= kl - ql
    allow = np.broadcast_to(allow, s.shape).copy()
    if mask is not None and mask.dtype == bool:
        allow &= np.broadcast_to(mask, s.shape)
    elif mask is not None:
        s = s + mask
    if norm == "softmax":
        z = np.where(allow, s, -np.inf)
        top = z.max(-1, keepdims=True)
        top = np.where(np.isfinite(top), top, 0.0)
        e = np.where(allow, np.exp(z - top), 0.0)
        tot = e.sum(-1, keepdims=True)
        p = np.divide(e, tot, out=np.zeros_like(e), where=tot > 0)
    else:
        p = np.where(allow, s, 0.0)
    if quant == "fp8":
        p = torch.tensor(np.clip(p / sq, -448, 448)).to(torch.float8_e4m3fn).double().numpy() * sq
    elif quant == "int8":
        p = np.clip(np.round(p / sq), -128, 127) * sq
    p = np.where(allow, p, 0.0)
    return p @ vv


@pytest.mark.parametrize("causal", ["none", "upper_left", "lower_right"])
@pytest.mark.parametrize("norm", ["softmax", "none"])
@pytest.mark.parametrize("quant", [None, "fp8", "int8"])
@pytest.mark.parametrize("maskkind", [None, "bool", "add"])
def test_brute_force_tiny(causal, norm, quant, maskkind):
    rng = np.random.default_rng(hash((causal, norm, quant, maskkind)) % 2**32)
    for trial in range(6):
        ql, kl = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        Hkv = int(rng.integers(1, 3))
        Hq = Hkv * int(rng.integers(1, 3))
        D = 4
        q = torch.tensor(rng.standard_normal((1, Hq, ql, D))).half()
        k = torch.tensor(rng.standard_normal((1, Hkv, kl, D))).half()
        v = torch.tensor(rng.standard_normal((1, Hkv, kl, D))).half()
        mask = None
        if maskkind == "bool":
            mask = rng.random((Hq, ql, kl)) > 0.3
        elif maskkind == "add":
            mask = rng.standard_normal((1, ql, kl))
        sq = 1 / 448 if quant == "fp8" else 1 / 127
        y = oracle.attention(q, k, v, scale=0.6, causal=causal, norm=norm,
                             mask=mask, quant=quant, quant_scale=sq)
        want = _direct(q[0].double().numpy(), k[0].double().numpy(),
                       v[0].double().numpy(), ql, kl, 0.6, causal, norm,
                       mask, quant, sq)
        np.testing.assert_allclose(y[0], want, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# Q/DQ ambiguity bound (quantised codes that sit on a rounding midpoint)
# ----------------------------------------------------------------------------
def _one_key(sval, quant, sq):
    q = np.array([[[[1.0, 0.0]]]])
    k = np.array([[[[sval, 0.0]]]])
    v = np.array([[[[3.0, -2.0]]]])
    return oracle.attention(q, k, v, scale=1.0, norm="none", quant=quant, quant_scale=sq,
                            ambiguity_eps=1e-9)


def test_ambiguity_marks_exact_midpoints_only():
    y, amb = _one_key(2.5, "int8", 1.0)            # 2.5 -> 2 (even); could be 3
    np.testing.assert_array_equal(y[0, 0, 0], [6.0, -4.0])
    np.testing.assert_array_equal(amb[0, 0, 0], [3.0, 2.0])   # one step * s * |v|
    y, amb = _one_key(2.3, "int8", 1.0)
    assert (amb == 0).all()
    y, amb = _one_key(1.0625, "fp8", 1.0)          # between 1.0 and 1.125
    np.testing.assert_array_equal(y[0, 0, 0], [3.0, -2.0])
    np.testing.assert_array_equal(amb[0, 0, 0], [0.375, 0.25])
    y, amb = _one_key(1.1, "fp8", 1.0)
    assert (amb == 0).all()


@pytest.mark.parametrize("quant", ["fp8", "int8"])
@pytest.mark.parametrize("norm", ["softmax", "none"])
def test_ambiguity_bounds_perturbed_evaluation(quant, norm):
    """Scores perturbed by a relative 1e-9 (another evaluation order) move the
    output by no more than the bound computed with eps = 1e-8."""
    c = _case(q_lens=[40, 30, 50], kv_lens=[60, 30, 50], causal="upper_left")
    sq = 1 / 448 if quant == "fp8" else 1 / 127
    sc = 0.05 if norm == "none" else c.scale
    y0, amb = _run(c, quant=quant, quant_scale=sq, norm=norm, scale=sc, ambiguity_eps=1e-8)
    for f in (1 + 1e-9, 1 - 1e-9):
        y1 = _run(c, quant=quant, quant_scale=sq, norm=norm, scale=sc * f)
        ok = ~np.isnan(y0)
        assert (np.abs(y1[ok] - y0[ok]) <= amb[ok] + 1e-6).all()


# ----------------------------------------------------------------------------
# FP8 KV cache ("TensorRT Plugins Guide", AttentionPlugin: kv_cache_type FP8):
# dequantisation against PyTorch's float8_e4m3fn decoding, the attention on
# dequantised keys and values against SDPA, and closed forms that tell the K
# scale from the V scale.
# ----------------------------------------------------------------------------
def test_e4m3_dequant_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    for s in (1.0, 1.0 / 56.0, 3.0):
        got = oracle.dequant_e4m3(codes, s)
        ref = codes.view(torch.float8_e4m3fn).double().numpy() * s
        nan = np.isnan(ref)
        assert (np.isnan(got) == nan).all()
        np.testing.assert_array_equal(got[~nan], ref[~nan])
        assert (np.signbit(got[~nan]) == np.signbit(ref[~nan])).all()


def _codes(shape, seed, s):
    return (_rand(shape, seed, torch.float32) / s).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8)


@pytest.mark.parametrize("causal", ["none", "upper_left"])
def test_fp8_kv_matches_torch_sdpa_on_decoded_cache(causal):
    B, H, N, D = 2, 3, 29, 16
    sk, sv = 1.0 / 56.0, 1.0 / 20.0
    q = _rand((B, H, N, D), 11)
    kc, vc = _codes((B, H, N, D), 12, sk), _codes((B, H, N, D), 13, sv)
    y = oracle.attention(q, kc, vc, scale=0.4, causal=causal, kv_fp8_scales=(sk, sv))
    kd = kc.view(torch.float8_e4m3fn).double() * sk
    vd = vc.view(torch.float8_e4m3fn).double() * sv
    ref = F.scaled_dot_product_attention(q.double(), kd, vd, is_causal=(causal == "upper_left"),
                                         scale=0.4)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_fp8_kv_constant_value_code_returns_its_value():
    # every value code 0x3A (1.25): softmax rows average to 1.25 * s_v, for
    # any keys and any K scale
    B, H, N, D = 1, 2, 17, 8
    q = _rand((B, H, N, D), 14)
    kc = _codes((B, H, N, D), 15, 0.05)
    vc = torch.full((B, H, N, D), 0x3A, dtype=torch.uint8)
    y = oracle.attention(q, kc, vc, scale=1.0, kv_fp8_scales=(0.05, 0.375))
    np.testing.assert_allclose(y, 1.25 * 0.375, rtol=1e-13)


def test_fp8_kv_zero_key_codes_give_uniform_weights():
    # all key codes zero: every score is 0 whatever s_k, so each row is the
    # plain mean of the dequantised values (V scale applied, K scale not)
    B, H, N, D = 1, 1, 9, 4
    q = _rand((B, H, N, D), 16)
    kc = torch.zeros((B, H, N, D), dtype=torch.uint8)
    vc = _codes((B, H, N, D), 17, 0.1)
    y = oracle.attention(q, kc, vc, kv_fp8_scales=(123.0, 0.1))
    vd = np.array([[oracle.e4m3_decode(int(c)) for c in row] for row in vc[0, 0]]) * 0.1
    np.testing.assert_allclose(y[0, 0], np.tile(vd.mean(axis=0), (N, 1)), rtol=1e-13)


# ----------------------------------------------------------------------------
# Paged KV cache: the gather that turns pools + page table into the linear
# cache, pinned by brute force and by round trips through known layouts.
# ----------------------------------------------------------------------------
def test_gather_pages_brute_force():
    g = torch.Generator().manual_seed(31)
    P, H, ps, D, B, mp = 7, 2, 32, 4, 3, 3
    pool = torch.randn(P, H, ps, D, generator=g).to(torch.float16)
    table = torch.tensor([[[4, 0, -1], [1, 2, -1]], [[-1, -1, -1], [-1, -1, -1]],
                          [[6, 5, 3], [0, 4, 6]]], dtype=torch.int32)
    kv = [40, 0, 70]
    for which in (0, 1):
        got = oracle.gather_pages(pool, table, which, kv)
        assert got.shape == (B, H, mp * ps, D)
        for b in range(B):
            for h in range(H):
                for n in range(mp * ps):
                    row = got[b, h, n]
                    if n < kv[b]:
                        src = pool[int(table[b, which, n // ps]), h, n % ps]
                        assert torch.equal(row.view(torch.int16), src.view(torch.int16))
                    else:
                        assert torch.isnan(row).all()


def test_gather_pages_inverts_the_paged_layout():
    from ragged_gqa_attention_gb300 import workloads as W
    c = W.make_case("g", 32, batch=4, q_heads=4, kv_heads=2, head_dim=16, q_lens=[1] * 4,
                    kv_lens=[0, 31, 64, 100], q_form="packed", kv_form="padded", kv_seq=128,
                    dtype=torch.bfloat16, causal="lower_right")
    for ps in (32, 64, 128):
        pc = W.paged(c, ps, seed=ps)
        for which, src in ((0, c.k), (1, c.v)):
            got = oracle.gather_pages(pc.k if which == 0 else pc.v, pc.page_table, which,
                                      c.kv_lens)
            for b, n in enumerate(c.kv_lens):
                assert torch.equal(got[b, :, :n].view(torch.int16), src[b, :, :n].view(torch.int16))

