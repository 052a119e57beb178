"""GPU parity: the CUDA library (through the C ABI) against the fp64 CPU
oracle on the same seeded inputs, element by element.

Tolerances (stated for the fused attention forward): max-abs 1e-2 and
mean-abs 1e-3 for fp16/bf16 with unquantised P; max-abs 3e-2 when P goes
through the fp8/int8 Q/DQ.  Rows outside the sequences and guard bands
around Y must keep their NaN sentinel bits exactly.
"""
import math

import numpy as np
import pytest
import torch

from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import workloads as W

from helpers import check, run_gpu, run_oracle, valid_row_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load(build_if_missing=True)


def _parity(case, tol=None):
    y, raw, st = run_gpu(case)
    assert binding.device_status(st) == 0
    ref = run_oracle(case)
    return check(case, y, raw, ref, tol)


def test_workload1_small_padded():
    _parity(W.workload(1))


# --------------------------------------------------------------------------
# option sweep on small ragged shapes that span several tiles and tails
# --------------------------------------------------------------------------
SWEEP = []
for qf in ("padded", "packed"):
    for kf in ("padded", "packed"):
        for causal in ("none", "upper_left", "lower_right"):
            for G in (1, 4):
                for D in (64, 128):
                    SWEEP.append((qf, kf, causal, G, D))


@pytest.mark.parametrize("qf,kf,causal,G,D", SWEEP)
def test_prefill_sweep(qf, kf, causal, G, D):
    dtype = torch.bfloat16 if (G + D + len(causal)) % 2 else torch.float16
    Hkv = 2
    c = W.make_case("sweep", 100 + len(SWEEP), batch=3, q_heads=Hkv * G, kv_heads=Hkv,
                    head_dim=D, q_lens=[1, 150, 277], kv_lens=[200, 131, 300],
                    q_form=qf, kv_form=kf, dtype=dtype, causal=causal,
                    pass_query_lengths=True, tail=3)
    _parity(c)


@pytest.mark.parametrize("G", [2, 8, 16, 32])
def test_prefill_gqa_ratios(G):
    c = W.make_case("gqa", 7, batch=2, q_heads=2 * G, kv_heads=2, head_dim=128,
                    q_lens=[190, 33], kv_lens=[190, 300], q_form="packed", kv_form="packed",
                    dtype=torch.bfloat16, causal="lower_right")
    _parity(c)


def test_prefill_odd_group_size():
    # G = 3: 42 tokens x 3 heads fill 126 of the 128 tile rows
    c = W.make_case("g3", 8, batch=2, q_heads=6, kv_heads=2, head_dim=64,
                    q_lens=[100, 45], kv_lens=[100, 45], q_form="packed", kv_form="padded",
                    dtype=torch.float16, causal="upper_left")
    _parity(c)


@pytest.mark.parametrize("mdtype", [torch.bool, torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", ["full", "key", "head_row"])
def test_prefill_masks(mdtype, shape):
    B, H, N, Nk = 2, 4, 140, 260
    g = torch.Generator().manual_seed(5)

    def mk(gen):
        dims = {"full": (B, H, N, Nk), "key": (B, 1, 1, Nk), "head_row": (1, H, N, 1)}[shape]
        if mdtype == torch.bool:
            m = torch.rand(dims, generator=gen) > 0.3
        else:
            m = (torch.randn(dims, generator=gen) * 2).to(mdtype)
        return m

    c = W.make_case("mask", 9, batch=B, q_heads=H, kv_heads=2, head_dim=128,
                    q_lens=[N, 77], kv_lens=[Nk, 201], q_seq=N, kv_seq=Nk,
                    dtype=torch.float16, mask=mk, pass_query_lengths=True)
    _parity(c)


@pytest.mark.parametrize("quant", [None, "fp8"])
def test_key_mask_hiding_the_start_of_a_tile(quant):
    # a key-only bool mask that excludes the first 64 keys of the first tile
    # (and scattered keys later): the rows' first reference must come from
    # keys past the first half of the tile
    B, N = 2, 300

    def mk(gen):
        keep = torch.rand((B, 1, 1, N), generator=gen) > 0.2
        keep[..., :64] = False
        keep[1, ..., 128:200] = False
        return keep

    c = W.make_case("latekeys", 24, batch=B, q_heads=4, kv_heads=2, head_dim=128,
                    q_lens=[N, 131], kv_lens=[N, N], q_seq=N, kv_seq=N,
                    dtype=torch.bfloat16, mask=mk, quant=quant, pass_query_lengths=True)
    _parity(c)


@pytest.mark.parametrize("causal", ["none", "upper_left"])
def test_prefill_norm_none(causal):
    c = W.make_case("none", 10, batch=2, q_heads=4, kv_heads=4, head_dim=64,
                    q_lens=[130, 64], kv_lens=[130, 250], dtype=torch.float16,
                    causal=causal, norm="none", scale=0.01, pass_query_lengths=True)
    _parity(c)


def _minus_inf_mask(B, H, Nq, Nkv, q_lens, kv_lens, seed):
    """Additive fp32 mask [B, H, Nq, Nkv]: zeros, with -inf at a few allowed
    pairs (inside both lengths) and +inf at one."""
    rng = np.random.default_rng(seed)
    m = torch.zeros(B, H, Nq, Nkv, dtype=torch.float32)
    for b in range(B):
        for _ in range(3):
            m[b, int(rng.integers(H)), int(rng.integers(q_lens[b])),
              int(rng.integers(kv_lens[b]))] = -math.inf
    m[0, 0, int(rng.integers(q_lens[0])), int(rng.integers(kv_lens[0]))] = math.inf
    return m


@pytest.mark.parametrize("path", ["prefill", "decode", "quantized"])
def test_none_with_infinite_mask_values_follows_the_formula(path):
    """Under 'none' the additive mask value is added to the scaled score and
    the sum multiplies V with no normalisation ("TensorRT Custom Operator
    Schemas", TRT_Attention: attn_mask, TRT_normalization_op).  An allowed
    pair whose value is -inf (or +inf) therefore gives a non-finite output
    row, as in the oracle; under the quantized op the infinite score
    saturates to the largest code and the row stays finite.  Excluded pairs
    (past the lengths) still contribute 0."""
    if path == "decode":
        B, H, N = 3, 8, 300
        q_lens, kv_lens = [1] * B, [300, 120, 299]
        mask = _minus_inf_mask(B, H, 1, N, q_lens, kv_lens, 31)
        c = W.make_case("none_inf_dec", 31, batch=B, q_heads=H, kv_heads=2, head_dim=128,
                        q_lens=q_lens, kv_lens=kv_lens, q_form="packed", kv_form="padded",
                        kv_seq=N, dtype=torch.float16, norm="none", scale=0.01, mask=mask)
    else:
        B, H = 2, 4
        q_lens, kv_lens = [130, 70], [200, 90]
        mask = _minus_inf_mask(B, H, 130, 200, q_lens, kv_lens, 32)
        c = W.make_case("none_inf", 32, batch=B, q_heads=H, kv_heads=H, head_dim=64,
                        q_lens=q_lens, kv_lens=kv_lens, dtype=torch.float16, norm="none",
                        scale=0.01, mask=mask, pass_query_lengths=True,
                        quant="int8" if path == "quantized" else None,
                        quant_scale=torch.tensor(1 / 127) if path == "quantized" else None)
    y, raw, st = run_gpu(c)
    assert binding.device_status(st) == 0
    ref = run_oracle(c)
    if path == "quantized":
        check(c, y, raw, ref)
        return
    rows = valid_row_mask(c)
    g, r = y[rows], ref[rows]
    bad = ~np.isfinite(r)
    assert bad.any(), "the case must produce non-finite oracle rows"
    np.testing.assert_array_equal(~np.isfinite(g), bad)
    err = np.abs(g[~bad] - r[~bad])
    assert err.max() <= 1e-2 and err.mean() <= 1e-3, err.max()


# --------------------------------------------------------------------------
# quantized P (TRT_QuantizedAttention)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("quant", ["fp8", "int8"])
@pytest.mark.parametrize("norm", ["softmax", "none"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_quantized(quant, norm, dtype):
    B, N = 2, 300

    def suffix(gen):
        m = torch.floor(torch.rand(B, generator=gen) * 0.25 * N).long()
        return (torch.arange(N)[None, :] < (N - m)[:, None]).reshape(B, 1, 1, N)

    c = W.make_case("quant", 11, batch=B, q_heads=4, kv_heads=4, head_dim=128,
                    q_lens=[N, N], dtype=dtype, causal="upper_left", mask=suffix,
                    quant=quant, norm=norm, scale=(0.005 if norm == "none" else None),
                    pass_kv_lengths=False)
    _parity(c)


@pytest.mark.parametrize("quant", ["fp8", "int8"])
@pytest.mark.parametrize("kind", ["bool_rows", "additive"])
def test_quantized_softmax_under_row_masks(quant, kind):
    # masks that depend on the query row take the kernel's general path for
    # both passes of the quantized softmax (each P grid in its own copy of
    # the probability loop)
    B, H, Nq, N = 2, 4, 200, 260

    def mk(gen):
        if kind == "bool_rows":
            return torch.rand((B, 1, Nq, N), generator=gen) > 0.25
        return (torch.randn((B, H, Nq, N), generator=gen) * 2).to(torch.float16)

    c = W.make_case("qrows", 41 + (kind == "additive"), batch=B, q_heads=H, kv_heads=2,
                    head_dim=128, q_lens=[Nq, 131], kv_lens=[N, 190], q_seq=Nq, kv_seq=N,
                    dtype=torch.float16, mask=mk, quant=quant, pass_query_lengths=True)
    _parity(c)


@pytest.mark.parametrize("sdtype", [torch.float16, torch.bfloat16])
def test_quantized_scale_dtypes(sdtype):
    c = W.make_case("qs", 12, batch=1, q_heads=2, kv_heads=1, head_dim=64,
                    q_lens=[200], kv_lens=[260], q_form="packed", kv_form="packed",
                    dtype=torch.float16, causal="lower_right", quant="int8",
                    quant_scale=torch.tensor(1 / 127).to(sdtype))
    _parity(c)


# --------------------------------------------------------------------------
# decode (split-KV) path
# --------------------------------------------------------------------------
@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_packed_q(G, dtype):
    B = 6
    kv = [1, 31, 32, 513, 1100, 2049]
    c = W.make_case("dec", 13, batch=B, q_heads=2 * G, kv_heads=2, head_dim=128,
                    q_lens=[1] * B, kv_lens=kv, q_form="packed", kv_form="padded",
                    kv_seq=2100, dtype=dtype, causal="lower_right")
    _parity(c)


@pytest.mark.parametrize("causal", ["none", "upper_left", "lower_right"])
def test_decode_padded_q_packed_kv(causal):
    c = W.make_case("dec2", 14, batch=3, q_heads=8, kv_heads=2, head_dim=64,
                    q_lens=[1, 1, 1], kv_lens=[700, 5, 1600], q_form="padded",
                    kv_form="packed", dtype=torch.bfloat16, causal=causal, tail=5)
    _parity(c)


def test_decode_multi_token_rows():
    # two tokens x 8 heads = 16 rows per (batch, kv head); one sequence with
    # more rows than a row block goes through the single-split loop
    c = W.make_case("dec3", 15, batch=4, q_heads=8, kv_heads=1, head_dim=128,
                    q_lens=[2, 0, 1, 1], kv_lens=[900, 10, 2000, 600], q_form="packed",
                    kv_form="padded", dtype=torch.bfloat16, causal="lower_right")
    _parity(c)
    c = W.make_case("dec4", 16, batch=4, q_heads=8, kv_heads=1, head_dim=128,
                    q_lens=[4, 0, 0, 0], kv_lens=[900, 10, 20, 600], q_form="packed",
                    kv_form="padded", dtype=torch.bfloat16, causal="lower_right")
    _parity(c)


def test_decode_zero_keys_and_range_edges():
    # sequences without keys (their rows are zero and no warp's range holds
    # them), and many short sequences whose pairs are cut by the ends of the
    # warps' tile ranges
    c = W.make_case("dec5", 21, batch=5, q_heads=16, kv_heads=2, head_dim=128,
                    q_lens=[1] * 5, kv_lens=[0, 1, 0, 700, 3000], q_form="packed",
                    kv_form="padded", kv_seq=3000, dtype=torch.bfloat16, causal="lower_right")
    _parity(c)
    g = torch.Generator().manual_seed(22)
    kv = torch.randint(1, 300, (257,), generator=g).tolist()
    c = W.make_case("dec6", 23, batch=257, q_heads=16, kv_heads=2, head_dim=64,
                    q_lens=[1] * 257, kv_lens=kv, q_form="packed", kv_form="padded",
                    kv_seq=300, dtype=torch.float16, causal="lower_right")
    _parity(c)


def test_decode_masks_and_none():
    B, N = 3, 1000
    c = W.make_case("decm", 17, batch=B, q_heads=8, kv_heads=2, head_dim=128,
                    q_lens=[1] * B, kv_lens=[N, 600, 999], q_form="packed", kv_form="padded",
                    kv_seq=N, dtype=torch.float16,
                    mask=lambda g: torch.rand((B, 8, 1, N), generator=g) > 0.2)
    _parity(c)
    c = W.make_case("decn", 18, batch=B, q_heads=8, kv_heads=2, head_dim=128,
                    q_lens=[1] * B, kv_lens=[N, 600, 999], q_form="packed", kv_form="padded",
                    kv_seq=N, dtype=torch.float16, norm="none", scale=0.01)
    _parity(c)


@pytest.mark.parametrize("D,dtype", [(64, torch.float16), (128, torch.bfloat16)])
@pytest.mark.parametrize("norm", ["softmax", "none"])
@pytest.mark.parametrize("q_form", ["packed", "padded"])
def test_decode_sixteen_row_pairs(D, dtype, norm, q_form):
    # more than 8 query rows per (batch, KV head) on average: the 16-bit
    # decode tile takes 16 rows per pair as two N-blocks.  G = 4 with 3, 1,
    # 2 and 3 tokens gives 12, 4, 8 and 12 rows: second N-blocks that are
    # half full or empty, a first row that sees no key (2 keys for 3 tokens,
    # lower right) and pairs that the stream-K ranges cut.  'none' sums up to
    # 2049 unnormalised terms: scale 0.001 keeps |y| below 2, where bf16
    # output rounding stays inside the tolerance
    kw = dict(q_seq=3, pass_query_lengths=True) if q_form == "padded" else dict(tail=3)
    c = W.make_case("dec16", 30 + D + (norm == "none") + 2 * (q_form == "padded"), batch=4,
                    q_heads=8, kv_heads=2, head_dim=D, q_lens=[3, 1, 2, 3],
                    kv_lens=[2, 33, 700, 2049], q_form=q_form, kv_form="padded", kv_seq=2100,
                    dtype=dtype, causal="lower_right", norm=norm,
                    scale=0.001 if norm == "none" else None, **kw)
    _parity(c)


@pytest.mark.parametrize("G", [2, 8])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_tree_decoding(G, dtype):
    # 8 draft tokens per sequence under a tree mask on the split-KV decode
    # kernel: 16 rows per (batch, KV head) with G = 2 (one row chunk), 64
    # rows with G = 8 (four chunks)
    from helpers import tree_mask
    B, T = 3, 8
    cache = [40, 700, 129]
    N = max(cache) + T + 5
    c = W.make_case("tree", 24 + G, batch=B, q_heads=2 * G, kv_heads=2, head_dim=128,
                    q_lens=[T] * B, kv_lens=[x + T for x in cache], q_form="packed",
                    kv_form="padded", kv_seq=N, dtype=dtype, mask=tree_mask(B, T, N, cache))
    _parity(c)


@pytest.mark.parametrize("shape", ["rounds", "partial_round", "long", "d64_none", "padded_q"])
def test_grouped_decode(shape):
    """More than two 16-row chunks per (batch, KV head) on average: warps in
    groups of four share each K/V tile (one chunk each), units with more than
    four chunks take several rounds, and units cut by the groups' ranges are
    merged from partials."""
    from helpers import tree_mask
    D, dtype, norm, q_form = 128, torch.bfloat16, "softmax", "packed"
    if shape == "rounds":          # 16 x 8 = 128 rows: 8 chunks, two rounds
        G, T, cache = 16, 8, [40, 700, 129]
    elif shape == "partial_round":   # 8 x 5 = 40 rows: 3 chunks, the last half full
        G, T, cache = 8, 5, [0, 333, 1025, 64]
    elif shape == "long":          # few units over long caches: ranges cut them
        G, T, cache = 8, 8, [3900, 2500]
    elif shape == "d64_none":
        G, T, cache, D, dtype, norm = 8, 8, [100, 517, 31], 64, torch.float16, "none"
    else:
        G, T, cache, q_form = 8, 6, [77, 640, 1], "padded"
    B = len(cache)
    N = max(cache) + T + 5
    kw = dict(q_seq=T, pass_query_lengths=True) if q_form == "padded" else {}
    c = W.make_case(f"grp_{shape}", 60 + len(shape), batch=B, q_heads=2 * G, kv_heads=2,
                    head_dim=D, q_lens=[T] * B, kv_lens=[x + T for x in cache], q_form=q_form,
                    kv_form="padded", kv_seq=N, dtype=dtype, norm=norm,
                    scale=0.002 if norm == "none" else None, mask=tree_mask(B, T, N, cache), **kw)
    _parity(c)


def test_grouped_decode_paged():
    from helpers import tree_mask
    B, T, G = 3, 8, 8
    cache = [40, 1500, 129]
    N = max(cache) + T + 5
    c = W.make_case("grp_paged", 77, batch=B, q_heads=2 * G, kv_heads=2, head_dim=128,
                    q_lens=[T] * B, kv_lens=[x + T for x in cache], q_form="packed",
                    kv_form="padded", kv_seq=N, dtype=torch.bfloat16,
                    mask=tree_mask(B, T, N, cache))
    _parity(W.paged(c, 64, seed=17))


# --------------------------------------------------------------------------
# degenerate shapes and device-side length errors
# --------------------------------------------------------------------------
def test_empty_and_degenerate_rows():
    # kv_len 0 (zero rows), q_len 0 (nothing written), lower_right with
    # q_len > kv_len (leading rows have no key)
    c = W.make_case("deg", 19, batch=4, q_heads=4, kv_heads=2, head_dim=64,
                    q_lens=[5, 0, 200, 1], kv_lens=[0, 7, 150, 1], q_form="padded",
                    kv_form="padded", q_seq=200, dtype=torch.float16, causal="lower_right",
                    pass_query_lengths=True)
    _parity(c)


def test_all_keys_masked_rows_are_zero():
    c = W.make_case("allmask", 20, batch=1, q_heads=2, kv_heads=2, head_dim=64,
                    q_lens=[64], kv_lens=[64], dtype=torch.float16,
                    mask=torch.zeros((1, 1, 64, 64), dtype=torch.bool))
    y, raw, st = run_gpu(c)
    assert (y == 0).all()


def test_bad_lengths_set_status_and_leave_y_untouched():
    c = W.make_case("bad", 21, batch=2, q_heads=2, kv_heads=2, head_dim=64,
                    q_lens=[10, 20], q_form="packed", kv_form="packed", dtype=torch.float16)
    c.query_lengths = torch.tensor([0, 25, 20], dtype=torch.int32)   # decreasing
    y, raw, st = run_gpu(c)
    assert binding.device_status(st) == 4
    from helpers import SENTINEL
    assert (raw == np.int16(SENTINEL)).all()


def test_invalid_arguments_return_codes():
    c = W.to_device(W.workload(1), "cuda")
    y = torch.empty_like(c.q)
    with pytest.raises(binding.RgaError) as e:   # mask together with causal
        binding.trt_attention(c.q, c.k, c.v, out=y, causal="upper_left",
                              mask=torch.ones(64, 64, dtype=torch.bool, device="cuda"))
    assert e.value.code == 1
    with pytest.raises(binding.RgaError) as e:   # head_dim 32 is not implemented
        q = torch.zeros(1, 2, 8, 32, dtype=torch.float16, device="cuda")
        binding.trt_attention(q, q, q)
    assert e.value.code == 2
    with pytest.raises(binding.RgaError) as e:   # 3 query heads over 2 KV heads
        q = torch.zeros(1, 3, 8, 64, dtype=torch.float16, device="cuda")
        kv = torch.zeros(1, 2, 8, 64, dtype=torch.float16, device="cuda")
        binding.trt_attention(q, kv, kv)
    assert e.value.code == 1


def test_repeat_calls_reuse_workspace():
    c = W.workload(1)
    y1, _, _ = run_gpu(c)
    y2, _, _ = run_gpu(c)
    np.testing.assert_array_equal(y1, y2)
