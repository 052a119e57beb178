"""Seeded synthetic inputs for ragged GQA attention.

This module only draws random numbers and lays them out in the padded_bhnd /
packed_nhd forms of the "TensorRT Custom Operator Schemas" page (TRT_Attention,
tensor format notation).  It holds none of the attention arithmetic, so both
the CUDA path and the CPU oracle can take their inputs from it.

Recipe (every workload): ``torch.Generator('cpu').manual_seed(seed)``; the draw
order is lengths, Q, K, V, mask; Q/K/V are drawn as fp32 N(0, 1) and cast to
the workload dtype with round-to-nearest-even; integer lengths are uniform
with inclusive bounds.  Rows of padded KV at or beyond a sequence's kv length
hold ``kv_pad`` (NaN by default, so that any read of them shows in the
output); packed tensors may carry ``tail`` extra rows past the last sequence,
filled the same way.

FP8 KV cache workloads draw K and V the same way, divide them by the
tensor's scale (s_k, s_v), clamp to +-448 and store them as E4M3FN codes
with PyTorch's round-to-nearest-even cast to float8_e4m3fn (uint8 tensors);
padding rows then hold the code of ``kv_pad`` (0x7F, a NaN code, by
default).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

PADDED = "padded"
PACKED = "packed"
PAGED = "paged"     # K, V in page pools [num_pages, Hkv, page_size, D] + a page table


@dataclass
class Case:
    """One attention problem on host memory (CPU tensors)."""
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    q_form: str
    kv_form: str
    batch: int
    query_lengths: Optional[torch.Tensor]   # int32 [B+1] cumulative, or None
    kv_lengths: Optional[torch.Tensor]      # int32 [B+1] cumulative or [B]
    q_lens: list                            # per-batch valid query rows
    kv_lens: list                           # per-batch valid key rows
    scale: float = 1.0
    causal: str = "none"
    norm: str = "softmax"
    mask: Optional[torch.Tensor] = None
    quant: Optional[str] = None
    quant_scale: Optional[torch.Tensor] = None
    kv_scales: Optional[tuple] = None       # fp8 KV cache: (s_k, s_v) fp32 [1] tensors
    page_table: Optional[torch.Tensor] = None   # paged: int32 [B, 2, max_pages]
    meta: dict = field(default_factory=dict)

    @property
    def q_heads(self):
        return self.q.shape[-2] if self.q_form == PACKED else self.q.shape[1]

    @property
    def kv_heads(self):   # padded [B, H, N, D], packed [T, H, D], paged pools [P, H, ps, D]
        return self.k.shape[-2] if self.kv_form == PACKED else self.k.shape[1]

    @property
    def head_dim(self):
        return self.q.shape[-1]


def _cum(lens):
    out = [0]
    for n in lens:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32)


def _randn(g, shape, dtype):
    return torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)


def make_case(name, seed, *, batch, q_heads, kv_heads, head_dim, q_lens,
              kv_lens=None, q_form=PADDED, kv_form=PADDED, q_seq=None,
              kv_seq=None, dtype=torch.float16, scale=None, causal="none",
              norm="softmax", mask=None, quant=None, quant_scale=None,
              pass_query_lengths=None, pass_kv_lengths=True, kv_pad=math.nan,
              tail=0, g=None, kv_fp8=None):
    """Build a Case from explicit per-batch lengths.

    q_lens / kv_lens: per-batch valid lengths (python ints).  For padded forms
    the padded extent is ``q_seq`` / ``kv_seq`` (default: the max length).
    ``pass_query_lengths`` (padded Q) passes the optional cumulative
    query_lengths; ``pass_kv_lengths`` (padded KV) passes the optional [B]
    kv_lengths.  ``mask`` is either a ready tensor or a callable
    ``mask(g) -> tensor`` drawn after V.  ``g`` continues an existing
    generator (used when the lengths were drawn from it).  ``kv_fp8 = (s_k,
    s_v)`` stores K and V as E4M3FN codes of K / s_k and V / s_v.
    """
    if g is None:
        g = torch.Generator("cpu").manual_seed(seed)
    kv_lens = list(q_lens) if kv_lens is None else list(kv_lens)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    D = head_dim
    if q_form == PACKED:
        T = sum(q_lens) + tail
        q = _randn(g, (T, q_heads, D), dtype)
        if tail:
            q[sum(q_lens):] = kv_pad
        query_lengths = _cum(q_lens)
    else:
        q_seq = max(q_lens + [0]) if q_seq is None else q_seq
        q = _randn(g, (batch, q_heads, q_seq, D), dtype)
        query_lengths = _cum(q_lens) if pass_query_lengths else None
    if kv_form == PACKED:
        Tk = sum(kv_lens) + tail
        k = _randn(g, (Tk, kv_heads, D), dtype)
        v = _randn(g, (Tk, kv_heads, D), dtype)
        if tail:
            k[sum(kv_lens):] = kv_pad
            v[sum(kv_lens):] = kv_pad
        kv_lengths = _cum(kv_lens)
    else:
        kv_seq = max(kv_lens + [0]) if kv_seq is None else kv_seq
        k = _randn(g, (batch, kv_heads, kv_seq, D), dtype)
        v = _randn(g, (batch, kv_heads, kv_seq, D), dtype)
        for b, n in enumerate(kv_lens):
            k[b, :, n:] = kv_pad
            v[b, :, n:] = kv_pad
        kv_lengths = (torch.tensor(kv_lens, dtype=torch.int32)
                      if pass_kv_lengths else None)
    kv_scales = None
    if kv_fp8 is not None:
        k, v = _to_e4m3_codes(k, kv_fp8[0], kv_pad), _to_e4m3_codes(v, kv_fp8[1], kv_pad)
        kv_scales = tuple(torch.tensor([float(x)], dtype=torch.float32) for x in kv_fp8)
    if callable(mask):
        mask = mask(g)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if quant is not None and quant_scale is None:
        quant_scale = torch.tensor(1.0 / 448.0 if quant == "fp8" else 1.0 / 127.0,
                                   dtype=torch.float32)
    return Case(name=name, q=q, k=k, v=v, q_form=q_form, kv_form=kv_form,
                batch=batch, query_lengths=query_lengths,
                kv_lengths=kv_lengths, q_lens=q_lens, kv_lens=kv_lens,
                scale=scale, causal=causal, norm=norm, mask=mask, quant=quant,
                quant_scale=quant_scale, kv_scales=kv_scales)


def _to_e4m3_codes(x, s, pad):
    """E4M3FN codes (uint8) of x / s; elements that hold ``pad`` (the
    padding fill) get the code of ``pad`` itself."""
    pad_t = torch.tensor(pad, dtype=torch.float32)
    is_pad = torch.isnan(x) if math.isnan(pad) else (x == pad_t)
    codes = (x.float() / s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    codes[is_pad] = pad_t.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes


def paged(case: Case, page_size: int, seed: int, spare: int = 3, pad=math.nan) -> Case:
    """The same problem with its padded K/V cache moved into page pools:
    each sequence's keys fill ceil(kv_len / page_size) pages, K and V pages
    each placed at a seeded random permutation of a pool that holds
    ``spare`` extra pages; unused pages and the rows past a sequence's end
    hold ``pad`` (its E4M3 code for code pools); page-table entries past a
    sequence's last page are -1 (never read).  Layout and random draws only."""
    assert case.kv_form == PADDED and page_size % 32 == 0
    B, H, N, D = case.k.shape
    mp = max(1, (N + page_size - 1) // page_size)
    need = [(n + page_size - 1) // page_size for n in case.kv_lens]
    P = sum(need) + spare
    g = torch.Generator("cpu").manual_seed(seed)
    table = torch.full((B, 2, mp), -1, dtype=torch.int32)
    pools = []
    for which, src in enumerate((case.k, case.v)):
        pool = torch.empty((P, H, page_size, D), dtype=src.dtype)
        if src.dtype == torch.uint8:
            pool.fill_(int(torch.tensor(pad, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)))
        else:
            pool.fill_(pad)
        perm = torch.randperm(P, generator=g)
        k = 0
        for b in range(B):
            for i in range(need[b]):
                pg = int(perm[k])
                k += 1
                rows = min(page_size, N - i * page_size)
                pool[pg, :, :rows] = src[b, :, i * page_size:i * page_size + rows]
                table[b, which, i] = pg
        pools.append(pool)
    return replace(case, name=f"{case.name}_paged{page_size}", k=pools[0], v=pools[1],
                   kv_form=PAGED, page_table=table)


def rope_cos_sin(positions, rotary_dim, base=10000.0):
    """RoPE input table [T, rotary_dim] fp32 for the given positions: the
    cosines of angles position * base^(-2i / rotary_dim), i < rotary_dim/2,
    then their sines (the usual rotary frequencies; rows of negative
    positions, padding, get angle 0).  An input of the rotation, built in
    fp64 and rounded once."""
    pos = torch.as_tensor(positions, dtype=torch.float64).clamp(min=0.0)
    half = rotary_dim // 2
    inv = base ** (-2.0 * torch.arange(half, dtype=torch.float64) / rotary_dim)
    ang = pos[:, None] * inv[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32)


def _uniform_int(g, lo, hi, n):
    """n integers uniform on [lo, hi] (inclusive)."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


# The named workloads.  Each entry: (name, description).
WORKLOADS = {
    1: ("padded_selfattn_b2_h4_n64_d64_fp16",
        "padded_bhnd B=2 Hq=Hkv=4 N=64 D=64 fp16, scale 1/8, no causal"),
    2: ("packed_ragged_prefill_gqa32x8_d128_bf16",
        "packed_nhd Q/KV, B=8 lengths U[128,2048], Hq=32 Hkv=8 D=128 bf16, "
        "upper_left"),
    3: ("chunked_packedq_paddedkv8192_gqa32x8_d128_bf16",
        "packed Q chunks U[64,512], padded KV N=8192 with kv_len "
        "U[q_len,8192], B=16, Hq=32 Hkv=8 D=128 bf16, lower_right"),
    4: ("decode_b64_gqa64x8_kv4096_d128_bf16",
        "packed Q (one token each), padded KV N=4096 with kv_len "
        "U[256,4096], B=64, Hq=64 Hkv=8 D=128 bf16, lower_right"),
    5: ("quantized_padded_b4_h16_n4096_d128_fp16",
        "padded B=4 Hq=Hkv=16 N=4096 D=128 fp16, upper_left, bool key-suffix "
        "mask [B,1,1,N] of 0-25%, P Q/DQ to fp8 (s=1/448) or int8 (s=1/127)"),
    6: ("tree_decode_b16_draft8_gqa64x8_kv4096_d128_bf16",
        "tree (speculative) decoding: packed Q of 8 draft tokens per sequence, "
        "padded KV N=4104 holding the cache (U[256,4096] keys) then the 8 drafts, "
        "bool mask [B,1,8,N]: every cached key, and of the drafts the token's "
        "ancestors in a seeded random tree and itself; B=16, Hq=64 Hkv=8 D=128 bf16"),
    7: ("decode_fp8kv_b64_gqa64x8_kv4096_d128_bf16",
        "decode over an FP8 (E4M3) KV cache: packed Q (one token each), padded KV "
        "N=4096 with kv_len U[256,4096], B=64, Hq=64 Hkv=8 D=128, bf16 Q/Y, "
        "lower_right; K, V stored as E4M3FN codes with per-tensor scales "
        "s_k = 1/56, s_v = 1/48"),
    8: ("decode_b64_gqa64x8_kv4096_d128_bf16_paged64",
        "workload 4 over a paged KV cache: each sequence's keys in pages of 64 "
        "keys placed at seeded random positions of K and V pools (16 spare "
        "pages each), page table [64, 2, 64]"),
    9: ("chunked_packedq_fp8kv8192_gqa32x8_d128_bf16",
        "workload 3 (its draws) over an FP8 (E4M3) KV cache: K and V stored as "
        "E4M3FN codes with per-tensor scales s_k = 1/56, s_v = 1/48; bf16 Q and Y"),
    10: ("chunked_packedq_paddedkv8192_gqa32x8_d128_bf16_paged64",
         "workload 3 over a paged KV cache: each sequence's keys in pages of 64 "
         "keys at seeded random positions of K and V pools (16 spare pages each), "
         "page table [16, 2, 128]"),
}

# per-tensor scales of the fp8 KV cache workload (K, V ~ N(0, 1) land near
# code magnitude 56 and 48, far inside the E4M3 range)
FP8_KV_SCALES = (1.0 / 56.0, 1.0 / 48.0)


def workload(index, *, quant="fp8", kv_pad=math.nan, seed=None):
    """The named workload ``index`` (1..10) as a Case on host memory.

    ``quant`` selects the fp8 or int8 variant of workload 5.
    """
    seed = index if seed is None else seed
    g = torch.Generator("cpu").manual_seed(seed)
    name = WORKLOADS[index][0]
    if index == 1:
        return make_case(name, seed, batch=2, q_heads=4, kv_heads=4,
                         head_dim=64, q_lens=[64, 64], dtype=torch.float16,
                         scale=1.0 / 8.0, kv_pad=kv_pad, g=g)
    if index == 2:
        lens = _uniform_int(g, 128, 2048, 8)
        return make_case(name, seed, batch=8, q_heads=32, kv_heads=8,
                         head_dim=128, q_lens=lens, kv_lens=lens,
                         q_form=PACKED, kv_form=PACKED, dtype=torch.bfloat16,
                         causal="upper_left", kv_pad=kv_pad, g=g)
    if index in (3, 9):
        if index == 9:   # workload 3's draws
            g = torch.Generator("cpu").manual_seed(3)
        qls = _uniform_int(g, 64, 512, 16)
        kvls = [_uniform_int(g, ql, 8192, 1)[0] for ql in qls]
        return make_case(name, seed, batch=16, q_heads=32, kv_heads=8,
                         head_dim=128, q_lens=qls, kv_lens=kvls,
                         q_form=PACKED, kv_form=PADDED, kv_seq=8192,
                         dtype=torch.bfloat16, causal="lower_right",
                         kv_pad=kv_pad, g=g, kv_fp8=FP8_KV_SCALES if index == 9 else None)
    if index == 10:
        return paged(workload(3, kv_pad=kv_pad), 64, seed=10, spare=16, pad=kv_pad)
    if index == 4:
        kvls = _uniform_int(g, 256, 4096, 64)
        return make_case(name, seed, batch=64, q_heads=64, kv_heads=8,
                         head_dim=128, q_lens=[1] * 64, kv_lens=kvls,
                         q_form=PACKED, kv_form=PADDED, kv_seq=4096,
                         dtype=torch.bfloat16, causal="lower_right",
                         kv_pad=kv_pad, g=g)
    if index == 8:
        return paged(workload(4, kv_pad=kv_pad), 64, seed=8, spare=16, pad=kv_pad)
    if index == 7:
        kvls = _uniform_int(g, 256, 4096, 64)
        return make_case(name, seed, batch=64, q_heads=64, kv_heads=8,
                         head_dim=128, q_lens=[1] * 64, kv_lens=kvls,
                         q_form=PACKED, kv_form=PADDED, kv_seq=4096,
                         dtype=torch.bfloat16, causal="lower_right",
                         kv_pad=kv_pad, g=g, kv_fp8=FP8_KV_SCALES)
    if index == 6:
        B, T, N = 16, 8, 4096 + 8
        cache = _uniform_int(g, 256, 4096, B)

        def tree_mask(gen):
            keep = torch.zeros(B, 1, T, N, dtype=torch.bool)
            for b in range(B):
                parent = [-1] + [int(torch.randint(0, i, (1,), generator=gen)) for i in range(1, T)]
                keep[b, 0, :, :cache[b]] = True
                for i in range(T):
                    j = i
                    while j >= 0:   # the token and its ancestors
                        keep[b, 0, i, cache[b] + j] = True
                        j = parent[j]
            return keep

        return make_case(name, seed, batch=B, q_heads=64, kv_heads=8, head_dim=128,
                         q_lens=[T] * B, kv_lens=[c + T for c in cache], q_form=PACKED,
                         kv_form=PADDED, kv_seq=N, dtype=torch.bfloat16, mask=tree_mask,
                         kv_pad=kv_pad, g=g)
    if index == 5:
        N, B = 4096, 4

        def suffix_mask(gen):
            # masked key suffix of m_b = floor(U[0, 0.25] * N) keys
            m = torch.floor(torch.rand(B, generator=gen) * 0.25 * N).to(torch.int64)
            keep = torch.arange(N)[None, :] < (N - m)[:, None]
            return keep.reshape(B, 1, 1, N)

        c = make_case(name, seed, batch=B, q_heads=16, kv_heads=16,
                      head_dim=128, q_lens=[N] * B, kv_lens=[N] * B,
                      dtype=torch.float16, causal="upper_left",
                      mask=suffix_mask, quant=quant, kv_pad=kv_pad,
                      pass_kv_lengths=False, g=g)
        c.name = f"{name}_{quant}"
        return c
    raise KeyError(index)


def to_device(case: Case, device, non_blocking=False) -> Case:
    """Copy every tensor of ``case`` to ``device``."""
    def mv(t):
        return None if t is None else t.to(device, non_blocking=non_blocking)
    return replace(case, q=mv(case.q), k=mv(case.k), v=mv(case.v),
                   query_lengths=mv(case.query_lengths),
                   kv_lengths=mv(case.kv_lengths), mask=mv(case.mask),
                   quant_scale=mv(case.quant_scale),
                   kv_scales=None if case.kv_scales is None else tuple(
                       mv(t) for t in case.kv_scales),
                   page_table=mv(case.page_table))
