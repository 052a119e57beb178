"""Rotary position embedding on the GPU against the oracle: in place on Q and
K (full and partial rotary dims, padding rows), and fused with the KV cache
update of the new keys (rotated rows land in their windows, every other
cache element and the update tensor keep their bits, Q rotated in the same
launch, a bad window changes nothing)."""
import numpy as np
import pytest
import torch

import oracle
from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load(build_if_missing=True)


def _close(got, ref, dtype):
    # fp32 arithmetic rounded once to the element type: within one unit in
    # the last place of the reference (plus the dtype's smallest normal step)
    ulp = 2.0 ** -7 if dtype == torch.bfloat16 else 2.0 ** -10
    g = got.detach().cpu().double().numpy()
    err = np.abs(g - ref)
    assert (err <= ulp * np.abs(ref) + 1e-6).all(), err.max()


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
# (the kernel takes eight pairs per unit where the rotary dims are a multiple
# of 16 and every base address 16-byte aligned, else four: R = 24 and 40
# take the four-pair units)
@pytest.mark.parametrize("D,R", [(128, 128), (128, 64), (64, 64), (128, 24), (64, 40)])
def test_rope_in_place(dtype, D, R):
    g = torch.Generator().manual_seed(D + R)
    T, Hq, Hk = 37, 8, 2
    q = torch.randn(T, Hq, D, generator=g).to(dtype)
    k = torch.randn(T, Hk, D, generator=g).to(dtype)
    pos = torch.randint(0, 8192, (T,), generator=g, dtype=torch.int32)
    pos[[3, 20]] = -1
    cs = W.rope_cos_sin(pos, R)
    qd, kd = q.cuda(), k.cuda()
    binding.rope_apply(qd, kd, cos_sin=cs.cuda(), positions=pos.cuda())
    torch.cuda.synchronize()
    _close(qd, oracle.rope(q, cs, pos), dtype)
    _close(kd, oracle.rope(k, cs, pos), dtype)
    for t in (3, 20):   # padding rows keep their bits
        assert np.array_equal(_bits(qd[t]), _bits(q[t])) and np.array_equal(_bits(kd[t]), _bits(k[t]))
    if R < D:           # dims past the rotary ones keep their bits
        assert np.array_equal(_bits(qd[..., R:]), _bits(q[..., R:]))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("R", [128, 32, 40])
def test_fused_kv_update_rope(dtype, R):
    g = torch.Generator().manual_seed(7 + R)
    B, H, N, D, Hq = 5, 2, 96, 128, 8
    cache = torch.randn(B, H, N, D, generator=g).to(dtype)
    lens = torch.tensor([3, 0, 1, 7, 2])
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0)
    T = int(cu[-1])
    wi = torch.tensor([0, 5, 95, 40, 94], dtype=torch.int32)
    upd = torch.randn(T, H, D, generator=g).to(dtype)
    q = torch.randn(T, Hq, D, generator=g).to(dtype)
    pos = (wi.repeat_interleave(lens) + torch.cat([torch.arange(int(n)) for n in lens])).to(torch.int32)
    pos[4] = -1
    cs = W.rope_cos_sin(pos, R)
    cd, ud, qd = cache.cuda(), upd.cuda(), q.cuda()
    _, st = binding.trt_kv_cache_update_rope(cd, ud, cos_sin=cs.cuda(), update_lengths=cu.cuda(),
                                             write_indices=wi.cuda(), q=qd, positions=pos.cuda(),
                                             return_status=True)
    torch.cuda.synchronize()
    assert binding.device_status(st) == 0
    assert np.array_equal(_bits(ud), _bits(upd))            # the update is only read
    _close(qd, oracle.rope(q, cs, pos), dtype)
    rot = oracle.rope(upd, cs, pos)
    want_bits = _bits(cache).copy()
    got = cd.cpu()
    for b in range(B):
        for t in range(int(lens[b])):
            tg = int(cu[b]) + t
            n = int(wi[b]) + t
            _close(got[b, :, n], rot[tg], dtype)
            want_bits[b, :, n] = _bits(got[b, :, n])        # checked above
    assert np.array_equal(_bits(got), want_bits)           # every other row untouched
    # the same as rotating a copy of the update and a plain KV cache update
    cache2, upd2 = cache.cuda(), upd.cuda()
    binding.rope_apply(None, upd2, cos_sin=cs.cuda(), positions=pos.cuda())
    binding.trt_kv_cache_update(cache2, upd2, update_form="packed", write_indices=wi.cuda(),
                                update_lengths=cu.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_bits(cache2), _bits(cd))


def test_rope_in_place_on_8_byte_aligned_rows():
    # Q and K views that start 8 bytes into their buffers: the four-pair units
    g = torch.Generator().manual_seed(11)
    T, Hq, Hk, D, R = 19, 4, 2, 64, 64
    qb = torch.randn(T * Hq * D + 4, generator=g).to(torch.bfloat16)
    kb = torch.randn(T * Hk * D + 4, generator=g).to(torch.bfloat16)
    pos = torch.randint(0, 4096, (T,), generator=g, dtype=torch.int32)
    cs = W.rope_cos_sin(pos, R)
    qd, kd = qb.cuda()[4:].view(T, Hq, D), kb.cuda()[4:].view(T, Hk, D)
    assert qd.data_ptr() % 16 == 8
    q0, k0 = qd.cpu().clone(), kd.cpu().clone()
    binding.rope_apply(qd, kd, cos_sin=cs.cuda(), positions=pos.cuda())
    torch.cuda.synchronize()
    _close(qd, oracle.rope(q0, cs, pos), torch.bfloat16)
    _close(kd, oracle.rope(k0, cs, pos), torch.bfloat16)


def test_fused_bad_window_changes_nothing():
    g = torch.Generator().manual_seed(9)
    cache = torch.randn(2, 2, 16, 64, generator=g).to(torch.bfloat16)
    upd = torch.randn(4, 2, 64, generator=g).to(torch.bfloat16)
    q = torch.randn(4, 4, 64, generator=g).to(torch.bfloat16)
    cs = W.rope_cos_sin(torch.arange(4), 64)
    cd, qd = cache.cuda(), q.cuda()
    _, st = binding.trt_kv_cache_update_rope(
        cd, upd.cuda(), cos_sin=cs.cuda(), update_lengths=torch.tensor([0, 2, 4], dtype=torch.int32).cuda(),
        write_indices=torch.tensor([0, 15], dtype=torch.int32).cuda(), q=qd, return_status=True)
    torch.cuda.synchronize()
    assert binding.device_status(st) == 4
    assert np.array_equal(_bits(cd), _bits(cache)) and np.array_equal(_bits(qd), _bits(q))
