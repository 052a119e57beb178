"""TRT_KVCacheUpdate on the GPU against the oracle, bit for bit: padded and
packed updates, in place and into a separate Y, every element width and
vector width the kernel picks, optional write_indices / update_lengths,
empty updates, the decode-step and chunk shapes, and device-side rejection
of windows outside the cache (nothing written)."""
import numpy as np
import pytest
import torch

import oracle
from ragged_gqa_attention_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load(build_if_missing=True)


def _bits(t):
    view = {2: torch.int16, 4: torch.int32}[t.element_size()]
    return t.detach().cpu().contiguous().view(view).numpy()


def _case(seed, B, H, N, D, nu, form, dtype, zero_some=False):
    g = torch.Generator().manual_seed(seed)
    cache = torch.randn(B, H, N, D, generator=g).to(dtype)
    lens = torch.randint(0, nu + 1, (B,), generator=g)
    if zero_some:
        lens[::3] = 0
    wi = torch.tensor([int(torch.randint(0, N - int(l) + 1, (1,), generator=g)) for l in lens],
                      dtype=torch.int32)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0)
    if form == "padded":
        upd = torch.randn(B, H, nu, D, generator=g).to(dtype)
    else:
        upd = torch.randn(int(cu[-1]), H, D, generator=g).to(dtype)
    return cache, upd, wi, cu


def _run(cache, upd, form, wi, cu, in_place):
    dev = lambda t: None if t is None else t.cuda()
    c, u = dev(cache), dev(upd)
    out = None if in_place else torch.full_like(c, float("nan"))
    y, st = binding.trt_kv_cache_update(c, u, update_form=form, write_indices=dev(wi),
                                        update_lengths=dev(cu), out=out, return_status=True)
    torch.cuda.synchronize()
    return y, binding.device_status(st)


@pytest.mark.parametrize("form", ["padded", "packed"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("in_place", [True, False])
def test_parity(form, dtype, in_place):
    cache, upd, wi, cu = _case(31, B=5, H=3, N=40, D=64, nu=7, form=form, dtype=dtype,
                               zero_some=True)
    y, st = _run(cache, upd, form, wi, cu, in_place)
    assert st == 0
    want = oracle.kv_cache_update(cache, upd, update_form=form, write_indices=wi, update_lengths=cu)
    assert np.array_equal(_bits(y), want)


@pytest.mark.parametrize("D,dtype", [(6, torch.float16), (3, torch.float16), (5, torch.float32)])
@pytest.mark.parametrize("form", ["padded", "packed"])
def test_narrow_rows_use_smaller_vectors(D, dtype, form):
    # rows of 12 or 6 bytes (16-bit) and 20 bytes (32-bit): 4- and 2-byte moves
    cache, upd, wi, cu = _case(32, B=4, H=2, N=17, D=D, nu=5, form=form, dtype=dtype)
    for in_place in (True, False):
        y, st = _run(cache, upd, form, wi, cu, in_place)
        assert st == 0
        want = oracle.kv_cache_update(cache, upd, update_form=form, write_indices=wi,
                                      update_lengths=cu)
        assert np.array_equal(_bits(y), want)


def test_optional_inputs_absent():
    # padded update, no lengths (all N_u tokens), no write_indices (position 0)
    cache, upd, _, _ = _case(33, B=3, H=2, N=12, D=64, nu=4, form="padded", dtype=torch.bfloat16)
    for in_place in (True, False):
        y, st = _run(cache, upd, "padded", None, None, in_place)
        assert st == 0
        want = oracle.kv_cache_update(cache, upd, update_form="padded")
        assert np.array_equal(_bits(y), want)


def test_decode_step_and_chunk_shapes():
    # one new token per sequence at its end (decode), and a prefill chunk
    g = torch.Generator().manual_seed(34)
    B, H, N, D = 64, 8, 1024, 128
    cache = torch.randn(B, H, N, D, generator=g).to(torch.bfloat16)
    kv_len = torch.randint(1, N + 1, (B,), generator=g)
    upd = torch.randn(B, H, D, generator=g).to(torch.bfloat16)
    cu = torch.arange(B + 1, dtype=torch.int32)
    wi = (kv_len - 1).to(torch.int32)
    y, st = _run(cache, upd, "packed", wi, cu, True)
    assert st == 0
    want = oracle.kv_cache_update(cache, upd, update_form="packed", write_indices=wi,
                                  update_lengths=cu)
    assert np.array_equal(_bits(y), want)
    cache, upd, wi, cu = _case(35, B=8, H=8, N=2048, D=128, nu=512, form="packed",
                               dtype=torch.bfloat16)
    y, st = _run(cache, upd, "packed", wi, cu, True)
    assert st == 0
    want = oracle.kv_cache_update(cache, upd, update_form="packed", write_indices=wi,
                                  update_lengths=cu)
    assert np.array_equal(_bits(y), want)


@pytest.mark.parametrize("bad", ["window_past_end", "negative_index", "lengths_past_update",
                                 "lengths_not_from_zero"])
@pytest.mark.parametrize("in_place", [True, False])
def test_bad_windows_set_status_and_write_nothing(bad, in_place):
    cache, upd, wi, cu = _case(36, B=4, H=2, N=16, D=64, nu=4, form="packed",
                               dtype=torch.float16)
    cu = torch.tensor([0, 2, 3, 5, 7], dtype=torch.int32)
    upd = torch.randn(7, 2, 64, generator=torch.Generator().manual_seed(37)).to(torch.float16)
    wi = torch.tensor([0, 4, 8, 12], dtype=torch.int32)
    if bad == "window_past_end":
        wi[3] = 15
    elif bad == "negative_index":
        wi[1] = -1
    elif bad == "lengths_past_update":
        cu[4] = 8
    else:
        cu = cu + 1
    y, st = _run(cache, upd, "packed", wi, cu, in_place)
    assert st == 4
    if in_place:
        assert np.array_equal(_bits(y), _bits(cache))
    else:
        assert torch.isnan(y).all()
