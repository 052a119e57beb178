"""Thin ctypes binding of the C ABI in include/rga.h.

Argument marshalling only: every step of the attention runs in the CUDA
library (librga.so).  There is no CPU or PyTorch fallback: if the library is
not built, or the tensors are not CUDA tensors, the call raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import buildlib as _build

c_int, c_i32, c_i64 = ctypes.c_int, ctypes.c_int32, ctypes.c_int64
c_vp, c_size, c_float = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float

# enums of rga.h
RGA_OK = 0
STATUS_NAMES = {0: "RGA_OK", 1: "RGA_ERR_INVALID_ARG", 2: "RGA_ERR_UNSUPPORTED",
                3: "RGA_ERR_CUDA", 4: "RGA_ERR_DEVICE_LENGTHS", 5: "RGA_ERR_TIMEOUT",
                6: "RGA_ERR_WORKSPACE", 7: "RGA_ERR_DEBUG_BOUNDS"}
FORMS = {"padded": 0, "padded_bhnd": 0, "packed": 1, "packed_nhd": 1}
CAUSAL = {"none": 0, "upper_left": 1, "lower_right": 2}
NORM = {"softmax": 0, "none": 1}
QUANT = {"fp8": 0, "int8": 1}
DTYPES = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2, torch.bool: 3,
          torch.float8_e4m3fn: 4}
# tensors that may carry E4M3 codes (an fp8 KV cache)
FP8_CODE_DTYPES = (torch.float8_e4m3fn, torch.uint8)

EXPORTED = ("rga_attention_workspace_size", "trt_attention", "trt_quantized_attention",
            "rga_get_device_status", "rga_status_string", "rga_abi_version",
            "trt_attention_static_scratch", "trt_kv_cache_update", "rga_selftest_wait_timeout",
            "trt_attention_fp8_kv", "rga_selftest_e4m3_decode", "trt_attention_paged_kv",
            "rga_rope_apply", "trt_kv_cache_update_rope", "rga_selftest_bounds_check")


class Args(ctypes.Structure):
    """Mirror of rga_attention_args."""
    _fields_ = [
        ("q", c_vp), ("k", c_vp), ("v", c_vp), ("y", c_vp),
        ("dtype", c_int), ("q_form", c_int), ("kv_form", c_int),
        ("batch", c_i32), ("q_heads", c_i32), ("kv_heads", c_i32), ("head_dim", c_i32),
        ("q_seq", c_i32), ("kv_seq", c_i32),
        ("query_lengths", c_vp), ("kv_lengths", c_vp),
        ("mask", c_vp), ("mask_dtype", c_int), ("mask_rank", c_i32), ("mask_dims", c_i64 * 4),
        ("scale", c_float), ("causal", c_int), ("norm", c_int), ("nb_rank", c_i32),
        ("workspace", c_vp), ("workspace_bytes", c_size), ("device_status", c_vp),
    ]


class KvArgs(ctypes.Structure):
    """Mirror of rga_kv_update_args."""
    _fields_ = [
        ("past_cache", c_vp), ("update", c_vp), ("y", c_vp),
        ("dtype", c_int), ("update_form", c_int),
        ("batch", c_i32), ("heads", c_i32), ("cache_seq", c_i32), ("head_dim", c_i32),
        ("update_seq", c_i32),
        ("write_indices", c_vp), ("update_lengths", c_vp), ("device_status", c_vp),
    ]


class PagedKv(ctypes.Structure):
    """Mirror of rga_paged_kv."""
    _fields_ = [
        ("k_pool", c_vp), ("v_pool", c_vp), ("kv_dtype", c_int),
        ("k_scale", c_vp), ("v_scale", c_vp), ("page_table", c_vp),
        ("num_pages", c_i32), ("page_size", c_i32), ("max_pages_per_seq", c_i32),
    ]


class RopeArgs(ctypes.Structure):
    """Mirror of rga_rope_args."""
    _fields_ = [
        ("q", c_vp), ("k", c_vp), ("dtype", c_int),
        ("tokens", c_i32), ("q_heads", c_i32), ("kv_heads", c_i32), ("head_dim", c_i32),
        ("rotary_dim", c_i32), ("cos_sin", c_vp), ("positions", c_vp),
    ]


class RgaError(RuntimeError):
    def __init__(self, code, where=""):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")
        self.code = code


_lib = None
_lock = threading.Lock()


def debug_checks() -> bool:
    """RGA_DEBUG_CHECKS=1 in the environment selects librga_debug.so, the
    build whose kernels check their accesses (status 7 on a violation)."""
    return os.environ.get("RGA_DEBUG_CHECKS", "0") not in ("", "0")


def library_path() -> str:
    return _build.DEBUG_LIB_PATH if debug_checks() else _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load librga.so, or librga_debug.so (RGA_DEBUG_CHECKS=1), optionally
    building it first."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if build_if_missing:
                _build.build(debug_checks=debug_checks())
            if not os.path.exists(path):
                raise RuntimeError(
                    f"the CUDA library {path} is not built; run "
                    "ragged_gqa_attention_gb300.buildlib.build() (there is no fallback)")
            lib = ctypes.CDLL(path)
            P = ctypes.POINTER(Args)
            lib.rga_attention_workspace_size.restype = c_size
            lib.rga_attention_workspace_size.argtypes = [P]
            lib.trt_attention.restype = c_int
            lib.trt_attention.argtypes = [P, c_vp]
            lib.trt_quantized_attention.restype = c_int
            lib.trt_quantized_attention.argtypes = [P, c_int, c_vp, c_int, c_vp]
            lib.trt_attention_static_scratch.restype = c_int
            lib.trt_attention_static_scratch.argtypes = [P, c_vp]
            lib.rga_get_device_status.restype = c_int
            lib.rga_get_device_status.argtypes = [c_vp, c_vp, ctypes.POINTER(c_i32)]
            lib.rga_status_string.restype = ctypes.c_char_p
            lib.rga_status_string.argtypes = [c_int]
            lib.rga_abi_version.restype = c_i32
            lib.rga_abi_version.argtypes = []
            lib.rga_selftest_wait_timeout.restype = c_int
            lib.rga_selftest_wait_timeout.argtypes = [c_vp, c_i64, c_vp]
            lib.trt_attention_fp8_kv.restype = c_int
            lib.trt_attention_fp8_kv.argtypes = [P, c_vp, c_vp, c_vp]
            lib.rga_selftest_e4m3_decode.restype = c_int
            lib.rga_selftest_e4m3_decode.argtypes = [c_vp, c_vp, c_vp]
            lib.rga_selftest_bounds_check.restype = c_int
            lib.rga_selftest_bounds_check.argtypes = [c_vp, c_i64, c_i64, c_vp, c_vp]
            lib.trt_attention_paged_kv.restype = c_int
            lib.trt_attention_paged_kv.argtypes = [P, ctypes.POINTER(PagedKv), c_vp]
            lib.rga_rope_apply.restype = c_int
            lib.rga_rope_apply.argtypes = [ctypes.POINTER(RopeArgs), c_vp]
            lib.trt_kv_cache_update_rope.restype = c_int
            lib.trt_kv_cache_update_rope.argtypes = [ctypes.POINTER(KvArgs),
                                                     ctypes.POINTER(RopeArgs), c_vp]
            lib.trt_kv_cache_update.restype = c_int
            lib.trt_kv_cache_update.argtypes = [ctypes.POINTER(KvArgs), c_vp]
            _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need_cuda(name, t):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t is not None and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_args(q, k, v, y, *, q_form="padded", kv_form="padded", query_lengths=None,
              kv_lengths=None, mask=None, scale=1.0, causal="none", norm="softmax",
              workspace=None, status=None, batch=None, nb_rank=1) -> Args:
    """Fill an rga_attention_args from tensors (no device work)."""
    qf, kf = FORMS[q_form], FORMS[kv_form]
    for name, t in (("q", q), ("k", k), ("v", v), ("y", y), ("query_lengths", query_lengths),
                    ("kv_lengths", kv_lengths), ("mask", mask), ("workspace", workspace),
                    ("status", status)):
        _need_cuda(name, t)
    a = Args()
    a.q, a.k, a.v, a.y = _ptr(q), _ptr(k), _ptr(v), _ptr(y)
    a.dtype = DTYPES.get(q.dtype, 99)
    a.q_form, a.kv_form = qf, kf
    if batch is None:
        if qf == 1:
            batch = query_lengths.numel() - 1
        elif kf == 1:
            batch = kv_lengths.numel() - 1
        else:
            batch = q.shape[0]
    a.batch = batch
    a.q_heads = q.shape[-2] if qf == 1 else q.shape[1]
    a.kv_heads = k.shape[-2] if kf == 1 else k.shape[1]
    a.head_dim = q.shape[-1]
    a.q_seq = q.shape[0] if qf == 1 else q.shape[2]
    a.kv_seq = k.shape[0] if kf == 1 else k.shape[2]
    a.query_lengths, a.kv_lengths = _ptr(query_lengths), _ptr(kv_lengths)
    if mask is not None:
        a.mask = _ptr(mask)
        a.mask_dtype = DTYPES[mask.dtype]
        a.mask_rank = mask.dim()
        for i, d in enumerate(mask.shape):
            a.mask_dims[i] = d
    a.scale = float(scale)
    a.causal, a.norm, a.nb_rank = CAUSAL[causal], NORM[norm], nb_rank
    if workspace is not None:
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    a.device_status = _ptr(status)
    return a


def workspace_size(args: Args) -> int:
    return load().rga_attention_workspace_size(ctypes.byref(args))


_ws_cache = {}


def _workspace(device, nbytes):
    key = (device.index if device.index is not None else torch.cuda.current_device())
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _stream_handle(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _call(kind, q, k, v, out, extra, stream, **kw):
    """kind: 'plain' (trt_attention), 'quant' (extra = (qtype, quant_scale)),
    'fp8kv' (extra = (k_scale, v_scale)) or 'paged' (extra = a filled
    PagedKv, k and v being the pools)."""
    lib = load()
    y = torch.full_like(q, float("nan")) if out is None else out
    status = kw.pop("status", None)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=q.device)
    workspace = kw.pop("workspace", None)
    a = make_args(q, k, v, y, status=status, workspace=workspace, **kw)
    if kind == "paged":   # a sequence may hold up to max_pages_per_seq * page_size keys
        a.kv_seq = extra.max_pages_per_seq * extra.page_size
    if workspace is None:
        n = lib.rga_attention_workspace_size(ctypes.byref(a))
        if n > 0:   # n == 0: invalid arguments; the call below reports which
            ws = _workspace(q.device, n)
            a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    h = _stream_handle(stream)
    if kind == "quant":
        qt, qs = extra
        rc = lib.trt_quantized_attention(ctypes.byref(a), QUANT[qt], qs.data_ptr(),
                                         DTYPES[qs.dtype], h)
        name = "trt_quantized_attention"
    elif kind == "fp8kv":
        ks, vs = extra
        rc = lib.trt_attention_fp8_kv(ctypes.byref(a), ks.data_ptr(), vs.data_ptr(), h)
        name = "trt_attention_fp8_kv"
    elif kind == "paged":
        rc = lib.trt_attention_paged_kv(ctypes.byref(a), ctypes.byref(extra), h)
        name = "trt_attention_paged_kv"
    else:
        rc = lib.trt_attention(ctypes.byref(a), h)
        name = "trt_attention"
    if rc != RGA_OK:
        raise RgaError(rc, name)
    return y, status


def trt_attention(q, k, v, *, q_form="padded", kv_form="padded", query_lengths=None,
                  kv_lengths=None, mask=None, scale=1.0, causal="none", norm="softmax",
                  out=None, workspace=None, status=None, stream=None, return_status=False):
    """TRT_Attention forward.  Tensors are CUDA tensors; returns Y (and the
    device status word when ``return_status``).  ``scale`` defaults to 1.0:
    the operator itself does not scale Q/K/V."""
    y, st = _call("plain", q, k, v, out, None, stream, q_form=q_form, kv_form=kv_form,
                  query_lengths=query_lengths, kv_lengths=kv_lengths, mask=mask,
                  scale=scale, causal=causal, norm=norm, workspace=workspace, status=status)
    return (y, st) if return_status else y


def trt_quantized_attention(q, k, v, *, quant_scale, quant="fp8", q_form="padded",
                            kv_form="padded", query_lengths=None, kv_lengths=None, mask=None,
                            scale=None, causal=None, is_causal=False, norm="softmax",
                            out=None, workspace=None, status=None, stream=None,
                            return_status=False):
    """TRT_QuantizedAttention forward.  ``scale`` defaults to 1/sqrt(D);
    ``is_causal`` selects upper_left unless ``causal`` is given;
    ``quant_scale`` is a one-element CUDA tensor (fp32, fp16 or bf16)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    if causal is None:
        causal = "upper_left" if is_causal else "none"
    _need_cuda("quant_scale", quant_scale)
    y, st = _call("quant", q, k, v, out, (quant, quant_scale), stream, q_form=q_form,
                  kv_form=kv_form, query_lengths=query_lengths, kv_lengths=kv_lengths,
                  mask=mask, scale=scale, causal=causal, norm=norm, workspace=workspace,
                  status=status)
    return (y, st) if return_status else y


def trt_attention_fp8_kv(q, k, v, *, k_scale, v_scale, q_form="padded", kv_form="padded",
                         query_lengths=None, kv_lengths=None, mask=None, scale=1.0,
                         causal="none", norm="softmax", out=None, workspace=None, status=None,
                         stream=None, return_status=False):
    """Attention over an FP8 KV cache: ``k`` and ``v`` hold E4M3 codes
    (torch.float8_e4m3fn, or uint8 holding the codes), dequantised with the
    one-element fp32 CUDA tensors ``k_scale`` and ``v_scale``; ``q`` and the
    returned Y are f16 or bf16.  Every shape: decode shapes run the decode
    kernels, the others the prefill kernel."""
    for name, t in (("k", k), ("v", v)):
        if t.dtype not in FP8_CODE_DTYPES:
            raise ValueError(f"{name} must hold E4M3 codes (float8_e4m3fn or uint8)")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _need_cuda(name, t)
        if t.dtype != torch.float32 or t.numel() != 1:
            raise ValueError(f"{name} must be a one-element fp32 CUDA tensor")
    y, st = _call("fp8kv", q, k, v, out, (k_scale, v_scale), stream, q_form=q_form,
                  kv_form=kv_form, query_lengths=query_lengths, kv_lengths=kv_lengths,
                  mask=mask, scale=scale, causal=causal, norm=norm, workspace=workspace,
                  status=status)
    return (y, st) if return_status else y


def make_paged(k_pool, v_pool, page_table, *, k_scale=None, v_scale=None) -> PagedKv:
    """rga_paged_kv for device pools [num_pages, Hkv, page_size, D] and a
    device int32 page table [B, 2, max_pages_per_seq].  Pools of E4M3 codes
    (float8_e4m3fn or uint8) need k_scale and v_scale."""
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool), ("page_table", page_table)):
        _need_cuda(name, t)
    if k_pool.dim() != 4 or v_pool.shape != k_pool.shape:
        raise ValueError("k_pool and v_pool must be [num_pages, Hkv, page_size, D]")
    if page_table.dtype != torch.int32 or page_table.dim() != 3 or page_table.shape[1] != 2:
        raise ValueError("page_table must be int32 [B, 2, max_pages_per_seq]")
    pk = PagedKv()
    pk.k_pool, pk.v_pool, pk.page_table = _ptr(k_pool), _ptr(v_pool), _ptr(page_table)
    if k_pool.dtype in FP8_CODE_DTYPES:
        if k_scale is None or v_scale is None:
            raise ValueError("E4M3 pools need k_scale and v_scale")
        for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
            _need_cuda(name, t)
        pk.kv_dtype = 4
        pk.k_scale, pk.v_scale = _ptr(k_scale), _ptr(v_scale)
    else:
        pk.kv_dtype = DTYPES.get(k_pool.dtype, 99)
    pk.num_pages, pk.page_size = k_pool.shape[0], k_pool.shape[2]
    pk.max_pages_per_seq = page_table.shape[2]
    return pk


def trt_attention_paged_kv(q, k_pool, v_pool, page_table, kv_lengths, *, k_scale=None,
                           v_scale=None, q_form="padded", query_lengths=None, mask=None,
                           scale=1.0, causal="none", norm="softmax", out=None, workspace=None,
                           status=None, stream=None, return_status=False):
    """Attention over a paged KV cache: pools [num_pages, Hkv, page_size, D]
    (q's dtype, or E4M3 codes with k_scale / v_scale), an int32 page table
    [B, 2, max_pages_per_seq] (K pages, V pages) and per-sequence key counts
    kv_lengths [B].  Every shape: decode shapes run the decode kernels,
    the others the prefill kernel."""
    pk = make_paged(k_pool, v_pool, page_table, k_scale=k_scale, v_scale=v_scale)
    y, st = _call("paged", q, k_pool, v_pool, out, pk, stream, q_form=q_form,
                  kv_form="padded", query_lengths=query_lengths, kv_lengths=kv_lengths,
                  mask=mask, scale=scale, causal=causal, norm=norm, workspace=workspace,
                  status=status, batch=(page_table.shape[0]))
    return (y, st) if return_status else y


def selftest_e4m3_decode(device=None):
    """(f16 bits, bf16 bits) of all 256 E4M3 codes through the decode
    kernel's in-register conversion, as int16 CUDA tensors."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    f16 = torch.zeros(256, dtype=torch.int16, device=dev)
    bf16 = torch.zeros(256, dtype=torch.int16, device=dev)
    rc = load().rga_selftest_e4m3_decode(f16.data_ptr(), bf16.data_ptr(),
                                         c_vp(_stream_handle(None)))
    if rc != RGA_OK:
        raise RgaError(rc, "rga_selftest_e4m3_decode")
    return f16, bf16


def selftest_bounds_check(buf, index, status, stream=None) -> int:
    """One store of 1 to element `index` of the int32 CUDA tensor `buf`
    through the debug-checks build's bounds check (status 7 and no store
    when index is outside).  Returns the call's status: RGA_ERR_UNSUPPORTED
    (2) from the ordinary build."""
    return load().rga_selftest_bounds_check(buf.data_ptr(), buf.numel(), index,
                                            status.data_ptr(), c_vp(_stream_handle(stream)))


def device_status(status, stream=None) -> int:
    """Read the status word (synchronises the stream)."""
    out = c_i32(0)
    rc = load().rga_get_device_status(ctypes.c_void_p(status.data_ptr()),
                                      ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(out))
    if rc != RGA_OK:
        raise RgaError(rc, "rga_get_device_status")
    return int(out.value)


def make_kv_args(past_cache, update, y, *, update_form="padded", write_indices=None,
                 update_lengths=None, status=None) -> KvArgs:
    """rga_kv_update_args for device tensors (see include/rga.h)."""
    for name, t in (("past_cache", past_cache), ("update", update), ("y", y),
                    ("write_indices", write_indices), ("update_lengths", update_lengths),
                    ("status", status)):
        _need_cuda(name, t)
    if past_cache.dim() != 4:
        raise ValueError("past_cache must be [B, H, N, D]")
    if update.dtype != past_cache.dtype or y.dtype != past_cache.dtype:
        raise ValueError("past_cache, update and y must share one dtype")
    a = KvArgs()
    a.past_cache, a.update, a.y = _ptr(past_cache), _ptr(update), _ptr(y)
    a.dtype = 4 if past_cache.dtype == torch.uint8 else DTYPES.get(past_cache.dtype, -1)
    a.update_form = FORMS[update_form]
    B, H, N, D = past_cache.shape
    a.batch, a.heads, a.cache_seq, a.head_dim = B, H, N, D
    a.update_seq = update.shape[2] if a.update_form == 0 else update.shape[0]
    a.write_indices, a.update_lengths = _ptr(write_indices), _ptr(update_lengths)
    a.device_status = _ptr(status)
    return a


def trt_kv_cache_update(past_cache, update, *, update_form="padded", write_indices=None,
                        update_lengths=None, out=None, status=None, stream=None,
                        return_status=False):
    """TRT_KVCacheUpdate: returns Y ([B, H, N, D]).  With out=None the cache
    is updated in place and returned; otherwise Y is written to `out`."""
    lib = load()
    y = past_cache if out is None else out
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=past_cache.device)
    a = make_kv_args(past_cache, update, y, update_form=update_form, write_indices=write_indices,
                     update_lengths=update_lengths, status=status)
    rc = lib.trt_kv_cache_update(ctypes.byref(a), c_vp(_stream_handle(stream)))
    if rc != RGA_OK:
        raise RgaError(rc, "trt_kv_cache_update")
    return (y, status) if return_status else y


def make_rope_args(q, k, cos_sin, positions=None, kv_heads=None) -> RopeArgs:
    """rga_rope_args for packed rows q [T, Hq, D] and/or k [T, Hkv, D] (either
    may be None), an fp32 table cos_sin [T, R] and optional int32 positions."""
    for name, t in (("q", q), ("k", k), ("cos_sin", cos_sin), ("positions", positions)):
        _need_cuda(name, t)
    x = q if q is not None else k
    r = RopeArgs()
    r.q, r.k = _ptr(q), _ptr(k)
    r.dtype = DTYPES.get(x.dtype, 99) if x is not None else 99
    if cos_sin.dtype != torch.float32 or cos_sin.dim() != 2:
        raise ValueError("cos_sin must be fp32 [T, rotary_dim]")
    r.tokens = cos_sin.shape[0]
    r.q_heads = q.shape[1] if q is not None else 0
    r.kv_heads = k.shape[1] if k is not None else (kv_heads or 0)
    r.head_dim = x.shape[2] if x is not None else 0
    r.rotary_dim = cos_sin.shape[1]
    r.cos_sin, r.positions = _ptr(cos_sin), _ptr(positions)
    return r


def rope_apply(q=None, k=None, *, cos_sin, positions=None, stream=None):
    """Rotary position embedding in place on q [T, Hq, D] and/or k [T, Hkv, D]."""
    r = make_rope_args(q, k, cos_sin, positions)
    rc = load().rga_rope_apply(ctypes.byref(r), c_vp(_stream_handle(stream)))
    if rc != RGA_OK:
        raise RgaError(rc, "rga_rope_apply")


def trt_kv_cache_update_rope(past_cache, update, *, cos_sin, update_lengths, write_indices=None,
                             q=None, positions=None, status=None, stream=None,
                             return_status=False):
    """TRT_KVCacheUpdate of the new keys (packed update [T, H, D]) into
    past_cache in place, each written row rotated by RoPE, and q (packed
    [T, Hq, D], optional) rotated in place, in one launch."""
    lib = load()
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=past_cache.device)
    a = make_kv_args(past_cache, update, past_cache, update_form="packed",
                     write_indices=write_indices, update_lengths=update_lengths, status=status)
    r = make_rope_args(q, None, cos_sin, positions, kv_heads=past_cache.shape[1])
    r.dtype = a.dtype
    r.head_dim = past_cache.shape[3]
    rc = lib.trt_kv_cache_update_rope(ctypes.byref(a), ctypes.byref(r),
                                      c_vp(_stream_handle(stream)))
    if rc != RGA_OK:
        raise RgaError(rc, "trt_kv_cache_update_rope")
    return (past_cache, status) if return_status else past_cache

