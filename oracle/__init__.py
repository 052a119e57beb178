"""Plain fp64 CPU oracle for ragged GQA attention (test infrastructure only).

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, loads or calls it, and it imports nothing
from the product package.

What it computes is the plain definition of the fused attention forward of the
"TensorRT Custom Operator Schemas" page (TRT_Attention and
TRT_QuantizedAttention sections), for every query row:

    A     = keys j < kv_len allowed by the causal kind and the bool mask
    s_j   = scale * <q_i, k_j> + additive_mask(i, j)
    p     = softmax over A  (or p_j = s_j on A for normalization op 'none')
    p     = s_q * Q(p / s_q)            (quantized op only; fp8 E4M3FN or int8)
    y_i   = sum_{j in A} p_j v_j

in double precision from the stored fp16/bf16 input values.  For an FP8 KV
cache ("TensorRT Plugins Guide", AttentionPlugin: kv_cache_type FP8) the
keys and values are first dequantised: decoded E4M3FN code times the
tensor's scale (``dequant_e4m3``, ``attention(..., kv_fp8_scales=...)``).  The arithmetic
lives in ``rga_oracle.c`` (compiled with gcc on first use); this module only
marshals arrays.

Parity pins for every function here live in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rga_oracle.c")
_LIB_PATH = os.path.join(_HERE, "librga_oracle.so")
_lib = None
_lock = threading.Lock()

PADDED, PACKED = 0, 1
CAUSAL = {"none": 0, "upper_left": 1, "lower_right": 2}
NORM = {"softmax": 0, "none": 1}
QUANT = {None: -1, "fp8": 0, "int8": 1}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (host code only, no CUDA)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call([
            "gcc", "-O2", "-std=c99", "-D_GNU_SOURCE", "-shared", "-fPIC",
            "-o", tmp, _SRC, "-lpthread", "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.c_double
            p = ctypes.c_void_p
            i = ctypes.c_int
            lib.rga_oracle_attention.restype = i
            lib.rga_oracle_attention.argtypes = [
                p, p, p, p, i, i, i, i, i, i, i, i, p, p, p, p, p,
                d, i, i, i, d, i, p, d]
            lib.rga_oracle_e4m3_decode.restype = d
            lib.rga_oracle_e4m3_decode.argtypes = [i]
            lib.rga_oracle_e4m3_round.restype = d
            lib.rga_oracle_e4m3_round.argtypes = [d]
            lib.rga_oracle_e4m3_encode.restype = i
            lib.rga_oracle_e4m3_encode.argtypes = [d]
            lib.rga_oracle_e4m3_dequant.restype = None
            lib.rga_oracle_e4m3_dequant.argtypes = [p, ctypes.c_long, d, p]
            lib.rga_oracle_int8_round.restype = d
            lib.rga_oracle_int8_round.argtypes = [d]
            _lib = lib
    return _lib


def _f64(x):
    """Exact float64 copy of a torch tensor or array (stored values)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def torch_bool():
    import torch
    return torch.bool


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__(f"oracle rejected the arguments (code {code})")
        self.code = code


def attention(q, k, v, *, q_form="padded", kv_form="padded", query_lengths=None,
              kv_lengths=None, mask=None, scale=1.0, causal="none",
              norm="softmax", quant=None, quant_scale=None, y_init=None,
              nthreads=None, ambiguity_eps=None, kv_fp8_scales=None):
    """Plain fp64 attention.  Returns a float64 array shaped like ``q``.

    q: padded [B,Hq,Nq,D] or packed [Tq,Hq,D]; k, v likewise for KV.
    query_lengths: [B+1] cumulative (required for packed q; optional for padded
    q, where its differences give the valid rows of each batch).
    kv_lengths: [B+1] cumulative for packed KV, [B] per-batch for padded KV.
    mask: None, a bool array (True = may attend) or a float array (added to
    the scaled scores), rank <= 4, right-aligned to [B, Hq, Nq, Nkv].
    quant: None, 'fp8' or 'int8'; quant_scale the stored scale value.
    Rows that are not valid query rows keep ``y_init`` (default NaN).
    kv_fp8_scales: (k_scale, v_scale) when k and v hold E4M3FN codes (uint8
    or float8_e4m3fn tensors / uint8 arrays): they are dequantised first.
    With ``ambiguity_eps`` (quantized op), returns ``(y, amb)``: amb bounds
    how far a quantised code within relative ``ambiguity_eps`` of a rounding
    midpoint may move each output element if it rounds the other way.
    """
    lib = _load()
    qf = PACKED if q_form in ("packed", "packed_nhd", PACKED) else PADDED
    kf = PACKED if kv_form in ("packed", "packed_nhd", PACKED) else PADDED
    if kv_fp8_scales is not None:
        K, V = dequant_e4m3(k, kv_fp8_scales[0]), dequant_e4m3(v, kv_fp8_scales[1])
    else:
        K, V = _f64(k), _f64(v)
    Q = _f64(q)
    D = Q.shape[-1]
    Hq = Q.shape[-2] if qf == PACKED else Q.shape[1]
    Hkv = K.shape[-2] if kf == PACKED else K.shape[1]
    q_seq = Q.shape[0] if qf == PACKED else Q.shape[2]
    kv_seq = K.shape[0] if kf == PACKED else K.shape[2]
    ql, kl = _i32(query_lengths), _i32(kv_lengths)
    if qf == PACKED:
        B = len(ql) - 1
    elif kf == PACKED:
        B = len(kl) - 1
    else:
        B = Q.shape[0]
    Y = np.full(Q.shape, np.nan) if y_init is None else _f64(y_init).copy()
    madd = mbool = None
    mdims = np.ones(4, dtype=np.int64)
    if mask is not None:
        if hasattr(mask, "detach"):   # torch: bool stays bool, others widen exactly
            mask = mask.detach().cpu()
            m = mask.numpy() if mask.dtype == torch_bool() else mask.double().numpy()
        else:
            m = np.asarray(mask)
        assert m.ndim <= 4
        mdims[4 - m.ndim:] = m.shape
        if m.dtype == np.bool_:
            mbool = np.ascontiguousarray(m.astype(np.uint8))
        else:
            madd = np.ascontiguousarray(m.astype(np.float64))
    qs = 1.0 if quant_scale is None else float(_f64(quant_scale).reshape(-1)[0])
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    amb = np.zeros(Q.shape) if ambiguity_eps is not None else None
    rc = lib.rga_oracle_attention(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(Y), qf, kf, B, Hq, Hkv, D, q_seq,
        kv_seq, _ptr(ql), _ptr(kl), _ptr(madd), _ptr(mbool), _ptr(mdims),
        float(scale), CAUSAL[causal], NORM[norm], QUANT[quant], qs,
        int(nthreads), _ptr(amb), float(ambiguity_eps or 0.0))
    if rc != 0:
        raise OracleError(rc)
    return Y if amb is None else (Y, amb)



def _codes(x):
    """uint8 numpy copy of E4M3 codes (uint8 / float8_e4m3fn tensor or array)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu()
        if x.dtype != torch.uint8:
            x = x.view(torch.uint8)
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.uint8))


def dequant_e4m3(codes, scale):
    """fp64 values of an FP8 KV cache tensor: decoded code times ``scale``
    (a float or a one-element tensor holding the stored fp32 scale)."""
    c = _codes(codes)
    s = float(_f64(scale).reshape(-1)[0]) if hasattr(scale, "detach") or isinstance(
        scale, np.ndarray) else float(scale)
    out = np.empty(c.shape, dtype=np.float64)
    _load().rga_oracle_e4m3_dequant(_ptr(c), c.size, s, _ptr(out))
    return out


def e4m3_decode(code: int) -> float:
    return _load().rga_oracle_e4m3_decode(int(code))


def e4m3_round(x: float) -> float:
    return _load().rga_oracle_e4m3_round(float(x))


def e4m3_encode(x: float) -> int:
    return _load().rga_oracle_e4m3_encode(float(x))


def int8_round(x: float) -> float:
    return _load().rga_oracle_int8_round(float(x))


def gather_pages(pool, page_table, which, kv_lens, pad=None):
    """The linear cache [B, H, N, D] (N = max_pages * page_size) of a paged
    KV pool ("TensorRT Plugins Guide", AttentionPlugin: kv_page_table
    [N, 2, max_pages_per_sequence]): key n < kv_lens[b] of batch b is row
    n % page_size of page page_table[b, which, n // page_size] of
    pool [num_pages, H, page_size, D]; which = 0 for K, 1 for V.  Rows past
    kv_lens[b] hold ``pad`` (default NaN, or the NaN code 0x7F for uint8 /
    float8 codes) and page entries past a sequence's last page are not read.
    Index work only: the element bits are copied unchanged (torch tensors in,
    a torch tensor of the pool's dtype out)."""
    import torch
    pool = pool.detach().cpu()
    pt = page_table.detach().cpu()
    B, mp = pt.shape[0], pt.shape[2]
    _, H, ps, D = pool.shape
    codes = pool.dtype in (torch.uint8, torch.float8_e4m3fn)
    out = torch.empty((B, H, mp * ps, D), dtype=pool.dtype)
    if codes:
        out.view(torch.uint8).fill_(0x7F if pad is None else int(pad))
    else:
        out.fill_(float("nan") if pad is None else float(pad))
    for b in range(B):
        n = int(kv_lens[b])
        for i in range((n + ps - 1) // ps):
            rows = min(ps, n - i * ps)
            out[b, :, i * ps:i * ps + rows] = pool[int(pt[b, which, i]), :, :rows]
    return out


# TRT_KVCacheUpdate (a plain scatter; see kv_update.py)
from .kv_update import kv_cache_update  # noqa: E402,F401
# rotary position embedding (see rope.py)
from .rope import rope  # noqa: E402,F401
