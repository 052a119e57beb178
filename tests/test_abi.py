"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/rga.h declares, the ctypes mirror of the argument
struct has the C layout, and argument validation returns its codes without
touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

from ragged_gqa_attention_gb300 import binding
from ragged_gqa_attention_gb300 import buildlib as B

HEADER = os.path.join(B.INCLUDE, "rga.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return binding.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in binding.EXPORTED:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    for n in declared_functions():
        assert n in exported, f"{n} declared in rga.h but not exported"
        assert hasattr(lib, n)


def _layout_matches_c(tmp_path, struct, cname):
    fields = [f[0] for f in struct._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", f'#include "{HEADER}"',
            "int main(void){",
            f'printf("%zu\\n", sizeof({cname}));']
    for f in fields:
        prog.append(f'printf("%zu\\n", offsetof({cname}, {f}));')
    prog.append("return 0;}")
    c = tmp_path / f"layout_{cname}.c"
    c.write_text("\n".join(prog))
    exe = tmp_path / f"layout_{cname}"
    subprocess.check_call(["gcc", "-I", "/usr/local/cuda/include", str(c), "-o", str(exe)])
    vals = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert vals[0] == ctypes.sizeof(struct)
    for f, off in zip(fields, vals[1:]):
        assert getattr(struct, f).offset == off, f


def test_struct_layout_matches_c(tmp_path):
    _layout_matches_c(tmp_path, binding.Args, "rga_attention_args")


def test_kv_update_struct_layout_matches_c(tmp_path):
    _layout_matches_c(tmp_path, binding.KvArgs, "rga_kv_update_args")


def test_status_strings_and_version(lib):
    assert lib.rga_abi_version() == 1
    for code, name in binding.STATUS_NAMES.items():
        assert lib.rga_status_string(code).decode() == name


def _args(**kw):
    a = binding.Args()
    a.q = a.k = a.v = a.y = 0x10000
    a.dtype, a.q_form, a.kv_form = 1, 0, 0
    a.batch, a.q_heads, a.kv_heads, a.head_dim = 2, 8, 2, 128
    a.q_seq, a.kv_seq = 256, 256
    a.scale, a.causal, a.norm, a.nb_rank = 1.0, 0, 0, 1
    a.device_status = 0x20000
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(q_heads=6, kv_heads=4), 1),          # heads not a multiple
    (dict(head_dim=96), 2),                    # not implemented
    (dict(dtype=2), 2),                        # fp32 Q/K/V not implemented
    (dict(nb_rank=2), 2),                      # single device only
    (dict(causal=7), 1),
    (dict(q_form=1), 1),                       # packed Q needs query_lengths
    (dict(kv_form=1), 1),                      # packed KV needs kv_lengths
    (dict(q=0x10008), 1),                      # misaligned
    (dict(device_status=None), 1),
    (dict(mask=0x30000, mask_dtype=3, mask_rank=2, causal=1), 1),   # mask + causal
    (dict(mask=0x30000, mask_dtype=3, mask_rank=4), 1),             # mask dims 0
])
def test_validation_codes_without_a_device(lib, kw, code):
    a = _args(**kw)
    if "mask_rank" in kw and kw["mask_rank"] == 2:
        a.mask_dims[0], a.mask_dims[1] = 256, 256
    rc = lib.trt_attention(ctypes.byref(a), None)
    assert rc == code


def test_workspace_missing_is_reported(lib):
    a = _args()
    assert lib.trt_attention(ctypes.byref(a), None) == 6
    n = lib.rga_attention_workspace_size(ctypes.byref(a))
    assert n >= 256 and n % 256 == 0


def test_quantized_requires_scale(lib):
    a = _args(workspace=0x100000, workspace_bytes=1 << 30)
    assert lib.trt_quantized_attention(ctypes.byref(a), 0, None, 2, None) == 1
    assert lib.trt_quantized_attention(ctypes.byref(a), 5, 0x40000, 2, None) == 1


def test_python_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 2, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        binding.trt_attention(q, q, q)


def _kv_args(**kw):
    a = binding.KvArgs()
    a.past_cache = a.update = a.y = 0x10000
    a.dtype, a.update_form = 1, 0
    a.batch, a.heads, a.cache_seq, a.head_dim, a.update_seq = 2, 8, 64, 128, 4
    a.device_status = 0x20000
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(past_cache=None), 1),
    (dict(update=None), 1),
    (dict(y=None), 1),
    (dict(device_status=None), 1),
    (dict(dtype=3), 1),                  # element type outside F16/BF16/F32
    (dict(update_form=5), 1),
    (dict(batch=-1), 1),
    (dict(head_dim=0), 1),
    (dict(update_form=1), 1),            # packed update needs update_lengths
    (dict(batch=9000), 2),               # more batches than the kernel lists
])
def test_kv_update_validation_codes_without_a_device(lib, kw, code):
    a = _kv_args(**kw)
    assert lib.trt_kv_cache_update(ctypes.byref(a), None) == code


def test_selftest_validates_its_arguments(lib):
    assert lib.rga_selftest_wait_timeout(None, 1000, None) == 1
    assert lib.rga_selftest_wait_timeout(0x20000, 0, None) == 1
    assert lib.rga_selftest_wait_timeout(0x20000, (1 << 32) + 1, None) == 1


def test_fp8_kv_validation_without_a_device(lib):
    a = _args(workspace=0x100000, workspace_bytes=1 << 30)
    assert lib.trt_attention_fp8_kv(ctypes.byref(a), None, 0x40000, None) == 1   # k_scale
    assert lib.trt_attention_fp8_kv(ctypes.byref(a), 0x40000, None, None) == 1   # v_scale
    # prefill shapes (256 query rows per sequence) pass validation and go to
    # the prefill kernel: with no device here, the launch set-up fails
    assert lib.trt_attention_fp8_kv(ctypes.byref(a), 0x40000, 0x40010, None) == 3
    # argument errors come first, as for trt_attention
    a = _args(q_heads=6, kv_heads=4)
    assert lib.trt_attention_fp8_kv(ctypes.byref(a), 0x40000, 0x40010, None) == 1


def test_fp8_codes_are_a_kv_update_element_type(lib):
    # E4M3 codes move as bytes: an odd head dim is valid (1-byte moves)
    a = _kv_args(dtype=4, head_dim=3)
    a.batch = 0            # nothing to move: validation only, no launch
    assert lib.trt_kv_cache_update(ctypes.byref(a), None) == 0



def test_e4m3_selftest_validates_its_arguments(lib):
    assert lib.rga_selftest_e4m3_decode(None, 0x20000, None) == 1
    assert lib.rga_selftest_e4m3_decode(0x20000, None, None) == 1


def test_paged_kv_validation_without_a_device(lib):
    def paged(**kw):
        pk = binding.PagedKv()
        pk.k_pool = pk.v_pool = 0x50000
        pk.kv_dtype = 1
        pk.page_table = 0x60000
        pk.num_pages, pk.page_size, pk.max_pages_per_seq = 16, 64, 8
        for k, v in kw.items():
            setattr(pk, k, v)
        return pk
    # one token per sequence (decode shape), padded KV with per-batch lengths
    a = _args(q_seq=1, kv_lengths=0x70000, workspace=0x100000, workspace_bytes=1 << 30)
    call = lambda a, pk: lib.trt_attention_paged_kv(ctypes.byref(a), ctypes.byref(pk), None)
    assert call(a, paged(page_size=48)) == 1            # not a multiple of 32
    assert call(a, paged(page_size=0)) == 1
    assert call(a, paged(k_pool=None)) == 1
    assert call(a, paged(page_table=None)) == 1
    assert call(a, paged(num_pages=0)) == 1
    assert call(a, paged(kv_dtype=0)) == 1              # neither Q's dtype nor E4M3
    assert call(a, paged(kv_dtype=4)) == 1              # E4M3 pools without scales
    assert call(_args(q_seq=1, kv_form=1, kv_lengths=0x70000), paged()) == 1   # packed KV
    assert call(_args(q_seq=1), paged()) == 1           # kv_lengths required
    # 256 query rows: a prefill shape, accepted (no device here: launch set-up fails)
    assert call(_args(kv_lengths=0x70000, workspace=0x100000, workspace_bytes=1 << 30),
                paged()) == 3


def test_rope_validation_without_a_device(lib):
    def rope(**kw):
        r = binding.RopeArgs()
        r.q = 0x10000
        r.dtype, r.tokens, r.q_heads, r.kv_heads, r.head_dim, r.rotary_dim = 1, 8, 4, 2, 128, 128
        r.cos_sin = 0x20000
        for k, v in kw.items():
            setattr(r, k, v)
        return r
    call = lambda r: lib.rga_rope_apply(ctypes.byref(r), None)
    assert call(rope(rotary_dim=12)) == 1        # not a multiple of 8
    assert call(rope(rotary_dim=136)) == 1       # past the head dim
    assert call(rope(head_dim=66)) == 1
    assert call(rope(cos_sin=None)) == 1
    assert call(rope(cos_sin=0x20008)) == 1      # table not 16-byte aligned
    assert call(rope(q=None)) == 1               # nothing to rotate
    assert call(rope(q=0x10004)) == 1            # rows not 8-byte aligned
    assert call(rope(dtype=2)) == 1
    assert call(rope(tokens=0)) == 0             # nothing to do, nothing launched
    kv = _kv_args(update_form=1, update_lengths=0x30000, update_seq=8, heads=2)
    fused = lambda a, r: lib.trt_kv_cache_update_rope(ctypes.byref(a), ctypes.byref(r), None)
    assert fused(_kv_args(update_form=0, heads=2, update_seq=8), rope()) == 1   # padded update
    assert fused(_kv_args(update_form=1, update_lengths=0x30000, update_seq=8, heads=2,
                          y=0x40000), rope()) == 1                              # not in place
    assert fused(_kv_args(update_form=1, update_lengths=0x30000, update_seq=8, heads=4),
                 rope()) == 1                                                    # heads differ
    assert fused(kv, rope(dtype=0)) == 1                                         # dtypes differ



def test_fp8_and_paged_report_a_small_workspace_before_any_device_work(lib):
    # one token per sequence: a decode shape; the workspace is checked after
    # the arguments and before anything is enqueued
    a = _args(q_seq=1, kv_lengths=0x70000)
    need = lib.rga_attention_workspace_size(ctypes.byref(a))
    assert need >= 256 and need % 256 == 0
    a.workspace, a.workspace_bytes = 0x100000, need - 256
    assert lib.trt_attention_fp8_kv(ctypes.byref(a), 0x40000, 0x40010, None) == 6
    pk = binding.PagedKv()
    pk.k_pool = pk.v_pool = 0x50000
    pk.kv_dtype = 1
    pk.page_table = 0x60000
    pk.num_pages, pk.page_size, pk.max_pages_per_seq = 16, 64, 4
    a.kv_seq = 4 * 64
    need = lib.rga_attention_workspace_size(ctypes.byref(a))
    a.workspace_bytes = need - 256
    assert lib.trt_attention_paged_kv(ctypes.byref(a), ctypes.byref(pk), None) == 6
    a.workspace = 0x100010          # not 256-byte aligned
    a.workspace_bytes = need
    assert lib.trt_attention_paged_kv(ctypes.byref(a), ctypes.byref(pk), None) == 6


def test_decode_pairs_take_sixteen_rows_past_eight_rows_per_kv_head(lib):
    # a (batch, KV head) with more than 8 query rows takes pairs of 16 rows
    # (two N-blocks) on a 16-bit cache: the partial slots of the workspace
    # double.  Padded Q, 2 KV heads: 16 query heads (G = 8) with 1 token and
    # 8 (G = 4) with 2 tokens are 8 rows; 16 heads with 2 tokens and 8 with 3
    # are 16 and 12 rows.  (The fp8 layout, also sized by the query, keeps 8.)
    def need(q_seq, q_heads):
        return lib.rga_attention_workspace_size(ctypes.byref(_args(q_seq=q_seq, q_heads=q_heads)))
    eight = need(1, 16)
    assert eight == need(2, 8)
    slot_rows = 16 * 8 * 128 * 4   # at least 16 slots of 8 more rows of 128 fp32 dims
    assert need(2, 16) - eight >= slot_rows
    assert need(3, 8) - eight >= slot_rows
