"""The C-ABI library loads, exports every function include/kvdec.h declares,
and agrees with the binding's struct mirrors.  Host-side argument checks are
exercised on calls that are rejected before any CUDA work (no GPU here)."""
import ctypes
import os
import re

import pytest

from decode_attention_kv_softmax_b300 import build, kvdec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kvdec.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvdec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvdec_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(kvdec.EXPORTS)


def test_struct_layouts(lib):
    assert lib.kvdec_abi_version() == kvdec.ABI_VERSION == 3
    for kind, st in enumerate([kvdec.GqaParams, kvdec.MlaParams, kvdec.AppendParams,
                               kvdec.CombineParams, kvdec.MlaProjParams, kvdec.MlaExpandParams,
                               kvdec.MlaPrefillParams]):
        assert lib.kvdec_params_size(kind) == ctypes.sizeof(st)
    assert lib.kvdec_params_size(99) == -1


def test_status_strings(lib):
    for s, txt in kvdec.STATUS.items():
        assert lib.kvdec_status_string(s).decode() == txt


def test_host_argument_checks(lib):
    # rejected before touching the device
    assert lib.kvdec_gqa_decode(None, None) == 1
    p = kvdec.GqaParams()
    p.batch, p.num_heads, p.num_kv_heads, p.head_dim = 2, 8, 3, 128
    assert lib.kvdec_gqa_decode(ctypes.byref(p), None) == 1
    assert "multiple" in lib.kvdec_last_error().decode()
    p.num_kv_heads, p.head_dim = 2, 96
    assert lib.kvdec_gqa_decode(ctypes.byref(p), None) == 2
    assert lib.kvdec_gqa_workspace_bytes(ctypes.byref(p)) == 0
    p.head_dim, p.batch = 128, 0
    assert lib.kvdec_gqa_decode(ctypes.byref(p), None) == 1
    c = kvdec.CombineParams()
    assert lib.kvdec_combine_splits(ctypes.byref(c), None) == 1
    a = kvdec.AppendParams()
    a.batch = 1
    assert lib.kvdec_append_rope(ctypes.byref(a), None) == 1
    a.mode = 7
    a.seqlens = 16
    assert lib.kvdec_append_rope(ctypes.byref(a), None) == 1
    m = kvdec.MlaParams()
    assert lib.kvdec_mla_decode_absorbed(ctypes.byref(m), None) != 0
    assert lib.kvdec_selftest_wait_timeout(1000, None, None) == 1


def test_projection_argument_checks(lib):
    """The MLA projections reject bad arguments before any launch."""
    assert lib.kvdec_mla_absorb_q(None, None) == 1
    p = kvdec.MlaProjParams()
    assert lib.kvdec_mla_project_out(ctypes.byref(p), None) == 1
    assert "non-NULL" in lib.kvdec_last_error().decode()
    p.x, p.w, p.y = 256, 512, 1024          # aligned, never dereferenced on the host
    p.batch, p.num_heads, p.out_dtype = 0, 128, kvdec.F32
    assert lib.kvdec_mla_absorb_q(ctypes.byref(p), None) == 1
    assert "batch" in lib.kvdec_last_error().decode()
    p.batch, p.out_dtype = 4, 7
    assert lib.kvdec_mla_project_out(ctypes.byref(p), None) == 1
    assert "out_dtype" in lib.kvdec_last_error().decode()
    p.out_dtype, p.x = kvdec.F32, 257
    assert lib.kvdec_mla_absorb_q(ctypes.byref(p), None) == 1
    assert "aligned" in lib.kvdec_last_error().decode()


def test_fp8_and_window_argument_checks(lib):
    """FP8 cache and sliding-window arguments that are rejected on the host
    before any device query."""
    p = kvdec.GqaParams()
    p.batch, p.num_heads, p.num_kv_heads, p.head_dim = 2, 8, 2, 64
    p.kv_format = kvdec.KV_FP8_E4M3
    assert lib.kvdec_gqa_decode(ctypes.byref(p), None) == 2       # FP8 needs head_dim 128
    assert "FP8" in lib.kvdec_last_error().decode()
    p.kv_format = 5
    assert lib.kvdec_gqa_decode(ctypes.byref(p), None) == 1
    assert "kv_format" in lib.kvdec_last_error().decode()
    p.kv_format, p.head_dim, p.window = kvdec.KV_BF16, 128, -1
    assert lib.kvdec_gqa_decode(ctypes.byref(p), None) == 1
    assert "window" in lib.kvdec_last_error().decode()
    assert lib.kvdec_gqa_workspace_bytes(ctypes.byref(p)) == 0
    a = kvdec.AppendParams()
    a.mode, a.batch, a.seqlens = kvdec.APPEND_MLA, 1, 16
    a.window = 8
    assert lib.kvdec_append_rope(ctypes.byref(a), None) == 2      # MLA takes no window
    a.mode, a.window = kvdec.APPEND_GQA, 0
    a.k_new, a.v_new, a.k, a.v = 256, 512, 1024, 2048
    a.num_kv_heads, a.head_dim, a.capacity = 2, 128, 64
    a.kv_format = kvdec.KV_FP8_E4M3                                # no scales
    assert lib.kvdec_append_rope(ctypes.byref(a), None) == 1
    assert "k_scale" in lib.kvdec_last_error().decode()
    a.kv_format, a.window = kvdec.KV_BF16, 65                      # more than the 64 slots
    assert lib.kvdec_append_rope(ctypes.byref(a), None) == 1
    assert "window" in lib.kvdec_last_error().decode()


def test_prefill_argument_checks(lib):
    """The prefill entry points reject bad arguments before any launch."""
    assert lib.kvdec_mla_prefill(None, None) == 1
    assert lib.kvdec_mla_prefill_expand(None, None) == 1
    p = kvdec.MlaPrefillParams()
    p.q_nope, p.q_rope, p.k_nope, p.k_rope, p.v, p.out = 256, 512, 768, 1024, 1280, 1536
    p.s_q, p.s_kv, p.num_heads, p.kv_offset = 8, 4, 128, -1      # chunk longer than the keys
    assert lib.kvdec_mla_prefill(ctypes.byref(p), None) == 1
    assert "s_kv" in lib.kvdec_last_error().decode()
    p.s_kv, p.kv_offset = 16, 9                                   # 9 + 8 > 16
    assert lib.kvdec_mla_prefill(ctypes.byref(p), None) == 1
    p.kv_offset, p.out_dtype = 8, 7
    assert lib.kvdec_mla_prefill(ctypes.byref(p), None) == 1
    p.out_dtype, p.scale = kvdec.F32, -1.0
    assert lib.kvdec_mla_prefill(ctypes.byref(p), None) == 1
    p.scale, p.k_rope = 0.0, 1025                                 # misaligned
    assert lib.kvdec_mla_prefill(ctypes.byref(p), None) == 1
    e = kvdec.MlaExpandParams()
    e.c_kv, e.w_uk, e.w_uv, e.k_nope, e.v = 256, 512, 768, 1024, 1280
    e.s, e.num_heads = 0, 128
    assert lib.kvdec_mla_prefill_expand(ctypes.byref(e), None) == 1


def test_mla_batch_limit(lib):
    """The MLA decode keeps a tile table of batch + 1 ints in shared memory
    beside five 36 KB cache stages, the 16 KB exchange and P buffers, the
    8 KB rope part of Q and a 4 KB hand-off; the largest batch that fits in
    the 227 KB a CTA may use is the limit (411), and one more sequence is
    rejected on the host (INVALID_ARG) before any device query."""
    limit = lib.kvdec_mla_max_batch()
    assert limit == 411
    m = kvdec.MlaParams()
    m.num_heads, m.num_pages, m.max_blocks = 128, 4, 4
    m.batch = limit + 1
    assert lib.kvdec_mla_decode_absorbed(ctypes.byref(m), None) == 1
    assert f"outside [1, {limit}]" in lib.kvdec_last_error().decode()
    assert lib.kvdec_mla_workspace_bytes(ctypes.byref(m)) == 0
    m.batch = limit                  # passes the batch check; no device here
    st = lib.kvdec_mla_decode_absorbed(ctypes.byref(m), None)
    assert st != 1 or "batch" not in lib.kvdec_last_error().decode()
