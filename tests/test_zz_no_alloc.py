"""kvdec_gqa_decode_noalloc: the GQA decode for callers that cannot allocate
device memory (a plugin inside a runtime that owns all device memory, a
serving loop that allows no allocation while decoding).  It keeps its split
scratch in a fixed array inside the library, so these tests check, through
the C ABI, that it gives the same results as kvdec_gqa_decode with a caller
workspace and as the fp64 oracle -- on two calls in a row, the second
finding whatever the first left in the shared array -- and that problems too
big for the array are rejected with a clear error.

This file is collected last on purpose: if it fails, a run stopped at the
first failure has already run every other test."""
import ctypes

import pytest
import torch

import kvgen
from decode_attention_kv_softmax_b300 import kvdec
from parity import assert_attn_close, assert_lse_close, f64, gqa_full_oracle

pytestmark = pytest.mark.gpu


def test_matches_workspace_entry_point_on_two_calls(cuda_lib):
    cases = [
        # ragged contiguous GQA, sequences cut across CTAs
        kvgen.gqa_case(4, 32, 8, 128, seqlens=[3000, 1, 700, 4096], cap=4096, seed=71,
                       device="cuda"),
        # a different shape next: paged, d = 64, MQA-like group of 16
        kvgen.gqa_case(3, 16, 1, 64, seqlens=[90, 2000, 5], paged=True, seed=72, device="cuda"),
    ]
    for i, case in enumerate(cases):
        ref, lref = cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens, case.block_table,
                                        scale=case.scale)
        out, lse = cuda_lib.gqa_decode_noalloc(case.q, case.k, case.v, case.seqlens,
                                               case.block_table, scale=case.scale)
        torch.cuda.synchronize()
        assert_attn_close(out, f64(ref), f"call {i}")
        assert_lse_close(lse, f64(lref), f"call {i}")
        # and against the oracle, so that a defect shared by both entry
        # points cannot pass
        oref, olse = gqa_full_oracle(case)
        assert_attn_close(out, oref, f"call {i} vs oracle")
        assert_lse_close(lse, olse, f"call {i} vs oracle")


@pytest.mark.parametrize("paged,window", [(False, 0), (True, 0), (True, 300)])
def test_fp8_and_window_through_the_array(cuda_lib, paged, window):
    """The E4M3 cache and the sliding-window ring through the same entry
    point, against the oracle, with the split counters left in the array by
    the calls before (an empty sequence and one cut across many CTAs)."""
    case = kvgen.gqa_case(3, 32, 8, 128, seqlens=[0, 2600, 450], cap=2688, paged=paged,
                          seed=73 + window, device="cuda", kv_dtype="fp8", window=window)
    flag = cuda_lib.new_error_flag()
    out, lse = cuda_lib.gqa_decode_noalloc(case.q, case.k, case.v, case.seqlens, case.block_table,
                                           scale=case.scale, k_scale=case.k_scale, v_scale=case.v_scale,
                                           window=case.window, error_flag=flag, max_ctas=40)
    torch.cuda.synchronize()
    assert flag.item() == 0
    ref, lref = gqa_full_oracle(case)
    assert_attn_close(out, ref, f"fp8 paged={paged} window={window}")
    assert_lse_close(lse, lref)
    assert torch.all(out[0] == 0) and torch.isneginf(lse[0]).all()


def test_rejects_problems_beyond_the_array(cuda_lib):
    lib = kvdec.load()
    p = kvdec.GqaParams()
    # 8192 sequences x 256 KV heads: the split counters alone exceed 16 MiB
    p.batch, p.num_heads, p.num_kv_heads, p.head_dim, p.capacity = 8192, 256, 256, 128, 64
    status = lib.kvdec_gqa_decode_noalloc(ctypes.byref(p), None)
    assert status == 4
    msg = lib.kvdec_last_error().decode()
    assert "16777216" in msg and "needs" in msg
