"""The decode entry points captured in a CUDA graph and replayed: the split
counters carry the call's epoch, which a captured launch keeps on every
replay, so the last piece of each split unit must return its counter to
zero for the next replay to merge again.  Checked for GQA and MLA against
the eager call and the oracle, over several replays."""
import pytest
import torch

import kvgen
from parity import assert_attn_close, assert_lse_close, f64, gqa_full_oracle, mla_full_oracle

pytestmark = pytest.mark.gpu

REPLAYS = 3


def capture(fn):
    """Eager warm-up call (the library's per-thread memos fill there), then
    one captured call; returns the graph and the captured outputs."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            res = fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g, res


def test_gqa_decode_replays(cuda_lib):
    # sequences cut across many CTAs: every unit has several pieces
    case = kvgen.gqa_case(3, 32, 8, 128, seqlens=[4000, 700, 2500], cap=4096, seed=81, device="cuda")
    run = lambda: cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens, scale=case.scale,
                                      max_ctas=40)
    g, (out, lse) = capture(run)
    ref, lref = gqa_full_oracle(case)
    for r in range(REPLAYS):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_attn_close(out, ref, f"replay {r}")
        assert_lse_close(lse, lref, f"replay {r}")


def test_mla_decode_replays(cuda_lib):
    case = kvgen.mla_case(3, 128, seqlens=[2500, 640, 1800], seed=82, device="cuda")
    run = lambda: cuda_lib.mla_decode_absorbed(case.q_abs, case.q_rope, case.cache, case.block_table,
                                               case.seqlens, scale=case.scale, max_ctas=10)
    g, (out, lse) = capture(run)
    ref, lref = mla_full_oracle(case)
    for r in range(REPLAYS):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_attn_close(out, ref, f"replay {r}")
        assert_lse_close(lse, lref, f"replay {r}")


def test_mla_fp8_decode_replays(cuda_lib):
    """The E4M3 latent cache: the widening pass and the decode captured
    together; between replays the cache's codes change, and every replay
    widens the new codes (the copy is rewritten, not reused)."""
    case = kvgen.mla_case(3, 128, seqlens=[2500, 640, 1800], seed=83, device="cuda", kv_dtype="fp8")
    run = lambda: cuda_lib.mla_decode_absorbed(case.q_abs, case.q_rope, case.cache, case.block_table,
                                               case.seqlens, scale=case.scale, max_ctas=10,
                                               kv_scale=case.kv_scale)
    g, (out, lse) = capture(run)
    gen = torch.Generator(device="cuda").manual_seed(84)
    for r in range(REPLAYS):
        if r > 0:   # new codes in place (same tensor the graph reads)
            x = torch.randn(case.cache.shape, generator=gen, device="cuda").to(torch.bfloat16)
            case.cache.copy_(kvgen.mla_fp8_codes(x, gen, "cuda")[0])
        ref, lref = mla_full_oracle(case)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_attn_close(out, ref, f"replay {r}")
        assert_lse_close(lse, lref, f"replay {r}")


def test_gqa_fp8_window_replays(cuda_lib):
    case = kvgen.gqa_case(2, 32, 8, 128, seqlens=[3000, 700], paged=True, seed=85, device="cuda",
                          kv_dtype="fp8", window=512)
    run = lambda: cuda_lib.gqa_decode(case.q, case.k, case.v, case.seqlens, case.block_table,
                                      scale=case.scale, k_scale=case.k_scale, v_scale=case.v_scale,
                                      window=case.window, max_ctas=24)
    g, (out, lse) = capture(run)
    ref, lref = gqa_full_oracle(case)
    for r in range(REPLAYS):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_attn_close(out, ref, f"replay {r}")
        assert_lse_close(lse, lref, f"replay {r}")
