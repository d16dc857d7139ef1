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
