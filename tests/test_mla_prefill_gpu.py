"""GPU parity of the non-absorbed MLA prefill: kvdec_mla_prefill_expand
(up-projection) and kvdec_mla_prefill (causal attention, head dims 192 / 128)
against the fp64 oracle, through the C ABI ([ARG]
"attention-variants-and-kv-cache" §四.6)."""
import numpy as np
import pytest
import torch

import kvgen
import oracle
from parity import assert_attn_close, assert_lse_close, f64

pytestmark = pytest.mark.gpu


def case(s_kv, s_q, n_h, seed):
    c = kvgen.mla_prefill_case(s_kv, s_q, n_h, seed=seed, device="cuda")
    return c


@pytest.mark.parametrize("s,n_h", [(1, 2), (100, 4), (257, 128)])
def test_expand_parity(cuda_lib, s, n_h):
    c = case(s, 1, n_h, 40 + s)
    k_nope, v = cuda_lib.mla_prefill_expand(c["c_kv"], c["W_UK"], c["W_UV"])
    torch.cuda.synchronize()
    kr, vr = oracle.mla_prefill_expand(f64(c["c_kv"]), f64(c["W_UK"]), f64(c["W_UV"]))
    assert_attn_close(k_nope, kr, "k_nope")
    assert_attn_close(v, vr, "v")


SHAPES = [
    # s_kv, s_q, n_h, kv_offset
    (64, 64, 2, -1),          # one full tile, square causal
    (130, 130, 2, -1),        # ragged tail, three tiles
    (300, 77, 3, -1),         # chunk of the newest 77 tokens
    (300, 77, 3, 100),        # chunk in the middle of the keys
    (65, 1, 128, -1),         # one query: a decode step on the literal path
    (1000, 200, 4, -1),
    (513, 513, 1, -1),
    (700, 384, 2, 200),       # odd query-block count with an offset: pairs with a lone tail tile, an idle partner
]


@pytest.mark.parametrize("s_kv,s_q,n_h,off", SHAPES)
def test_prefill_attention_parity(cuda_lib, s_kv, s_q, n_h, off):
    """The attention kernel on the device's own up-projected K/V."""
    c = case(s_kv, s_q, n_h, 50 + s_kv + s_q)
    k_nope, v = cuda_lib.mla_prefill_expand(c["c_kv"], c["W_UK"], c["W_UV"])
    out, lse = cuda_lib.mla_prefill(c["q_nope"], c["q_rope"], k_nope, c["k_rope"], v, kv_offset=off)
    torch.cuda.synchronize()
    ref, lref = oracle.mla_prefill(f64(c["q_nope"]), f64(c["q_rope"]), f64(k_nope), f64(c["k_rope"]),
                                   f64(v), kv_offset=None if off < 0 else off)
    assert_attn_close(out, ref, "out")
    assert_lse_close(lse, lref, "lse")


def test_prefill_repeatable(cuda_lib):
    """Two launches on the same inputs agree bit for bit: paired query blocks
    share K/V tiles through multicast loads and joint stage releases, and a
    slip in that hand-off would show up as run-to-run differences."""
    s_kv, s_q, n_h = 2048, 1920, 8
    c = case(s_kv, s_q, n_h, 83)
    k_nope, v = cuda_lib.mla_prefill_expand(c["c_kv"], c["W_UK"], c["W_UV"])
    o1, l1 = cuda_lib.mla_prefill(c["q_nope"], c["q_rope"], k_nope, c["k_rope"], v)
    o2, l2 = cuda_lib.mla_prefill(c["q_nope"], c["q_rope"], k_nope, c["k_rope"], v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_prefill_end_to_end_and_bf16_out(cuda_lib):
    """Expand + attention against the oracle's own fp64 up-projection."""
    s_kv, s_q, n_h = 200, 150, 4
    c = case(s_kv, s_q, n_h, 61)
    k_nope, v = cuda_lib.mla_prefill_expand(c["c_kv"], c["W_UK"], c["W_UV"])
    out, lse = cuda_lib.mla_prefill(c["q_nope"], c["q_rope"], k_nope, c["k_rope"], v,
                                    out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    kr, vr = oracle.mla_prefill_expand(f64(c["c_kv"]), f64(c["W_UK"]), f64(c["W_UV"]))
    ref, lref = oracle.mla_prefill(f64(c["q_nope"]), f64(c["q_rope"]), kr, f64(c["k_rope"]), vr)
    assert_attn_close(out, ref, "out")
    assert_lse_close(lse, lref, "lse")


def test_prefill_full_size_sampled(cuda_lib):
    """DeepSeek-V3-shaped chunk: 4096 tokens, 128 heads, causal; sampled
    (row, head) pairs against the oracle row by row."""
    s, n_h = 4096, 128
    c = case(s, s, n_h, 71)
    k_nope, v = cuda_lib.mla_prefill_expand(c["c_kv"], c["W_UK"], c["W_UV"])
    out, lse = cuda_lib.mla_prefill(c["q_nope"], c["q_rope"], k_nope, c["k_rope"], v)
    torch.cuda.synchronize()
    g = np.random.default_rng(5)
    rows = [(int(i), int(h)) for i, h in zip(g.integers(0, s, 40), g.integers(0, n_h, 40))] + [(0, 0), (s - 1, 127), (63, 5), (64, 5)]
    kr = f64(c["k_rope"])
    for i, h in rows:
        K = np.concatenate([f64(k_nope[: i + 1, h]), kr[: i + 1]], axis=1)
        q = np.concatenate([f64(c["q_nope"][i, h]), f64(c["q_rope"][i, h])])[None]
        o, l = oracle.attend(q, K, f64(v[: i + 1, h]), 1 / np.sqrt(192))
        assert_attn_close(out[i, h:h + 1], o, f"row {i} head {h}")
        assert_lse_close(lse[i, h:h + 1], l, f"lse {i} {h}")
