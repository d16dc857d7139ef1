"""Pins for the fp64 oracle: each test ties an oracle function to something
other than itself -- values the pages print, hand-worked examples, closed
forms, special cases with a known answer, and invariants the pages state.
CPU only."""
import math

import numpy as np
import pytest
import torch

import kvgen
import oracle
from oracle import closed_forms as cf
from conftest import read_golden

RNG = np.random.default_rng(20261202)


# ---------------------------------------------------------------- worked examples

def test_two_token_hand_example():
    g = read_golden("two_token_hand.txt")
    q = np.array([g["q"]])
    K = np.array([g["k0"], g["k1"]])
    V = np.array([g["v0"], g["v1"]])
    out, lse = oracle.attend(q, K, V, 1.0)
    np.testing.assert_allclose(out[0], g["out"], rtol=0, atol=1e-14)
    assert abs(lse[0] - g["lse"][0]) < 1e-14


def test_gqa_hand_example_head_mapping():
    g = read_golden("gqa_hand.txt")
    q = np.ones((1, 4, 1))
    k = np.zeros((1, 2, 2, 1))
    v = np.zeros((1, 2, 2, 1))
    v[0, 0, :, 0] = g["v_head0"]
    v[0, 1, :, 0] = g["v_head1"]
    out, lse = oracle.gqa_decode(q, k, v, [2], scale=1.0)
    np.testing.assert_allclose(out[0, :, 0], g["out"], atol=1e-14)
    np.testing.assert_allclose(lse[0], g["lse"][0] * np.ones(4), atol=1e-14)
    # the wrong (tiled) head mapping is distinguishable on this example
    assert not np.allclose(out[0, :, 0], [3, 20, 3, 20])


# ---------------------------------------------------------------- special cases

def test_single_token_returns_its_value_row():
    q = RNG.normal(size=(3, 16))
    K = RNG.normal(size=(1, 16))
    V = RNG.normal(size=(1, 8))
    out, lse = oracle.attend(q, K, V, 0.25)
    np.testing.assert_allclose(out, np.repeat(V, 3, 0), atol=1e-15)
    np.testing.assert_allclose(lse, 0.25 * q @ K[0], atol=1e-14)


def test_equal_keys_average_values():
    L = 37
    q = RNG.normal(size=(2, 8))
    K = np.repeat(RNG.normal(size=(1, 8)), L, 0)
    V = RNG.normal(size=(L, 5))
    out, lse = oracle.attend(q, K, V, 0.5)
    np.testing.assert_allclose(out, np.repeat(V.mean(0, keepdims=True), 2, 0), atol=1e-13)
    np.testing.assert_allclose(lse, 0.5 * q @ K[0] + math.log(L), atol=1e-12)


def test_dominant_key_selects_its_value():
    L, d = 20, 8
    q = RNG.normal(size=(1, d))
    K = RNG.normal(size=(L, d)) * 0.01
    K[13] = 60.0 * q[0] / np.linalg.norm(q[0]) ** 2   # score 60 vs ~0
    V = RNG.normal(size=(L, 4))
    out, _ = oracle.attend(q, K, V, 1.0)
    np.testing.assert_allclose(out[0], V[13], atol=1e-12)


def test_probabilities_sum_to_one():
    q = RNG.normal(size=(4, 32))
    K = RNG.normal(size=(300, 32))
    out, _ = oracle.attend(q, K, np.ones((300, 3)), 1 / math.sqrt(32))
    np.testing.assert_allclose(out, 1.0, atol=1e-12)


def test_empty_sequence():
    out, lse = oracle.attend(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 3)), 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_brute_force_tiny_gqa():
    """Scalar loops (math.exp) on a tiny GQA problem with ragged lengths."""
    B, h, n_kv, d = 2, 4, 2, 3
    q = RNG.normal(size=(B, h, d))
    k = RNG.normal(size=(B, n_kv, 5, d))
    v = RNG.normal(size=(B, n_kv, 5, d))
    sl = [5, 2]
    out, lse = oracle.gqa_decode(q, k, v, sl, scale=0.7)
    for b in range(B):
        for hh in range(h):
            kv = hh // 2
            s = [0.7 * sum(q[b, hh, i] * k[b, kv, j, i] for i in range(d)) for j in range(sl[b])]
            z = sum(math.exp(x) for x in s)
            for i in range(d):
                ref = sum(math.exp(s[j]) / z * v[b, kv, j, i] for j in range(sl[b]))
                assert abs(out[b, hh, i] - ref) < 1e-13
            assert abs(lse[b, hh] - math.log(z)) < 1e-13


# ---------------------------------------------------------------- GQA invariants

def test_repeat_kv_equals_mha():
    """[KVC-LLM] §四 (difference 3) and [CH7] §7.3: expanding each KV head g
    times along the head axis turns GQA into MHA with the same result."""
    B, h, n_kv, d, L = 2, 8, 2, 16, 40
    q = RNG.normal(size=(B, h, d))
    k = RNG.normal(size=(B, n_kv, L, d))
    v = RNG.normal(size=(B, n_kv, L, d))
    sl = [40, 23]
    o1, l1 = oracle.gqa_decode(q, k, v, sl)
    kr = np.repeat(k, h // n_kv, axis=1)
    vr = np.repeat(v, h // n_kv, axis=1)
    o2, l2 = oracle.gqa_decode(q, kr, vr, sl)
    # equal up to fp64 rounding order (a group's heads share one product);
    # a head read from the wrong KV head differs by O(1)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)
    # MQA is the g = h end of the same family
    o3, _ = oracle.gqa_decode(q, k[:, :1], v[:, :1], sl)
    o4, _ = oracle.gqa_decode(q, np.repeat(k[:, :1], h, 1), np.repeat(v[:, :1], h, 1), sl)
    np.testing.assert_allclose(o3, o4, rtol=0, atol=1e-12)
    assert np.abs(o1[:, 0] - o1[:, h // n_kv]).max() > 0.1     # the groups do differ


def test_head_axis_detector():
    """[CH7] §7.3: a broadcast on the wrong axis keeps shapes but breaks the
    logits.  Give each KV head a distinct constant value; head hh must read
    KV head hh // g."""
    B, h, n_kv, d, L = 1, 12, 3, 4, 9
    q = RNG.normal(size=(B, h, d))
    k = RNG.normal(size=(B, n_kv, L, d))
    v = np.zeros((B, n_kv, L, d))
    for kv in range(n_kv):
        v[:, kv] = kv + 1
    out, _ = oracle.gqa_decode(q, k, v, [L])
    np.testing.assert_allclose(out[0, :, 0], [hh // 4 + 1 for hh in range(h)], atol=1e-13)


def test_paged_equals_contiguous():
    """[ARG] §六.1: paging only changes where a token lives."""
    case = kvgen.gqa_case(3, 4, 2, 16, seqlens=[130, 64, 1], paged=True, seed=7)
    k = oracle.bf16_to_f64(case.k)
    v = oracle.bf16_to_f64(case.v)
    q = oracle.bf16_to_f64(case.q)
    bt = case.block_table.numpy()
    sl = case.seqlens.numpy()
    cap = bt.shape[1] * 64
    kc = np.zeros((3, 2, cap, 16))
    vc = np.zeros((3, 2, cap, 16))
    for b in range(3):
        for j in range(sl[b]):
            kc[b, :, j] = k[bt[b, j // 64], :, j % 64]
            vc[b, :, j] = v[bt[b, j // 64], :, j % 64]
    o1, l1 = oracle.gqa_decode(q, k, v, sl, block_table=bt)
    o2, l2 = oracle.gqa_decode(q, kc, vc, sl)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ---------------------------------------------------------------- split / combine

@pytest.mark.parametrize("S", [1, 2, 3, 7, 61])
def test_split_invariance(S):
    """[ARG] §五.2: softmax pieces merge exactly by their normalisers."""
    L = 61
    q = RNG.normal(size=(5, 24))
    K = RNG.normal(size=(L, 24))
    V = RNG.normal(size=(L, 10))
    ref, lref = oracle.attend(q, K, V, 0.3)
    bounds = [round(i * L / S) for i in range(S + 1)]
    O, ls = oracle.split_partials(q, K, V, 0.3, bounds)
    out, lse = oracle.combine_splits(O, ls)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, lref, atol=1e-12)


def test_combine_with_empty_split_and_counts():
    q = RNG.normal(size=(2, 8))
    K = RNG.normal(size=(10, 8))
    V = RNG.normal(size=(10, 3))
    ref, lref = oracle.attend(q, K, V, 1.0)
    # three splits, the middle one empty, plus one trailing unused slot
    O, ls = oracle.split_partials(q, K, V, 1.0, [0, 4, 4, 10])
    assert np.all(np.isneginf(ls[1]))
    O = np.concatenate([O, np.full((1, 2, 3), 1e30)])
    ls = np.concatenate([ls, np.full((1, 2), 50.0)])
    out, lse = oracle.combine_splits(O, ls, counts=[3, 3])
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, lref, atol=1e-12)
    out0, lse0 = oracle.combine_splits(O, ls, counts=[0, 3])
    assert np.all(out0[0] == 0) and np.isneginf(lse0[0])


# ---------------------------------------------------------------- MLA

def _mla_small(B=2, n_h=4, sl=(70, 9)):
    case = kvgen.mla_case(B, n_h, seqlens=list(sl), seed=11)
    return (oracle.bf16_to_f64(case.q_abs), oracle.bf16_to_f64(case.q_rope),
            oracle.bf16_to_f64(case.cache), case.block_table.numpy(),
            case.seqlens.numpy())


def test_mla_absorbed_equals_nonabsorbed():
    """[ARG] §四.5 and [MLA] §4: q~_h = W_UK,h^T q^C_h against the latent
    gives the same scores as up-projecting every cached latent; applying
    W_UV,h to the latent output gives the standard per-head output; the
    scale stays 1/sqrt(128 + 64)."""
    _, q_rope, cache, bt, sl = _mla_small()
    B, n_h = q_rope.shape[:2]
    W_UK = RNG.normal(size=(n_h, 128, 512)) / math.sqrt(512)
    W_UV = RNG.normal(size=(n_h, 128, 512)) / math.sqrt(512)
    q_nope = RNG.normal(size=(B, n_h, 128))
    q_abs = oracle.mla_absorb_q(q_nope, W_UK)
    lat, lse_a = oracle.mla_decode_absorbed(q_abs, q_rope, cache, bt, sl)
    o_abs = oracle.mla_project_out(lat, W_UV)
    o_ref, lse_n = oracle.mla_decode_nonabsorbed(q_nope, q_rope, cache, bt, sl, W_UK, W_UV)
    np.testing.assert_allclose(o_abs, o_ref, atol=1e-11)
    np.testing.assert_allclose(lse_a, lse_n, atol=1e-11)
    # W_UV with its latent axis reversed (a plausible slip) does not reach the same output
    assert not np.allclose(oracle.mla_project_out(lat, W_UV[:, :, ::-1]), o_ref, atol=1e-3)
    # 1/sqrt(576) is a different (wrong) reading and shows up
    lat2, _ = oracle.mla_decode_absorbed(q_abs, q_rope, cache, bt, sl, scale=1 / 24.0)
    assert not np.allclose(lat2, lat, atol=1e-6)


def test_mla_score_is_concatenated_dot():
    """[AIFAQ]: [q_c ; q_r] . [k_c ; k_r] = q_c.k_c + q_r.k_r, and V is the
    first 512 values of the same cached row ([ARG] §四.5): MLA equals one
    MQA head of key dim 576 and value dim 512."""
    q_abs, q_rope, cache, bt, sl = _mla_small()
    lat, lse = oracle.mla_decode_absorbed(q_abs, q_rope, cache, bt, sl)
    for b in range(len(sl)):
        rows = oracle.gather_tokens(cache, b, int(sl[b]), bt)
        qf = np.concatenate([q_abs[b], q_rope[b]], axis=1)
        o, l = oracle.attend(qf, rows, rows[:, :512], 1 / math.sqrt(192))
        np.testing.assert_allclose(lat[b], o, atol=1e-12)
        np.testing.assert_allclose(lse[b], l, atol=1e-12)


def test_mla_rope_term_matters():
    q_abs, q_rope, cache, bt, sl = _mla_small()
    a, _ = oracle.mla_decode_absorbed(q_abs, q_rope, cache, bt, sl)
    b, _ = oracle.mla_decode_absorbed(q_abs, 0 * q_rope, cache, bt, sl)
    assert not np.allclose(a, b, atol=1e-6)


def test_mla_single_token():
    q_abs, q_rope, cache, bt, _ = _mla_small()
    lat, _ = oracle.mla_decode_absorbed(q_abs, q_rope, cache, bt, np.array([1, 1]))
    for b in range(2):
        np.testing.assert_allclose(lat[b], np.repeat(cache[bt[b, 0], 0:1, :512], 4, 0), atol=0)


# ---------------------------------------------------------------- RoPE

def test_rope_identity_at_zero_and_norm():
    x = RNG.normal(size=(5, 64))
    np.testing.assert_array_equal(oracle.rope_rotate(x, np.zeros(5)), x)
    y = oracle.rope_rotate(x, np.arange(5) * 1000.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_relative_position():
    """[ARG] §四.4: R_m^T R_n = R_{n-m}, so <R_m q, R_n k> depends on n - m."""
    for m, n in [(3, 10), (100, 4), (131000, 131072)]:
        Rm, Rn, Rd = (oracle.rope_matrix(p, 8) for p in (m, n, n - m))
        np.testing.assert_allclose(Rm.T @ Rn, Rd, atol=1e-9)
    q, k = RNG.normal(size=64), RNG.normal(size=64)
    a = oracle.rope_rotate(q, 17.0) @ oracle.rope_rotate(k, 29.0)
    b = oracle.rope_rotate(q, 1017.0) @ oracle.rope_rotate(k, 1029.0)
    assert abs(a - b) < 1e-10


def test_rope_known_angles():
    """Reading: interleaved pairs, angle_i = pos * theta^(-2i/dim)."""
    y = oracle.rope_rotate(np.array([1.0, 0.0]), 1.0)
    np.testing.assert_allclose(y, [math.cos(1), math.sin(1)], atol=1e-16)
    y = oracle.rope_rotate(np.array([0.0, 0.0, 1.0, 0.0]), 100.0)   # 10000^(-2/4) = 1/100
    np.testing.assert_allclose(y, [0, 0, math.cos(1), math.sin(1)], atol=1e-15)
    y = oracle.rope_rotate(np.array([0.0, 1.0]), math.pi / 2)
    np.testing.assert_allclose(y, [-1, 0], atol=1e-15)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rounding_known_values():
    f = oracle.f64_to_bf16_bits
    assert f(np.array([1.0]))[0] == 0x3F80
    assert f(np.array([1.0 + 2 ** -8]))[0] == 0x3F80          # tie -> even
    assert f(np.array([1.0 + 3 * 2 ** -8]))[0] == 0x3F82      # tie -> even (up)
    assert f(np.array([1.0 + 2 ** -8 + 2 ** -30]))[0] == 0x3F81
    assert f(np.array([-2.0]))[0] == 0xC000


def test_bf16_rounding_matches_fp32_cast():
    """One RNE step from binary32 (a library routine) is the special case of
    the fp64 rounding for inputs that are exact binary32 values."""
    x = torch.randn(100000, dtype=torch.float32) * 3
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16_bits(x.numpy().astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    back = oracle.bf16_bits_to_f64(ref)
    np.testing.assert_array_equal(back, x.to(torch.bfloat16).to(torch.float64).numpy())


# ---------------------------------------------------------------- cache append

def test_append_mla_slot_and_rotation():
    sl = np.array([0, 63, 64, 200])
    case = kvgen.mla_case(4, 2, seqlens=[1, 64, 65, 201], seed=3, spare_pages=2)
    bits = case.cache.view(torch.int16).numpy().view(np.uint16)
    bt = case.block_table.numpy()
    ckv, kr = kvgen.append_inputs_mla(4, seed=5)
    cb = ckv.view(torch.int16).numpy().view(np.uint16)
    kb = kr.view(torch.int16).numpy().view(np.uint16)
    new = oracle.append_rope_mla(bits, bt, sl, cb, kb)
    changed = np.argwhere(np.any(new != bits, axis=2))
    expect = {(int(bt[b, sl[b] // 64]), int(sl[b] % 64)) for b in range(4)}
    assert {tuple(x) for x in changed} <= expect
    for b in range(4):
        page, row = bt[b, sl[b] // 64], sl[b] % 64
        np.testing.assert_array_equal(new[page, row, :512], cb[b])
        back = oracle.rope_rotate(oracle.bf16_bits_to_f64(new[page, row, 512:]), -float(sl[b]))
        np.testing.assert_allclose(back, oracle.bf16_bits_to_f64(kb[b]), atol=0.02)
    # position 0 is the identity rotation
    np.testing.assert_array_equal(new[bt[0, 0], 0, 512:], kb[0])


def test_append_gqa_contiguous_and_paged():
    sl = np.array([5, 0])
    k_new, v_new = kvgen.append_inputs_gqa(2, 2, 8, seed=9)
    kn = k_new.view(torch.int16).numpy().view(np.uint16)
    vn = v_new.view(torch.int16).numpy().view(np.uint16)
    K = np.zeros((2, 2, 16, 8), np.uint16)
    V = np.zeros((2, 2, 16, 8), np.uint16)
    K2, V2 = oracle.append_rope_gqa(K, V, sl, kn, vn)
    np.testing.assert_array_equal(V2[0, :, 5], vn[0])
    np.testing.assert_array_equal(K2[1, :, 0], kn[1])       # pos 0: no rotation
    rot = oracle.rope_rotate(oracle.bf16_bits_to_f64(kn[0]), 5.0)
    np.testing.assert_array_equal(K2[0, :, 5], oracle.f64_to_bf16_bits(rot))
    mask = np.ones(K.shape, bool)
    mask[0, :, 5] = False
    mask[1, :, 0] = False
    assert np.all(K2[mask] == 0) and np.all(V2[mask] == 0)
    bt = np.array([[1, 0], [2, 3]])
    Kp = np.zeros((4, 2, 64, 8), np.uint16)
    Vp = np.zeros((4, 2, 64, 8), np.uint16)
    Kp2, Vp2 = oracle.append_rope_gqa(Kp, Vp, np.array([70, 3]), kn, vn, block_table=bt)
    np.testing.assert_array_equal(Vp2[0, :, 6], vn[0])
    np.testing.assert_array_equal(Vp2[2, :, 3], vn[1])


# ---------------------------------------------------------------- MLA prefill (non-absorbed)

def _prefill_case(s_kv, s_q, n_h, seed):
    r = np.random.default_rng(seed)
    c_kv = r.normal(size=(s_kv, 512))
    k_rope = r.normal(size=(s_kv, 64))
    q_nope = r.normal(size=(s_q, n_h, 128)) / 4
    q_rope = r.normal(size=(s_q, n_h, 64)) / 4
    W_UK = r.normal(size=(n_h, 128, 512)) / math.sqrt(512)
    W_UV = r.normal(size=(n_h, 128, 512)) / math.sqrt(512)
    return c_kv, k_rope, q_nope, q_rope, W_UK, W_UV


def test_mla_prefill_rows_equal_absorbed_path():
    """Every query row of the non-absorbed causal prefill equals the absorbed
    decode over that row's prefix ([ARG] §四.5-6: the two paths are the same
    attention; the pinned absorbed functions serve as the check)."""
    s_kv, s_q, n_h = 70, 6, 2
    c_kv, k_rope, q_nope, q_rope, W_UK, W_UV = _prefill_case(s_kv, s_q, n_h, 31)
    k_nope, v = oracle.mla_prefill_expand(c_kv, W_UK, W_UV)
    out, lse = oracle.mla_prefill(q_nope, q_rope, k_nope, k_rope, v)
    cache = np.zeros((2, 64, 576))
    rows = np.concatenate([c_kv, k_rope], axis=1)
    cache.reshape(128, 576)[:s_kv] = rows
    bt = np.array([[0, 1]] * s_q)
    sl = np.array([s_kv - s_q + i + 1 for i in range(s_q)])
    q_abs = oracle.mla_absorb_q(q_nope, W_UK)
    lat, lse_a = oracle.mla_decode_absorbed(q_abs, q_rope, cache, bt, sl)
    np.testing.assert_allclose(out, oracle.mla_project_out(lat, W_UV), atol=1e-11)
    np.testing.assert_allclose(lse, lse_a, atol=1e-11)
    # a chunk placed at another offset is a different (wrong) causal window
    wrong, _ = oracle.mla_prefill(q_nope, q_rope, k_nope, k_rope, v, kv_offset=s_kv - s_q - 3)
    assert not np.allclose(wrong, out, atol=1e-6)


def test_mla_prefill_is_causal():
    """Query i sees positions <= s_kv - s_q + i and nothing after them."""
    s_kv, s_q, n_h = 40, 8, 1
    c_kv, k_rope, q_nope, q_rope, W_UK, W_UV = _prefill_case(s_kv, s_q, n_h, 32)
    k_nope, v = oracle.mla_prefill_expand(c_kv, W_UK, W_UV)
    out, _ = oracle.mla_prefill(q_nope, q_rope, k_nope, k_rope, v)
    i = 3
    last = s_kv - s_q + i
    k2, v2, r2 = k_nope.copy(), v.copy(), k_rope.copy()
    k2[last + 1:] += 5.0
    v2[last + 1:] -= 7.0
    r2[last + 1:] *= -1
    out2, _ = oracle.mla_prefill(q_nope, q_rope, k2, r2, v2)
    np.testing.assert_array_equal(out2[: i + 1], out[: i + 1])
    assert not np.allclose(out2[i + 1:], out[i + 1:])
    v3 = v.copy()
    v3[last] += 1.0
    out3, _ = oracle.mla_prefill(q_nope, q_rope, k_nope, k_rope, v3)
    assert not np.allclose(out3[i], out[i])


def test_mla_prefill_single_query_is_decode():
    """A one-token chunk is a decode step on the literal path."""
    s_kv, n_h = 65, 3
    c_kv, k_rope, q_nope, q_rope, W_UK, W_UV = _prefill_case(s_kv, 1, n_h, 33)
    k_nope, v = oracle.mla_prefill_expand(c_kv, W_UK, W_UV)
    out, lse = oracle.mla_prefill(q_nope, q_rope, k_nope, k_rope, v)
    cache = np.zeros((2, 64, 576))
    cache.reshape(128, 576)[:s_kv] = np.concatenate([c_kv, k_rope], axis=1)
    ref, lref = oracle.mla_decode_nonabsorbed(q_nope, q_rope, cache, np.array([[0, 1]]),
                                              np.array([s_kv]), W_UK, W_UV)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, lref, atol=1e-12)


# ---------------------------------------------------------------- E4M3 (FP8 KV cache)

def test_e4m3_decode_golden():
    """Code values written out from the format definition."""
    for key, (val,) in read_golden("e4m3_codes.txt").items():
        code = int(key[4:])
        got = oracle.e4m3_bits_to_f64(np.array([code], np.uint8))[0]
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)
    assert np.isnan(oracle.e4m3_bits_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_matches_library_cast():
    """All 256 codes against torch's float8_e4m3fn widening."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_bits_to_f64(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_e4m3_encode_matches_library_cast():
    """Nearest-even rounding against torch's float32 -> float8_e4m3fn cast on
    values across the whole finite range, including every midpoint between
    neighbouring codes (the ties)."""
    mags = oracle.e4m3_bits_to_f64(np.arange(0x7F))
    mids = (mags[:-1] + mags[1:]) / 2
    rnd = np.exp2(RNG.uniform(-12, np.log2(448.0), 20000))
    x = np.concatenate([mags, mids, rnd, np.nextafter(mids, 0), np.nextafter(mids, 1e9)])
    x = np.concatenate([x, -x]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.f64_to_e4m3_bits(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_ties_saturation_roundtrip():
    enc = oracle.f64_to_e4m3_bits
    # ties go to the even code: 1.0625 between 1 (0x38) and 1.125 (0x39)
    assert enc([1.0625])[0] == 0x38 and enc([1.1875])[0] == 0x3A
    # subnormal ties: 2^-10 between 0 and 2^-9; 3 * 2^-10 between codes 1 and 2
    assert enc([2.0 ** -10])[0] == 0x00 and enc([3 * 2.0 ** -10])[0] == 0x02
    # saturation to the largest finite value, sign kept
    assert enc([1e6])[0] == 0x7E and enc([-500.0])[0] == 0xFE and enc([464.0])[0] == 0x7E
    assert enc([np.nan])[0] == 0x7F and enc([-0.0])[0] == 0x80
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    np.testing.assert_array_equal(enc(oracle.e4m3_bits_to_f64(finite)), finite)


def test_dequant_scales_the_kv_head_axis():
    codes = np.full((2, 3, 5, 4), 0x38, np.uint8)          # every value 1.0
    sc = np.array([0.5, 2.0, 8.0])
    v = oracle.dequant_e4m3(codes, sc)
    for hh in range(3):
        assert np.all(v[:, hh] == sc[hh])


def test_fp8_decode_equals_decode_of_dequantised_bf16():
    """With power-of-two scales every dequantised value is a bf16 number, so
    the FP8 decode must equal the bf16 decode of the same values; a scale
    taken from the wrong head, or K's scale used for V, must not."""
    c = kvgen.gqa_case(2, 8, 2, 16, seqlens=[9, 70], seed=3)
    kc = RNG.integers(0, 256, c.k.shape).astype(np.uint8)
    vc = RNG.integers(0, 256, c.v.shape).astype(np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x3C                      # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x3C
    kc = kc & 0xBF                                       # exponent field <= 7: |value| < 2
    vc = vc & 0xBF
    ks = np.array([2.0 ** -3, 2.0 ** 1])
    vs = np.array([2.0 ** 2, 2.0 ** -1])
    q = oracle.bf16_to_f64(c.q)
    out, lse = oracle.gqa_decode_fp8(q, kc, vc, ks, vs, c.seqlens.numpy())
    kf = oracle.e4m3_bits_to_f64(kc) * ks[None, :, None, None]
    vf = oracle.e4m3_bits_to_f64(vc) * vs[None, :, None, None]
    assert np.array_equal(oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(kf)), kf)
    out2, lse2 = oracle.gqa_decode(q, kf, vf, c.seqlens.numpy())
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)
    bad, _ = oracle.gqa_decode_fp8(q, kc, vc, ks[::-1], vs, c.seqlens.numpy())
    assert not np.allclose(bad, out, atol=1e-3)
    bad, _ = oracle.gqa_decode_fp8(q, kc, vc, ks, ks, c.seqlens.numpy())
    assert not np.allclose(bad, out, atol=1e-3)


def test_fp8_append_codes():
    """FP8 append: K codes are the nearest codes to RoPE(k) / k_scale (the
    quantisation error bound: half a code step); V codes equal the library
    cast of the binary32 quotient v / v_scale."""
    B, n_kv, d = 3, 2, 16
    k_new, v_new = kvgen.append_inputs_gqa(B, n_kv, d, seed=21)
    kn = k_new.view(torch.int16).numpy().view(np.uint16)
    vn = v_new.view(torch.int16).numpy().view(np.uint16)
    ks = np.array([0.01, 0.03], np.float32)
    vs = np.array([0.02, 0.005], np.float32)
    sl = np.array([5, 0, 131])
    K = np.zeros((B, n_kv, 192, d), np.uint8)
    V = np.zeros((B, n_kv, 192, d), np.uint8)
    K2, V2 = oracle.append_rope_gqa(K, V, sl, kn, vn, k_scale=ks, v_scale=vs)
    for b in range(B):
        rot = oracle.rope_rotate(oracle.bf16_bits_to_f64(kn[b]), float(sl[b])) / ks[:, None].astype(np.float64)
        got = oracle.e4m3_bits_to_f64(K2[b, :, sl[b]])
        # |x - Q(x)| <= half the gap between the two codes around x
        mags = oracle.e4m3_bits_to_f64(np.arange(0x7F))
        hi = np.searchsorted(mags, np.abs(rot))
        gap = mags[np.minimum(hi, 126)] - mags[np.maximum(hi - 1, 0)]
        assert np.all(np.abs(got - rot) <= gap / 2 + 1e-15)
        quot = torch.from_numpy(v_new[b].float().numpy() / vs[:, None])
        ref = quot.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(V2[b, :, sl[b]], ref)


def test_dequant_mla_splits_the_row():
    """The latent row's first 512 values take the c_kv scale, its last 64
    the k_R scale."""
    codes = np.full((2, 3, 576), 0x38, np.uint8)            # every value 1.0
    codes[0, 0, 511] = 0xC0                                 # -2.0
    v = oracle.dequant_mla_e4m3(codes, [0.5, 4.0])
    assert np.all(v[..., 512:] == 4.0)
    assert v[0, 0, 511] == -1.0
    assert np.all(np.delete(v[..., :512].reshape(-1), 511) == 0.5)


def _mla_codes(shape):
    c = RNG.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C                            # no NaN codes
    return c


def test_mla_fp8_decode_equals_decode_of_dequantised_bf16():
    """With power-of-two scales every dequantised value is a bf16 number, so
    the FP8 MLA decode must equal the (pinned) bf16 absorbed decode of the
    same rows; swapping the c_kv and k_R scales must not."""
    case = kvgen.mla_case(2, 4, seqlens=[70, 9], seed=31)
    codes = _mla_codes(case.cache.shape) & 0xBF               # exponent field <= 7
    ks = np.array([2.0 ** -3, 2.0 ** 1])
    qa, qr = oracle.bf16_to_f64(case.q_abs), oracle.bf16_to_f64(case.q_rope)
    bt, sl = case.block_table.numpy(), case.seqlens.numpy()
    out, lse = oracle.mla_decode_absorbed_fp8(qa, qr, codes, ks, bt, sl)
    rows = oracle.e4m3_bits_to_f64(codes)
    rows[..., :512] *= ks[0]
    rows[..., 512:] *= ks[1]
    assert np.array_equal(oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(rows)), rows)
    out2, lse2 = oracle.mla_decode_absorbed(qa, qr, rows, bt, sl)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)
    bad, _ = oracle.mla_decode_absorbed_fp8(qa, qr, codes, ks[::-1], bt, sl)
    assert not np.allclose(bad, out, atol=1e-3)


def test_mla_fp8_scale_homogeneity():
    """Scaling the whole cache row by s is the same as scaling both query
    pieces by s (scores) and the latent output by s (values): with scales
    (s_c, s_R), out = s_c * out(scales 1, q_abs * s_c, q_rope * s_R) and the
    lse is unchanged.  A scale missing on the values, or applied to the
    wrong piece of the row, breaks it."""
    case = kvgen.mla_case(2, 4, seqlens=[130, 64], seed=32)
    codes = _mla_codes(case.cache.shape)
    qa, qr = oracle.bf16_to_f64(case.q_abs), oracle.bf16_to_f64(case.q_rope)
    bt, sl = case.block_table.numpy(), case.seqlens.numpy()
    sc, sr = 0.0125, 0.07
    out, lse = oracle.mla_decode_absorbed_fp8(qa, qr, codes, [sc, sr], bt, sl)
    out1, lse1 = oracle.mla_decode_absorbed_fp8(qa * sc, qr * sr, codes, [1.0, 1.0], bt, sl)
    np.testing.assert_allclose(out, sc * out1, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse, lse1, rtol=1e-12, atol=1e-12)
    assert np.abs(out).max() > 1e-3


def test_fp8_mla_append_codes():
    """Quantising MLA append: the row lands at the slot of pos = seqlens[b];
    c_kv codes equal the library cast of the binary32 quotient c_kv /
    scale_c; k_R codes are the nearest codes to RoPE(k_R) / scale_R (half a
    code step); nothing else changes."""
    sl = np.array([0, 63, 64, 200])
    case = kvgen.mla_case(4, 2, seqlens=[1, 64, 65, 201], seed=33, spare_pages=2,
                          kv_dtype="fp8")
    codes = case.cache.numpy()
    bt = case.block_table.numpy()
    ckv, kr = kvgen.append_inputs_mla(4, seed=34)
    cb = ckv.view(torch.int16).numpy().view(np.uint16)
    kb = kr.view(torch.int16).numpy().view(np.uint16)
    ks = np.array([0.02, 0.011], np.float32)
    new = oracle.append_rope_mla(codes, bt, sl, cb, kb, kv_scale=ks)
    changed = np.argwhere(np.any(new != codes, axis=2))
    expect = {(int(bt[b, sl[b] // 64]), int(sl[b] % 64)) for b in range(4)}
    assert {tuple(x) for x in changed} <= expect
    mags = oracle.e4m3_bits_to_f64(np.arange(0x7F))
    for b in range(4):
        page, row = bt[b, sl[b] // 64], sl[b] % 64
        quot = torch.from_numpy(ckv[b].float().numpy() / ks[0])
        np.testing.assert_array_equal(new[page, row, :512],
                                      quot.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        rot = oracle.rope_rotate(oracle.bf16_bits_to_f64(kb[b]), float(sl[b])) / np.float64(ks[1])
        got = oracle.e4m3_bits_to_f64(new[page, row, 512:])
        hi = np.searchsorted(mags, np.abs(rot))
        gap = mags[np.minimum(hi, 126)] - mags[np.maximum(hi - 1, 0)]
        assert np.all(np.abs(got - rot) <= gap / 2 + 1e-15)


# ---------------------------------------------------------------- sliding window

def test_window_matches_printed_mask():
    """window_slots reads exactly the keys the figure marks for w = 4."""
    g = read_golden("sliding_window_w4.txt")
    w = 4
    for t in range(12):
        slots = oracle.window_slots(t + 1, w)
        # invert the ring: the position p in (t - w, t] with p mod w == slot
        pos = sorted(t - ((t - s) % w) for s in slots)
        mask = np.zeros(12)
        mask[pos] = 1
        np.testing.assert_array_equal(mask, g["t%d" % t])
    # the text's "[t - w, t]" (w + 1 keys) is a different reading
    assert len(oracle.window_slots(12, w)) == w


@pytest.mark.parametrize("paged", [False, True])
def test_window_ring_equals_last_w_positions(paged):
    """A ring of w slots holding position p at slot p mod w gives the same
    decode as plain attention over the last w positions of a linear cache."""
    w, d, n_kv, h = 37, 8, 2, 4
    lens = [5, 37, 38, 100, 0]
    B = len(lens)
    T = max(lens)
    q = RNG.normal(size=(B, h, d))
    Klin = RNG.normal(size=(B, n_kv, T, d))
    Vlin = RNG.normal(size=(B, n_kv, T, d))
    Kr = np.zeros((B, n_kv, w, d))
    Vr = np.zeros((B, n_kv, w, d))
    for b, n in enumerate(lens):
        for p in range(max(0, n - w), n):
            Kr[b, :, p % w] = Klin[b, :, p]
            Vr[b, :, p % w] = Vlin[b, :, p]
    bt = None
    if paged:
        bt = np.array([[2 * b + 1, 2 * b] for b in range(B)])
        Kp = np.zeros((2 * B, n_kv, 64, d))
        Vp = np.zeros((2 * B, n_kv, 64, d))
        for b in range(B):
            for s_ in range(w):
                Kp[bt[b, s_ // 64], :, s_ % 64] = Kr[b, :, s_]
                Vp[bt[b, s_ // 64], :, s_ % 64] = Vr[b, :, s_]
        Kr, Vr = Kp, Vp
    out, lse = oracle.gqa_decode(q, Kr, Vr, np.array(lens), 0.3, bt, window=w)
    for b, n in enumerate(lens):
        lo = max(0, n - w)
        for hh in range(h):
            o, l = oracle.attend(q[b, hh:hh + 1], Klin[b, hh // 2, lo:n], Vlin[b, hh // 2, lo:n], 0.3)
            np.testing.assert_allclose(out[b, hh], o[0], atol=1e-12)
            assert (l[0] == lse[b, hh]) if n == 0 else abs(l[0] - lse[b, hh]) < 1e-12
    # w >= length: the full decode
    full, _ = oracle.gqa_decode(q, Klin, Vlin, np.array(lens), 0.3)
    wide, _ = oracle.gqa_decode(q, Klin, Vlin, np.array(lens), 0.3, window=T)
    np.testing.assert_array_equal(full, wide)


def test_window_append_ring_keeps_last_w():
    """Appending positions 0..N-1 one by one into a ring of w slots leaves
    slot s holding the newest position p = s (mod w), rotated to p."""
    w, n_kv, d, N = 5, 1, 8, 13
    K = np.zeros((1, n_kv, 8, d), np.uint16)
    V = np.zeros((1, n_kv, 8, d), np.uint16)
    ks_, vs_ = [], []
    for p in range(N):
        k_new, v_new = kvgen.append_inputs_gqa(1, n_kv, d, seed=100 + p)
        kn = k_new.view(torch.int16).numpy().view(np.uint16)
        vn = v_new.view(torch.int16).numpy().view(np.uint16)
        ks_.append(kn)
        vs_.append(vn)
        K, V = oracle.append_rope_gqa(K, V, np.array([p]), kn, vn, window=w)
    for p in range(N - w, N):
        rot = oracle.f64_to_bf16_bits(oracle.rope_rotate(oracle.bf16_bits_to_f64(ks_[p][0]), float(p)))
        np.testing.assert_array_equal(K[0, :, p % w], rot)
        np.testing.assert_array_equal(V[0, :, p % w], vs_[p][0])
    assert np.all(K[0, :, w:] == 0)


# ---------------------------------------------------------------- closed forms

def test_closed_forms_match_printed_values():
    g = {k: v[0] for k, v in read_golden("cache_sizes.txt").items()}
    per_layer_values = lambda heads, d: cf.kv_cache_bytes_per_token(1, heads, d, elem_bytes=1)
    mla = cf.mla_latent_values_per_token(512, 64)
    assert mla == g["mla_elems_per_token_per_layer"]
    assert 64 / 512 == g["mla_rope_overhead"]
    mha5120 = per_layer_values(40, 128)               # 2 * d_model at d_model = 5120
    assert mha5120 == 10240
    assert round(mha5120 / mla, 1) == g["mha_vs_mla_ratio_dmodel5120"]
    assert mha5120 / cf.mla_latent_values_per_token(512, 0) == g["mha_vs_pure_mla_ratio_dmodel5120"]
    assert cf.mla_cache_bytes_per_token(60) == g["mla_60_layer_bytes_per_token"]
    assert cf.mla_cache_bytes_per_token(60) / 1024 == 67.5
    assert per_layer_values(32, 128) == g["llama2_mha_elems"]
    assert per_layer_values(8, 128) == g["llama2_gqa8_elems"]
    assert per_layer_values(1, 128) == g["llama2_mqa_elems"]
    assert cf.mla_latent_values_per_token(512, 0) == g["llama2_mla_elems"]
    assert cf.kv_cache_bytes_per_token(32, 8, 128) == g["llama3_8b_gqa_bytes_per_token"]
    assert cf.kv_cache_bytes_per_token(32, 32, 128) == g["llama3_8b_mha_bytes_per_token"]
    assert cf.kv_cache_bytes_per_token(80, 8, 128) == g["llama3_70b_gqa_bytes_per_token"]
    v3 = cf.mla_cache_bytes_per_token(61)
    assert v3 == g["deepseek_v3_mla_bytes_per_token"]
    v3m = cf.kv_cache_bytes_per_token(61, 128, 128)
    assert v3m == g["deepseek_v3_as_mha_bytes_per_token"]
    assert round(v3m / v3, 1) == g["deepseek_v3_mha_over_mla"]
    gib = 1024 ** 3
    assert round(cf.kv_cache_bytes_per_token(32, 8, 128) * 131072 / gib, 1) == g["llama3_8b_128k_gib"]
    assert round(cf.kv_cache_bytes_per_token(80, 8, 128) * 131072 / gib, 1) == g["llama3_70b_128k_gib"]
    assert round(v3 * 131072 / gib, 1) == g["deepseek_v3_128k_gib"]
    assert cf.grouped_decode_intensity(1) == g["intensity_mha"]
    assert cf.grouped_decode_intensity(32 // 8) == g["intensity_llama3_8b"]
    assert cf.grouped_decode_intensity(64 // 8) == g["intensity_llama3_70b"]
    assert round(cf.mla_decode_intensity(128)) == g["intensity_deepseek_v3"]
    assert cf.mla_decode_flops_per_token(128) == g["mla_flops_per_token_per_layer"]
    assert cf.mla_cache_bytes_per_token(1) == g["mla_bytes_per_token_per_layer"]
    assert cf.kv_cache_bytes_per_token(1, 8, 128) == g["llama3_8b_gqa_bytes_per_token_per_layer"]
    # [ARG] §四.6 prints the Llama-3-8B GQA FLOPs per cached token per layer:
    # 32 heads, a 128-long dot and a 128-long weighted sum each
    assert 32 * 2 * (128 + 128) == g["llama3_8b_gqa_flops_per_token_per_layer"]
    assert (g["llama3_8b_gqa_flops_per_token_per_layer"] / g["llama3_8b_gqa_bytes_per_token_per_layer"]
            == cf.grouped_decode_intensity(4))
    assert 192 + 128 == g["dot_len_unabsorbed"] and 576 + 512 == g["dot_len_absorbed"]
    assert round(cf.mla_vs_mha_read_ratio(20), 2) == g["mla_mha_read_ratio_s20"]
    assert abs(cf.mla_vs_mha_read_ratio(1e12) - g["mla_mha_read_ratio_limit"]) < 1e-9
