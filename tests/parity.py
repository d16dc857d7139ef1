"""Shared parity helpers: tolerance checks and oracle slices for GPU tests.

Tolerance (floating point, bf16 inputs, fp32 accumulation): max-abs error
<= 2e-2 over all elements AND per-row relative L2 error
||gpu - ref|| / ||ref|| <= 1e-2.  The row-wise relative error is the reading
of "max-rel 1e-2": an element-wise relative error is unbounded where the
exact output is near zero, which an average of N(0,1) values often is.
lse is compared with max-abs 2e-2.  Integer and byte results are compared
bit-exactly by the tests themselves.
"""
import math

import numpy as np
import torch

import oracle

ATOL = 2e-2
ROW_RTOL = 1e-2


def f64(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    if t.dtype == torch.bfloat16:
        return oracle.bf16_to_f64(t)
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_attn_close(got, ref, what="", atol=ATOL, row_rtol=ROW_RTOL):
    got = f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    num = np.linalg.norm((got - ref).reshape(-1, ref.shape[-1]), axis=1)
    den = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1)
    rel = np.where(den > 0, num / np.maximum(den, 1e-300), num)
    assert max_abs <= atol, f"{what}: max-abs {max_abs:.3e} > {atol}"
    assert float(rel.max()) <= row_rtol, f"{what}: row rel {rel.max():.3e} > {row_rtol}"
    return max_abs, float(rel.max())


def assert_lse_close(got, ref, what="", atol=ATOL):
    got = f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{what}: -inf pattern differs"
    d = np.abs(got[~inf_ref] - ref[~inf_ref])
    assert (d.max() if d.size else 0.0) <= atol, f"{what}: lse max-abs {d.max():.3e}"


def gqa_rows_oracle(case, rows):
    """Oracle output and lse for selected (b, h) rows of a GqaCase, computed
    one row at a time from the row's own tokens (works at full size)."""
    g = case.h // case.n_kv
    sl = case.seqlens.to("cpu").numpy()
    bt = None if case.block_table is None else case.block_table.to("cpu").numpy()
    outs, lses = [], []
    for b, h in rows:
        kv = h // g
        L = int(sl[b])
        if bt is None:
            K = f64(case.k[b, kv, :L])
            V = f64(case.v[b, kv, :L])
        else:
            npg = (L + 63) // 64
            pages = torch.as_tensor(bt[b, :npg], dtype=torch.long, device=case.k.device)
            K = f64(case.k[pages, kv].reshape(-1, case.d)[:L])
            V = f64(case.v[pages, kv].reshape(-1, case.d)[:L])
        o, l = oracle.attend(f64(case.q[b, h:h + 1]), K, V, case.scale)
        outs.append(o[0])
        lses.append(l[0])
    return np.array(outs), np.array(lses)


def mla_rows_oracle(case, rows):
    """Oracle latent output and lse for selected (b, h) rows of an MlaCase:
    the sequence's pages are gathered in logical order and passed to the
    oracle's MLA definition with an identity block table."""
    sl = case.seqlens.to("cpu").numpy()
    bt = case.block_table.to("cpu").numpy()
    outs, lses = [], []
    seq_cache = {}
    for b, h in rows:
        L = int(sl[b])
        npg = (L + 63) // 64
        if b not in seq_cache:
            pages = torch.as_tensor(bt[b, :npg], dtype=torch.long, device=case.cache.device)
            seq_cache[b] = f64(case.cache[pages]) if npg else np.zeros((0, 64, 576))
        o, l = oracle.mla_decode_absorbed(
            f64(case.q_abs[b, h:h + 1])[None], f64(case.q_rope[b, h:h + 1])[None],
            seq_cache[b], np.arange(max(npg, 1))[None], [L], case.scale)
        outs.append(o[0, 0])
        lses.append(l[0, 0])
    return np.array(outs), np.array(lses)


def gqa_full_oracle(case):
    """Oracle output and lse of a whole GqaCase, one oracle call per
    (sequence, KV head): the sequence's tokens of that head (its pages, for
    a paged cache, gathered in logical order) and the g query heads that
    read it.  Bounded memory at any size: only one head's rows are widened
    to fp64 at a time.  Handles E4M3 caches (k_scale set) and ring caches
    (window > 0) through the oracle's own functions."""
    B, h, d, n_kv = case.B, case.h, case.d, case.n_kv
    g = h // n_kv
    sl = case.seqlens.to("cpu").numpy()
    bt = None if case.block_table is None else case.block_table.to("cpu").numpy()
    window = getattr(case, "window", 0) or 0
    fp8 = getattr(case, "k_scale", None) is not None
    ks = case.k_scale.to("cpu").numpy() if fp8 else None
    vs = case.v_scale.to("cpu").numpy() if fp8 else None
    out = np.zeros((B, h, d))
    lse = np.zeros((B, h))
    raw = (lambda t: t.detach().to("cpu").numpy()) if fp8 else f64
    for b in range(B):
        held = min(int(sl[b]), window) if window > 0 else int(sl[b])
        for kv in range(n_kv):
            heads = slice(kv * g, (kv + 1) * g)
            q = f64(case.q[b:b + 1, heads])
            if bt is None:
                n_slots = max(held, window) if window > 0 else held
                K = raw(case.k[b:b + 1, kv:kv + 1, :max(n_slots, 1)])
                V = raw(case.v[b:b + 1, kv:kv + 1, :max(n_slots, 1)])
                bt_b = None
            else:
                npg = max((max(held, window) if window > 0 else held) + 63, 64) // 64
                pages = torch.as_tensor(bt[b, :npg], dtype=torch.long, device=case.k.device)
                K = raw(case.k[pages, kv:kv + 1])
                V = raw(case.v[pages, kv:kv + 1])
                bt_b = np.arange(npg)[None]
            if fp8:
                o, l = oracle.gqa_decode_fp8(q, K, V, ks[kv:kv + 1], vs[kv:kv + 1], [int(sl[b])],
                                             case.scale, bt_b, window)
            else:
                o, l = oracle.gqa_decode(q, K, V, [int(sl[b])], case.scale, bt_b, window)
            out[b, heads], lse[b, heads] = o[0], l[0]
    return out, lse


def mla_full_oracle(case):
    """Oracle latent output and lse of a whole MlaCase, one oracle call per
    sequence on that sequence's pages (gathered in logical order).  E4M3
    caches (kv_scale set) go through the oracle's FP8 decode on the raw
    codes."""
    sl = case.seqlens.to("cpu").numpy()
    bt = case.block_table.to("cpu").numpy()
    fp8 = getattr(case, "kv_scale", None) is not None
    ks = case.kv_scale.to("cpu").numpy() if fp8 else None
    out = np.zeros((case.B, case.n_h, 512))
    lse = np.zeros((case.B, case.n_h))
    for b in range(case.B):
        L = int(sl[b])
        npg = max((L + 63) // 64, 1)
        pages = torch.as_tensor(bt[b, :npg], dtype=torch.long, device=case.cache.device)
        qa, qr = f64(case.q_abs[b:b + 1]), f64(case.q_rope[b:b + 1])
        if fp8:
            o, l = oracle.mla_decode_absorbed_fp8(qa, qr, case.cache[pages].to("cpu").numpy(), ks,
                                                  np.arange(npg)[None], [L], case.scale)
        else:
            o, l = oracle.mla_decode_absorbed(qa, qr, f64(case.cache[pages]), np.arange(npg)[None], [L],
                                              case.scale)
        out[b], lse[b] = o[0], l[0]
    return out, lse


def sample_rows(B, H, n, seed=0):
    rng = np.random.default_rng(seed)
    rows = {(0, 0), (B - 1, H - 1)}
    while len(rows) < min(n, B * H):
        rows.add((int(rng.integers(B)), int(rng.integers(H))))
    return sorted(rows)


def default_scale(d):
    return 1.0 / math.sqrt(d)
