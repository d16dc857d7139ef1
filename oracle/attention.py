"""fp64 reference definitions of the decode-attention hot path.

TEST INFRASTRUCTURE ONLY (see the package docstring): imported by tests,
``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py``; never by
the library.

Sources (the pages this library follows), cited by page title and section:

* [KVC-LLM] "KV Cache 如何影响了 LLM Inference" (kakack.github.io),
  §2.2 decode with a KV cache, §四 the unified MHA/GQA/MQA module
  (difference 3: expand+reshape of K/V heads).
* [ARG] "attention-variants-and-kv-cache" (arganzheng.life),
  §二.1-2 decode attention, §三.2 GQA head grouping, §四.2-5 MLA structure,
  decoupled RoPE and matrix absorption, §五.2 FlashAttention IO and the
  flash-decoding split of the sequence with a merge of the normalisers,
  §六.1 paging.
* [MLA] "multi-head-latent-attention" (jianzhnie.github.io), §2 KV equations
  (output with scale 1/sqrt(d_h + d_h^R)), §4 absorption.
* [AIFAQ] aifaq.phimes.top, the decoupled-RoPE Q&A (cache = [c_kv ; k_rope],
  score = content dot + rope dot).
* [CH7] shippingwang.com ch.7 "KV Cache 优化", §7.3 (query head h reads KV
  head h // g; never replicate, check the head axis).

Readings where the pages are silent:

* RoPE: the pages state only that R_m depends on the position m and that
  R_m^T R_n = R_{n-m} ([ARG] §四.4); the frequencies are deferred to another
  article.  Reading: RoFormer-style rotation of interleaved coordinate pairs
  (2i, 2i+1) by the angle pos * theta^(-2i/d_rot), theta = 10000, pos = the
  token's 0-based slot.
* The appended token's slot is the current length seqlens[b]; the caller
  increments the length afterwards ([KVC-LLM] §2.2, [ARG] §二.2: the cache
  only grows by one row per step).
* Empty sequence: output 0, lse = -inf.  An empty split has weight 0.
* Split partials are stored normalised (O_s = o_s / l_s) with
  lse_s = m_s + ln l_s.
"""
from __future__ import annotations

import math

import numpy as np

PAGE = 64

# ----------------------------------------------------------------------------
# bf16 <-> fp64, from the bfloat16 format definition (1 sign bit, 8 exponent
# bits, 7 stored mantissa bits: the top half of an IEEE binary32)
# ----------------------------------------------------------------------------


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening: a bf16 bit pattern is the high 16 bits of a binary32."""
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def bf16_to_f64(t) -> np.ndarray:
    """torch bf16 tensor -> numpy float64 (exact)."""
    import torch
    return bf16_bits_to_f64(t.detach().to("cpu").contiguous()
                            .view(torch.int16).numpy().view(np.uint16))


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even) in one step,
    returning uint16 bit patterns.  Finite normal inputs within bf16 range
    (the only ones this library produces)."""
    x = np.asarray(x, dtype=np.float64)
    u = x.view(np.uint64)
    # bf16 keeps 7 of binary64's 52 mantissa bits: drop 45 bits with RNE
    drop = np.uint64(45)
    lsb = (u >> drop) & np.uint64(1)
    u = (u + (np.uint64(1) << (drop - np.uint64(1))) - np.uint64(1) + lsb)
    u = u & ~((np.uint64(1) << drop) - np.uint64(1))
    r = u.view(np.float64).astype(np.float32)   # exact: 8 significant bits
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------
# E4M3, the 8-bit float of an FP8 KV cache ([ARG] §六.3: FP8 (E4M3) halves the
# bytes per element, with one scale per head or per token).  The format is the
# E4M3 of "FP8 Formats for Deep Learning" (Micikevicius et al., 2022): 1 sign
# bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds
# the subnormals (m/8) * 2^-6; S.1111.111 is NaN; there is no infinity, so
# the largest finite magnitude is 1.75 * 2^8 = 448.
# ----------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_bits_to_f64(codes) -> np.ndarray:
    """Exact value of each E4M3 code (uint8 array)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where(c & 0x80, -mag, mag)


# magnitudes of codes 0x00..0x7E, strictly increasing with the code
_E4M3_MAGS = e4m3_bits_to_f64(np.arange(0x7F))


def f64_to_e4m3_bits(x) -> np.ndarray:
    """Nearest E4M3 code to each value, ties to the even code (mantissa LSB
    0); magnitudes above 448 saturate to 448; NaN gives 0x7F; the sign bit is
    the input's (so a negative value that rounds to zero gives 0x80)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(np.nan_to_num(x)), E4M3_MAX)
    hi = np.searchsorted(_E4M3_MAGS, a, side="left")      # first magnitude >= a
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_MAGS[lo]
    d_hi = _E4M3_MAGS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def dequant_e4m3(codes, scale, head_axis: int = 1) -> np.ndarray:
    """Cache values of an FP8 cache with one scale per KV head ([ARG] §六.3):
    value = E4M3(code) * scale[head], the head on ``head_axis`` (1 for both
    the contiguous [B, n_kv, cap, d] and the paged [pages, n_kv, PAGE, d]
    layouts)."""
    v = e4m3_bits_to_f64(codes)
    shape = [1] * v.ndim
    shape[head_axis] = -1
    return v * np.asarray(scale, dtype=np.float64).reshape(shape)


def gqa_decode_fp8(q, k_codes, v_codes, k_scale, v_scale, seqlens, scale=None,
                   block_table=None, window=0):
    """GQA decode over an E4M3 K/V cache with per-KV-head scales: the plain
    decode of the dequantised cache ([ARG] §六.3: quantisation changes only
    the bytes per element, not the attention)."""
    return gqa_decode(q, dequant_e4m3(k_codes, k_scale), dequant_e4m3(v_codes, v_scale),
                      seqlens, scale, block_table, window)


def dequant_mla_e4m3(codes, kv_scale) -> np.ndarray:
    """Latent rows of an E4M3 MLA cache ([ARG] §六.3: FP8 halves the bytes
    per cached element -- for DeepSeek-V3's 576-value row as for every
    other cache -- with one scale per head or per token; the latent cache
    has a single head).  Reading: one scale for the 512 c_kv values of every
    row and one for its 64 k_R values (the two pieces of the row are
    different tensors, [ARG] §四.2), value = E4M3(code) * scale.
    codes uint8 [..., 576], kv_scale [c_kv scale, k_R scale]."""
    v = e4m3_bits_to_f64(codes)
    s = np.asarray(kv_scale, dtype=np.float64)
    v[..., :512] *= s[0]
    v[..., 512:] *= s[1]
    return v


def mla_decode_absorbed_fp8(q_abs, q_rope, codes, kv_scale, block_table, seqlens,
                            scale=None):
    """MLA absorbed decode over an E4M3 latent cache: the plain absorbed
    decode of the dequantised rows ([ARG] §六.3: quantisation changes the
    bytes per element, not the attention)."""
    return mla_decode_absorbed(q_abs, q_rope, dequant_mla_e4m3(codes, kv_scale),
                               block_table, seqlens, scale)


# ----------------------------------------------------------------------------
# softmax attention of one query block over one key/value sequence
# ----------------------------------------------------------------------------


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Single-step decode attention ([ARG] §二.1, [KVC-LLM] §2.2):
    s_j = scale * q . K_j, p = softmax(s), out = sum_j p_j V_j,
    lse = log sum_j exp(s_j).

    q [H, dk], K [L, dk], V [L, dv] -> out [H, dv], lse [H].  L = 0 gives
    out = 0 and lse = -inf."""
    H = q.shape[0]
    L = K.shape[0]
    if L == 0:
        return np.zeros((H, V.shape[1])), np.full(H, -np.inf)
    s = scale * (q @ K.T)                       # [H, L]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    p = e / l
    out = p @ V
    lse = (m + np.log(l))[:, 0]
    return out, lse


def gather_slots(cache, b: int, slots, block_table=None, head=None):
    """Cache rows ``slots`` of sequence b.  Contiguous caches are
    [B, heads, cap, d] (head given) or [B, cap, d]; paged caches are
    [pages, heads, PAGE, d] or [pages, PAGE, d] with slot j at
    (block_table[b, j // PAGE], j % PAGE) ([ARG] §六.1: the kernel looks up
    logical -> physical block)."""
    j = np.asarray(slots, dtype=np.int64)
    if block_table is None:
        return cache[b, head, j] if head is not None else cache[b, j]
    pages = np.asarray(block_table)[b, j // PAGE]
    if head is not None:
        return cache[pages, head, j % PAGE]
    return cache[pages, j % PAGE]


def gather_tokens(cache, b: int, L: int, block_table=None, head=None):
    """Rows 0..L-1 of sequence b (see gather_slots)."""
    return gather_slots(cache, b, np.arange(L), block_table, head)


def window_slots(n: int, window: int) -> np.ndarray:
    """Cache slots a decode step reads for a sequence of n tokens.

    window = 0: every position 0..n-1, slot = position.  window = w > 0
    (sliding-window attention, [ARG] §五.3 and its mask figure): the query at
    position t = n-1 sees the w positions t-w+1 .. t (the figure marks w
    cells per row; the text's "[t - w, t]" would be w+1 -- reading: w), and
    the cache keeps only those, so position p lives in ring slot p mod w."""
    if window <= 0:
        return np.arange(n)
    pos = np.arange(max(0, n - window), n)
    return pos % window


def gqa_decode(q, k, v, seqlens, scale=None, block_table=None, window=0):
    """MHA / GQA / MQA decode ([ARG] §三.2; [CH7] §7.3; [KVC-LLM] §四).

    q [B, h, d]; k, v contiguous [B, n_kv, cap, d] or paged
    [pages, n_kv, PAGE, d] with block_table [B, max_blocks].  Query head hh
    reads KV head hh // g, g = h / n_kv.  ``window`` > 0 reads a ring cache
    of the last ``window`` positions (window_slots).  Returns out [B, h, d],
    lse [B, h] (natural log)."""
    B, h, d = q.shape
    n_kv = k.shape[1]
    assert h % n_kv == 0
    g = h // n_kv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, h, d))
    lse = np.zeros((B, h))
    for b in range(B):
        slots = window_slots(int(seqlens[b]), window)
        for kv in range(n_kv):
            # the query heads hh with hh // g == kv share this KV head's rows
            heads = slice(kv * g, (kv + 1) * g)
            K = gather_slots(k, b, slots, block_table, kv)
            V = gather_slots(v, b, slots, block_table, kv)
            out[b, heads], lse[b, heads] = attend(q[b, heads], K, V, scale)
    return out, lse


def mla_decode_absorbed(q_abs, q_rope, cache, block_table, seqlens, scale=None):
    """MLA decode with matrix absorption ([ARG] §四.5; [MLA] §4; [AIFAQ]).

    Per head: score_j = scale * (q_abs . c_kv_j + q_rope . k_R_j) with the
    cached row [c_kv (512) ; k_R (64)]; scale defaults to 1/sqrt(128 + 64)
    (the pre-absorption head dim, not 1/sqrt(576)); the output stays in the
    512-d latent space: out = sum_j p_j c_kv_j (V is the first 512 values of
    the same cached row).  q_abs [B, n_h, 512], q_rope [B, n_h, 64],
    cache [pages, PAGE, 576]."""
    B, n_h, dc = q_abs.shape
    if scale is None:
        scale = 1.0 / math.sqrt(128 + 64)
    out = np.zeros((B, n_h, dc))
    lse = np.zeros((B, n_h))
    for b in range(B):
        L = int(seqlens[b])
        rows = gather_tokens(cache, b, L, block_table)       # [L, 576]
        c_kv, k_r = rows[:, :dc], rows[:, dc:]
        if L == 0:
            lse[b] = -np.inf
            continue
        s = scale * (q_abs[b] @ c_kv.T + q_rope[b] @ k_r.T)   # content + rope
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        out[b] = (e / l) @ c_kv
        lse[b] = (m + np.log(l))[:, 0]
    return out, lse


def mla_decode_nonabsorbed(q_nope, q_rope, cache, block_table, seqlens,
                           W_UK, W_UV, scale=None):
    """The literal (prefill-style) MLA path ([ARG] §四.2 and the §四.5
    figure; [MLA] §2): up-project every cached latent to per-head keys and
    values, k^C_{j,h} = W_UK,h c_kv_j and v^C_{j,h} = W_UV,h c_kv_j with
    W_UK [n_h, d_h, 512] and W_UV [n_h, d_v, 512] (column-vector form, W_UK,h
    being head h's 128x512 block), then standard attention of
    q = [q^C ; q^R] against k = [k^C ; k^R] with values v^C.
    Returns the per-head output in value space [B, n_h, d_v]."""
    B, n_h, dh = q_nope.shape
    if scale is None:
        scale = 1.0 / math.sqrt(dh + q_rope.shape[2])
    dv = W_UV.shape[1]
    out = np.zeros((B, n_h, dv))
    lse = np.zeros((B, n_h))
    for b in range(B):
        L = int(seqlens[b])
        rows = gather_tokens(cache, b, L, block_table)
        c_kv, k_r = rows[:, :512], rows[:, 512:]
        for hh in range(n_h):
            kC = c_kv @ W_UK[hh].T                    # [L, d_h]
            vC = c_kv @ W_UV[hh].T                    # [L, d_v]
            K = np.concatenate([kC, k_r], axis=1)
            qf = np.concatenate([q_nope[b, hh], q_rope[b, hh]])[None]
            o, l = attend(qf, K, vC, scale)
            out[b, hh] = o[0]
            lse[b, hh] = l[0]
    return out, lse


def mla_prefill_expand(c_kv, W_UK, W_UV):
    """The up-projection of a prefill chunk ([ARG] §四.6: one ordinary
    weight GEMM over all s tokens; [MLA] §4.2.1: prefill computes k and v
    explicitly): K^C[t, h, :] = W_UK,h c_kv_t and V[t, h, :] = W_UV,h c_kv_t
    for c_kv [s, 512] and W_UK, W_UV [n_h, 128, 512].  Returns both
    [s, n_h, 128]."""
    c = np.asarray(c_kv, dtype=np.float64)
    return (np.einsum("tc,hdc->thd", c, np.asarray(W_UK, dtype=np.float64)),
            np.einsum("tc,hdc->thd", c, np.asarray(W_UV, dtype=np.float64)))


def mla_prefill(q_nope, q_rope, k_nope, k_rope, v, scale=None, kv_offset=None):
    """Causal MLA attention of a prefill chunk on the non-absorbed path
    ([ARG] §四.6: after the up-projection, standard causal attention with
    head dims 192 (q.k) and 128 (v); §五.3 causal mask).

    q_nope [s_q, n_h, 128], q_rope [s_q, n_h, 64] (rotated); k_nope
    [s_kv, n_h, 128], k_rope [s_kv, 64] (rotated, shared by every head),
    v [s_kv, n_h, 128].  Query i sits at position kv_offset + i (default
    s_kv - s_q: the chunk is the newest s_q tokens) and sees keys
    j <= kv_offset + i.  scale defaults to 1/sqrt(192).  Returns out
    [s_q, n_h, 128] and lse [s_q, n_h]."""
    s_q, n_h, dn = q_nope.shape
    s_kv = k_nope.shape[0]
    if kv_offset is None:
        kv_offset = s_kv - s_q
    if scale is None:
        scale = 1.0 / math.sqrt(dn + q_rope.shape[2])
    out = np.zeros((s_q, n_h, v.shape[2]))
    lse = np.zeros((s_q, n_h))
    for hh in range(n_h):
        K = np.concatenate([k_nope[:, hh], k_rope], axis=1)       # [s_kv, 192]
        for i in range(s_q):
            L = min(s_kv, kv_offset + i + 1)
            q = np.concatenate([q_nope[i, hh], q_rope[i, hh]])[None]
            o, l = attend(q, K[:L], v[:L, hh], scale)
            out[i, hh] = o[0]
            lse[i, hh] = l[0]
    return out, lse


# ----------------------------------------------------------------------------
# MLA absorption projections on either side of the absorbed decode ([ARG]
# §四.5; [MLA] §4): W_UK folded into the query, W_UV applied to the latent
# output
# ----------------------------------------------------------------------------


def mla_absorb_q(q_nope, W_UK):
    """Query-side absorption ([ARG] "attention-variants-and-kv-cache" §四.5;
    [MLA] "multi-head-latent-attention" §4): q~_{b,h} = W_UK,h^T q^C_{b,h},
    the 128-wide per-head no-rope query taken into the 512-wide latent space,
    so that q~_{b,h} . c = q^C_{b,h} . (W_UK,h c).  q_nope [B, n_h, d_h],
    W_UK [n_h, d_h, 512] -> [B, n_h, 512]."""
    B, n_h, d_h = q_nope.shape
    out = np.zeros((B, n_h, W_UK.shape[2]))
    for h in range(n_h):
        out[:, h, :] = q_nope[:, h, :] @ W_UK[h]
    return out


def mla_project_out(lat, W_UV):
    """Value-side absorption ([ARG] §四.5; [MLA] §4): the latent output
    o~_{b,h} = sum_j p_j c_j taken to head h's value space,
    o_{b,h} = W_UV,h o~_{b,h} = sum_j p_j (W_UV,h c_j).  lat [B, n_h, 512],
    W_UV [n_h, d_v, 512] -> [B, n_h, d_v]."""
    B, n_h, _ = lat.shape
    out = np.zeros((B, n_h, W_UV.shape[1]))
    for h in range(n_h):
        out[:, h, :] = lat[:, h, :] @ W_UV[h].T
    return out


# ----------------------------------------------------------------------------
# flash-decoding split and merge ([ARG] §五.2, last paragraph: split the KV
# along the sequence, softmax each piece locally, then merge the normalisers)
# ----------------------------------------------------------------------------


def split_partials(q, K, V, scale, bounds):
    """Local softmax over each token range [bounds[s], bounds[s+1]):
    normalised partial outputs O_s [S, H, dv] and lse_s [S, H]."""
    S = len(bounds) - 1
    H = q.shape[0]
    O = np.zeros((S, H, V.shape[1]))
    lse = np.zeros((S, H))
    for s in range(S):
        a, e = bounds[s], bounds[s + 1]
        O[s], lse[s] = attend(q, K[a:e], V[a:e], scale)
    return O, lse


def combine_splits(partial_o, partial_lse, counts=None):
    """Merge S normalised partials per row: M = max_s lse_s,
    w_s = exp(lse_s - M), out = sum_s w_s O_s / sum_s w_s,
    lse = M + ln sum_s w_s.  partial_o [S, R, D], partial_lse [S, R];
    counts [R] limits row r to its first counts[r] partials (None: all S).
    Rows whose partials are all empty get out = 0, lse = -inf."""
    S, R, D = partial_o.shape
    out = np.zeros((R, D))
    lse = np.full(R, -np.inf)
    for r in range(R):
        n = S if counts is None else int(counts[r])
        ls = partial_lse[:n, r]
        if n == 0 or not np.isfinite(ls).any():
            continue
        M = ls.max()
        w = np.exp(ls - M)
        out[r] = (w[:, None] * partial_o[:n, r]).sum(axis=0) / w.sum()
        lse[r] = M + math.log(w.sum())
    return out, lse


# ----------------------------------------------------------------------------
# rotary position embedding and the cache append
# ----------------------------------------------------------------------------


def rope_matrix(pos: float, dim: int, theta: float = 10000.0) -> np.ndarray:
    """The block-diagonal rotation R_pos (reading: interleaved pairs,
    angle_i = pos * theta^(-2i/dim)).  Used by the tests to check
    R_m^T R_n = R_{n-m} ([ARG] §四.4)."""
    R = np.zeros((dim, dim))
    for i in range(dim // 2):
        a = pos * theta ** (-2.0 * i / dim)
        c, s = math.cos(a), math.sin(a)
        R[2 * i, 2 * i], R[2 * i, 2 * i + 1] = c, -s
        R[2 * i + 1, 2 * i], R[2 * i + 1, 2 * i + 1] = s, c
    return R


def rope_rotate(x: np.ndarray, pos, theta: float = 10000.0) -> np.ndarray:
    """Rotate the last axis of x (interleaved pairs) to position(s) ``pos``
    (broadcast over the leading axes)."""
    x = np.asarray(x, dtype=np.float64)
    dim = x.shape[-1]
    i = np.arange(dim // 2)
    inv = theta ** (-2.0 * i / dim)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


def append_rope_mla(cache_bits, block_table, seqlens, c_kv_bits, kr_bits,
                    theta=10000.0, kv_scale=None):
    """Write one new token per sequence into the paged latent cache
    ([ARG] §四.2: c_kv is cached as is, k_R is cached already rotated;
    [KVC-LLM] §2.2: the cache grows by one row).  Inputs are bf16 bit
    patterns (uint16).  Slot: pos = seqlens[b], page block_table[b, pos//64],
    row pos % 64.  Returns a new cache array.

    bf16 cache (kv_scale None): bf16 bit patterns in and out.  E4M3 cache
    (kv_scale = [c_kv scale, k_R scale], [ARG] §六.3; uint8 codes): c_kv code
    = E4M3(c_kv / scale_c) taken from the binary32 quotient (the precision
    the kernel divides in, so these codes are exact), k_R code =
    E4M3(RoPE(k_R) / scale_R) from the binary64 rotation (within one code of
    the kernel's binary32 rotation)."""
    out = np.array(cache_bits, copy=True)
    fp8 = kv_scale is not None
    for b in range(len(seqlens)):
        pos = int(seqlens[b])
        page = int(block_table[b, pos // PAGE])
        row = pos % PAGE
        rot = rope_rotate(bf16_bits_to_f64(kr_bits[b]), pos, theta)
        if fp8:
            s32 = np.asarray(kv_scale, np.float32)
            cq = bf16_bits_to_f64(c_kv_bits[b]).astype(np.float32) / s32[0]
            out[page, row, :512] = f64_to_e4m3_bits(cq.astype(np.float64))
            out[page, row, 512:] = f64_to_e4m3_bits(rot / np.float64(s32[1]))
        else:
            out[page, row, :512] = c_kv_bits[b]
            out[page, row, 512:] = f64_to_bf16_bits(rot)
    return out


def append_rope_gqa(k_bits, v_bits, seqlens, k_new_bits, v_new_bits,
                    block_table=None, theta=10000.0, window=0, k_scale=None,
                    v_scale=None):
    """GQA cache append: K[.., slot, :] = RoPE_pos(k_new) over the whole head
    dim, V[.., slot, :] = v_new, pos = seqlens[b].  slot = pos, or pos mod
    window for a sliding-window ring cache ([ARG] §五.3: the cache keeps the
    last window tokens).  Contiguous [B, n_kv, cap, d] or paged
    [pages, n_kv, PAGE, d] layouts.

    bf16 cache (k_scale None): bf16 bit patterns in and out.  E4M3 cache
    (k_scale, v_scale fp32 [n_kv], [ARG] §六.3): K code = E4M3(RoPE(k) /
    k_scale) from the binary64 rotation; V code = E4M3(v / v_scale) taken
    from the binary32 quotient -- the quantised code is decided in the
    precision the kernel divides in, so V codes are exact while K codes carry
    the rotation's rounding (within one code)."""
    K = np.array(k_bits, copy=True)
    V = np.array(v_bits, copy=True)
    B, n_kv, d = k_new_bits.shape
    fp8 = k_scale is not None
    for b in range(B):
        pos = int(seqlens[b])
        slot = pos % window if window > 0 else pos
        rot = rope_rotate(bf16_bits_to_f64(k_new_bits[b]), pos, theta)
        if fp8:
            kq = f64_to_e4m3_bits(rot / np.asarray(k_scale, np.float64)[:, None])
            vq32 = (bf16_bits_to_f64(v_new_bits[b]).astype(np.float32)
                    / np.asarray(v_scale, np.float32)[:, None])
            vq = f64_to_e4m3_bits(vq32.astype(np.float64))
        else:
            kq = f64_to_bf16_bits(rot)
            vq = v_new_bits[b]
        if block_table is None:
            K[b, :, slot] = kq
            V[b, :, slot] = vq
        else:
            page = int(block_table[b, slot // PAGE])
            K[page, :, slot % PAGE] = kq
            V[page, :, slot % PAGE] = vq
    return K, V
