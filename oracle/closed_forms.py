"""Closed-form KV-cache sizes and decode-attention intensities, restated from
the pages' prose formulas.

TEST INFRASTRUCTURE ONLY: imported by the tests that pin the oracle to the
numbers the pages print.  ``bench.py`` keeps its own byte and FLOP counts.

Each function is one formula of the text, in that text's terms:

* [ARG] "attention-variants-and-kv-cache", §二.3 (the KV-cache size
  formula: K and V, for every layer and every KV head, d_head values each),
  §三.3 (a KV element read once feeds g query heads at 2 FLOPs each),
  §四.3 (MLA caches one latent of d_c values plus one decoupled rope key of
  d_h^R values per token per layer, shared by all heads), §四.6 (per cached
  token and layer: a (d_c + d_h^R)-long score dot and a d_c-long weighted
  sum for each of the n_h heads).
* [AIFAQ] aifaq.phimes.top, decoupled-RoPE Q&A (the same 512 + 64 values,
  compared with 2 * d_model for MHA).
* [MLA] "multi-head-latent-attention", §4.2.3 (memory read by the absorbed
  decode over the standard one).
"""
from __future__ import annotations


def kv_cache_bytes_per_token(layers: int, n_kv_heads: int, head_dim: int,
                             elem_bytes: int = 2) -> int:
    """[ARG] §二.3: the factor 2 counts K and V; MHA has n_kv_heads = n_h,
    MQA n_kv_heads = 1.  With layers = 1 and elem_bytes = 1 this is the
    number of cached values per token per layer."""
    return 2 * layers * n_kv_heads * head_dim * elem_bytes


def mla_latent_values_per_token(d_c: int = 512, d_rope: int = 64) -> int:
    """[ARG] §四.3 / [AIFAQ]: c_kv (d_c values) and k_R (d_rope values) are
    the whole per-layer cache entry of a token."""
    return d_c + d_rope


def mla_cache_bytes_per_token(layers: int, d_c: int = 512, d_rope: int = 64,
                              elem_bytes: int = 2) -> int:
    """[ARG] §四.3: one latent entry per layer, no per-head factor."""
    return layers * mla_latent_values_per_token(d_c, d_rope) * elem_bytes


def grouped_decode_intensity(group: int, elem_bytes: int = 2) -> float:
    """[ARG] §三.3: FLOPs per byte of KV read in a decode step.  A K element
    meets the query of each of the `group` heads sharing it in one
    multiply-add (2 FLOPs), and so does the V element in the weighted sum;
    each of them costs elem_bytes of reading."""
    return 2.0 * group / elem_bytes


def mla_decode_flops_per_token(n_heads: int, d_c: int = 512, d_rope: int = 64) -> int:
    """[ARG] §四.6: every head takes one dot of the full cached row for its
    score and one weighted sum of the latent for its output, 2 FLOPs per
    dimension of each."""
    score_dims = d_c + d_rope
    out_dims = d_c
    return n_heads * 2 * (score_dims + out_dims)


def mla_decode_intensity(n_heads: int, d_c: int = 512, d_rope: int = 64,
                         elem_bytes: int = 2) -> float:
    """[ARG] §四.6: those FLOPs over the bytes of one cached row."""
    return mla_decode_flops_per_token(n_heads, d_c, d_rope) / (
        mla_latent_values_per_token(d_c, d_rope) * elem_bytes)


def mla_vs_mha_read_ratio(s: float, d_c: int = 512, d_h: int = 128, n_h: int = 128) -> float:
    """[MLA] §4.2.3: the absorbed decode reads n_h query rows and s latent
    rows of d_c values, standard MHA reads one query row and s cached rows of
    d_h values for each of the n_h heads."""
    read_absorbed = d_c * (n_h + s)
    read_mha = d_h * n_h * (1 + s)
    return read_absorbed / read_mha
