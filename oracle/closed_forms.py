"""Closed-form KV-cache sizes and decode-attention intensities.

TEST INFRASTRUCTURE ONLY: imported by the tests that pin the oracle to the
numbers the pages print.  ``bench.py`` keeps its own byte and FLOP counts.
These formulas are restated from the pages:

* [ARG] "attention-variants-and-kv-cache", §二.3 (bytes per token
  = 2 * layers * n_kv * d_head * bytes/elem), §三.3 (decode intensity: each
  KV element read serves g query heads at 2 FLOPs each -> g FLOP/byte in
  bf16), §四.3 (MLA caches d_c + d_h^R = 576 values per token per layer),
  §四.6 (MLA FLOPs per cached token per layer = n_h * 2 * (576 + 512)).
* [AIFAQ] aifaq.phimes.top, decoupled-RoPE Q&A (576 elements, 17.8x vs MHA
  at d_model = 5120, 60 layers * 576 * 2 B).
* [MLA] "multi-head-latent-attention", §4.2.3 (memory-read ratio
  M_MLA / M_MHA = d_c (n_h + s) / (d_h n_h (1 + s))).
"""
from __future__ import annotations


def kv_elems_per_token_per_layer(attn: str, n_heads=0, n_kv_heads=0,
                                 head_dim=0, d_c=0, d_rope=0) -> int:
    if attn == "mha":
        return 2 * n_heads * head_dim
    if attn == "gqa":
        return 2 * n_kv_heads * head_dim
    if attn == "mqa":
        return 2 * head_dim
    if attn == "mla":
        return d_c + d_rope
    raise ValueError(attn)


def kv_bytes_per_token(layers: int, elems_per_layer: int, bytes_per_elem=2) -> int:
    return layers * elems_per_layer * bytes_per_elem


def decode_intensity(attn: str, n_heads: int, elems_per_layer: int,
                     head_dim=0, d_c=0, d_rope=0, bytes_per_elem=2) -> float:
    """FLOPs per byte of KV read, per cached token per layer: every query
    head does a K dot and a V weighted sum, 2 FLOPs per dimension."""
    if attn == "mla":
        flops = n_heads * 2 * ((d_c + d_rope) + d_c)
    else:
        flops = n_heads * 2 * (head_dim + head_dim)
    return flops / (elems_per_layer * bytes_per_elem)


def mla_flops_per_token(n_heads: int, d_c=512, d_rope=64) -> int:
    return n_heads * 2 * ((d_c + d_rope) + d_c)


def mla_vs_mha_read_ratio(s: float, d_c=512, d_h=128, n_h=128) -> float:
    return d_c * (n_h + s) / (d_h * n_h * (1 + s))
