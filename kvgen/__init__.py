"""Seeded synthetic inputs for single-token decode attention.

This module is shared by the fp64 oracle (``oracle/``) and the CUDA path
(``decode_attention_kv_softmax_b300``).  It only draws random numbers and lays
them out in the cache formats; it holds none of the attention arithmetic
(no dot products, no softmax, no rotary embedding), so the two sides that it
feeds stay independent.

Workloads (the five decode configurations the library is measured on):

=====  =====================================================================
name   shapes
=====  =====================================================================
C0     tiny GQA: B=1, h=4, n_kv=2, d=64, L=128 cached tokens, fp32 out
C1     Llama-3-8B-shaped GQA: B=32, h=32, n_kv=8, d=128, seqlens U[1024,4096],
       contiguous K/V [B, 8, 4096, 128]
C2     Llama-2-7B-shaped MHA (n_kv=32) and MQA (n_kv=1): B=16, h=32, d=128,
       L=4096; one q shared by both
C3     DeepSeek-V3-shaped MLA absorbed decode: B=64, n_h=128, seqlens
       U[512,4096], paged latent cache [pages, 64, 576], shuffled block table
C4     long ragged mix: MLA as C3 with B=8 and seqlens U[16384,131072]; GQA
       h=64, n_kv=8, d=128 (Llama-3-70B shape), B=8, same seqlen range,
       paged 64-token blocks in shuffled order
=====  =====================================================================

Every tensor is bf16 drawn from N(0, 1) (q of MLA: N(0,1)/sqrt(512)) with a
``torch.Generator`` seeded per configuration (seed = 1000 + config index).
The decoupled rope key k_R of the MLA cache is drawn directly from N(0, 1):
a rotary embedding rotates each coordinate pair by an angle, and a standard
2-D normal is invariant under rotation, so RoPE(N(0,1)) has exactly the
N(0,1) distribution the workload names.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE = 64          # tokens per KV page (block) in every paged layout here
D_C = 512          # MLA latent width (kv_lora_rank)
D_R = 64           # MLA decoupled rope key width (qk_rope_head_dim)
D_LATENT = D_C + D_R

SEED_BASE = 1000


@dataclass
class GqaCase:
    """One GQA/MQA/MHA decode problem.  ``k``/``v`` are contiguous
    [B, n_kv, cap, d] when ``block_table`` is None, else paged
    [num_pages, n_kv, PAGE, d]."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    seqlens: torch.Tensor            # int32 [B]
    block_table: torch.Tensor | None  # int32 [B, max_blocks] or None
    scale: float
    cap: int                          # tokens addressable per sequence
    meta: dict = field(default_factory=dict)
    # E4M3 caches: k, v hold uint8 codes and these the per-KV-head fp32 scales
    k_scale: torch.Tensor | None = None
    v_scale: torch.Tensor | None = None
    window: int = 0                   # > 0: ring cache of the last `window` tokens

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def h(self):
        return self.q.shape[1]

    @property
    def d(self):
        return self.q.shape[2]

    @property
    def n_kv(self):
        return self.k.shape[1]


@dataclass
class MlaCase:
    """One MLA absorbed decode problem over a paged latent cache."""
    q_abs: torch.Tensor      # bf16 [B, n_h, 512]
    q_rope: torch.Tensor     # bf16 [B, n_h, 64]
    cache: torch.Tensor      # bf16 [num_pages, PAGE, 576]
    seqlens: torch.Tensor    # int32 [B]
    block_table: torch.Tensor  # int32 [B, max_blocks]
    scale: float
    meta: dict = field(default_factory=dict)
    # E4M3 cache: cache holds uint8 codes and this the fp32 scales
    # [c_kv scale, k_R scale]
    kv_scale: torch.Tensor | None = None

    @property
    def B(self):
        return self.q_abs.shape[0]

    @property
    def n_h(self):
        return self.q_abs.shape[1]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g, device, std=1.0):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def draw_seqlens(B: int, lo: int, hi: int, g, device) -> torch.Tensor:
    """Integer sequence lengths uniform on [lo, hi] (inclusive)."""
    return torch.randint(lo, hi + 1, (B,), generator=g, device=device,
                         dtype=torch.int64).to(torch.int32)


def shuffled_block_table(seqlens: torch.Tensor, g, device, spare_pages: int = 0,
                         max_blocks: int | None = None):
    """Give each sequence ceil(len/PAGE) pages drawn from one random
    permutation of all pages, so logical order and physical order disagree.
    Returns (block_table int32 [B, max_blocks], num_pages).  Unused table
    entries are -1.  ``spare_pages`` extra physical pages stay unreferenced
    (used as canaries by the tests)."""
    sl = seqlens.to("cpu").tolist()
    need = [(s + PAGE - 1) // PAGE for s in sl]
    total = sum(need)
    num_pages = total + spare_pages
    mb = max(need + [1]) if max_blocks is None else max_blocks
    perm = torch.randperm(num_pages, generator=g, device=device).to("cpu")
    bt = torch.full((len(sl), mb), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    return bt.to(device), num_pages


# ----------------------------------------------------------------------------
# generic builders
# ----------------------------------------------------------------------------

def gqa_case(B, h, n_kv, d, *, seqlens=None, lo=None, hi=None, cap=None,
             paged=False, seed=SEED_BASE, device="cpu", q=None,
             spare_pages=0, scale=None, kv_dtype="bf16", window=0) -> GqaCase:
    """Build a GQA decode problem.  Either pass explicit ``seqlens`` (list or
    tensor) or a range [lo, hi].  ``cap`` defaults to the longest cached
    length rounded up to PAGE for contiguous caches.

    ``window`` > 0 makes a ring cache of ``window`` slots: seqlens count every
    token of the sequence (and may exceed the capacity) while only
    min(seqlen, window) slots hold data.  ``kv_dtype="fp8"`` turns K and V
    into E4M3 codes (see fp8_codes)."""
    g = _gen(seed, device)
    if seqlens is None:
        sl = draw_seqlens(B, lo, hi, g, device)
    else:
        sl = torch.as_tensor(seqlens, dtype=torch.int32).to(device)
    if q is None:
        q = _randn_bf16((B, h, d), g, device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    held = sl.clamp(max=window) if window > 0 else sl      # slots holding data
    ring_pages = (window + PAGE - 1) // PAGE                 # a ring has >= window slots
    if not paged:
        if cap is None:
            mx = int(held.max().item()) if B > 0 else 0
            cap = max(PAGE, (mx + PAGE - 1) // PAGE * PAGE, ring_pages * PAGE)
        k = _randn_bf16((B, n_kv, cap, d), g, device)
        v = _randn_bf16((B, n_kv, cap, d), g, device)
        case = GqaCase(q, k, v, sl, None, scale, cap, window=window)
    else:
        need = [(int(x) + PAGE - 1) // PAGE for x in held.to("cpu").tolist()]
        mb = max(need + [1, ring_pages])
        bt, num_pages = shuffled_block_table(held, g, device, spare_pages, mb)
        k = _randn_bf16((num_pages, n_kv, PAGE, d), g, device)
        v = _randn_bf16((num_pages, n_kv, PAGE, d), g, device)
        cap = bt.shape[1] * PAGE
        case = GqaCase(q, k, v, sl, bt, scale, cap, {"num_pages": num_pages},
                       window=window)
    if kv_dtype == "fp8":
        case.k, case.k_scale = fp8_codes(case.k, g, device)
        case.v, case.v_scale = fp8_codes(case.v, g, device)
    elif kv_dtype != "bf16":
        raise ValueError(kv_dtype)
    return case


def fp8_codes(x: torch.Tensor, g, device):
    """Stand-in for a quantised E4M3 cache with one scale per KV head (axis
    1): each head's values are the drawn N(0,1) values times a per-head
    spread sigma_h ~ U[0.25, 4] (so that a scale taken from the wrong head is
    visible), cast by torch to float8_e4m3fn with scale_h = max|x_h| / 448.
    Returns (uint8 codes of x's shape, fp32 scales [n_kv])."""
    n_kv = x.shape[1]
    sigma = torch.empty(n_kv, device=device).uniform_(0.25, 4.0, generator=g)
    xs = x.float() * sigma.view(1, -1, 1, 1)
    amax = xs.abs().amax(dim=(0, 2, 3)).clamp(min=1e-6)
    scale = (amax / 448.0).to(torch.float32)
    codes = (xs / scale.view(1, -1, 1, 1)).clamp(-448.0, 448.0)
    codes = codes.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def mla_fp8_codes(cache: torch.Tensor, g, device):
    """Stand-in for a quantised E4M3 latent cache: the drawn N(0,1) values
    of the row (the same distribution as the bf16 cache), cast by torch to
    float8_e4m3fn with one scale per piece, max|x| / 448 over the c_kv values
    and over the k_R values.  Returns (uint8 codes of the cache's shape,
    fp32 [scale_c, scale_R]).  ``g`` is unused (kept for a uniform call)."""
    x = cache.float()
    amax = torch.stack([x[..., :D_C].abs().amax(), x[..., D_C:].abs().amax()]).clamp(min=1e-6)
    scale = (amax / 448.0).to(torch.float32)
    x[..., :D_C] /= scale[0]
    x[..., D_C:] /= scale[1]
    codes = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def mla_case(B, n_h=128, *, seqlens=None, lo=None, hi=None, seed=SEED_BASE,
             device="cpu", spare_pages=0, max_blocks=None, kv_dtype="bf16") -> MlaCase:
    """An MLA decode problem; ``kv_dtype="fp8"`` turns the latent cache into
    E4M3 codes (see mla_fp8_codes) drawn after every other input, so the
    queries, lengths and block table are those of the bf16 case."""
    g = _gen(seed, device)
    if seqlens is None:
        sl = draw_seqlens(B, lo, hi, g, device)
    else:
        sl = torch.as_tensor(seqlens, dtype=torch.int32).to(device)
    q_abs = _randn_bf16((B, n_h, D_C), g, device, std=1.0 / math.sqrt(512))
    q_rope = _randn_bf16((B, n_h, D_R), g, device, std=1.0 / math.sqrt(512))
    bt, num_pages = shuffled_block_table(sl, g, device, spare_pages, max_blocks)
    cache = _randn_bf16((num_pages, PAGE, D_LATENT), g, device)
    scale = 1.0 / math.sqrt(128 + 64)
    case = MlaCase(q_abs, q_rope, cache, sl, bt, scale, {"num_pages": num_pages})
    if kv_dtype == "fp8":
        case.cache, case.kv_scale = mla_fp8_codes(cache, g, device)
    elif kv_dtype != "bf16":
        raise ValueError(kv_dtype)
    return case


def mla_proj_case(B, n_h=128, *, seed=SEED_BASE, device="cpu"):
    """Inputs of the two MLA absorption projections: q_nope [B, n_h, 128],
    W_UK and W_UV [n_h, 128, 512], all bf16 ~ N(0, 1) scaled so that every
    output element has unit variance (W_UK by 1/sqrt(128): 128 terms;
    W_UV by 1/sqrt(512): 512 terms)."""
    g = _gen(seed, device)
    q_nope = _randn_bf16((B, n_h, 128), g, device)
    W_UK = _randn_bf16((n_h, 128, D_C), g, device, std=1.0 / math.sqrt(128))
    W_UV = _randn_bf16((n_h, 128, D_C), g, device, std=1.0 / math.sqrt(D_C))
    return q_nope, W_UK, W_UV


def mla_prefill_case(s_kv, s_q, n_h=128, *, seed=SEED_BASE, device="cpu"):
    """Inputs of a non-absorbed MLA prefill chunk: c_kv [s_kv, 512] and the
    rotated rope key k_rope [s_kv, 64] ~ N(0, 1) (a rotation keeps N(0,1),
    see the module docstring), W_UK, W_UV [n_h, 128, 512] ~ N(0, 1/512) so
    that the up-projected keys and values are ~N(0, 1), and the chunk's
    queries q_nope [s_q, n_h, 128], q_rope [s_q, n_h, 64] ~ N(0, 1); all
    bf16.  Returns a dict."""
    g = _gen(seed, device)
    return {
        "c_kv": _randn_bf16((s_kv, D_C), g, device),
        "k_rope": _randn_bf16((s_kv, D_R), g, device),
        "W_UK": _randn_bf16((n_h, 128, D_C), g, device, std=1.0 / math.sqrt(D_C)),
        "W_UV": _randn_bf16((n_h, 128, D_C), g, device, std=1.0 / math.sqrt(D_C)),
        "q_nope": _randn_bf16((s_q, n_h, 128), g, device),
        "q_rope": _randn_bf16((s_q, n_h, D_R), g, device),
    }


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------

CONFIGS = {
    "C0": dict(kind="gqa", B=1, h=4, n_kv=2, d=64, L=128),
    "C1": dict(kind="gqa", B=32, h=32, n_kv=8, d=128, lo=1024, hi=4096, cap=4096),
    "C2-MHA": dict(kind="gqa", B=16, h=32, n_kv=32, d=128, L=4096),
    "C2-MQA": dict(kind="gqa", B=16, h=32, n_kv=1, d=128, L=4096),
    "C3": dict(kind="mla", B=64, n_h=128, lo=512, hi=4096),
    "C4-MLA": dict(kind="mla", B=8, n_h=128, lo=16384, hi=131072),
    "C4-GQA": dict(kind="gqa", B=8, h=64, n_kv=8, d=128, lo=16384, hi=131072,
                   paged=True),
}
CONFIG_INDEX = {"C0": 0, "C1": 1, "C2-MHA": 2, "C2-MQA": 2, "C3": 3,
                "C4-MLA": 4, "C4-GQA": 4}


def config_case(name: str, device="cpu", kv_dtype="bf16"):
    """The named workload with its seed (1000 + config index).  C2-MHA and
    C2-MQA draw the same q (the seed's first draw) and independent K/V.
    ``kv_dtype="fp8"`` turns the cache into E4M3 codes (GQA: per-KV-head
    scales; MLA: a c_kv and a k_R scale)."""
    c = CONFIGS[name]
    if kv_dtype != "bf16":
        if kv_dtype != "fp8":
            raise ValueError(kv_dtype)
        case = config_case(name, device)
        if c["kind"] == "mla":
            g = _gen(SEED_BASE + 500 + CONFIG_INDEX[name], device)
            case.cache, case.kv_scale = mla_fp8_codes(case.cache, g, device)
            return case
        g = _gen(SEED_BASE + 500 + CONFIG_INDEX[name], device)
        case.k, case.k_scale = fp8_codes(case.k, g, device)
        case.v, case.v_scale = fp8_codes(case.v, g, device)
        return case
    seed = SEED_BASE + CONFIG_INDEX[name]
    if c["kind"] == "mla":
        return mla_case(c["B"], c["n_h"], lo=c["lo"], hi=c["hi"], seed=seed,
                        device=device)
    if name.startswith("C2"):
        gq = _gen(seed, device)
        q = _randn_bf16((c["B"], c["h"], c["d"]), gq, device)
        sub = 1 if name == "C2-MHA" else 2
        return gqa_case(c["B"], c["h"], c["n_kv"], c["d"],
                        seqlens=[c["L"]] * c["B"], cap=c["L"],
                        seed=seed * 10 + sub, device=device, q=q)
    if "L" in c:
        return gqa_case(c["B"], c["h"], c["n_kv"], c["d"],
                        seqlens=[c["L"]] * c["B"], cap=c["L"], seed=seed,
                        device=device)
    return gqa_case(c["B"], c["h"], c["n_kv"], c["d"], lo=c["lo"], hi=c["hi"],
                    cap=c.get("cap"), paged=c.get("paged", False), seed=seed,
                    device=device)


def append_inputs_mla(B, seed, device="cpu"):
    """New-token latent row pieces: c_kv [B,512] and the un-rotated rope key
    [B,64], both bf16 N(0,1)."""
    g = _gen(seed, device)
    return _randn_bf16((B, D_C), g, device), _randn_bf16((B, D_R), g, device)


def append_inputs_gqa(B, n_kv, d, seed, device="cpu"):
    """New-token k (un-rotated) and v, bf16 N(0,1) [B, n_kv, d]."""
    g = _gen(seed, device)
    return _randn_bf16((B, n_kv, d), g, device), _randn_bf16((B, n_kv, d), g, device)
