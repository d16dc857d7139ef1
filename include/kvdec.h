/*
 * kvdec.h -- C ABI of libkvdec: single-token decode attention over a KV cache
 * on NVIDIA B300 (sm_103a).
 *
 * Four operations (plus helpers):
 *   kvdec_gqa_decode           MHA / GQA / MQA split-KV decode
 *   kvdec_mla_decode_absorbed  MLA decode over the 576-wide latent cache
 *   kvdec_append_rope          write one new token per sequence into a cache
 *   kvdec_combine_splits       log-sum-exp merge of split partial outputs
 *
 * Sources, cited by page title and section:
 *   [KVC-LLM] "KV Cache 如何影响了 LLM Inference" (kakack.github.io)
 *   [ARG]     "attention-variants-and-kv-cache" (arganzheng.life)
 *   [MLA]     "multi-head-latent-attention" (jianzhnie.github.io)
 *   [AIFAQ]   aifaq.phimes.top (decoupled-RoPE Q&A)
 *   [CH7]     shippingwang.com ch.7 "KV Cache 优化"
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller, dense
 *     row-major in the stated shape.  bf16 is IEEE-style bfloat16.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and allocates nothing.
 *   - Host-side argument checks run before any launch; a failed check returns
 *     an error status and launches nothing.  C++ exceptions never cross the
 *     ABI.  kvdec_last_error() gives a human-readable reason (per thread).
 *   - Device-side problems (a block-table entry outside [0, num_pages), a
 *     sequence length outside [0, capacity], a bounded wait that ran out) do
 *     not fault or trap: kernels keep every access in bounds, OR a
 *     KVDEC_DEVERR_* bit into *error_flag (when error_flag is not NULL) and
 *     the affected outputs are unspecified.  The caller reads the word after
 *     synchronising.
 *   - Calls that share a workspace or an output buffer must not overlap on
 *     the GPU.
 */
#ifndef KVDEC_H
#define KVDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVDEC_ABI_VERSION 3
#define KVDEC_PAGE_SIZE 64      /* tokens per KV page (block) */
#define KVDEC_MLA_DC 512        /* MLA latent width d_c */
#define KVDEC_MLA_DR 64         /* MLA decoupled rope key width d_h^R */

typedef enum kvdec_status {
    KVDEC_OK = 0,
    KVDEC_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment */
    KVDEC_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim 96) */
    KVDEC_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    KVDEC_ERR_WORKSPACE = 4      /* workspace missing or too small */
} kvdec_status;

/* bits OR-ed into *error_flag by the kernels */
#define KVDEC_DEVERR_BAD_PAGE 0x1u   /* block-table entry outside [0, num_pages) */
#define KVDEC_DEVERR_SEQLEN 0x2u     /* seqlen < 0 or > capacity (clamped) */
#define KVDEC_DEVERR_TIMEOUT 0x4u    /* a bounded device wait ran out */

typedef enum kvdec_dtype { KVDEC_F32 = 0, KVDEC_BF16 = 1 } kvdec_dtype;

/* Element format of a K/V cache ([ARG] §六.3: quantising the cache to FP8
 * E4M3 halves the bytes per element, with one scale per head or per token).
 * KVDEC_KV_FP8_E4M3: every cached element is one E4M3 byte (the format of
 * "FP8 Formats for Deep Learning", Micikevicius et al. 2022), and the value
 * it stands for is E4M3(code) * scale: for a GQA cache one fp32 scale per KV
 * head for K and one for V; for the MLA latent cache one for the 512 c_kv
 * values of every row and one for its 64 k_R values. */
typedef enum kvdec_kv_format { KVDEC_KV_BF16 = 0, KVDEC_KV_FP8_E4M3 = 1 } kvdec_kv_format;

/* ------------------------------------------------------------------------ */
/* MHA / GQA / MQA decode                                                   */
/* ------------------------------------------------------------------------ */
/*
 * For every sequence b and query head h (g = num_heads / num_kv_heads):
 *   s_j  = scale * q[b,h,:] . K[b, h/g, j, :]            for j < seqlens[b]
 *   out[b,h,:] = sum_j softmax(s)_j V[b, h/g, j, :],   lse[b,h] = ln sum_j e^{s_j}
 * ([ARG] §二.1 decode attention, §三.2 grouping; [CH7] §7.3: query head h
 * reads KV head h // g and KV is never replicated; [KVC-LLM] §2.2).
 * The sequence is split across CTAs and the pieces merged by their
 * log-sum-exp ([ARG] §五.2, flash-decoding); the result does not depend on
 * the split.  seqlens[b] == 0 gives out = 0, lse = -inf.
 *
 * Layouts
 *   q      bf16 [batch, num_heads, head_dim]
 *   k, v   block_table == NULL: bf16 [batch, num_kv_heads, capacity, head_dim]
 *          else paged:          bf16 [num_pages, num_kv_heads, 64, head_dim];
 *          token j of sequence b lives in page block_table[b, j/64], row j%64
 *          ([ARG] §六.1).  Pages may be shared between sequences.
 *   block_table int32 [batch, max_blocks] (paged only)
 *   seqlens int32 [batch]
 *   out    [batch, num_heads, head_dim], F32 or BF16 (out_dtype)
 *   lse    fp32 [batch, num_heads] or NULL
 * FP8 cache (kv_format = KVDEC_KV_FP8_E4M3, head_dim 128 only): k and v hold
 *   one E4M3 byte per element in the same layouts; k_scale and v_scale are
 *   fp32 [num_kv_heads] device arrays (required); K = E4M3(k) * k_scale[kv],
 *   V = E4M3(v) * v_scale[kv].  q is taken in f16 (|q| < 65504).
 * Sliding window (window = w > 0, [ARG] §五.3: the query at position t sees
 *   positions t-w+1 .. t and the cache keeps only those): the cache is a ring
 *   of w slots, position p in slot p mod w (kvdec_append_rope with the same
 *   window writes it so); seqlens[b] counts every token of the sequence and
 *   may exceed the capacity, and the step reads the min(seqlens[b], w) slots.
 *   w must not exceed the capacity (contiguous) or max_blocks * 64 (paged).
 * Supported: head_dim in {64, 128}; num_heads % num_kv_heads == 0;
 * q, k, v, out 16-byte aligned.  scale == 0 selects 1/sqrt(head_dim); any other
 * scale must be positive and finite (KVDEC_ERR_INVALID_ARG otherwise).
 * Workspace: at least kvdec_gqa_workspace_bytes(p) bytes, 256-byte aligned,
 * no initialisation needed (split counters are tagged with a per-call epoch).
 * It holds the split partials and their counters; calls that share it must
 * not overlap on the GPU.  Its size follows the launch the call will make:
 * batch, the head counts, head_dim, kv_format, the cache's capacity
 * (capacity, or max_blocks when paged), window and max_ctas all enter it, so
 * query it with the same values the decode call will carry.
 */
typedef struct kvdec_gqa_params {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* block_table;
    const int32_t* seqlens;
    int32_t batch;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t capacity;        /* contiguous: cached tokens per (b, kv head) */
    int32_t num_pages;       /* paged only */
    int32_t max_blocks;      /* paged only */
    float scale;
    void* out;
    int32_t out_dtype;       /* kvdec_dtype */
    float* lse;
    void* workspace;
    size_t workspace_bytes;
    uint32_t* error_flag;    /* optional */
    int32_t max_ctas;        /* work items (CTAs); 0 = one wave of resident CTAs */
    int32_t kv_format;       /* kvdec_kv_format; 0 = bf16 */
    const float* k_scale;    /* FP8 only: fp32 [num_kv_heads] */
    const float* v_scale;    /* FP8 only: fp32 [num_kv_heads] */
    int32_t window;          /* 0 = all seqlens[b] tokens; w > 0 = ring cache of w slots */
    int32_t reserved;
} kvdec_gqa_params;

size_t kvdec_gqa_workspace_bytes(const kvdec_gqa_params* p);
kvdec_status kvdec_gqa_decode(const kvdec_gqa_params* p, void* stream);

/* ------------------------------------------------------------------------ */
/* GQA decode for callers that cannot allocate                               */
/* ------------------------------------------------------------------------ */
/*
 * No counterpart in the source pages: this is a deployment variant of
 * kvdec_gqa_decode, not part of the method.
 *
 * Same operation, arguments and results as kvdec_gqa_decode, for callers that
 * cannot hand the library a device workspace -- for example a plugin inside
 * another runtime that owns all device memory through its own allocator, or
 * a serving loop that commits all free HBM to the KV cache at start-up and
 * allows no allocation while decoding.  p->workspace and p->workspace_bytes
 * are ignored: the split scratch lives in a fixed array of
 * KVDEC_NOALLOC_SCRATCH_BYTES bytes inside the library, held on every GPU
 * where the library's code is loaded until the process exits.  The call
 * allocates nothing.
 *   - The first call on each device looks up the array's device address
 *     (with that device current); make it before any stream capture there.
 *     After a reset of the device (cudaDeviceReset) the next call looks the
 *     address up again in the new context: make that call before any
 *     capture too.
 *   - Problems whose scratch would exceed the array are rejected with
 *     KVDEC_ERR_WORKSPACE and a message giving the size needed (lower
 *     max_ctas or batch, or use kvdec_gqa_decode).
 *   - All calls on a device share the array and it keeps the last call's
 *     contents; nothing in it needs to start at zero (the split counters
 *     carry a per-call epoch).  Calls that overlap on the GPU race on it:
 *     serialise them.
 */
#define KVDEC_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
kvdec_status kvdec_gqa_decode_noalloc(const kvdec_gqa_params* p, void* stream);

/* ------------------------------------------------------------------------ */
/* MLA absorbed decode                                                       */
/* ------------------------------------------------------------------------ */
/*
 * DeepSeek-style MLA after matrix absorption ([ARG] §四.5; [MLA] §4;
 * [AIFAQ]): every cached token stores one 576-value row
 * [c_kv (512) ; k_R (64, already rotated)] shared by all heads.  For each
 * sequence b and head h:
 *   s_j  = scale * (q_absorbed[b,h,:] . c_kv_j + q_rope[b,h,:] . k_R_j)
 *   out[b,h,:] = sum_j softmax(s)_j c_kv_j        (latent space, 512 wide)
 * V is the first 512 values of the same row.  scale == 0 selects
 * 1/sqrt(128 + 64) = 1/sqrt(192), the pre-absorption head dim; any other
 * scale must be positive and finite (KVDEC_ERR_INVALID_ARG otherwise).
 * W_UK (folded into q_absorbed) and W_UV / W_O (applied to out) are the
 * caller's.
 *
 * Layouts
 *   q_absorbed bf16 [batch, num_heads, 512]; q_rope bf16 [batch, num_heads, 64]
 *   cache bf16 [num_pages, 64, 576]; block_table int32 [batch, max_blocks]
 *   seqlens int32 [batch]; out [batch, num_heads, 512] F32 or BF16;
 *   lse fp32 [batch, num_heads] or NULL
 * FP8 latent cache (kv_format = KVDEC_KV_FP8_E4M3): cache holds uint8 E4M3
 *   codes [num_pages, 64, 576] (576 bytes a token); kv_scale is a device
 *   array fp32 [2] (required): c_kv = E4M3(code[0:512]) * kv_scale[0],
 *   k_R = E4M3(code[512:576]) * kv_scale[1].  The call first widens the
 *   pages it reads into a bf16 copy in the workspace (each value
 *   E4M3(code) * scale rounded once to bf16, nearest-even), then runs the
 *   bf16 decode on the copy: the FP8 cache halves the bytes held in HBM,
 *   not the bytes a step moves.  The workspace grows by
 *   batch * max_blocks * (73728 + 4) bytes; batch * max_blocks * 64 must stay
 *   below 2^31.
 * Supported: num_heads == 128 (tensor-core tile height) and
 * batch <= kvdec_mla_max_batch(): the kernel keeps a per-sequence tile table
 * in shared memory beside its cache stages, so a larger batch is rejected
 * with KVDEC_ERR_INVALID_ARG before any launch (split it into calls).
 * Workspace: as for kvdec_gqa_decode (no initialisation needed), plus the
 * widened copy for an FP8 cache.
 */
typedef struct kvdec_mla_params {
    const void* q_absorbed;
    const void* q_rope;
    const void* cache;
    const int32_t* block_table;
    const int32_t* seqlens;
    int32_t batch;
    int32_t num_heads;
    int32_t num_pages;
    int32_t max_blocks;
    float scale;
    void* out;
    int32_t out_dtype;
    float* lse;
    void* workspace;
    size_t workspace_bytes;
    uint32_t* error_flag;
    int32_t max_ctas;        /* 0 = one full wave of CTA pairs */
    int32_t kv_format;       /* kvdec_kv_format; 0 = bf16 */
    const float* kv_scale;   /* FP8 only: fp32 [2] = {c_kv scale, k_R scale} */
} kvdec_mla_params;

size_t kvdec_mla_workspace_bytes(const kvdec_mla_params* p);
kvdec_status kvdec_mla_decode_absorbed(const kvdec_mla_params* p, void* stream);
/* Largest batch one kvdec_mla_decode_absorbed call accepts (a build
 * constant; makes no CUDA call). */
int32_t kvdec_mla_max_batch(void);

/* ------------------------------------------------------------------------ */
/* Cache append with RoPE                                                    */
/* ------------------------------------------------------------------------ */
/*
 * Writes one new token per sequence at slot pos = seqlens[b] (0-based; the
 * caller increments seqlens afterwards) -- the cache only grows by one row
 * per decode step ([KVC-LLM] §2.2; [ARG] §二.2).  RoPE rotates interleaved
 * pairs (2i, 2i+1) by pos * rope_theta^(-2i/dim) ([ARG] §四.4: R_m depends
 * only on the position; the pairing and frequencies are this library's
 * reading).  Rotated values are rounded to bf16 (nearest-even); copied values
 * are bit-exact.
 *
 * mode KVDEC_APPEND_MLA ([ARG] §四.2: c_kv cached as is, k_R cached rotated):
 *   c_kv bf16 [batch, 512], k_rope bf16 [batch, 64] (un-rotated)
 *   -> cache bf16 [num_pages, 64, 576] row (block_table[b, pos/64], pos%64)
 *      = [c_kv ; RoPE_pos(k_rope)]
 * mode KVDEC_APPEND_GQA:
 *   k_new, v_new bf16 [batch, num_kv_heads, head_dim]
 *   -> K[.., pos, :] = RoPE_pos(k_new) (all head_dim values rotated),
 *      V[.., pos, :] = v_new, contiguous (block_table NULL) or paged layout
 *      exactly as in kvdec_gqa_decode.
 *   window = w > 0 (GQA only): the row goes to ring slot pos mod w (the
 *   rotation still uses pos), matching kvdec_gqa_decode's sliding window.
 *   kv_format = KVDEC_KV_FP8_E4M3 (GQA: head_dim 128): K code =
 *   E4M3(RoPE_pos(k_new) / k_scale[kv]) from the binary32 rotation, V code =
 *   E4M3(v_new / v_scale[kv]) from the correctly rounded binary32 quotient;
 *   nearest-even, magnitudes above 448 saturate to 448.
 *   kv_format = KVDEC_KV_FP8_E4M3 (MLA): the cache holds uint8 codes
 *   [num_pages, 64, 576] and k_scale is the fp32 [2] array {c_kv scale,
 *   k_R scale} of kvdec_mla_decode_absorbed; c_kv codes = E4M3(c_kv /
 *   k_scale[0]) from the correctly rounded binary32 quotient, k_R codes =
 *   E4M3(RoPE_pos(k_rope) / k_scale[1]) from the binary32 rotation.
 * pos (or its ring slot) outside [0, capacity) or a bad page entry sets the
 * error bit and the row is skipped.
 */
typedef enum kvdec_append_mode { KVDEC_APPEND_MLA = 0, KVDEC_APPEND_GQA = 1 } kvdec_append_mode;

typedef struct kvdec_append_params {
    int32_t mode;
    int32_t batch;
    const int32_t* seqlens;
    const int32_t* block_table;  /* MLA: required; GQA: NULL = contiguous */
    int32_t num_pages;
    int32_t max_blocks;
    float rope_theta;            /* 0 selects 10000 */
    /* MLA */
    const void* c_kv;
    const void* k_rope;
    void* cache;
    /* GQA */
    const void* k_new;
    const void* v_new;
    void* k;
    void* v;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t capacity;            /* GQA contiguous */
    int32_t reserved;
    uint32_t* error_flag;        /* optional */
    int32_t kv_format;           /* GQA: kvdec_kv_format; 0 = bf16 */
    int32_t window;              /* GQA: 0, or w > 0 for a ring cache of w slots */
    const float* k_scale;        /* FP8: fp32 [num_kv_heads] (MLA: {c_kv, k_R} scales) */
    const float* v_scale;        /* FP8 GQA: fp32 [num_kv_heads] */
} kvdec_append_params;

kvdec_status kvdec_append_rope(const kvdec_append_params* p, void* stream);


/* ------------------------------------------------------------------------ */
/* MLA absorption projections                                                */
/* ------------------------------------------------------------------------ */
/*
 * The two absorbed projections around kvdec_mla_decode_absorbed ([ARG]
 * "attention-variants-and-kv-cache" §四.5; [MLA] "multi-head-latent-
 * attention" §4): for every sequence b and head h,
 *   kvdec_mla_absorb_q:    q_absorbed[b,h,:] = W_UK[h]^T q_nope[b,h,:]   (128 -> 512)
 *   kvdec_mla_project_out: out[b,h,:]        = W_UV[h]   latent[b,h,:]   (512 -> 128)
 * with W_UK, W_UV [num_heads, 128, 512] bf16 (row v or d of head h holds the
 * 512 latent weights).  Together with the decode they give one MLA attention
 * layer in value space; the pages carry no counterpart kernel, only the
 * algebra.
 *
 * Layouts (row-major, bf16 inputs, fp32 accumulation):
 *   absorb:  x = q_nope bf16 [batch, num_heads, 128], y [batch, num_heads, 512]
 *   project: x = latent bf16 [batch, num_heads, 512], y [batch, num_heads, 128]
 *   y is F32 or BF16 (out_dtype).
 * Ownership: the caller owns every buffer; nothing is allocated.
 * Errors: KVDEC_ERR_INVALID_ARG for NULL or misaligned (16 B) pointers, a
 * batch or head count below 1 (batch above 2^20), or another out_dtype; the
 * call is asynchronous on `stream`.
 */
typedef struct kvdec_mla_proj_params {
    const void* x;
    const void* w;
    void* y;
    int32_t batch;
    int32_t num_heads;
    int32_t out_dtype;
    int32_t reserved;
} kvdec_mla_proj_params;

kvdec_status kvdec_mla_absorb_q(const kvdec_mla_proj_params* p, void* stream);
kvdec_status kvdec_mla_project_out(const kvdec_mla_proj_params* p, void* stream);

/* ------------------------------------------------------------------------ */
/* MLA prefill on the non-absorbed path                                      */
/* ------------------------------------------------------------------------ */
/*
 * A prefill (or chunked-prefill) step of MLA attention does not absorb:
 * it up-projects the chunk's latents with one weight GEMM and runs ordinary
 * causal attention with head dims 192 (q.k) and 128 (v) ([ARG]
 * "attention-variants-and-kv-cache" §四.6: absorbing would cost ~3.4x the
 * FLOPs of the s^2 term, which dominates a compute-bound prefill; [MLA]
 * "multi-head-latent-attention" §4.2.1; causal mask [ARG] §五.3).
 *
 * kvdec_mla_prefill_expand: for every token t and head h
 *   k_nope[t, h, :] = W_UK[h] c_kv[t, :],   v[t, h, :] = W_UV[h] c_kv[t, :]
 *   c_kv bf16 [s, 512]; W_UK, W_UV bf16 [num_heads, 128, 512] (as for
 *   kvdec_mla_absorb_q / kvdec_mla_project_out); k_nope, v bf16
 *   [s, num_heads, 128] (fp32 accumulation, one rounding to bf16).  An even
 *   num_heads runs as one tcgen05 GEMM per output, [s, 512] x [512, 128 n_h];
 *   an odd one on the per-head projection kernel.
 *
 * kvdec_mla_prefill: for every query i (position kv_offset + i) and head h
 *   s_j = scale [q_nope ; q_rope][i, h] . [k_nope[j, h] ; k_rope[j]],
 *         j <= kv_offset + i
 *   out[i, h, :] = sum_j softmax(s)_j v[j, h, :],  lse[i, h] = ln sum_j e^{s_j}
 *   q_nope bf16 [s_q, num_heads, 128], q_rope bf16 [s_q, num_heads, 64]
 *   (rotated); k_nope, v bf16 [s_kv, num_heads, 128]; k_rope bf16 [s_kv, 64]
 *   (rotated, shared by every head: the second half of the latent cache
 *   row); out [s_q, num_heads, 128] F32 or BF16; lse fp32 [s_q, num_heads]
 *   or NULL.  kv_offset < 0 selects s_kv - s_q (the chunk is the newest
 *   tokens); 0 <= kv_offset and kv_offset + s_q <= s_kv are required.
 *   scale == 0 selects 1/sqrt(192); otherwise positive and finite.
 * Ownership: the caller owns every buffer; nothing is allocated; both calls
 * are asynchronous on `stream`.  Errors: KVDEC_ERR_INVALID_ARG for NULL or
 * misaligned (16 B) pointers, sizes out of range or another out_dtype.
 */
typedef struct kvdec_mla_expand_params {
    const void* c_kv;
    const void* w_uk;
    const void* w_uv;
    void* k_nope;
    void* v;
    int32_t s;
    int32_t num_heads;
} kvdec_mla_expand_params;

kvdec_status kvdec_mla_prefill_expand(const kvdec_mla_expand_params* p, void* stream);

typedef struct kvdec_mla_prefill_params {
    const void* q_nope;
    const void* q_rope;
    const void* k_nope;
    const void* k_rope;
    const void* v;
    int32_t s_q;
    int32_t s_kv;
    int32_t num_heads;
    int32_t kv_offset;   /* < 0: s_kv - s_q */
    float scale;         /* 0 selects 1/sqrt(192) */
    int32_t out_dtype;
    void* out;
    float* lse;          /* optional */
} kvdec_mla_prefill_params;

kvdec_status kvdec_mla_prefill(const kvdec_mla_prefill_params* p, void* stream);

/* ------------------------------------------------------------------------ */
/* Split combine                                                             */
/* ------------------------------------------------------------------------ */
/*
 * Merges normalised split partials of rows = batch * num_heads rows
 * ([ARG] §五.2, last paragraph: softmax each piece locally, then merge the
 * normalisers).  For row r with n = split_counts[r] (or num_splits):
 *   M = max_s lse_s,  w_s = e^{lse_s - M},
 *   out[r,:] = sum_s w_s O_s[r,:] / sum_s w_s,   lse[r] = M + ln sum_s w_s
 * Partials with lse = -inf (empty pieces) weigh 0; a row whose partials are
 * all empty gets out = 0, lse = -inf; a row with split_counts[r] == 0 is left
 * untouched.
 *
 * Layouts
 *   partial_o   fp32 [num_splits, rows, head_dim]   (O_s = o_s / l_s)
 *   partial_lse fp32 [num_splits, rows]             (natural log)
 *   split_counts int32 [rows] or NULL (all rows use num_splits)
 *   out [rows, head_dim] F32 or BF16; lse fp32 [rows] or NULL
 * Supported: head_dim a multiple of 4 and <= 1024; partial_o and out
 * 16-byte aligned.
 */
typedef struct kvdec_combine_params {
    const float* partial_o;
    const float* partial_lse;
    const int32_t* split_counts;
    int32_t num_splits;
    int32_t rows;
    int32_t head_dim;
    int32_t out_dtype;
    void* out;
    float* lse;
} kvdec_combine_params;

kvdec_status kvdec_combine_splits(const kvdec_combine_params* p, void* stream);

/* ------------------------------------------------------------------------ */
/* helpers                                                                   */
/* ------------------------------------------------------------------------ */
int kvdec_abi_version(void);
/* sizeof() of each params struct, so a binding can check its mirror:
 * kind 0 gqa, 1 mla, 2 append, 3 combine, 4 mla_proj, 5 mla_expand,
 * 6 mla_prefill; -1 for an unknown kind. */
int64_t kvdec_params_size(int kind);
const char* kvdec_status_string(kvdec_status s);
const char* kvdec_last_error(void);
/* Self-test of the bounded device wait: one CTA waits on a barrier that
 * nothing completes, gives up after about timeout_ns nanoseconds, ORs
 * KVDEC_DEVERR_TIMEOUT into *error_flag (device) and returns.  Lets a test
 * check the timeout path without hanging the GPU. */
kvdec_status kvdec_selftest_wait_timeout(uint64_t timeout_ns, uint32_t* error_flag,
                                         void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVDEC_H */
