// Argument blocks and launchers shared between the host API (api.cu) and
// the kernel translation units.
#pragma once

#include "common.cuh"
#include "launch_cache.h"

namespace kvdec {

struct GqaArgs {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* seqlens;
    void* out;
    float* lse;
    float* part_o;       // [2*grid, rows, D]
    float* part_lse;     // [2*grid, rows]
    unsigned long long* counters;  // [units], see arrive_piece
    uint32_t epoch;
    uint32_t* err;
    int B, H, n_kv, g, n_hc, hc_rows;
    int cap;             // tokens addressable per sequence
    int paged, num_pages, max_blocks;
    int out_bf16;
    float scale_log2;
    int min_tiles;
    uint64_t timeout_ns;
    // E4M3 cache: per-KV-head fp32 scales (dequantised value = code * scale)
    const float* k_scale;
    const float* v_scale;
    int window;          // > 0: ring cache of the last `window` tokens
};

struct CombineArgs {
    const float* po;
    const float* plse;
    const int32_t* counts;
    void* out;
    float* lse;
    int S, rows, D;
    int out_bf16;
};

constexpr int kMaxRopePairs = 64;

struct AppendArgs {
    int mode;  // 0 MLA, 1 GQA
    int B;
    const int32_t* seqlens;
    const int32_t* block_table;
    int num_pages, max_blocks;
    double inv_freq[kMaxRopePairs];   // theta^(-2i/dim), computed on the host in binary64
    const __nv_bfloat16* c_kv;
    const __nv_bfloat16* k_rope;
    __nv_bfloat16* cache;
    const __nv_bfloat16* k_new;
    const __nv_bfloat16* v_new;
    void* k;             // bf16, or E4M3 bytes when fp8
    void* v;
    int n_kv, d, cap;
    uint32_t* err;
    int fp8;             // E4M3 cache (GQA: per-KV-head scales; MLA: k_scale = [c_kv, k_R])
    int window;          // GQA: > 0 ring cache of `window` slots
    const float* k_scale;
    const float* v_scale;
};

struct MlaMaps {
    CUtensorMap c128;  // cache [pages*64, 576], box 64 x 64, 128-byte swizzle
    CUtensorMap c64;   // cache [pages*64, 576], box 32 x 64, 64-byte swizzle
    CUtensorMap part;  // partial O [2*pairs*128, 512] fp32, box 32 x 32, 128-byte swizzle (stores)
    CUtensorMap outf;  // out [B*128, 512] fp32, same box (stores; unused for bf16 out)
};

struct MlaArgs {
    const __nv_bfloat16* q_abs;     // [B, 128, 512]
    const __nv_bfloat16* q_rope;    // [B, 128, 64]
    const int32_t* block_table;
    const int32_t* seqlens;
    void* out;
    float* lse;
    float* part_o;                  // [2*pairs, 128, 512]
    float* part_lse;                // [2 CTAs][2*pairs, 128]
    unsigned long long* counters;   // [B][2 CTAs][4 head quadrants]
    uint32_t epoch;
    uint32_t* err;
    int B, num_pages, max_blocks;
    int out_bf16;
    float scale_log2;
    int min_tiles;
    int seg_cost;                   // start cost of a sequence, in pages (schedule.cuh)
    uint64_t timeout_ns;
};

// Widening of the pages an MLA decode reads from an E4M3 latent cache into a
// bf16 copy laid out in logical order (mla_widen.cu): tile lt of sequence b
// (lt < its page count) goes to copy page b * max_blocks + lt, and the copy's
// block table is the identity on [B, max_blocks].
struct MlaWidenArgs {
    const uint8_t* codes;       // [num_pages, 64, 576] E4M3
    const int32_t* block_table; // [B, max_blocks]
    const int32_t* seqlens;     // [B]
    const float* kv_scale;      // [c_kv scale, k_R scale]
    __nv_bfloat16* copy;        // [B * max_blocks, 64, 576]
    int32_t* copy_table;        // [B, max_blocks], identity
    int B, num_pages, max_blocks;
    uint32_t* err;
};
cudaError_t launch_mla_widen(const MlaWidenArgs& a, cudaStream_t st);

// Start cost of a sequence in the MLA decode schedule, in pages: loading a
// new Q into TMEM and flushing O takes about as long as this many pages.
constexpr int kMlaSeqStartCost = 4;

struct MlaProjArgs {
    const __nv_bfloat16* x;   // absorb: q_nope [B, H, 128]; project: latent [B, H, 512]
    const __nv_bfloat16* w;   // [H, 128, 512]
    void* y;                  // absorb: [B, H, 512]; project: [B, H, 128]
    int batch, num_heads, out_bf16;
    int x_shared;             // x is one [B, K] matrix for every head (prefill up-projection)
};

cudaError_t launch_mla(const MlaMaps& maps, const MlaArgs& a, int pairs, cudaStream_t st);
cudaError_t launch_mla_proj(bool absorb, const MlaProjArgs& a, cudaStream_t st);

// Causal MLA prefill attention on the non-absorbed path (mla_prefill_tc.cu)
struct MlaPrefillArgs {
    const __nv_bfloat16* q_nope;   // [s_q, H, 128]
    const __nv_bfloat16* q_rope;   // [s_q, H, 64]
    const __nv_bfloat16* k_nope;   // [s_kv, H, 128]
    const __nv_bfloat16* k_rope;   // [s_kv, 64]
    const __nv_bfloat16* v;        // [s_kv, H, 128]
    void* out;                     // [s_q, H, 128]
    float* lse;                    // [s_q, H] or null
    int s_q, s_kv, num_heads, kv_offset, out_bf16;
    float scale_log2;
    uint32_t* err;
    uint64_t timeout_ns;
};
// Tensor maps of the tcgen05 prefill: q_nope, q_rope, k_nope, v as 3-D
// [tokens][heads][dims] (box 64 dims x 1 head x 128 or 64 tokens, 128-byte
// swizzle), k_rope 2-D [tokens][64] (box 64 x 64).
struct MlaPrefillMaps {
    CUtensorMap qn, qr, kn, kr, v;
};
cudaError_t launch_mla_prefill_tc(const MlaPrefillMaps& maps, const MlaPrefillArgs& a, cudaStream_t st);

// Up-projection of a prefill chunk on tcgen05 (mla_expand_tc.cu): maps over
// c_kv [s, 512] (box 64 x 128) and W_UK, W_UV viewed as [n_h 128, 512]
// (box 64 x 256), 128-byte swizzle.
struct MlaExpandMaps {
    CUtensorMap c, wk, wv;
};
struct MlaExpandArgs {
    __nv_bfloat16* k_nope;   // [s, n_h 128]
    __nv_bfloat16* v;
    int s, N;                // N = n_h 128 (a multiple of 256)
    uint32_t* err;
    uint64_t timeout_ns;
};
cudaError_t launch_mla_expand_tc(const MlaExpandMaps& maps, const MlaExpandArgs& a, cudaStream_t st);
int max_pairs_mla(int B);
int max_batch_mla();   // largest batch whose tile table fits in shared memory

// MT: head-row tiles of 16 (1 or 2), or 0 for the transposed FP8 form (at
// most 8 head rows); dense selects that form's three-CTAs-per-SM build.
cudaError_t launch_gqa(int D, int MT, bool F8, bool dense, const CUtensorMap& tk, const CUtensorMap& tv,
                       const GqaArgs& a, int grid, cudaStream_t st);
int occupancy_gqa(int D, int MT, bool F8, bool dense, int B);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st);
cudaError_t launch_append(const AppendArgs& a, cudaStream_t st);
cudaError_t launch_selftest_wait(uint64_t timeout_ns, uint32_t* err, cudaStream_t st);
void set_last_error(const char* msg);

}  // namespace kvdec
