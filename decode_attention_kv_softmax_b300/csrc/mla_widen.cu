// Widening pass of the MLA decode over an E4M3 latent cache ([ARG]
// "attention-variants-and-kv-cache" §六.3: an FP8 cache halves the bytes per
// cached element; §四.2: the latent row is [c_kv ; k_R]).
//
// The pages a decode call reads are dequantised into a bf16 copy in the
// call's workspace, and the bf16 tcgen05 decode (mla_decode.cu) then runs on
// that copy unchanged: value = E4M3(code) * scale (the c_kv scale for the
// first 512 values of a row, the k_R scale for the last 64), rounded once to
// bf16 (nearest-even).  The copy is laid out in logical order -- tile lt of
// sequence b lands in copy page b * max_blocks + lt -- so its block table is
// the identity, written here as well.  Pages shared between sequences are
// widened once per reference.
//
// One CTA per (sequence, tile) slot; slots past the sequence's page count
// only write their identity entry.  An HBM stream: 576 bytes read and 1152
// written per token, coalesced 16-byte loads and 32-byte stores (the copy's
// pages start on 32-byte boundaries: the workspace is 256-byte aligned and a
// page is 73,728 bytes).
#include "common.cuh"
#include "kernels.h"

namespace kvdec {

namespace {
// 32-byte global store (one instruction for 16 widened values; 32-byte aligned)
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
constexpr int kRow = KVDEC_MLA_DC + KVDEC_MLA_DR;        // 576 values a token
constexpr int kPageVals = KVDEC_PAGE_SIZE * kRow;         // 36864
constexpr int kChunks = kPageVals / 16;                   // 16 codes per chunk
constexpr int kThreads = 256;
static_assert(kRow % 16 == 0 && KVDEC_MLA_DC % 16 == 0, "a chunk never straddles a row or the c_kv / k_R split");
static_assert(kChunks % kThreads == 0, "whole chunks per thread");
}  // namespace

__global__ void __launch_bounds__(kThreads) mla_widen_kernel(const MlaWidenArgs a) {
    const int lt = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
    const size_t slot = (size_t)b * a.max_blocks + lt;
    if (t == 0) a.copy_table[slot] = (int32_t)slot;
    const int len = min(max(__ldg(a.seqlens + b), 0), a.max_blocks * KVDEC_PAGE_SIZE);
    if (lt * KVDEC_PAGE_SIZE >= len) return;
    const int page = __ldg(a.block_table + slot);
    uint4* dst = reinterpret_cast<uint4*>(a.copy + slot * kPageVals);
    if (page < 0 || page >= a.num_pages) {
        if (t == 0) report(a.err, KVDEC_DEVERR_BAD_PAGE);
        for (int i = t; i < 2 * kChunks; i += kThreads) dst[i] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(a.codes + (size_t)page * kPageVals);
    const float sc = __ldg(a.kv_scale), sr = __ldg(a.kv_scale + 1);
    uint4 x[kChunks / kThreads];
#pragma unroll
    for (int k = 0; k < kChunks / kThreads; ++k) x[k] = __ldg(src + t + kThreads * k);
#pragma unroll
    for (int k = 0; k < kChunks / kThreads; ++k) {
        const int c = t + kThreads * k;                 // chunk: 16 values of row c / 36
        const float s = (c % (kRow / 16)) < KVDEC_MLA_DC / 16 ? sc : sr;
        const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t lo, hi;
            e4m3x4_to_f16x2x2(w[q], lo, hi);   // exact
            const float2 f0 = unpack_half2(lo), f1 = unpack_half2(hi);
            o[2 * q] = pack_bf16x2(f0.x * s, f0.y * s);
            o[2 * q + 1] = pack_bf16x2(f1.x * s, f1.y * s);
        }
        st_global_v8(dst + 2 * c, o);
    }
}

cudaError_t launch_mla_widen(const MlaWidenArgs& a, cudaStream_t st) {
    mla_widen_kernel<<<dim3(a.max_blocks, a.B), kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvdec
