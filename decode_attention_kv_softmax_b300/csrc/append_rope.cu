// Cache append with RoPE: one new token per sequence ([KVC-LLM] "KV Cache
// 如何影响了 LLM Inference" §2.2: each step appends the new k, v row;
// [ARG] "attention-variants-and-kv-cache" §四.2: the MLA cache row is
// [c_kv ; k_R] with k_R stored already rotated, §四.4: R_m depends only on the
// position m).
//
// RoPE reading: interleaved pairs (2i, 2i+1) rotated by
// pos * theta^(-2i/dim).  The angle reaches 1.3e5 rad at 128K context, where
// a binary32 angle is off by ~1e-2 rad; the angle and its reduction modulo
// 2 pi are therefore taken in binary64 (the frequencies come from the host
// in binary64), the sine/cosine of the reduced angle and the rotation in
// binary32, and the result is rounded once to bf16 (nearest-even).  The kernel moves a few KB per call: it is launch-latency
// bound, so it is written for simplicity, one CTA per (sequence, head).
//
// Options: an FP8 cache ([ARG] §六.3) stores E4M3(x / scale) (nearest-even,
// saturating at 448; the quotient is the correctly rounded binary32 one),
// with one scale per KV head (GQA) or one for c_kv and one for k_R (MLA);
// and (GQA) a sliding window of w tokens ([ARG] §五.3) writes the
// ring slot pos mod w while the rotation keeps the position pos.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace kvdec {


// Rotated pair i of x at position pos, in binary32.
KVDEC_DEVINL float2 rope_pair_f32(const __nv_bfloat16* x, int i, int pos, const double* inv_freq) {
    // angle in binary64, reduced to [-pi, pi] in binary64, then sine/cosine
    // and the rotation in binary32 (|error| ~1e-7, far below one bf16 ulp)
    const double ang = (double)pos * inv_freq[i];
    const double r = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
    float s, c;
    sincosf((float)r, &s, &c);
    const float x0 = __bfloat162float(x[2 * i]);
    const float x1 = __bfloat162float(x[2 * i + 1]);
    return make_float2(fmaf(x0, c, -x1 * s), fmaf(x0, s, x1 * c));
}

KVDEC_DEVINL void rope_pair(const __nv_bfloat16* x, __nv_bfloat16* y, int i, int pos,
                            const double* inv_freq) {
    const float2 r = rope_pair_f32(x, i, pos, inv_freq);
    y[2 * i] = __float2bfloat16_rn(r.x);
    y[2 * i + 1] = __float2bfloat16_rn(r.y);
}

KVDEC_DEVINL uint8_t to_e4m3(float x) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

__global__ void __launch_bounds__(64) append_rope_kernel(const AppendArgs a) {
    const int b = blockIdx.x, head = blockIdx.y, t = threadIdx.x;
    const int pos_abs = __ldg(a.seqlens + b);
    // ring slot of a sliding-window cache; the rotation uses pos_abs
    const int pos = (a.window > 0 && pos_abs >= 0) ? pos_abs % a.window : pos_abs;
    const int cap = a.block_table ? a.max_blocks * KVDEC_PAGE_SIZE : a.cap;
    if (pos < 0 || pos >= cap) {
        if (t == 0 && head == 0) report(a.err, KVDEC_DEVERR_SEQLEN);
        return;
    }
    int page = 0;
    if (a.block_table) {
        page = __ldg(a.block_table + (size_t)b * a.max_blocks + pos / KVDEC_PAGE_SIZE);
        if (page < 0 || page >= a.num_pages) {
            if (t == 0 && head == 0) report(a.err, KVDEC_DEVERR_BAD_PAGE);
            return;
        }
    }
    const int slot = pos % KVDEC_PAGE_SIZE;
    if (a.mode == 0 && a.fp8) {
        // E4M3 latent row: [E4M3(c_kv / s_c) ; E4M3(RoPE(k_rope) / s_R)], s = k_scale[0..1]
        uint8_t* row = reinterpret_cast<uint8_t*>(a.cache) +
                       ((size_t)page * KVDEC_PAGE_SIZE + slot) * (KVDEC_MLA_DC + KVDEC_MLA_DR);
        const float sc = __ldg(a.k_scale), sr = __ldg(a.k_scale + 1);
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(a.c_kv + (size_t)b * KVDEC_MLA_DC) + t);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t c[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {   // 8 values of 64 threads = 512
            const uint32_t bits = (i & 1) ? (w[i >> 1] & 0xffff0000u) : (w[i >> 1] << 16);
            c[i >> 2] |= (uint32_t)to_e4m3(__fdiv_rn(__uint_as_float(bits), sc)) << (8 * (i & 3));
        }
        *reinterpret_cast<uint2*>(row + 8 * t) = make_uint2(c[0], c[1]);
        if (t < KVDEC_MLA_DR / 2) {
            const float2 r = rope_pair_f32(a.k_rope + (size_t)b * KVDEC_MLA_DR, t, pos, a.inv_freq);
            row[KVDEC_MLA_DC + 2 * t] = to_e4m3(__fdiv_rn(r.x, sr));
            row[KVDEC_MLA_DC + 2 * t + 1] = to_e4m3(__fdiv_rn(r.y, sr));
        }
        return;
    }
    if (a.mode == 0) {
        // MLA latent row: [c_kv (512, copied) ; RoPE(k_rope) (64)]
        __nv_bfloat16* row = a.cache + ((size_t)page * KVDEC_PAGE_SIZE + slot) * (KVDEC_MLA_DC + KVDEC_MLA_DR);
        const uint4* src = reinterpret_cast<const uint4*>(a.c_kv + (size_t)b * KVDEC_MLA_DC);
        reinterpret_cast<uint4*>(row)[t] = __ldg(src + t);     // 64 threads x 16 B = 512 bf16
        if (t < KVDEC_MLA_DR / 2)
            rope_pair(a.k_rope + (size_t)b * KVDEC_MLA_DR, row + KVDEC_MLA_DC, t, pos, a.inv_freq);
        return;
    }
    // GQA: K row rotated over the whole head dim, V row copied
    const size_t src_off = ((size_t)b * a.n_kv + head) * a.d;
    size_t dst_off;
    if (a.block_table) dst_off = (((size_t)page * a.n_kv + head) * KVDEC_PAGE_SIZE + slot) * a.d;
    else dst_off = (((size_t)b * a.n_kv + head) * a.cap + pos) * a.d;
    if (a.fp8) {
        uint8_t* k8 = static_cast<uint8_t*>(a.k) + dst_off;
        uint8_t* v8 = static_cast<uint8_t*>(a.v) + dst_off;
        const float ks = __ldg(a.k_scale + head), vs = __ldg(a.v_scale + head);
        if (t < a.d / 2) {
            const float2 r = rope_pair_f32(a.k_new + src_off, t, pos_abs, a.inv_freq);
            k8[2 * t] = to_e4m3(__fdiv_rn(r.x, ks));
            k8[2 * t + 1] = to_e4m3(__fdiv_rn(r.y, ks));
        }
        for (int i = t; i < a.d; i += blockDim.x)
            v8[i] = to_e4m3(__fdiv_rn(__bfloat162float(a.v_new[src_off + i]), vs));
        return;
    }
    __nv_bfloat16* k16 = static_cast<__nv_bfloat16*>(a.k);
    __nv_bfloat16* v16 = static_cast<__nv_bfloat16*>(a.v);
    if (t < a.d / 2) rope_pair(a.k_new + src_off, k16 + dst_off, t, pos_abs, a.inv_freq);
    if (t < a.d / 8)
        reinterpret_cast<uint4*>(v16 + dst_off)[t] = __ldg(reinterpret_cast<const uint4*>(a.v_new + src_off) + t);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st) {
    dim3 grid(a.B, a.mode == 0 ? 1 : a.n_kv);
    append_rope_kernel<<<grid, 64, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvdec
