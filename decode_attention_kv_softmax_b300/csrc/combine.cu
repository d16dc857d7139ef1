// Log-sum-exp merge of split partial outputs ([ARG]
// "attention-variants-and-kv-cache" §五.2: the sequence is split, softmax is
// taken per piece, and the pieces are merged through their normalisers).
//
// One warp per output row; each lane owns head_dim/32 (rounded up to float4
// groups) columns.  The row's partial lse values are read once per split
// with a warp-wide max, then the weighted sum streams the partials with
// 16-byte loads.
#include "common.cuh"
#include "kernels.h"

namespace kvdec {


__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= a.rows) return;
    const int r = warp;
    int n = a.counts ? __ldg(a.counts + r) : a.S;
    if (n <= 0) return;               // row left untouched
    if (n > a.S) n = a.S;
    float M = -INFINITY;
    for (int s = lane; s < n; s += 32) M = fmaxf(M, __ldg(a.plse + (size_t)s * a.rows + r));
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const int n4 = a.D >> 2;
    float den = 0.f;
    if (M == -INFINITY) {
        // every piece empty: out = 0, lse = -inf
        for (int c = lane; c < n4; c += 32) {
            const size_t off = (size_t)r * a.D + c * 4;
            if (a.out_bf16) *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off) = make_uint2(0u, 0u);
            else *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (lane == 0 && a.lse) a.lse[r] = -INFINITY;
        return;
    }
    for (int c0 = 0; c0 < n4; c0 += 32) {
        const int c = c0 + lane;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float dsum = 0.f;
        for (int s = 0; s < n; ++s) {
            const float ls = __ldg(a.plse + (size_t)s * a.rows + r);
            const float wgt = (ls == -INFINITY) ? 0.f : fast_exp2((ls - M) * kLog2e);
            dsum += wgt;
            if (c < n4 && wgt != 0.f) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(a.po + ((size_t)s * a.rows + r) * a.D) + c);
                acc.x = fmaf(wgt, v.x, acc.x);
                acc.y = fmaf(wgt, v.y, acc.y);
                acc.z = fmaf(wgt, v.z, acc.z);
                acc.w = fmaf(wgt, v.w, acc.w);
            }
        }
        den = dsum;
        if (c < n4) {
            const float inv = 1.f / dsum;
            acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
            const size_t off = (size_t)r * a.D + c * 4;
            if (a.out_bf16) {
                *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off) =
                    make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
            } else {
                *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off) = acc;
            }
        }
    }
    if (lane == 0 && a.lse) a.lse[r] = M + __logf(den);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
    const int warps_per_block = 8;
    const int grid = (a.rows + warps_per_block - 1) / warps_per_block;
    combine_kernel<<<grid, 32 * warps_per_block, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvdec
