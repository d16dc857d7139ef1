// Causal MLA attention of a prefill chunk on the non-absorbed path
// ([ARG] "attention-variants-and-kv-cache" §四.6: prefill reads c_kv,
// up-projects K and V with one weight GEMM and runs ordinary causal
// attention with head dims 192 (q.k) and 128 (v), because absorption would
// cost ~3.4x the FLOPs of the s^2 term; [MLA] "multi-head-latent-attention"
// §4.2.1: prefill computes k and v explicitly; [ARG] §五.3: causal mask).
//
// For head h and query i (position kv_offset + i):
//   s_j = scale [q_nope ; q_rope]_i . [k_nope_{j,h} ; k_rope_j],  j <= kv_offset + i
//   out[i, h] = sum_j softmax(s)_j v_{j,h},  lse[i, h] = ln sum_j e^{s_j}
// k_rope is one rotated 64-vector per token shared by all heads.
//
// CTA = 4 warps, one head and 64 query rows (16 per warp); the KV of the
// head streams through a two-stage cp.async ring in 64-token tiles, K as
// three 128-byte-swizzled boxes of 64 dims (k_nope dims 0-63, 64-127,
// k_rope) and V as two.  Each warp runs FlashAttention's online softmax on
// warp-level m16n8k16 bf16 MMAs (fp32 accumulation): S = Q K^T from
// ldmatrix fragments of K, O += P V with P taken from the S accumulators and
// V through ldmatrix.trans.  Tiles wholly above the diagonal are never
// loaded; the diagonal and the sequence tail are masked.  The query blocks
// with the most tiles are launched first.
#include "common.cuh"
#include "kernels.h"

namespace kvdec {

namespace pf {
constexpr int kQ = 64;                    // query rows per CTA
constexpr int kT = 64;                    // keys per tile
constexpr int kDn = 128, kDr = 64, kDv = 128;
constexpr int kBox = 64 * 128;            // 64 rows x 128 B
constexpr int kKBytes = 3 * kBox;         // k_nope (2 boxes) + k_rope (1 box)
constexpr int kVBytes = 2 * kBox;
constexpr int kStage = kKBytes + kVBytes; // 40 KB
constexpr int kSmem = 2 * kStage + 1024;
}  // namespace pf

KVDEC_DEVINL void pf_cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__global__ void __launch_bounds__(128, 2) mla_prefill_kernel(const MlaPrefillArgs a) {
    using namespace pf;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane >> 2, qc = lane & 3;
    const int qb = gridDim.x - 1 - blockIdx.x;   // heaviest query blocks first
    const int hh = blockIdx.y;
    const int H = a.num_heads;
    const int i0 = qb * kQ;
    // keys any row of this CTA may see: positions < kv_offset + last row + 1
    const int kend = min(a.s_kv, a.kv_offset + min(i0 + kQ, a.s_q));
    const int ntiles = (kend + kT - 1) / kT;

    // Q fragments of the warp's 16 rows over the 192 dims (12 k-steps)
    uint32_t qa[12][4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = i0 + 16 * warp + quad + 8 * half;
        const bool ok = r < a.s_q;
        const int rr = ok ? r : 0;
        const uint32_t* qn = reinterpret_cast<const uint32_t*>(a.q_nope + ((size_t)rr * H + hh) * kDn);
        const uint32_t* qr = reinterpret_cast<const uint32_t*>(a.q_rope + ((size_t)rr * H + hh) * kDr);
#pragma unroll
        for (int ks = 0; ks < 12; ++ks) {
            const uint32_t* src = ks < 8 ? qn + 8 * ks : qr + 8 * (ks - 8);
            qa[ks][half] = ok ? __ldg(src + qc) : 0u;
            qa[ks][half + 2] = ok ? __ldg(src + 4 + qc) : 0u;
        }
    }

    // tile t of the head's keys -> stage s (rows past s_kv are zero-filled)
    auto load_tile = [&](int t, int s) {
        const uint32_t kb = smem_addr(smem + s * kStage), vb = kb + kKBytes;
        for (int i = tid; i < kT * 24; i += 128) {
            const int r = i / 24, c = i % 24;   // 16-byte chunk c of the 384-byte key row
            const int tok = t * kT + r;
            const bool ok = tok < a.s_kv;
            const size_t tk = (size_t)(ok ? tok : 0);
            const __nv_bfloat16* src = (c < 16) ? a.k_nope + (tk * H + hh) * kDn + c * 8
                                                : a.k_rope + tk * kDr + (c - 16) * 8;
            pf_cp_async16(kb + (c >> 3) * kBox + swz128(r, c & 7), src, ok);
        }
        for (int i = tid; i < kT * 16; i += 128) {
            const int r = i / 16, c = i % 16;
            const int tok = t * kT + r;
            const bool ok = tok < a.s_kv;
            const __nv_bfloat16* src = a.v + ((size_t)(ok ? tok : 0) * H + hh) * kDv + c * 8;
            pf_cp_async16(vb + (c >> 3) * kBox + swz128(r, c & 7), src, ok);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    float o[kDv / 8][4];
#pragma unroll
    for (int nd = 0; nd < kDv / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    const float sl2 = a.scale_log2;
    const int qpos0 = a.kv_offset + i0 + 16 * warp;   // position of the warp's first row

    if (ntiles > 0) load_tile(0, 0);
    for (int t = 0; t < ntiles; ++t) {
        if (t + 1 < ntiles) load_tile(t + 1, (t + 1) & 1);
        else asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncthreads();
        const uint32_t kb = smem_addr(smem + (t & 1) * kStage), vb = kb + kKBytes;

        // ---- S = Q K^T: the warp's 16 rows x 64 keys
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            const uint32_t tok = nt * 8 + (lane & 7);
#pragma unroll
            for (int kk = 0; kk < 6; ++kk) {
                const uint32_t chunk = 4 * kk + (lane >> 3);
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kb + (chunk >> 3) * kBox + swz128(tok, chunk & 7), r0, r1, r2, r3);
                mma_bf16_16816(s[nt], qa[2 * kk], r0, r1);
                mma_bf16_16816(s[nt], qa[2 * kk + 1], r2, r3);
            }
        }
        // ---- causal mask (key position > query position) and the tail
        const int kp0 = t * kT;
        if (kp0 + kT - 1 > qpos0 || kp0 + kT > a.s_kv) {
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kp = kp0 + nt * 8 + 2 * qc + (e & 1);
                    const int qp = qpos0 + quad + 8 * (e >> 1);
                    if (kp > qp || kp >= a.s_kv) s[nt][e] = -INFINITY;
                }
        }
        // ---- online softmax (base 2, scaled), P fragments in bf16
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m[0], mx0 * sl2), mn1 = fmaxf(m[1], mx1 * sl2);
        const float b0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float b1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float al0 = fast_exp2(m[0] - b0), al1 = fast_exp2(m[1] - b1);
        m[0] = mn0;
        m[1] = mn1;
        float ps0 = 0.f, ps1 = 0.f;
        uint32_t pa[4][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const float p0 = fast_exp2(fmaf(s[nt][0], sl2, -b0));
            const float p1 = fast_exp2(fmaf(s[nt][1], sl2, -b0));
            const float p2 = fast_exp2(fmaf(s[nt][2], sl2, -b1));
            const float p3 = fast_exp2(fmaf(s[nt][3], sl2, -b1));
            ps0 += p0 + p1;
            ps1 += p2 + p3;
            pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p0, p1);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p2, p3);
        }
        l[0] = fmaf(l[0], al0, ps0);
        l[1] = fmaf(l[1], al1, ps1);
#pragma unroll
        for (int nd = 0; nd < kDv / 8; ++nd) {
            o[nd][0] *= al0;
            o[nd][1] *= al0;
            o[nd][2] *= al1;
            o[nd][3] *= al1;
        }
        // ---- O += P V, 16 keys at a time
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int nd2 = 0; nd2 < kDv / 16; ++nd2) {
                const int mat = lane >> 3;
                const uint32_t tok = 16 * ks + (mat & 1) * 8 + (lane & 7);
                const uint32_t chunk = 2 * nd2 + (mat >> 1);
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(vb + (chunk >> 3) * kBox + swz128(tok, chunk & 7), r0, r1, r2, r3);
                mma_bf16_16816(o[2 * nd2], pa[ks], r0, r1);
                mma_bf16_16816(o[2 * nd2 + 1], pa[ks], r2, r3);
            }
        }
        __syncthreads();   // the stage is refilled by the next iteration's load
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");

    // ---- normalise and store: thread holds rows quad (+8), columns 8 nd + 2 qc (+1)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float lr = l[half];
        lr += __shfl_xor_sync(0xffffffffu, lr, 1);
        lr += __shfl_xor_sync(0xffffffffu, lr, 2);
        const int r = i0 + 16 * warp + quad + 8 * half;
        if (r >= a.s_q) continue;
        const float inv = lr > 0.f ? 1.f / lr : 0.f;
        const size_t base = ((size_t)r * H + hh) * kDv;
#pragma unroll
        for (int nd = 0; nd < kDv / 8; ++nd) {
            const float v0 = o[nd][2 * half] * inv, v1 = o[nd][2 * half + 1] * inv;
            const size_t off = base + nd * 8 + 2 * qc;
            if (a.out_bf16)
                *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off) = pack_bf16x2(v0, v1);
            else
                *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + off) = make_float2(v0, v1);
        }
        if (a.lse && qc == 0)
            a.lse[(size_t)r * H + hh] = lr > 0.f ? (m[half] + __log2f(lr)) * kLn2 : -INFINITY;
    }
}

cudaError_t launch_mla_prefill(const MlaPrefillArgs& a, cudaStream_t st) {
    const dim3 grid((a.s_q + pf::kQ - 1) / pf::kQ, a.num_heads);
    cudaError_t e = cudaFuncSetAttribute(mla_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pf::kSmem);
    if (e != cudaSuccess) return e;
    mla_prefill_kernel<<<grid, 128, pf::kSmem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvdec
