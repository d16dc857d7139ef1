// Causal MLA prefill attention on the non-absorbed path with fifth-generation
// tensor cores ([ARG] "attention-variants-and-kv-cache" §四.6: prefill
// up-projects K and V and runs ordinary causal attention with head dims 192
// and 128; [ARG] §五.2: FlashAttention's tiled online softmax; §五.3: causal
// mask).
//
// CTA = one head and 128 query rows, 6 warps:
//   warp 0  TMA producer: Q once (3 boxes of 128 rows x 64 dims), then
//           64-key K tiles (k_nope 0-63, 64-127, k_rope) and V tiles
//           (2 boxes of 64 dims) through NS stages;
//   warp 1  owns TMEM (256 columns) and issues the MMAs from one thread:
//           S(j) = Q K_j^T into TMEM buffer j mod 2 (12 MMAs of
//           M=128, N=64, K=16), then O += P(j-1) V_(j-1) (4 MMAs of N=128,
//           P from shared memory, V MN-major);
//   warps 2-5  softmax, one thread per query row (TMEM lane): load S(j),
//           mask the diagonal and the tail, row max, exponentials into bf16
//           P (128-byte-swizzled rows in shared memory), row sums; O is
//           rescaled in TMEM only when a row's max passes its reference
//           max by more than 2^8 (then after PV(j-1) has completed).
// S(j+1) runs on the tensor cores while the softmax works on S(j).  All
// waits are bounded; a timeout sets the error word and unwinds.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace kvdec {

namespace pft {
constexpr int kBM = 128, kBN = 64;
constexpr int kNS = 3;
constexpr int kQBytes = 3 * 128 * 128;     // 3 boxes [128 rows x 128 B]
constexpr int kKBox = 64 * 128;            // [64 keys x 128 B]
constexpr int kStage = 5 * kKBox;          // K: 3 boxes, V: 2 boxes = 40 KB
constexpr int kPBytes = 128 * 128;         // [128 rows x 64 keys] bf16
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQBytes;
constexpr int kOffP = kOffKV + kNS * kStage;
constexpr int kOffBars = kOffP + kPBytes;
enum { B_Q, B_SFULL, B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PFREE, B_ODONE, B_DONE, B_KV };
constexpr int kBars = B_KV + 2 * kNS;
constexpr int kOffMisc = kOffBars + kBars * 8;           // [0] TMEM base, [1] abort word
constexpr int kSmem = kOffMisc + 16 + 1024;
constexpr uint32_t kTmemCols = 256;                      // S buffers [0,128), O [128,256)
constexpr uint32_t kTmemO = 128;
}  // namespace pft

__global__ void __launch_bounds__(192, 1)
    mla_prefill_tc_kernel(const __grid_constant__ MlaPrefillMaps maps, const MlaPrefillArgs a) {
    using namespace pft;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qb = gridDim.x - 1 - blockIdx.x;   // heaviest query blocks first
    const int hh = blockIdx.y;
    const int q0 = qb * kBM;
    const int kend = min(a.s_kv, a.kv_offset + min(q0 + kBM, a.s_q));
    const int nt = (kend + kBN - 1) / kBN;      // >= 1: kv_offset >= 0

    const uint32_t bar0 = smem_addr(smem + kOffBars);
    auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };
    auto kv_full = [bar0](int s) { return bar0 + 8u * (uint32_t)(B_KV + s); };
    auto kv_empty = [bar0](int s) { return bar0 + 8u * (uint32_t)(B_KV + kNS + s); };
    volatile int* misc = reinterpret_cast<volatile int*>(smem + kOffMisc);
    volatile int* abort_word = misc + 1;
    const uint32_t sQ = smem_addr(smem + kOffQ), sKV = smem_addr(smem + kOffKV), sP = smem_addr(smem + kOffP);

    if (tid == 0) {
        mbar_init(bar(B_Q), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_SFULL + i), 1);
            mbar_init(bar(B_SFREE + i), 4);
        }
        mbar_init(bar(B_PFULL), 4);
        mbar_init(bar(B_PFREE), 1);
        mbar_init(bar(B_ODONE), 1);
        mbar_init(bar(B_DONE), 1);
        for (int s = 0; s < kNS; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(smem + kOffMisc), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = (uint32_t)misc[0];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&maps.qn);
            prefetch_tensormap(&maps.qr);
            prefetch_tensormap(&maps.kn);
            prefetch_tensormap(&maps.kr);
            prefetch_tensormap(&maps.v);
            const uint64_t keep = l2_policy_evict_last();   // K/V are read by every query block
            mbar_arrive_expect_tx(bar(B_Q), kQBytes);
            tma_load_3d(sQ, &maps.qn, bar(B_Q), 0, hh, q0);
            tma_load_3d(sQ + 16384, &maps.qn, bar(B_Q), 64, hh, q0);
            tma_load_3d(sQ + 32768, &maps.qr, bar(B_Q), 0, hh, q0);
            int issued = 0;
            for (int j = 0; j < nt; ++j) {
                const int s = j % kNS;
                if (!wait_or_abort(kv_empty(s), (uint32_t)(((j / kNS) & 1) ^ 1), abort_word, a.err, a.timeout_ns))
                    break;
                const uint32_t fb = kv_full(s), dst = sKV + s * kStage;
                mbar_arrive_expect_tx(fb, kStage);
                const int k0 = j * kBN;
                tma_load_3d_hint(dst, &maps.kn, fb, 0, hh, k0, keep);
                tma_load_3d_hint(dst + kKBox, &maps.kn, fb, 64, hh, k0, keep);
                tma_load_2d(dst + 2 * kKBox, &maps.kr, fb, 0, k0, keep);
                tma_load_3d_hint(dst + 3 * kKBox, &maps.v, fb, 0, hh, k0, keep);
                tma_load_3d_hint(dst + 4 * kKBox, &maps.v, fb, 64, hh, k0, keep);
                ++issued;
            }
            // never leave TMA writes in flight
            if (!mbar_wait_bounded(bar(B_Q), 0, a.timeout_ns)) report(a.err, KVDEC_DEVERR_TIMEOUT);
            for (int i = (issued > kNS ? issued - kNS : 0); i < issued; ++i)
                if (!mbar_wait_bounded(kv_full(i % kNS), (uint32_t)((i / kNS) & 1), a.timeout_ns)) {
                    report(a.err, KVDEC_DEVERR_TIMEOUT);
                    break;
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t iS = umma_idesc_bf16(128, 64, false, false);
            constexpr uint32_t iP = umma_idesc_bf16(128, 128, false, true);
            auto pv = [&](int j) -> bool {
                if (!wait_or_abort(bar(B_PFULL), (uint32_t)(j & 1), abort_word, a.err, a.timeout_ns)) return false;
                tc_fence_after();
                const uint32_t vb = sKV + (j % kNS) * kStage + 3 * kKBox;
                for (int ks = 0; ks < 4; ++ks)
                    umma_bf16_ss(tmem + kTmemO, umma_desc(sP + ks * 32, 16, 1024, kSwizzle128B),
                                 umma_desc(vb + ks * 2048, 8192, 1024, kSwizzle128B), iP,
                                 (j > 0 || ks > 0) ? 1u : 0u);
                umma_commit(bar(B_PFREE));
                umma_commit(kv_empty(j % kNS));
                return true;
            };
            bool ok = wait_or_abort(bar(B_Q), 0, abort_word, a.err, a.timeout_ns);
            for (int j = 0; ok && j < nt; ++j) {
                const int s = j % kNS, sb = j & 1;
                if (!wait_or_abort(kv_full(s), (uint32_t)((j / kNS) & 1), abort_word, a.err, a.timeout_ns)) break;
                if (j >= 2 && !wait_or_abort(bar(B_SFREE + sb), (uint32_t)(((j - 2) >> 1) & 1), abort_word, a.err,
                                             a.timeout_ns))
                    break;
                tc_fence_after();
                const uint32_t kb = sKV + s * kStage;
                for (int ks = 0; ks < 12; ++ks)
                    umma_bf16_ss(tmem + 64u * sb,
                                 umma_desc(sQ + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024, kSwizzle128B),
                                 umma_desc(kb + (ks >> 2) * kKBox + (ks & 3) * 32, 16, 1024, kSwizzle128B), iS,
                                 ks > 0 ? 1u : 0u);
                umma_commit(bar(B_SFULL + sb));
                if (j >= 1 && !pv(j - 1)) ok = false;
            }
            if (ok) pv(nt - 1);
            umma_commit(bar(B_ODONE));
            // every MMA issued by this thread has completed before TMEM is freed
            umma_commit(bar(B_DONE));
            if (!mbar_wait_bounded(bar(B_DONE), 0, a.timeout_ns)) report(a.err, KVDEC_DEVERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int qd = warp & 3;                 // TMEM lane quadrant of this warp
        const int row = 32 * qd + lane;          // query row in the block
        const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16);
        const int qpos = a.kv_offset + q0 + row; // this row's position
        const float sl2 = a.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        uint8_t* prow = smem + kOffP + row * 128;
        for (int j = 0; j < nt; ++j) {
            const int sb = j & 1;
            if (!wait_or_abort(bar(B_SFULL + sb), (uint32_t)((j >> 1) & 1), abort_word, a.err, a.timeout_ns)) break;
            tc_fence_after();
            float s[64];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld16(trow + 64u * sb + 16 * c, *reinterpret_cast<float(*)[16]>(s + 16 * c));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_SFREE + sb));
            // causal mask and the tail of the keys
            const int kp0 = j * kBN;
            if (kp0 + kBN - 1 > a.kv_offset + q0 || kp0 + kBN > a.s_kv) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (kp0 + c > qpos || kp0 + c >= a.s_kv) s[c] = -INFINITY;
            }
            float mt[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) mt[i] = fmaxf(s[i], s[i + 32]);
#pragma unroll
            for (int w2 = 16; w2 >= 1; w2 >>= 1)
#pragma unroll
                for (int i = 0; i < w2; ++i) mt[i] = fmaxf(mt[i], mt[i + w2]);
            const float mx = mt[0] * sl2;
            // P(j-1) has been consumed (and O holds PV(j-1)) before P(j) or a rescale
            if (j >= 1 && !wait_or_abort(bar(B_PFREE), (uint32_t)((j - 1) & 1), abort_word, a.err, a.timeout_ns))
                break;
            if (mx > m_ref + 8.f) {
                // new reference max: rescale the running sum and, after a PV, O
                const float alpha = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - mx);
                l *= alpha;
                if (j >= 1) {
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        float o[16];
                        tmem_ld16(trow + kTmemO + 16 * c, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] *= alpha;
                        tmem_st16(trow + kTmemO + 16 * c, o);
                    }
                    tmem_st_wait();
                }
                m_ref = mx;
            }
            const float b = (m_ref == -INFINITY) ? 0.f : m_ref;
            float ls = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = fast_exp2(fmaf(s[8 * k + 2 * e], sl2, -b));
                    const float p1 = fast_exp2(fmaf(s[8 * k + 2 * e + 1], sl2, -b));
                    ls += p0 + p1;
                    pk[e] = pack_bf16x2(p0, p1);
                }
                *reinterpret_cast<uint4*>(prow + ((k ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            l += ls;
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PFULL));
        }
        // ---- O / l out
        if (wait_or_abort(bar(B_ODONE), 0, abort_word, a.err, a.timeout_ns)) {
            tc_fence_after();
            const int r = q0 + row;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                float o[16];
                tmem_ld16(trow + kTmemO + 16 * c, o);
                tmem_ld_wait();
                if (r < a.s_q) {
                    const size_t base = ((size_t)r * a.num_heads + hh) * 128 + 16 * c;
                    if (a.out_bf16) {
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + base);
                        dst[0] = make_uint4(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv),
                                            pack_bf16x2(o[4] * inv, o[5] * inv), pack_bf16x2(o[6] * inv, o[7] * inv));
                        dst[1] = make_uint4(pack_bf16x2(o[8] * inv, o[9] * inv), pack_bf16x2(o[10] * inv, o[11] * inv),
                                            pack_bf16x2(o[12] * inv, o[13] * inv),
                                            pack_bf16x2(o[14] * inv, o[15] * inv));
                    } else {
                        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + base);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv,
                                                 o[4 * e + 3] * inv);
                    }
                }
            }
            if (a.lse && r < a.s_q)
                a.lse[(size_t)r * a.num_heads + hh] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

cudaError_t launch_mla_prefill_tc(const MlaPrefillMaps& maps, const MlaPrefillArgs& a, cudaStream_t st) {
    const dim3 grid((a.s_q + pft::kBM - 1) / pft::kBM, a.num_heads);
    cudaError_t e = cudaFuncSetAttribute(mla_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         pft::kSmem);
    if (e != cudaSuccess) return e;
    mla_prefill_tc_kernel<<<grid, 192, pft::kSmem, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace kvdec
