// Causal MLA prefill attention on the non-absorbed path with fifth-generation
// tensor cores ([ARG] "attention-variants-and-kv-cache" §四.6: prefill
// up-projects K and V and runs ordinary causal attention with head dims 192
// and 128; [ARG] §五.2: FlashAttention's tiled online softmax; §五.3: causal
// mask).
//
// CTA = one head and 128 query rows, 8 warps; the CTAs are independent (the
// query blocks of a head read the same K/V tiles, which L2 serves again):
//   warp 0  TMA producer of Q (3 boxes of 128 rows x 64 dims) and, per
//           128-key tile, K (k_nope 0-63, 64-127, k_rope) into a 2-stage ring;
//   warp 6  TMA producer of V (2 boxes of 64 dims) into a 2-stage ring;
//           a stage refills once this CTA's MMAs have released it;
//   warp 1  owns TMEM and issues S(j) = Q K_j^T into S buffer j mod 2 (12
//           MMAs of M=128, N=128, K=16; the K stage is released when they
//           complete);
//   warp 7  issues O += P(j) V_j (8 MMAs of N=128 with P read from TMEM, V
//           MN-major; the V stage is released when they complete).  Both
//           issuers run warp-uniform code and one elected lane issues, and
//           two issuers halve the serial wait-and-issue chain per tile;
//   warps 2-5  softmax, one thread per query row (TMEM lane): load S(j),
//           mask the diagonal and the tail, row max, exponentials packed to
//           bf16 pairs into P buffer j mod 2 in TMEM, row sums.  O is
//           rescaled in TMEM only when a row's max passes its reference max
//           by more than 2^8 (after PV(j-1) has completed).
// TMEM columns: S [0,128) and [128,256), O [256,384), P [384,448) and
// [448,512).  With two S and two P buffers the tensor cores run S(j+1) and
// PV(j-1) while the softmax works on tile j.  N=128 MMAs run at the tensor
// cores' full rate where N=64 ones reach about 55 % of it, and a 128-key
// tile halves the barrier traffic per key.  All waits are bounded; a
// timeout sets the error word and unwinds.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace kvdec {

namespace pft {
constexpr int kBM = 128, kBN = 128;
constexpr int kNK = 2, kNV = 2;            // K and V ring depths
constexpr int kQBytes = 3 * 128 * 128;     // 3 boxes [128 rows x 128 B]
constexpr int kBox = 128 * 128;            // [128 keys x 128 B], loaded as two 64-key halves
constexpr int kHalf = kBox / 2;
constexpr int kKStage = 3 * kBox;          // k_nope 0-63, 64-127, k_rope: 48 KB
constexpr int kVStage = 2 * kBox;          // v 0-63, 64-127: 32 KB
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kNK * kKStage;
constexpr int kOffBars = kOffV + kNV * kVStage;
enum {
    B_Q,
    B_SFULL,
    B_SFREE = B_SFULL + 2,
    B_PFULL = B_SFREE + 2,
    B_PFREE = B_PFULL + 2,
    B_ODONE = B_PFREE + 2,
    B_DONE,
    B_KFULL,
    B_KEMPTY = B_KFULL + kNK,
    B_VFULL = B_KEMPTY + kNK,
    B_VEMPTY = B_VFULL + kNV,
    kBars = B_VEMPTY + kNV
};
constexpr int kOffMisc = kOffBars + kBars * 8;           // [0] TMEM base, [1] abort word
constexpr int kSmem = kOffMisc + 16 + 1024;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0, kTmemO = 256, kTmemP = 384;

// key tiles of query block qb (the causal triangle up to its last row)
__device__ __forceinline__ int block_tiles(const MlaPrefillArgs& a, int qb) {
    const int q0 = qb * kBM;
    const int kend = min(a.s_kv, a.kv_offset + min(q0 + kBM, a.s_q));
    return (kend + kBN - 1) / kBN;
}
}  // namespace pft

__global__ void __launch_bounds__(pft::kThreads, 1)
    mla_prefill_tc_kernel(const __grid_constant__ MlaPrefillMaps maps, const MlaPrefillArgs a) {
    using namespace pft;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // heaviest query blocks first
    const int G = (a.s_q + kBM - 1) / kBM;
    const int qb = G - 1 - (int)blockIdx.x;
    const int hh = blockIdx.y;
    const int q0 = qb * kBM;
    const int nt = block_tiles(a, qb);

    const uint32_t bar0 = smem_addr(smem + kOffBars);
    auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };
    volatile int* misc = reinterpret_cast<volatile int*>(smem + kOffMisc);
    volatile int* abort_word = misc + 1;
    const uint32_t sQ = smem_addr(smem + kOffQ), sK = smem_addr(smem + kOffK), sV = smem_addr(smem + kOffV);

    if (tid == 0) {
        mbar_init(bar(B_Q), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_SFULL + i), 1);
            mbar_init(bar(B_SFREE + i), 4);
            mbar_init(bar(B_PFULL + i), 4);
            mbar_init(bar(B_PFREE + i), 1);
        }
        mbar_init(bar(B_ODONE), 1);
        mbar_init(bar(B_DONE), 1);
        for (int s = 0; s < kNK; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_KEMPTY + s), 1);
        }
        for (int s = 0; s < kNV; ++s) {
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_VEMPTY + s), 1);
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

    if (nt > 0 && (warp == 0 || warp == 6)) {
        // ------------------------------------------------------- producers
        if (lane == 0) {
            const bool is_k = warp == 0;
            const uint64_t keep = l2_policy_evict_last();   // K/V are read by every query block
            if (is_k) {
                prefetch_tensormap(&maps.qn);
                prefetch_tensormap(&maps.qr);
                prefetch_tensormap(&maps.kn);
                prefetch_tensormap(&maps.kr);
                mbar_arrive_expect_tx(bar(B_Q), kQBytes);
                tma_load_3d(sQ, &maps.qn, bar(B_Q), 0, hh, q0);
                tma_load_3d(sQ + 16384, &maps.qn, bar(B_Q), 64, hh, q0);
                tma_load_3d(sQ + 32768, &maps.qr, bar(B_Q), 0, hh, q0);
            } else {
                prefetch_tensormap(&maps.v);
            }
            const int NS = is_k ? kNK : kNV;
            const int empty0 = is_k ? B_KEMPTY : B_VEMPTY, full0 = is_k ? B_KFULL : B_VFULL;
            const int stage_bytes = is_k ? kKStage : kVStage;
            const uint32_t ring = is_k ? sK : sV;
            int issued = 0;
            for (int j = 0; j < nt; ++j) {
                const int k0 = j * kBN, st = j % NS;
                const uint32_t ep = (uint32_t)(((j / NS) & 1) ^ 1);
                if (!wait_or_abort(bar(empty0 + st), ep, abort_word, a.err, a.timeout_ns)) break;
                const uint32_t fb = bar(full0 + st), dst = ring + st * stage_bytes;
                mbar_arrive_expect_tx(fb, stage_bytes);
                // the tile's 128 token rows as two 64-row boxes per dim block
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t d = dst + h * kHalf;
                    const int t = k0 + 64 * h;
                    if (is_k) {
                        tma_load_3d_hint(d, &maps.kn, fb, 0, hh, t, keep);
                        tma_load_3d_hint(d + kBox, &maps.kn, fb, 64, hh, t, keep);
                        tma_load_2d(d + 2 * kBox, &maps.kr, fb, 0, t, keep);
                    } else {
                        tma_load_3d_hint(d, &maps.v, fb, 0, hh, t, keep);
                        tma_load_3d_hint(d + kBox, &maps.v, fb, 64, hh, t, keep);
                    }
                }
                ++issued;
            }
            // never leave TMA writes in flight
            if (is_k && !mbar_wait_bounded(bar(B_Q), 0, a.timeout_ns)) report(a.err, KVDEC_DEVERR_TIMEOUT);
            for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
                if (!mbar_wait_bounded(bar(full0 + i % NS), (uint32_t)((i / NS) & 1), a.timeout_ns)) {
                    report(a.err, KVDEC_DEVERR_TIMEOUT);
                    break;
                }
        }
    } else if (nt > 0 && (warp == 1 || warp == 7)) {
        // ------------------------------------------------------- MMA issuers
        // warp 1 issues S(j) = Q K_j^T, warp 7 O += P(j) V_j.  Each whole warp
        // runs its loop (warp-uniform operands) and one elected lane issues
        // each MMA and commit; a commit covers the MMAs of its own warp.
        // Descriptors are a base plus constant offsets (16-byte units; no
        // carry out of the 14-bit address field below 256 KB).
        auto wait1 = [&](uint32_t b, uint32_t par) -> bool {
            if (__all_sync(0xffffffffu, mbar_try_wait(b, par) ? 1 : 0)) return true;
            int ok = 1;
            if (lane == 0) ok = wait_or_abort(b, par, abort_word, a.err, a.timeout_ns) ? 1 : 0;
            return __all_sync(0xffffffffu, ok) != 0;
        };
        if (warp == 1) {
            constexpr uint32_t iS = umma_idesc_bf16(128, 128, false, false);
            const uint64_t dQ = umma_desc(sQ, 16, 1024, kSwizzle128B);
            const uint64_t dK = umma_desc(sK, 16, 1024, kSwizzle128B);
            bool ok = wait1(bar(B_Q), 0);
            for (int j = 0; ok && j < nt; ++j) {
                const int ks_ = j % kNK, sb = j & 1;
                if (!wait1(bar(B_KFULL + ks_), (uint32_t)((j / kNK) & 1))) break;
                if (j >= 2 && !wait1(bar(B_SFREE + sb), (uint32_t)(((j - 2) >> 1) & 1))) break;
                tc_fence_after();
                const uint64_t dk = dK + (uint64_t)((ks_ * kKStage) >> 4);
#pragma unroll
                for (int ks = 0; ks < 12; ++ks)
                    umma_bf16_ss_w(tmem + kTmemS + 128u * sb,
                                   dQ + (uint64_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                                   dk + (uint64_t)(((ks >> 2) * kBox + (ks & 3) * 32) >> 4), iS, ks > 0 ? 1u : 0u);
                umma_commit_w(bar(B_SFULL + sb));
                umma_commit_w(bar(B_KEMPTY + ks_));   // the K stage may refill
            }
            // every MMA of this warp has completed before TMEM is freed
            umma_commit_w(bar(B_DONE));
            if (lane == 0 && !mbar_wait_bounded(bar(B_DONE), 0, a.timeout_ns)) report(a.err, KVDEC_DEVERR_TIMEOUT);
        } else {
            constexpr uint32_t iP = umma_idesc_bf16(128, 128, false, true);
            const uint64_t dV = umma_desc(sV, kBox, 1024, kSwizzle128B);
            for (int j = 0; j < nt; ++j) {
                const int pb = j & 1, vs = j % kNV;
                if (!wait1(bar(B_PFULL + pb), (uint32_t)((j >> 1) & 1))) break;
                if (!wait1(bar(B_VFULL + vs), (uint32_t)((j / kNV) & 1))) break;
                tc_fence_after();
                const uint64_t dv = dV + (uint64_t)((vs * kVStage) >> 4);
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks)
                    umma_bf16_ts_w(tmem + kTmemO, tmem + kTmemP + 64u * pb + 8u * ks,
                                   dv + (uint64_t)((ks * 2048) >> 4), iP, (j > 0 || ks > 0) ? 1u : 0u);
                umma_commit_w(bar(B_PFREE + pb));
                umma_commit_w(bar(B_VEMPTY + vs));    // the V stage may refill
            }
            // O is final (or the loop was abandoned) once every PV has completed
            umma_commit_w(bar(B_ODONE));
            if (lane == 0 && !mbar_wait_bounded(bar(B_ODONE), 0, a.timeout_ns)) report(a.err, KVDEC_DEVERR_TIMEOUT);
        }
    } else if (nt > 0 && warp >= 2 && warp <= 5) {
        // ------------------------------------------------------------ softmax
        const int qd = warp & 3;                 // TMEM lane quadrant of this warp
        const int row = 32 * qd + lane;          // query row in the block
        const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16);
        const int qpos = a.kv_offset + q0 + row; // this row's position
        const float sl2 = a.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        // completed phases are checked first (no abort-word load on that path)
        auto waitf = [&](uint32_t b, uint32_t par) -> bool {
            return mbar_try_wait(b, par) || wait_or_abort(b, par, abort_word, a.err, a.timeout_ns);
        };
        for (int j = 0; j < nt; ++j) {
            const int sb = j & 1;
            if (!waitf(bar(B_SFULL + sb), (uint32_t)((j >> 1) & 1))) break;
            tc_fence_after();
            float s[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c)
                tmem_ld32(trow + kTmemS + 128u * sb + 32 * c, *reinterpret_cast<float(*)[32]>(s + 32 * c));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_SFREE + sb));
            // causal mask and the tail of the keys
            const int kp0 = j * kBN;
            if (kp0 + kBN - 1 > a.kv_offset + q0 || kp0 + kBN > a.s_kv) {
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (kp0 + c > qpos || kp0 + c >= a.s_kv) s[c] = -INFINITY;
            }
            // row max: three-input maxima, 128 -> 32 -> 11 -> 4 -> 1
            float mt[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) mt[i] = fmaxf(fmax3f(s[i], s[i + 32], s[i + 64]), s[i + 96]);
            float m2[11];
#pragma unroll
            for (int i = 0; i < 10; ++i) m2[i] = fmax3f(mt[3 * i], mt[3 * i + 1], mt[3 * i + 2]);
            m2[10] = fmaxf(mt[30], mt[31]);
            const float m3a = fmax3f(m2[0], m2[1], m2[2]), m3b = fmax3f(m2[3], m2[4], m2[5]);
            const float m3c = fmax3f(m2[6], m2[7], m2[8]), m3d = fmaxf(m2[9], m2[10]);
            const float mx = fmaxf(fmax3f(m3a, m3b, m3c), m3d) * sl2;
            if (mx > m_ref + 8.f) {
                // new reference max: rescale the running sum and, once O holds
                // PV(j-1), O itself
                const float alpha = (m_ref == -INFINITY) ? 0.f : fast_exp2(m_ref - mx);
                l *= alpha;
                if (j >= 1) {
                    if (!wait_or_abort(bar(B_PFREE + ((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1), abort_word,
                                       a.err, a.timeout_ns))
                        break;
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
            // P buffer sb is free once PV(j-2) has completed
            if (j >= 2 && !waitf(bar(B_PFREE + sb), (uint32_t)(((j - 2) >> 1) & 1))) break;
            const float b = (m_ref == -INFINITY) ? 0.f : m_ref;
            // p = 2^(s sl2 - b) with packed f32x2 FMAs and adds (two keys each)
            const float2 sl2x2 = make_float2(sl2, sl2), nbx2 = make_float2(-b, -b);
            float2 ls2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int h = 0; h < kBN / 64; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float2 x = __ffma2_rn(make_float2(s[64 * h + 2 * e], s[64 * h + 2 * e + 1]), sl2x2, nbx2);
                    const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                    ls2 = __fadd2_rn(ls2, p);
                    pk[e] = pack_bf16x2(p.x, p.y);
                }
                tmem_st32u(trow + kTmemP + 64u * sb + 32 * h, pk);
            }
            l += ls2.x + ls2.y;
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PFULL + sb));
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
    const int G = (a.s_q + pft::kBM - 1) / pft::kBM;
    const dim3 grid(G, a.num_heads);
    cudaError_t e = allow_max_dynamic_smem(reinterpret_cast<const void*>(mla_prefill_tc_kernel));
    if (e != cudaSuccess) return e;
    mla_prefill_tc_kernel<<<grid, pft::kThreads, pft::kSmem, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace kvdec

