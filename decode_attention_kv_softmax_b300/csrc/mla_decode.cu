// MLA absorbed decode on the fifth-generation tensor cores (tcgen05, TMEM).
//
// What it computes ([ARG] "attention-variants-and-kv-cache" §四.5; [MLA]
// "multi-head-latent-attention" §4; [AIFAQ] decoupled-RoPE Q&A): for every
// sequence b and head h,
//   s_j = scale * (q_abs[b,h] . c_kv_j + q_rope[b,h] . k_R_j),
//   out[b,h] = sum_j softmax(s)_j c_kv_j        (512-wide latent output),
// over the paged cache of 576-value rows [c_kv ; k_R]; V is the first 512
// values of the same row, so one load serves both products.
//
// Design (B300).  128 heads x 576 make each 64-token page a dense
// [128 x 576] . [576 x 64] contraction (242 FLOP per byte of cache), so the
// products run on tcgen05 MMAs with fp32 accumulators in TMEM.  The output
// accumulator O[128 x 512] fp32 alone would fill the 512 TMEM columns of an
// SM, so a cluster of two CTAs splits every cache row by columns:
//   CTA 0 holds dims [0,256) and [512,544), CTA 1 holds [256,512) and [544,576).
// Each CTA computes a partial S = Q_r K_r^T over its 288 dims (M=128, N=64,
// K=288), the pair swaps partial S rows through distributed shared memory,
// both run the same online softmax on S = S_0 + S_1, and each accumulates
// O_r += P V_r for its own 256 output columns (M=128, N=256, K=64).  Every
// cache byte is read from HBM once and no MMA is duplicated.
//   TMEM per CTA: O_r at columns [0,256), S at [256,320).
//   Shared memory per CTA: Q_r 72 KB, two 36 KB cache stages, two 16 KB P
//   buffers, the 34 KB partial-S receive buffer.
// Roles: warps 0-3 own one head (TMEM lane) per thread: S readout, the S
// exchange, softmax (base 2, lazy rescale: O is rescaled only when a row's
// running max grows by more than 2^8), P to shared memory, output; warp 4
// issues the MMAs (one thread) and owns the TMEM allocation; warp 5 issues
// the TMA loads (one thread).
// The split-KV schedule (schedule.cuh) gives each CTA pair an equal share of
// all pages; sequences cut across pairs leave normalised partials, merged by
// log-sum-exp ([ARG] §五.2) by the last piece to finish, per head quarter.
#include "common.cuh"
#include "kernels.h"
#include "schedule.cuh"
#include "tcgen05.cuh"

namespace kvdec {

namespace mla {
constexpr int kHeads = 128;
constexpr int kNS = 2;                          // cache stages
constexpr int kQBytes = 4 * 16384 + 8192;       // q_abs 4 x [128 x 64] SW128 + q_rope [128 x 32] SW64
constexpr int kStageBytes = 4 * 8192 + 4096;    // c_kv 4 x [64 x 64] SW128 + rope [64 x 32] SW64
constexpr int kPBytes = 16384;                  // P [128 x 64] bf16, SW128
constexpr int kRecvStride = 68;                 // floats per received partial-S row (padded)
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQBytes;
constexpr int kOffP = kOffKV + kNS * kStageBytes;
constexpr int kOffRecv = kOffP + 2 * kPBytes;
constexpr int kOffBars = kOffRecv + kHeads * kRecvStride * 4;
enum {
    B_Q_FULL, B_Q_FREE, B_KV_FULL, B_KV_EMPTY = B_KV_FULL + kNS, B_S_FULL = B_KV_EMPTY + kNS,
    B_S_FREE, B_P_FULL, B_P_FREE = B_P_FULL + 2, B_O_FREE = B_P_FREE + 2, B_RECV_FULL,
    B_RECV_EMPTY, B_DONE, B_COUNT
};
constexpr int kOffMisc = kOffBars + B_COUNT * 8;   // [0] TMEM base, [1] abort word
constexpr int kThreads = 192;
constexpr int kOffScratch = kOffMisc + 16;
constexpr int kOffCum = kOffScratch + kThreads * 4;
constexpr int smem_bytes(int B) { return kOffCum + (B + 1) * 4 + 1024; }
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;
static_assert(kOffKV % 1024 == 0 && kStageBytes % 1024 == 0 && kOffP % 1024 == 0, "alignment");
static_assert(kOffRecv % 16 == 0 && kOffBars % 8 == 0, "alignment");
}  // namespace mla

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(mla::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ MlaMaps maps, const MlaArgs a) {
    using namespace mla;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    const uint32_t bar0 = smem_addr(bars);
    auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };
    volatile int* misc = reinterpret_cast<volatile int*>(smem + kOffMisc);
    int* scratch = reinterpret_cast<int*>(smem + kOffScratch);
    int* cum = reinterpret_cast<int*>(smem + kOffCum);
    const uint32_t sQ = smem_addr(smem + kOffQ), sKV = smem_addr(smem + kOffKV);
    const uint32_t sP = smem_addr(smem + kOffP);
    float* recv = reinterpret_cast<float*>(smem + kOffRecv);

    if (tid == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        mbar_init(bar(B_Q_FREE), 1);
        for (int s = 0; s < kNS; ++s) {
            mbar_init(bar(B_KV_FULL + s), 1);
            mbar_init(bar(B_KV_EMPTY + s), 1);
        }
        mbar_init(bar(B_S_FULL), 1);
        mbar_init(bar(B_S_FREE), 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_P_FULL + i), 4);
            mbar_init(bar(B_P_FREE + i), 1);
        }
        mbar_init(bar(B_O_FREE), 4);
        mbar_init(bar(B_RECV_FULL), 4);
        mbar_init(bar(B_RECV_EMPTY), 4);
        mbar_init(bar(B_DONE), 1);
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_addr(smem + kOffMisc), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    const int cap = a.max_blocks * kTileTokens;
    build_cum(cum, scratch, a.seqlens, a.B, cap, a.err);   // ends with __syncthreads
    tc_fence_after();
    cluster_sync_all();                                    // the peer's barriers exist
    const uint32_t tmem = (uint32_t)misc[0];

    TileSchedule S;
    S.cum = cum;
    S.B = a.B;
    S.upb = 1;
    S.T = cum[a.B];
    S.W = effective_items(S.T, npairs, a.min_tiles);
    const int w = pair;
    const long long t_begin = (w < S.W && S.T > 0) ? S.item_begin(w) : 0;
    const long long t_end = (w < S.W && S.T > 0) ? S.item_begin(w + 1) : 0;

    if (warp == 5) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && t_begin < t_end) {
            const uint64_t pol = l2_policy_evict_first();
            prefetch_tensormap(&maps.qa);
            prefetch_tensormap(&maps.qr);
            prefetch_tensormap(&maps.c128);
            prefetch_tensormap(&maps.c64);
            TileCursor cur;
            cur.start(S, t_begin);
            int stage = 0, seg = 0;
            uint32_t phase = 0;
            long long issued = 0;
            for (long long t = t_begin; t < t_end; ++t) {
                if (t == t_begin || cur.lt == 0) {
                    if (seg > 0 && !wait_or_abort(bar(B_Q_FREE), (seg - 1) & 1, misc + 1, a.err, a.timeout_ns))
                        break;
                    mbar_arrive_expect_tx(bar(B_Q_FULL), kQBytes);
                    const int row = cur.b * kHeads;
                    for (int c = 0; c < 4; ++c)
                        tma_load_2d(sQ + c * 16384, &maps.qa, bar(B_Q_FULL), 256 * rank + 64 * c, row, pol);
                    tma_load_2d(sQ + 65536, &maps.qr, bar(B_Q_FULL), 32 * rank, row, pol);
                    ++seg;
                }
                if (!wait_or_abort(bar(B_KV_EMPTY + stage), phase ^ 1, misc + 1, a.err, a.timeout_ns)) break;
                int page = __ldg(a.block_table + (size_t)cur.b * a.max_blocks + cur.lt);
                if (page < 0 || page >= a.num_pages) {
                    report(a.err, KVDEC_DEVERR_BAD_PAGE);
                    page = 0;
                }
                const uint32_t fb = bar(B_KV_FULL + stage);
                const uint32_t dst = sKV + stage * kStageBytes;
                mbar_arrive_expect_tx(fb, kStageBytes);
                for (int c = 0; c < 4; ++c)
                    tma_load_2d(dst + c * 8192, &maps.c128, fb, 256 * rank + 64 * c, page * kTileTokens, pol);
                tma_load_2d(dst + 32768, &maps.c64, fb, 512 + 32 * rank, page * kTileTokens, pol);
                ++issued;
                if (++stage == kNS) {
                    stage = 0;
                    phase ^= 1;
                }
                cur.advance(S);
            }
            // never leave TMA writes in flight
            for (long long i = (issued > kNS ? issued - kNS : 0); i < issued; ++i)
                if (!mbar_wait_bounded(bar(B_KV_FULL + (int)(i % kNS)), (uint32_t)((i / kNS) & 1), a.timeout_ns)) {
                    report(a.err, KVDEC_DEVERR_TIMEOUT);
                    break;
                }
            if (seg > 0 && !mbar_wait_bounded(bar(B_Q_FULL), (seg - 1) & 1, a.timeout_ns))
                report(a.err, KVDEC_DEVERR_TIMEOUT);
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && t_begin < t_end) {
            constexpr uint32_t iS = umma_idesc_bf16(128, 64, false, false);
            constexpr uint32_t iP = umma_idesc_bf16(128, 256, false, true);
            TileCursor cur;
            cur.start(S, t_begin);
            int stage = 0, seg = -1;
            uint32_t phase = 0;
            long long it = 0;
            bool pending = false, ok = true;
            long long p_it = 0;
            int p_stage = 0, p_seg = 0;
            bool p_first = false;
            auto issue_pv = [&](long long pit, int pst, bool pfirst, int pseg) -> bool {
                if (!wait_or_abort(bar(B_P_FULL + (int)(pit & 1)), (uint32_t)((pit >> 1) & 1), misc + 1, a.err,
                                   a.timeout_ns))
                    return false;
                if (pfirst && pseg > 0 &&
                    !wait_or_abort(bar(B_O_FREE), (uint32_t)((pseg - 1) & 1), misc + 1, a.err, a.timeout_ns))
                    return false;
                tc_fence_after();
                const uint32_t pb = sP + (uint32_t)(pit & 1) * kPBytes;
                const uint32_t vb = sKV + pst * kStageBytes;
                for (int ks = 0; ks < 4; ++ks)
                    umma_bf16_ss(tmem + kTmemO, umma_desc(pb + ks * 32, 16, 1024, kSwizzle128B),
                                 umma_desc(vb + ks * 2048, 8192, 1024, kSwizzle128B), iP,
                                 (pfirst && ks == 0) ? 0u : 1u);
                umma_commit(bar(B_P_FREE + (int)(pit & 1)));
                umma_commit(bar(B_KV_EMPTY + pst));
                return true;
            };
            for (long long t = t_begin; t < t_end && ok; ++t) {
                const bool seg_first = (t == t_begin) || cur.lt == 0;
                const bool seg_last = (cur.lt == cur.nt - 1) || (t == t_end - 1);
                if (seg_first) {
                    ++seg;
                    if (pending) {          // S of this tile waits for a new Q anyway
                        ok = issue_pv(p_it, p_stage, p_first, p_seg);
                        pending = false;
                        if (!ok) break;
                    }
                    if (!wait_or_abort(bar(B_Q_FULL), (uint32_t)(seg & 1), misc + 1, a.err, a.timeout_ns)) break;
                }
                if (!wait_or_abort(bar(B_KV_FULL + stage), phase, misc + 1, a.err, a.timeout_ns)) break;
                if (it > 0 && !wait_or_abort(bar(B_S_FREE), (uint32_t)((it - 1) & 1), misc + 1, a.err, a.timeout_ns))
                    break;
                tc_fence_after();
                const uint32_t kb = sKV + stage * kStageBytes;
                int n = 0;
                for (int c = 0; c < 4; ++c)
                    for (int ks = 0; ks < 4; ++ks, ++n)
                        umma_bf16_ss(tmem + kTmemS, umma_desc(sQ + c * 16384 + ks * 32, 16, 1024, kSwizzle128B),
                                     umma_desc(kb + c * 8192 + ks * 32, 16, 1024, kSwizzle128B), iS, n > 0);
                for (int ks = 0; ks < 2; ++ks)
                    umma_bf16_ss(tmem + kTmemS, umma_desc(sQ + 65536 + ks * 32, 16, 512, kSwizzle64B),
                                 umma_desc(kb + 32768 + ks * 32, 16, 512, kSwizzle64B), iS, 1u);
                umma_commit(bar(B_S_FULL));
                if (seg_last) umma_commit(bar(B_Q_FREE));
                if (pending) {
                    ok = issue_pv(p_it, p_stage, p_first, p_seg);
                    if (!ok) break;
                }
                pending = true;
                p_it = it;
                p_stage = stage;
                p_first = seg_first;
                p_seg = seg;
                if (++stage == kNS) {
                    stage = 0;
                    phase ^= 1;
                }
                ++it;
                cur.advance(S);
            }
            if (ok && pending && !*(misc + 1)) issue_pv(p_it, p_stage, p_first, p_seg);
            // every MMA issued by this thread has completed before TMEM is freed
            umma_commit(bar(B_DONE));
            if (!mbar_wait_bounded(bar(B_DONE), 0, a.timeout_ns)) report(a.err, KVDEC_DEVERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int row = tid;                                  // head = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        float* my_recv = recv + row * kRecvStride;
        const uint32_t peer_recv = mapa_shared(smem_addr(my_recv), peer);
        const uint32_t peer_full = mapa_shared(bar(B_RECV_FULL), peer);
        const uint32_t peer_empty = mapa_shared(bar(B_RECV_EMPTY), peer);
        const float sl2 = a.scale_log2;
        volatile int* abort_word = misc + 1;

        // sequences with no tokens
        for (int b = 0; b < a.B; ++b) {
            if (S.ntiles(b) != 0 || b % S.W != w || w >= S.W) continue;
            const size_t base = ((size_t)b * kHeads + row) * 512 + 256 * rank;
            for (int c = 0; c < 256; c += 4) {
                if (a.out_bf16)
                    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + base + c) = make_uint2(0u, 0u);
                else
                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + base + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (rank == 0 && a.lse) a.lse[(size_t)b * kHeads + row] = -INFINITY;
        }

        TileCursor cur;
        if (t_begin < t_end) cur.start(S, t_begin);
        float m_run = -INFINITY, l_run = 0.f;
        int len = 0;
        bool seg_item_first = true, seg_unit_first = true;
        long long it = 0;
        for (long long t = t_begin; t < t_end; ++t, ++it) {
            const bool seg_first = (t == t_begin) || cur.lt == 0;
            const bool seg_last = (cur.lt == cur.nt - 1) || (t == t_end - 1);
            if (seg_first) {
                m_run = -INFINITY;
                l_run = 0.f;
                len = clamp_len(__ldg(a.seqlens + cur.b), cap, nullptr);
                seg_item_first = (t == t_begin);
                seg_unit_first = (cur.lt == 0);
            }
            const int n_valid = min(kTileTokens, len - cur.lt * kTileTokens);
            // ---- partial S of this CTA's 288 dims
            if (!wait_or_abort(bar(B_S_FULL), (uint32_t)(it & 1), abort_word, a.err, a.timeout_ns)) break;
            tc_fence_after();
            float s[64];
#pragma unroll
            for (int k = 0; k < 4; ++k) tmem_ld16(trow + kTmemS + 16 * k, *reinterpret_cast<float(*)[16]>(s + 16 * k));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_S_FREE));
            // ---- swap partial rows with the peer: S = S_0 + S_1
            if (it > 0 && !wait_cluster_or_abort(bar(B_RECV_EMPTY), (uint32_t)((it - 1) & 1), abort_word, a.err,
                                                 a.timeout_ns))
                break;
#pragma unroll
            for (int k = 0; k < 16; ++k)
                st_cluster_f4(peer_recv + 16 * k, s[4 * k], s[4 * k + 1], s[4 * k + 2], s[4 * k + 3]);
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(peer_full);
            if (!wait_cluster_or_abort(bar(B_RECV_FULL), (uint32_t)(it & 1), abort_word, a.err, a.timeout_ns))
                break;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float4 v = *reinterpret_cast<const float4*>(my_recv + 4 * k);
                s[4 * k] += v.x;
                s[4 * k + 1] += v.y;
                s[4 * k + 2] += v.z;
                s[4 * k + 3] += v.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(peer_empty);
            // ---- online softmax, base 2, lazy rescale
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                if (j >= n_valid) s[j] = -INFINITY;
                mx = fmaxf(mx, s[j]);
            }
            mx *= sl2;
            float alpha = 1.f;
            bool resc = false;
            if (mx > m_run + 8.f) {
                resc = (m_run != -INFINITY);
                alpha = resc ? fast_exp2(m_run - mx) : 0.f;
                m_run = mx;
            }
            float lsum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float p0 = fast_exp2(fmaf(s[2 * j], sl2, -m_run));
                const float p1 = fast_exp2(fmaf(s[2 * j + 1], sl2, -m_run));
                lsum += p0 + p1;
                pk[j] = pack_bf16x2(p0, p1);
            }
            l_run = l_run * alpha + lsum;
            // ---- P row -> shared memory (K-major, 128-byte swizzle)
            if (it >= 2 && !wait_or_abort(bar(B_P_FREE + (int)(it & 1)), (uint32_t)(((it - 2) >> 1) & 1), abort_word,
                                          a.err, a.timeout_ns))
                break;
            uint8_t* prow = smem + kOffP + (it & 1) * kPBytes + row * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            // ---- tail page: zero the unused V rows (stale bytes may be NaN)
            if (n_valid < kTileTokens) {
                uint8_t* st = smem + kOffKV + (int)(it % kNS) * kStageBytes;
                const int nz = (kTileTokens - n_valid) * 32;   // 16-byte chunks over 4 boxes
                for (int i = row; i < nz; i += 128) {
                    const int r = n_valid + (i >> 5), bx = (i >> 3) & 3, ch = i & 7;
                    *reinterpret_cast<uint4*>(st + bx * 8192 + r * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // ---- rescale O rows whose running max moved (rare)
            if (!seg_first && __any_sync(0xffffffffu, resc)) {
                if (!wait_or_abort(bar(B_P_FREE + (int)((it - 1) & 1)), (uint32_t)(((it - 1) >> 1) & 1), abort_word,
                                   a.err, a.timeout_ns))
                    break;
                tc_fence_after();
                for (int c0 = 0; c0 < 256; c0 += 16) {
                    float v[16];
                    tmem_ld16(trow + kTmemO + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= alpha;
                    tmem_st16(trow + kTmemO + c0, v);
                }
                tmem_st_wait();
            }
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + (int)(it & 1)));

            if (seg_last) {
                // ---------------------------------------------------- flush
                if (!wait_or_abort(bar(B_P_FREE + (int)(it & 1)), (uint32_t)((it >> 1) & 1), abort_word, a.err,
                                   a.timeout_ns))
                    break;
                tc_fence_after();
                const bool complete = seg_unit_first && (cur.lt == cur.nt - 1);
                const int slot = 2 * w + (seg_item_first ? 0 : 1);
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                const float lse_v = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
                const size_t orow = (size_t)cur.b * kHeads + row;
                float* pdst = a.part_o + ((size_t)slot * kHeads + row) * 512 + 256 * rank;
                for (int c0 = 0; c0 < 256; c0 += 16) {
                    float v[16];
                    tmem_ld16(trow + kTmemO + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= inv;
                    if (!complete) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(pdst + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    } else if (a.out_bf16) {
                        __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(a.out) + orow * 512 + 256 * rank + c0;
#pragma unroll
                        for (int i = 0; i < 16; i += 8)
                            *reinterpret_cast<uint4*>(d + i) =
                                make_uint4(pack_bf16x2(v[i], v[i + 1]), pack_bf16x2(v[i + 2], v[i + 3]),
                                           pack_bf16x2(v[i + 4], v[i + 5]), pack_bf16x2(v[i + 6], v[i + 7]));
                    } else {
                        float* d = reinterpret_cast<float*>(a.out) + orow * 512 + 256 * rank + c0;
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(d + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_O_FREE));
                if (complete) {
                    if (rank == 0 && a.lse) a.lse[orow] = lse_v;
                } else {
                    float* plse = a.part_lse + (size_t)rank * (2 * npairs) * kHeads;
                    plse[(size_t)slot * kHeads + row] = lse_v;
                    __threadfence();
                    __syncwarp();
                    int last = 0;
                    if (lane == 0)
                        last = arrive_piece(a.counters + ((size_t)cur.b * 2 + rank) * 4 + warp, a.epoch,
                                            (uint32_t)S.num_pieces(cur.b, 0))
                                   ? 1
                                   : 0;
                    last = __shfl_sync(0xffffffffu, last, 0);
                    if (last) {
                        // merge this warp's 32 heads, this CTA's 256 columns
                        __threadfence();
                        const int np = S.num_pieces(cur.b, 0);
                        int w0, kind0;
                        S.first_piece(cur.b, 0, w0, kind0);
                        float M = -INFINITY, den = 0.f;
                        for (int s2 = 0; s2 < np; ++s2) {
                            const int sl = 2 * (w0 + s2) + (s2 == 0 ? kind0 : 0);
                            M = fmaxf(M, __ldcg(plse + (size_t)sl * kHeads + row));
                        }
                        for (int s2 = 0; s2 < np; ++s2) {
                            const int sl = 2 * (w0 + s2) + (s2 == 0 ? kind0 : 0);
                            const float ls = __ldcg(plse + (size_t)sl * kHeads + row);
                            den += (ls == -INFINITY) ? 0.f : fast_exp2((ls - M) * kLog2e);
                        }
                        if (rank == 0 && a.lse) a.lse[orow] = den > 0.f ? M + __logf(den) : -INFINITY;
                        for (int rr = 0; rr < 32; ++rr) {
                            const int hrow = warp * 32 + rr;
                            const float Mr = __shfl_sync(0xffffffffu, M, rr);
                            const float dr = __shfl_sync(0xffffffffu, den, rr);
                            const float invd = dr > 0.f ? 1.f / dr : 0.f;
                            for (int c4 = lane; c4 < 64; c4 += 32) {
                                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                                for (int s2 = 0; s2 < np; ++s2) {
                                    const int sl = 2 * (w0 + s2) + (s2 == 0 ? kind0 : 0);
                                    const float ls = __ldcg(plse + (size_t)sl * kHeads + hrow);
                                    const float wgt = (ls == -INFINITY) ? 0.f : fast_exp2((ls - Mr) * kLog2e) * invd;
                                    const float4 v = __ldcg(reinterpret_cast<const float4*>(
                                        a.part_o + ((size_t)sl * kHeads + hrow) * 512 + 256 * rank) + c4);
                                    acc.x = fmaf(wgt, v.x, acc.x);
                                    acc.y = fmaf(wgt, v.y, acc.y);
                                    acc.z = fmaf(wgt, v.z, acc.z);
                                    acc.w = fmaf(wgt, v.w, acc.w);
                                }
                                const size_t off = ((size_t)cur.b * kHeads + hrow) * 512 + 256 * rank + 4 * c4;
                                if (a.out_bf16)
                                    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off) =
                                        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
                                else
                                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off) = acc;
                            }
                        }
                    }
                }
            }
            cur.advance(S);
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync_all();   // the peer no longer touches this CTA's shared memory
}

cudaError_t launch_mla(const MlaMaps& maps, const MlaArgs& a, int pairs, cudaStream_t st) {
    const int smem = mla::smem_bytes(a.B);
    cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    mla_decode_kernel<<<2 * pairs, mla::kThreads, smem, st>>>(maps, a);
    return cudaGetLastError();
}

int max_pairs_mla(int B) {
    const int smem = mla::smem_bytes(B);
    if (cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(mla::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace kvdec
