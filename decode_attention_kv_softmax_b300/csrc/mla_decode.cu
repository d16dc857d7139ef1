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
// K=288), the pair swaps partial S through distributed shared memory, both
// run the same online softmax on S = S_0 + S_1, and each accumulates
// O_r += P V_r for its own 256 output columns (M=128, N=256, K=64).  Every
// cache byte is read from HBM once and no MMA is duplicated.
//   TMEM per CTA (512 columns): O_r [0,256), Q_r [256,400) (bf16 pairs),
//   S [400,464), P [464,496) (bf16 pairs).  Both MMAs take their A operand
//   (Q, P) from TMEM, so shared memory holds only cache pages (five 36 KB
//   stages, TMA with 128/64-byte swizzle) and two 16 KB exchange buffers.
// The partial-S exchange is pipelined one page ahead: while a page's
// softmax runs, the next page's partial S already travels to the peer (as
// fp16) with asynchronous remote stores that complete on the peer's
// mbarrier; the MMA thread keeps S up to two pages ahead of PV.
// Roles: warps 0-7 run the softmax, two warps per TMEM lane quadrant (one
// head per lane, 32 of the 64 columns each; the row max is shared through a
// small buffer); warp 8 issues the MMAs (one thread) and owns the TMEM
// allocation; warp 9 issues the TMA loads (one thread).  Softmax is base 2
// with lazy rescaling: O is rescaled only when a row's running max grows by
// more than 2^8.
// The split-KV schedule (schedule.cuh) gives each CTA pair an equal share of
// all pages; sequences cut across pairs leave normalised partials, merged by
// log-sum-exp ([ARG] §五.2) by the last piece to finish, per warp tile.
#include "common.cuh"
#include "kernels.h"
#include "schedule.cuh"
#include "tcgen05.cuh"

namespace kvdec {

namespace mla {
constexpr int kHeads = 128;
constexpr int kNS = 5;                          // cache stages
constexpr int kStageBytes = 4 * 8192 + 4096;    // c_kv 4 x [64 x 64] SW128 + rope [64 x 32] SW64
constexpr int kOffKV = 0;
constexpr int kOffRecv = kOffKV + kNS * kStageBytes;          // [2][8][128] uint4 (8 fp16) partial S
constexpr int kRecvBytes = 8 * kHeads * 16;                   // one buffer
constexpr int kOffRed = kOffRecv + 2 * kRecvBytes;            // row max: [2 parity][2 halves][128]
constexpr int kOffRedL = kOffRed + 2 * 2 * kHeads * 4;        // row sum at a flush: [2 halves][128]
constexpr int kOffBars = kOffRedL + 2 * kHeads * 4;
enum {
    B_Q_FULL, B_Q_FREE, B_KV_FULL, B_KV_EMPTY = B_KV_FULL + kNS, B_S_FULL = B_KV_EMPTY + kNS,
    B_S_FREE, B_P_FULL, B_P_FREE, B_O_FREE, B_RECV_FULL, B_RECV_EMPTY = B_RECV_FULL + 2,
    B_PAIR = B_RECV_EMPTY + 2, B_DONE = B_PAIR + 4,
    B_COUNT
};
constexpr int kOffMisc = kOffBars + B_COUNT * 8;   // [0] TMEM base, [1] abort word
constexpr int kSoftWarps = 8;
constexpr int kThreads = 32 * (kSoftWarps + 2);
constexpr int kOffScratch = kOffMisc + 16;
constexpr int kOffCum = kOffScratch + kThreads * 4;
constexpr int smem_bytes(int B) { return kOffCum + (B + 1) * 4 + 1024; }
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemQ = 256;
constexpr uint32_t kTmemS = 400;
constexpr uint32_t kTmemP = 464;
static_assert(kStageBytes % 1024 == 0 && kOffRecv % 1024 == 0, "alignment");
static_assert(kOffBars % 8 == 0, "alignment");
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
    volatile int* abort_word = misc + 1;
    int* scratch = reinterpret_cast<int*>(smem + kOffScratch);
    int* cum = reinterpret_cast<int*>(smem + kOffCum);
    const uint32_t sKV = smem_addr(smem + kOffKV);

    if (tid == 0) {
        mbar_init(bar(B_Q_FULL), kSoftWarps);
        mbar_init(bar(B_Q_FREE), 1);
        for (int s = 0; s < kNS; ++s) {
            mbar_init(bar(B_KV_FULL + s), 1);
            mbar_init(bar(B_KV_EMPTY + s), 1);
        }
        mbar_init(bar(B_S_FULL), 1);
        mbar_init(bar(B_S_FREE), kSoftWarps);
        mbar_init(bar(B_P_FULL), kSoftWarps);
        mbar_init(bar(B_P_FREE), 1);
        mbar_init(bar(B_O_FREE), kSoftWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_RECV_FULL + i), 1);           // expect_tx by the receiver
            mbar_init(bar(B_RECV_EMPTY + i), kSoftWarps); // remote arrivals of the peer's warps
        }
        for (int q = 0; q < 4; ++q) mbar_init(bar(B_PAIR + q), 2);
        mbar_init(bar(B_DONE), 1);
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == kSoftWarps) {
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

    if (warp == kSoftWarps + 1) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && t_begin < t_end) {
            const uint64_t pol = l2_policy_evict_first();
            prefetch_tensormap(&maps.c128);
            prefetch_tensormap(&maps.c64);
            TileCursor cur;
            cur.start(S, t_begin);
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            // block-table entry of the cursor's tile; -1 (reported below) if the
            // cursor were ever outside the table
            auto page_of = [&](const TileCursor& c) -> int {
                return (c.b < a.B && c.lt < a.max_blocks)
                           ? __ldg(a.block_table + (size_t)c.b * a.max_blocks + c.lt)
                           : -1;
            };
            int page = page_of(cur);
            for (long long t = t_begin; t < t_end; ++t) {
                if (!wait_or_abort(bar(B_KV_EMPTY + stage), phase ^ 1, abort_word, a.err, a.timeout_ns)) break;
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
                // fetch the next page index now, so its latency overlaps the next wait
                if (t + 1 < t_end) page = page_of(cur);
            }
            // never leave TMA writes in flight
            for (long long i = (issued > kNS ? issued - kNS : 0); i < issued; ++i)
                if (!mbar_wait_bounded(bar(B_KV_FULL + (int)(i % kNS)), (uint32_t)((i / kNS) & 1), a.timeout_ns)) {
                    report(a.err, KVDEC_DEVERR_TIMEOUT);
                    break;
                }
        }
    } else if (warp == kSoftWarps) {
        // ------------------------------------------------------------ MMA issuer
        // Issues S(next) as soon as its page, its Q and a free S buffer are
        // there (at most two pages ahead of PV), and PV(next) as soon as its
        // P is in TMEM; never blocks on one while the other could go.
        if (lane == 0 && t_begin < t_end) {
            constexpr uint32_t iS = umma_idesc_bf16(128, 64, false, false);
            constexpr uint32_t iP = umma_idesc_bf16(128, 256, false, true);
            const long long n = t_end - t_begin;
            TileCursor cs;                       // page of the next S
            cs.start(S, t_begin);
            long long ns = 0, np = 0;            // next S / next PV page index
            int seg_s = -1;                      // segment of the last issued S
            int ring_seg[4];
            bool ring_first[4];
            uint64_t t_wait = 0;
            bool stuck = false;
            while (np < n) {
                bool progress = false;
                if (ns < n && ns <= np + 2) {
                    const bool first = (ns == 0) || cs.lt == 0;
                    const bool last = (cs.lt == cs.nt - 1) || (ns == n - 1);
                    const int stage = (int)(ns % kNS);
                    const bool ready =
                        (!first || mbar_try_wait(bar(B_Q_FULL), (uint32_t)((seg_s + 1) & 1))) &&
                        mbar_try_wait(bar(B_KV_FULL + stage), (uint32_t)((ns / kNS) & 1)) &&
                        (ns == 0 || mbar_try_wait(bar(B_S_FREE), (uint32_t)((ns - 1) & 1)));
                    if (ready) {
                        if (first) ++seg_s;
                        tc_fence_after();
                        const uint32_t kb = sKV + stage * kStageBytes;
                        for (int q = 0; q < 16; ++q)
                            umma_bf16_ts(tmem + kTmemS, tmem + kTmemQ + 8 * q,
                                         umma_desc(kb + (q >> 2) * 8192 + (q & 3) * 32, 16, 1024, kSwizzle128B),
                                         iS, q > 0);
                        for (int q = 0; q < 2; ++q)
                            umma_bf16_ts(tmem + kTmemS, tmem + kTmemQ + 128 + 8 * q,
                                         umma_desc(kb + 32768 + q * 32, 16, 512, kSwizzle64B), iS, 1u);
                        umma_commit(bar(B_S_FULL));
                        if (last) umma_commit(bar(B_Q_FREE));
                        ring_seg[ns & 3] = seg_s;
                        ring_first[ns & 3] = first;
                        ++ns;
                        cs.advance(S);
                        progress = true;
                    }
                }
                if (np < ns) {
                    const bool pfirst = ring_first[np & 3];
                    const int pseg = ring_seg[np & 3];
                    const bool ready =
                        mbar_try_wait(bar(B_P_FULL), (uint32_t)(np & 1)) &&
                        (!pfirst || pseg == 0 || mbar_try_wait(bar(B_O_FREE), (uint32_t)((pseg - 1) & 1)));
                    if (ready) {
                        tc_fence_after();
                        const int pst = (int)(np % kNS);
                        const uint32_t vb = sKV + pst * kStageBytes;
                        for (int ks = 0; ks < 4; ++ks)
                            umma_bf16_ts(tmem + kTmemO, tmem + kTmemP + 8 * ks,
                                         umma_desc(vb + ks * 2048, 8192, 1024, kSwizzle128B), iP,
                                         (pfirst && ks == 0) ? 0u : 1u);
                        umma_commit(bar(B_P_FREE));
                        umma_commit(bar(B_KV_EMPTY + pst));
                        ++np;
                        progress = true;
                    }
                }
                if (progress) {
                    t_wait = 0;
                } else {
                    if (*abort_word) break;
                    const uint64_t now = global_timer_ns();
                    if (t_wait == 0) {
                        t_wait = now;
                    } else if (now - t_wait > a.timeout_ns) {
                        stuck = true;
                        break;
                    }
                }
            }
            if (stuck) {
                *abort_word = 1;
                report(a.err, KVDEC_DEVERR_TIMEOUT);
            }
            // every MMA issued by this thread has completed before TMEM is freed
            umma_commit(bar(B_DONE));
            if (!mbar_wait_bounded(bar(B_DONE), 0, a.timeout_ns)) report(a.err, KVDEC_DEVERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int qd = warp & 3, half = warp >> 2;
        const int row = qd * 32 + lane;                       // head = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
        const uint4* recv4 = reinterpret_cast<const uint4*>(smem + kOffRecv);    // [2][8][128]
        float* red = reinterpret_cast<float*>(smem + kOffRed);       // [2][2][128]
        float* red_l = reinterpret_cast<float*>(smem + kOffRedL);    // [2][128]
        const uint32_t peer_recv = mapa_shared(smem_addr(smem + kOffRecv), peer);
        const uint32_t peer_full = mapa_shared(bar(B_RECV_FULL), peer);
        const uint32_t peer_empty = mapa_shared(bar(B_RECV_EMPTY), peer);
        const uint32_t pair_bar = bar(B_PAIR + qd);
        const float sl2 = a.scale_log2;
        uint32_t pair_uses = 0;
        // row-wide exchange with the other half of this quadrant
        auto pair_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(pair_bar);
            const bool ok = wait_or_abort(pair_bar, pair_uses & 1, abort_word, a.err, a.timeout_ns);
            ++pair_uses;
            return ok;
        };

        // sequences with no tokens
        for (int b = 0; b < a.B; ++b) {
            if (w >= S.W || S.ntiles(b) != 0 || b % S.W != w) continue;
            const size_t base = ((size_t)b * kHeads + row) * 512 + 256 * rank + 128 * half;
            for (int c = 0; c < 128; c += 4) {
                if (a.out_bf16)
                    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + base + c) = make_uint2(0u, 0u);
                else
                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + base + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (rank == 0 && half == 0 && a.lse) a.lse[(size_t)b * kHeads + row] = -INFINITY;
        }

        const long long n = t_end - t_begin;
        int qseg = -1;
        // Q_r of a sequence -> TMEM (bf16 pairs), once the previous sequence's
        // last S has completed
        auto load_q = [&](int b) -> bool {
            ++qseg;
            if (qseg > 0 &&
                !wait_or_abort(bar(B_Q_FREE), (uint32_t)((qseg - 1) & 1), abort_word, a.err, a.timeout_ns))
                return false;
            const uint4* qa_row = reinterpret_cast<const uint4*>(
                a.q_abs + ((size_t)b * kHeads + row) * 512 + 256 * rank + 128 * half);
            uint32_t v[16];
#pragma unroll
            for (int c = 0; c < 4; ++c) {       // 128 bf16 of q_abs = 64 columns
                const uint4 x0 = __ldg(qa_row + 4 * c), x1 = __ldg(qa_row + 4 * c + 1);
                const uint4 x2 = __ldg(qa_row + 4 * c + 2), x3 = __ldg(qa_row + 4 * c + 3);
                v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
                v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
                v[8] = x2.x; v[9] = x2.y; v[10] = x2.z; v[11] = x2.w;
                v[12] = x3.x; v[13] = x3.y; v[14] = x3.z; v[15] = x3.w;
                tmem_st16u(trow + kTmemQ + 64 * half + 16 * c, v);
            }
            if (half == 1) {                    // 32 bf16 of q_rope = 16 columns
                const uint4* qr_row = reinterpret_cast<const uint4*>(
                    a.q_rope + ((size_t)b * kHeads + row) * 64 + 32 * rank);
                const uint4 x0 = __ldg(qr_row), x1 = __ldg(qr_row + 1);
                const uint4 x2 = __ldg(qr_row + 2), x3 = __ldg(qr_row + 3);
                v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
                v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
                v[8] = x2.x; v[9] = x2.y; v[10] = x2.z; v[11] = x2.w;
                v[12] = x3.x; v[13] = x3.y; v[14] = x3.z; v[15] = x3.w;
                tmem_st16u(trow + kTmemQ + 128, v);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_Q_FULL));
            return true;
        };
        // partial S of page j (this half's 32 columns) -> registers and, with
        // asynchronous remote stores, the peer's receive buffer j & 1
        auto read_send = [&](long long j, float (&dst)[32]) -> bool {
            if (!wait_or_abort(bar(B_S_FULL), (uint32_t)(j & 1), abort_word, a.err, a.timeout_ns)) return false;
            tc_fence_after();
            tmem_ld16(trow + kTmemS + 32 * half, *reinterpret_cast<float(*)[16]>(dst));
            tmem_ld16(trow + kTmemS + 32 * half + 16, *reinterpret_cast<float(*)[16]>(dst + 16));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_S_FREE));
            const uint32_t buf = (uint32_t)(j & 1);
            if (j >= 2 && !wait_cluster_or_abort(bar(B_RECV_EMPTY + (int)buf), (uint32_t)(((j - 2) >> 1) & 1),
                                                 abort_word, a.err, a.timeout_ns))
                return false;
            // sent as fp16: the error this adds to a probability is relative,
            // about scale * |S_peer| * 2^-12, no larger than the bf16 rounding of P
            const uint32_t dst_base = peer_recv + buf * kRecvBytes;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint4 hv;
                hv.x = pack_half2(dst[8 * k], dst[8 * k + 1]);
                hv.y = pack_half2(dst[8 * k + 2], dst[8 * k + 3]);
                hv.z = pack_half2(dst[8 * k + 4], dst[8 * k + 5]);
                hv.w = pack_half2(dst[8 * k + 6], dst[8 * k + 7]);
                st_async_u4(dst_base + (uint32_t)(((4 * half + k) * kHeads + row) * 16), hv, peer_full + 8u * buf);
            }
            return true;
        };

        TileCursor cur, nxt;
        float s_cur[32], s_nxt[32];
        bool ok = true;
        if (n > 0) {
            cur.start(S, t_begin);
            nxt = cur;
            ok = load_q(cur.b) && read_send(0, s_cur);
        }
        float m_run = -INFINITY, l_run = 0.f;
        int len = 0;
        bool seg_item_first = true, seg_unit_first = true;
        for (long long it = 0; ok && it < n; ++it) {
            const long long t = t_begin + it;
            const bool seg_first = (t == t_begin) || cur.lt == 0;
            const bool seg_last = (cur.lt == cur.nt - 1) || (t == t_end - 1);
            // ---- look ahead: the next page's partial S leaves for the peer now
            if (it + 1 < n) {
                nxt.advance(S);
                if (nxt.lt == 0 && !load_q(nxt.b)) break;
                if (!read_send(it + 1, s_nxt)) break;
            }
            if (seg_first) {
                // warm L2 with the next sequence's Q rows, needed at the next switch
                if (cur.b + 1 < a.B) {
                    const char* nq = reinterpret_cast<const char*>(
                        a.q_abs + ((size_t)(cur.b + 1) * kHeads + row) * 512 + 256 * rank + 128 * half);
                    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(nq));
                    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(nq + 128));
                    if (half == 1)
                        asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(reinterpret_cast<const char*>(
                            a.q_rope + ((size_t)(cur.b + 1) * kHeads + row) * 64 + 32 * rank)));
                }
                m_run = -INFINITY;
                l_run = 0.f;
                len = clamp_len(__ldg(a.seqlens + cur.b), cap, nullptr);
                seg_item_first = (t == t_begin);
                seg_unit_first = (cur.lt == 0);
            }
            const int n_valid = min(kTileTokens, len - cur.lt * kTileTokens);
            // ---- the peer's partial S of this page
            const int buf = (int)(it & 1);
            if (tid == 0) mbar_arrive_expect_tx(bar(B_RECV_FULL + buf), kRecvBytes);
            if (!wait_cluster_or_abort(bar(B_RECV_FULL + buf), (uint32_t)((it >> 1) & 1), abort_word, a.err,
                                       a.timeout_ns))
                break;
            float s[32];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 x = recv4[(buf * 8 + 4 * half + k) * kHeads + row];
                const float2 a0 = unpack_half2(x.x), a1 = unpack_half2(x.y);
                const float2 a2 = unpack_half2(x.z), a3 = unpack_half2(x.w);
                s[8 * k] = s_cur[8 * k] + a0.x;
                s[8 * k + 1] = s_cur[8 * k + 1] + a0.y;
                s[8 * k + 2] = s_cur[8 * k + 2] + a1.x;
                s[8 * k + 3] = s_cur[8 * k + 3] + a1.y;
                s[8 * k + 4] = s_cur[8 * k + 4] + a2.x;
                s[8 * k + 5] = s_cur[8 * k + 5] + a2.y;
                s[8 * k + 6] = s_cur[8 * k + 6] + a3.x;
                s[8 * k + 7] = s_cur[8 * k + 7] + a3.y;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(peer_empty + 8u * (uint32_t)buf);
            // ---- row max over both halves, lazy rescale, base-2 probabilities
            float mx = -INFINITY;
#pragma unroll
            for (int j2 = 0; j2 < 32; ++j2) {
                if (32 * half + j2 >= n_valid) s[j2] = -INFINITY;
                mx = fmaxf(mx, s[j2]);
            }
            red[((it & 1) * 2 + half) * kHeads + row] = mx;
            if (!pair_sync()) break;
            mx = fmaxf(mx, red[((it & 1) * 2 + (half ^ 1)) * kHeads + row]) * sl2;
            float alpha = 1.f;
            bool resc = false;
            if (mx > m_run + 8.f) {
                resc = (m_run != -INFINITY);
                alpha = resc ? fast_exp2(m_run - mx) : 0.f;
                m_run = mx;
            }
            float lsum = 0.f;
            uint32_t pk[16];
#pragma unroll
            for (int j2 = 0; j2 < 16; ++j2) {
                const float p0 = fast_exp2(fmaf(s[2 * j2], sl2, -m_run));
                const float p1 = fast_exp2(fmaf(s[2 * j2 + 1], sl2, -m_run));
                lsum += p0 + p1;
                pk[j2] = pack_bf16x2(p0, p1);
            }
            l_run = l_run * alpha + lsum;      // this half's share of the row sum
            // ---- P (this half's 32 tokens) -> TMEM once PV of the previous page is done
            if (it > 0 &&
                !wait_or_abort(bar(B_P_FREE), (uint32_t)((it - 1) & 1), abort_word, a.err, a.timeout_ns))
                break;
            tc_fence_after();
            tmem_st16u(trow + kTmemP + 16 * half, pk);
            // ---- tail page: zero the unused V rows (stale bytes may be NaN)
            if (n_valid < kTileTokens) {
                uint8_t* st = smem + kOffKV + (int)(it % kNS) * kStageBytes;
                const int nz = (kTileTokens - n_valid) * 32;   // 16-byte chunks over 4 boxes
                for (int i2 = tid; i2 < nz; i2 += 32 * kSoftWarps) {
                    const int r = n_valid + (i2 >> 5), bx = (i2 >> 3) & 3, ch = i2 & 7;
                    *reinterpret_cast<uint4*>(st + bx * 8192 + r * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async();
            }
            // ---- rescale this half's 128 O columns where the running max moved (rare)
            if (!seg_first && __any_sync(0xffffffffu, resc)) {
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    float o[16];
                    tmem_ld16(trow + kTmemO + 128 * half + c0, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2) o[i2] *= alpha;
                    tmem_st16(trow + kTmemO + 128 * half + c0, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL));

            if (seg_last) {
                // ---------------------------------------------------- flush
                red_l[half * kHeads + row] = l_run;
                if (!pair_sync()) break;
                const float l_tot = l_run + red_l[(half ^ 1) * kHeads + row];
                if (!wait_or_abort(bar(B_P_FREE), (uint32_t)(it & 1), abort_word, a.err, a.timeout_ns)) break;
                tc_fence_after();
                const bool complete = seg_unit_first && (cur.lt == cur.nt - 1);
                const int slot = 2 * w + (seg_item_first ? 0 : 1);
                const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
                const float lse_v = l_tot > 0.f ? (m_run + __log2f(l_tot)) * kLn2 : -INFINITY;
                const size_t orow = (size_t)cur.b * kHeads + row;
                const int col0 = 256 * (int)rank + 128 * half;
                float* pdst = a.part_o + ((size_t)slot * kHeads + row) * 512 + col0;
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    float o[16];
                    tmem_ld16(trow + kTmemO + 128 * half + c0, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2) o[i2] *= inv;
                    if (!complete) {
#pragma unroll
                        for (int i2 = 0; i2 < 16; i2 += 4)
                            *reinterpret_cast<float4*>(pdst + c0 + i2) = make_float4(o[i2], o[i2 + 1], o[i2 + 2], o[i2 + 3]);
                    } else if (a.out_bf16) {
                        __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(a.out) + orow * 512 + col0 + c0;
#pragma unroll
                        for (int i2 = 0; i2 < 16; i2 += 8)
                            *reinterpret_cast<uint4*>(d + i2) =
                                make_uint4(pack_bf16x2(o[i2], o[i2 + 1]), pack_bf16x2(o[i2 + 2], o[i2 + 3]),
                                           pack_bf16x2(o[i2 + 4], o[i2 + 5]), pack_bf16x2(o[i2 + 6], o[i2 + 7]));
                    } else {
                        float* d = reinterpret_cast<float*>(a.out) + orow * 512 + col0 + c0;
#pragma unroll
                        for (int i2 = 0; i2 < 16; i2 += 4)
                            *reinterpret_cast<float4*>(d + i2) = make_float4(o[i2], o[i2 + 1], o[i2 + 2], o[i2 + 3]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_O_FREE));
                if (complete) {
                    if (rank == 0 && half == 0 && a.lse) a.lse[orow] = lse_v;
                } else {
                    // this warp's own copy of the partial lse: [rank][half][slot][row]
                    float* plse = a.part_lse + (size_t)(rank * 2 + half) * (2 * npairs) * kHeads;
                    plse[(size_t)slot * kHeads + row] = lse_v;
                    __threadfence();
                    __syncwarp();
                    int last = 0;
                    if (lane == 0)
                        last = arrive_piece(a.counters + ((size_t)cur.b * 2 + rank) * kSoftWarps + warp, a.epoch,
                                            (uint32_t)S.num_pieces(cur.b, 0))
                                   ? 1
                                   : 0;
                    last = __shfl_sync(0xffffffffu, last, 0);
                    if (last) {
                        // merge this warp's 32 heads x 128 columns over every piece
                        __threadfence();
                        const int npc = S.num_pieces(cur.b, 0);
                        int w0, kind0;
                        S.first_piece(cur.b, 0, w0, kind0);
                        float M = -INFINITY, den = 0.f;
                        for (int s2 = 0; s2 < npc; ++s2) {
                            const int sl = 2 * (w0 + s2) + (s2 == 0 ? kind0 : 0);
                            M = fmaxf(M, __ldcg(plse + (size_t)sl * kHeads + row));
                        }
                        for (int s2 = 0; s2 < npc; ++s2) {
                            const int sl = 2 * (w0 + s2) + (s2 == 0 ? kind0 : 0);
                            const float ls = __ldcg(plse + (size_t)sl * kHeads + row);
                            den += (ls == -INFINITY) ? 0.f : fast_exp2((ls - M) * kLog2e);
                        }
                        if (rank == 0 && half == 0 && a.lse) a.lse[orow] = den > 0.f ? M + __logf(den) : -INFINITY;
                        const float invd = den > 0.f ? 1.f / den : 0.f;
                        // 8 rows at a time, every row's load in flight together
                        for (int r0 = 0; r0 < 32; r0 += 8) {
                            float4 acc[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                            for (int s2 = 0; s2 < npc; ++s2) {
                                const int sl = 2 * (w0 + s2) + (s2 == 0 ? kind0 : 0);
                                const float ls = __ldcg(plse + (size_t)sl * kHeads + row);
                                const float wm = (ls == -INFINITY) ? 0.f : fast_exp2((ls - M) * kLog2e) * invd;
                                const float4* src = reinterpret_cast<const float4*>(
                                    a.part_o + ((size_t)sl * kHeads + qd * 32 + r0) * 512 + col0) + lane;
                                float4 v[8];
#pragma unroll
                                for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (size_t)u * 128);
#pragma unroll
                                for (int u = 0; u < 8; ++u) {
                                    const float wgt = __shfl_sync(0xffffffffu, wm, r0 + u);
                                    acc[u].x = fmaf(wgt, v[u].x, acc[u].x);
                                    acc[u].y = fmaf(wgt, v[u].y, acc[u].y);
                                    acc[u].z = fmaf(wgt, v[u].z, acc[u].z);
                                    acc[u].w = fmaf(wgt, v[u].w, acc[u].w);
                                }
                            }
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const size_t off = ((size_t)cur.b * kHeads + qd * 32 + r0 + u) * 512 + col0 + 4 * lane;
                                if (a.out_bf16)
                                    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off) =
                                        make_uint2(pack_bf16x2(acc[u].x, acc[u].y), pack_bf16x2(acc[u].z, acc[u].w));
                                else
                                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off) = acc[u];
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) s_cur[k] = s_nxt[k];
            cur.advance(S);
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kSoftWarps) {
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
