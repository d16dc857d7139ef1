// MHA / GQA / MQA split-KV decode attention for sm_103a.
//
// What it computes ([ARG] "attention-variants-and-kv-cache" §二.1, §三.2;
// [CH7] shippingwang.com ch.7 §7.3): for sequence b and query head h,
//   out[b,h] = softmax_j(scale * q[b,h] . K[b, h/g, j]) V[b, h/g, j],
// reading each KV head once for all g query heads of its group.
//
// Design (B300):
//  * One CTA = 1 producer warp + 4 consumer warps.  The producer streams
//    64-token K and V tiles with 2-D TMA (128-byte swizzle, L2 evict-first)
//    into an NS-stage shared-memory ring guarded by mbarriers.
//  * Each consumer warp takes 16 of a tile's 64 tokens and runs the whole
//    softmax-attention step on the tensor cores with warp-level
//    m16n8k16 bf16 MMA: S = Q K^T with the group's query heads as the 16
//    MMA rows (zero padded; g > 16 uses two row tiles), an online softmax
//    with quad shuffles (exp2 on the SFU), then O += P V with P taken straight
//    from the S accumulators.  The contraction is tiny (16 x 64 x D per tile),
//    so the kernel stays HBM-bound; the tensor cores only keep the issue
//    slots free for the memory pipeline.
//  * Work is split by the balanced tile schedule in schedule.cuh: every CTA
//    streams the same number of tiles; pieces of a (b, kv head) unit that
//    cross CTAs are merged by log-sum-exp ([ARG] §五.2) in the same kernel by
//    the last CTA to finish the unit.
//  * FP8 cache (F8, [ARG] §六.3: E4M3 halves the bytes per element, one scale
//    per head): the tiles arrive as 8-bit codes, half the bytes, and the
//    MMAs run in f16, to which every E4M3 value widens exactly.  K: ldmatrix
//    on the 8-bit rows hands a thread 4 consecutive dims of one token, so
//    the contraction order inside each 16-dim step is permuted (thread t
//    holds dims 4t..4t+3) and the Q fragments are loaded in that order.  V:
//    each thread reads its 16 dims of each of its 4 tokens with one 16-byte
//    load per token, and byte permutes pair the tokens per dim, giving the
//    B fragment of dim 16g + 4c + i for output tile 4c + i; the output
//    columns are mapped back at the flush.  The K scale folds into the
//    softmax scale, the V scale into the final normalisation.
//  * FP8 with at most 8 query heads per KV head (MT = 0): the same step
//    transposed, S^T = K Q^T and O^T = V^T P^T, so that the warp's 16 tokens
//    and then 16-dim slices of the head fill the MMA's 16 rows and the heads
//    its 8 columns.  Against 16 padded head rows this halves the MMAs, the
//    rescaled accumulators and the Q registers per token; the K codes widen
//    straight into A fragments, P^T reaches the B operand through an in-
//    register 8x8 transpose (movmatrix), and a thread ends up holding 16
//    consecutive dims of two heads.  Built with two CTAs per SM of six
//    stages, and with three of four stages (128 registers) for caches of at
//    most 256 tiles per SM.
//  * Sliding window ([ARG] §五.3): with a ring cache of w slots a step reads
//    the min(seqlen, w) slots holding the last w tokens (read_len).
#include "common.cuh"
#include "kernels.h"
#include "schedule.cuh"

namespace kvdec {


template <int D, int MT, int NS, bool F8>
struct GqaSmem {
    static constexpr int kBoxBytes = 64 * 128;                // 64 rows x 128 B
    static constexpr int kBoxElems = F8 ? 128 : 64;           // elements per box row
    static constexpr int kBoxes = D / kBoxElems;
    static constexpr int kTileBytes = kBoxes * kBoxBytes;     // K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRows = MT == 0 ? 8 : 16 * MT;        // head rows of a chunk
    // padded fp32 row; in the transposed form a thread writes 16 consecutive
    // dims of rows 2 qc, 2 qc + 1, and D + 4 spreads those rows over the banks
    static constexpr int kOStride = MT == 0 ? D + 4 : D + 8;
    static constexpr int kObuf = NS * kStageBytes;
    static constexpr int kStat = kObuf + kRows * kOStride * 4;  // [4 warps][16][2]
    static constexpr int kRowML = kStat + 4 * 16 * 2 * 4;       // [rows][2]
    static constexpr int kBars = kRowML + kRows * 2 * 4;
    static constexpr int kMisc = kBars + 2 * NS * 8;            // ints
    static constexpr int kScratch = kMisc + 4 * 4;
    static constexpr int kCum = kScratch + 160 * 4;
    static constexpr int bytes(int B) { return kCum + (B + 1) * 4 + 1024; }
};

// Transpose of an 8x8 matrix of 16-bit values spread over the warp as an
// MMA fragment (thread t holds row t / 4, columns 2 (t % 4) and 2 (t % 4) + 1),
// returned in the same layout.
KVDEC_DEVINL uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// 16-byte shared-memory load
KVDEC_DEVINL uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

template <int D, int MT, int NS, bool F8>
__global__ void __launch_bounds__(160, (MT == 0 && NS == 4) ? 3 : 2)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const GqaArgs a) {
    static_assert(!F8 || D == 128, "the FP8 path is built for head_dim 128");
    // MT = 0: at most 8 head rows, computed transposed (S^T = K Q^T and
    // O^T = V^T P^T: tokens and dims fill the MMA's 16 rows, the head rows
    // its 8 columns)
    constexpr bool SW = (MT == 0);
    static_assert(!SW || F8, "the transposed form is built for the FP8 cache");
    using L = GqaSmem<D, MT, NS, F8>;
    constexpr int ROWS = L::kRows;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* obuf = reinterpret_cast<float*>(smem + L::kObuf);
    float* stat = reinterpret_cast<float*>(smem + L::kStat);
    float* rowml = reinterpret_cast<float*>(smem + L::kRowML);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
    volatile int* misc = reinterpret_cast<volatile int*>(smem + L::kMisc);
    int* scratch = reinterpret_cast<int*>(smem + L::kScratch);
    int* cum = reinterpret_cast<int*>(smem + L::kCum);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + NS);
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 4);
        }
        misc[0] = 0;
        misc[1] = 0;
        fence_barrier_init();
    }
    build_cum(cum, scratch, a.seqlens, a.B, a.cap, a.err, a.window);

    TileSchedule S;
    S.cum = cum;
    S.B = a.B;
    S.upb = a.n_kv * a.n_hc;
    S.T = (long long)cum[a.B] * S.upb;
    S.W = effective_items(S.T, gridDim.x, a.min_tiles);
    const int w = blockIdx.x;
    if (w >= S.W) return;
    const long long t_begin = S.item_begin(w), t_end = S.item_begin(w + 1);

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        const uint64_t pol = l2_policy_evict_first();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        TileCursor cur;
        if (t_begin < t_end) cur.start(S, t_begin);
        long long issued = 0;
        int stage = 0;
        uint32_t phase = 0;
        for (long long t = t_begin; t < t_end; ++t) {
            if (!wait_or_abort(empty0 + 8 * stage, phase ^ 1, misc, a.err, a.timeout_ns)) break;
            const int kvh = cur.j / a.n_hc;
            int row;
            if (a.paged) {
                int page = (cur.b < a.B && cur.lt < a.max_blocks)
                               ? __ldg(a.block_table + (size_t)cur.b * a.max_blocks + cur.lt)
                               : -1;
                if (page < 0 || page >= a.num_pages) {
                    report(a.err, KVDEC_DEVERR_BAD_PAGE);
                    page = 0;
                }
                row = (page * a.n_kv + kvh) * kTileTokens;
            } else {
                row = (cur.b * a.n_kv + kvh) * a.cap + cur.lt * kTileTokens;
            }
            const uint32_t fb = full0 + 8 * stage;
            mbar_arrive_expect_tx(fb, L::kStageBytes);
            const uint32_t dst = smem_addr(smem + stage * L::kStageBytes);
#pragma unroll
            for (int x = 0; x < L::kBoxes; ++x) {
                tma_load_2d(dst + x * L::kBoxBytes, &tmK, fb, x * L::kBoxElems, row, pol);
                tma_load_2d(dst + L::kTileBytes + x * L::kBoxBytes, &tmV, fb, x * L::kBoxElems, row, pol);
            }
            ++issued;
            if (++stage == NS) {
                stage = 0;
                phase ^= 1;
            }
            cur.advance(S);
        }
        // drain: never leave the CTA with TMA writes in flight
        for (long long i = (issued > NS ? issued - NS : 0); i < issued; ++i) {
            const int st = (int)(i % NS);
            const uint32_t par = (uint32_t)((i / NS) & 1);
            if (!mbar_wait_bounded(full0 + 8 * st, par, a.timeout_ns)) {
                report(a.err, KVDEC_DEVERR_TIMEOUT);
                break;
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Warp roles: warp w owns M-tile mt_w (16 head rows) and TPW tokens of
    // every tile, so a warp's registers do not depend on the group size.
    // Transposed (SW): every warp holds all 8 rows and 16 tokens of a tile.
    constexpr int WPM = SW ? 4 : 4 / MT; // warps per M-tile
    constexpr int TPW = SW ? 16 : 16 * MT;  // tokens per warp per tile
    constexpr int NT = TPW / 8;          // 8-token MMA column tiles per warp
    const int quad = lane >> 2, qc = lane & 3;
    const int mt_w = warp / WPM;
    const int tok_base = (warp % WPM) * TPW;

    // units with no tokens: out = 0, lse = -inf (unit u is handled by item
    // u mod W: step through this item's units only)
    for (int u = w; u < a.B * S.upb; u += S.W) {
        const int b = u / S.upb, j = u % S.upb;
        if (S.ntiles(b) != 0) continue;
        {
            const int kvh = j / a.n_hc, hc = j % a.n_hc;
            const int nr = min(a.hc_rows, a.g - hc * a.hc_rows);
            for (int i = tid; i < nr * D; i += 128) {
                const int r = i / D, c = i % D;
                const size_t o = ((size_t)b * a.H + kvh * a.g + hc * a.hc_rows + r) * D + c;
                if (a.out_bf16) reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16(0.f);
                else reinterpret_cast<float*>(a.out)[o] = 0.f;
            }
            if (a.lse && tid < nr)
                a.lse[(size_t)b * a.H + kvh * a.g + hc * a.hc_rows + tid] = -INFINITY;
        }
    }
    if (t_begin >= t_end) return;

    TileCursor cur;
    cur.start(S, t_begin);
    int stage = 0;
    uint32_t phase = 0;

    // SW: qa[ks] = the B fragment of Q^T for 16-dim step ks; o[nd] = O^T for
    // dims 16 quad + 2 nd, + 1 (rows 2 qc, 2 qc + 1)
    uint32_t qa[D / 16][SW ? 2 : 4];
    float o[SW ? D / 16 : D / 8][4];
    float m[2], l[2];
    int len = 0, nrows = 0;
    bool seg_start = true, seg_item_first = true, seg_unit_first = true;
    float sl2 = a.scale_log2;

    for (long long t = t_begin; t < t_end; ++t) {
        if (seg_start) {
            seg_start = false;
            seg_item_first = (t == t_begin);
            seg_unit_first = (cur.lt == 0);
            len = read_len(__ldg(a.seqlens + cur.b), a.window, a.cap, nullptr);
            const int kvh = cur.j / a.n_hc, hc = cur.j % a.n_hc;
            nrows = min(a.hc_rows, a.g - hc * a.hc_rows);
            const int h0 = kvh * a.g + hc * a.hc_rows;
            if (F8) sl2 = a.scale_log2 * __ldg(a.k_scale + kvh);
            if constexpr (SW) {
                // column quad of Q^T = head row quad; its k order within each
                // 16-dim step follows the K fragments (dims 4 qc .. 4 qc + 3)
                const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                    a.q + ((size_t)cur.b * a.H + h0 + min(quad, nrows - 1)) * D);
                const bool ok = quad < nrows;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint2 u = ok ? __ldg(reinterpret_cast<const uint2*>(qrow + ks * 8 + 2 * qc))
                                       : make_uint2(0u, 0u);
                    qa[ks][0] = bf16x2_to_f16x2(u.x);
                    qa[ks][1] = bf16x2_to_f16x2(u.y);
                }
            } else {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int r = 16 * mt_w + quad + 8 * half;
                    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                        a.q + ((size_t)cur.b * a.H + h0 + min(r, nrows - 1)) * D);
                    const bool ok = r < nrows;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        if constexpr (F8) {
                            // dims 16 ks + 4 qc .. +3, in the order the K fragments use
                            const uint2 u = ok ? __ldg(reinterpret_cast<const uint2*>(qrow + ks * 8 + 2 * qc))
                                               : make_uint2(0u, 0u);
                            qa[ks][half] = bf16x2_to_f16x2(u.x);
                            qa[ks][half + 2] = bf16x2_to_f16x2(u.y);
                        } else {
                            qa[ks][half] = ok ? __ldg(qrow + ks * 8 + qc) : 0u;
                            qa[ks][half + 2] = ok ? __ldg(qrow + ks * 8 + 4 + qc) : 0u;
                        }
                    }
                }
            }
            m[0] = m[1] = -INFINITY;
            l[0] = l[1] = 0.f;
#pragma unroll
            for (int nd = 0; nd < (SW ? D / 16 : D / 8); ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
        }
        const int n_valid = min(kTileTokens, len - cur.lt * kTileTokens);

        if (wait_or_abort(full0 + 8 * stage, phase, misc, a.err, a.timeout_ns)) {
            const uint32_t kb = smem_addr(smem + stage * L::kStageBytes);
            const uint32_t vb = kb + L::kTileBytes;
            if constexpr (SW) {
                // ---- S^T = K Q^T: rows = this warp's 16 tokens, columns = the
                // 8 head rows.  An x4 ldmatrix on the 8-bit rows gives tokens
                // 0-7 / 8-15 of two 16-dim steps; a thread gets 4 consecutive
                // dims of one token, widened to the A fragment in the k order
                // of the Q^T fragments.  Two chains of four MMAs.
                float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t krow = tok_base + (lane & 7) + (lane & 8);
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(kb + swz128(krow, 2 * kk + (lane >> 4)), r0, r1, r2, r3);
                    uint32_t ka[4], kc[4];
                    e4m3x4_to_f16x2x2(r0, ka[0], ka[2]);
                    e4m3x4_to_f16x2x2(r1, ka[1], ka[3]);
                    e4m3x4_to_f16x2x2(r2, kc[0], kc[2]);
                    e4m3x4_to_f16x2x2(r3, kc[1], kc[3]);
                    mma_f16_16816(s, ka, qa[2 * kk][0], qa[2 * kk][1]);
                    mma_f16_16816(s2, kc, qa[2 * kk + 1][0], qa[2 * kk + 1][1]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) s[e] += s2[e];
                // s[0], s[1]: token tok_base + quad, head rows 2 qc, 2 qc + 1;
                // s[2], s[3]: token tok_base + quad + 8, the same rows
                const bool partial = n_valid < kTileTokens;
                if (partial) {
                    if (tok_base + quad >= n_valid) s[0] = s[1] = -INFINITY;
                    if (tok_base + quad + 8 >= n_valid) s[2] = s[3] = -INFINITY;
                }
                // ---- online softmax down the columns (across the 8 quads)
                float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
                for (int x = 4; x < 32; x <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
                }
                const float mn0 = fmaxf(m[0], mx0 * sl2), mn1 = fmaxf(m[1], mx1 * sl2);
                const float b0 = (mn0 == -INFINITY) ? 0.f : mn0;
                const float b1 = (mn1 == -INFINITY) ? 0.f : mn1;
                const float al0 = fast_exp2(m[0] - b0), al1 = fast_exp2(m[1] - b1);
                m[0] = mn0;
                m[1] = mn1;
                const float p0 = fast_exp2(fmaf(s[0], sl2, -b0)), p1 = fast_exp2(fmaf(s[1], sl2, -b1));
                const float p2 = fast_exp2(fmaf(s[2], sl2, -b0)), p3 = fast_exp2(fmaf(s[3], sl2, -b1));
                l[0] = fmaf(l[0], al0, p0 + p2);
                l[1] = fmaf(l[1], al1, p1 + p3);
                // P^T transposed in registers = the B fragment of V^T P^T
                // (k = tokens 2 qc, 2 qc + 1 | + 8, + 9; n = head row quad)
                const uint32_t pb0 = movmatrix_t(pack_half2(p0, p1));
                const uint32_t pb1 = movmatrix_t(pack_half2(p2, p3));
#pragma unroll
                for (int nd = 0; nd < D / 16; ++nd) {
                    o[nd][0] *= al0;
                    o[nd][1] *= al1;
                    o[nd][2] *= al0;
                    o[nd][3] *= al1;
                }
                // ---- O^T += V^T P^T: the thread reads dims 16 quad .. + 15 of
                // tokens tk, tk + 1, tk + 8, tk + 9 (one 16-byte load each);
                // byte permutes pair the tokens per dim.  Dim tile 2 c + h has
                // rows quad / quad + 8 = dims 16 quad + 4 c + 2 h / + 1.
                const int tk = tok_base + 2 * qc;
                const uint32_t keep_lo = (tk < n_valid ? 0x0000ffffu : 0u) | (tk + 1 < n_valid ? 0xffff0000u : 0u);
                const uint32_t keep_hi = (tk + 8 < n_valid ? 0x0000ffffu : 0u) | (tk + 9 < n_valid ? 0xffff0000u : 0u);
                const uint4 x0 = ld_shared_v4(vb + swz128(tk, quad));
                const uint4 x1 = ld_shared_v4(vb + swz128(tk + 1, quad));
                const uint4 x2 = ld_shared_v4(vb + swz128(tk + 8, quad));
                const uint4 x3 = ld_shared_v4(vb + swz128(tk + 9, quad));
                const uint32_t y0[4] = {x0.x, x0.y, x0.z, x0.w}, y1[4] = {x1.x, x1.y, x1.z, x1.w};
                const uint32_t y2[4] = {x2.x, x2.y, x2.z, x2.w}, y3[4] = {x3.x, x3.y, x3.z, x3.w};
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    // lo[i] = dim 16 quad + 4 c + i of tokens (tk, tk + 1),
                    // hi[i] = the same dim of tokens (tk + 8, tk + 9)
                    uint32_t lo[4], hi[4];
                    e4m3x4_to_f16x2x2(__byte_perm(y0[c], y1[c], 0x5140), lo[0], lo[1]);
                    e4m3x4_to_f16x2x2(__byte_perm(y0[c], y1[c], 0x7362), lo[2], lo[3]);
                    e4m3x4_to_f16x2x2(__byte_perm(y2[c], y3[c], 0x5140), hi[0], hi[1]);
                    e4m3x4_to_f16x2x2(__byte_perm(y2[c], y3[c], 0x7362), hi[2], hi[3]);
                    if (partial) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            lo[i] &= keep_lo;
                            hi[i] &= keep_hi;
                        }
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t va[4] = {lo[2 * h], lo[2 * h + 1], hi[2 * h], hi[2 * h + 1]};
                        mma_f16_16816(o[2 * c + h], va, pb0, pb1);
                    }
                }
            } else {
                // ---- S = Q K^T over this warp's TPW tokens
                float s[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint32_t tok = tok_base + nt * 8 + (lane & 7);
                    if constexpr (F8) {
                        // 8-bit rows of 128 dims: matrix i of the x4 load is the
                        // 16-dim step 4 kk + i; a thread gets dims 4 qc .. 4 qc + 3.
                        // Odd steps accumulate apart, so two chains of four
                        // dependent MMAs run side by side instead of one of eight.
                        float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int kk = 0; kk < D / 64; ++kk) {
                            const uint32_t chunk = 4 * kk + (lane >> 3);
                            uint32_t r[4];
                            ldsm_x4(kb + swz128(tok, chunk), r[0], r[1], r[2], r[3]);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                uint32_t b0, b1;
                                e4m3x4_to_f16x2x2(r[i], b0, b1);
                                mma_f16_16816((i & 1) ? s2 : s[nt], qa[4 * kk + i], b0, b1);
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) s[nt][e] += s2[e];
                    } else {
#pragma unroll
                        for (int kk = 0; kk < D / 32; ++kk) {
                            const uint32_t chunk = 4 * kk + (lane >> 3);
                            uint32_t r0, r1, r2, r3;
                            ldsm_x4(kb + (chunk >> 3) * L::kBoxBytes + swz128(tok, chunk & 7), r0, r1, r2, r3);
                            mma_bf16_16816(s[nt], qa[2 * kk], r0, r1);
                            mma_bf16_16816(s[nt], qa[2 * kk + 1], r2, r3);
                        }
                    }
                }
                const bool partial = n_valid < kTileTokens;
                if (partial) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int tk = tok_base + nt * 8 + 2 * qc;
                        if (tk >= n_valid) s[nt][0] = s[nt][2] = -INFINITY;
                        if (tk + 1 >= n_valid) s[nt][1] = s[nt][3] = -INFINITY;
                    }
                }
                // ---- online softmax (base 2, scaled) and P fragments
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
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
                uint32_t pa[MT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float p0 = fast_exp2(fmaf(s[nt][0], sl2, -b0));
                    const float p1 = fast_exp2(fmaf(s[nt][1], sl2, -b0));
                    const float p2 = fast_exp2(fmaf(s[nt][2], sl2, -b1));
                    const float p3 = fast_exp2(fmaf(s[nt][3], sl2, -b1));
                    ps0 += p0 + p1;
                    ps1 += p2 + p3;
                    pa[nt >> 1][(nt & 1) * 2 + 0] = F8 ? pack_half2(p0, p1) : pack_bf16x2(p0, p1);
                    pa[nt >> 1][(nt & 1) * 2 + 1] = F8 ? pack_half2(p2, p3) : pack_bf16x2(p2, p3);
                }
                l[0] = fmaf(l[0], al0, ps0);
                l[1] = fmaf(l[1], al1, ps1);
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd) {
                    o[nd][0] *= al0;
                    o[nd][1] *= al0;
                    o[nd][2] *= al1;
                    o[nd][3] *= al1;
                }
                // ---- O += P V, one 16-token k-step at a time
#pragma unroll
                for (int ks = 0; ks < MT; ++ks) {
                    const int tk = tok_base + 16 * ks + 2 * qc;
                    const uint32_t keep_lo = (tk < n_valid ? 0x0000ffffu : 0u) | (tk + 1 < n_valid ? 0xffff0000u : 0u);
                    const uint32_t keep_hi = (tk + 8 < n_valid ? 0x0000ffffu : 0u) | (tk + 9 < n_valid ? 0xffff0000u : 0u);
                    if constexpr (F8) {
                        // tokens tk, tk+1, tk+8, tk+9 (the B fragment's k rows): a
                        // thread takes dims 16 quad .. 16 quad + 15 of each, one
                        // 16-byte load per token (a quarter-warp's loads hit eight
                        // distinct bank groups under the swizzle); word c holds dims
                        // 16 quad + 4 c .. +3
                        const uint4 x0 = ld_shared_v4(vb + swz128(tk, quad));
                        const uint4 x1 = ld_shared_v4(vb + swz128(tk + 1, quad));
                        const uint4 x2 = ld_shared_v4(vb + swz128(tk + 8, quad));
                        const uint4 x3 = ld_shared_v4(vb + swz128(tk + 9, quad));
                        const uint32_t y0[4] = {x0.x, x0.y, x0.z, x0.w}, y1[4] = {x1.x, x1.y, x1.z, x1.w};
                        const uint32_t y2[4] = {x2.x, x2.y, x2.z, x2.w}, y3[4] = {x3.x, x3.y, x3.z, x3.w};
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            const uint32_t w0 = y0[c], w1 = y1[c], w2 = y2[c], w3 = y3[c];
                            // byte pairs per dim (dims 0, 1 | dims 2, 3), widened:
                            // bl[i] = tokens (tk, tk+1) of dim i, bh[i] = (tk+8, tk+9)
                            uint32_t bl[4], bh[4];
                            e4m3x4_to_f16x2x2(__byte_perm(w0, w1, 0x5140), bl[0], bl[1]);
                            e4m3x4_to_f16x2x2(__byte_perm(w0, w1, 0x7362), bl[2], bl[3]);
                            e4m3x4_to_f16x2x2(__byte_perm(w2, w3, 0x5140), bh[0], bh[1]);
                            e4m3x4_to_f16x2x2(__byte_perm(w2, w3, 0x7362), bh[2], bh[3]);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                uint32_t b0 = bl[i], b1 = bh[i];
                                if (partial) {
                                    b0 &= keep_lo;
                                    b1 &= keep_hi;
                                }
                                mma_f16_16816(o[4 * c + i], pa[ks], b0, b1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int nd2 = 0; nd2 < D / 16; ++nd2) {
                            const int mat = lane >> 3;
                            const uint32_t tok = tok_base + 16 * ks + (mat & 1) * 8 + (lane & 7);
                            const uint32_t chunk = 2 * nd2 + (mat >> 1);
                            uint32_t r0, r1, r2, r3;
                            ldsm_x4_t(vb + (chunk >> 3) * L::kBoxBytes + swz128(tok, chunk & 7), r0, r1, r2, r3);
                            if (partial) {
                                r0 &= keep_lo;
                                r2 &= keep_lo;
                                r1 &= keep_hi;
                                r3 &= keep_hi;
                            }
                            mma_bf16_16816(o[2 * nd2], pa[ks], r0, r1);
                            mma_bf16_16816(o[2 * nd2 + 1], pa[ks], r2, r3);
                    }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);
        if (++stage == NS) {
            stage = 0;
            phase ^= 1;
        }

        const bool seg_end = (cur.lt == cur.nt - 1) || (t == t_end - 1);
        if (seg_end) {
            // ---------------------------------------------------------- flush
            const bool unit_last = (cur.lt == cur.nt - 1);
            const bool complete = seg_unit_first && unit_last;
            const int kvh = cur.j / a.n_hc, hc = cur.j % a.n_hc;
            const int h0 = kvh * a.g + hc * a.hc_rows;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if constexpr (SW) {
                    // rows 2 qc + r: the tokens are spread over the quads
                    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 4);
                    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 8);
                    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 16);
                    if (quad == 0) {
                        stat[(warp * 16 + 2 * qc + r) * 2] = m[r];
                        stat[(warp * 16 + 2 * qc + r) * 2 + 1] = l[r];
                    }
                } else {
                    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
                    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
                    if (qc == 0) {
                        stat[(warp * 16 + quad + 8 * r) * 2] = m[r];
                        stat[(warp * 16 + quad + 8 * r) * 2 + 1] = l[r];
                    }
                }
            }
            named_barrier(1, 128);
            if (tid < ROWS) {
                // row tid of the chunk = row (tid % 16) of M-tile tid / 16
                const int mt = tid >> 4, lr = tid & 15;
                float M = -INFINITY;
                for (int ww = mt * WPM; ww < (mt + 1) * WPM; ++ww) M = fmaxf(M, stat[(ww * 16 + lr) * 2]);
                float Lsum = 0.f;
                if (M != -INFINITY)
                    for (int ww = mt * WPM; ww < (mt + 1) * WPM; ++ww)
                        Lsum += stat[(ww * 16 + lr) * 2 + 1] * fast_exp2(stat[(ww * 16 + lr) * 2] - M);
                rowml[tid * 2] = M;
                rowml[tid * 2 + 1] = Lsum;
            }
            named_barrier(1, 128);
            // The warps of a row tile add their partial O into obuf in WPM
            // ordered steps, all of them in every step: in step s warp i takes
            // the output tiles of slice (i + s) mod WPM, so every element is
            // summed in the same warp order each call.
            for (int step = 0; step < WPM; ++step) {
                const int part = (warp % WPM + step) % WPM;
                {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int row = SW ? 2 * qc + r : 16 * mt_w + quad + 8 * r;
                        const float M = rowml[row * 2];
                        float sc = (M == -INFINITY) ? 0.f : fast_exp2(m[r] - M);
                        if constexpr (SW) {
                            // o[nd][r], o[nd][2 + r] = dims 16 quad + 2 nd, + 1 of this row
                            sc *= __ldg(a.v_scale + kvh);
                            float* dst = obuf + row * L::kOStride + 16 * quad;
#pragma unroll
                            for (int nd = 0; nd < D / 16; nd += 2) {
                                if (nd / (D / 16 / WPM) != part) continue;
                                const float4 v = make_float4(o[nd][r] * sc, o[nd][2 + r] * sc,
                                                             o[nd + 1][r] * sc, o[nd + 1][2 + r] * sc);
                                float4* p4 = reinterpret_cast<float4*>(dst + 2 * nd);
                                if (step == 0) *p4 = v;
                                else {
                                    const float4 u = *p4;
                                    *p4 = make_float4(u.x + v.x, u.y + v.y, u.z + v.z, u.w + v.w);
                                }
                            }
                        } else if constexpr (F8) {
                            // FP8: output tile nd = 4 c + i holds dims 32 qc + 4 c + i (+16)
                            sc *= __ldg(a.v_scale + kvh);
                            float* dst = obuf + row * L::kOStride + 32 * qc;
#pragma unroll
                            for (int nd = 0; nd < D / 8; ++nd) {
                                if (nd / (D / 8 / WPM) != part) continue;
                                float* p0 = dst + 4 * (nd >> 2) + (nd & 3);
                                const float v0 = o[nd][2 * r] * sc, v1 = o[nd][2 * r + 1] * sc;
                                if (step == 0) {
                                    p0[0] = v0;
                                    p0[16] = v1;
                                } else {
                                    p0[0] += v0;
                                    p0[16] += v1;
                                }
                            }
                        } else {
                            float* dst = obuf + row * L::kOStride + 2 * qc;
#pragma unroll
                            for (int nd = 0; nd < D / 8; ++nd) {
                                if (nd / (D / 8 / WPM) != part) continue;
                                float2 v = make_float2(o[nd][2 * r] * sc, o[nd][2 * r + 1] * sc);
                                float2* p2 = reinterpret_cast<float2*>(dst + nd * 8);
                                if (step == 0) *p2 = v;
                                else {
                                    float2 u = *p2;
                                    *p2 = make_float2(u.x + v.x, u.y + v.y);
                                }
                            }
                        }
                    }
                }
                named_barrier(1, 128);
            }
            // normalised result rows -> final output or a partial slot
            const int unit = cur.b * S.upb + cur.j;
            int slot = 0;
            if (!complete) slot = 2 * w + (seg_item_first ? 0 : 1);
            for (int i = tid; i < nrows * (D / 4); i += 128) {
                const int r = i / (D / 4), c4 = i % (D / 4);
                const float Lr = rowml[r * 2 + 1];
                const float inv = Lr > 0.f ? 1.f / Lr : 0.f;
                float4 v = *reinterpret_cast<const float4*>(obuf + r * L::kOStride + c4 * 4);
                v.x *= inv; v.y *= inv; v.z *= inv; v.w *= inv;
                if (complete) {
                    const size_t off = ((size_t)cur.b * a.H + h0 + r) * D + c4 * 4;
                    if (a.out_bf16) {
                        uint2 pk = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
                        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off) = pk;
                    } else {
                        *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off) = v;
                    }
                } else {
                    *reinterpret_cast<float4*>(a.part_o + ((size_t)slot * a.hc_rows + r) * D + c4 * 4) = v;
                }
            }
            if (tid < nrows) {
                const float M = rowml[tid * 2], Lr = rowml[tid * 2 + 1];
                const float lse_v = (Lr > 0.f) ? (M + __log2f(Lr)) * kLn2 : -INFINITY;
                if (complete) {
                    if (a.lse) a.lse[(size_t)cur.b * a.H + h0 + tid] = lse_v;
                } else {
                    a.part_lse[(size_t)slot * a.hc_rows + tid] = lse_v;
                }
            }
            if (!complete) {
                __threadfence();
                named_barrier(1, 128);
                if (tid == 0)
                    misc[1] = arrive_piece(a.counters + unit, a.epoch,
                                           (uint32_t)S.num_pieces(cur.b, cur.j)) ? 1 : 0;
                named_barrier(1, 128);
                if (misc[1]) {
                    // last piece of this unit: merge every piece's partial.
                    // Piece s lives in slot 2 (w0 + s) (+ kind0 for s = 0).
                    __threadfence();
                    const int np = S.num_pieces(cur.b, cur.j);
                    int w0, kind0;
                    S.first_piece(cur.b, cur.j, w0, kind0);
                    if (tid < nrows) {
                        // max and denominator in one pass, four pieces' loads in flight
                        float M = -INFINITY, den = 0.f;
                        for (int s2 = 0; s2 < np; s2 += 4) {
                            float ls[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int sp = s2 + u;
                                const int sl = 2 * (w0 + sp) + (sp == 0 ? kind0 : 0);
                                ls[u] = sp < np ? __ldcg(a.part_lse + (size_t)sl * a.hc_rows + tid) : -INFINITY;
                            }
                            const float Mn = fmaxf(fmaxf(M, fmaxf(ls[0], ls[1])), fmaxf(ls[2], ls[3]));
                            if (Mn != -INFINITY) {
                                den = (M == -INFINITY) ? 0.f : den * fast_exp2((M - Mn) * kLog2e);
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    den += (ls[u] == -INFINITY) ? 0.f : fast_exp2((ls[u] - Mn) * kLog2e);
                                M = Mn;
                            }
                        }
                        rowml[tid * 2] = M;
                        rowml[tid * 2 + 1] = den;
                        if (a.lse)
                            a.lse[(size_t)cur.b * a.H + h0 + tid] = (den > 0.f) ? M + __logf(den) : -INFINITY;
                    }
                    named_barrier(1, 128);
                    for (int i = tid; i < nrows * (D / 4); i += 128) {
                        const int r = i / (D / 4), c4 = i % (D / 4);
                        const float M = rowml[r * 2], den = rowml[r * 2 + 1];
                        const float inv = den > 0.f ? 1.f / den : 0.f;
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                        // four pieces' loads in flight per round trip
                        for (int s2 = 0; s2 < np; s2 += 4) {
                            float ls[4];
                            float4 v[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int sp = s2 + u;
                                const int sl = 2 * (w0 + sp) + (sp == 0 ? kind0 : 0);
                                const bool ok = sp < np;
                                ls[u] = ok ? __ldcg(a.part_lse + (size_t)sl * a.hc_rows + r) : -INFINITY;
                                v[u] = ok ? __ldcg(reinterpret_cast<const float4*>(
                                               a.part_o + ((size_t)sl * a.hc_rows + r) * D + c4 * 4))
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const float wgt = (ls[u] == -INFINITY) ? 0.f : fast_exp2((ls[u] - M) * kLog2e) * inv;
                                acc.x = fmaf(wgt, v[u].x, acc.x);
                                acc.y = fmaf(wgt, v[u].y, acc.y);
                                acc.z = fmaf(wgt, v[u].z, acc.z);
                                acc.w = fmaf(wgt, v[u].w, acc.w);
                            }
                        }
                        const size_t off = ((size_t)cur.b * a.H + h0 + r) * D + c4 * 4;
                        if (a.out_bf16) {
                            uint2 pk = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
                            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + off) = pk;
                        } else {
                            *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + off) = acc;
                        }
                    }
                    if (tid == 0) a.counters[unit] = 0ull;
                }
            }
            named_barrier(1, 128);
            seg_start = true;
        }
        cur.advance(S);
    }
}

// ---------------------------------------------------------------- launcher

template <int D, int MT, int NS, bool F8>
static cudaError_t launch_gqa_t(const CUtensorMap& tk, const CUtensorMap& tv, const GqaArgs& a,
                                int grid, cudaStream_t st) {
    using L = GqaSmem<D, MT, NS, F8>;
    const int smem = L::bytes(a.B);
    auto kern = gqa_decode_kernel<D, MT, NS, F8>;
    cudaError_t e = allow_max_dynamic_smem(reinterpret_cast<const void*>(kern));
    if (e != cudaSuccess) return e;
    kern<<<grid, 160, smem, st>>>(tk, tv, a);
    return cudaGetLastError();
}

template <int D, int MT, int NS, bool F8>
static int occupancy_gqa_t(int B) {
    using L = GqaSmem<D, MT, NS, F8>;
    const int smem = L::bytes(B);
    auto kern = gqa_decode_kernel<D, MT, NS, F8>;
    if (allow_max_dynamic_smem(reinterpret_cast<const void*>(kern)) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 160, smem) != cudaSuccess) return 0;
    return n;
}

// Stages per configuration: a 64-token K+V tile is 32 KB at D=128 (16 KB
// with the FP8 cache), 16 KB at D=64; three (six) of them keep ~96 KB in
// flight per CTA, two CTAs per SM.  MT = 0 (FP8, at most 8 head rows) is the
// transposed form, built twice: two CTAs per SM of six stages, or (dense)
// three of four stages under a 128-register cap.
#define KVDEC_GQA_DISPATCH(FN, ...)                                                          \
    (F8 ? (MT == 0   ? (dense ? FN<128, 0, 4, true>(__VA_ARGS__)                           \
                              : FN<128, 0, 6, true>(__VA_ARGS__))                          \
           : MT == 1 ? FN<128, 1, 6, true>(__VA_ARGS__)                                    \
                     : FN<128, 2, 6, true>(__VA_ARGS__))                                   \
        : D == 128 ? (MT == 1 ? FN<128, 1, 3, false>(__VA_ARGS__) : FN<128, 2, 3, false>(__VA_ARGS__)) \
                   : (MT == 1 ? FN<64, 1, 6, false>(__VA_ARGS__) : FN<64, 2, 6, false>(__VA_ARGS__)))

cudaError_t launch_gqa(int D, int MT, bool F8, bool dense, const CUtensorMap& tk, const CUtensorMap& tv,
                       const GqaArgs& a, int grid, cudaStream_t st) {
    return KVDEC_GQA_DISPATCH(launch_gqa_t, tk, tv, a, grid, st);
}

int occupancy_gqa(int D, int MT, bool F8, bool dense, int B) {
    return KVDEC_GQA_DISPATCH(occupancy_gqa_t, B);
}

}  // namespace kvdec
