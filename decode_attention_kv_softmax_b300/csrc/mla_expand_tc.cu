// The up-projection of an MLA prefill chunk on fifth-generation tensor cores
// ([ARG] "attention-variants-and-kv-cache" §四.6: one ordinary weight GEMM
// [s, 512] x [512, n_h 128] per K and V; [MLA] "multi-head-latent-attention"
// §4.2.1):
//   k_nope[t, h, :] = W_UK[h] c_kv[t, :],   v[t, h, :] = W_UV[h] c_kv[t, :]
// With W viewed as [n_h 128, 512] (row h 128 + d) and the outputs as
// [s, n_h 128], both are D = C W^T with C = c_kv [s, 512]: a K-major x
// K-major GEMM, M = s, N = n_h 128, K = 512.
//
// CTA = one 128-token x 256-column output tile (two heads) of K or V
// (blockIdx.z), 6 warps: warp 0 streams the 64-wide K chunks of C (128 x 64)
// and W (256 x 64) by TMA through two stages; warp 1 owns 256 TMEM columns
// and issues M=128, N=256, K=16 MMAs from one thread; warps 2-5 turn the
// fp32 accumulator rows (thread = token = TMEM lane) into bf16 and store
// them.  ~97 KB of shared memory: two CTAs per SM, one's epilogue under the
// other's MMAs.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace kvdec {

namespace ext {
constexpr int kBM = 128, kBN = 256, kBK = 64, kK = 512;
constexpr int kNS = 2;
constexpr int kABytes = kBM * kBK * 2;     // 16 KB
constexpr int kBBytes = kBN * kBK * 2;     // 32 KB
constexpr int kStage = kABytes + kBBytes;
constexpr int kOffBars = kNS * kStage;
enum { B_ACC, B_DONE, B_KV };
constexpr int kBars = B_KV + 2 * kNS;
constexpr int kOffMisc = kOffBars + kBars * 8;
constexpr int kSmem = kOffMisc + 16 + 1024;
constexpr uint32_t kTmemCols = 256;
}  // namespace ext

__global__ void __launch_bounds__(192, 2)
    mla_expand_tc_kernel(const __grid_constant__ MlaExpandMaps maps, const MlaExpandArgs a) {
    using namespace ext;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
    const bool is_v = blockIdx.z != 0;
    const CUtensorMap* wmap = is_v ? &maps.wv : &maps.wk;
    __nv_bfloat16* out = is_v ? a.v : a.k_nope;

    const uint32_t bar0 = smem_addr(smem + kOffBars);
    auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };
    auto kv_full = [bar0](int s) { return bar0 + 8u * (uint32_t)(B_KV + s); };
    auto kv_empty = [bar0](int s) { return bar0 + 8u * (uint32_t)(B_KV + kNS + s); };
    volatile int* misc = reinterpret_cast<volatile int*>(smem + kOffMisc);
    volatile int* abort_word = misc + 1;
    const uint32_t s0 = smem_addr(smem);

    if (tid == 0) {
        mbar_init(bar(B_ACC), 1);
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
    constexpr int NK = kK / kBK;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&maps.c);
            prefetch_tensormap(wmap);
            const uint64_t keep = l2_policy_evict_last();   // C and W are reused by many tiles
            int issued = 0;
            for (int kc = 0; kc < NK; ++kc) {
                const int s = kc % kNS;
                if (!wait_or_abort(kv_empty(s), (uint32_t)(((kc / kNS) & 1) ^ 1), abort_word, a.err, a.timeout_ns))
                    break;
                const uint32_t fb = kv_full(s), dst = s0 + s * kStage;
                mbar_arrive_expect_tx(fb, kStage);
                tma_load_2d(dst, &maps.c, fb, kc * kBK, m0, keep);
                tma_load_2d(dst + kABytes, wmap, fb, kc * kBK, n0, keep);
                ++issued;
            }
            for (int i = (issued > kNS ? issued - kNS : 0); i < issued; ++i)
                if (!mbar_wait_bounded(kv_full(i % kNS), (uint32_t)((i / kNS) & 1), a.timeout_ns)) {
                    report(a.err, KVDEC_DEVERR_TIMEOUT);
                    break;
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(128, 256, false, false);
            for (int kc = 0; kc < NK; ++kc) {
                const int s = kc % kNS;
                if (!wait_or_abort(kv_full(s), (uint32_t)((kc / kNS) & 1), abort_word, a.err, a.timeout_ns)) break;
                tc_fence_after();
                const uint32_t sa = s0 + s * kStage, sb = sa + kABytes;
#pragma unroll
                for (int ks = 0; ks < kBK / 16; ++ks)
                    umma_bf16_ss(tmem, umma_desc(sa + ks * 32, 16, 1024, kSwizzle128B),
                                 umma_desc(sb + ks * 32, 16, 1024, kSwizzle128B), idesc, (kc > 0 || ks > 0) ? 1u : 0u);
                umma_commit(kv_empty(s));
            }
            umma_commit(bar(B_ACC));
            umma_commit(bar(B_DONE));
            if (!mbar_wait_bounded(bar(B_DONE), 0, a.timeout_ns)) report(a.err, KVDEC_DEVERR_TIMEOUT);
        }
    } else {
        // epilogue: thread = token row = TMEM lane
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16);
        if (wait_or_abort(bar(B_ACC), 0, abort_word, a.err, a.timeout_ns)) {
            tc_fence_after();
            const int t = m0 + row;
            uint4* dst = reinterpret_cast<uint4*>(out + (size_t)(t < a.s ? t : 0) * a.N + n0);
#pragma unroll 1
            for (int c = 0; c < kBN / 16; ++c) {
                float v[16];
                tmem_ld16(trow + 16 * c, v);
                tmem_ld_wait();
                if (t < a.s) {
                    dst[2 * c] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                    dst[2 * c + 1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                                                pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

cudaError_t launch_mla_expand_tc(const MlaExpandMaps& maps, const MlaExpandArgs& a, cudaStream_t st) {
    const dim3 grid(a.N / ext::kBN, (a.s + ext::kBM - 1) / ext::kBM, 2);
    cudaError_t e = allow_max_dynamic_smem(reinterpret_cast<const void*>(mla_expand_tc_kernel));
    if (e != cudaSuccess) return e;
    mla_expand_tc_kernel<<<grid, 192, ext::kSmem, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace kvdec
