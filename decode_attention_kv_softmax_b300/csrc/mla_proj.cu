// The two absorbed projections around the MLA decode ([ARG]
// "attention-variants-and-kv-cache" §四.5; [MLA] "multi-head-latent-attention"
// §4), per sequence b and head h:
//   absorb:  q~[b,h,:]  = W_UK[h]^T q^C[b,h,:]   (128 -> 512)
//   project: o[b,h,:]   = W_UV[h]   o~[b,h,:]    (512 -> 128)
// with W_UK, W_UV [n_h, 128, 512] bf16.  With x_shared the input rows are
// one [batch, K] matrix for every head: the prefill up-projection
// K^C[t, h] = W_UK[h] c_kv[t], V[t, h] = W_UV[h] c_kv[t] ([ARG] §四.6).  For every head this is a small
// GEMM over the batch: Y_h[B x N] = X_h[B x K] . W_h (absorb: K = 128,
// N = 512, W_h stored [K][N]) or X_h . W_h^T (project: K = 512, N = 128, W_h
// stored [N][K]).  At decode batch sizes it reads the 16.8 MB of weights
// once per call and moves little else, so it is HBM-bound; warp-level
// m16n8k16 bf16 MMA keeps the issue slots free while cp.async streams the
// tiles.
//
// CTA: 4 warps, a 64-row x 128-column output tile of one head; K in chunks
// of 64 through a shared-memory ring (A: 64 x 64, W: 64 x 128; all chunks
// of the absorb in flight, four of the project's eight),
// each row 128 or 256 B with the 16-byte chunks XOR-swizzled by row so that
// ldmatrix reads are conflict-free.  Rows past the batch are zero-filled and
// never stored.
#include "common.cuh"
#include "kernels.h"

namespace kvdec {

namespace proj {
constexpr int kM = 64, kN = 128, kKC = 64;
constexpr int kABytes = kM * kKC * 2;        // 8 KB
constexpr int kWBytes = kKC * kN * 2;        // 16 KB
constexpr int kStage = kABytes + kWBytes;
// ring depth: every chunk of the contraction in flight at once (absorb: 2;
// project: 4 of its 8)
template <bool ABSORB>
__host__ __device__ constexpr int stages() { return ABSORB ? 2 : 4; }
template <bool ABSORB>
__host__ __device__ constexpr int smem() { return stages<ABSORB>() * kStage + 1024; }
}  // namespace proj

KVDEC_DEVINL void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
template <int N>
KVDEC_DEVINL void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool ABSORB>
__global__ void __launch_bounds__(128) mla_proj_kernel(const MlaProjArgs a) {
    using namespace proj;
    constexpr int K = ABSORB ? 128 : 512;     // contraction
    constexpr int N = ABSORB ? 512 : 128;     // output width
    constexpr int NK = K / kKC;
    constexpr int NS = stages<ABSORB>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, m0 = blockIdx.y * kM, n0 = blockIdx.z * kN;
    const __nv_bfloat16* X = a.x;
    const __nv_bfloat16* W = a.w + (size_t)h * 128 * 512;

    // chunk kc of the contraction -> ring slot s
    auto load = [&](int kc, int s) {
        const uint32_t sa = smem_addr(smem + s * kStage);
        const uint32_t sw = sa + kABytes;
        // A: 64 rows x 8 chunks of 16 B
        for (int i = tid; i < kM * 8; i += 128) {
            const int r = i >> 3, c = i & 7;
            const bool ok = m0 + r < a.batch;
            const size_t xr = (size_t)(ok ? m0 + r : 0);
            const __nv_bfloat16* src = X + (a.x_shared ? xr : xr * a.num_heads + h) * K + kc * kKC + c * 8;
            cp_async16(sa + swz128(r, c), src, ok);
        }
        if (ABSORB) {
            // W rows k (64) x 16 chunks of n (256 B per row), chunk c at c ^ (k & 7)
            for (int i = tid; i < kKC * 16; i += 128) {
                const int r = i >> 4, c = i & 15;
                const __nv_bfloat16* src = W + (size_t)(kc * kKC + r) * 512 + n0 + c * 8;
                cp_async16(sw + r * 256 + ((c ^ (r & 7)) << 4), src, true);
            }
        } else {
            // W rows n (128) x 8 chunks of k (128 B per row)
            for (int i = tid; i < kN * 8; i += 128) {
                const int r = i >> 3, c = i & 7;
                const __nv_bfloat16* src = W + (size_t)(n0 + r) * 512 + kc * kKC + c * 8;
                cp_async16(sw + swz128(r, c), src, true);
            }
        }
        cp_async_commit();
    };

    float acc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

    // NS - 1 chunks ahead; an empty group keeps the count uniform at the tail
#pragma unroll
    for (int i = 0; i < NS - 1; ++i) {
        if (i < NK) load(i, i);
        else cp_async_commit();
    }
    for (int kc = 0; kc < NK; ++kc) {
        if (kc + NS - 1 < NK) load(kc + NS - 1, (kc + NS - 1) % NS);
        else cp_async_commit();
        cp_async_wait<NS - 1>();   // chunk kc has landed
        __syncthreads();
        const uint32_t sa = smem_addr(smem + (kc % NS) * kStage);
        const uint32_t sw = sa + kABytes;
#pragma unroll
        for (int ks = 0; ks < kKC / 16; ++ks) {
            // A fragment: rows 16 warp + [0,16), k 16 ks + [0,16)
            uint32_t af[4];
            {
                const int r = 16 * warp + (lane & 15), c = 2 * ks + (lane >> 4);
                ldsm_x4(sa + swz128(r, c), af[0], af[1], af[2], af[3]);
            }
#pragma unroll
            for (int np = 0; np < 8; ++np) {        // pairs of 8-column n tiles
                uint32_t b0, b1, b2, b3;
                if (ABSORB) {
                    // W^T fragments from [k][n] rows: transposed 8x8 loads
                    const int mat = lane >> 3;
                    const int kr = 16 * ks + (mat & 1) * 8 + (lane & 7);
                    const int nc = 2 * np + (mat >> 1);            // 16-byte chunk of n
                    ldsm_x4_t(sw + kr * 256 + ((nc ^ (kr & 7)) << 4), b0, b1, b2, b3);
                } else {
                    // [n][k] rows: n 16 np + [0,16), k 16 ks + [0,16)
                    const int mat = lane >> 3;
                    const int nr = 16 * np + (mat >> 1) * 8 + (lane & 7);
                    const int kc2 = 2 * ks + (mat & 1);
                    ldsm_x4(sw + swz128(nr, kc2), b0, b1, b2, b3);
                }
                mma_bf16_16816(acc[2 * np], af, b0, b1);
                mma_bf16_16816(acc[2 * np + 1], af, b2, b3);
            }
        }
        __syncthreads();   // the slot is refilled NS - 1 chunks later
    }

    // ---- store: thread holds rows (lane / 4) and (lane / 4 + 8) of its warp's
    // 16, columns 8 nt + 2 (lane % 4) + {0, 1}
    const int qrow = lane >> 2, qc = lane & 3;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int b = m0 + 16 * warp + qrow + 8 * half;
        if (b >= a.batch) continue;
        const size_t base = ((size_t)b * a.num_heads + h) * N + n0;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const float v0 = acc[nt][2 * half], v1 = acc[nt][2 * half + 1];
            const int col = 8 * nt + 2 * qc;
            if (a.out_bf16)
                *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.y) + base + col) = pack_bf16x2(v0, v1);
            else
                *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.y) + base + col) = make_float2(v0, v1);
        }
    }
}

cudaError_t launch_mla_proj(bool absorb, const MlaProjArgs& a, cudaStream_t st) {
    const dim3 grid(a.num_heads, (a.batch + proj::kM - 1) / proj::kM, absorb ? 512 / proj::kN : 1);
    if (absorb) {
        cudaError_t e = allow_max_dynamic_smem(reinterpret_cast<const void*>(mla_proj_kernel<true>));
        if (e != cudaSuccess) return e;
        mla_proj_kernel<true><<<grid, 128, proj::smem<true>(), st>>>(a);
    } else {
        cudaError_t e = allow_max_dynamic_smem(reinterpret_cast<const void*>(mla_proj_kernel<false>));
        if (e != cudaSuccess) return e;
        mla_proj_kernel<false><<<grid, 128, proj::smem<false>(), st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kvdec
