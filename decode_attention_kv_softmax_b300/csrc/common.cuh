// Shared device helpers for libkvdec (sm_103a): mbarriers with bounded waits,
// TMA tensor loads, warp-level tensor-core fragments, and small numerics.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvdec.h"

#define KVDEC_DEVINL __device__ __forceinline__
#define KVDEC_HDINL __host__ __device__ __forceinline__

namespace kvdec {

// Default limit of every device wait (ns of %globaltimer); a correct run
// never comes near it.
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

KVDEC_DEVINL uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

KVDEC_DEVINL uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// True once more than timeout_ns have passed since t0.  The global timer is
// not guaranteed to be monotonic (it may be stepped), so a reading below t0
// counts as no time passed rather than wrapping around to a huge interval.
KVDEC_DEVINL bool timed_out(uint64_t t0, uint64_t timeout_ns) {
    const uint64_t now = global_timer_ns();
    return now > t0 && now - t0 > timeout_ns;
}

KVDEC_DEVINL void report(uint32_t* flag, uint32_t bits) {
    if (flag) atomicOr(flag, bits);
}

// ---------------------------------------------------------------- mbarrier

KVDEC_DEVINL void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

KVDEC_DEVINL void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

KVDEC_DEVINL void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

KVDEC_DEVINL void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

KVDEC_DEVINL bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity (never suspends the
// thread, unlike try_wait): for polling loops that have other work to do.
KVDEC_DEVINL bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// timeout_ns and returns false (the caller reports and unwinds).
KVDEC_DEVINL bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (timed_out(t0, timeout_ns)) return false;
    }
}

// Wait that also honours a CTA-wide abort word in shared memory: once any
// thread of the CTA has timed out, later waits return false at once so that
// every warp still walks the same control flow (and reaches the same named
// barriers) without touching data that never arrived.
KVDEC_DEVINL bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_word,
                                uint32_t* err, uint64_t timeout_ns) {
    if (*abort_word) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_word) return false;
        if (timed_out(t0, timeout_ns)) {
            *abort_word = 1;
            report(err, KVDEC_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// ---------------------------------------------------------------- clusters

KVDEC_DEVINL uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in cluster CTA `rank`.
KVDEC_DEVINL uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

KVDEC_DEVINL void st_cluster_f4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// Asynchronous store of 16 bytes into another CTA's shared memory; the
// bytes are counted as transaction bytes on that CTA's mbarrier `rbar`.
KVDEC_DEVINL void st_async_f4(uint32_t addr, float a, float b, float c, float d, uint32_t rbar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
        "f"(a), "f"(b), "f"(c), "f"(d), "r"(rbar)
        : "memory");
}

KVDEC_DEVINL void st_async_u4(uint32_t addr, uint4 v, uint32_t rbar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
        "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
        : "memory");
}

// Relaxed arrive on an mbarrier of another CTA of the cluster: orders
// nothing, so it does not wait for this thread's outstanding remote stores.
// Used only to hand back a buffer whose loads have already returned their
// values (a warp issues in order, and those values have been consumed).
KVDEC_DEVINL void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// Arrive (release, cluster scope) on an mbarrier of another CTA of the cluster.
KVDEC_DEVINL void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

KVDEC_DEVINL bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on a local barrier whose phases are completed by arrivals
// from another CTA of the cluster (acquire at cluster scope).
KVDEC_DEVINL bool wait_cluster_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_word,
                                        uint32_t* err, uint64_t timeout_ns) {
    if (*abort_word) return false;
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_acq_cluster(bar, parity)) return true;
        if (*abort_word) return false;
        if (timed_out(t0, timeout_ns)) {
            *abort_word = 1;
            report(err, KVDEC_DEVERR_TIMEOUT);
            return false;
        }
    }
}

KVDEC_DEVINL void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// ---------------------------------------------------------------- TMA

KVDEC_DEVINL uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

KVDEC_DEVINL uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled TMA load into this CTA's shared memory, completion counted in
// bytes on `bar`.  c0 is the innermost (element) coordinate and must be a
// multiple of 8 for bf16 (16 bytes).
KVDEC_DEVINL void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// 3-D tiled TMA load (coordinates innermost first) with an L2 cache hint.
KVDEC_DEVINL void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1, int c2,
                                   uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
        : "memory");
}

// 16-byte asynchronous copy global -> shared memory through L2 only (data
// other SMs wrote), completed by cp_async_wait_all.
KVDEC_DEVINL void cp_async16(uint32_t dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
KVDEC_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
KVDEC_DEVINL void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// wait until at most N of this thread's cp.async groups are pending
template <int N>
KVDEC_DEVINL void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Bring a tensor-map box into L2 ahead of its load (no shared memory, no
// barrier; boxes past the tensor's edge are ignored).
KVDEC_DEVINL void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

KVDEC_DEVINL void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

KVDEC_DEVINL void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 2-D TMA store of a box from (swizzled) shared memory; completion tracked
// by the issuing thread's bulk groups.
KVDEC_DEVINL void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
KVDEC_DEVINL void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared memory of every committed bulk store has been read
KVDEC_DEVINL void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed bulk store has completed (its writes are done)
KVDEC_DEVINL void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

KVDEC_DEVINL void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a TMA
// box written with CU_TENSOR_MAP_SWIZZLE_128B (128-byte rows, box base
// 1024-byte aligned): the chunk index is XOR-ed with the row index mod 8.
KVDEC_DEVINL uint32_t swz128(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// ---------------------------------------------------------------- warp MMA

KVDEC_DEVINL void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

KVDEC_DEVINL void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                            uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
KVDEC_DEVINL void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// f16 inputs, fp32 accumulation (the FP8 path: E4M3 widens exactly to f16)
KVDEC_DEVINL void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

KVDEC_DEVINL uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Four E4M3 codes (byte k = code k) -> two f16x2: lo = (code 0, code 1),
// hi = (code 2, code 3), the first of each pair in the low half.  The 32-bit
// register is split into its 16-bit halves in place, one conversion each.
// Exact: every E4M3 value, subnormals included, is an f16 number.
KVDEC_DEVINL void e4m3x4_to_f16x2x2(uint32_t codes, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(codes));
}

// bf16x2 -> f16x2 (exact for |x| in f16's normal range)
KVDEC_DEVINL uint32_t bf16x2_to_f16x2(uint32_t u) {
    const __half2 h = __floats2half2_rn(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------- numerics

// 2^x on the special-function unit (ex2.approx: a PTX instruction).
// Three-input maximum (one instruction on sm_100 and later).
KVDEC_DEVINL float fmax3f(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

KVDEC_DEVINL float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

KVDEC_DEVINL uint32_t pack_half2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

KVDEC_DEVINL float2 unpack_half2(uint32_t u) {
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

KVDEC_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

KVDEC_DEVINL void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace kvdec
