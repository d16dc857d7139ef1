// kvdec_gqa_decode_noalloc: the GQA split-KV decode for callers that cannot
// allocate device memory.
//
// kvdec_gqa_decode needs a caller-owned workspace for its split scratch (the
// partial outputs of sequences cut across CTAs and their arrival counters).
// Some callers have no way to provide one: a plugin running inside another
// runtime that owns every byte of device memory through its own allocator,
// or a serving loop that commits all free HBM to the KV cache at start-up and
// forbids any allocation on the decode path (an allocation there can block,
// fragment the pool, or fail under memory pressure).  This entry point runs
// the same kernel with its scratch in a fixed array that the library itself
// holds in device memory, so the caller passes only inputs and outputs.
//
// The array is KVDEC_NOALLOC_SCRATCH_BYTES (16 MiB) per GPU and lives from
// the moment the library's code is loaded on that GPU until the process
// exits.  Its device address is looked up once per device, on the first call
// made with that device current; make that first call before any stream
// capture on that device.  A device reset (cudaDeviceReset) gives the device
// a new context where the array is loaded again; the next call sees the new
// context and looks the address up again, so after a reset that call too
// must come before any capture.  Every call on a device shares the one array, and
// it keeps whatever the previous call left there.  Nothing in it has to start
// at zero: the split counters carry a per-call epoch, so a stale word counts
// as zero.  Calls that overlap on the GPU (two streams, or two host threads)
// race on the array and must be serialised by the caller.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KVDEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
// per device: the array's address and the unique id of the context it was
// looked up in (a reset device gets a new context, where the module and its
// array are loaded again, possibly at another address)
void* g_scratch_addr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the current context (0 if the driver cannot say).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// Device address of the array on the current device, looked up once per
// device (and again if the device's context has changed since).
kvdec_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        kvdec::set_last_error("kvdec_gqa_decode_noalloc: no current CUDA device");
        return KVDEC_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        kvdec::set_last_error("kvdec_gqa_decode_noalloc: device index out of range");
        return KVDEC_ERR_UNSUPPORTED;
    }
    // the context id is read before the lookup on later calls and after it on
    // the first (the lookup itself brings up the device's context)
    const unsigned long long ctx_now = current_context_id();
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx_now) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char buf[256];
            snprintf(buf, sizeof(buf),
                     "kvdec_gqa_decode_noalloc: cudaGetSymbolAddress of the scratch array failed: %s",
                     cudaGetErrorString(e));
            kvdec::set_last_error(buf);
            return KVDEC_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_context_id();
    }
    *out = g_scratch_addr[dev];
    return KVDEC_OK;
}

}  // namespace

extern "C" kvdec_status kvdec_gqa_decode_noalloc(const kvdec_gqa_params* p, void* stream) {
    if (!p) {
        kvdec::set_last_error("kvdec_gqa_decode_noalloc: params is NULL");
        return KVDEC_ERR_INVALID_ARG;
    }
    kvdec_gqa_params q = *p;
    q.workspace = nullptr;
    q.workspace_bytes = 0;
    // Size check first: it needs only the shapes, not the array.
    const size_t need = kvdec_gqa_workspace_bytes(&q);
    if (need == 0) return kvdec_gqa_decode(&q, stream);  // reports the argument error
    if (need > (size_t)KVDEC_NOALLOC_SCRATCH_BYTES) {
        char buf[320];
        snprintf(buf, sizeof(buf),
                 "kvdec_gqa_decode_noalloc: this problem needs %zu bytes of split scratch, more "
                 "than the library's fixed %zu-byte array; lower max_ctas or batch, or call "
                 "kvdec_gqa_decode with a workspace",
                 need, (size_t)KVDEC_NOALLOC_SCRATCH_BYTES);
        kvdec::set_last_error(buf);
        return KVDEC_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    const kvdec_status s = scratch_address(&scratch);
    if (s != KVDEC_OK) return s;
    q.workspace = scratch;
    q.workspace_bytes = KVDEC_NOALLOC_SCRATCH_BYTES;
    return kvdec_gqa_decode(&q, stream);
}
