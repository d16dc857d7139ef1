// Host-side memos that keep repeated calls with the same arguments off the
// driver: a kernel's dynamic shared-memory limit is raised once per (kernel,
// device), and callers look up per-thread memos before taking any lock.
#pragma once

#include <cuda_runtime.h>

#include <mutex>
#include <set>
#include <utility>

namespace kvdec {

// Raises `fn`'s dynamic shared-memory limit to everything the current device
// lets one CTA opt in to, once per (kernel, device).  Every launch of the
// library's kernels asks for at most that much, and the limit never moves
// again, so no launch pays for cudaFuncSetAttribute and no thread can lower
// a limit that another thread's launch relies on.
inline cudaError_t allow_max_dynamic_smem(const void* fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    constexpr int kMemo = 32;
    thread_local const void* memo_fn[kMemo];
    thread_local int memo_dev[kMemo];
    thread_local int memo_n = 0;
    for (int i = 0; i < memo_n; ++i)
        if (memo_fn[i] == fn && memo_dev[i] == dev) return cudaSuccess;
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!done.count({fn, dev})) {
            int optin = 0;
            e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
            if (e != cudaSuccess) return e;
            done.insert({fn, dev});
        }
    }
    if (memo_n < kMemo) {
        memo_fn[memo_n] = fn;
        memo_dev[memo_n] = dev;
        ++memo_n;
    }
    return cudaSuccess;
}

}  // namespace kvdec
