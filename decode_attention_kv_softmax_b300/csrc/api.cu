// Host side of the C ABI declared in include/kvdec.h: argument checks,
// workspace layout, TMA tensor-map encoding and kernel launches.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "common.cuh"

#include "kernels.h"

namespace {

thread_local std::string g_last_error;

kvdec_status fail(kvdec_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kvdec_status fail(kvdec_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

kvdec_status cuda_fail(cudaError_t e, const char* what) {
    return fail(KVDEC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- devices

struct DeviceInfo {
    int sm_count = 0;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<std::tuple<int, int, int, int, int>, int> g_occupancy;  // (dev, kind, D, MT, B)

bool device_info(DeviceInfo& out, int& dev) {
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    // per-thread memo first: the common case takes no lock
    constexpr int kMemo = 8;
    thread_local int memo_dev[kMemo];
    thread_local DeviceInfo memo_info[kMemo];
    thread_local int memo_n = 0;
    for (int i = 0; i < memo_n; ++i)
        if (memo_dev[i] == dev) {
            out = memo_info[i];
            return true;
        }
    std::lock_guard<std::mutex> lk(g_mu);
    if (memo_n < kMemo) {
        auto it = g_devices.find(dev);
        DeviceInfo d;
        if (it != g_devices.end()) {
            d = it->second;
        } else {
            if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return false;
            g_devices[dev] = d;
        }
        memo_dev[memo_n] = dev;
        memo_info[memo_n] = d;
        ++memo_n;
        out = d;
        return true;
    }
    auto it = g_devices.find(dev);
    if (it != g_devices.end()) {
        out = it->second;
        return true;
    }
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    g_devices[dev] = d;
    out = d;
    return true;
}

// Resident CTAs (or CTA pairs) per launch shape, keyed (device, kind, D, MT,
// batch): a per-thread memo in front of the process-wide map.
using OccKey = std::tuple<int, int, int, int, int>;
template <typename F>
int cached_occupancy(const OccKey& key, F&& query) {
    constexpr int kMemo = 16;
    thread_local OccKey memo_key[kMemo];
    thread_local int memo_val[kMemo];
    thread_local int memo_n = 0, memo_next = 0;
    for (int i = 0; i < memo_n; ++i)
        if (memo_key[i] == key) return memo_val[i];
    int v;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occupancy.find(key);
        if (it == g_occupancy.end()) {
            v = query();
            g_occupancy[key] = v;
        } else {
            v = it->second;
        }
    }
    const int slot = memo_n < kMemo ? memo_n++ : (memo_next++ % kMemo);
    memo_key[slot] = key;
    memo_val[slot] = v;
    return v;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Per-thread memo of encoded 2-D tensor maps.  An encoded map is a pure
// function of its encode arguments, so a hit returns the bytes the driver
// would produce again; a decode loop that passes the same buffers every step
// encodes each of its maps once per thread.
struct MapKey {
    const void* base;
    uint64_t rows, cols, stride;
    uint32_t box_cols, box_rows;
    int32_t swz, dt;
};
struct MapMemo {
    MapKey key;
    CUtensorMap map;
};
constexpr int kMapMemo = 32;
thread_local MapMemo t_maps[kMapMemo];
thread_local int t_maps_n = 0, t_maps_next = 0;

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box of
// box_cols x box_rows elements, given swizzle.
kvdec_status encode_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                       CUtensorMapSwizzle swz,
                       CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    MapKey key;
    memset(&key, 0, sizeof(key));
    key.base = base;
    key.rows = rows;
    key.cols = cols;
    key.stride = row_stride_bytes;
    key.box_cols = box_cols;
    key.box_rows = box_rows;
    key.swz = (int32_t)swz;
    key.dt = (int32_t)dt;
    for (int i = 0; i < t_maps_n; ++i)
        if (memcmp(&t_maps[i].key, &key, sizeof(key)) == 0) {
            *map = t_maps[i].map;
            return KVDEC_OK;
        }
    auto enc = tensor_map_encoder();
    if (!enc) return fail(KVDEC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVDEC_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    MapMemo& slot = t_maps[t_maps_n < kMapMemo ? t_maps_n++ : (t_maps_next++ % kMapMemo)];
    slot.key = key;
    slot.map = *map;
    return KVDEC_OK;
}

// 3-D bf16 tensor map over [d2][d1][d0] (d0 innermost), 128-byte swizzle.
kvdec_status encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                       uint32_t box2) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(KVDEC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVDEC_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
    return KVDEC_OK;
}

// ---------------------------------------------------------------- GQA layout

struct GqaPlan {
    int D, MT, g, n_hc, hc_rows, units;
    bool f8, dense;
    int grid;
    size_t off_lse, off_o, bytes;
};

constexpr int kMaxBatch = 8192;

// Call epoch for the split-piece counters (see arrive_piece): kept in
// [1, 2^23) so that a counter word never looks like a normal float pair.
uint32_t next_epoch() {
    static std::atomic<uint32_t> e{0};
    return (e.fetch_add(1, std::memory_order_relaxed) % ((1u << 23) - 1u)) + 1u;
}

kvdec_status plan_gqa(const kvdec_gqa_params* p, GqaPlan& pl) {
    if (!p) return fail(KVDEC_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->batch > kMaxBatch)
        return fail(KVDEC_ERR_INVALID_ARG, "batch %d outside [1, %d]", p->batch, kMaxBatch);
    if (p->num_heads < 1 || p->num_kv_heads < 1 || p->num_heads % p->num_kv_heads)
        return fail(KVDEC_ERR_INVALID_ARG, "num_heads %d must be a positive multiple of num_kv_heads %d",
                    p->num_heads, p->num_kv_heads);
    if (p->head_dim != 64 && p->head_dim != 128)
        return fail(KVDEC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", p->head_dim);
    if (p->kv_format != KVDEC_KV_BF16 && p->kv_format != KVDEC_KV_FP8_E4M3)
        return fail(KVDEC_ERR_INVALID_ARG, "kv_format %d", p->kv_format);
    pl.f8 = p->kv_format == KVDEC_KV_FP8_E4M3;
    if (pl.f8 && p->head_dim != 128)
        return fail(KVDEC_ERR_UNSUPPORTED, "FP8 cache with head_dim %d (supported: 128)", p->head_dim);
    if (p->window < 0) return fail(KVDEC_ERR_INVALID_ARG, "window %d", p->window);
    pl.D = p->head_dim;
    pl.g = p->num_heads / p->num_kv_heads;
    DeviceInfo di;
    int dev;
    if (!device_info(di, dev)) return fail(KVDEC_ERR_CUDA, "no current CUDA device");
    // Head chunks of up to 32 rows.  With more than 16 heads per KV head and
    // fewer (sequence, KV head) units than SMs (MQA-like shapes at small
    // batch), chunks of 16 double the CTAs at work and halve each tile's MMA
    // work; the sibling chunk reads the same K/V tiles, from L2.
    pl.hc_rows = pl.g <= 32 ? pl.g : 32;
    if (pl.g > 16 && (long long)p->batch * p->num_kv_heads * ((pl.g + 31) / 32) < di.sm_count) pl.hc_rows = 16;
    pl.n_hc = (pl.g + pl.hc_rows - 1) / pl.hc_rows;
    // row tiles of 16 head rows; an FP8 cache with at most 8 rows per chunk
    // takes the transposed form (the rows as the MMA's 8 columns)
    pl.MT = pl.hc_rows > 16 ? 2 : (pl.f8 && pl.hc_rows <= 8) ? 0 : 1;
    pl.units = p->batch * p->num_kv_heads * pl.n_hc;
    int occ = cached_occupancy(std::make_tuple(dev, pl.f8 ? 2 : 0, pl.D, pl.MT, p->batch),
                               [&] { return kvdec::occupancy_gqa(pl.D, pl.MT, pl.f8, false, p->batch); });
    if (occ < 1) return fail(KVDEC_ERR_CUDA, "GQA kernel does not fit on this device");
    // The transposed FP8 form runs three CTAs per SM when the cache holds at
    // most 256 tiles per SM (short contexts: the kernel's start and tail weigh
    // most there); longer caches stream better through two CTAs of six stages.
    pl.dense = false;
    if (pl.MT == 0) {
        long long slots = p->block_table ? (long long)p->max_blocks * KVDEC_PAGE_SIZE : p->capacity;
        if (p->window > 0 && p->window < slots) slots = p->window;
        const long long max_tiles =
            (long long)pl.units * ((std::max(slots, 0ll) + KVDEC_PAGE_SIZE - 1) / KVDEC_PAGE_SIZE);
        if (max_tiles <= 256ll * di.sm_count) {
            const int occ3 = cached_occupancy(std::make_tuple(dev, 3, pl.D, pl.MT, p->batch), [&] {
                return kvdec::occupancy_gqa(pl.D, pl.MT, pl.f8, true, p->batch);
            });
            if (occ3 >= 3) {
                pl.dense = true;
                occ = occ3;
            }
        }
    }
    pl.grid = di.sm_count * occ;
    // max_ctas > 0 sets the number of work items (CTAs); above one resident
    // wave the hardware hands the equal-size items out as SMs free up.
    if (p->max_ctas > 0) pl.grid = std::min(p->max_ctas, 64 * di.sm_count * occ);
    const size_t slots = 2 * (size_t)pl.grid;
    pl.off_lse = round_up((size_t)pl.units * 8, 256);
    pl.off_o = pl.off_lse + round_up(slots * pl.hc_rows * 4, 256);
    pl.bytes = pl.off_o + slots * pl.hc_rows * pl.D * 4;
    return KVDEC_OK;
}

// The kernels take the row max before scaling, so the scale must be positive.
bool scale_ok(float s) { return s == 0.f || (s > 0.f && std::isfinite(s)); }

// ---------------------------------------------------------------- MLA layout

struct MlaPlan {
    int pairs;
    size_t off_lse, off_o, bytes;
    // E4M3 cache: the widened bf16 copy of the pages the call reads and its
    // identity block table (mla_widen.cu)
    size_t off_table, off_copy;
};

kvdec_status plan_mla(const kvdec_mla_params* p, MlaPlan& pl) {
    if (!p) return fail(KVDEC_ERR_INVALID_ARG, "params is NULL");
    if (p->num_heads != 128)
        return fail(KVDEC_ERR_UNSUPPORTED, "num_heads %d (the MLA kernel is built for 128)", p->num_heads);
    if (p->batch < 1 || p->batch > kvdec::max_batch_mla())
        return fail(KVDEC_ERR_INVALID_ARG, "batch %d outside [1, %d]", p->batch, kvdec::max_batch_mla());
    if (p->num_pages < 1 || p->max_blocks < 1)
        return fail(KVDEC_ERR_INVALID_ARG, "num_pages and max_blocks must be >= 1");
    if (p->kv_format != KVDEC_KV_BF16 && p->kv_format != KVDEC_KV_FP8_E4M3)
        return fail(KVDEC_ERR_INVALID_ARG, "kv_format %d", p->kv_format);
    DeviceInfo di;
    int dev;
    if (!device_info(di, dev)) return fail(KVDEC_ERR_CUDA, "no current CUDA device");
    int pairs = cached_occupancy(std::make_tuple(dev, 1, 0, 0, p->batch),
                                 [&] { return kvdec::max_pairs_mla(p->batch); });
    if (pairs < 1) return fail(KVDEC_ERR_CUDA, "MLA kernel clusters do not fit on this device");
    if (p->max_ctas > 0) pairs = std::min(std::max(1, p->max_ctas / 2), 64 * pairs);
    pl.pairs = pairs;
    const size_t slots = 2 * (size_t)pairs;
    pl.off_lse = round_up((size_t)p->batch * 2 * 4 * 8, 256);
    pl.off_o = pl.off_lse + round_up(2 * slots * 128 * 4, 256);
    pl.bytes = pl.off_o + slots * 128 * 512 * 4;
    pl.off_table = pl.off_copy = 0;
    if (p->kv_format == KVDEC_KV_FP8_E4M3) {
        const size_t copy_pages = (size_t)p->batch * p->max_blocks;
        pl.off_table = round_up(pl.bytes, 256);
        pl.off_copy = round_up(pl.off_table + copy_pages * 4, 256);
        pl.bytes = pl.off_copy + copy_pages * KVDEC_PAGE_SIZE * 576 * 2;
    }
    return KVDEC_OK;
}

}  // namespace

namespace kvdec {
// Lets other translation units of the library set the kvdec_last_error text.
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace kvdec

extern "C" {

int kvdec_abi_version(void) { return KVDEC_ABI_VERSION; }

int32_t kvdec_mla_max_batch(void) { return kvdec::max_batch_mla(); }

int64_t kvdec_params_size(int kind) {
    switch (kind) {
        case 0: return (int64_t)sizeof(kvdec_gqa_params);
        case 1: return (int64_t)sizeof(kvdec_mla_params);
        case 2: return (int64_t)sizeof(kvdec_append_params);
        case 3: return (int64_t)sizeof(kvdec_combine_params);
        case 4: return (int64_t)sizeof(kvdec_mla_proj_params);
        case 5: return (int64_t)sizeof(kvdec_mla_expand_params);
        case 6: return (int64_t)sizeof(kvdec_mla_prefill_params);
        default: return -1;
    }
}

const char* kvdec_status_string(kvdec_status s) {
    switch (s) {
        case KVDEC_OK: return "ok";
        case KVDEC_ERR_INVALID_ARG: return "invalid argument";
        case KVDEC_ERR_UNSUPPORTED: return "unsupported";
        case KVDEC_ERR_CUDA: return "CUDA error";
        case KVDEC_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

const char* kvdec_last_error(void) { return g_last_error.c_str(); }

size_t kvdec_gqa_workspace_bytes(const kvdec_gqa_params* p) {
    GqaPlan pl;
    if (plan_gqa(p, pl) != KVDEC_OK) return 0;
    return pl.bytes;
}

kvdec_status kvdec_gqa_decode(const kvdec_gqa_params* p, void* stream) {
    GqaPlan pl;
    kvdec_status st = plan_gqa(p, pl);
    if (st != KVDEC_OK) return st;
    if (!p->q || !p->k || !p->v || !p->seqlens || !p->out)
        return fail(KVDEC_ERR_INVALID_ARG, "q, k, v, seqlens and out must be non-NULL");
    if (!aligned(p->q, 16) || !aligned(p->k, 16) || !aligned(p->v, 16) || !aligned(p->out, 16))
        return fail(KVDEC_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
    if (!aligned(p->seqlens, 4) || (p->lse && !aligned(p->lse, 4)))
        return fail(KVDEC_ERR_INVALID_ARG, "seqlens and lse must be 4-byte aligned");
    if (p->out_dtype != KVDEC_F32 && p->out_dtype != KVDEC_BF16)
        return fail(KVDEC_ERR_INVALID_ARG, "out_dtype %d", p->out_dtype);
    if (!p->workspace || !aligned(p->workspace, 256))
        return fail(KVDEC_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
    if (p->workspace_bytes < pl.bytes)
        return fail(KVDEC_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", p->workspace_bytes,
                    pl.bytes);
    const bool paged = p->block_table != nullptr;
    uint64_t rows;
    int cap;
    if (paged) {
        if (p->num_pages < 1 || p->max_blocks < 1)
            return fail(KVDEC_ERR_INVALID_ARG, "paged cache needs num_pages >= 1 and max_blocks >= 1");
        if (!aligned(p->block_table, 4)) return fail(KVDEC_ERR_INVALID_ARG, "block_table alignment");
        rows = (uint64_t)p->num_pages * p->num_kv_heads * KVDEC_PAGE_SIZE;
        if ((uint64_t)p->max_blocks * KVDEC_PAGE_SIZE > 0x7fffffffull)
            return fail(KVDEC_ERR_INVALID_ARG, "max_blocks too large");
        cap = p->max_blocks * KVDEC_PAGE_SIZE;
    } else {
        if (p->capacity < 1) return fail(KVDEC_ERR_INVALID_ARG, "capacity must be >= 1");
        rows = (uint64_t)p->batch * p->num_kv_heads * p->capacity;
        cap = p->capacity;
    }
    if (rows + KVDEC_PAGE_SIZE >= 0x7fffffffull)
        return fail(KVDEC_ERR_UNSUPPORTED, "cache has %llu rows (limit 2^31 - 64)",
                    (unsigned long long)rows);
    if (p->window > cap)
        return fail(KVDEC_ERR_INVALID_ARG, "window %d exceeds the %d cache slots", p->window, cap);
    if (pl.f8 && (!p->k_scale || !p->v_scale || !aligned(p->k_scale, 4) || !aligned(p->v_scale, 4)))
        return fail(KVDEC_ERR_INVALID_ARG, "an FP8 cache needs 4-byte aligned k_scale and v_scale");
    CUtensorMap tk, tv;
    if (pl.f8) {
        // one byte per element: a 64-token box of 128-byte rows
        st = encode_2d(&tk, p->k, rows, pl.D, (uint64_t)pl.D, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_DATA_TYPE_UINT8);
        if (st != KVDEC_OK) return st;
        st = encode_2d(&tv, p->v, rows, pl.D, (uint64_t)pl.D, 128, 64, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_DATA_TYPE_UINT8);
    } else {
        st = encode_2d(&tk, p->k, rows, pl.D, (uint64_t)pl.D * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != KVDEC_OK) return st;
        st = encode_2d(&tv, p->v, rows, pl.D, (uint64_t)pl.D * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (st != KVDEC_OK) return st;

    kvdec::GqaArgs a;
    memset(&a, 0, sizeof(a));
    a.q = static_cast<const __nv_bfloat16*>(p->q);
    a.block_table = p->block_table;
    a.seqlens = p->seqlens;
    a.out = p->out;
    a.lse = p->lse;
    uint8_t* ws = static_cast<uint8_t*>(p->workspace);
    a.counters = reinterpret_cast<unsigned long long*>(ws);
    a.epoch = next_epoch();
    a.part_lse = reinterpret_cast<float*>(ws + pl.off_lse);
    a.part_o = reinterpret_cast<float*>(ws + pl.off_o);
    a.err = p->error_flag;
    a.B = p->batch;
    a.H = p->num_heads;
    a.n_kv = p->num_kv_heads;
    a.g = pl.g;
    a.n_hc = pl.n_hc;
    a.hc_rows = pl.hc_rows;
    a.cap = cap;
    a.paged = paged ? 1 : 0;
    a.num_pages = p->num_pages;
    a.max_blocks = p->max_blocks;
    a.out_bf16 = p->out_dtype == KVDEC_BF16;
    if (!scale_ok(p->scale)) return fail(KVDEC_ERR_INVALID_ARG, "scale %g (must be 0 or positive and finite)", (double)p->scale);
    const double scale = p->scale != 0.f ? (double)p->scale : 1.0 / std::sqrt((double)pl.D);
    a.scale_log2 = (float)(scale * 1.4426950408889634);
    a.min_tiles = 8;
    a.timeout_ns = kvdec::kDefaultTimeoutNs;
    a.k_scale = p->k_scale;
    a.v_scale = p->v_scale;
    a.window = p->window;
    cudaError_t e = kvdec::launch_gqa(pl.D, pl.MT, pl.f8, pl.dense, tk, tv, a, pl.grid,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "GQA decode launch");
    return KVDEC_OK;
}


size_t kvdec_mla_workspace_bytes(const kvdec_mla_params* p) {
    MlaPlan pl;
    if (plan_mla(p, pl) != KVDEC_OK) return 0;
    return pl.bytes;
}

kvdec_status kvdec_mla_decode_absorbed(const kvdec_mla_params* p, void* stream) {
    MlaPlan pl;
    kvdec_status st = plan_mla(p, pl);
    if (st != KVDEC_OK) return st;
    if (!p->q_absorbed || !p->q_rope || !p->cache || !p->block_table || !p->seqlens || !p->out)
        return fail(KVDEC_ERR_INVALID_ARG,
                    "q_absorbed, q_rope, cache, block_table, seqlens and out must be non-NULL");
    if (!aligned(p->q_absorbed, 16) || !aligned(p->q_rope, 16) || !aligned(p->cache, 16) ||
        !aligned(p->out, 16))
        return fail(KVDEC_ERR_INVALID_ARG, "q_absorbed, q_rope, cache and out must be 16-byte aligned");
    if (!aligned(p->block_table, 4) || !aligned(p->seqlens, 4) || (p->lse && !aligned(p->lse, 4)))
        return fail(KVDEC_ERR_INVALID_ARG, "block_table, seqlens and lse must be 4-byte aligned");
    if (p->out_dtype != KVDEC_F32 && p->out_dtype != KVDEC_BF16)
        return fail(KVDEC_ERR_INVALID_ARG, "out_dtype %d", p->out_dtype);
    if (!p->workspace || !aligned(p->workspace, 256))
        return fail(KVDEC_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
    if (p->workspace_bytes < pl.bytes)
        return fail(KVDEC_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", p->workspace_bytes,
                    pl.bytes);
    const uint64_t rows = (uint64_t)p->num_pages * KVDEC_PAGE_SIZE;
    if (rows >= 0x7fffffffull || (uint64_t)p->max_blocks * KVDEC_PAGE_SIZE >= 0x7fffffffull)
        return fail(KVDEC_ERR_UNSUPPORTED, "cache too large (rows >= 2^31)");
    if (!scale_ok(p->scale)) return fail(KVDEC_ERR_INVALID_ARG, "scale %g (must be 0 or positive and finite)", (double)p->scale);
    uint8_t* ws = static_cast<uint8_t*>(p->workspace);
    // E4M3 cache: widen the pages this call reads into the workspace's bf16
    // copy, then decode the copy through its identity block table
    const bool fp8 = p->kv_format == KVDEC_KV_FP8_E4M3;
    const void* cache = p->cache;
    const int32_t* block_table = p->block_table;
    int num_pages = p->num_pages;
    if (fp8) {
        if (!p->kv_scale || !aligned(p->kv_scale, 4))
            return fail(KVDEC_ERR_INVALID_ARG, "an E4M3 latent cache needs kv_scale = fp32 [c_kv scale, k_R scale]");
        const uint64_t copy_rows = (uint64_t)p->batch * p->max_blocks * KVDEC_PAGE_SIZE;
        if (copy_rows >= 0x7fffffffull)
            return fail(KVDEC_ERR_UNSUPPORTED, "batch * max_blocks * 64 >= 2^31 (split the call)");
        kvdec::MlaWidenArgs w;
        w.codes = static_cast<const uint8_t*>(p->cache);
        w.block_table = p->block_table;
        w.seqlens = p->seqlens;
        w.kv_scale = p->kv_scale;
        w.copy = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_copy);
        w.copy_table = reinterpret_cast<int32_t*>(ws + pl.off_table);
        w.B = p->batch;
        w.num_pages = p->num_pages;
        w.max_blocks = p->max_blocks;
        w.err = p->error_flag;
        cudaError_t e = kvdec::launch_mla_widen(w, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "MLA widening launch");
        cache = w.copy;
        block_table = w.copy_table;
        num_pages = p->batch * p->max_blocks;
    }
    const uint64_t crows = (uint64_t)num_pages * KVDEC_PAGE_SIZE;
    kvdec::MlaMaps maps;
    if ((st = encode_2d(&maps.c128, cache, crows, 576, 1152, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))) return st;
    if ((st = encode_2d(&maps.c64, cache, crows, 576, 1152, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B))) return st;
    // stores of O / l, 32 rows x 32 fp32 columns per box: partials, and out when it is fp32
    if ((st = encode_2d(&maps.part, static_cast<uint8_t*>(p->workspace) + pl.off_o, 2 * (uint64_t)pl.pairs * 128, 512,
                        2048, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32)))
        return st;
    maps.outf = maps.part;
    if (p->out_dtype == KVDEC_F32 &&
        (st = encode_2d(&maps.outf, p->out, (uint64_t)p->batch * 128, 512, 2048, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_DATA_TYPE_FLOAT32)))
        return st;
    kvdec::MlaArgs a;
    memset(&a, 0, sizeof(a));
    a.q_abs = static_cast<const __nv_bfloat16*>(p->q_absorbed);
    a.q_rope = static_cast<const __nv_bfloat16*>(p->q_rope);
    a.block_table = block_table;
    a.seqlens = p->seqlens;
    a.out = p->out;
    a.lse = p->lse;
    a.counters = reinterpret_cast<unsigned long long*>(ws);
    a.part_lse = reinterpret_cast<float*>(ws + pl.off_lse);
    a.part_o = reinterpret_cast<float*>(ws + pl.off_o);
    a.epoch = next_epoch();
    a.err = p->error_flag;
    a.B = p->batch;
    a.num_pages = num_pages;
    a.max_blocks = p->max_blocks;
    a.out_bf16 = p->out_dtype == KVDEC_BF16;
    const double scale = p->scale != 0.f ? (double)p->scale : 1.0 / std::sqrt(192.0);
    a.scale_log2 = (float)(scale * 1.4426950408889634);
    a.min_tiles = 4;
    a.seg_cost = kvdec::kMlaSeqStartCost;
    a.timeout_ns = kvdec::kDefaultTimeoutNs;
    cudaError_t e = kvdec::launch_mla(maps, a, pl.pairs, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "MLA decode launch");
    return KVDEC_OK;
}

static kvdec_status mla_proj(const kvdec_mla_proj_params* p, void* stream, bool absorb) {
    const char* name = absorb ? "kvdec_mla_absorb_q" : "kvdec_mla_project_out";
    if (!p) return fail(KVDEC_ERR_INVALID_ARG, "%s: params is NULL", name);
    if (!p->x || !p->w || !p->y) return fail(KVDEC_ERR_INVALID_ARG, "%s: x, w and y must be non-NULL", name);
    if (!aligned(p->x, 16) || !aligned(p->w, 16) || !aligned(p->y, 16))
        return fail(KVDEC_ERR_INVALID_ARG, "%s: x, w and y must be 16-byte aligned", name);
    if (p->batch < 1 || p->batch > (1 << 20) || p->num_heads < 1 || p->num_heads > 65535)
        return fail(KVDEC_ERR_INVALID_ARG, "%s: batch %d, num_heads %d", name, p->batch, p->num_heads);
    if (p->out_dtype != KVDEC_F32 && p->out_dtype != KVDEC_BF16)
        return fail(KVDEC_ERR_INVALID_ARG, "%s: out_dtype %d", name, p->out_dtype);
    kvdec::MlaProjArgs a;
    a.x = static_cast<const __nv_bfloat16*>(p->x);
    a.w = static_cast<const __nv_bfloat16*>(p->w);
    a.y = p->y;
    a.batch = p->batch;
    a.num_heads = p->num_heads;
    a.out_bf16 = p->out_dtype == KVDEC_BF16;
    a.x_shared = 0;
    cudaError_t e = kvdec::launch_mla_proj(absorb, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, name);
    return KVDEC_OK;
}

kvdec_status kvdec_mla_absorb_q(const kvdec_mla_proj_params* p, void* stream) { return mla_proj(p, stream, true); }

kvdec_status kvdec_mla_project_out(const kvdec_mla_proj_params* p, void* stream) {
    return mla_proj(p, stream, false);
}

kvdec_status kvdec_mla_prefill_expand(const kvdec_mla_expand_params* p, void* stream) {
    const char* name = "kvdec_mla_prefill_expand";
    if (!p) return fail(KVDEC_ERR_INVALID_ARG, "%s: params is NULL", name);
    if (!p->c_kv || !p->w_uk || !p->w_uv || !p->k_nope || !p->v)
        return fail(KVDEC_ERR_INVALID_ARG, "%s: c_kv, w_uk, w_uv, k_nope and v must be non-NULL", name);
    if (!aligned(p->c_kv, 16) || !aligned(p->w_uk, 16) || !aligned(p->w_uv, 16) || !aligned(p->k_nope, 16) ||
        !aligned(p->v, 16))
        return fail(KVDEC_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", name);
    if (p->s < 1 || p->s > (1 << 20) || p->num_heads < 1 || p->num_heads > 65535)
        return fail(KVDEC_ERR_INVALID_ARG, "%s: s %d, num_heads %d", name, p->s, p->num_heads);
    if (p->num_heads % 2 == 0) {
        // tcgen05 GEMM: D [s, n_h 128] = c_kv [s, 512] . W^T, W as [n_h 128, 512]
        const uint64_t N = (uint64_t)p->num_heads * 128;
        kvdec::MlaExpandMaps maps;
        kvdec_status st;
        if ((st = encode_2d(&maps.c, p->c_kv, p->s, 512, 1024, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) != KVDEC_OK)
            return st;
        if ((st = encode_2d(&maps.wk, p->w_uk, N, 512, 1024, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B)) != KVDEC_OK)
            return st;
        if ((st = encode_2d(&maps.wv, p->w_uv, N, 512, 1024, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B)) != KVDEC_OK)
            return st;
        kvdec::MlaExpandArgs e;
        e.k_nope = static_cast<__nv_bfloat16*>(p->k_nope);
        e.v = static_cast<__nv_bfloat16*>(p->v);
        e.s = p->s;
        e.N = (int)N;
        e.err = nullptr;
        e.timeout_ns = kvdec::kDefaultTimeoutNs;
        cudaError_t ce = kvdec::launch_mla_expand_tc(maps, e, static_cast<cudaStream_t>(stream));
        if (ce != cudaSuccess) return cuda_fail(ce, name);
        return KVDEC_OK;
    }
    // an odd head count: the per-head projection kernel, every head reading the same rows
    kvdec::MlaProjArgs a;
    a.x = static_cast<const __nv_bfloat16*>(p->c_kv);
    a.batch = p->s;
    a.num_heads = p->num_heads;
    a.out_bf16 = 1;
    a.x_shared = 1;
    a.w = static_cast<const __nv_bfloat16*>(p->w_uk);
    a.y = p->k_nope;
    cudaError_t e = kvdec::launch_mla_proj(false, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, name);
    a.w = static_cast<const __nv_bfloat16*>(p->w_uv);
    a.y = p->v;
    e = kvdec::launch_mla_proj(false, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, name);
    return KVDEC_OK;
}

kvdec_status kvdec_mla_prefill(const kvdec_mla_prefill_params* p, void* stream) {
    const char* name = "kvdec_mla_prefill";
    if (!p) return fail(KVDEC_ERR_INVALID_ARG, "%s: params is NULL", name);
    if (!p->q_nope || !p->q_rope || !p->k_nope || !p->k_rope || !p->v || !p->out)
        return fail(KVDEC_ERR_INVALID_ARG, "%s: q_nope, q_rope, k_nope, k_rope, v and out must be non-NULL", name);
    if (!aligned(p->q_nope, 16) || !aligned(p->q_rope, 16) || !aligned(p->k_nope, 16) || !aligned(p->k_rope, 16) ||
        !aligned(p->v, 16) || !aligned(p->out, 16) || (p->lse && !aligned(p->lse, 4)))
        return fail(KVDEC_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", name);
    if (p->s_q < 1 || p->s_kv < 1 || p->s_kv > (1 << 24) || p->num_heads < 1 || p->num_heads > 65535)
        return fail(KVDEC_ERR_INVALID_ARG, "%s: s_q %d, s_kv %d, num_heads %d", name, p->s_q, p->s_kv, p->num_heads);
    const int off = p->kv_offset < 0 ? p->s_kv - p->s_q : p->kv_offset;
    if (off < 0 || (int64_t)off + p->s_q > p->s_kv)
        return fail(KVDEC_ERR_INVALID_ARG, "%s: queries at positions %d..%d need s_kv %d >= that", name, off,
                    off + p->s_q - 1, p->s_kv);
    if (p->out_dtype != KVDEC_F32 && p->out_dtype != KVDEC_BF16)
        return fail(KVDEC_ERR_INVALID_ARG, "%s: out_dtype %d", name, p->out_dtype);
    if (!scale_ok(p->scale)) return fail(KVDEC_ERR_INVALID_ARG, "%s: scale %g", name, (double)p->scale);
    kvdec::MlaPrefillArgs a;
    a.q_nope = static_cast<const __nv_bfloat16*>(p->q_nope);
    a.q_rope = static_cast<const __nv_bfloat16*>(p->q_rope);
    a.k_nope = static_cast<const __nv_bfloat16*>(p->k_nope);
    a.k_rope = static_cast<const __nv_bfloat16*>(p->k_rope);
    a.v = static_cast<const __nv_bfloat16*>(p->v);
    a.out = p->out;
    a.lse = p->lse;
    a.s_q = p->s_q;
    a.s_kv = p->s_kv;
    a.num_heads = p->num_heads;
    a.kv_offset = off;
    a.out_bf16 = p->out_dtype == KVDEC_BF16;
    const double scale = p->scale != 0.f ? (double)p->scale : 1.0 / std::sqrt(192.0);
    a.scale_log2 = (float)(scale * 1.4426950408889634);
    a.err = nullptr;
    a.timeout_ns = kvdec::kDefaultTimeoutNs;
    // tensor maps: [tokens][heads][dims] for q and the up-projected k, v;
    // boxes of 64 dims x 1 head x (128 query | 64 key) tokens
    const uint64_t H = (uint64_t)p->num_heads;
    kvdec::MlaPrefillMaps maps;
    kvdec_status st;
    if ((st = encode_3d(&maps.qn, p->q_nope, 128, H, p->s_q, 256, H * 256, 64, 1, 128)) != KVDEC_OK) return st;
    if ((st = encode_3d(&maps.qr, p->q_rope, 64, H, p->s_q, 128, H * 128, 64, 1, 128)) != KVDEC_OK) return st;
    if ((st = encode_3d(&maps.kn, p->k_nope, 128, H, p->s_kv, 256, H * 256, 64, 1, 64)) != KVDEC_OK) return st;
    if ((st = encode_3d(&maps.v, p->v, 128, H, p->s_kv, 256, H * 256, 64, 1, 64)) != KVDEC_OK) return st;
    if ((st = encode_2d(&maps.kr, p->k_rope, p->s_kv, 64, 128, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != KVDEC_OK)
        return st;
    cudaError_t e = kvdec::launch_mla_prefill_tc(maps, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, name);
    return KVDEC_OK;
}

kvdec_status kvdec_combine_splits(const kvdec_combine_params* p, void* stream) {
    if (!p) return fail(KVDEC_ERR_INVALID_ARG, "params is NULL");
    if (!p->partial_o || !p->partial_lse || !p->out)
        return fail(KVDEC_ERR_INVALID_ARG, "partial_o, partial_lse and out must be non-NULL");
    if (p->num_splits < 1 || p->rows < 1)
        return fail(KVDEC_ERR_INVALID_ARG, "num_splits and rows must be >= 1");
    if (p->head_dim < 4 || p->head_dim % 4 || p->head_dim > 1024)
        return fail(KVDEC_ERR_UNSUPPORTED, "head_dim %d (multiple of 4, <= 1024)", p->head_dim);
    if (!aligned(p->partial_o, 16) || !aligned(p->out, 16))
        return fail(KVDEC_ERR_INVALID_ARG, "partial_o and out must be 16-byte aligned");
    if (p->out_dtype != KVDEC_F32 && p->out_dtype != KVDEC_BF16)
        return fail(KVDEC_ERR_INVALID_ARG, "out_dtype %d", p->out_dtype);
    kvdec::CombineArgs a;
    a.po = p->partial_o;
    a.plse = p->partial_lse;
    a.counts = p->split_counts;
    a.out = p->out;
    a.lse = p->lse;
    a.S = p->num_splits;
    a.rows = p->rows;
    a.D = p->head_dim;
    a.out_bf16 = p->out_dtype == KVDEC_BF16;
    cudaError_t e = kvdec::launch_combine(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    return KVDEC_OK;
}

kvdec_status kvdec_append_rope(const kvdec_append_params* p, void* stream) {
    if (!p) return fail(KVDEC_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1) return fail(KVDEC_ERR_INVALID_ARG, "batch must be >= 1");
    if (!p->seqlens) return fail(KVDEC_ERR_INVALID_ARG, "seqlens is NULL");
    kvdec::AppendArgs a;
    memset(&a, 0, sizeof(a));
    a.B = p->batch;
    a.seqlens = p->seqlens;
    a.block_table = p->block_table;
    a.num_pages = p->num_pages;
    a.max_blocks = p->max_blocks;
    a.err = p->error_flag;
    if (p->block_table && (p->num_pages < 1 || p->max_blocks < 1))
        return fail(KVDEC_ERR_INVALID_ARG, "paged append needs num_pages >= 1 and max_blocks >= 1");
    if (p->mode == KVDEC_APPEND_MLA) {
        if (p->window != 0) return fail(KVDEC_ERR_UNSUPPORTED, "MLA append takes no window");
        if (p->kv_format != KVDEC_KV_BF16 && p->kv_format != KVDEC_KV_FP8_E4M3)
            return fail(KVDEC_ERR_INVALID_ARG, "kv_format %d", p->kv_format);
        if (!p->block_table || !p->c_kv || !p->k_rope || !p->cache)
            return fail(KVDEC_ERR_INVALID_ARG, "MLA append needs block_table, c_kv, k_rope and cache");
        if (!aligned(p->c_kv, 16) || !aligned(p->cache, 16) || !aligned(p->k_rope, 4))
            return fail(KVDEC_ERR_INVALID_ARG, "c_kv and cache must be 16-byte aligned");
        a.mode = 0;
        a.fp8 = p->kv_format == KVDEC_KV_FP8_E4M3;
        if (a.fp8 && (!p->k_scale || !aligned(p->k_scale, 4)))
            return fail(KVDEC_ERR_INVALID_ARG, "an E4M3 latent cache needs k_scale = fp32 [c_kv scale, k_R scale]");
        a.k_scale = p->k_scale;
        a.c_kv = static_cast<const __nv_bfloat16*>(p->c_kv);
        a.k_rope = static_cast<const __nv_bfloat16*>(p->k_rope);
        a.cache = static_cast<__nv_bfloat16*>(p->cache);
    } else if (p->mode == KVDEC_APPEND_GQA) {
        if (!p->k_new || !p->v_new || !p->k || !p->v)
            return fail(KVDEC_ERR_INVALID_ARG, "GQA append needs k_new, v_new, k and v");
        if (p->head_dim != 64 && p->head_dim != 128)
            return fail(KVDEC_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", p->head_dim);
        if (p->num_kv_heads < 1 || p->num_kv_heads > 65535)
            return fail(KVDEC_ERR_INVALID_ARG, "num_kv_heads %d", p->num_kv_heads);
        if (!p->block_table && p->capacity < 1)
            return fail(KVDEC_ERR_INVALID_ARG, "contiguous append needs capacity >= 1");
        if (!aligned(p->v_new, 16) || !aligned(p->v, 16) || !aligned(p->k_new, 4) || !aligned(p->k, 4))
            return fail(KVDEC_ERR_INVALID_ARG, "v_new and v must be 16-byte aligned");
        if (p->kv_format != KVDEC_KV_BF16 && p->kv_format != KVDEC_KV_FP8_E4M3)
            return fail(KVDEC_ERR_INVALID_ARG, "kv_format %d", p->kv_format);
        a.fp8 = p->kv_format == KVDEC_KV_FP8_E4M3;
        if (a.fp8 && (!p->k_scale || !p->v_scale || !aligned(p->k_scale, 4) || !aligned(p->v_scale, 4)))
            return fail(KVDEC_ERR_INVALID_ARG, "an FP8 cache needs 4-byte aligned k_scale and v_scale");
        const int slots = p->block_table ? p->max_blocks * KVDEC_PAGE_SIZE : p->capacity;
        if (p->window < 0 || p->window > slots)
            return fail(KVDEC_ERR_INVALID_ARG, "window %d (must be 0 or at most the %d cache slots)",
                        p->window, slots);
        a.window = p->window;
        a.k_scale = p->k_scale;
        a.v_scale = p->v_scale;
        a.mode = 1;
        a.k_new = static_cast<const __nv_bfloat16*>(p->k_new);
        a.v_new = static_cast<const __nv_bfloat16*>(p->v_new);
        a.k = p->k;
        a.v = p->v;
        a.n_kv = p->num_kv_heads;
        a.d = p->head_dim;
        a.cap = p->capacity;
    } else {
        return fail(KVDEC_ERR_INVALID_ARG, "mode %d", p->mode);
    }
    const double theta = p->rope_theta != 0.f ? (double)p->rope_theta : 10000.0;
    const int rot_dim = p->mode == KVDEC_APPEND_MLA ? KVDEC_MLA_DR : p->head_dim;
    if (rot_dim < 2 || rot_dim > 2 * kvdec::kMaxRopePairs || rot_dim % 2)
        return fail(KVDEC_ERR_UNSUPPORTED, "rotary dim %d", rot_dim);
    for (int i = 0; i < rot_dim / 2; ++i)
        a.inv_freq[i] = std::pow(theta, -2.0 * (double)i / (double)rot_dim);
    cudaError_t e = kvdec::launch_append(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return KVDEC_OK;
}

kvdec_status kvdec_selftest_wait_timeout(uint64_t timeout_ns, uint32_t* error_flag, void* stream) {
    if (!error_flag) return fail(KVDEC_ERR_INVALID_ARG, "error_flag is NULL");
    if (timeout_ns > 10000000000ull) return fail(KVDEC_ERR_INVALID_ARG, "timeout above 10 s");
    cudaError_t e = kvdec::launch_selftest_wait(timeout_ns, error_flag, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return KVDEC_OK;
}

}  // extern "C"
