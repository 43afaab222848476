// host_common.cuh -- host-side helpers shared by the library's translation units:
// the per-device facts and process-wide knobs, TMA tensor-map encoding, and the
// launch helper of one kernel instantiation.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/fp8gemm.h"
#include "gemm_kernel.cuh"

namespace fgh {

using fg::GemmParams;

constexpr int kMaxDevices = 64;
constexpr uint32_t kDefaultWatchdogMs = 2000;

// Process-wide knobs (defined in fp8gemm.cu; see include/fp8gemm.h).
extern std::atomic<int> g_num_sms_override;
extern std::atomic<uint32_t> g_watchdog_ms;
extern std::atomic<int> g_debug_skip_iter;
extern std::atomic<int> g_force_bn;
extern std::atomic<int> g_pdl;  // programmatic dependent launch of the GEMM kernels
extern std::atomic<int> g_force_split;
extern std::atomic<int> g_pair_mode;  // CTA-pair tiles: -1 where they apply, 0 never, 1 whenever allowed
extern std::atomic<int> g_swap_mode;  // swapped operand roles: -1 automatic (never), 0 never, 1 wherever they apply
extern std::atomic<int> g_debug_bad_coord;  // debug build: K iteration whose A load is sent past K (-1: none)

// Per-device facts read once.  `ready` is published with release after the
// other fields are written, and read with acquire, so a thread that sees it
// set also sees the status address and the SM count.
struct DeviceInfo {
    std::atomic<int> ready{0};
    int num_sms = 0;
    uint32_t *status = nullptr;
};
inline fg_status cuda_fail() { return FG_ERR_CUDA; }

// The calling thread's current device: its SM count and status word.
fg_status device_info(DeviceInfo **out);

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Everything a tensor map is encoded from.  The 128-byte map is a pure
// function of these fields (the address is encoded, the memory behind it is
// not read), so a map made once can be reused by any later call with the
// same fields, whatever happened to the memory in between.
struct MapKey {
    const void *base;
    uint64_t dims[3];
    uint64_t strides[2];
    uint32_t box[3];
    int32_t rank, dt, swizzle, pad;
};

// Encoded maps of this thread's recent calls: a small ring searched linearly
// (a call encodes three or four maps; a thread that alternates between a few
// problems finds all of them here).  Per thread, so no lock is taken.
constexpr int kMapCacheSize = 32;
struct MapCache {
    MapKey key[kMapCacheSize];
    CUtensorMap map[kMapCacheSize];
    int used = 0, next = 0;
};

#ifndef FG_TENSOR_MAP_CACHE
#define FG_TENSOR_MAP_CACHE 1
#endif

// Tiled tensor map (rank 2 or 3) over a row-major array: dims[0] innermost,
// strides[i] = bytes between consecutive indices of dimension i+1.
inline bool encode(CUtensorMap *map, CUtensorMapDataType dt, const void *base, int rank, const uint64_t *dims,
                   const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle swizzle) {
    MapKey key;
    std::memset(&key, 0, sizeof(key));
    key.base = base;
    key.rank = rank;
    key.dt = (int32_t)dt;
    key.swizzle = (int32_t)swizzle;
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) key.strides[i] = strides[i];
#if FG_TENSOR_MAP_CACHE
    thread_local MapCache cache;
    for (int i = 0; i < cache.used; ++i) {
        if (std::memcmp(&cache.key[i], &key, sizeof(key)) == 0) {
            *map = cache.map[i];
            return true;
        }
    }
#endif
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[3], st[2];
    cuuint32_t bx[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
    CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void *>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
#if FG_TENSOR_MAP_CACHE
    cache.key[cache.next] = key;
    cache.map[cache.next] = *map;
    cache.next = (cache.next + 1) % kMapCacheSize;
    if (cache.used < kMapCacheSize) ++cache.used;
#endif
    return true;
}

inline bool encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    const uint64_t dims[2] = {inner, outer};
    const uint64_t strides[1] = {row_bytes};
    const uint32_t box[2] = {box_inner, box_outer};
    return encode(map, dt, base, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// LHS scales, MN-major: 2-D {rows, kb} with row pitch ld (dense, contiguous) or
// 3-D {M_cap, kb, G} (masked); each load brings the 128 scales of one K block.
inline bool encode_scales_a(CUtensorMap *map, const float *sA, int ld, int rows, int kb, int groups, bool masked) {
    const uint64_t dims[3] = {(uint64_t)rows, (uint64_t)kb, (uint64_t)groups};
    const uint64_t strides[2] = {(uint64_t)ld * 4, (uint64_t)ld * 4 * (uint64_t)kb};
    const uint32_t box[3] = {(uint32_t)fg::BLOCK_M, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sA, masked ? 3 : 2, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }


// Launch helper of one kernel instantiation F with BYTES of dynamic shared
// memory; CLUSTERED kernels always carry a cluster dimension.
template <auto F, int BYTES, bool CLUSTERED, int THREADS = fg::NUM_THREADS>
struct Launcher {
    // launch configuration: a cluster dimension and/or programmatic dependent
    // launch (`at` holds room for two attributes)
    static cudaLaunchConfig_t config(int grid, int cluster, cudaStream_t stream, cudaLaunchAttribute *at,
                                     bool pdl = false) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(grid, 1, 1);
        cfg.blockDim = dim3(THREADS, 1, 1);
        cfg.dynamicSmemBytes = BYTES;
        cfg.stream = stream;
        unsigned n = 0;
        if (cluster > 1 || CLUSTERED) {
            at[n].id = cudaLaunchAttributeClusterDimension;
            at[n].val.clusterDim.x = cluster;
            at[n].val.clusterDim.y = 1;
            at[n].val.clusterDim.z = 1;
            ++n;
        }
        if (pdl) {
            at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            at[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        cfg.attrs = at;
        cfg.numAttrs = n;
        return cfg;
    }

    // dynamic shared memory attribute, once per device
    static bool configure() {
        static std::atomic<uint64_t> configured{0};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return false;
        const uint64_t bit = 1ull << (dev & 63);
        if (configured.load(std::memory_order_acquire) & bit) return true;
        if (cudaFuncSetAttribute(F, cudaFuncAttributeMaxDynamicSharedMemorySize, BYTES) != cudaSuccess)
            return false;
        configured.fetch_or(bit, std::memory_order_acq_rel);
        return true;
    }

    // clusters of `cluster` CTAs that can be resident at once (one wave)
    static int max_active_clusters(int cluster) {
        static std::atomic<int> cache[kMaxDevices][9];
        int dev = 0;
        if (cluster < 1 || cluster > 8 || cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices) return 0;
        const int v = cache[dev][cluster].load();
        if (v > 0) return v;
        if (!configure()) return 0;
        cudaLaunchAttribute at[2];
        cudaLaunchConfig_t cfg = config(cluster, cluster, nullptr, at);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, F, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cache[dev][cluster].store(n);
        return n;
    }

    static fg_status launch(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &td,
                            const CUtensorMap &tsa, const GemmParams &p, int grid, int cluster,
                            cudaStream_t stream) {
        if (!configure()) return cuda_fail();
        cudaLaunchAttribute at[2];
        cudaLaunchConfig_t cfg = config(grid, cluster, stream, at, g_pdl.load() != 0);
        if (cudaLaunchKernelEx(&cfg, F, ta, tb, td, tsa, p) != cudaSuccess) return cuda_fail();
        return cudaPeekAtLastError() == cudaSuccess ? FG_OK : cuda_fail();
    }
};

}  // namespace fgh
