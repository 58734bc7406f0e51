// device.cu -- host state shared by the kernels' launch code: SM counts,
// raised dynamic shared-memory limits and occupancy queries, per device (function
// attributes and occupancy belong to each device's context, so those caches are
// keyed by device ordinal and kernel; a failed query is not cached), and TMA
// tensor-map descriptors.
#include <cudaTypedefs.h>

#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <unordered_map>

#include <atomic>

#include "common.cuh"

namespace lowbit {
namespace {

struct Key {
    int dev;
    const void *fn;
    int a, b;
    uint32_t c;
    bool operator<(const Key &o) const { return std::tie(dev, fn, a, b, c) < std::tie(o.dev, o.fn, o.a, o.b, o.c); }
};

std::mutex g_mu;
std::map<int, int> g_sms;                 // device -> SM count
std::map<Key, int> g_smem;                // (device, kernel, bytes) -> limit raised
std::map<Key, int> g_occ;                 // (device, kernel, threads, -, smem) -> CTAs per SM
std::map<Key, int> g_clusters;            // (device, kernel, ks, threads, smem) -> clusters

// Tensor-map descriptors by their encoding arguments.  A descriptor is a pure
// function of those arguments (it names an address, not an allocation), so a
// cached one is exactly what encoding again would return; encoding costs far
// more host time than a lookup, and eager callers encode on every call.
constexpr size_t kMaxMaps = 4096;
std::mutex g_map_mu;
std::unordered_map<std::string, CUtensorMap> g_maps;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

}  // namespace

bool encode_tiled(CUtensorMap *map, CUtensorMapDataType type, uint32_t rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                  CUtensorMapSwizzle swizzle) {
    if (rank < 1 || rank > 5) return false;
    std::string key(sizeof(uint32_t) * 3 + sizeof(void *) + rank * (2 * sizeof(uint64_t) + sizeof(uint32_t)), '\0');
    char *k = key.data();
    const uint32_t head[3] = {(uint32_t)type, rank, (uint32_t)swizzle};
    std::memcpy(k, head, sizeof head);
    k += sizeof head;
    std::memcpy(k, &base, sizeof base);
    k += sizeof base;
    std::memcpy(k, dims, rank * sizeof(uint64_t));
    k += rank * sizeof(uint64_t);
    if (rank > 1) std::memcpy(k, strides, (rank - 1) * sizeof(uint64_t));
    k += rank * sizeof(uint64_t);
    std::memcpy(k, box, rank * sizeof(uint32_t));
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *map = it->second;
            return true;
        }
    }
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], es[5];
    for (uint32_t i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    if (enc(map, type, rank, const_cast<void *>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() >= kMaxMaps) g_maps.clear();
    g_maps.emplace(std::move(key), *map);
    return true;
}

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

int device_sm_count(int dev) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_sms.find(dev);
        if (it != g_sms.end()) return it->second;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_sms[dev] = v;
    return v;
}

cudaError_t raise_smem_limit(const void *fn, int dev, int bytes) {
    const Key key{dev, fn, bytes, 0, 0};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_smem.count(key)) return cudaSuccess;
    }
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_smem[key] = 1;
    return cudaSuccess;
}

int blocks_per_sm(const void *fn, int dev, int threads, uint32_t smem) {
    const Key key{dev, fn, threads, 0, smem};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 0) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ[key] = n;
    return n;
}

int clusters_at_once(const void *fn, int dev, int ks, int threads, uint32_t smem) {
    const Key key{dev, fn, ks, threads, smem};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_clusters.find(key);
        if (it != g_clusters.end()) return it->second;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)ks;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 0) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_clusters[key] = n;
    return n;
}

}  // namespace lowbit
