// device.cu -- per-device host state shared by the kernels' launch code: SM
// counts, raised dynamic shared-memory limits and occupancy queries.  Function
// attributes and occupancy belong to each device's context, so every cache is
// keyed by device ordinal (and kernel); a failed query is not cached.
#include <map>
#include <mutex>
#include <tuple>

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

}  // namespace

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
