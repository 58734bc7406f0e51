// qmv_mma_host.cu -- host side of the warp-level tensor-core decode kernel
// (qmv_mma.cuh): bit-width dispatch, the shared-memory padding model, and
// per-device caches of the launch limits.
#include <map>
#include <mutex>
#include <tuple>

#include "qmv_mma.cuh"

namespace lowbit {
namespace mma {

#define LOWBIT_MMA_DECL(B)                                                                                  \
    cudaError_t launch_b##B(const uint16_t *, const uint8_t *, const uint16_t *, const uint16_t *,          \
                            const uint16_t *, uint16_t *, int64_t, int, int, int, int, cudaStream_t);       \
    uint32_t timeouts_b##B(bool);
LOWBIT_MMA_DECL(1)
LOWBIT_MMA_DECL(2)
LOWBIT_MMA_DECL(3)
LOWBIT_MMA_DECL(4)
LOWBIT_MMA_DECL(5)
LOWBIT_MMA_DECL(6)
LOWBIT_MMA_DECL(7)
#undef LOWBIT_MMA_DECL

namespace {

// Shared-memory wavefronts of one pass of the consumers' weight reads for a
// staged-row stride: lane 4 gid + t reads, for blocks beta = 0, 1, the b words
// at row gid, byte (128 beta + 32 t) b / 8, with the widest aligned loads.
int model_wavefronts(int bits, uint32_t stride) {
    const int width = bits == 4 ? 16 : ((bits == 2 || bits == 6) ? 8 : 4);
    const int per_phase = width == 16 ? 8 : (width == 8 ? 16 : 32);
    int total = 0;
    for (int beta = 0; beta < 2; ++beta) {
        for (int i = 0; i < 4 * bits; i += width) {
            for (int ph = 0; ph < 32; ph += per_phase) {
                int words_in_bank[32] = {};
                uint32_t seen[32][32];
                int nseen[32] = {};
                int worst = 1;
                for (int lane = ph; lane < ph + per_phase; ++lane) {
                    const int gid = lane >> 2, t = lane & 3;
                    const uint32_t a = (uint32_t)gid * stride + (uint32_t)(((128 * beta + 32 * t) * bits) >> 3) + i;
                    for (uint32_t wd = a / 4; wd < (a + width) / 4; ++wd) {
                        const int bank = (int)(wd % 32);
                        bool dup = false;
                        for (int k = 0; k < nseen[bank]; ++k) dup = dup || seen[bank][k] == wd;
                        if (!dup && nseen[bank] < 32) {
                            seen[bank][nseen[bank]++] = wd;
                            words_in_bank[bank]++;
                            worst = std::max(worst, words_in_bank[bank]);
                        }
                    }
                }
                total += worst;
            }
        }
    }
    return total;
}

// Wavefronts of one warp-wide shared load: `addr` per lane, `width` bytes
// each (phases of 32, 16 or 8 lanes for 4-, 8- and 16-byte loads).
int warp_wavefronts(const uint32_t (&addr)[32], int width) {
    const int per_phase = width == 16 ? 8 : (width == 8 ? 16 : 32);
    int total = 0;
    for (int ph = 0; ph < 32; ph += per_phase) {
        uint32_t words[32][8];
        int n[32] = {};
        int worst = 1;
        for (int l = ph; l < ph + per_phase; ++l)
            for (uint32_t wd = addr[l] / 4; wd < (addr[l] + (uint32_t)std::max(width, 4)) / 4; ++wd) {
                const int bank = (int)(wd % 32);
                bool dup = false;
                for (int k = 0; k < n[bank]; ++k) dup = dup || words[bank][k] == wd;
                if (!dup && n[bank] < 8) {
                    words[bank][n[bank]++] = wd;
                    worst = std::max(worst, n[bank]);
                }
            }
        total += worst;
    }
    return total;
}

// The epilogue's scale reads for a staged row of spg fp16: lane 4 gid + t
// of warp w reads row gid at group w * gsl + c, c = 2t as a 32-bit pair (one
// row of x, two or more groups per slice) or (2t) / MP as 16 bits.
int sz_model(int spg, int gsl, int MP, int W) {
    int total = 0;
    const bool pair = MP == 1 && gsl >= 2;
    for (int w = 0; w < W; ++w) {
        uint32_t a[32];
        for (int l = 0; l < 32; ++l) {
            const int gid = l >> 2, t = l & 3;
            const int c = pair ? ((2 * t < gsl) ? 2 * t : 0) : std::min((2 * t) / MP, gsl - 1);
            a[l] = (uint32_t)((gid * spg + w * gsl + c) * 2);
        }
        total += warp_wavefronts(a, pair ? 4 : 2);
    }
    return total;
}

std::mutex g_spg_mu;
std::map<std::tuple<int, int, int, int>, int> g_spg_cache;

std::atomic<uint32_t> g_pad_cache[8][8];   // [bits][(crow % 128) / 16]: pad + 1 (0 = unknown)


}  // namespace

uint32_t row_pad(int bits, uint32_t crow_bytes) {
    const uint32_t key = (crow_bytes % 128u) / 16u;
    std::atomic<uint32_t> &slot = g_pad_cache[bits & 7][key];
    uint32_t v = slot.load(std::memory_order_relaxed);
    if (v != 0) return v - 1;
    uint32_t best = 16;
    int best_w = 1 << 30;
    for (uint32_t pad = 16; pad < 128; pad += 16) {
        const int w = model_wavefronts(bits, crow_bytes + pad);
        if (w < best_w) {
            best_w = w;
            best = pad;
        }
    }
    slot.store(best + 1, std::memory_order_relaxed);
    return best;
}

int sz_pitch(int groups, int gsl, int MP, int W) {
    const auto key = std::make_tuple(groups, gsl, MP, W);
    {
        std::lock_guard<std::mutex> lk(g_spg_mu);
        auto it = g_spg_cache.find(key);
        if (it != g_spg_cache.end()) return it->second;
    }
    const int base = std::max(8, (groups + 7) & ~7);
    int best = base, best_w = 1 << 30;
    for (int spg = base; spg <= base + 32; spg += 8) {
        const int wf = sz_model(spg, gsl, MP, W);
        if (wf < best_w) {
            best_w = wf;
            best = spg;
        }
    }
    std::lock_guard<std::mutex> lk(g_spg_mu);
    g_spg_cache[key] = best;
    return best;
}

bool encode_2d(CUtensorMap *map, CUtensorMapDataType type, const void *base, uint64_t inner, uint64_t rows,
               uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
    const uint64_t dims[2] = {inner, rows};
    const uint64_t strides[1] = {row_stride_bytes};
    const uint32_t box[2] = {box_inner, box_rows};
    return encode_tiled(map, type, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

int max_clusters(const void *fn, int dev, int ks, uint32_t smem, int threads) {
    if (ks == 1) return blocks_per_sm(fn, dev, threads, smem) * device_sm_count(dev);
    return clusters_at_once(fn, dev, ks, threads, smem);
}

}  // namespace mma

cudaError_t launch_qmv_mma(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                           const uint16_t *bias, uint16_t *y, int64_t M, int64_t K, int64_t N, int bits, int group,
                           int64_t F, cudaStream_t stream) {
    const int k = (int)K, n = (int)N, f = (int)F;
    switch (bits) {
        case 1: return mma::launch_b1(x, w, s, z, bias, y, M, k, n, group, f, stream);
        case 2: return mma::launch_b2(x, w, s, z, bias, y, M, k, n, group, f, stream);
        case 3: return mma::launch_b3(x, w, s, z, bias, y, M, k, n, group, f, stream);
        case 4: return mma::launch_b4(x, w, s, z, bias, y, M, k, n, group, f, stream);
        case 5: return mma::launch_b5(x, w, s, z, bias, y, M, k, n, group, f, stream);
        case 6: return mma::launch_b6(x, w, s, z, bias, y, M, k, n, group, f, stream);
        case 7: return mma::launch_b7(x, w, s, z, bias, y, M, k, n, group, f, stream);
        default: return cudaErrorInvalidValue;
    }
}

bool qmv_mma_shape_ok(int64_t K, int group) {
    if (K <= 0 || K % mma::kSlice != 0 || K % group != 0 || ((K / group) * 2) % 16 != 0) return false;
    for (int k = 1; k <= 8; ++k)
        if (K % (mma::kSlice * k) == 0 && K / k <= mma::kSlice * mma::kMaxW) return true;
    return false;
}

int qmv_mma_rows(int group) { return mma::max_rows(group); }

uint32_t mma_timeouts(bool reset) {
    return mma::timeouts_b1(reset) + mma::timeouts_b2(reset) + mma::timeouts_b3(reset) +
           mma::timeouts_b4(reset) + mma::timeouts_b5(reset) + mma::timeouts_b6(reset) + mma::timeouts_b7(reset);
}

}  // namespace lowbit
