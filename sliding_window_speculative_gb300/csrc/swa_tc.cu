// Host side of the tensor-core path: per-configuration constants, TMA tensor
// maps for the cache and the queries, and the persistent launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "swa_pair.cuh"
#include "swa_rows.cuh"
#include "swa_tc.cuh"
#include "swa_tc_host.h"

namespace swa {
namespace {

// Per (head_dim, padded rows): ring slots of one 128-key tile and Q / P
// buffer counts, sized to one CTA per SM (at most 227 KB of shared memory).
template <int D, int N>
struct Conf {
    // A ring of three K-or-V tiles lets V(t+1) load while V(t) waits for its
    // PV; at head_dim 256 (64 KB tiles) that leaves room for one Q and one P
    // buffer beside it (two at 16 rows).  O^T (2N columns per head-dim half)
    // is double-buffered unless TMEM runs out (head_dim 256, 64 rows).
    static constexpr int NT = D == 256 ? (N <= 32 ? 3 : 2) : 5;
    static constexpr int QB = (D == 256 && N >= 32) ? 1 : (D == 128 && N == 64) ? 1 : 2;
    static constexpr int PB = (D == 256 && N >= 32) ? 1 : (N == 64) ? 1 : 2;
    static constexpr int OB = (D == 256 && N == 64) ? 1 : 2;
    using C = TcCfg<D, N, NT, QB, PB, OB>;
};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

template <int D, int N, bool AP>
cudaError_t launch_ap(const TcLaunch &L, const TcMaps &maps, cudaStream_t stream) {
    using Cf = Conf<D, N>;
    using C = typename Cf::C;
    auto kern = swa_tc_kernel<D, N, Cf::NT, Cf::QB, Cf::PB, Cf::OB, AP>;
    static std::atomic<bool> attr_done[64];
    cudaError_t e = raise_smem_limit(kern, C::SMEM_BYTES, attr_done);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(L.grid), dim3(AP ? kTcThreads + 32 : kTcThreads),
                         C::SMEM_BYTES, stream, L.T, maps);
}

// The plain kernel, or (fused append) its variant with the append warp.
template <int D, int N>
cudaError_t launch(const TcLaunch &L, const TcMaps &maps, cudaStream_t stream) {
    return L.T.a.k_new != nullptr ? launch_ap<D, N, true>(L, maps, stream)
                                  : launch_ap<D, N, false>(L, maps, stream);
}

// Rows-major kernel: per (head_dim, Q rows) the ring tiles and Q buffers
// that fit one CTA per SM.
template <int D, int QR>
struct RowsConf {
    static constexpr int NT = D == 256 ? (QR == 32 ? 3 : 2) : (QR == 128 ? 5 : 6);
    static constexpr int QB = D == 256 ? (QR == 64 ? 2 : 1) : (QR == 32 ? 2 : 1);
    using C = RowsCfg<D, QR, NT, QB>;
};

template <int D, int QR, bool AP>
cudaError_t launch_rows_ap(const TcLaunch &L, const TcMaps &maps, cudaStream_t stream) {
    using Cf = RowsConf<D, QR>;
    using C = typename Cf::C;
    auto kern = swa_rows_kernel<D, QR, Cf::NT, Cf::QB, AP>;
    static std::atomic<bool> attr_done[64];
    cudaError_t e = raise_smem_limit(kern, C::SMEM_BYTES, attr_done);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(L.grid), dim3(AP ? kRowsThreads + 32 : kRowsThreads),
                         C::SMEM_BYTES, stream, L.T, maps);
}

template <int D, int QR>
cudaError_t launch_rows(const TcLaunch &L, const TcMaps &maps, cudaStream_t stream) {
    return L.T.a.k_new != nullptr ? launch_rows_ap<D, QR, true>(L, maps, stream)
                                  : launch_rows_ap<D, QR, false>(L, maps, stream);
}

template <int D>
cudaError_t launch_rows_d(const TcLaunch &L, const TcMaps &maps, cudaStream_t s) {
    switch (L.N) {
        case 32: return launch_rows<D, 32>(L, maps, s);
        case 64: return launch_rows<D, 64>(L, maps, s);
        case 128: return launch_rows<D, 128>(L, maps, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

// CTA-pair kernel: clusters of two CTAs, as many pairs as the plan's grid
// holds and the device runs at once (queried once per device).
template <int D>
cudaError_t launch_pairs(const TcLaunch &L, const TcMaps &maps, const PairMaps &pm,
                         cudaStream_t stream) {
    using C = PairCfg<D, kPairSlots>;
    auto kern = swa_pair_kernel<D, kPairSlots>;
    static std::atomic<bool> attr_done[64];
    static std::atomic<int> max_pairs[64];
    cudaError_t e = raise_smem_limit(kern, C::SMEM_BYTES, attr_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int fit = dev >= 0 && dev < 64 ? max_pairs[dev].load(std::memory_order_acquire) : 0;
    if (fit == 0) {
        cfg.gridDim = dim3((unsigned)L.grid);
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&fit, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (fit < 1) return cudaErrorInvalidConfiguration;
        if (dev >= 0 && dev < 64) max_pairs[dev].store(fit, std::memory_order_release);
    }
    const int pairs = L.grid / 2 < fit ? L.grid / 2 : fit;
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    if (launch_fault_due()) return cudaErrorLaunchOutOfResources;
    return cudaLaunchKernelEx(&cfg, kern, L.T, maps, pm);
}

template <int D>
cudaError_t launch_d(const TcLaunch &L, const TcMaps &maps, cudaStream_t s) {
    switch (L.N) {
        case 16: return launch<D, 16>(L, maps, s);
        case 32: return launch<D, 32>(L, maps, s);
        case 64: return launch<D, 64>(L, maps, s);
        default: return cudaErrorInvalidConfiguration;
    }
}

template <int D, int N>
void conf_info(TcConfInfo *c) {
    using C = typename Conf<D, N>::C;
    c->nslot = Conf<D, N>::NT;
    c->smem_bytes = C::SMEM_BYTES;
    c->tmem_cols = C::TMEM_COLS;
    c->ctas_per_sm = 1;  // persistent: one CTA per SM
}

}  // namespace

bool tc_conf(int D, int N, TcConfInfo *c) {
    if (D == 256) {
        switch (N) {
            case 16: conf_info<256, 16>(c); return true;
            case 32: conf_info<256, 32>(c); return true;
            case 64: conf_info<256, 64>(c); return true;
        }
    } else if (D == 128) {
        switch (N) {
            case 16: conf_info<128, 16>(c); return true;
            case 32: conf_info<128, 32>(c); return true;
            case 64: conf_info<128, 64>(c); return true;
        }
    }
    return false;
}

cudaError_t tc_launch(const TcLaunch &L, cudaStream_t stream, char *err, size_t errlen) {
    if (!load_encode()) {
        snprintf(err, errlen, "cuTensorMapEncodeTiled is not available from the driver");
        return cudaErrorNotSupported;
    }
    const AttnParams &P = L.T.a;
    const int D = L.D;
    // K and V cache viewed as rows of D bf16 (B * Hkv * L rows, or every
    // page's rows of a paged cache).  4D maps
    // (x = 64 dims, y = row, z = 64-dim slab, w = 8-row atom; strides D*2,
    // 128 and 8*D*2 bytes) with boxes of 16, 8, 4 and 2 atoms, and a 3D
    // one-atom map (x, y, z) whose rows are bounds-checked one by one.
    // Both land as [atom][slab][8 rows][128 bytes], 128-byte swizzled.
    TcMaps maps{};
    const cuuint64_t rows = (cuuint64_t)L.cache_rows;
    const cuuint32_t slabs = (cuuint32_t)(D / 64);
    for (int kv = 0; kv < 2; ++kv) {
        const void *base = kv ? L.v : L.k;
        CUtensorMap *m4 = kv ? maps.v_atoms : maps.k_atoms;
        for (int bi = 0; bi < 5; ++bi) {
            const bool atom = bi == 4;
            const cuuint32_t A = atom ? 1u : (16u >> bi);
            cuuint64_t dims[4] = {64, rows, slabs, 16};
            cuuint64_t strides[3] = {(cuuint64_t)D * 2, 128, (cuuint64_t)D * 2 * 8};
            cuuint32_t box[4] = {64, 8, slabs, A};
            cuuint32_t es[4] = {1, 1, 1, 1};
            CUresult r = g_encode(atom ? (kv ? &maps.v_atom : &maps.k_atom) : &m4[bi],
                                  CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, atom ? 3 : 4,
                                  const_cast<void *>(base), dims, strides, box, es,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) {
                snprintf(err, errlen, "cuTensorMapEncodeTiled(%s cache, %u-atom box) failed: %d",
                         kv ? "V" : "K", (unsigned)A, (int)r);
                return cudaErrorInvalidValue;
            }
        }
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)P.Hq, (cuuint64_t)P.B * P.q_len};
        cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)P.Hq * D * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)P.G, (cuuint32_t)L.T.q_rows_per_tile};
        cuuint32_t es[3] = {1, 1, 1};
        CUresult r = g_encode(&maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                              const_cast<void *>(L.q), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            snprintf(err, errlen, "cuTensorMapEncodeTiled(q) failed: %d", (int)r);
            return cudaErrorInvalidValue;
        }
    }
    if (P.k_new != nullptr) {
        for (int kv = 0; kv < 2; ++kv) {
            cuuint64_t dims[5] = {64, (cuuint64_t)P.q_len, slabs, (cuuint64_t)P.Hkv,
                                  (cuuint64_t)P.B};
            cuuint64_t strides[4] = {(cuuint64_t)P.Hkv * D * 2, 128, (cuuint64_t)D * 2,
                                     (cuuint64_t)P.q_len * P.Hkv * D * 2};
            cuuint32_t box[5] = {64, 8, slabs, 1, 1};
            cuuint32_t es[5] = {1, 1, 1, 1, 1};
            CUresult r = g_encode(kv ? &maps.vn_atom : &maps.kn_atom,
                                  CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                                  const_cast<__nv_bfloat16 *>(kv ? P.v_new : P.k_new), dims,
                                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) {
                snprintf(err, errlen, "cuTensorMapEncodeTiled(%s new rows) failed: %d",
                         kv ? "V" : "K", (int)r);
                return cudaErrorInvalidValue;
            }
        }
    }
    if (L.pairs) {
        // V as D / 2 head dims per CTA: boxes of half the slabs, otherwise as
        // the full maps above
        if (D != 256 || L.grid < 2) return cudaErrorInvalidConfiguration;
        PairMaps pm{};
        for (int bi = 0; bi < 5; ++bi) {
            const bool atom = bi == 4;
            const cuuint32_t A = atom ? 1u : (16u >> bi);
            cuuint64_t dims[4] = {64, rows, slabs, 16};
            cuuint64_t strides[3] = {(cuuint64_t)D * 2, 128, (cuuint64_t)D * 2 * 8};
            cuuint32_t box[4] = {64, 8, slabs / 2, A};
            cuuint32_t es[4] = {1, 1, 1, 1};
            CUresult r = g_encode(atom ? &pm.vh_atom : &pm.vh_atoms[bi],
                                  CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, atom ? 3 : 4,
                                  const_cast<void *>(L.v), dims, strides, box, es,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) {
                snprintf(err, errlen, "cuTensorMapEncodeTiled(V cache halves, %u-atom box) failed: %d",
                         (unsigned)A, (int)r);
                return cudaErrorInvalidValue;
            }
        }
        if (P.G <= 32 && 32 % P.G == 0) {
            cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)P.Hq, (cuuint64_t)P.B * P.q_len};
            cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)P.Hq * D * 2};
            cuuint32_t box[3] = {32, (cuuint32_t)P.G, (cuuint32_t)(32 / P.G)};
            cuuint32_t es[3] = {1, 1, 1};
            CUresult r = g_encode(&pm.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, P.out, dims, strides,
                                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) {
                snprintf(err, errlen, "cuTensorMapEncodeTiled(out) failed: %d", (int)r);
                return cudaErrorInvalidValue;
            }
            pm.out_ok = 1;
        }
        return launch_pairs<256>(L, maps, pm, stream);
    }
    if (L.rows_major) {
        if (D == 256) return launch_rows_d<256>(L, maps, stream);
        return launch_rows_d<128>(L, maps, stream);
    }
    if (D == 256) return launch_d<256>(L, maps, stream);
    return launch_d<128>(L, maps, stream);
}

}  // namespace swa
