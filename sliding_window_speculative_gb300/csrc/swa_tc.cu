// Host side of the tensor-core path: per-configuration constants, TMA tensor
// maps for the cache and the queries, and the persistent launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "swa_tc.cuh"
#include "swa_tc_host.h"

namespace swa {
namespace {

// Ring slots per (head_dim, padded rows).  Small row tiles keep the CTA
// under half of the SM's shared memory so two CTAs share an SM; large row
// tiles take the SM alone with a deeper ring.
constexpr int nslot_for(int D, int N) {
    return D == 256 ? (N <= 32 ? 4 : 8) : (N <= 32 ? 4 : N == 64 ? 8 : 6);
}

template <int D, int N>
struct Conf {
    static constexpr int NSLOT = nslot_for(D, N);
    using C = TcCfg<D, N, NSLOT>;
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

template <int D, int N>
cudaError_t launch(const TcLaunch &L, const CUtensorMap &mk, const CUtensorMap &mv,
                   const CUtensorMap &mq, cudaStream_t stream) {
    using C = typename Conf<D, N>::C;
    auto kern = swa_tc_kernel<D, N, Conf<D, N>::NSLOT>;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    kern<<<L.grid, kTcThreads, C::SMEM_BYTES, stream>>>(L.T, mk, mv, mq);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const TcLaunch &L, const CUtensorMap &mk, const CUtensorMap &mv,
                     const CUtensorMap &mq, cudaStream_t s) {
    switch (L.N) {
        case 16: return launch<D, 16>(L, mk, mv, mq, s);
        case 32: return launch<D, 32>(L, mk, mv, mq, s);
        case 64: return launch<D, 64>(L, mk, mv, mq, s);
        default:
            if constexpr (D == 128) return launch<D, 128>(L, mk, mv, mq, s);
            return cudaErrorInvalidConfiguration;  // D = 256 row tiles stop at 64 rows
    }
}

template <int D, int N>
void conf_info(TcConfInfo *c) {
    using C = typename Conf<D, N>::C;
    c->nslot = Conf<D, N>::NSLOT;
    c->smem_bytes = C::SMEM_BYTES;
    c->tmem_cols = C::TMEM_COLS;
    // the register budget (launch bounds) is sized for MIN_BLOCKS CTAs per SM
    const int by_tmem = 512 / C::TMEM_COLS;
    c->ctas_per_sm = C::MIN_BLOCKS < by_tmem ? C::MIN_BLOCKS : by_tmem;
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
            case 128: conf_info<128, 128>(c); return true;
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
    CUtensorMap mk, mv, mq;
    // cache viewed as [B * Hkv * L rows, D]: boxes of 128 keys x 64 dims
    {
        cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)P.B * P.Hkv * (cuuint64_t)P.L};
        cuuint64_t strides[1] = {(cuuint64_t)D * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)kTcTileKeys};
        cuuint32_t es[2] = {1, 1};
        for (int which = 0; which < 2; ++which) {
            CUresult r = g_encode(which ? &mv : &mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                  const_cast<void *>(which ? L.v : L.k), dims, strides, box, es,
                                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) {
                snprintf(err, errlen, "cuTensorMapEncodeTiled(%s cache) failed: %d",
                         which ? "V" : "K", (int)r);
                return cudaErrorInvalidValue;
            }
        }
    }
    // queries viewed as [B * q_len, Hq, D]: boxes of (draft rows x G heads x 64 dims)
    {
        cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)P.Hq, (cuuint64_t)P.B * P.q_len};
        cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)P.Hq * D * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)P.G, (cuuint32_t)L.T.q_rows_per_tile};
        cuuint32_t es[3] = {1, 1, 1};
        CUresult r = g_encode(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(L.q),
                              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            snprintf(err, errlen, "cuTensorMapEncodeTiled(q) failed: %d", (int)r);
            return cudaErrorInvalidValue;
        }
    }
    if (D == 256) return launch_d<256>(L, mk, mv, mq, stream);
    return launch_d<128>(L, mk, mv, mq, stream);
}

}  // namespace swa
