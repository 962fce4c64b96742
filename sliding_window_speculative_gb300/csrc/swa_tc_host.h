// Internal interface between the C-ABI layer and the tensor-core path.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include <atomic>
#include <utility>

#include "swa_simt.cuh"

namespace swa {

// Kernel parameters of the tensor-core path (plain data).
struct TcParams {
    AttnParams a;
    int rows_per_tile;    // packed rows per item (a multiple of G, <= N)
    int q_rows_per_tile;  // draft rows per item
    int items;            // splits * Hkv * row_tiles * B
    // items_per_cta > 0: CTA c takes the contiguous block of items_per_cta (+1
    // for c < items_extra) items starting at c * items_per_cta +
    // min(c, items_extra); 0: CTA c takes items c, c + grid, c + 2 grid, ...
    int items_per_cta, items_extra;
    // fills of a CTA's first item issued ahead of the producer loop, at most
    // (1 when the launch covers half the SMs or more: every CTA loading at
    // once saturates HBM and the first K tile should land first)
    int early_max;
};

// TMA tensor maps of one call.  The cache is viewed as rows of D bf16
// (B * Hkv * L rows); a map with box "A atoms" loads 8*A consecutive rows
// from any start row as A blocks of [head-dim slab][8 rows][128 bytes], so
// a 128-key tile arrives in one copy and a partial tile in a few.
struct TcMaps {
    CUtensorMap k_atoms[4];  // 4D boxes of 16, 8, 4, 2 atoms
    CUtensorMap k_atom;      // 3D box of one atom (rows past the cache are zero-filled)
    CUtensorMap v_atoms[4];
    CUtensorMap v_atom;
    CUtensorMap q;           // 3D box (64 dims x G heads x draft rows)
    // fused append only: the new rows k_new / v_new [B, q_len, Hkv, D] as 5D
    // (x = 64 dims, y = draft row, z = slab, w = KV head, v = sequence), a
    // box of one atom (8 draft rows; rows past q_len are zero-filled)
    CUtensorMap kn_atom;
    CUtensorMap vn_atom;
};

struct TcConfInfo {
    int nslot;        // ring slots of one 128-key tile each
    int smem_bytes;   // dynamic shared memory per CTA
    int tmem_cols;    // TMEM columns per CTA
    int ctas_per_sm;  // resident CTAs per SM the plan assumes
};

struct TcLaunch {
    TcParams T;
    int rows_major;  // 1: the kernel with packed rows as the MMA's M (swa_rows_kernel)
    // 1 (with rows_major): the CTA-pair kernel (swa_pair_kernel), clusters of
    // two CTAs; T.rows_per_tile / T.q_rows_per_tile are one CTA's rows, an
    // item holds twice that, and grid counts CTAs (two per item at once)
    int pairs;
    int D, N;   // head_dim, padded rows per item (rows kernel: 32, 64 or 128)
    int grid;   // persistent CTAs
    long long cache_rows;  // rows of D elements in each of the K and V tensors
    const void *k, *v, *q;
};

// Kernels are launched with programmatic stream serialization (programmatic
// dependent launch): each may begin its prologue while the previous kernel
// in the stream finishes, and waits (griddepcontrol.wait) before it reads
// any caller memory.  On unless a test or sweep turned it off through
// swa_set_debug_options (defined with the C ABI).
bool pdl_enabled();

// True when a test asked (swa_set_debug_options, fail_launch) that this
// launch not be made; counts the launches down to it.
bool launch_fault_due();

// A kernel's dynamic shared memory limit raised to `smem` on the current
// device, once per device: `done` holds one flag per device (NDEV of them;
// devices past that set the attribute on every call).  Calls racing on a
// device's first launch may both set it, which is harmless.
template <typename K, int NDEV>
cudaError_t raise_smem_limit(K kern, int smem, std::atomic<bool> (&done)[NDEV]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < NDEV;
    if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess && cached) done[dev].store(true, std::memory_order_release);
    return e;
}

template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    if (launch_fault_due()) return cudaErrorLaunchOutOfResources;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Constants of the (head_dim, padded rows) configuration; false if none.
bool tc_conf(int D, int N, TcConfInfo *c);

// Encodes the TMA tensor maps and launches; on failure writes a message.
cudaError_t tc_launch(const TcLaunch &L, cudaStream_t stream, char *err, size_t errlen);

}  // namespace swa
