// Tensor-core (tcgen05) split-KV kernel for sliding-window verify attention.
//
// Persistent CTAs walk a list of work items (sequence, KV head, key chunk,
// row tile).  Keys are the MMA's M dimension: for every tile of 128 keys
//
//   S^T[128 keys x N rows] = K_tile[128 x D] . Q[N x D]^T      (TMEM, fp32)
//   O^T[D x N]            += V_tile^T[D x 128] . P^T[N x 128]^T (TMEM, fp32)
//
// P is carried into the second MMA as two bf16 tiles, P = P_hi + P_lo with
// P_hi = bf16(P) and P_lo = bf16(P - P_hi), so the weights keep about 16
// significant bits instead of bf16's 8; the PV product is issued twice.
//
// where the N rows are the packed query rows of one KV head (G query heads
// times the q_len draft rows, padded to a multiple of 16), so every K/V byte
// is read once per KV head and small draft blocks cost no M padding.  K and
// V tiles arrive by TMA in 16 KB slabs (128 keys x 64 dims, 128-byte
// swizzle) through a ring of shared-memory slots; Q arrives once per item.
//
// Warp roles (192 threads):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM owner and MMA issuer (one lane)
//   warps 2..5  softmax / correction / epilogue, one thread per TMEM lane:
//               a thread owns one key of the S^T tile and one head-dim row
//               of the O^T accumulator.
//
// Softmax runs in the log2 domain with a lazily raised reference maximum:
// each row keeps m_ref; a tile whose scaled score exceeds m_ref + 8 (a
// factor 256) for any row triggers an exact per-row tile maximum, a raise of
// m_ref and, if O already holds data, a rescale of O^T in TMEM.  Otherwise
// P = 2^(s - m_ref) <= 256, exact in the ratio the normaliser divides out.
// Row sums are reduced across lanes with a reduce-scatter butterfly.
//
// Every wait on an mbarrier is bounded; a wait that gives up sets the fault
// word, the roles leave their loops together, and TMEM is freed.
#pragma once

#include "swa_simt.cuh"
#include "swa_tc_host.h"
#include "swa_tc_ptx.cuh"

namespace swa {

constexpr int kTcThreads = 192;
constexpr int kTcTileKeys = 128;

template <int D, int N, int NSLOT>
struct TcCfg {
    static constexpr int SLABS = D / 64;
    static constexpr int SLOT_BYTES = 16384;
    static constexpr int Q_SLAB = N * 128;
    static constexpr int P_SLAB = N * 128;
    static constexpr int RING_OFF = 0;
    static constexpr int Q_OFF = RING_OFF + NSLOT * SLOT_BYTES;
    static constexpr int P_OFF = Q_OFF + SLABS * Q_SLAB;
    static constexpr int P_LO = 2 * P_SLAB;               // P_lo tile after P_hi
    static constexpr int RED_OFF = P_OFF + 4 * P_SLAB;  // float [4][N]
    static constexpr int MREF_OFF = RED_OFF + 4 * N * 4;  // float [N]
    static constexpr int ALPHA_OFF = MREF_OFF + N * 4;    // float [N]
    static constexpr int LSUM_OFF = ALPHA_OFF + N * 4;    // float [N]
    static constexpr int BAR_OFF = LSUM_OFF + N * 4;
    static constexpr int NBARS = 2 * NSLOT + 10;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
    static constexpr int END = MISC_OFF + 16;
    static constexpr int SMEM_BYTES = END + 1024;  // slack for 1024-byte alignment
    static constexpr int TMEM_USED = 2 * N + (D / 128) * N;
    static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                     : TMEM_USED <= 64  ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256
                                                        : 512;
    static constexpr int CW = N >= 32 ? 32 : 16;  // TMEM columns per load
    static constexpr int NCH = N / CW;
    static constexpr bool LOOKAHEAD = NSLOT >= 2 * SLABS;
    // two CTAs share an SM when shared memory allows it
    static constexpr int MIN_BLOCKS = SMEM_BYTES + 1024 <= 113 * 1024 ? 2 : 1;
    static_assert(NSLOT % 2 == 0 && NSLOT >= SLABS, "ring holds whole K or V tiles in pairs");
    static_assert(N % 16 == 0 && N >= 16 && N <= 128, "rows per tile");
    static_assert(TMEM_USED <= 512, "TMEM");
    // barrier indices
    static constexpr int B_FULL = 0, B_EMPTY = NSLOT, B_QFULL = 2 * NSLOT, B_QEMPTY = 2 * NSLOT + 1,
                         B_SFULL = 2 * NSLOT + 2, B_SFREE = 2 * NSLOT + 4,
                         B_PFULL = 2 * NSLOT + 6, B_PVDONE = 2 * NSLOT + 7,
                         B_OFREE = 2 * NSLOT + 8, B_DRAIN = 2 * NSLOT + 9;
};

struct TcItem {
    int b, h, split, rt;
    ChunkRange cr;
    int n_tiles;
    int row0;  // first packed row of the item
    int rows;  // packed rows of the item
    int i0;    // first draft row
};

__device__ __forceinline__ TcItem tc_decode(const TcParams &T, int item) {
    const AttnParams &P = T.a;
    TcItem it;
    int rest = item;
    it.rt = rest % P.row_tiles;
    rest /= P.row_tiles;
    it.split = rest % P.splits;
    rest /= P.splits;
    it.h = rest % P.Hkv;
    it.b = rest / P.Hkv;
    it.cr = chunk_range(P, it.b, it.split);
    const int nk = it.cr.c_hi - it.cr.c_lo;
    it.n_tiles = nk > 0 ? (nk + kTcTileKeys - 1) / kTcTileKeys : 0;
    it.row0 = it.rt * T.rows_per_tile;
    it.rows = min(P.R - it.row0, T.rows_per_tile);
    it.i0 = it.rt * T.q_rows_per_tile;
    return it;
}

__device__ __forceinline__ void named_sync_softmax() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// True on every softmax thread if `v` is true on any of them.
__device__ __forceinline__ bool softmax_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 2, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Reduce-scatter of CW per-lane values across the warp with op `max` or
// `sum`: afterwards lane l holds the reduction of element (l % CW).
template <int CW, bool MAX>
__device__ __forceinline__ float lane_reduce(float (&v)[CW]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int half = CW / 2; half >= 1; half >>= 1) {
        const bool upper = (lane & half) != 0;
#pragma unroll
        for (int e = 0; e < half; ++e) {
            const float keep = upper ? v[e + half] : v[e];
            const float give = upper ? v[e] : v[e + half];
            const float got = __shfl_xor_sync(0xffffffffu, give, half);
            v[e] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    if constexpr (CW == 16) {
        const float got = __shfl_xor_sync(0xffffffffu, v[0], 16);
        v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
    }
    return v[0];
}

template <int CW>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t (&raw)[CW]) {
    if constexpr (CW == 32) {
        tc::tmem_ld32(taddr, raw);
    } else {
        tc::tmem_ld16(taddr, raw);
    }
    tc::tmem_wait_ld();
}

template <int D, int N, int NSLOT>
__global__ void __launch_bounds__(kTcThreads, (TcCfg<D, N, NSLOT>::MIN_BLOCKS))
    swa_tc_kernel(const __grid_constant__ TcParams T, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v,
                  const __grid_constant__ CUtensorMap map_q) {
    using C = TcCfg<D, N, NSLOT>;
    using namespace tc;
    constexpr int SLABS = C::SLABS;
    constexpr int CW = C::CW;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const AttnParams &P = T.a;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    uint8_t *ring = sm + C::RING_OFF;
    uint8_t *qs = sm + C::Q_OFF;
    uint8_t *ps = sm + C::P_OFF;
    float *red = reinterpret_cast<float *>(sm + C::RED_OFF);
    float *mref = reinterpret_cast<float *>(sm + C::MREF_OFF);
    float *alpha = reinterpret_cast<float *>(sm + C::ALPHA_OFF);
    float *lsum = reinterpret_cast<float *>(sm + C::LSUM_OFF);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::MISC_OFF + 4);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&bars[C::B_FULL + i], 1);
            mbar_init(&bars[C::B_EMPTY + i], 1);
        }
        mbar_init(&bars[C::B_QFULL], 1);
        mbar_init(&bars[C::B_QEMPTY], 1);
        mbar_init(&bars[C::B_SFULL], 1);
        mbar_init(&bars[C::B_SFULL + 1], 1);
        mbar_init(&bars[C::B_SFREE], 128);
        mbar_init(&bars[C::B_SFREE + 1], 128);
        mbar_init(&bars[C::B_PFULL], 128);
        mbar_init(&bars[C::B_PVDONE], 1);
        mbar_init(&bars[C::B_OFREE], 128);
        mbar_init(&bars[C::B_DRAIN], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // Q rows past the item's rows stay zero for the whole kernel (TMA
    // writes only the first rows_per_tile rows of each slab).
    for (int i = tid; i < SLABS * C::Q_SLAB / 16; i += kTcThreads)
        reinterpret_cast<uint4 *>(qs)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ======================================================= producer
        if (lane == 0) {
            prefetch_tmap(&map_k);
            prefetch_tmap(&map_v);
            prefetch_tmap(&map_q);
            const uint64_t policy = l2_policy_evict_first();
            uint32_t f = 0, qi = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < T.items && ok; item += gridDim.x) {
                const TcItem it = tc_decode(T, item);
                if (it.n_tiles == 0) continue;
                ok = mbar_wait_bounded(&bars[C::B_QEMPTY], (qi & 1) ^ 1, P.fault, kFaultCopyTimeout);
                if (!ok) break;
                mbar_arrive_expect_tx(&bars[C::B_QFULL], SLABS * T.rows_per_tile * 128);
                for (int s = 0; s < SLABS; ++s)
                    tma_load_3d(qs + s * C::Q_SLAB, &map_q, 64 * s, it.h * P.G,
                                it.b * P.q_len + it.i0, &bars[C::B_QFULL]);
                ++qi;
                const int y0 = (it.b * P.Hkv + it.h) * P.L + it.cr.c_lo;
                for (int t = 0; t < it.n_tiles && ok; ++t) {
                    for (int kv = 0; kv < 2 && ok; ++kv) {
                        for (int s = 0; s < SLABS; ++s) {
                            const uint32_t slot = f % NSLOT;
                            ok = mbar_wait_bounded(&bars[C::B_EMPTY + slot], ((f / NSLOT) & 1) ^ 1,
                                                   P.fault, kFaultCopyTimeout);
                            if (!ok) break;
                            mbar_arrive_expect_tx(&bars[C::B_FULL + slot], C::SLOT_BYTES);
                            tma_load_2d_hint(ring + slot * C::SLOT_BYTES, kv ? &map_v : &map_k,
                                             64 * s, y0 + kTcTileKeys * t,
                                             &bars[C::B_FULL + slot], policy);
                            ++f;
                        }
                    }
                }
            }
            if (!ok) *abort_flag = 1;
            // every copy this CTA issued has landed before it exits
            const uint32_t n_drain = f < (uint32_t)NSLOT ? f : (uint32_t)NSLOT;
            for (uint32_t k = 0; k < n_drain; ++k) {
                const uint32_t fi = f - 1 - k;
                mbar_wait_bounded(&bars[C::B_FULL + fi % NSLOT], (fi / NSLOT) & 1, P.fault,
                                  kFaultCopyTimeout);
            }
            if (qi > 0)
                mbar_wait_bounded(&bars[C::B_QFULL], (qi - 1) & 1, P.fault, kFaultCopyTimeout);
        }
    } else if (warp == 1) {
        // ============================================================ MMA
        if (lane == 0) {
            constexpr uint32_t ID_QK = idesc_bf16_f32(128, N, 0, 0);
            constexpr uint32_t ID_PV = idesc_bf16_f32(128, N, 1, 0);
            const uint32_t ring_a = smem_u32(ring);
            const uint32_t qs_a = smem_u32(qs);
            const uint32_t ps_a = smem_u32(ps);
            uint32_t f = 0, qi = 0, gt = 0, pc = 0, oc = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < T.items && ok; item += gridDim.x) {
                const TcItem it = tc_decode(T, item);
                if (it.n_tiles == 0) continue;
                ok = mbar_wait_bounded(&bars[C::B_QFULL], qi & 1, P.fault, kFaultCopyTimeout);
                if (!ok) break;
                ++qi;
                fence_after_sync();
                const uint32_t fbase = f;
                f += (uint32_t)it.n_tiles * 2 * SLABS;
                auto qk = [&](int t) -> bool {
                    const uint32_t g = gt + t;
                    const uint32_t sb = g & 1, use = g >> 1;
                    if (!mbar_wait_bounded(&bars[C::B_SFREE + sb], (use & 1) ^ 1, P.fault,
                                           kFaultCopyTimeout))
                        return false;
                    fence_after_sync();
                    for (int s = 0; s < SLABS; ++s) {
                        const uint32_t fi = fbase + (uint32_t)t * 2 * SLABS + s;
                        const uint32_t slot = fi % NSLOT;
                        if (!mbar_wait_bounded(&bars[C::B_FULL + slot], (fi / NSLOT) & 1, P.fault,
                                               kFaultCopyTimeout))
                            return false;
                        fence_after_sync();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a =
                                smem_desc_sw128(ring_a + slot * C::SLOT_BYTES + kk * 32, 16, 1024);
                            const uint64_t bdesc =
                                smem_desc_sw128(qs_a + s * C::Q_SLAB + kk * 32, 16, 1024);
                            mma_bf16_ss(tmem + sb * N, a, bdesc, ID_QK, (s | kk) != 0);
                        }
                        mma_commit(&bars[C::B_EMPTY + slot]);
                    }
                    mma_commit(&bars[C::B_SFULL + sb]);
                    return true;
                };
                if (C::LOOKAHEAD) ok = qk(0);
                for (int t = 0; t < it.n_tiles && ok; ++t) {
                    if (C::LOOKAHEAD) {
                        if (t + 1 < it.n_tiles) ok = qk(t + 1);
                    } else {
                        ok = qk(t);
                    }
                    if (!ok) break;
                    if (t == it.n_tiles - 1) mma_commit(&bars[C::B_QEMPTY]);
                    ok = mbar_wait_bounded(&bars[C::B_PFULL], pc & 1, P.fault, kFaultCopyTimeout);
                    if (!ok) break;
                    ++pc;
                    fence_after_sync();
                    if (t == 0) {
                        ok = mbar_wait_bounded(&bars[C::B_OFREE], (oc & 1) ^ 1, P.fault,
                                               kFaultCopyTimeout);
                        if (!ok) break;
                        ++oc;
                        fence_after_sync();
                    }
                    for (int mh = 0; mh < D / 128 && ok; ++mh) {
                        const uint32_t fi0 = fbase + (uint32_t)t * 2 * SLABS + SLABS + 2 * mh;
                        const uint32_t s0 = fi0 % NSLOT, s1 = (fi0 + 1) % NSLOT;  // s1 = s0 + 1
                        ok = mbar_wait_bounded(&bars[C::B_FULL + s0], (fi0 / NSLOT) & 1, P.fault,
                                               kFaultCopyTimeout) &&
                             mbar_wait_bounded(&bars[C::B_FULL + s1], ((fi0 + 1) / NSLOT) & 1,
                                               P.fault, kFaultCopyTimeout);
                        if (!ok) break;
                        fence_after_sync();
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk) {
                            // A = V^T: MN-major, the two 64-dim slabs one slot apart;
                            // B = P_hi for kk < 8, then P_lo
                            const int k8 = kk & 7;
                            const uint64_t a = smem_desc_sw128(
                                ring_a + s0 * C::SLOT_BYTES + k8 * 2048, C::SLOT_BYTES, 1024);
                            const uint64_t bdesc = smem_desc_sw128(
                                ps_a + (kk >> 3) * C::P_LO + (k8 >> 2) * C::P_SLAB + (k8 & 3) * 32,
                                16, 1024);
                            mma_bf16_ss(tmem + 2 * N + mh * N, a, bdesc, ID_PV,
                                        (t > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&bars[C::B_EMPTY + s0]);
                        mma_commit(&bars[C::B_EMPTY + s1]);
                    }
                    if (!ok) break;
                    mma_commit(&bars[C::B_PVDONE]);
                }
                gt += it.n_tiles;
            }
            if (!ok) *abort_flag = 1;
            // all issued MMAs complete before TMEM is released
            mma_commit(&bars[C::B_DRAIN]);
            mbar_wait_bounded(&bars[C::B_DRAIN], 0, P.fault, kFaultCopyTimeout);
        }
    } else {
        // ===================================================== softmax
        const int sw = warp - 2;           // softmax warp 0..3
        const int quad = warp & 3;         // TMEM lane quadrant of this warp
        const int lk = quad * 32 + lane;   // TMEM lane: key of S^T, dim row of O^T
        const int stid = tid - 64;         // 0..127
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t gt = 0, pvw = 0, fbase = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < T.items && ok; item += gridDim.x) {
            const TcItem it = tc_decode(T, item);
            const size_t bh = (size_t)it.b * P.Hkv + it.h;
            if (it.n_tiles == 0) {
                // no key in this chunk: empty result for every row
                for (int idx = stid; idx < it.rows * D; idx += 128) {
                    const int r = it.row0 + idx / D, d = idx % D;
                    const int i = r / P.G, gg = r - i * P.G;
                    const size_t orow =
                        ((size_t)it.b * P.q_len + i) * P.Hq + (size_t)it.h * P.G + gg;
                    if (P.splits == 1) {
                        P.out[orow * D + d] = __float2bfloat16_rn(0.f);
                        if (d == 0 && P.lse != nullptr) P.lse[orow] = NEG_INF;
                    } else {
                        const size_t prow = (bh * P.splits + it.split) * P.R + r;
                        P.part_acc[prow * D + d] = 0.f;
                        if (d == 0) {
                            P.part_ml[prow * 2] = NEG_INF;
                            P.part_ml[prow * 2 + 1] = 0.f;
                        }
                    }
                }
                continue;
            }
            for (int r = stid; r < N; r += 128) mref[r] = NEG_INF;
            float lpart[C::NCH];
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) lpart[c] = 0.f;
            named_sync_softmax();

            const int qp_i0 = it.cr.qp + it.i0;  // position of the item's first draft row
            for (int t = 0; t < it.n_tiles; ++t) {
                const uint32_t sb = gt & 1, use = gt >> 1;
                ok = !softmax_any(!mbar_wait_bounded(&bars[C::B_SFULL + sb], use & 1, P.fault,
                                                     kFaultCopyTimeout));
                if (!ok) break;
                fence_after_sync();
                const int j0 = it.cr.c_lo + kTcTileKeys * t;
                const int n_valid = min(kTcTileKeys, it.cr.c_hi - j0);
                const int j = j0 + lk;
                // packed rows [ra, rb) of this item whose window holds key j:
                // draft row i sees j iff p_i - W < j <= p_i, p_i = qp_i0 + i
                int ra = 0, rb = 0;
                if (lk < n_valid) {
                    const long long lo_i = (long long)j - qp_i0;
                    const long long hi_i = (long long)j + P.window - qp_i0;
                    const long long a = lo_i < 0 ? 0 : lo_i * P.G;
                    long long bnd = hi_i < 0 ? 0 : hi_i * P.G;
                    if (bnd > it.rows) bnd = it.rows;
                    ra = (int)(a < it.rows ? a : it.rows);
                    rb = (int)bnd;
                }
                const uint32_t scol = tl + sb * N;

                // pass 1: does any score exceed its row's reference by more than 2^8?
                bool flag = false;
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    uint32_t raw[CW];
                    tmem_load_cols<CW>(scol + c * CW, raw);
#pragma unroll
                    for (int e = 0; e < CW; ++e) {
                        const int r = c * CW + e;
                        const float v = (r >= ra && r < rb) ? __uint_as_float(raw[e]) * P.qk_scale
                                                            : NEG_INF;
                        flag |= v > mref[r] + 8.f;
                    }
                }
                const bool raise = softmax_any(flag);
                if (raise) {
                    // exact tile maximum per row, then raise the references
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c) {
                        uint32_t raw[CW];
                        tmem_load_cols<CW>(scol + c * CW, raw);
                        float v[CW];
#pragma unroll
                        for (int e = 0; e < CW; ++e) {
                            const int r = c * CW + e;
                            v[e] = (r >= ra && r < rb) ? __uint_as_float(raw[e]) * P.qk_scale
                                                       : NEG_INF;
                        }
                        const float m = lane_reduce<CW, true>(v);
                        if (lane < CW) red[sw * N + c * CW + lane] = m;
                    }
                    named_sync_softmax();
                    for (int r = stid; r < N; r += 128) {
                        const float tm = fmaxf(fmaxf(red[r], red[N + r]),
                                               fmaxf(red[2 * N + r], red[3 * N + r]));
                        const float mo = mref[r];
                        const float mn = fmaxf(mo, tm);
                        alpha[r] = (mn == mo) ? 1.f : fast_exp2(mo - mn);
                        mref[r] = mn;
                    }
                    named_sync_softmax();
                }
                // PV of the previous tile done: P buffer free, O^T stable
                if (t > 0) {
                    ok = !softmax_any(!mbar_wait_bounded(&bars[C::B_PVDONE], pvw & 1, P.fault,
                                                         kFaultCopyTimeout));
                    if (!ok) break;
                    ++pvw;
                    fence_after_sync();
                }
                if (raise && t > 0) {
#pragma unroll 1
                    for (int mh = 0; mh < D / 128; ++mh) {
#pragma unroll 1
                        for (int c0 = 0; c0 < N; c0 += 16) {
                            uint32_t o[16];
                            const uint32_t ocol = tl + 2 * N + mh * N + c0;
                            tmem_ld16(ocol, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha[c0 + e]);
                            tmem_st16(ocol, o);
                        }
                    }
                    tmem_wait_st();
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c) lpart[c] *= alpha[c * CW + (lane % CW)];
                }
                // pass 2: P = 2^(s - m_ref) into the swizzled P^T tile, row sums
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    uint32_t raw[CW];
                    tmem_load_cols<CW>(scol + c * CW, raw);
                    float pv[CW];
#pragma unroll
                    for (int e = 0; e < CW; ++e) {
                        const int r = c * CW + e;
                        const float m = mref[r];
                        const float mu = m == NEG_INF ? 0.f : m;
                        const float v = (r >= ra && r < rb) ? __uint_as_float(raw[e]) * P.qk_scale
                                                            : NEG_INF;
                        const float p = fast_exp2(v - mu);
                        const __nv_bfloat16 hi = __float2bfloat16_rn(p);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
                        const uint32_t off = (lk >> 6) * C::P_SLAB + sw128_offset(r, lk & 63);
                        *reinterpret_cast<__nv_bfloat16 *>(ps + off) = hi;
                        *reinterpret_cast<__nv_bfloat16 *>(ps + C::P_LO + off) = lo;
                        // the sum weights exactly what the two MMAs weight
                        pv[e] = __bfloat162float(hi) + __bfloat162float(lo);
                    }
                    lpart[c] += lane_reduce<CW, false>(pv);
                }
                fence_before_sync();
                mbar_arrive(&bars[C::B_SFREE + sb]);
                // Keys past the chunk's end: their V rows are zeroed so that
                // 0 * (whatever the cache holds there) cannot reach O; the
                // TMA box always spans 128 keys.
                if (n_valid < kTcTileKeys) {
                    const uint32_t fv = fbase + (uint32_t)t * 2 * SLABS + SLABS;
                    bool vok = true;
#pragma unroll
                    for (int s = 0; s < SLABS; ++s)
                        vok = vok && mbar_wait_bounded(&bars[C::B_FULL + (fv + s) % NSLOT],
                                                       ((fv + s) / NSLOT) & 1, P.fault,
                                                       kFaultCopyTimeout);
                    ok = !softmax_any(!vok);
                    if (!ok) break;
                    if (lk >= n_valid) {
#pragma unroll
                        for (int s = 0; s < SLABS; ++s) {
                            uint4 *row = reinterpret_cast<uint4 *>(
                                ring + ((fv + s) % NSLOT) * C::SLOT_BYTES + lk * 128);
#pragma unroll
                            for (int q = 0; q < 8; ++q) row[q] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_proxy_async_smem();
                fence_before_sync();
                mbar_arrive(&bars[C::B_PFULL]);
                ++gt;
            }
            if (!ok) break;

            // -------------------------------------------------- epilogue
            ok = !softmax_any(!mbar_wait_bounded(&bars[C::B_PVDONE], pvw & 1, P.fault,
                                                 kFaultCopyTimeout));
            if (!ok) break;
            ++pvw;
            fence_after_sync();
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
                if (lane < CW) red[sw * N + c * CW + lane] = lpart[c];
            named_sync_softmax();
            for (int r = stid; r < N; r += 128)
                lsum[r] = (red[r] + red[N + r]) + (red[2 * N + r] + red[3 * N + r]);
            named_sync_softmax();
#pragma unroll 1
            for (int mh = 0; mh < D / 128; ++mh) {
                const int d = mh * 128 + lk;
#pragma unroll 1
                for (int c0 = 0; c0 < N; c0 += 16) {
                    if (c0 >= it.rows) break;
                    uint32_t o[16];
                    tmem_ld16(tl + 2 * N + mh * N + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = c0 + e;
                        if (r >= it.rows) break;
                        const int rg = it.row0 + r;
                        const float ov = __uint_as_float(o[e]);
                        if (P.splits == 1) {
                            const int i = rg / P.G, gg = rg - i * P.G;
                            const size_t orow =
                                ((size_t)it.b * P.q_len + i) * P.Hq + (size_t)it.h * P.G + gg;
                            const float l = lsum[r];
                            P.out[orow * D + d] = __float2bfloat16_rn(l > 0.f ? ov / l : 0.f);
                        } else {
                            const size_t prow = (bh * P.splits + it.split) * P.R + rg;
                            P.part_acc[prow * D + d] = ov;
                        }
                    }
                }
            }
            for (int r = stid; r < it.rows; r += 128) {
                const int rg = it.row0 + r;
                const float l = lsum[r], m = mref[r];
                if (P.splits == 1) {
                    if (P.lse != nullptr) {
                        const int i = rg / P.G, gg = rg - i * P.G;
                        const size_t orow =
                            ((size_t)it.b * P.q_len + i) * P.Hq + (size_t)it.h * P.G + gg;
                        P.lse[orow] = l > 0.f ? (m + __log2f(l)) * kLn2 : NEG_INF;
                    }
                } else {
                    const size_t prow = (bh * P.splits + it.split) * P.R + rg;
                    P.part_ml[prow * 2] = l > 0.f ? m : NEG_INF;
                    P.part_ml[prow * 2 + 1] = l;
                }
            }
            fence_before_sync();
            mbar_arrive(&bars[C::B_OFREE]);
            fbase += (uint32_t)it.n_tiles * 2 * SLABS;
            named_sync_softmax();
        }
        if (!ok) *abort_flag = 1;
    }

    // ---------------------------------------------------------- teardown
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace swa
