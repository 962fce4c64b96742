// Tensor-core (tcgen05) split-KV kernel on CTA pairs, with query rows as the
// MMA's M dimension, for sliding-window verify attention.
//
// A cluster of two CTAs (ranks 0 and 1, on two SMs) takes a work item of up
// to 2 x 128 packed rows (sequence, KV head, key chunk, pair row tile); rank
// r holds the rows 128 r .. 128 r + 127 of it.  For every tile of 128 keys
//
//   S[256 rows x 128 keys] = Q[256 x D] . K_tile^T              (TMEM, fp32)
//   O[256 rows x D]       += P_hi . V_tile + P_lo . V_tile      (TMEM, fp32)
//
// as 2-CTA MMAs (M = 256) issued by rank 0.  Each CTA holds its own 128 rows
// of Q, keys 64 r .. 64 r + 63 of every K tile and head dims (D / 2) r ..
// (D / 2) (r + 1) - 1 of every V tile, and receives S, P and O of its own
// rows in its TMEM.  So every K/V byte is read once for all 256 rows, and a
// CTA's ring holds half tiles: four 32 KB slots where the one-CTA rows-major
// kernel has two 64 KB ones (at head_dim 256).
//
// Rank 0's producer posts the bytes of both CTAs on its ring and Q barriers
// and rank 1's copies complete there; the MMA commits arrive on the barrier
// of that name in both CTAs (slot free, scores ready, PV done).  The softmax
// of each CTA is the one-CTA rows-major kernel's (a thread pair per row, P
// written back to TMEM as bf16 hi/lo); its "P ready" and "O read" arrivals,
// one per warp, go to rank 0's barriers.  The last V tile of an item whose
// keys end inside a 16-key MMA step has the rows past the end zeroed before
// the MMA reads them (P is 0 there, but cache rows past a sequence's length
// may hold anything, NaN included): rank 0 zeroes its half in the MMA warp;
// rank 1 lands that tile on a barrier of its own, zeroes its half in warp 1
// and then arrives on rank 0's barrier of that slot.
//
// Warp roles (320 threads in each CTA):
//   warp 0      TMA producer (lane 0)
//   warp 1      TMEM owner; rank 0: the MMA issuer (one lane); rank 1: the
//               zeroing of its partial V tiles
//   warps 2..9  softmax / epilogue of the CTA's rows: warp w owns TMEM lanes
//               32 (w % 4).. and key half (w - 2) / 4 of every tile
//               (head-dim half of the output)
//
// TMEM (512 columns in each CTA): S/P buffers at columns 0 and 128, O at 256.
// Contiguous caches only (no block table, no fused append), head_dim 256.
// Every wait is bounded; a wait that gives up sets the fault word and the
// roles leave their loops; both CTAs then meet at a cluster barrier before
// TMEM is freed, so neither leaves while the other may still reach its
// shared memory.
#pragma once

#include "swa_tc.cuh"

namespace swa {

constexpr int kPairThreads = 320;
constexpr int kPairSlots = 4;

// V tensor maps of the pair kernel: boxes of D / 2 head dims (half the slabs),
// started at slab (D / 128) r by rank r; laid out as the full maps' boxes.
struct PairMaps {
    CUtensorMap vh_atoms[4];  // 4D boxes of 16, 8, 4, 2 atoms
    CUtensorMap vh_atom;      // 3D box of one atom (rows past the cache are zero-filled)
    // out [B * q_len rows][Hq][D] as 3D (x = head dim, y = query head, z = row),
    // a box of 32 dims x G heads x 32 / G rows (one softmax warp's 32 packed
    // rows), 64-byte swizzled: valid when out_ok (G divides 32)
    CUtensorMap out;
    int out_ok;
};

template <int D, int NT>
struct PairCfg {
    static constexpr int SLABS = D / 64;
    static constexpr int K_ATOM = SLABS * 1024;        // 8 keys x D
    static constexpr int V_ATOM = (SLABS / 2) * 1024;  // 8 keys x D / 2
    static constexpr int HALF_KEYS = kTcTileKeys / 2;
    static constexpr int SLOT_BYTES = (HALF_KEYS / 8) * K_ATOM;  // a K or a V half tile
    static constexpr int QR = 128;
    static constexpr int Q_SLAB = QR * 128;  // 128 rows x 64 dims
    static constexpr int Q_BUF = SLABS * Q_SLAB;
    static constexpr int Q_OFF = 0;
    static constexpr int RING_OFF = Q_BUF;
    static constexpr int META_OFF = RING_OFF + NT * SLOT_BYTES;  // TcItem [kTcMetaItems]
    // the softmax pairs' exchange: half maxima [tile parity][quadrant][half][lane],
    // half row sums [quadrant][half][lane]
    static constexpr int XM_OFF = (META_OFF + kTcMetaItems * (int)sizeof(TcItem) + 15) & ~15;
    static constexpr int XL_OFF = XM_OFF + 2 * 4 * 2 * 32 * 4;
    // (1024-byte aligned: the 64-byte swizzle of the output's tensor store
    // follows the shared-memory address)
    static constexpr int STG_OFF = (XL_OFF + 4 * 2 * 32 * 4 + 1023) & ~1023;
    static constexpr int STG_NEED = 8 * 2048;  // output staging, 2 KB per softmax warp
    static constexpr int BAR_OFF = STG_OFF + STG_NEED;
    // ring full / empty [NT], rank 1's own landing of a V half to zero [NT],
    // rank 1's zeroing done [NT] (on rank 0), q full / empty, s full [2],
    // s free [2], p full [2], pv done [2], o free, drain
    static constexpr int B_FULL = 0, B_EMPTY = NT, B_VLOC = 2 * NT, B_FIX = 3 * NT,
                         B_QFULL = 4 * NT, B_QEMPTY = B_QFULL + 1, B_SFULL = B_QEMPTY + 1,
                         B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PVDONE = B_PFULL + 2,
                         B_OFREE = B_PVDONE + 2, B_DRAIN = B_OFREE + 1, NBARS = B_DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base
    static constexpr int END = MISC_OFF + 16;
    static constexpr int SMEM_BYTES = END + 1024;  // slack for 1024-byte alignment
    static constexpr int O_COL = 256;
    static constexpr int TMEM_COLS = 512;
    static_assert(D == 256, "the pair kernel is built for head_dim 256");
    static_assert(SLOT_BYTES == (kTcTileKeys / 8) * V_ATOM, "K and V half tiles fill a slot");
    static_assert(O_COL + D <= TMEM_COLS, "TMEM");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(RING_OFF % 1024 == 0 && SLOT_BYTES % 1024 == 0, "swizzled tiles");
    static_assert(STG_OFF % 16 == 0 && BAR_OFF % 8 == 0 && META_OFF % 8 == 0, "alignment");
};

// The items of this CTA's pair (the cluster blockIdx.x / 2 of gridDim.x / 2),
// round-robin: items c, c + pairs, c + 2 pairs, ...
__device__ __forceinline__ int pair_items(const TcParams &T) {
    const int c = (int)(blockIdx.x >> 1), n = (int)(gridDim.x >> 1);
    return (T.items - c + n - 1) / n;
}
__device__ __forceinline__ int pair_item(int j) {
    return (int)(blockIdx.x >> 1) + j * (int)(gridDim.x >> 1);
}

// Work item `item` as rank `rank` sees it: the pair's key range (the windows
// of all its rows, so both CTAs walk the same tiles) and this CTA's rows.
// T.rows_per_tile / T.q_rows_per_tile are one CTA's packed / draft rows.
__device__ __forceinline__ TcItem pair_decode_global(const TcParams &T, int item, uint32_t rank) {
    const AttnParams &P = T.a;
    TcItem it;
    int rest = item;
    it.rt = rest % P.row_tiles;
    rest /= P.row_tiles;
    it.split = rest % P.splits;
    rest /= P.splits;
    it.h = rest % P.Hkv;
    it.b = rest / P.Hkv;
    const int prow0 = it.rt * 2 * T.rows_per_tile;
    const int prows = min(P.R - prow0, 2 * T.rows_per_tile);
    it.row0 = prow0 + (int)rank * T.rows_per_tile;
    it.rows = max(0, min(P.R - it.row0, T.rows_per_tile));
    const int pi0 = it.rt * 2 * T.q_rows_per_tile;
    it.i0 = pi0 + (int)rank * T.q_rows_per_tile;
    it.cr = chunk_range(P, it.b, it.split, pi0, (prow0 + prows - 1) / P.G);
    it.t0 = it.cr.c_lo;
    const int nk = it.cr.c_hi - it.t0;
    it.n_tiles = it.cr.c_hi > it.cr.c_lo ? (nk + kTcTileKeys - 1) / kTcTileKeys : 0;
    return it;
}

__device__ __forceinline__ TcItem pair_decode(const TcParams &T, int j, uint32_t rank,
                                              const TcItem *meta) {
    if (j < kTcMetaItems) return meta[j];
    return pair_decode_global(T, pair_item(j), rank);
}

// Keys of a tile's K half held by rank `rank` (of n_valid keys in the tile).
__device__ __forceinline__ int pair_half_keys(int n_valid, uint32_t rank) {
    const int n = n_valid - kTcTileKeys / 2 * (int)rank;
    return n < 0 ? 0 : (n > kTcTileKeys / 2 ? kTcTileKeys / 2 : n);
}

// A run of cache rows [y, y + 8 whole (+ 8 if partial)) into atoms of AB
// bytes at dst: whole atoms through the 4D boxes (m4[0..3]: 16, 8, 4, 2
// atoms), a single or a partial atom through the 3D one-atom box; z is the
// first head-dim slab; completion on `bar` (shared::cluster address).
template <int AB>
__device__ __forceinline__ void pair_atom_run(const CUtensorMap *m4, const CUtensorMap *m1, int y,
                                              int z, int whole, bool partial, uint8_t *dst,
                                              uint32_t bar, uint64_t policy) {
    using namespace tc;
    int w = 0;
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
        const int na = 16 >> bi;
        if (whole & na) {
            tma_load_4d_pair(dst + w * AB, &m4[bi], 0, y + 8 * w, z, 0, bar, policy);
            w += na;
        }
    }
    if (whole & 1) {
        tma_load_3d_pair(dst + w * AB, m1, 0, y + 8 * w, z, bar, policy);
        ++w;
    }
    if (partial) tma_load_3d_pair(dst + w * AB, m1, 0, y + 8 * w, z, bar, policy);
}

// Bytes one CTA's copies of fill kv (0 K, 1 V) of a tile with n_valid keys
// deliver: K, its key half; V, all keys of its head-dim half.
template <class C>
__device__ __forceinline__ uint32_t pair_fill_bytes(int kv, int n_valid, uint32_t rank) {
    return kv ? (uint32_t)((n_valid + 7) >> 3) * C::V_ATOM
              : (uint32_t)((pair_half_keys(n_valid, rank) + 7) >> 3) * C::K_ATOM;
}

// Zero rows [nv, 16 ceil(nv / 16)) of a V half tile ([atom][slab][8 rows][128
// bytes], D / 128 slabs) so the last 16-key MMA step reads zeros past the
// keys; the whole warp, then a proxy fence for the tensor core's reads.
template <class C>
__device__ __forceinline__ void pair_zero_v_tail(uint8_t *vt, int nv, int lane) {
    const int end = (nv + 15) & ~15;
    const int q = lane & 7;
#pragma unroll
    for (int s = 0; s < C::SLABS / 2; ++s) {
#pragma unroll
        for (int r4 = 0; r4 < 16; r4 += 4) {
            const int r = nv + (lane >> 3) + r4;
            if (r < end)
                reinterpret_cast<uint4 *>(vt + (r >> 3) * C::V_ATOM + s * 1024 + (r & 7) * 128)[q] =
                    make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    __syncwarp();
}

template <int D, int NT>
__global__ void __launch_bounds__(kPairThreads, 1)
    swa_pair_kernel(const __grid_constant__ TcParams T, const __grid_constant__ TcMaps M,
                    const __grid_constant__ PairMaps PM) {
    using C = PairCfg<D, NT>;
    using namespace tc;
    constexpr int SLABS = C::SLABS;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const AttnParams &P = T.a;

    extern __shared__ uint8_t smem_raw[];
    // the same offset in both CTAs: the MMAs address rank 1's operands by
    // rank 0's shared-memory offsets
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    uint8_t *qs = sm + C::Q_OFF;
    uint8_t *ring = sm + C::RING_OFF;
    TcItem *meta = reinterpret_cast<TcItem *>(sm + C::META_OFF);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::MISC_OFF);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank();
    // quadrants (warps of 32 rows) that hold packed rows of an item
    const int act_q = (T.rows_per_tile + 31) >> 5;

    // ---------------------------------------------------------------- setup
    if (warp == 0 && lane < 6) {
        const CUtensorMap *mp = lane < 2    ? &M.k_atoms[lane + 1]
                                : lane == 2 ? &M.k_atom
                                : lane == 3 ? &PM.vh_atoms[0]
                                : lane == 4 ? &PM.vh_atom
                                            : &M.q;
        prefetch_tmap(mp);
    }
    if (tid == 0) {
        for (int i = 0; i < NT; ++i) {
            mbar_init(&bars[C::B_FULL + i], 1);
            mbar_init(&bars[C::B_EMPTY + i], 1);
            mbar_init(&bars[C::B_VLOC + i], 1);
            mbar_init(&bars[C::B_FIX + i], 1);
        }
        mbar_init(&bars[C::B_QFULL], 1);
        mbar_init(&bars[C::B_QEMPTY], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[C::B_SFULL + i], 1);
            mbar_init(&bars[C::B_SFREE + i], 1);
            mbar_init(&bars[C::B_PFULL + i], 2 * 2 * act_q);  // a warp per quadrant and half, both CTAs
            mbar_init(&bars[C::B_PVDONE + i], 1);
        }
        mbar_init(&bars[C::B_OFREE], 2 * 2 * act_q);
        mbar_init(&bars[C::B_DRAIN], 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    fence_before_sync();
    // both CTAs' barriers initialised before either reaches the other's
    cluster_sync();
    fence_after_sync();
    grid_dep_wait();
    grid_dep_trigger();
    const int n_items = pair_items(T);
    for (int j = tid; j < kTcMetaItems; j += kPairThreads)
        if (j < n_items) meta[j] = pair_decode_global(T, pair_item(j), rank);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ======================================================= producer
        // For every item: K tile 0, this CTA's Q rows, V tile 0, K 1, V 1, ...
        // Fill f (two per tile, K then V) goes to ring slot f % NT.
        if (lane == 0) {
            const uint64_t policy =
                P.row_tiles > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
            const uint32_t full0 = cluster_addr(&bars[C::B_FULL], 0);
            const uint32_t qfull0 = cluster_addr(&bars[C::B_QFULL], 0);
            const int z_v = (int)rank * (SLABS / 2);
            uint32_t f = 0, k = 0;  // fills, items with keys
            bool ok = true;
            for (int j = 0; j < n_items && ok; ++j) {
                const TcItem it = pair_decode(T, j, rank, meta);
                if (it.n_tiles == 0) continue;
                const int last_keys = it.cr.c_hi - it.t0 - kTcTileKeys * (it.n_tiles - 1);
                for (int t = 0; t < it.n_tiles && ok; ++t) {
                    const int p = it.t0 + kTcTileKeys * t;
                    const int n_valid = min(kTcTileKeys, it.cr.c_hi - p);
                    for (int kv = 0; kv < 2 && ok; ++kv) {
                        if (t == 0 && kv == 1) {
                            // this CTA's Q rows, after the item's first K tile
                            ok = mbar_wait_bounded(&bars[C::B_QEMPTY], (k & 1) ^ 1, P.fault,
                                                   kFaultCopyTimeout, P.wait_limit);
                            if (!ok) break;
                            // both CTAs' boxes: SLABS x (G x q_rows_per_tile) rows x 128 B
                            if (rank == 0)
                                mbar_arrive_expect_tx(&bars[C::B_QFULL],
                                                      2u * SLABS * (uint32_t)T.rows_per_tile * 128u);
                            for (int s = 0; s < SLABS; ++s)
                                tma_load_3d_pair(qs + s * C::Q_SLAB, &M.q, 64 * s, it.h * P.G,
                                                 it.b * P.q_len + it.i0, qfull0, policy);
                            ++k;
                        }
                        const uint32_t slot = f % NT, use = f / NT;
                        ok = mbar_wait_bounded(&bars[C::B_EMPTY + slot], (use & 1) ^ 1, P.fault,
                                               kFaultCopyTimeout, P.wait_limit);
                        if (!ok) break;
                        // the last V tile with keys ending inside a 16-key step:
                        // rank 1 lands its half on VLOC and zeroes the tail itself
                        const bool fix = kv == 1 && t == it.n_tiles - 1 && (last_keys & 15) != 0;
                        const uint32_t own = pair_fill_bytes<C>(kv, n_valid, rank);
                        if (rank == 0)
                            mbar_arrive_expect_tx(
                                &bars[C::B_FULL + slot],
                                own + (fix ? 0u : pair_fill_bytes<C>(kv, n_valid, 1)));
                        uint32_t bar = full0 + 8 * slot;
                        if (rank == 1 && fix) {
                            mbar_arrive_expect_tx(&bars[C::B_VLOC + slot], own);
                            bar = smem_u32(&bars[C::B_VLOC + slot]);
                        }
                        // (tests of the bounded waits: this fill's copies are never issued)
                        if (!(P.withhold_fill == (int)f && blockIdx.x == 0)) {
                            uint8_t *dst = ring + slot * C::SLOT_BYTES;
                            if (kv == 0) {
                                const int n = pair_half_keys(n_valid, rank);
                                if (n > 0)
                                    pair_atom_run<C::K_ATOM>(
                                        M.k_atoms, &M.k_atom,
                                        (int)cache_row(P, it.b, it.h, p + kTcTileKeys / 2 * (int)rank), 0,
                                        n >> 3, (n & 7) != 0, dst, bar, policy);
                            } else {
                                pair_atom_run<C::V_ATOM>(PM.vh_atoms, &PM.vh_atom,
                                                         (int)cache_row(P, it.b, it.h, p), z_v,
                                                         n_valid >> 3, (n_valid & 7) != 0, dst,
                                                         bar, policy);
                            }
                        }
                        ++f;
                    }
                }
            }
            if (rank == 0) {
                // every copy of both CTAs landed (rank 0's ring and Q barriers
                // count rank 1's bytes too, but for the V halves rank 1 zeroes,
                // which its warp 1 waits for) before the CTAs exit
#pragma unroll
                for (int s2 = 0; s2 < NT; ++s2) {
                    const uint32_t uses = f / NT + ((uint32_t)s2 < f % NT ? 1u : 0u);
                    if (uses > 0)
                        mbar_wait_bounded(&bars[C::B_FULL + s2], (uses - 1) & 1, P.fault,
                                          kFaultCopyTimeout, P.wait_limit);
                }
                if (k > 0)
                    mbar_wait_bounded(&bars[C::B_QFULL], (k - 1) & 1, P.fault, kFaultCopyTimeout,
                                      P.wait_limit);
            }
        }
    } else if (warp == 1 && rank == 1) {
        // ============================== rank 1: zero the tails of its V halves
        uint32_t g = 0, par = 0;  // tiles so far, VLOC wait parities per slot
        for (int j = 0; j < n_items; ++j) {
            const TcItem it = pair_decode(T, j, rank, meta);
            if (it.n_tiles == 0) continue;
            g += (uint32_t)it.n_tiles;
            const int last_keys = it.cr.c_hi - it.t0 - kTcTileKeys * (it.n_tiles - 1);
            if ((last_keys & 15) == 0) continue;
            const uint32_t vslot = (2 * (g - 1) + 1) % NT;
            const bool ok = __all_sync(
                0xffffffffu, mbar_wait_bounded(&bars[C::B_VLOC + vslot], (par >> vslot) & 1,
                                               P.fault, kFaultCopyTimeout, P.wait_limit));
            if (!ok) break;
            par ^= 1u << vslot;
            pair_zero_v_tail<C>(ring + vslot * C::SLOT_BYTES, last_keys, lane);
            if (lane == 0) mbar_arrive_cluster(cluster_addr(&bars[C::B_FIX + vslot], 0));
        }
    } else if (warp == 1) {
        // ================================================== rank 0: MMA
        // Two cursors over the tile sequence: S = Q K^T of the next tile and
        // O += P_hi V + P_lo V of the oldest tile whose P is in TMEM, each
        // issued as soon as its operands are there in both CTAs (S at most
        // one tile ahead of PV).  The whole warp runs the loop; lane 0 issues.
        const bool leader = lane == 0;
        constexpr uint32_t ID_S = idesc_bf16_f32(256, 128, 0, 0);
        constexpr uint32_t ID_O = idesc_bf16_f32(256, D, 0, 1);
        const uint32_t ring_a = smem_u32(ring);
        const uint32_t qs_a = smem_u32(qs);
        struct Cursor {
            int j, t, n_tiles;
            int last_keys;  // keys of the item's last tile
            uint32_t k, g;
            bool valid;
        };
        auto seek = [&](Cursor &c) {
            for (; c.j < n_items; ++c.j) {
                const TcItem it = pair_decode(T, c.j, rank, meta);
                if (it.n_tiles > 0) {
                    c.n_tiles = it.n_tiles;
                    c.last_keys = it.cr.c_hi - it.t0 - kTcTileKeys * (it.n_tiles - 1);
                    c.t = 0;
                    c.valid = true;
                    return;
                }
            }
            c.valid = false;
        };
        auto advance = [&](Cursor &c) {
            ++c.g;
            if (++c.t < c.n_tiles) return;
            ++c.k;
            ++c.j;
            seek(c);
        };
        Cursor qc{0, 0, 0, 0, 0u, 0u, false};
        seek(qc);
        Cursor pc = qc;
        uint32_t fixpar = 0;  // FIX wait parities per slot
        long long idle_since = clock64();
        while (pc.valid) {
            bool progressed = false;
            // ---- PV of tile pc.g (its S was issued before)
            if (pc.g < qc.g || !qc.valid) {
                const uint32_t sb = pc.g & 1;
                const uint32_t vf = 2 * pc.g + 1, vslot = vf % NT;
                const bool last = pc.t == pc.n_tiles - 1;
                const int nv = last ? pc.last_keys : kTcTileKeys;
                const bool fix = (nv & 15) != 0;
                bool ready = mbar_test(&bars[C::B_PFULL + sb], (pc.g >> 1) & 1);
                if (ready && pc.t == 0) ready = mbar_test(&bars[C::B_OFREE], (pc.k & 1) ^ 1);
                ready = ready && mbar_test(&bars[C::B_FULL + vslot], (vf / NT) & 1);
                if (ready && fix) ready = mbar_test_cluster(&bars[C::B_FIX + vslot], (fixpar >> vslot) & 1);
                ready = __shfl_sync(0xffffffffu, ready, 0) != 0;  // one decision for the warp
                if (ready) {
                    fence_after_sync();
                    if (fix) {
                        fixpar ^= 1u << vslot;
                        pair_zero_v_tail<C>(ring + vslot * C::SLOT_BYTES, nv, lane);
                    }
                    if (leader) {
                        // B = V, MN-major: 64-dim blocks one slab (1024 B) apart,
                        // 8-key groups one atom apart; a 16-key step is two atoms
                        const uint64_t vbase =
                            smem_desc_sw128(ring_a + vslot * C::SLOT_BYTES, 1024, C::V_ATOM);
                        const uint32_t d_t = tmem + C::O_COL;
                        const uint32_t p_t = tmem + sb * 128;  // P_hi; P_lo at +64
                        const uint32_t acc0 = pc.t > 0 ? 1u : 0u;
                        const int steps = (nv + 15) >> 4;
                        for (int k8 = 0; k8 < steps; ++k8)
                            mma_bf16_ts_pair(d_t, p_t + k8 * 8,
                                             vbase + (uint64_t)(k8 * (2 * C::V_ATOM >> 4)), ID_O,
                                             (acc0 | (uint32_t)k8) != 0);
                        for (int k8 = 0; k8 < steps; ++k8)
                            mma_bf16_ts_pair(d_t, p_t + 64 + k8 * 8,
                                             vbase + (uint64_t)(k8 * (2 * C::V_ATOM >> 4)), ID_O, 1u);
                        mma_commit_pair_both(&bars[C::B_EMPTY + vslot]);
                        mma_commit_pair(&bars[C::B_SFREE + sb]);
                        mma_commit_pair_both(&bars[C::B_PVDONE + sb]);
                    }
                    __syncwarp();
                    advance(pc);
                    progressed = true;
                }
            }
            // ---- S of tile qc.g, at most one tile ahead of the PV cursor
            if (qc.valid && qc.g <= pc.g + 1) {
                const uint32_t sb = qc.g & 1;
                const uint32_t kf = 2 * qc.g, kslot = kf % NT;
                bool ready = mbar_test(&bars[C::B_SFREE + sb], ((qc.g >> 1) & 1) ^ 1) &&
                             mbar_test(&bars[C::B_QFULL], qc.k & 1) &&
                             mbar_test(&bars[C::B_FULL + kslot], (kf / NT) & 1);
                ready = __shfl_sync(0xffffffffu, ready, 0) != 0;
                if (ready) {
                    fence_after_sync();
                    if (leader) {
                        // A = Q, K-major: 8-row groups 1024 B apart, slab s at
                        // s * Q_SLAB; B = K, K-major: 8-key groups one atom apart,
                        // slab s at s * 1024
                        const uint64_t qbase = smem_desc_sw128(qs_a, 16, 1024);
                        const uint64_t kbase =
                            smem_desc_sw128(ring_a + kslot * C::SLOT_BYTES, 16, C::K_ATOM);
#pragma unroll
                        for (int s = 0; s < SLABS; ++s) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_bf16_ss_pair(tmem + sb * 128,
                                                 qbase + (uint64_t)(s * (C::Q_SLAB >> 4) + kk * 2),
                                                 kbase + (uint64_t)(s * 64 + kk * 2), ID_S,
                                                 (s | kk) != 0);
                        }
                        mma_commit_pair_both(&bars[C::B_EMPTY + kslot]);
                        mma_commit_pair_both(&bars[C::B_SFULL + sb]);
                        if (qc.t == qc.n_tiles - 1) mma_commit_pair_both(&bars[C::B_QEMPTY]);
                    }
                    __syncwarp();
                    advance(qc);
                    progressed = true;
                }
            }
            if (progressed) {
                idle_since = clock64();
            } else if (clock64() - idle_since > P.wait_limit) {
                atomicOr(P.fault, kFaultCopyTimeout);
                break;
            }
        }
        // all issued MMAs complete before either CTA leaves or TMEM is freed
        if (leader) {
            mma_commit_pair(&bars[C::B_DRAIN]);
            mbar_wait_bounded(&bars[C::B_DRAIN], 0, P.fault, kFaultCopyTimeout, P.wait_limit);
        }
        __syncwarp();
    } else {
        // ===================================================== softmax
        const int quad = warp & 3;         // TMEM lane quadrant = packed rows 32 quad ..
        const int half = (warp - 2) >> 2;  // key half of each tile, head-dim half of O
        if (quad < act_q) {
            const int r = quad * 32 + lane;  // packed row within this CTA's rows
            const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
            float *xm = reinterpret_cast<float *>(sm + C::XM_OFF);
            float *xl = reinterpret_cast<float *>(sm + C::XL_OFF) + (quad * 2) * 32 + lane;
            const int kh = 64 * half;  // first key of this thread's half
            constexpr int DH = D / 2;  // head dims of this thread's half of O
            const float sc = P.qk_scale;
            const uint32_t pfull0 = cluster_addr(&bars[C::B_PFULL], 0);
            const uint32_t ofree0 = cluster_addr(&bars[C::B_OFREE], 0);
            // the pair of warps of this quadrant (64 threads), barrier 1 + quad
            auto pair_sync = [&]() {
                asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
            };
            uint32_t g = 0;
            bool ok = true;
            for (int j = 0; j < n_items && ok; ++j) {
                const TcItem it = pair_decode(T, j, rank, meta);
                const bool live = r < it.rows;
                const int rg = it.row0 + r;  // packed row of the (sequence, KV head)
                const int i = rg / P.G, gg = rg - i * P.G;
                const size_t orow =
                    ((size_t)it.b * P.q_len + i) * P.Hq + (size_t)it.h * P.G + gg;
                const size_t prow =
                    (((size_t)it.b * P.Hkv + it.h) * P.splits + it.split) * P.R + rg;
                if (it.n_tiles == 0) {
                    // no key in this chunk: empty result (each half its dims)
                    if (live) {
                        if (P.splits == 1) {
                            for (int d = half * DH; d < (half + 1) * DH; d += 8)
                                *reinterpret_cast<uint4 *>(P.out + orow * D + d) =
                                    make_uint4(0, 0, 0, 0);
                            if (half == 0 && P.lse != nullptr) P.lse[orow] = NEG_INF;
                        } else {
                            for (int d = half * DH; d < (half + 1) * DH; d += 4)
                                *reinterpret_cast<float4 *>(P.part_acc + prow * D + d) =
                                    make_float4(0.f, 0.f, 0.f, 0.f);
                            if (half == 0) {
                                P.part_ml[prow * 2] = NEG_INF;
                                P.part_ml[prow * 2 + 1] = 0.f;
                            }
                        }
                    }
                    continue;
                }
                // keys of the chunk this row sees: [jlo, jhi]; draft row i sits at
                // position q_pos + i and sees (p - W, p]
                const long long pp = (long long)it.cr.qp + i;
                long long jlo = pp - P.window + 1, jhi = pp;
                if (jlo < it.cr.c_lo) jlo = it.cr.c_lo;
                if (jhi > it.cr.c_hi - 1) jhi = it.cr.c_hi - 1;
                if (!live) {
                    jlo = 1;
                    jhi = 0;
                }
                float mref = kNoRef, lsum = 0.f;
                for (int t = 0; t < it.n_tiles; ++t, ++g) {
                    const uint32_t sb = g & 1;
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[C::B_SFULL + sb], (g >> 1) & 1,
                                                                   P.fault, kFaultCopyTimeout, P.wait_limit));
                    if (!ok) break;
                    fence_after_sync();
                    // this thread's 64 scores (keys kh .. kh + 63 of the tile), masked
                    // to the row's keys, in log2 units
                    const long long j0 = (long long)it.t0 + (long long)kTcTileKeys * t + kh;
                    const long long ca_l = jlo - j0, cb_l = jhi - j0;
                    const int ca = ca_l < 0 ? 0 : (ca_l > 64 ? 64 : (int)ca_l);
                    const int cb = cb_l < -1 ? -1 : (cb_l > 63 ? 63 : (int)cb_l);
                    uint32_t sraw[64];
                    tmem_ld32(tl + sb * 128 + kh, *reinterpret_cast<uint32_t(*)[32]>(sraw));
                    tmem_ld32(tl + sb * 128 + kh + 32, *reinterpret_cast<uint32_t(*)[32]>(sraw + 32));
                    tmem_wait_ld();
                    float m4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
                    if (ca == 0 && cb == 63) {
                        const uint64_t sc2 = f2_pack(sc, sc);
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            float x0, x1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(sraw[c]), __uint_as_float(sraw[c + 1])),
                                             sc2),
                                      x0, x1);
                            sraw[c] = __float_as_uint(x0);
                            sraw[c + 1] = __float_as_uint(x1);
                            m4[(c >> 1) & 3] = fmax3(m4[(c >> 1) & 3], x0, x1);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            const float x0 =
                                (c >= ca && c <= cb) ? __uint_as_float(sraw[c]) * sc : NEG_INF;
                            const float x1 =
                                (c + 1 >= ca && c + 1 <= cb) ? __uint_as_float(sraw[c + 1]) * sc : NEG_INF;
                            sraw[c] = __float_as_uint(x0);
                            sraw[c + 1] = __float_as_uint(x1);
                            m4[(c >> 1) & 3] = fmax3(m4[(c >> 1) & 3], x0, x1);
                        }
                    }
                    // the pair's common tile maximum (one exchange per tile, buffers
                    // alternate with the tile so a slow partner is never overwritten)
                    float *xmt = xm + ((sb * 4 + quad) * 2) * 32 + lane;
                    xmt[half * 32] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                    pair_sync();
                    const float mt = fmaxf(xmt[0], xmt[32]);
                    // raise the reference when a score exceeds it by 2^8 (always on
                    // the row's first scores); O of the item's earlier tiles is then
                    // rescaled in TMEM (each half its head dims) once their PVs are done
                    const bool raise = mt > mref + 8.f;
                    if (__any_sync(0xffffffffu, raise && t > 0)) {
                        const uint32_t gp = g - 1;
                        ok = __all_sync(0xffffffffu,
                                        mbar_wait_bounded(&bars[C::B_PVDONE + (gp & 1)], (gp >> 1) & 1,
                                                          P.fault, kFaultCopyTimeout, P.wait_limit));
                        if (!ok) break;
                        fence_after_sync();
                        const float al = raise ? fast_exp2(mref - mt) : 1.f;
                        const uint32_t oc = tl + C::O_COL + half * DH;
#pragma unroll 1
                        for (int c0 = 0; c0 < DH; c0 += 32) {
                            uint32_t o[32];
                            tmem_ld32(oc + c0, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * al);
                            tmem_st32(oc + c0, o);
                        }
                        tmem_wait_st();
                    }
                    if (raise) {
                        lsum *= fast_exp2(mref - mt);
                        mref = mt;
                    }
                    // P = 2^(s - m_ref) for this half's keys into the S buffer's TMEM
                    // columns: P_hi (bf16 truncation) in 0..63, P_lo (the rest,
                    // rounded) in 64..127, two keys per column, even key low
                    // (pairs of keys through packed fp32 arithmetic)
                    {
                        uint32_t phi[32], plo[32];
                        const uint64_t m2 = f2_pack(mref, mref);
                        uint64_t ls2 = f2_pack(0.f, 0.f);
#pragma unroll
                        for (int c2 = 0; c2 < 32; ++c2) {
                            float d0, d1;
                            f2_unpack(f2_sub(f2_pack(__uint_as_float(sraw[2 * c2]),
                                                     __uint_as_float(sraw[2 * c2 + 1])),
                                             m2),
                                      d0, d1);
                            const float p0 = fast_exp2(d0), p1 = fast_exp2(d1);
                            const uint64_t p2 = f2_pack(p0, p1);
                            ls2 = f2_add(ls2, p2);
                            const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
                            phi[c2] = __byte_perm(u0, u1, 0x7632);
                            float l0, l1;
                            f2_unpack(f2_sub(p2, f2_pack(__uint_as_float(u0 & 0xffff0000u),
                                                         __uint_as_float(u1 & 0xffff0000u))),
                                      l0, l1);
                            plo[c2] = pack_bf16x2(l0, l1);
                        }
                        float ls0, ls1;
                        f2_unpack(ls2, ls0, ls1);
                        lsum += ls0 + ls1;
                        tmem_st32(tl + sb * 128 + (kh >> 1), phi);
                        tmem_st32(tl + sb * 128 + 64 + (kh >> 1), plo);
                    }
                    tmem_wait_st();
                    fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(pfull0 + 8 * sb);
                }
                if (!ok) break;

                // ------------------------------------------------ end of item
                // the row's sum: this half's plus the partner's
                xl[half * 32] = lsum;
                pair_sync();
                const float ltot = xl[0] + xl[32];
                const uint32_t gl = g - 1;  // the item's last tile
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[C::B_PVDONE + (gl & 1)],
                                                               (gl >> 1) & 1, P.fault,
                                                               kFaultCopyTimeout, P.wait_limit));
                if (!ok) break;
                fence_after_sync();
                const uint32_t oc = tl + C::O_COL + half * DH;
                if (P.splits == 1) {
                    // 32 dims of the warp's 32 rows at a time through a 2 KB staging
                    // buffer ([row][4 x 16 B], chunk index XOR (row >> 1) & 3 against
                    // bank conflicts), then stored as 8 rows x 64 B per instruction
                    const float inv = ltot > 0.f ? __frcp_rn(ltot) : 0.f;
                    uint8_t *stg = sm + C::STG_OFF + (warp - 2) * 2048;
                    // the warp's 32 rows all in the item and starting a query row:
                    // each staged chunk leaves in one tensor store, so the warp does
                    // not wait on the output's global stores
                    const int rw0 = it.row0 + quad * 32;
                    const bool tma_out = PM.out_ok && quad * 32 + 31 < it.rows && rw0 % P.G == 0;
                    const int oy = it.h * P.G, oz = it.b * P.q_len + rw0 / P.G;
                    const int wr = lane >> 2, wc = lane & 3;  // write-back row (+ 8 s), chunk
                    size_t wrow[4];
                    bool wlive[4];
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) {
                        const int rr = quad * 32 + wr + 8 * s2;
                        const int rg2 = it.row0 + rr;
                        const int i2 = rg2 / P.G, gg2 = rg2 - i2 * P.G;
                        wlive[s2] = rr < it.rows;
                        wrow[s2] = (((size_t)it.b * P.q_len + i2) * P.Hq + (size_t)it.h * P.G + gg2) * D;
                    }
                    // (the next chunk's TMEM load is in flight meanwhile)
                    uint32_t o[2][32];
                    tmem_ld32(oc, o[0]);
#pragma unroll
                    for (int c = 0; c < DH / 32; ++c) {
                        tmem_wait_ld();
                        if (c + 1 < DH / 32) tmem_ld32(oc + 32 * (c + 1), o[(c + 1) & 1]);
                        const uint32_t *oo = o[c & 1];
                        // the staging buffer's previous tensor store has read it
                        if (lane == 0) bulk_wait_read();
                        __syncwarp();
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(oo[8 * q4 + 0]) * inv,
                                              __uint_as_float(oo[8 * q4 + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(oo[8 * q4 + 2]) * inv,
                                              __uint_as_float(oo[8 * q4 + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(oo[8 * q4 + 4]) * inv,
                                              __uint_as_float(oo[8 * q4 + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(oo[8 * q4 + 6]) * inv,
                                              __uint_as_float(oo[8 * q4 + 7]) * inv);
                            *reinterpret_cast<uint4 *>(stg + lane * 64 +
                                                       ((q4 ^ ((lane >> 1) & 3)) << 4)) = w;
                        }
                        if (tma_out) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_3d(&PM.out, half * DH + 32 * c, oy, oz, stg);
                                bulk_commit();
                            }
                            continue;
                        }
                        __syncwarp();
#pragma unroll
                        for (int s2 = 0; s2 < 4; ++s2) {
                            const int rr = wr + 8 * s2;
                            const uint4 w = *reinterpret_cast<const uint4 *>(
                                stg + rr * 64 + ((wc ^ ((rr >> 1) & 3)) << 4));
                            if (wlive[s2])
                                *reinterpret_cast<uint4 *>(P.out + wrow[s2] + half * DH + 32 * c + wc * 8) = w;
                        }
                        __syncwarp();
                    }
                    if (live && half == 0 && P.lse != nullptr)
                        P.lse[orow] = ltot > 0.f ? (mref + __log2f(ltot)) * kLn2 : NEG_INF;
                } else {
#pragma unroll 1
                    for (int c0 = 0; c0 < DH; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(oc + c0, o);
                        tmem_wait_ld();
                        if (live) {
                            float4 *dst =
                                reinterpret_cast<float4 *>(P.part_acc + prow * D + half * DH + c0);
#pragma unroll
                            for (int q4 = 0; q4 < 8; ++q4)
                                dst[q4] = make_float4(__uint_as_float(o[4 * q4]), __uint_as_float(o[4 * q4 + 1]),
                                                      __uint_as_float(o[4 * q4 + 2]),
                                                      __uint_as_float(o[4 * q4 + 3]));
                        }
                    }
                    if (live && half == 0) {
                        P.part_ml[prow * 2] = ltot > 0.f ? mref : NEG_INF;
                        P.part_ml[prow * 2 + 1] = ltot;
                    }
                }
                fence_before_sync();
                __syncwarp();
                // O may be overwritten (its loads completed; the output stores
                // need no ordering with rank 0)
                if (lane == 0) mbar_arrive_cluster_relaxed(ofree0);
            }
            (void)ok;
            if (lane == 0) bulk_wait_all();  // this warp's output stores complete
        }
    }

    // ---------------------------------------------------------- teardown
    fence_before_sync();
    __syncthreads();
    cluster_sync();
    fence_after_sync();
    if (warp == 1) tmem_dealloc_pair(tmem, C::TMEM_COLS);
}

}  // namespace swa
