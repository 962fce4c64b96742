// Tensor-core (tcgen05) split-KV kernel for sliding-window verify attention.
//
// Persistent CTAs (one per SM) walk a list of work items (sequence, KV
// head, key chunk, row tile).  Keys are the MMA's M dimension: for every
// tile of 128 keys
//
//   S^T[128 keys x N rows] = K_tile[128 x D] . Q[N x D]^T      (TMEM, fp32)
//   O^T[D x N]            += V_tile^T[D x 128] . P^T[N x 128]^T (TMEM, fp32)
//
// where the N rows are the packed query rows of one KV head (G query heads
// times the draft rows, padded to a multiple of 16), so every K/V byte is
// read once per KV head and small draft blocks cost no M padding.
//
// P is carried into the second MMA as two bf16 tiles, P = P_hi + P_lo with
// P_hi = bf16(P) and P_lo = bf16(P - P_hi), so the weights keep about 16
// significant bits instead of bf16's 8.  The two tiles are stacked as one
// B operand of 2N rows (an M=128 MMA costs the same up to N=64), and O^T
// holds 2N columns whose halves the epilogue adds.
//
// K and V arrive by TMA a whole tile at a time into a ring of tile slots.
// A tile is laid out as 8-key atoms, each atom holding the D/64 head-dim
// slabs of its 8 keys as 1024-byte 128-byte-swizzled blocks:
//   [atom a][slab s][key row r][128 bytes]
// A 4D tensor map (x = 64 dims, y = cache row, z = slab, w = atom) loads
// 8*A consecutive rows from any start row in one copy, so a full tile is one
// TMA and a partial tile of n keys at most five (binary decomposition of
// n / 8 atoms, then a one-atom 3D box for the last n % 8 keys, whose rows
// past the cache the TMA zero-fills).  Q, P and O are double-buffered (where
// shared memory allows) so consecutive tiles and items overlap: the MMA lane
// issues the next tile's S (across item boundaries) before the current
// tile's PV, and the epilogue of one item runs while the next item's loads
// and scores proceed.
//
// Warp roles (320 threads, 352 under a fused append):
//   warp 0      TMA producer (lane 0 runs it; the warp issues a tile's copies)
//   warp 1      TMEM owner and MMA issuer (one lane)
//   warps 2..9  softmax / correction / epilogue in two warpgroups that split
//               the packed rows in halves; within a group a thread owns one
//               TMEM lane: one key of the S^T tile and one head-dim row of
//               the O^T accumulator (warps w and w + 4 read the same lanes).
//   warp 10     fused append only (the kernel's AP variant): mixed atoms of a
//               paged cache, and the new rows' cache stores
//
// Softmax runs in the log2 domain with a lazily raised reference maximum:
// each row keeps m_ref (in registers, identical in every thread of the
// group that owns the row);
// a tile whose scaled score exceeds m_ref + 8 (a factor 256) for any row
// triggers an exact per-row tile maximum, a raise of m_ref and, if O
// already holds data, a rescale of O^T in TMEM.  Otherwise
// P = 2^(s - m_ref) <= 256.  Row sums are reduced across lanes with a
// reduce-scatter butterfly.
//
// Every wait on an mbarrier is bounded; a wait that gives up sets the fault
// word, the roles leave their loops together, and TMEM is freed.
#pragma once

#include "swa_simt.cuh"
#include "swa_tc_host.h"
#include "swa_tc_ptx.cuh"

namespace swa {

constexpr int kTcThreads = 320;  // and one append warp more under a fused append
constexpr int kTcTileKeys = 128;
constexpr int kTcTailBox = 32;    // keys per box of a partial tile
constexpr int kTcMetaItems = 7;   // items per CTA decoded once into shared memory
// Ring slots are handed out in any order (the first free one), so a K tile,
// consumed as soon as its scores are computed, frees its slot long before
// the V tiles around it; a table of the recent fills tells the MMA lane
// where each landed: entry f % kFillTab = (f << 8) | (use parity << 4) | slot.
constexpr int kFillTab = 16;
// Initial per-row reference maximum (log2 units): finite, so P = 2^(s - m)
// needs no special case, yet below any score of a row with keys, so the
// first tile always raises it.
constexpr float kNoRef = -1.0e30f;

struct TcItem {
    int b, h, split, rt;
    ChunkRange cr;
    int t0;    // key position of tile 0: the chunk start, or that rounded down to
               // a multiple of 8 (paged cache: every atom inside one page) or to
               // q_pos mod 8 (fused append: new rows start on an atom)
    int n_tiles;
    int row0;  // first packed row of the item
    int rows;  // packed rows of the item
    int i0;    // first draft row
};

template <int D, int N, int NT, int QB, int PB, int OB>
struct TcCfg {
    static constexpr int SLABS = D / 64;
    static constexpr int ATOM_BYTES = SLABS * 1024;            // 8 keys x D
    static constexpr int TILE_BYTES = (kTcTileKeys / 8) * ATOM_BYTES;
    static constexpr int Q_SLAB = N * 128;
    static constexpr int Q_BUF = SLABS * Q_SLAB;
    static constexpr int P_KSLAB = 2 * N * 128;  // 64 keys x (N hi + N lo rows)
    static constexpr int P_BUF = 2 * P_KSLAB;     // 128 keys
    static constexpr int RING_OFF = 0;
    static constexpr int Q_OFF = RING_OFF + NT * TILE_BYTES;
    static constexpr int P_OFF = Q_OFF + QB * Q_BUF;
    static constexpr int RED_OFF = P_OFF + PB * P_BUF;        // float [2][4][N]
    static constexpr int LINV_OFF = RED_OFF + 2 * 4 * N * 4;  // float [N]
    static constexpr int ALPHA_OFF = LINV_OFF + N * 4;        // float [N]
    static constexpr int ROW_OFF = ALPHA_OFF + N * 4;          // uint32 [N] output rows
    static constexpr int META_OFF = ROW_OFF + N * 4;           // TcItem [kTcMetaItems]
    static constexpr int FTAB_OFF = META_OFF + kTcMetaItems * (int)sizeof(TcItem);  // uint32 [kFillTab]
    static constexpr int BAR_OFF = FTAB_OFF + kFillTab * 4;
    // ring full/empty [NT], q full/empty [QB], s full/free [2], p full [PB],
    // pv done [PB], o free [2] (OB used), drain, mixed atom of a fused append [NT]
    static constexpr int B_FULL = 0, B_EMPTY = NT, B_QFULL = 2 * NT, B_QEMPTY = B_QFULL + QB,
                         B_SFULL = B_QEMPTY + QB, B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2,
                         B_PVDONE = B_PFULL + PB, B_OFREE = B_PVDONE + PB, B_DRAIN = B_OFREE + 2,
                         B_MIX = B_DRAIN + 1, NBARS = B_MIX + NT;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base
    static constexpr int END = MISC_OFF + 16;
    static constexpr int SMEM_BYTES = END + 1024;  // slack for 1024-byte alignment
    static constexpr int O_COLS = (D / 128) * 2 * N;  // one O^T buffer: hi and lo halves
    static constexpr int TMEM_USED = 2 * N + OB * O_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                     : TMEM_USED <= 64  ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256
                                                        : 512;
    static constexpr int O_COL = 2 * N;           // O buffer ob at O_COL + ob * O_COLS
    static constexpr int CW = N >= 32 ? 32 : 16;  // TMEM columns per load
    static constexpr int NCH = N / CW;
    static_assert(NT >= 2, "ring holds at least a K and a V tile");
    static_assert(N % 16 == 0 && N >= 16 && N <= 64, "rows per tile");
    static_assert(TMEM_USED <= 512, "TMEM");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(PB * P_BUF >= N * 512, "epilogue staging fits in the P buffers");
    static_assert(RED_OFF % 16 == 0 && BAR_OFF % 8 == 0 && META_OFF % 8 == 0, "alignment");
};


// The work items of this CTA, numbered j = 0, 1, ...: a contiguous block of
// the item list (T.items_per_cta > 0: neighbouring (sequence, KV head) units
// run back to back on one SM) or every gridDim.x-th item (round-robin).
__device__ __forceinline__ int cta_items(const TcParams &T) {
    if (T.items_per_cta > 0) return T.items_per_cta + ((int)blockIdx.x < T.items_extra ? 1 : 0);
    return (T.items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
}
__device__ __forceinline__ int cta_item(const TcParams &T, int j) {
    if (T.items_per_cta > 0)
        return (int)blockIdx.x * T.items_per_cta + min((int)blockIdx.x, T.items_extra) + j;
    return (int)blockIdx.x + j * (int)gridDim.x;
}

// Work item `item` (its sequence's seq_len / q_pos read from global memory).
template <bool AP>
__device__ __forceinline__ TcItem tc_decode_global(const TcParams &T, int item) {
    const AttnParams &P = T.a;
    TcItem it;
    int rest = item;
    it.rt = rest % P.row_tiles;
    rest /= P.row_tiles;
    it.split = rest % P.splits;
    rest /= P.splits;
    it.h = rest % P.Hkv;
    it.b = rest / P.Hkv;
    it.row0 = it.rt * T.rows_per_tile;
    it.rows = min(P.R - it.row0, T.rows_per_tile);
    it.i0 = it.rt * T.q_rows_per_tile;
    it.cr = chunk_range(P, it.b, it.split, it.i0, (it.row0 + it.rows - 1) / P.G);
    // a contiguous cache under a fused append: rounded down to q_pos mod 8,
    // so the new block starts on an atom of every tile (not below position 0:
    // a box must not start at a negative row, whose bounds check would blank
    // the rows its later atoms hold)
    it.t0 = P.block_table != nullptr ? (it.cr.c_lo & ~7)
            : AP                     ? max(it.cr.c_lo - ((it.cr.c_lo - it.cr.qp) & 7), 0)
                                     : it.cr.c_lo;
    const int nk = it.cr.c_hi - it.t0;
    it.n_tiles = it.cr.c_hi > it.cr.c_lo ? (nk + kTcTileKeys - 1) / kTcTileKeys : 0;
    return it;
}

// Work item `item`, the j-th of this CTA: the first kTcMetaItems were
// decoded once at set-up into shared memory.
template <bool AP>
__device__ __forceinline__ TcItem tc_decode(const TcParams &T, int item, int j,
                                            const TcItem *meta) {
    if (j < kTcMetaItems) return meta[j];
    return tc_decode_global<AP>(T, item);
}

// Barrier of one softmax warpgroup (128 threads), ids 1 / 3.
__device__ __forceinline__ void group_sync(int wg) {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + 2 * wg) : "memory");
}

// True on every thread of softmax warpgroup `wg` if `v` is true on any of
// them (ids 2 / 4).
__device__ __forceinline__ bool group_any(int wg, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(2 + 2 * wg)
        : "memory");
    return r != 0;
}

// Reduce-scatter of CW (8, 16 or 32) per-lane values across the warp with
// op `max` or `sum`: afterwards lane l holds the reduction of element
// (l % CW) over all 32 lanes.  v is consumed.
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
#pragma unroll
    for (int off = CW; off < 32; off <<= 1) {
        const float got = __shfl_xor_sync(0xffffffffu, v[0], off);
        v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
    }
    return v[0];
}

// W (8, 16 or 32) consecutive TMEM columns of this thread's lane.
template <int W>
__device__ __forceinline__ void tmem_load(uint32_t taddr, uint32_t *r) {
    if constexpr (W == 32) {
        tc::tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(r));
    } else if constexpr (W == 16) {
        tc::tmem_ld16(taddr, r);
    } else {
        tc::tmem_ld8(taddr, r);
    }
}

template <int W>
__device__ __forceinline__ void tmem_store(uint32_t taddr, const uint32_t *r) {
    if constexpr (W == 16) {
        tc::tmem_st16(taddr, r);
    } else {
        static_assert(W == 8, "store width");
        tc::tmem_st8(taddr, r);
    }
}

// The copies of one K or V tile: key positions [p, p + n_valid) of
// (sequence b, KV head h) into ceil(n_valid / 8) atoms of AB bytes at dst,
// completing on `bar`.  Whole atoms go through the 4D boxes (16, 8, 4 or 2
// atoms: the rows of a run are consecutive cache rows); a single or a
// partial atom through the 3D one-atom box, whose rows past the cache the
// TMA zero-fills.  A contiguous cache is one run; a paged cache breaks runs
// at page ends (pages hold a multiple of 8 rows and its tiles start on an
// 8-key boundary, so no atom straddles two pages).
// Whole atoms [0, whole) and, if `partial`, one more through the 3D box: a
// run of consecutive cache rows starting at row y into dst.
template <int AB>
__device__ __forceinline__ void atom_run(const CUtensorMap *m4, const CUtensorMap *m1, int y,
                                         int whole, bool partial, uint8_t *dst, uint64_t *bar,
                                         uint64_t policy) {
    using namespace tc;
    int w = 0;
    if (whole == 16) {
        tma_load_4d_hint(dst, &m4[0], 0, y, 0, 0, bar, policy);
        return;
    }
#pragma unroll
    for (int bi = 1; bi < 4; ++bi) {
        const int na = 16 >> bi;
        if (whole & na) {
            tma_load_4d_hint(dst + w * AB, &m4[bi], 0, y + 8 * w, 0, 0, bar, policy);
            w += na;
        }
    }
    if (whole & 1) {
        tma_load_3d_hint(dst + w * AB, m1, 0, y + 8 * w, 0, bar, policy);
        ++w;
    }
    if (partial) tma_load_3d_hint(dst + w * AB, m1, 0, y + 8 * w, 0, bar, policy);
}

// The copies of one K or V tile: key positions [p, p + n_valid) of
// (sequence b, KV head h) into ceil(n_valid / 8) atoms of AB bytes at dst,
// completing on `bar`, issued by the lanes of the producer warp.  Whole
// atoms go through the 4D boxes (16, 8, 4 or 2 atoms: the rows of a run are
// consecutive cache rows); a single or a partial atom through the 3D
// one-atom box, whose rows past the cache the TMA zero-fills.  A contiguous
// cache is one run (lane 0); a paged cache breaks runs at page ends (pages
// hold a multiple of 8 rows and its tiles start on an 8-key boundary, so no
// atom straddles two pages) and lane k reads the page id of run k and
// issues its copies, so a tile over many small pages costs one round of
// copies, not one per page.
template <int AB>
__device__ __forceinline__ void tile_copies(const AttnParams &P, const TcMaps &M, int kv, int b,
                                            int h, int p, int n_valid, uint8_t *dst, uint64_t *bar,
                                            uint64_t policy, int lane) {
    const CUtensorMap *m4 = kv ? M.v_atoms : M.k_atoms;
    const CUtensorMap *m1 = kv ? &M.v_atom : &M.k_atom;
    const int full = n_valid >> 3, natoms = (n_valid + 7) >> 3;
    if (P.block_table == nullptr) {
        if (lane == 0)
            atom_run<AB>(m4, m1, (int)cache_row(P, b, h, p), full, natoms > full, dst, bar,
                         policy);
        return;
    }
    const int ps = P.page_size, pa = ps >> 3;           // rows, atoms per page
    const int k0 = p / ps, first = (ps - p % ps) >> 3;  // first page, its atoms
    const int a = lane == 0 ? 0 : first + (lane - 1) * pa;  // first atom of run `lane`
    if (a >= natoms) return;
    int run = lane == 0 ? first : pa;
    run = run < natoms - a ? run : natoms - a;
    int whole = full - a;
    whole = whole < 0 ? 0 : (whole > run ? run : whole);
    const int pg = checked_page(P, __ldg(P.block_table + (long long)b * P.max_blocks + k0 + lane),
                                nullptr);
    const int y = (pg * P.Hkv + h) * ps + (lane == 0 ? p % ps : 0);
    atom_run<AB>(m4, m1, y, whole, run > whole, dst + a * AB, bar, policy);
}

// How a K/V tile (key positions [p, p + n_valid), ceil(n_valid / 8) atoms)
// is sourced under a fused append (new rows at positions qp ..): atoms
// [0, a_m) hold cache rows only; atom a_m is mixed (cache rows, then new
// rows) when the new block starts inside it, which happens only on a paged
// cache; atoms [a_n, natoms) hold positions >= qp only and come from
// k_new / v_new.  A tile whose valid keys end before qp, and every tile
// without an append, has a_m = a_n = natoms.
__device__ __forceinline__ void append_split(const AttnParams &P, int qp, int p, int n_valid,
                                             int &a_m, int &a_n) {
    a_m = a_n = (n_valid + 7) >> 3;
    if (P.k_new == nullptr || p + n_valid <= qp) return;
    a_m = qp > p ? (qp - p) >> 3 : 0;
    a_n = qp > p && ((qp - p) & 7) ? a_m + 1 : a_m;
}

// Fills of the CTA's first work item issued ahead of the producer loop:
// its first min(NT, early_max, 2 * n_tiles) K/V fills (fill 2t + kv into
// ring slot 2t + kv) and its Q rows; 0 if none (paged cache, fused append,
// no item, an empty first item).  The producer loop computes the same count.
template <int NT, bool AP>
__device__ __forceinline__ int early_fills(const TcParams &T, const TcItem &it) {
    if (AP || T.a.block_table != nullptr || it.n_tiles == 0) return 0;
    return min(min(NT, T.early_max), 2 * it.n_tiles);
}

// Right after griddepcontrol.wait, lane 0 of warp w < early_fills issues
// fill w of the CTA's first item (and warp NT the item's Q rows), each warp
// decoding the item itself: the copies go out in parallel from separate
// warps, ahead of the CTA's set-up barrier and of the producer loop (whose
// first fills would otherwise leave one at a time).  The barriers and the
// fill table must be initialised and a CTA barrier passed beforehand; no
// other thread writes the bytes these copies land in (the Q rows TMA writes
// are never zeroed).  A withheld fill (tests of the bounded waits) is
// posted on its barrier but not copied.
template <class C, int NT, bool AP>
__device__ __forceinline__ void issue_early_fills(const TcParams &T, const TcMaps &M,
                                                  volatile uint32_t *ftab, uint8_t *ring,
                                                  uint8_t *qs, uint64_t *bars, int warp) {
    using namespace tc;
    const AttnParams &P = T.a;
    if (AP || P.block_table != nullptr || warp > NT || cta_items(T) < 1) return;
    const TcItem it = tc_decode_global<AP>(T, cta_item(T, 0));
    const int n = early_fills<NT, AP>(T, it);
    if (n == 0) return;
    if (warp == NT) {
        mbar_arrive_expect_tx(&bars[C::B_QFULL], C::SLABS * T.rows_per_tile * 128);
        for (int s = 0; s < C::SLABS; ++s)
            tma_load_3d(qs + s * C::Q_SLAB, &M.q, 64 * s, it.h * P.G, it.b * P.q_len + it.i0,
                        &bars[C::B_QFULL]);
        return;
    }
    if (warp >= n) return;
    const int t = warp >> 1, kv = warp & 1;
    const int p = it.t0 + kTcTileKeys * t;
    const int n_valid = min(kTcTileKeys, it.cr.c_hi - p);
    ftab[warp] = ((uint32_t)warp << 8) | (uint32_t)warp;  // fill w -> slot w, use parity 0
    mbar_arrive_expect_tx(&bars[C::B_FULL + warp], (uint32_t)((n_valid + 7) >> 3) * C::ATOM_BYTES);
    if (P.withhold_fill == warp && blockIdx.x == 0) return;
    const uint64_t policy = P.row_tiles > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
    tile_copies<C::ATOM_BYTES>(P, M, kv, it.b, it.h, p, n_valid, ring + warp * C::TILE_BYTES,
                               &bars[C::B_FULL + warp], policy, 0);
}

// The TMA producer (warp 0) of both tensor-core kernels: lane 0 runs the
// control (slots, barriers, the fill table, Q and the fused append's extra
// copies) and the warp issues each tile's copies.  For every item of the
// CTA, its K and V tiles into the first free ring slots
// (the fill table records where each landed) and its Q rows, issued after
// the item's first K tile so a single Q buffer does not hold back the K
// stream.  With a fused append, the atoms of a tile from the first new row
// on (a mixed atom from the cache, new-row atoms from k_new / v_new) land on
// B_MIX, for the append worker to complete the fill.  With `early`, the
// first item's first early_fills() fills and its Q rows were issued already
// (issue_early_fills).  Waits for every copy it issued before returning.
template <class C, int NT, int QB, bool AP>
__device__ __forceinline__ void tile_producer(const TcParams &T, const TcMaps &M,
                                              const TcItem *meta, volatile uint32_t *ftab,
                                              uint8_t *ring, uint8_t *qs, uint64_t *bars,
                                              bool early) {
    using namespace tc;
    const AttnParams &P = T.a;
    const int lane = (int)(threadIdx.x & 31);
    // The warp walks the loop together when a tile's copies are many (paged
    // cache) or the CTA has one item (latency-bound calls: measured faster);
    // a long run of items over a contiguous cache is faster with lane 0
    // alone (no per-fill warp synchronisation).
    const bool coop = P.block_table != nullptr || cta_items(T) <= 1;
    if (!coop && lane != 0) return;
    // K/V are read once per row tile: with one row tile nothing reads a line
    // again (evict first); with several, the row tiles of a (sequence, KV
    // head) run side by side on neighbouring CTAs and the later ones should
    // find the lines in L2
    const uint64_t policy = P.row_tiles > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
    uint32_t f = 0, k = 0;  // fills (two per tile: K then V), items with keys
    uint32_t mix_used = 0, mix_n = 0;  // slots that took a mixed atom; use count parity
    uint32_t uses[NT];              // fills handed to each slot so far
#pragma unroll
    for (int s2 = 0; s2 < NT; ++s2) uses[s2] = 0;
    const int n_items = cta_items(T);
    const int n_early = early && n_items > 0 ? early_fills<NT, AP>(T, tc_decode<AP>(T, cta_item(T, 0), 0, meta)) : 0;
#pragma unroll
    for (int s2 = 0; s2 < NT; ++s2)
        if (s2 < n_early) uses[s2] = 1;  // fill s2 went to slot s2
    f = (uint32_t)n_early;
    bool ok = true;
    for (int j = 0; j < n_items && ok; ++j) {
        const TcItem it = tc_decode<AP>(T, cta_item(T, j), j, meta);
        if (it.n_tiles == 0) continue;
        const uint32_t qb = k % QB, quse = k / QB;
        auto load_q = [&]() -> bool {
            if (!mbar_wait_bounded(&bars[C::B_QEMPTY + qb], (quse & 1) ^ 1, P.fault,
                                   kFaultCopyTimeout, P.wait_limit))
                return false;
            mbar_arrive_expect_tx(&bars[C::B_QFULL + qb], C::SLABS * T.rows_per_tile * 128);
            for (int s = 0; s < C::SLABS; ++s)
                tma_load_3d(qs + qb * C::Q_BUF + s * C::Q_SLAB, &M.q, 64 * s, it.h * P.G,
                            it.b * P.q_len + it.i0, &bars[C::B_QFULL + qb]);
            return true;
        };
        ++k;
        for (int t = 0; t < it.n_tiles && ok; ++t) {
            const int p = it.t0 + kTcTileKeys * t;
            const int n_valid = min(kTcTileKeys, it.cr.c_hi - p);
            const int natoms = (n_valid + 7) >> 3;
            int a_m = natoms, a_n = natoms;
            if constexpr (AP) append_split(P, it.cr.qp, p, n_valid, a_m, a_n);
            const bool worker_full = AP && a_n > a_m;  // the append worker completes a mixed atom
            for (int kv = 0; kv < 2 && ok; ++kv) {
                if (j == 0 && 2 * t + kv < n_early) continue;  // issued ahead of the loop
                if (t == 0 && kv == 1 && !(j == 0 && n_early > 0)) {
                    if (lane == 0) ok = load_q();
                    if (coop) ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
                    if (!ok) break;
                }
                // the first free slot: never used, or its last fill consumed
                int slot = -1;
                uint32_t par = 0;
                if (lane == 0) {
                    const long long w0 = clock64();
                    for (int spin = 0;; ++spin) {
#pragma unroll
                        for (int s2 = 0; s2 < NT; ++s2) {
                            if (slot < 0 &&
                                (uses[s2] == 0 ||
                                 mbar_test(&bars[C::B_EMPTY + s2], (uses[s2] - 1) & 1))) {
                                slot = s2;
                                par = uses[s2] & 1;
                                ++uses[s2];
                            }
                        }
                        if (slot >= 0) break;
                        if (clock64() - w0 > P.wait_limit) {
                            atomicOr(P.fault, kFaultCopyTimeout);
                            break;
                        }
                        if (spin > 8) __nanosleep(32);
                    }
                }
                if (coop) {
                    slot = __shfl_sync(0xffffffffu, slot, 0);
                    par = __shfl_sync(0xffffffffu, par, 0);
                }
                ok = slot >= 0;
                if (!ok) break;
                if (lane == 0) ftab[f % kFillTab] = (f << 8) | (par << 4) | (uint32_t)slot;
                // a fill completes (FULL) on this lane's arrival with the bytes;
                // under a fused append it takes a second arrival: this lane's,
                // or the append worker's after it completed a mixed atom
                uint64_t *bar = &bars[C::B_FULL + slot];
                uint8_t *dst = ring + slot * C::TILE_BYTES;
                if (lane == 0)
                    mbar_arrive_expect_tx(bar, (uint32_t)(a_m + natoms - a_n) * C::ATOM_BYTES);
                if (coop) __syncwarp();  // the expected bytes are posted before any copy
                // (tests of the bounded waits: this fill's copies are never issued)
                const bool withhold = P.withhold_fill == (int)f && blockIdx.x == 0;
                if (withhold) {
                    ++f;
                    continue;
                }
                if (a_m > 0)
                    tile_copies<C::ATOM_BYTES>(P, M, kv, it.b, it.h, p,
                                               a_m < natoms ? 8 * a_m : n_valid, dst, bar,
                                               policy, lane);
                if (lane == 0) {
                    for (int a = a_n; a < natoms; ++a)
                        tma_load_5d(dst + a * C::ATOM_BYTES, kv ? &M.vn_atom : &M.kn_atom, 0,
                                    p + 8 * a - it.cr.qp, 0, it.h, it.b, bar);
                    if (worker_full) {
                        // the mixed atom from the cache, on its own barrier
                        uint64_t *mb = &bars[C::B_MIX + slot];
                        mix_used |= 1u << slot;
                        mix_n ^= 1u << slot;
                        mbar_arrive_expect_tx(mb, C::ATOM_BYTES);
                        tma_load_3d_hint(dst + a_m * C::ATOM_BYTES, kv ? &M.v_atom : &M.k_atom,
                                         0, (int)cache_row(P, it.b, it.h, p + 8 * a_m), 0, mb,
                                         policy);
                    } else if (AP) {
                        mbar_arrive(bar);
                    }
                }
                ++f;
            }
        }
    }
    if (lane != 0) return;
    // every copy this CTA issued has landed before it exits
#pragma unroll
    for (int s2 = 0; s2 < NT; ++s2) {
        if (uses[s2] > 0)
            mbar_wait_bounded(&bars[C::B_FULL + s2], (uses[s2] - 1) & 1, P.fault,
                              kFaultCopyTimeout, P.wait_limit);
        if ((mix_used >> s2) & 1u)
            mbar_wait_bounded(&bars[C::B_MIX + s2], ((mix_n >> s2) & 1u) ^ 1u, P.fault,
                              kFaultCopyTimeout, P.wait_limit);
    }
    const uint32_t nq = k < (uint32_t)QB ? k : (uint32_t)QB;
    for (uint32_t q = 0; q < nq; ++q) {
        const uint32_t kq = k - 1 - q;
        mbar_wait_bounded(&bars[C::B_QFULL + kq % QB], (kq / QB) & 1, P.fault,
                          kFaultCopyTimeout, P.wait_limit);
    }
}

// The append warp (warp 10) under a fused append.  Over the tiles whose new
// block starts inside an atom (paged cache): the mixed atom landed
//   from the cache on B_MIX of the ring slot the fill table names; the warp
//   writes the new rows over its stale ones from registers loaded from
//   k_new / v_new ahead of time, fences the writes against the tensor
//   core's reads and gives FULL its second arrival.
// With at most two items per CTA it also stores the new rows the item owns
// (its own draft rows' positions inside its chunk) to the cache, overlapped
// with the attention; with more the CTA stores them together at the end
// (append_flush).
// It runs in a warp of its own: lanes of the TMA warp blocked on their
// loads would hold back the other, diverged path of that warp.
template <class C, int D>
__device__ __forceinline__ void append_worker(const TcParams &T, const TcItem *meta,
                                              const volatile uint32_t *ftab, uint8_t *ring,
                                              uint64_t *bars) {
    const AttnParams &P = T.a;
    constexpr int PR = D / 8;                   // 16-byte pieces per row
    constexpr int MP = (7 * PR + 31) / 32;      // pieces per lane of a mixed atom's new rows
    constexpr int U = 16;                       // pieces per lane in flight while storing
    const int t = (int)(threadIdx.x & 31);
    uint32_t f = 0, mixpar = 0;                 // fills seen; use parity of B_MIX per slot
    const int n_items = cta_items(T);
    for (int j = 0; j < n_items; ++j) {
        const TcItem it = tc_decode<true>(T, cta_item(T, j), j, meta);
        if (it.n_tiles == 0) continue;
        int ap_lo, ap_hi;
        append_range(P, it.cr, it.i0, (it.row0 + it.rows - 1) / P.G, ap_lo, ap_hi);
        const long long row_b = (long long)it.b * P.q_len;  // k_new row of draft row 0
        for (int tt = 0; tt < it.n_tiles; ++tt, f += 2) {
            const int p = it.t0 + kTcTileKeys * tt;
            const int n_valid = min(kTcTileKeys, it.cr.c_hi - p);
            int a_m, a_n;
            append_split(P, it.cr.qp, p, n_valid, a_m, a_n);
            if (a_n == a_m) continue;
            // the mixed atom's new rows (rows [m_lo, 8) of atom a_m), loaded early
            const int p_m = p + 8 * a_m;
            const int m_lo = it.cr.qp - p_m;
            const int np = (8 - m_lo) * PR;
            uint4 w[2][MP];
#pragma unroll
            for (int kv = 0; kv < 2; ++kv)
#pragma unroll
                for (int u = 0; u < MP; ++u) {
                    const int e = t + 32 * u;
                    const int i = e / PR;  // draft row of the piece
                    w[kv][u] = make_uint4(0, 0, 0, 0);
                    if (e < np && i < P.q_len)
                        w[kv][u] = __ldg(reinterpret_cast<const uint4 *>(
                            (kv ? P.v_new : P.k_new) + ((row_b + i) * P.Hkv + it.h) * D +
                            (e % PR) * 8));
                }
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
                // lane 0 waits for the fill's table entry and hands it on
                const uint32_t fill = f + kv;
                uint32_t e = 0;
                bool found = true;
                if (t == 0) {
                    e = ftab[fill % kFillTab];
                    const long long w0 = clock64();
                    while ((e >> 8) != (fill & 0xffffffu)) {
                        if (clock64() - w0 > P.wait_limit) {
                            atomicOr(P.fault, kFaultCopyTimeout);
                            found = false;
                            break;
                        }
                        __nanosleep(32);
                        e = ftab[fill % kFillTab];
                    }
                }
                if (!__shfl_sync(0xffffffffu, (int)found, 0)) return;
                const int slot = (int)(__shfl_sync(0xffffffffu, e, 0) & 15u);
                const bool landed = mbar_wait_bounded(&bars[C::B_MIX + slot],
                                                      (mixpar >> slot) & 1u, P.fault,
                                                      kFaultCopyTimeout, P.wait_limit);
                if (!__all_sync(0xffffffffu, landed)) return;
                mixpar ^= 1u << slot;
                uint8_t *atom = ring + slot * C::TILE_BYTES + a_m * C::ATOM_BYTES;
#pragma unroll
                for (int u = 0; u < MP; ++u) {
                    const int e2 = t + 32 * u;
                    if (e2 < np) {
                        const int r = m_lo + e2 / PR, c = e2 % PR;
                        *reinterpret_cast<uint4 *>(atom + (c >> 3) * 1024 + r * 128 +
                                                   (((c & 7) ^ r) << 4)) = w[kv][u];
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (t == 0) mbar_arrive(&bars[C::B_FULL + slot]);
            }
        }
        // with at most two items per CTA (latency-bound calls) the item's new
        // rows go to the cache here, overlapped with the attention; otherwise
        // the whole CTA stores them at the end (append_flush)
        if (n_items > 2 || ap_lo >= ap_hi) continue;
        const int half = (ap_hi - ap_lo) * PR, n = 2 * half;  // K then V
        for (int b0 = 0; b0 < n; b0 += 32 * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = b0 + t + 32 * u;
                if (e < n) {
                    const int kv = e >= half, rest = e - kv * half;
                    const int i = ap_lo + rest / PR - it.cr.qp;
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(
                        (kv ? P.v_new : P.k_new) + ((row_b + i) * P.Hkv + it.h) * D +
                        (rest % PR) * 8));
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = b0 + t + 32 * u;
                if (e < n) {
                    const int kv = e >= half, rest = e - kv * half;
                    __nv_bfloat16 *cache = const_cast<__nv_bfloat16 *>(kv ? P.v : P.k);
                    bool bad = false;
                    const long long row = cache_row(P, it.b, it.h, ap_lo + rest / PR, &bad);
                    if (!bad) *reinterpret_cast<uint4 *>(cache + row * D + (rest % PR) * 8) = v[u];
                }
            }
        }
    }
}

// The fused append's cache stores, by every thread of the CTA once its
// attention work is done (after the CTA-wide barrier: the ring is free then).
// Each item owns the new rows at its own draft rows' positions inside its
// chunk (append_range); their 16-byte pieces, K then V per item, form one
// sequence that the threads
// stride through with U loads in flight each, so a CTA's stores take about
// one memory round trip however many chunks it had.  A table of the chunks
// (sequence, head, rows, first piece) is built in `scratch` first.  No kernel
// reads a new row back from the cache: the stores only have to land before
// the kernel ends.
struct AppendChunk {
    int b, h, lo, qp, n, first;
};

template <int D>
__device__ __forceinline__ void append_flush(const TcParams &T, const TcItem *meta,
                                             uint8_t *scratch, int scratch_bytes, int nthreads) {
    const AttnParams &P = T.a;
    constexpr int PR = D / 8;  // 16-byte pieces per row
    constexpr int U = 8;
    const int tid = threadIdx.x;
    AppendChunk *tab = reinterpret_cast<AppendChunk *>(scratch);
    const int n_items = cta_items(T);
    const int cap = scratch_bytes / (int)sizeof(AppendChunk) - 1;
    for (int k0 = 0; k0 < n_items; k0 += cap) {
        const int nk = min(cap, n_items - k0);
        for (int k = tid; k < nk; k += nthreads) {
            const int j = k0 + k;
            const TcItem it = tc_decode<true>(T, cta_item(T, j), j, meta);
            int lo, hi;
            append_range(P, it.cr, it.i0, (it.row0 + it.rows - 1) / P.G, lo, hi);
            const bool own = lo < hi;
            tab[k] = AppendChunk{it.b, it.h, lo, it.cr.qp, own ? 2 * (hi - lo) * PR : 0, 0};
        }
        __syncthreads();
        if (tid == 0) {
            int off = 0;
            for (int k = 0; k < nk; ++k) {
                tab[k].first = off;
                off += tab[k].n;
            }
            tab[nk].first = off;  // total
        }
        __syncthreads();
        const int total = tab[nk].first;
        int k = 0;  // chunk of the current piece (pieces are visited in increasing order)
        for (int g0 = 0; g0 < total; g0 += nthreads * U) {
            uint4 v[U];
            long long dst[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int g = g0 + tid + nthreads * u;
                dst[u] = -1;
                if (g < total) {
                    while (tab[k + 1].first <= g) ++k;
                    const AppendChunk c = tab[k];
                    const int half = c.n / 2, e = g - c.first;
                    const int kv = e >= half, rest = e - kv * half;
                    const int pos = c.lo + rest / PR, pc = rest % PR;
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(
                        (kv ? P.v_new : P.k_new) +
                        (((long long)c.b * P.q_len + (pos - c.qp)) * P.Hkv + c.h) * D + pc * 8));
                    bool bad = false;
                    const long long row = cache_row(P, c.b, c.h, pos, &bad);
                    if (!bad) dst[u] = ((row * D + pc * 8) << 1) | kv;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (dst[u] >= 0) {
                    __nv_bfloat16 *cache = const_cast<__nv_bfloat16 *>((dst[u] & 1) ? P.v : P.k);
                    *reinterpret_cast<uint4 *>(cache + (dst[u] >> 1)) = v[u];
                }
            }
        }
        __syncthreads();  // the table is rebuilt for the next group of items
    }
}

template <int D, int N, int NT, int QB, int PB, int OB, bool AP>
__global__ void __launch_bounds__(AP ? kTcThreads + 32 : kTcThreads, 1)
    swa_tc_kernel(const __grid_constant__ TcParams T, const __grid_constant__ TcMaps M) {
    using C = TcCfg<D, N, NT, QB, PB, OB>;
    constexpr int NTHR = AP ? kTcThreads + 32 : kTcThreads;
    using namespace tc;
    constexpr int SLABS = C::SLABS;
    constexpr int MH = D / 128;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const AttnParams &P = T.a;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    uint8_t *ring = sm + C::RING_OFF;
    uint8_t *qs = sm + C::Q_OFF;
    uint8_t *ps = sm + C::P_OFF;
    float *red = reinterpret_cast<float *>(sm + C::RED_OFF);
    float *linv = reinterpret_cast<float *>(sm + C::LINV_OFF);
    float *alpha_sm = reinterpret_cast<float *>(sm + C::ALPHA_OFF);
    uint32_t *rowidx = reinterpret_cast<uint32_t *>(sm + C::ROW_OFF);
    TcItem *meta = reinterpret_cast<TcItem *>(sm + C::META_OFF);
    volatile uint32_t *ftab = reinterpret_cast<volatile uint32_t *>(sm + C::FTAB_OFF);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::MISC_OFF);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    // ---------------------------------------------------------------- setup
    // Nothing before grid_dep_wait() reads memory the previous kernel in the
    // stream may write: the tensor maps are kernel parameters, so their
    // descriptors are fetched while that kernel finishes.
    if (warp == 0 && lane < (AP ? 13 : 11)) {
        const CUtensorMap *mp = lane < 4    ? &M.k_atoms[lane]
                                : lane < 8  ? &M.v_atoms[lane - 4]
                                : lane == 8 ? &M.k_atom
                                : lane == 9 ? &M.v_atom
                                : lane == 10 ? &M.q
                                : lane == 11 ? &M.kn_atom
                                             : &M.vn_atom;
        prefetch_tmap(mp);
    }
    if (tid == 0) {
        for (int i = 0; i < NT; ++i) {
            // under a fused append a fill takes a second arrival
            mbar_init(&bars[C::B_FULL + i], AP ? 2 : 1);
            mbar_init(&bars[C::B_EMPTY + i], 1);
            mbar_init(&bars[C::B_MIX + i], 1);
        }
        for (int i = 0; i < QB; ++i) {
            mbar_init(&bars[C::B_QFULL + i], 1);
            mbar_init(&bars[C::B_QEMPTY + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[C::B_SFULL + i], 1);
            mbar_init(&bars[C::B_SFREE + i], 256);
            mbar_init(&bars[C::B_OFREE + i], 256);
        }
        for (int i = 0; i < PB; ++i) {
            mbar_init(&bars[C::B_PFULL + i], 256);
            mbar_init(&bars[C::B_PVDONE + i], 1);
        }
        mbar_init(&bars[C::B_DRAIN], 1);
        fence_barrier_init();
    }
    // Q rows past an item's rows stay zero for the whole kernel (TMA writes
    // only the first rows_per_tile rows of each slab, and those are never
    // zeroed, so the first Q copy may land before this block's barrier).
    {
        const int zr = (N - T.rows_per_tile) * 8;  // 16-byte pieces per slab
        for (int i = tid; i < QB * SLABS * zr; i += NTHR) {
            const int sl = i / zr, r = i - sl * zr;
            reinterpret_cast<uint4 *>(qs + sl * C::Q_SLAB + T.rows_per_tile * 128)[r] =
                make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    for (int i = tid; i < kFillTab; i += NTHR) ftab[i] = 0xffffffffu;
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();  // barriers and fill table ready for the early fills
    grid_dep_wait();
    grid_dep_trigger();
    // the first item's first fills and Q rows go out before anything else,
    // one warp each; then the metadata of this CTA's first items
    if (lane == 0) issue_early_fills<C, NT, AP>(T, M, ftab, ring, qs, bars, warp);
    for (int j = tid; j < kTcMetaItems; j += NTHR)
        if (j < cta_items(T)) meta[j] = tc_decode_global<AP>(T, cta_item(T, j));
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ======================================================= producer
        tile_producer<C, NT, QB, AP>(T, M, meta, ftab, ring, qs, bars, true);
    } else if (warp == 1) {
        // ============================================================ MMA
        // An event loop over two cursors on the same tile sequence: S = K Q^T
        // of the next tile and O += V^T P^T of the oldest tile whose P is
        // ready are each issued as soon as their operands have landed, so
        // neither waits behind the other.  The whole warp runs the loop (its
        // lanes zero the ragged end of a partial V tile); lane 0 issues.
        {
            const bool leader = lane == 0;
            constexpr uint32_t ID_QK = idesc_bf16_f32(128, N, 0, 0);
            constexpr uint32_t ID_PV = idesc_bf16_f32(128, 2 * N, 1, 0);
            const uint32_t ring_a = smem_u32(ring);
            const uint32_t qs_a = smem_u32(qs);
            const uint32_t ps_a = smem_u32(ps);
            // tile g of this CTA is fills 2g (K) and 2g + 1 (V); the fill table
            // says which slot (and use parity) each landed in
            struct Cursor {
                int item, j, t, n_tiles;
                int last_keys;  // keys of the item's last tile
                int head;       // key rows before the chunk in its first tile (paged cache)
                uint32_t k, g;
                bool valid;
                int slot;       // this cursor's fill: slot, parity (-1: not yet looked up)
                uint32_t par;
            };
            auto lookup = [&](Cursor &c, uint32_t fill) -> bool {
                if (c.slot >= 0) return true;
                const uint32_t e = ftab[fill % kFillTab];
                if ((e >> 8) != (fill & 0xffffffu)) return false;
                c.slot = (int)(e & 15u);
                c.par = (e >> 4) & 1u;
                return true;
            };
            // first tile of the next non-empty item at or after (item, j)
            const int n_items = cta_items(T);
            auto seek = [&](Cursor &c) {
                for (; c.j < n_items; ++c.j) {
                    c.item = cta_item(T, c.j);
                    const TcItem it = tc_decode<AP>(T, c.item, c.j, meta);
                    if (it.n_tiles > 0) {
                        c.n_tiles = it.n_tiles;
                        c.last_keys = it.cr.c_hi - it.t0 - kTcTileKeys * (it.n_tiles - 1);
                        c.head = it.cr.c_lo - it.t0;
                        c.t = 0;
                        c.valid = true;
                        return;
                    }
                }
                c.valid = false;
            };
            auto advance = [&](Cursor &c) {
                ++c.g;
                c.slot = -1;
                if (++c.t < c.n_tiles) return;
                ++c.k;
                ++c.j;
                seek(c);
            };
            Cursor qc{0, 0, 0, 0, 0, 0, 0u, 0u, false, -1, 0u};
            seek(qc);
            Cursor pc = qc;
            bool ok = true;
            long long idle_since = clock64();
            int idle = 0;
            while (pc.valid) {
                bool progressed = false;
                // ---- PV of tile pc.g (its S was issued before)
                if (pc.g < qc.g || !qc.valid) {
                    const uint32_t pb = pc.g % PB;
                    bool ready = mbar_test(&bars[C::B_PFULL + pb], (pc.g / PB) & 1);
                    if (ready && pc.t == 0)
                        ready = mbar_test(&bars[C::B_OFREE + pc.k % OB], ((pc.k / OB) & 1) ^ 1);
                    ready = ready && lookup(pc, 2 * pc.g + 1) &&
                            mbar_test(&bars[C::B_FULL + pc.slot], pc.par);
                    const uint32_t vslot = (uint32_t)pc.slot;
                    if (ready) {
                        fence_after_sync();
                        // a partial tile: only the 16-key steps that hold valid keys
                        // are multiplied; the rows of the last step past the chunk's
                        // end are zeroed first, so that 0 * (whatever the slot holds
                        // there) cannot reach O
                        const int nv = pc.t == pc.n_tiles - 1 ? pc.last_keys : kTcTileKeys;
                        const int steps = (nv + 15) >> 4;
                        uint8_t *vt = ring + vslot * C::TILE_BYTES;
                        if (nv & 15) {
                            // key rows [nv, 16 * steps) of every slab: a lane clears one
                            // 16-byte chunk of four rows per pass
                            const int row = nv + (lane >> 3), q = lane & 7;
#pragma unroll
                            for (int s = 0; s < SLABS; ++s) {
#pragma unroll
                                for (int r4 = 0; r4 < 16; r4 += 4) {
                                    const int r = row + r4;
                                    if (r < steps * 16)
                                        reinterpret_cast<uint4 *>(vt + (r >> 3) * C::ATOM_BYTES +
                                                                  s * 1024 + (r & 7) * 128)[q] =
                                            make_uint4(0, 0, 0, 0);
                                }
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                        }
                        if (pc.t == 0 && pc.head > 0) {
                            // (paged cache) the rows before the chunk in its first
                            // tile: P is 0 there, but they may hold anything
                            const int row = lane >> 3, q = lane & 7;
#pragma unroll
                            for (int s = 0; s < SLABS; ++s)
#pragma unroll
                                for (int r4 = 0; r4 < 8; r4 += 4)
                                    if (row + r4 < pc.head)
                                        reinterpret_cast<uint4 *>(vt + s * 1024 + (row + r4) * 128)[q] =
                                            make_uint4(0, 0, 0, 0);
                            fence_proxy_async_smem();
                            __syncwarp();
                        }
                        if (leader) {
                            // descriptors differ only in the start address (16-byte
                            // units in the low bits), so offsets are added to a base
                            const uint64_t bbase =
                                smem_desc_sw128(ps_a + pb * C::P_BUF, 16, 1024);
                            // A = V^T, MN-major: 64-dim blocks one slab (1024 B) apart,
                            // 8-key groups one atom apart
                            const uint64_t abase = smem_desc_sw128(
                                ring_a + vslot * C::TILE_BYTES, 1024, C::ATOM_BYTES);
                            const uint32_t ob = pc.k % OB;
                            const uint32_t acc0 = pc.t > 0 ? 1u : 0u;
#pragma unroll
                            for (int mh = 0; mh < MH; ++mh) {
                                const uint64_t ah = abase + (uint64_t)(mh * (2048 >> 4));
                                const uint32_t d_t = tmem + C::O_COL + ob * C::O_COLS + mh * 2 * N;
                                // B = [P_hi; P_lo], 2N rows
                                if (steps == 8) {
#pragma unroll
                                    for (int k8 = 0; k8 < 8; ++k8)
                                        mma_bf16_ss(d_t, ah + (uint64_t)(k8 * (2 * C::ATOM_BYTES >> 4)),
                                                    bbase + (uint64_t)((k8 >> 2) * (C::P_KSLAB >> 4) +
                                                                       (k8 & 3) * 2),
                                                    ID_PV, (acc0 | (uint32_t)k8) != 0);
                                } else {
                                    for (int k8 = 0; k8 < steps; ++k8)
                                        mma_bf16_ss(d_t, ah + (uint64_t)(k8 * (2 * C::ATOM_BYTES >> 4)),
                                                    bbase + (uint64_t)((k8 >> 2) * (C::P_KSLAB >> 4) +
                                                                       (k8 & 3) * 2),
                                                    ID_PV, (acc0 | (uint32_t)k8) != 0);
                                }
                            }
                            mma_commit(&bars[C::B_EMPTY + vslot]);
                            mma_commit(&bars[C::B_PVDONE + pb]);
                        }
                        __syncwarp();
                        advance(pc);
                        progressed = true;
                    }
                }
                // ---- S of tile qc.g, at most one tile ahead of the PV cursor: the
                // tensor pipe runs in issue order, so an S batch issued early
                // would hold back the PV that the softmax warps wait for
                if (qc.valid && qc.g <= pc.g + 1) {
                    const uint32_t sb = qc.g & 1;
                    bool ready = mbar_test(&bars[C::B_SFREE + sb], ((qc.g >> 1) & 1) ^ 1) &&
                                 mbar_test(&bars[C::B_QFULL + qc.k % QB], (qc.k / QB) & 1) &&
                                 lookup(qc, 2 * qc.g) &&
                                 mbar_test(&bars[C::B_FULL + qc.slot], qc.par);
                    const uint32_t kslot = (uint32_t)qc.slot;
                    if (ready) {
                        fence_after_sync();
                        if (leader) {
                            const uint64_t qbase =
                                smem_desc_sw128(qs_a + (qc.k % QB) * C::Q_BUF, 16, 1024);
                            // A = K, K-major: 8-key groups one atom apart, the 64-dim
                            // slab s at s * 1024 B
                            const uint64_t abase =
                                smem_desc_sw128(ring_a + kslot * C::TILE_BYTES, 16, C::ATOM_BYTES);
#pragma unroll
                            for (int s = 0; s < SLABS; ++s) {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_bf16_ss(tmem + sb * N, abase + (uint64_t)(s * 64 + kk * 2),
                                                qbase + (uint64_t)(s * (C::Q_SLAB >> 4) + kk * 2),
                                                ID_QK, (s | kk) != 0);
                            }
                            mma_commit(&bars[C::B_EMPTY + kslot]);
                            mma_commit(&bars[C::B_SFULL + sb]);
                            if (qc.t == qc.n_tiles - 1)
                                mma_commit(&bars[C::B_QEMPTY + qc.k % QB]);
                        }
                        __syncwarp();
                        advance(qc);
                        progressed = true;
                    }
                }
                if (progressed) {
                    idle_since = clock64();
                    idle = 0;
                } else if (clock64() - idle_since < P.wait_limit) {
                    ++idle;
                } else {
                    atomicOr(P.fault, kFaultCopyTimeout);
                    ok = false;
                    break;
                }
            }
            (void)ok;
            // all issued MMAs complete before TMEM is released
            if (leader) {
                mma_commit(&bars[C::B_DRAIN]);
                mbar_wait_bounded(&bars[C::B_DRAIN], 0, P.fault, kFaultCopyTimeout, P.wait_limit);
            }
            __syncwarp();
        }
    } else if (warp < 10) {
        // ===================================================== softmax
        constexpr int HN = N / 2;                 // rows per softmax warpgroup
        constexpr int CWH = HN >= 32 ? 32 : HN;  // TMEM columns per S load
        constexpr int NCH = HN / CWH;
        constexpr int OW = HN >= 16 ? 16 : 8;    // TMEM columns per O load / store
        const int wg = (warp - 2) >> 2;          // softmax warpgroup
        const int sw = (warp - 2) & 3;           // warp within the group
        const int quad = warp & 3;               // TMEM lane quadrant of this warp
        const int lk = quad * 32 + lane;         // TMEM lane: key of S^T, dim row of O^T
        const int gtid = sw * 32 + lane;         // 0..127 within the group
        const int r0 = wg * HN;                  // first packed row of this group
        const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
        // P^T address pieces of this thread's key: the 16-byte chunk index
        // of key lk inside a 128-byte row is XORed with (row & 7)
        const uint32_t p_key = (uint32_t)(lk >> 6) * C::P_KSLAB + (uint32_t)(lk & 7) * 2;
        const uint32_t p_chunk = (uint32_t)(lk & 63) >> 3;
        uint32_t g = 0, k = 0;
        bool ok = true;
        const int n_items = cta_items(T);
        for (int j = 0; j < n_items && ok; ++j) {
            const TcItem it = tc_decode<AP>(T, cta_item(T, j), j, meta);
            const size_t bh = (size_t)it.b * P.Hkv + it.h;
            const int my_rows = min(HN, it.rows - r0);  // rows of this group in the item
            if (it.n_tiles == 0) {
                // no key in this chunk: empty result for every row
                for (int idx = gtid; idx < my_rows * D; idx += 128) {
                    const int r = it.row0 + r0 + idx / D, d = idx % D;
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
            const uint32_t ob = k % OB;
            const uint32_t ocol0 = tl + C::O_COL + ob * C::O_COLS;  // this lane's O^T row
            float mref[HN], lrow[HN];
#pragma unroll
            for (int r = 0; r < HN; ++r) {
                mref[r] = kNoRef;
                lrow[r] = 0.f;
            }

            const int qp_i0 = it.cr.qp + it.i0;  // position of the item's first draft row
            for (int t = 0; t < it.n_tiles; ++t, ++g) {
                const uint32_t sb = g & 1, suse = g >> 1;
                // (a failed wait is voted on together with the raise below: one
                // group barrier per tile when nothing is raised)
                const bool got = mbar_wait_bounded(&bars[C::B_SFULL + sb], suse & 1, P.fault,
                                                   kFaultCopyTimeout, P.wait_limit);
                fence_after_sync();
                const int j0 = it.t0 + kTcTileKeys * t;
                const int n_valid = min(kTcTileKeys, it.cr.c_hi - j0);
                const int jk = j0 + lk;
                // packed rows [ra, rb) of this item whose window holds key jk:
                // draft row i sees jk iff p_i - W < jk <= p_i, p_i = qp_i0 + i;
                // shifted to this group's rows
                int ra = 0, rb = 0;
                if (lk < n_valid && jk >= it.cr.c_lo) {
                    const long long lo_i = (long long)jk - qp_i0;
                    const long long hi_i = (long long)jk + P.window - qp_i0;
                    const long long a = lo_i < 0 ? 0 : lo_i * P.G;
                    long long bnd = hi_i < 0 ? 0 : hi_i * P.G;
                    if (bnd > it.rows) bnd = it.rows;
                    ra = (int)(a < it.rows ? a : it.rows) - r0;
                    rb = (int)bnd - r0;
                }
                // this group's scores into registers, then hand the S buffer back
                float v[HN];
                {
                    uint32_t raw[HN];
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        tmem_load<CWH>(tl + sb * N + r0 + c * CWH, raw + c * CWH);
                    tmem_wait_ld();
                    if (ra <= 0 && rb >= HN) {
                        // (pairs of rows through packed fp32 arithmetic)
                        const uint64_t sc2 = f2_pack(P.qk_scale, P.qk_scale);
#pragma unroll
                        for (int r = 0; r < HN; r += 2)
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(raw[r]), __uint_as_float(raw[r + 1])),
                                             sc2),
                                      v[r], v[r + 1]);
                    } else {
#pragma unroll
                        for (int r = 0; r < HN; ++r)
                            v[r] = (r >= ra && r < rb) ? __uint_as_float(raw[r]) * P.qk_scale
                                                       : NEG_INF;
                    }
                }
                fence_before_sync();
                mbar_arrive(&bars[C::B_SFREE + sb]);

                bool flag = false;
#pragma unroll
                for (int r = 0; r < HN; ++r) flag |= v[r] > mref[r] + 8.f;
                const bool raise = group_any(wg, flag || !got);
                if (raise) {
                    ok = !group_any(wg, !got);
                    if (!ok) break;
                }
                if (raise) {
                    // exact tile maximum per row; raise the references
                    float *rd = red + (g & 1) * 4 * N + r0;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        float tmp[CWH];
#pragma unroll
                        for (int e = 0; e < CWH; ++e) tmp[e] = v[c * CWH + e];
                        const float m = lane_reduce<CWH, true>(tmp);
                        if (lane < CWH) rd[sw * N + c * CWH + lane] = m;
                    }
                    group_sync(wg);
                    const bool rescale = t > 0;
                    // all four warps' maxima first (no shared-memory store in
                    // between, so the loads issue back to back), then the
                    // references and the rescale factor
                    float tm[HN];
#pragma unroll
                    for (int r4 = 0; r4 < HN; r4 += 4) {
                        const float4 a0 = *reinterpret_cast<const float4 *>(rd + r4);
                        const float4 a1 = *reinterpret_cast<const float4 *>(rd + N + r4);
                        const float4 a2 = *reinterpret_cast<const float4 *>(rd + 2 * N + r4);
                        const float4 a3 = *reinterpret_cast<const float4 *>(rd + 3 * N + r4);
                        tm[r4] = fmaxf(fmaxf(a0.x, a1.x), fmaxf(a2.x, a3.x));
                        tm[r4 + 1] = fmaxf(fmaxf(a0.y, a1.y), fmaxf(a2.y, a3.y));
                        tm[r4 + 2] = fmaxf(fmaxf(a0.z, a1.z), fmaxf(a2.z, a3.z));
                        tm[r4 + 3] = fmaxf(fmaxf(a0.w, a1.w), fmaxf(a2.w, a3.w));
                    }
                    float my_alpha = 1.f;
                    if (!rescale) {
                        // the item's first tile: its maxima are the references (the
                        // row sums are still 0, so nothing is rescaled)
#pragma unroll
                        for (int r = 0; r < HN; ++r) mref[r] = fmaxf(mref[r], tm[r]);
                    } else {
#pragma unroll
                        for (int r = 0; r < HN; ++r) {
                            const float mo = mref[r];
                            const float mn = fmaxf(mo, tm[r]);
                            const float al = mn == mo ? 1.f : fast_exp2(mo - mn);
                            if (gtid == r) my_alpha = al;
                            lrow[r] *= al;
                            mref[r] = mn;
                        }
                    }
                    if (rescale && gtid < HN) alpha_sm[r0 + gtid] = my_alpha;
                    if (rescale) {
                        // every PV of this item so far has completed before O is scaled
                        const uint32_t gp = g - 1;
                        ok = !group_any(wg, !mbar_wait_bounded(&bars[C::B_PVDONE + gp % PB],
                                                               (gp / PB) & 1, P.fault,
                                                               kFaultCopyTimeout, P.wait_limit));
                        if (!ok) break;
                        fence_after_sync();  // (the vote also published alpha_sm)
#pragma unroll 1
                        for (int mh = 0; mh < 2 * MH; ++mh) {  // hi and lo halves of each
#pragma unroll 1
                            for (int c0 = 0; c0 < HN; c0 += OW) {
                                uint32_t o[OW];
                                const uint32_t ocol = ocol0 + mh * N + r0 + c0;
                                tmem_load<OW>(ocol, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int e = 0; e < OW; ++e)
                                    o[e] = __float_as_uint(__uint_as_float(o[e]) *
                                                           alpha_sm[r0 + c0 + e]);
                                tmem_store<OW>(ocol, o);
                            }
                        }
                        tmem_wait_st();
                    }
                }
                // P buffer free: its previous PV has completed
                const uint32_t pb = g % PB;
                if (g >= (uint32_t)PB && !(raise && t > 0 && PB == 1)) {
                    const uint32_t gp = g - PB;
                    ok = !group_any(wg, !mbar_wait_bounded(&bars[C::B_PVDONE + pb],
                                                           (gp / PB) & 1, P.fault,
                                                           kFaultCopyTimeout, P.wait_limit));
                    if (!ok) break;
                }
                // the previous item's epilogue staged its output in the P buffers
                if (t == 0 && k > 0) group_sync(wg);
                // P = 2^(s - m_ref) as bf16 hi + lo into the swizzled P^T tiles:
                // P_hi = P truncated to bf16, P_lo = the rest rounded to bf16
                // (P_hi + P_lo within 2^-16 of P).  Row r0 + r of the tile; r0
                // is a multiple of 8, so the row's swizzle phase is r & 7.
                uint8_t *pt = ps + pb * C::P_BUF + p_key + r0 * 128;
                // (pairs of rows through packed fp32 arithmetic)
#pragma unroll
                for (int r = 0; r < HN; r += 2) {
                    float d0, d1;
                    f2_unpack(f2_sub(f2_pack(v[r], v[r + 1]), f2_pack(mref[r], mref[r + 1])), d0, d1);
                    const float p0 = fast_exp2(d0), p1 = fast_exp2(d1);
                    const uint64_t p2 = f2_pack(p0, p1);
                    f2_unpack(f2_add(f2_pack(lrow[r], lrow[r + 1]), p2), lrow[r], lrow[r + 1]);
                    const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
                    float lo0, lo1;
                    f2_unpack(f2_sub(p2, f2_pack(__uint_as_float(b0 & 0xffff0000u),
                                                 __uint_as_float(b1 & 0xffff0000u))),
                              lo0, lo1);
                    const uint32_t sw0 = (p_chunk ^ (uint32_t)(r & 7)) << 4;
                    const uint32_t sw1 = (p_chunk ^ (uint32_t)((r + 1) & 7)) << 4;
                    *reinterpret_cast<uint16_t *>(pt + r * 128 + sw0) = (uint16_t)(b0 >> 16);
                    *reinterpret_cast<uint16_t *>(pt + (r + 1) * 128 + sw1) = (uint16_t)(b1 >> 16);
                    *reinterpret_cast<uint16_t *>(pt + (N + r) * 128 + sw0) =
                        __bfloat16_as_ushort(__float2bfloat16_rn(lo0));
                    *reinterpret_cast<uint16_t *>(pt + (N + r + 1) * 128 + sw1) =
                        __bfloat16_as_ushort(__float2bfloat16_rn(lo1));
                }
                fence_proxy_async_smem();
                mbar_arrive(&bars[C::B_PFULL + pb]);
            }
            if (!ok) break;

            // -------------------------------------------------- epilogue
            // row sums (they do not depend on the last PV): lanes, then the
            // group's four warps
            float *rl = red + (g & 1) * 4 * N + r0;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                float tmp[CWH];
#pragma unroll
                for (int e = 0; e < CWH; ++e) tmp[e] = lrow[c * CWH + e];
                const float s = lane_reduce<CWH, false>(tmp);
                if (lane < CWH) rl[sw * N + c * CWH + lane] = s;
            }
            group_sync(wg);
            if (gtid < my_rows) {
                const int r = gtid;
                const float l = (rl[r] + rl[N + r]) + (rl[2 * N + r] + rl[3 * N + r]);
                float m = NEG_INF;
#pragma unroll
                for (int q = 0; q < HN; ++q)
                    if (q == r) m = mref[q];
                linv[r0 + r] = l > 0.f ? __frcp_rn(l) : 0.f;
                const int rg = it.row0 + r0 + r;
                if (P.splits == 1) {
                    // output row of packed row rg: draft row rg / G of query head
                    // h * G + rg % G (below 2^31 by the plan's size checks)
                    const int i = rg / P.G, gg = rg - i * P.G;
                    const uint32_t orow =
                        (uint32_t)(((size_t)it.b * P.q_len + i) * P.Hq + (size_t)it.h * P.G + gg);
                    rowidx[r0 + r] = orow;
                    if (P.lse != nullptr)
                        P.lse[orow] = l > 0.f ? (m + __log2f(l)) * kLn2 : NEG_INF;
                } else {
                    const size_t prow = (bh * P.splits + it.split) * P.R + rg;
                    P.part_ml[prow * 2] = l > 0.f ? m : NEG_INF;
                    P.part_ml[prow * 2 + 1] = l;
                }
            }
            const uint32_t gl = g - 1;  // the item's last tile
            ok = !group_any(wg, !mbar_wait_bounded(&bars[C::B_PVDONE + gl % PB], (gl / PB) & 1,
                                                   P.fault, kFaultCopyTimeout, P.wait_limit));
            if (!ok) break;
            fence_after_sync();  // (the vote also published linv)
            // O^T through shared memory (the P buffers are idle now) into
            // 16-byte row stores: a bf16 row of D dims at a time, an fp32
            // partial row in halves of 128 dims.  A group stages its rows only
            // in the bytes of its own P rows (hi and lo, both key slabs), so
            // the other group's P writes for the next item cannot collide.
            // Staged row rr (RB bytes) of the group sits in the group's
            // 128-byte P rows, RPC staged rows per P row.
            auto stg_row = [&](int rr, int RB, int RPC) -> uint8_t * {
                const int c = rr / RPC;
                return ps + (c >> 1) * C::P_KSLAB + ((c & 1) * N + r0) * 128 + (rr % RPC) * RB;
            };
            if (P.splits == 1) {
                constexpr int RB = D * 2, RPC = HN * 128 / RB;
                // 1/l of the group's rows into registers first: no shared-memory
                // load then sits between the staging stores
                float li[HN];
#pragma unroll
                for (int r = 0; r < HN; ++r) li[r] = linv[r0 + r];
#pragma unroll
                for (int mh = 0; mh < MH; ++mh) {
#pragma unroll
                    for (int c0 = 0; c0 < HN; c0 += OW) {
                        uint32_t o[OW], ol[OW];
                        tmem_load<OW>(ocol0 + mh * 2 * N + r0 + c0, o);
                        tmem_load<OW>(ocol0 + mh * 2 * N + N + r0 + c0, ol);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < OW; ++e) {
                            const float ov = __uint_as_float(o[e]) + __uint_as_float(ol[e]);
                            *reinterpret_cast<__nv_bfloat16 *>(stg_row(c0 + e, RB, RPC) +
                                                               (mh * 128 + lk) * 2) =
                                __float2bfloat16_rn(ov * li[c0 + e]);
                        }
                    }
                }
                fence_before_sync();
                mbar_arrive(&bars[C::B_OFREE + ob]);  // O buffer may be reused
                group_sync(wg);
                constexpr int CPR = D / 8;  // 16-byte chunks per row
                for (int idx = gtid; idx < my_rows * CPR; idx += 128) {
                    const int r = idx / CPR, c = idx % CPR;
                    *reinterpret_cast<uint4 *>(P.out + (size_t)rowidx[r0 + r] * D + c * 8) =
                        *reinterpret_cast<const uint4 *>(stg_row(r, RB, RPC) + c * 16);
                }
                // (the group synchronises again before the staging area, a P
                // buffer, is written by the next item)
            } else {
                constexpr int RB = 512, RPC = HN * 128 / RB;
                const size_t prow0 = (bh * P.splits + it.split) * P.R + it.row0 + r0;
#pragma unroll 1
                for (int mh = 0; mh < MH; ++mh) {
#pragma unroll
                    for (int c0 = 0; c0 < HN; c0 += OW) {
                        uint32_t o[OW], ol[OW];
                        tmem_load<OW>(ocol0 + mh * 2 * N + r0 + c0, o);
                        tmem_load<OW>(ocol0 + mh * 2 * N + N + r0 + c0, ol);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < OW; ++e)
                            *reinterpret_cast<float *>(stg_row(c0 + e, RB, RPC) + lk * 4) =
                                __uint_as_float(o[e]) + __uint_as_float(ol[e]);
                    }
                    if (mh == MH - 1) {
                        fence_before_sync();
                        mbar_arrive(&bars[C::B_OFREE + ob]);  // O buffer may be reused
                    }
                    group_sync(wg);
                    for (int idx = gtid; idx < my_rows * 32; idx += 128) {
                        const int r = idx / 32, c = idx % 32;
                        *reinterpret_cast<uint4 *>(P.part_acc + (prow0 + r) * D + mh * 128 + c * 4) =
                            *reinterpret_cast<const uint4 *>(stg_row(r, RB, RPC) + c * 16);
                    }
                    group_sync(wg);
                }
            }
            ++k;
        }
    } else if constexpr (AP) {
        // ================================================= append worker
        append_worker<C, D>(T, meta, ftab, ring, bars);
    }

    // ---------------------------------------------------------- teardown
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
    if constexpr (AP) {
        if (cta_items(T) > 2) append_flush<D>(T, meta, ring, NT * C::TILE_BYTES, NTHR);
    }
}

}  // namespace swa
