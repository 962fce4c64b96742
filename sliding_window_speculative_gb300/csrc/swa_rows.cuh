// Tensor-core (tcgen05) split-KV kernel with query rows as the MMA's M
// dimension, for sliding-window verify attention.
//
// For every tile of 128 keys of a work item (sequence, KV head, key chunk,
// row tile of up to 128 packed rows):
//
//   S[128 rows x 128 keys] = Q[128 x D] . K_tile^T          (TMEM, fp32)
//   O[128 rows x D]       += P_hi . V_tile + P_lo . V_tile  (TMEM, fp32)
//
// The packed rows (G query heads of the KV head times the draft rows) are
// the TMEM lanes.  Two softmax threads own a row, one per half of the tile's
// keys (warps w and w + 4 share a TMEM lane quadrant): each keeps its half's
// maximum and sum in registers, the pair swaps the half maxima through
// shared memory once per tile so both use the same reference, and each
// writes P for its keys back into the TMEM columns of the S buffer (P_hi =
// bf16 truncation in columns 0..63, P_lo = the rest rounded to bf16 in
// 64..127) as the A operand of the two PV MMAs.  P never touches shared
// memory.
//
// Q sits in shared memory as [slab][QR rows][128 bytes] (QR = 32, 64 or
// 128); an MMA reads 128 rows per slab, so with fewer rows it reads past the
// buffer into the ring: those S rows are never used.  K and V tiles arrive
// exactly as for the key-major kernel (one 4D TMA per tile into first-free
// ring slots, atoms of [slab][8 rows][128 B]); K is the B operand of the
// score MMA (K-major), V the B operand of the PV MMAs (MN-major, N = D).
//
// Warp roles (320 threads, 352 under a fused append):
//   warp 0      TMA producer (lane 0 runs it; the warp issues a tile's copies)
//   warp 1      TMEM owner and MMA issuer (one lane)
//   warps 2..9  softmax / epilogue; warp w owns TMEM lanes 32 (w % 4)..,
//               i.e. packed rows 32 (w % 4).., and key half (w - 2) / 4 of
//               every tile (head-dim half of the output); quadrants without
//               rows idle.
//   warp 10     fused append only (the kernel's AP variant): mixed atoms of a
//               paged cache, and the new rows' cache stores
//
// TMEM: S/P buffers at columns 0 and 128, O at 256 (two O buffers at head
// dim 128).  Every wait is bounded; a wait that gives up sets the fault
// word and the roles leave their loops.
#pragma once

#include "swa_tc.cuh"

namespace swa {

constexpr int kRowsThreads = 320;  // and one append warp more under a fused append

template <int D, int QR, int NT, int QB>
struct RowsCfg {
    static constexpr int SLABS = D / 64;
    static constexpr int ATOM_BYTES = SLABS * 1024;  // 8 keys x D
    static constexpr int TILE_BYTES = (kTcTileKeys / 8) * ATOM_BYTES;
    static constexpr int Q_SLAB = QR * 128;          // QR rows x 64 dims
    static constexpr int Q_BUF = SLABS * Q_SLAB;
    static constexpr int Q_OFF = 0;                  // Q first: short-Q reads run into the ring
    static constexpr int RING_OFF = QB * Q_BUF;
    static constexpr int META_OFF = RING_OFF + NT * TILE_BYTES;  // TcItem [kTcMetaItems]
    static constexpr int FTAB_OFF = META_OFF + kTcMetaItems * (int)sizeof(TcItem);
    // the pairs' exchange: half maxima [tile parity][quadrant][half][lane],
    // half row sums [quadrant][half][lane]
    static constexpr int XM_OFF = (FTAB_OFF + kFillTab * 4 + 15) & ~15;
    static constexpr int XL_OFF = XM_OFF + 2 * 4 * 2 * 32 * 4;
    static constexpr int STG_OFF = (XL_OFF + 4 * 2 * 32 * 4 + 15) & ~15;  // 16-byte stores
    // output staging, 2 KB per softmax warp (32 rows x 64 bytes), where it fits
    static constexpr int STG_NEED = 8 * 2048;
    static constexpr bool STAGE = STG_OFF + STG_NEED + 1024 + 512 <= 227 * 1024;
    static constexpr int BAR_OFF = STG_OFF + (STAGE ? STG_NEED : 0);
    static constexpr int OB = D == 128 ? 2 : 1;      // O buffers in TMEM
    // ring full/empty [NT], q full/empty [QB], s full [2], s free [2],
    // p full [2], pv done [2], o free [OB], drain, mixed atom of a fused append [NT]
    static constexpr int B_FULL = 0, B_EMPTY = NT, B_QFULL = 2 * NT, B_QEMPTY = B_QFULL + QB,
                         B_SFULL = B_QEMPTY + QB, B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2,
                         B_PVDONE = B_PFULL + 2, B_OFREE = B_PVDONE + 2, B_DRAIN = B_OFREE + OB,
                         B_MIX = B_DRAIN + 1, NBARS = B_MIX + NT;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base
    static constexpr int END = MISC_OFF + 16;
    static constexpr int SMEM_BYTES = END + 1024;  // slack for 1024-byte alignment
    static constexpr int O_COL = 256;
    static constexpr int TMEM_COLS = 512;
    static_assert(QR == 32 || QR == 64 || QR == 128, "Q rows");
    static_assert(NT >= 2, "ring holds at least a K and a V tile");
    static_assert(O_COL + OB * D <= TMEM_COLS, "TMEM");
    static_assert(QB * Q_BUF - Q_SLAB + 128 * 128 <= RING_OFF + NT * TILE_BYTES,
                  "an MMA's 128-row read of the last Q slab stays in shared memory");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(STG_OFF % 16 == 0 && BAR_OFF % 8 == 0 && META_OFF % 8 == 0, "alignment");
};

template <int D, int QR, int NT, int QB, bool AP>
__global__ void __launch_bounds__(AP ? kRowsThreads + 32 : kRowsThreads, 1)
    swa_rows_kernel(const __grid_constant__ TcParams T, const __grid_constant__ TcMaps M) {
    using C = RowsCfg<D, QR, NT, QB>;
    constexpr int NTHR = AP ? kRowsThreads + 32 : kRowsThreads;
    using namespace tc;
    constexpr int SLABS = C::SLABS;
    constexpr int OB = C::OB;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const AttnParams &P = T.a;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    uint8_t *qs = sm + C::Q_OFF;
    uint8_t *ring = sm + C::RING_OFF;
    TcItem *meta = reinterpret_cast<TcItem *>(sm + C::META_OFF);
    volatile uint32_t *ftab = reinterpret_cast<volatile uint32_t *>(sm + C::FTAB_OFF);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + C::MISC_OFF);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // quadrants (warps of 32 rows) that hold packed rows of an item
    const int act_q = (T.rows_per_tile + 31) >> 5;
    const uint32_t n_act = 32u * (uint32_t)act_q;

    // ---------------------------------------------------------------- setup
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
            mbar_init(&bars[C::B_SFREE + i], 1);
            mbar_init(&bars[C::B_PFULL + i], 2 * n_act);
            mbar_init(&bars[C::B_PVDONE + i], 1);
        }
        for (int i = 0; i < OB; ++i) mbar_init(&bars[C::B_OFREE + i], 2 * n_act);
        mbar_init(&bars[C::B_DRAIN], 1);
        fence_barrier_init();
    }
    for (int i = tid; i < kFillTab; i += NTHR) ftab[i] = 0xffffffffu;
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    grid_dep_wait();
    grid_dep_trigger();
    for (int j = tid; j < kTcMetaItems; j += NTHR)
        if (j < cta_items(T)) meta[j] = tc_decode_global<AP>(T, cta_item(T, j));
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ======================================================= producer
        tile_producer<C, NT, QB, AP>(T, M, meta, ftab, ring, qs, bars, false);
    } else if (warp == 1) {
        // ============================================================ MMA
        // Two cursors over the tile sequence: S = Q K^T of the next tile and
        // O += P_hi V + P_lo V of the oldest tile whose P is in TMEM, each
        // issued as soon as its operands are there (S at most one tile ahead
        // of PV).  The whole warp runs the loop; lane 0 issues.
        {
            const bool leader = lane == 0;
            constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t ID_O = idesc_bf16_f32(128, D, 0, 1);
            const uint32_t ring_a = smem_u32(ring);
            const uint32_t qs_a = smem_u32(qs);
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
            while (pc.valid) {
                bool progressed = false;
                // ---- PV of tile pc.g (its S was issued before)
                if (pc.g < qc.g || !qc.valid) {
                    const uint32_t sb = pc.g & 1;
                    bool ready = mbar_test(&bars[C::B_PFULL + sb], (pc.g >> 1) & 1);
                    if (ready && pc.t == 0)
                        ready = mbar_test(&bars[C::B_OFREE + pc.k % OB], ((pc.k / OB) & 1) ^ 1);
                    ready = ready && lookup(pc, 2 * pc.g + 1) &&
                            mbar_test(&bars[C::B_FULL + pc.slot], pc.par);
                    if (ready) {
                        const uint32_t vslot = (uint32_t)pc.slot;
                        fence_after_sync();
                        // a partial tile: only the 16-key steps that hold valid keys
                        // are multiplied; the V rows of the last step past the
                        // chunk's end are zeroed first (P is 0 there, but the slot
                        // may hold anything)
                        const int nv = pc.t == pc.n_tiles - 1 ? pc.last_keys : kTcTileKeys;
                        const int steps = (nv + 15) >> 4;
                        uint8_t *vt = ring + vslot * C::TILE_BYTES;
                        if (nv & 15) {
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
                            // B = V, MN-major: 64-dim blocks one slab (1024 B) apart,
                            // 8-key groups one atom apart; a 16-key step is two atoms
                            const uint64_t vbase = smem_desc_sw128(ring_a + vslot * C::TILE_BYTES,
                                                                   1024, C::ATOM_BYTES);
                            const uint32_t d_t = tmem + C::O_COL + (pc.k % OB) * D;
                            const uint32_t p_t = tmem + sb * 128;  // P_hi; P_lo at +64
                            const uint32_t acc0 = pc.t > 0 ? 1u : 0u;
                            for (int k8 = 0; k8 < steps; ++k8)
                                mma_bf16_ts(d_t, p_t + k8 * 8,
                                            vbase + (uint64_t)(k8 * (2 * C::ATOM_BYTES >> 4)), ID_O,
                                            (acc0 | (uint32_t)k8) != 0);
                            for (int k8 = 0; k8 < steps; ++k8)
                                mma_bf16_ts(d_t, p_t + 64 + k8 * 8,
                                            vbase + (uint64_t)(k8 * (2 * C::ATOM_BYTES >> 4)), ID_O, 1u);
                            mma_commit(&bars[C::B_EMPTY + vslot]);
                            mma_commit(&bars[C::B_SFREE + sb]);
                            mma_commit(&bars[C::B_PVDONE + sb]);
                        }
                        __syncwarp();
                        advance(pc);
                        progressed = true;
                    }
                }
                // ---- S of tile qc.g, at most one tile ahead of the PV cursor
                if (qc.valid && qc.g <= pc.g + 1) {
                    const uint32_t sb = qc.g & 1;
                    bool ready = mbar_test(&bars[C::B_SFREE + sb], ((qc.g >> 1) & 1) ^ 1) &&
                                 mbar_test(&bars[C::B_QFULL + qc.k % QB], (qc.k / QB) & 1) &&
                                 lookup(qc, 2 * qc.g) &&
                                 mbar_test(&bars[C::B_FULL + qc.slot], qc.par);
                    if (ready) {
                        const uint32_t kslot = (uint32_t)qc.slot;
                        fence_after_sync();
                        if (leader) {
                            // A = Q, K-major: 8-row groups 1024 B apart, slab s at
                            // s * Q_SLAB; B = K, K-major: 8-key groups one atom apart,
                            // slab s at s * 1024
                            const uint64_t qbase =
                                smem_desc_sw128(qs_a + (qc.k % QB) * C::Q_BUF, 16, 1024);
                            const uint64_t kbase =
                                smem_desc_sw128(ring_a + kslot * C::TILE_BYTES, 16, C::ATOM_BYTES);
#pragma unroll
                            for (int s = 0; s < SLABS; ++s) {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_bf16_ss(tmem + sb * 128,
                                                qbase + (uint64_t)(s * (C::Q_SLAB >> 4) + kk * 2),
                                                kbase + (uint64_t)(s * 64 + kk * 2), ID_S,
                                                (s | kk) != 0);
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
                } else if (clock64() - idle_since > P.wait_limit) {
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
        const int quad = warp & 3;        // TMEM lane quadrant = packed rows 32 quad ..
        const int half = (warp - 2) >> 2;  // key half of each tile, head-dim half of O
        if (quad < act_q) {
            const int r = quad * 32 + lane;  // packed row within the row tile
            const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
            float *xm = reinterpret_cast<float *>(sm + C::XM_OFF);
            float *xl = reinterpret_cast<float *>(sm + C::XL_OFF) + (quad * 2) * 32 + lane;
            const int kh = 64 * half;  // first key of this thread's half
            constexpr int DH = D / 2;  // head dims of this thread's half of O
            const float sc = P.qk_scale;
            // the pair of warps of this quadrant (64 threads), barrier 1 + quad
            auto pair_sync = [&]() {
                asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
            };
            uint32_t g = 0, k = 0;
            bool ok = true;
            const int n_items = cta_items(T);
            for (int j = 0; j < n_items && ok; ++j) {
                const TcItem it = tc_decode<AP>(T, cta_item(T, j), j, meta);
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
                const uint32_t ob = k % OB;
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
                        const uint32_t oc = tl + C::O_COL + ob * D + half * DH;
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
                    mbar_arrive(&bars[C::B_PFULL + sb]);
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
                const uint32_t oc = tl + C::O_COL + ob * D + half * DH;
                if (P.splits == 1 && C::STAGE) {
                    // 32 dims of the warp's 32 rows at a time through a 2 KB staging
                    // buffer ([row][4 x 16 B], chunk index XOR (row >> 1) & 3 against
                    // bank conflicts), then stored as 8 rows x 64 B per instruction
                    const float inv = ltot > 0.f ? __frcp_rn(ltot) : 0.f;
                    uint8_t *stg = sm + C::STG_OFF + (warp - 2) * 2048;
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
                } else if (P.splits == 1) {
                    const float inv = ltot > 0.f ? __frcp_rn(ltot) : 0.f;
#pragma unroll 1
                    for (int c0 = 0; c0 < DH; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(oc + c0, o);
                        tmem_wait_ld();
                        if (live) {
                            uint4 *dst = reinterpret_cast<uint4 *>(P.out + orow * D + half * DH + c0);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                uint4 w;
                                w.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv,
                                                  __uint_as_float(o[8 * q4 + 1]) * inv);
                                w.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv,
                                                  __uint_as_float(o[8 * q4 + 3]) * inv);
                                w.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv,
                                                  __uint_as_float(o[8 * q4 + 5]) * inv);
                                w.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv,
                                                  __uint_as_float(o[8 * q4 + 7]) * inv);
                                dst[q4] = w;
                            }
                        }
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
                mbar_arrive(&bars[C::B_OFREE + ob]);  // O buffer may be reused
                ++k;
            }
            (void)ok;
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
