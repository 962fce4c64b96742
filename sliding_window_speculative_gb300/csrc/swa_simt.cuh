// CUDA-core split-KV chunk kernel for sliding-window verify attention.
//
// One CTA = one (chunk of the window span, KV head, row tile, sequence).
// The K and V rows of the chunk stream through a ring of shared-memory
// stages, each filled by two bulk copies on the TMA engine (a sequence's
// rows of one KV head are contiguous, so a tile of keys is one contiguous
// block).  Four warps split the CTA's packed query rows (the G query heads
// of the KV head times the q_len draft rows, so each K/V byte is read once
// per KV head) and/or the keys of each tile.  Scores, an online softmax in
// the log2 domain and the PV accumulation run in fp32 on the CUDA cores:
//
//   lanes split head_dim; a lane holds RPW query rows x D/32 dims in
//   registers; for every group of 32/RPW keys the 32 (key, row) partial
//   dot products are summed across the warp with a reduce-scatter
//   butterfly (31 shuffles) that leaves one finished score per lane.
//
// The chunk's result is either the final output (one chunk per sequence)
// or a partial (m, l, acc) for the log-sum-exp merge kernel.
#pragma once

#include "swa_common.cuh"

namespace swa {

constexpr int kSimtThreads = 128;
constexpr int kSimtTileKeys = 32;

struct AttnParams {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k;
    const __nv_bfloat16 *v;
    const int32_t *seq_lens;
    const int32_t *q_pos;
    __nv_bfloat16 *out;
    float *lse;
    float *part_acc;  // [B*Hkv, splits, R, D]  (splits > 1)
    float *part_ml;   // [B*Hkv, splits, R, 2]
    uint32_t *fault;  // device fault word (bounded waits that gave up)
    // paged cache (block_table non-null): k/v are [pages, Hkv, page_size, D]
    // and key position j of sequence b lives in page block_table[b][j / page_size]
    const int32_t *block_table;  // [B, max_blocks]
    int page_size, max_blocks, num_pages;
    // fused append (k_new non-null): the q_len new rows [B, q_len, Hkv, D] of
    // every KV head, key positions q_pos + i, are attended from here and
    // stored to the cache; k / v then point at writable caches
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    int B, q_len, Hq, Hkv, G, L, window, R;
    int splits, chunk, row_tiles, rows_per_tile;
    float qk_scale;   // scale * log2(e)
    // bounded waits give up after this many SM cycles (kWaitLimitCycles
    // unless a test shortened it)
    long long wait_limit;
    // tests of the bounded waits only (-1 otherwise): the producer of the
    // first CTA posts this fill (K/V tile, or stage) but never issues its
    // copies, so every wait on it runs out
    int withhold_fill;
};

// Chunk `split` [lo, hi) of sequence b's window span (clamped to the
// sequence's own slab [0, L)), and the keys [c_lo, c_hi) a work item reads:
// the chunk, narrowed to the windows of the item's draft rows.
struct ChunkRange {
    int lo, hi;     // the chunk
    int c_lo, c_hi; // keys read
    int qp;         // q_pos of the sequence
};

__device__ __forceinline__ ChunkRange chunk_range_of(const AttnParams &P, long long qp,
                                                     long long sl, int split) {
    ChunkRange c;
    if constexpr (kDebugChecks)
        if (sl < 0 || sl > P.L) debug_oob(P.fault);
    long long hi = qp + P.q_len;
    if (hi > sl) hi = sl;
    if (hi > P.L) hi = P.L;
    if (hi < 0) hi = 0;
    long long lo = qp - P.window + 1;
    if (lo < 0) lo = 0;
    if (lo > hi) lo = hi;
    long long clo = lo + (long long)split * P.chunk;
    long long chi = clo + P.chunk;
    if (clo > hi) clo = hi;
    if (chi > hi) chi = hi;
    c.lo = c.c_lo = (int)clo;
    c.hi = c.c_hi = (int)chi;
    c.qp = (int)(qp < -(1LL << 30) ? -(1LL << 30) : (qp > (1LL << 30) ? (1LL << 30) : qp));
    return c;
}

// The chunk of a work item holding draft rows [i_first, i_last]: the keys
// it reads narrowed to the union of those rows' windows,
// [q_pos + i_first - W + 1, q_pos + i_last] (a row tile of a long block,
// e.g. a 512-token prefill chunk, sees W + its rows - 1 keys, not the whole
// span).
__device__ __forceinline__ ChunkRange chunk_range(const AttnParams &P, int b, int split,
                                                  int i_first, int i_last) {
    ChunkRange c = chunk_range_of(P, P.q_pos[b], P.seq_lens[b], split);
    const long long lo = (long long)c.qp + i_first - P.window + 1;
    const long long hi = (long long)c.qp + i_last + 1;
    if (lo > c.c_lo) c.c_lo = (int)(lo < c.c_hi ? lo : c.c_hi);
    if (hi < c.c_hi) c.c_hi = (int)(hi > c.c_lo ? hi : c.c_lo);
    return c;
}

// A block-table page, checked in SWA_DEBUG_CHECKS builds: one outside
// [0, num_pages) is counted, `bad` set and page 0 used instead.
__device__ __forceinline__ int checked_page(const AttnParams &P, int page, bool *bad) {
    if constexpr (kDebugChecks) {
        if (page < 0 || page >= P.num_pages) {
            debug_oob(P.fault);
            if (bad != nullptr) *bad = true;
            return 0;
        }
    }
    return page;
}

// Cache row (in rows of D elements) of key position j of (sequence b, KV
// head h): contiguous [B, Hkv, L] or, with a block table, the page's row.
// `bad` (stores pass it) is set when a debug check replaced the page.
__device__ __forceinline__ long long cache_row(const AttnParams &P, int b, int h, int j,
                                               bool *bad = nullptr) {
    if (P.block_table == nullptr) return ((long long)b * P.Hkv + h) * P.L + j;
    const int page =
        checked_page(P, P.block_table[(long long)b * P.max_blocks + j / P.page_size], bad);
    return ((long long)page * P.Hkv + h) * P.page_size + (j % P.page_size);
}

// The new rows of a fused append that a work item (draft rows
// [i_first, i_last], its chunk cr) stores to the cache: positions
// q_pos + i of its own draft rows inside its chunk, so every new row has
// exactly one owner; empty without an append.  The kernels read new rows
// straight from k_new / v_new and no kernel reads one back from the cache,
// so the stores need no ordering against the tile loads.
__device__ __forceinline__ void append_range(const AttnParams &P, const ChunkRange &cr,
                                             int i_first, int i_last, int &lo, int &hi) {
    const long long a = (long long)cr.qp + i_first, e = (long long)cr.qp + i_last + 1;
    lo = (int)(a > cr.lo ? (a < cr.hi ? a : cr.hi) : cr.lo);
    hi = (int)(e < cr.hi ? (e > lo ? e : lo) : cr.hi);
    if (P.k_new == nullptr || hi < lo) hi = lo;
}

template <int D>
__device__ __forceinline__ void load_row_f32(const __nv_bfloat16 *src, float *dst) {
    // D/32 consecutive bf16 of one row owned by this lane.
    constexpr int DPL = D / 32;
    if constexpr (DPL == 8) {
        const uint4 w = *reinterpret_cast<const uint4 *>(src);
        dst[0] = bf16lo(w.x); dst[1] = bf16hi(w.x);
        dst[2] = bf16lo(w.y); dst[3] = bf16hi(w.y);
        dst[4] = bf16lo(w.z); dst[5] = bf16hi(w.z);
        dst[6] = bf16lo(w.w); dst[7] = bf16hi(w.w);
    } else if constexpr (DPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(src);
        dst[0] = bf16lo(w.x); dst[1] = bf16hi(w.x);
        dst[2] = bf16lo(w.y); dst[3] = bf16hi(w.y);
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(src);
        dst[0] = bf16lo(w); dst[1] = bf16hi(w);
    }
}

// Reduce-scatter of 32 per-lane values: afterwards lane l holds
// sum over all lanes of v[l].  v is consumed.
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int half = 16; half >= 1; half >>= 1) {
        const bool upper = (lane & half) != 0;
#pragma unroll
        for (int e = 0; e < half; ++e) {
            const float keep = upper ? v[e + half] : v[e];
            const float give = upper ? v[e] : v[e + half];
            v[e] = keep + __shfl_xor_sync(0xffffffffu, give, half);
        }
    }
    return v[0];
}

template <int D, int RPW, int NRG>
struct SimtCfg {
    static constexpr int NKG = 4 / NRG;                 // key groups (warps per row group)
    static constexpr int RPT = RPW * NRG;               // packed rows per CTA
    static constexpr int DPL = D / 32;                  // dims per lane
    static constexpr int KPG = 32 / RPW;                // keys per butterfly group
    static constexpr int KB = kSimtTileKeys / NKG;      // keys per warp per tile
    static constexpr int NG = KB / KPG;                 // butterfly groups per warp per tile
    static constexpr int STAGES = D == 256 ? 3 : 4;
    static constexpr int TILE_BYTES = kSimtTileKeys * D * 2;         // one of K or V
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int COMB_BYTES = NKG * RPT * D * 4 + NKG * RPT * 2 * 4;
    static constexpr int MAIN_BYTES = RING_BYTES > COMB_BYTES ? RING_BYTES : COMB_BYTES;
    static constexpr int PBUF_BYTES = 4 * KB * RPW * 4;
    static constexpr int SMEM_BYTES = MAIN_BYTES + PBUF_BYTES + STAGES * 8;
    static_assert(KB % KPG == 0, "key block must hold whole butterfly groups");
};

template <int D, int RPW, int NRG, bool AP>
__global__ void __launch_bounds__(kSimtThreads) swa_simt_kernel(const AttnParams P) {
    using C = SimtCfg<D, RPW, NRG>;
    constexpr int DPL = C::DPL;
    const float NEG_INF = -__int_as_float(0x7f800000);

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    float *pbuf_all = reinterpret_cast<float *>(smem + C::MAIN_BYTES);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::MAIN_BYTES + C::PBUF_BYTES);

    const int split = blockIdx.x;
    const int h = blockIdx.y / P.row_tiles;
    const int rt = blockIdx.y % P.row_tiles;
    const int b = blockIdx.z;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = warp % NRG, kg = warp / NRG;
    float *pbuf = pbuf_all + warp * (C::KB * RPW);

    grid_dep_wait();
    grid_dep_trigger();
    // draft rows of this CTA's packed rows [rt * RPT, min(R, rt * RPT + RPT))
    const int i_first = rt * C::RPT / P.G;
    const int i_last = (min(P.R, rt * C::RPT + C::RPT) - 1) / P.G;
    const ChunkRange cr = chunk_range(P, b, split, i_first, i_last);
    const int n_keys = cr.c_hi - cr.c_lo;
    const int n_tiles = n_keys > 0 ? (n_keys + kSimtTileKeys - 1) / kSimtTileKeys : 0;


    // keys read from k_new / v_new (every position >= q_pos under an append)
    // and the new rows this CTA stores to the cache; both empty in the plain
    // variant (AP false)
    int nw_lo = 0, nw_hi = 0, ap_lo = 0, ap_hi = 0;
    if constexpr (AP) {
        nw_lo = cr.c_lo > cr.qp ? cr.c_lo : cr.qp;
        nw_hi = cr.c_hi > nw_lo ? cr.c_hi : nw_lo;
        append_range(P, cr, i_first, i_last, ap_lo, ap_hi);
    }
    auto issue = [&](int t) {
        const int s = t % C::STAGES;
        const int j0 = cr.c_lo + t * kSimtTileKeys;
        const int n = min(kSimtTileKeys, cr.c_hi - j0);
        const uint32_t bytes = (uint32_t)n * D * 2;
        uint8_t *dst = ring + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        if (P.withhold_fill == t && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) return;
        // one copy per run of rows contiguous in the cache (a page's rows, or
        // the whole tile of a contiguous cache); a new row of a fused append
        // is one copy from k_new / v_new
        for (int j = j0; j < j0 + n;) {
            const uint32_t off = (uint32_t)(j - j0) * D * 2;
            if (AP && j >= nw_lo && j < nw_hi) {
                const size_t src = (((size_t)b * P.q_len + (j - cr.qp)) * P.Hkv + h) * D;
                bulk_copy_g2s(dst + off, P.k_new + src, D * 2, &full[s]);
                bulk_copy_g2s(dst + C::TILE_BYTES + off, P.v_new + src, D * 2, &full[s]);
                ++j;
                continue;
            }
            int run = (AP && nw_lo < nw_hi && j < nw_lo && nw_lo < j0 + n ? nw_lo : j0 + n) - j;
            if (P.block_table != nullptr) {
                const int left = P.page_size - j % P.page_size;
                run = run < left ? run : left;
            }
            const size_t row = (size_t)cache_row(P, b, h, j);
            const uint32_t rb = (uint32_t)run * D * 2;
            bulk_copy_g2s(dst + off, P.k + row * D, rb, &full[s]);
            bulk_copy_g2s(dst + C::TILE_BYTES + off, P.v + row * D, rb, &full[s]);
            j += run;
        }
    };
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int t = 0; t < C::STAGES - 1 && t < n_tiles; ++t) issue(t);
    }

    // ---- this lane's query rows (pre-scaled into the log2 domain)
    const int row0 = rt * C::RPT + rg * RPW;  // first packed row of this warp
    float qf[RPW][DPL];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int r = row0 + rr;
        if (r < P.R) {
            const int i = r / P.G, gg = r - (r / P.G) * P.G;
            const __nv_bfloat16 *src =
                P.q + (((size_t)b * P.q_len + i) * P.Hq + (size_t)h * P.G + gg) * D + lane * DPL;
            load_row_f32<D>(src, qf[rr]);
#pragma unroll
            for (int d = 0; d < DPL; ++d) qf[rr][d] *= P.qk_scale;
        } else {
#pragma unroll
            for (int d = 0; d < DPL; ++d) qf[rr][d] = 0.f;
        }
    }

    // ---- the row whose finished scores this lane holds after a butterfly
    const int r_own = row0 + (lane % RPW);
    int jlo_own = 1, jhi_own = 0;  // inclusive, empty by default
    if (r_own < P.R) {
        const int p = cr.qp + r_own / P.G;
        jlo_own = max(max(cr.c_lo, p - P.window + 1), 0);
        jhi_own = min(p, cr.c_hi - 1);
    }

    float m_own = NEG_INF, l_own = 0.f;
    float acc[RPW][DPL];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[rr][d] = 0.f;

    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
        if (tid == 0 && t + C::STAGES - 1 < n_tiles) {
            fence_proxy_async_smem();
            issue(t + C::STAGES - 1);
        }
        const int s = t % C::STAGES;
        if (!mbar_wait_bounded(&full[s], (t / C::STAGES) & 1, P.fault, kFaultCopyTimeout,
                               P.wait_limit)) {
            // the stages issued after this one land before the CTA leaves
            if (tid == 0)
                for (int t2 = t + 1; t2 < n_tiles && t2 < t + C::STAGES; ++t2)
                    mbar_wait_bounded(&full[t2 % C::STAGES], (t2 / C::STAGES) & 1, P.fault,
                                      kFaultCopyTimeout, P.wait_limit);
            ok = false;
            break;
        }
        const __nv_bfloat16 *Ks = reinterpret_cast<const __nv_bfloat16 *>(ring + s * C::STAGE_BYTES);
        const __nv_bfloat16 *Vs = Ks + kSimtTileKeys * D;
        const int j0 = cr.c_lo + t * kSimtTileKeys;
        const int n = min(kSimtTileKeys, cr.c_hi - j0);
        if constexpr (AP) {
            // the fused append's new rows of this tile that this CTA owns, from
            // the stage to the cache
            const int r0 = max(ap_lo, j0) - j0, r1 = min(ap_hi, j0 + n) - j0;
            constexpr int PR = D / 8;
            for (int e = tid; e < 2 * (r1 - r0) * PR; e += kSimtThreads) {
                const int kv = e >= (r1 - r0) * PR, rest = e - kv * (r1 - r0) * PR;
                const int r = r0 + rest / PR, c = rest % PR;
                const uint4 w = *reinterpret_cast<const uint4 *>((kv ? Vs : Ks) + (size_t)r * D + c * 8);
                __nv_bfloat16 *cache = const_cast<__nv_bfloat16 *>(kv ? P.v : P.k);
                bool bad = false;
                const long long row = cache_row(P, b, h, j0 + r, &bad);
                if (!bad) *reinterpret_cast<uint4 *>(cache + row * D + c * 8) = w;
            }
        }
        const int kb0 = kg * C::KB;

        // scores of this warp's key block: one finished (key, row) per lane per group
        float sc[C::NG];
#pragma unroll
        for (int grp = 0; grp < C::NG; ++grp) {
            float v[32];
#pragma unroll
            for (int kk = 0; kk < C::KPG; ++kk) {
                float kf[DPL];
                load_row_f32<D>(Ks + (size_t)(kb0 + grp * C::KPG + kk) * D + lane * DPL, kf);
#pragma unroll
                for (int rr = 0; rr < RPW; ++rr) {
                    float a = 0.f;
#pragma unroll
                    for (int d = 0; d < DPL; ++d) a = fmaf(qf[rr][d], kf[d], a);
                    v[kk * RPW + rr] = a;
                }
            }
            const float red = warp_reduce_scatter32(v);
            const int j = j0 + kb0 + grp * C::KPG + lane / RPW;
            sc[grp] = (j >= jlo_own && j <= jhi_own) ? red : NEG_INF;
        }

        // online softmax for the row this lane holds
        float tmax = sc[0];
#pragma unroll
        for (int grp = 1; grp < C::NG; ++grp) tmax = fmaxf(tmax, sc[grp]);
#pragma unroll
        for (int off = RPW; off < 32; off <<= 1)
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        const float m_new = fmaxf(m_own, tmax);
        const float m_use = m_new == NEG_INF ? 0.f : m_new;
        const float alpha = fast_exp2(m_own - m_use);
        float psum = 0.f;
#pragma unroll
        for (int grp = 0; grp < C::NG; ++grp) {
            const float pv = fast_exp2(sc[grp] - m_use);
            psum += pv;
            pbuf[grp * 32 + lane] = pv;  // = pbuf[key_in_block * RPW + row]
        }
#pragma unroll
        for (int off = RPW; off < 32; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l_own = l_own * alpha + psum;
        m_own = m_new;
        __syncwarp();

        // rescale and accumulate P V
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const float a = __shfl_sync(0xffffffffu, alpha, rr);
#pragma unroll
            for (int d = 0; d < DPL; ++d) acc[rr][d] *= a;
        }
        const int kmax = min(C::KB, n - kb0);  // keys past the tile's end hold stale data
        for (int kk = 0; kk < kmax; ++kk) {
            float vf[DPL];
            load_row_f32<D>(Vs + (size_t)(kb0 + kk) * D + lane * DPL, vf);
            float pr[RPW];
            if constexpr (RPW == 4) {
                const float4 p4 = *reinterpret_cast<const float4 *>(pbuf + kk * 4);
                pr[0] = p4.x; pr[1] = p4.y; pr[2] = p4.z; pr[3] = p4.w;
            } else {
                const float4 a4 = *reinterpret_cast<const float4 *>(pbuf + kk * 8);
                const float4 b4 = *reinterpret_cast<const float4 *>(pbuf + kk * 8 + 4);
                pr[0] = a4.x; pr[1] = a4.y; pr[2] = a4.z; pr[3] = a4.w;
                pr[4] = b4.x; pr[5] = b4.y; pr[6] = b4.z; pr[7] = b4.w;
            }
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
                for (int d = 0; d < DPL; ++d) acc[rr][d] = fmaf(pr[rr], vf[d], acc[rr][d]);
        }
        __syncthreads();  // stage s and pbuf free for reuse
    }
    if (!ok) return;  // a copy never landed; the fault word is set

    // ---- combine the key groups of each row group, then write out
    float *comb_acc = reinterpret_cast<float *>(ring);
    float *comb_ml = comb_acc + C::NKG * C::RPT * D;
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        float *dst = comb_acc + ((size_t)kg * C::RPT + rg * RPW + rr) * D + lane * DPL;
#pragma unroll
        for (int d = 0; d < DPL; ++d) dst[d] = acc[rr][d];
    }
    if (lane < RPW) {
        float *ml = comb_ml + ((size_t)kg * C::RPT + rg * RPW + lane) * 2;
        ml[0] = m_own;
        ml[1] = l_own;
    }
    __syncthreads();

    constexpr int CPR = D / 8;  // 8-dim chunks per row
    for (int idx = tid; idx < C::RPT * CPR; idx += kSimtThreads) {
        const int rloc = idx / CPR, dc = idx % CPR;
        const int r = rt * C::RPT + rloc;
        if (r >= P.R) continue;
        float M = NEG_INF;
#pragma unroll
        for (int q = 0; q < C::NKG; ++q) M = fmaxf(M, comb_ml[((size_t)q * C::RPT + rloc) * 2]);
        float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float Lam = 0.f;
        if (M != NEG_INF) {
#pragma unroll
            for (int q = 0; q < C::NKG; ++q) {
                const float mq = comb_ml[((size_t)q * C::RPT + rloc) * 2];
                const float w = fast_exp2(mq - M);
                Lam += w * comb_ml[((size_t)q * C::RPT + rloc) * 2 + 1];
                const float *a = comb_acc + ((size_t)q * C::RPT + rloc) * D + dc * 8;
#pragma unroll
                for (int d = 0; d < 8; ++d) o[d] = fmaf(w, a[d], o[d]);
            }
        }
        const int i = r / P.G, gg = r - (r / P.G) * P.G;
        const size_t orow = ((size_t)b * P.q_len + i) * P.Hq + (size_t)h * P.G + gg;
        if (P.splits == 1) {
            const float inv = Lam > 0.f ? 1.f / Lam : 0.f;
            uint4 w;
            w.x = pack_bf16x2(o[0] * inv, o[1] * inv);
            w.y = pack_bf16x2(o[2] * inv, o[3] * inv);
            w.z = pack_bf16x2(o[4] * inv, o[5] * inv);
            w.w = pack_bf16x2(o[6] * inv, o[7] * inv);
            *reinterpret_cast<uint4 *>(P.out + orow * D + dc * 8) = w;
            if (dc == 0 && P.lse != nullptr)
                P.lse[orow] = Lam > 0.f ? (M + __log2f(Lam)) * kLn2 : NEG_INF;
        } else {
            const size_t prow = (((size_t)b * P.Hkv + h) * P.splits + split) * P.R + r;
            float4 *dst = reinterpret_cast<float4 *>(P.part_acc + prow * D + dc * 8);
            dst[0] = make_float4(o[0], o[1], o[2], o[3]);
            dst[1] = make_float4(o[4], o[5], o[6], o[7]);
            if (dc == 0) {
                P.part_ml[prow * 2] = M;
                P.part_ml[prow * 2 + 1] = Lam;
            }
        }
    }
}

// Log-sum-exp merge of the split partials of every packed row:
//   M = max_s m_s, Lambda = sum_s l_s 2^(m_s - M),
//   out = sum_s acc_s 2^(m_s - M) / Lambda, lse = (M + log2 Lambda) ln 2.
// One block per packed row (sequence, KV head, row).  The block first turns
// the splits' (m, l) into weights in shared memory; then each thread sums a
// residue class of splits for one 8-dim chunk, so all of a row's partial
// loads are in flight at once, and the classes are added up in shared
// memory.
constexpr int kMergeThreads = 256;
constexpr int kMergeMaxSplits = 64;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) swa_merge_kernel(const AttnParams P) {
    const float NEG_INF = -__int_as_float(0x7f800000);
    constexpr int CPR = D / 8;                    // 8-dim chunks per row
    constexpr int NG = kMergeThreads / CPR;       // split classes
    __shared__ float w_s[kMergeMaxSplits];        // 2^(m_s - M), 0 for empty splits
    __shared__ float red[2];                      // M, Lambda
    __shared__ __align__(16) float part[NG][D];   // per-class sums
    grid_dep_wait();
    grid_dep_trigger();
    const long long grow = blockIdx.x;            // (b*Hkv + h) * R + r
    const long long bh = grow / P.R;
    const int r = (int)(grow % P.R);
    const int b = (int)(bh / P.Hkv), h = (int)(bh % P.Hkv);
    const size_t base = (size_t)bh * P.splits * P.R + r;  // split s at base + s*R
    const int tid = threadIdx.x;
    if (tid < 32) {
        // warp 0: M and the weights (splits <= 64, two per lane)
        float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
        if (tid < P.splits) {
            m0 = P.part_ml[(base + (size_t)tid * P.R) * 2];
            l0 = P.part_ml[(base + (size_t)tid * P.R) * 2 + 1];
        }
        if (tid + 32 < P.splits) {
            m1 = P.part_ml[(base + (size_t)(tid + 32) * P.R) * 2];
            l1 = P.part_ml[(base + (size_t)(tid + 32) * P.R) * 2 + 1];
        }
        float M = fmaxf(m0, m1);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float w0 = (M == NEG_INF || m0 == NEG_INF) ? 0.f : fast_exp2(m0 - M);
        const float w1 = (M == NEG_INF || m1 == NEG_INF) ? 0.f : fast_exp2(m1 - M);
        float lam = w0 * l0 + w1 * l1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lam += __shfl_xor_sync(0xffffffffu, lam, off);
        w_s[tid] = w0;
        w_s[tid + 32] = w1;
        if (tid == 0) {
            red[0] = M;
            red[1] = lam;
        }
    }
    __syncthreads();
    const int c = tid % CPR, sg = tid / CPR;
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int sp = sg; sp < P.splits; sp += NG) {
        const float w = w_s[sp];
        const float4 *a = reinterpret_cast<const float4 *>(P.part_acc + (base + (size_t)sp * P.R) * D + c * 8);
        const float4 a0 = a[0], a1 = a[1];
        o[0] = fmaf(w, a0.x, o[0]); o[1] = fmaf(w, a0.y, o[1]);
        o[2] = fmaf(w, a0.z, o[2]); o[3] = fmaf(w, a0.w, o[3]);
        o[4] = fmaf(w, a1.x, o[4]); o[5] = fmaf(w, a1.y, o[5]);
        o[6] = fmaf(w, a1.z, o[6]); o[7] = fmaf(w, a1.w, o[7]);
    }
    *reinterpret_cast<float4 *>(&part[sg][c * 8]) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4 *>(&part[sg][c * 8 + 4]) = make_float4(o[4], o[5], o[6], o[7]);
    __syncthreads();
    if (tid < CPR) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int g2 = 0; g2 < NG; ++g2) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += part[g2][tid * 8 + e];
        }
        const float Lam = red[1];
        const float inv = Lam > 0.f ? 1.f / Lam : 0.f;
        const int i = r / P.G, gg = r % P.G;
        const size_t orow = ((size_t)b * P.q_len + i) * P.Hq + (size_t)h * P.G + gg;
        uint4 wv;
        wv.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        wv.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        wv.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        wv.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4 *>(P.out + orow * D + tid * 8) = wv;
        if (tid == 0 && P.lse != nullptr)
            P.lse[orow] = Lam > 0.f ? (red[0] + __log2f(Lam)) * kLn2 : NEG_INF;
    }
}

}  // namespace swa
