// C-ABI of the sliding-window split-KV verify-attention library: argument
// validation, the split heuristic, workspace management and kernel launch.
// Every entry point is declared (with its contract) in include/swa.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/swa.h"
#include "swa_simt.cuh"
#include "swa_accept.cuh"
#include "swa_tc_host.h"

// Fault word of each device that loads the library; kernels receive its
// address and OR bits into it when a bounded wait gives up.  The word after
// it counts out-of-range index attempts in a library built with
// SWA_DEBUG_CHECKS.
__device__ uint32_t g_fault_word[2] = {0, 0};

namespace {

constexpr int kMaxSplits = 64;
constexpr int kTcKeysPerTile = 128;  // keys per tensor-core tile (MMA M)
static_assert(kMaxSplits <= swa::kMergeMaxSplits, "the merge kernel weighs at most 64 splits");
constexpr int kMaxQLen = 64;      // SPLITKV_VERIFY_MAX_Q: draft rows of a greedy verification
constexpr int kMaxBlockLen = 512; // MAX_NUM_BATCHED_TOKENS: rows of an attention call
                                  // (verify blocks up to 64, prefill chunks up to 512)
constexpr int kMaxDevices = 64;

thread_local char t_last_error[512] = "";

swa_status fail(swa_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return st;
}

swa_status cuda_fail(cudaError_t e, const char *what) {
    return fail(SWA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

swa_status validate_dims(const swa_dims *d, int32_t window) {
    if (d == nullptr) return fail(SWA_ERR_INVALID_ARG, "dims is NULL");
    if (d->batch < 1 || d->batch > 65535)
        return fail(SWA_ERR_INVALID_ARG, "batch %d outside [1, 65535]", d->batch);
    if (d->q_len < 1 || d->q_len > kMaxBlockLen)
        return fail(SWA_ERR_INVALID_ARG, "q_len %d outside [1, %d]", d->q_len, kMaxBlockLen);
    if (d->num_q_heads < 1 || d->num_kv_heads < 1)
        return fail(SWA_ERR_INVALID_ARG, "head counts must be >= 1 (Hq %d, Hkv %d)",
                    d->num_q_heads, d->num_kv_heads);
    if (d->num_q_heads % d->num_kv_heads != 0)
        return fail(SWA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                    d->num_q_heads, d->num_kv_heads);
    if (d->num_kv_heads > 65535)
        return fail(SWA_ERR_INVALID_ARG, "num_kv_heads %d too large", d->num_kv_heads);
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
        return fail(SWA_ERR_UNSUPPORTED, "head_dim %d not in {64, 128, 256}", d->head_dim);
    if (d->max_len < 1) return fail(SWA_ERR_INVALID_ARG, "max_len %d < 1", d->max_len);
    if (window < 1) return fail(SWA_ERR_INVALID_ARG, "window %d < 1", window);
    if (d->num_splits < 0) return fail(SWA_ERR_INVALID_ARG, "num_splits %d < 0", d->num_splits);
    const long long R = (long long)d->q_len * (d->num_q_heads / d->num_kv_heads);
    if (R > 4096) return fail(SWA_ERR_UNSUPPORTED, "q_len * G = %lld rows per KV head > 4096", R);
    // cache and query element counts must fit the kernels' size_t arithmetic
    // and the grid: Hkv * row_tiles <= 65535
    const long long row_tiles = (R + 31) / 32;
    if ((long long)d->num_kv_heads * row_tiles > 65535)
        return fail(SWA_ERR_UNSUPPORTED, "num_kv_heads * row tiles exceeds the grid limit");
    return SWA_OK;
}

struct Plan {
    int kernel;       // 1 = CUDA-core (SIMT) chunk kernel, 2 = key-major tensor-core kernel,
                      // 3 = rows-major tensor-core kernel, 4 = its CTA-pair form
    int rpw, nrg;     // SIMT row layout
    int rows_per_tile, row_tiles;
    int q_rows_per_tile;  // tensor-core path: draft rows per item
    int tc_n;             // tensor-core path: padded rows per item (MMA N)
    int splits, chunk;
    long long workspace;
    long long grid;   // CTAs of the attention kernel
    long long items;  // tensor-core path: work items
    int sms;          // SMs of the device the plan is for
};

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Test and sweep controls (swa_set_debug_options); relaxed atomics, read on
// every call.
std::atomic<int> g_opt_force{0};
std::atomic<int> g_opt_pdl{1};
std::atomic<long long> g_opt_wait_limit{0};
std::atomic<int> g_opt_withhold{-1};
std::atomic<int> g_opt_rows{0};
std::atomic<int> g_opt_fail_launch{0};

// Kernel override of a test or sweep: 0 none, 1 CUDA-core, 2 key-major, 3 rows-major,
// 4 rows-major on CTA pairs.
int forced_kernel() { return g_opt_force.load(std::memory_order_relaxed); }

// Split heuristic.  Host-only: seq_lens live on the device, so the
// worst-case span W + q_len - 1 (bounded by the cache length) is used; a
// work item reads only the windows of its own draft rows, W + rows - 1 keys
// (the kernels narrow each item's chunk), and that decides the splits.
//  - Rows-major tensor-core kernel for more than 32 packed rows, up to 128
//    rows per item; same chunking as below.
//  - Tensor-core path (head_dim 128/256; >= 16 packed rows, or a batch whose
//    (sequence, KV head) units cover half the SMs): one chunk per (sequence,
//    KV head, row tile) once those units cover half the SMs or the span is at
//    most three 128-key tiles; otherwise enough chunks of >= 128 keys to reach
//    every SM.  Persistent grid of at most SMs x resident CTAs.
//  - CUDA-core path: enough CTAs to cover every SM about twice, chunks of at
//    least one 32-key tile.
// Chunks are multiples of 16 keys; at most kMaxSplits chunks.
Plan make_plan_with(const swa_dims *d, int32_t window, int num_sms, int force, bool pairs_ok) {
    Plan p{};
    p.sms = num_sms;
    const int G = d->num_q_heads / d->num_kv_heads;
    const int R = d->q_len * G;
    const int D = d->head_dim;
    if (num_sms < 1) num_sms = 148;
    long long span = (long long)window + d->q_len - 1;
    if (span > d->max_len) span = d->max_len;
    if (span < 1) span = 1;

    const bool tc_shape = (D == 128 || D == 256) && G <= 64 &&
                          (long long)d->batch * d->num_kv_heads * d->max_len < (1LL << 31) &&
                          (long long)d->batch * d->q_len < (1LL << 31) &&
                          (long long)d->batch * d->num_kv_heads * d->q_len * kMaxSplits <
                              (1LL << 31);
    // The tensor-core kernel needs >= 16 packed rows to fill an MMA without
    // waste, but below that it still wins once the (sequence, KV head) units
    // alone cover half the SMs: its MMAs cost the same for 4 rows as for 16,
    // and its K/V stream is the faster one.
    const bool big_batch = (long long)d->batch * d->num_kv_heads * 2 >= num_sms;
    const bool use_tc = tc_shape && (force == 2 || (force == 0 && (R >= 16 || big_batch)));
    int splits;
    // More than 32 packed rows (q_len > 8 at 4:1 GQA) go to the rows-major
    // kernel: its softmax keeps a row in one thread pair and P in TMEM, and
    // an item holds up to 128 rows, so K/V are re-read less often; up to 32
    // rows the key-major kernel's eight warps share the work better.
    const bool use_rows = tc_shape && (force == 3 || force == 4 || (force == 0 && R > 32));
    // More than 128 packed rows (two or more row tiles of a (sequence, KV
    // head)) at head_dim 256 over a contiguous cache: the rows-major kernel on
    // CTA pairs, 2 x 128 rows per item, each K/V byte read once per item.
    const bool use_pairs = use_rows && pairs_ok && D == 256 && (force == 4 || (force == 0 && R > 128));
    if (use_pairs) {
        p.kernel = 4;
        const int cta_rows = (128 / G) * G;
        p.rows_per_tile = 2 * cta_rows;
        p.q_rows_per_tile = 2 * (128 / G);
        p.row_tiles = ceil_div(d->q_len, p.q_rows_per_tile);
        p.tc_n = 128;
    } else if (use_rows) {
        // rows-major kernel: up to 128 packed rows per item (the MMA's M)
        p.kernel = 3;
        const int max_rows = 128;
        p.rows_per_tile = R <= max_rows ? R : (max_rows / G) * G;
        p.q_rows_per_tile = p.rows_per_tile / G;
        p.row_tiles = ceil_div(d->q_len, p.q_rows_per_tile);
        p.tc_n = p.rows_per_tile <= 32 ? 32 : p.rows_per_tile <= 64 ? 64 : 128;
    } else if (use_tc) {
        p.kernel = 2;
        // rows per item: at most 64 (shared memory holds Q and P tiles beside
        // the ring; the softmax keeps a row's reference maximum in registers);
        // fewer when SMs would stay idle (below, once the key split is known)
        const int max_rows = 64;
        p.rows_per_tile = R <= max_rows ? R : (max_rows / G) * G;
        p.q_rows_per_tile = p.rows_per_tile / G;
        p.row_tiles = ceil_div(d->q_len, p.q_rows_per_tile);
        p.tc_n = p.rows_per_tile <= 16 ? 16 : p.rows_per_tile <= 32 ? 32 : 64;
    }
    if (use_rows || use_tc) {
        const int ctas_per_sm = 1;  // the tensor-core kernels: one persistent CTA per SM
        const int unit_ctas = use_pairs ? 2 : 1;  // CTAs that work on one item at once
        const long long units = (long long)d->batch * d->num_kv_heads * p.row_tiles * unit_ctas;
        long long item_span = (long long)window + p.q_rows_per_tile - 1;
        if (item_span > span) item_span = span;
        long long chunk;
        if (d->num_splits > 0) {
            splits = d->num_splits;
            chunk = (span + splits - 1) / splits;
        } else {
            int per_item;  // chunks across one item's keys
            if (units * 2 >= num_sms || item_span <= 3 * kTcKeysPerTile) {
                // a split costs a partial round trip, a dependent merge launch
                // and the merge (~2.5 us measured on GB300), which a span of up
                // to three 128-key tiles (~1.2 us each) does not win back
                per_item = 1;
            } else {
                const long long s = (num_sms + units - 1) / units;
                const long long by_len = (item_span + kTcKeysPerTile - 1) / kTcKeysPerTile;
                per_item = (int)(s < by_len ? s : by_len);
            }
            chunk = (item_span + per_item - 1) / per_item;
            if (per_item == 1) chunk = span;  // one chunk: the whole span
            chunk = (chunk + 15) / 16 * 16;
            if ((span + chunk - 1) / chunk > kMaxSplits) chunk = (span + kMaxSplits - 1) / kMaxSplits;
            splits = ceil_div(span, chunk);
        }
        if (splits < 1) splits = 1;
        if (splits > kMaxSplits) {
            splits = kMaxSplits;
            chunk = (span + splits - 1) / splits;
        }
        if (chunk < 1) chunk = 1;
        splits = ceil_div(span, chunk);
        p.splits = splits;
        p.chunk = (int)chunk;
        if (use_tc && !use_rows && d->num_splits == 0) {
            // Key-major kernel, key split fixed: cut the rows into smaller
            // items while many SMs would stay idle, so more SMs share each
            // tile's softmax (the row tiles' extra K/V reads come from L2): 8
            // rows while the 8-row items fill at most a sixteenth of the SMs,
            // else 16 while the 16-row items fill at most ~60% of them.
            // Measured on GB300 (q8, 4:1 GQA, us, rows 8 / 16 / 32): W188 one
            // sequence 7.21 / 7.38 / 8.66, 2 sequences 7.50 / 7.33 / 8.66, 8:
            // 7.90 / 7.70 / 8.87, 16: 9.77 / 8.07 / 8.95, 24: 13.99 / 10.01 /
            // 9.21, 32: 14.78 / 10.34 / 9.62; W512 4 sequences 13.07 / 9.71 /
            // 10.33; W1024 one sequence 9.40 / 9.14 / 9.87, 4: 14.48 / 11.29 /
            // 10.66; W4096 one sequence 15.5 / 10.48 / 10.34.
            const long long per_unit = (long long)d->batch * d->num_kv_heads * splits;
            for (int r : {8, 16}) {
                const int rows = r < G ? G : (r / G) * G;
                if (rows >= p.rows_per_tile) break;
                const long long rt = ceil_div(d->q_len, rows / G);
                const long long n = per_unit * rt;
                if (r == 8 ? n * 16 <= num_sms : n * 5 <= 3LL * num_sms) {
                    p.rows_per_tile = rows;
                    p.q_rows_per_tile = rows / G;
                    p.row_tiles = (int)rt;
                    p.tc_n = 16 * ((rows + 15) / 16);
                    break;
                }
            }
        }
        const int force_rows = g_opt_rows.load(std::memory_order_relaxed);
        if (force_rows > 0 && d->num_splits == 0 && !use_pairs) {
            // a sweep's override of the rows per item
            const int max_rows = use_rows ? 128 : 64;
            int rows = force_rows < max_rows ? force_rows : max_rows;
            rows = rows < R ? rows : R;
            rows = rows < G ? G : (rows / G) * G;
            if (rows <= max_rows) {
                p.rows_per_tile = rows;
                p.q_rows_per_tile = rows / G;
                p.row_tiles = ceil_div(d->q_len, p.q_rows_per_tile);
                p.tc_n = use_rows ? (rows <= 32 ? 32 : rows <= 64 ? 64 : 128)
                                  : 16 * ((rows + 15) / 16);
            }
        }
        p.items = (long long)splits * d->batch * d->num_kv_heads * p.row_tiles;
        long long slots = (long long)num_sms * ctas_per_sm / unit_ctas;
        if (slots < 1) slots = 1;
        p.grid = (p.items < slots ? p.items : slots) * unit_ctas;
    } else {
        p.kernel = 1;
        if (R <= 4) { p.rpw = 4; p.nrg = 1; }
        else if (R <= 8) { p.rpw = 8; p.nrg = 1; }
        else if (R <= 16) { p.rpw = 8; p.nrg = 2; }
        else { p.rpw = 8; p.nrg = 4; }
        p.rows_per_tile = p.rpw * p.nrg;
        p.row_tiles = ceil_div(R, p.rows_per_tile);
        const long long units = (long long)d->batch * d->num_kv_heads * p.row_tiles;
        // keys one CTA reads: the windows of its draft rows
        long long item_span = (long long)window + (p.rows_per_tile + G - 1) / G;
        if (item_span > span) item_span = span;
        long long chunk;
        if (d->num_splits > 0) {
            splits = d->num_splits;
            if (splits > kMaxSplits) splits = kMaxSplits;
            chunk = (span + splits - 1) / splits;
        } else {
            const long long target = 2LL * num_sms;
            long long s = (target + units - 1) / units;
            const long long by_len = (item_span + swa::kSimtTileKeys - 1) / swa::kSimtTileKeys;
            if (s > by_len) s = by_len;
            if (s < 1) s = 1;
            chunk = (item_span + s - 1) / s;
            chunk = (chunk + 15) / 16 * 16;
            if ((span + chunk - 1) / chunk > kMaxSplits) chunk = (span + kMaxSplits - 1) / kMaxSplits;
        }
        if (chunk < 1) chunk = 1;
        splits = ceil_div(span, chunk);
        p.splits = splits;
        p.chunk = (int)chunk;
        p.grid = (long long)splits * d->num_kv_heads * p.row_tiles * d->batch;
        p.items = p.grid;
    }
    p.workspace = p.splits > 1 ? (long long)d->batch * d->num_kv_heads * p.splits * R *
                                     ((long long)D + 2) * 4
                               : 0;
    return p;
}

// The plan of a call.  More than 32 packed rows go to the rows-major kernel
// unless the key-major kernel's items (up to 64 rows each) fit in one wave of
// its persistent CTAs, one item per SM, or it cuts its rows into 8- or
// 16-row items: then the key-major plan is taken.  Measured on GB300, W188,
// us, rows-major / key-major: q16 one sequence 11.5 / 7.3, 8 sequences 12.1 /
// 8.0, 16: 12.4 / 11.9, 64: 14.9 / 13.7, 128 (256 key-major items): 23.0 /
// 22.8; q32 8 sequences 13.3 / 12.0, 32: 14.7 / 14.0, 64 (256 items): 17.4 /
// 23.4; q64 4 sequences 13.3 / 11.8, 16: 14.4 / 13.8, 32 (256 items): 16.6 /
// 22.7; a 512-token prefill chunk of one sequence 13.6 / 12.1.
//
// Against the CTA-pair kernel (above 128 rows) the key-major plan wins only
// when it cuts the rows into 8- or 16-row items.  Measured on GB300, W188,
// us, key-major / pairs: q64 one sequence 7.6 / 11.0 (16-row items), 4
// sequences 11.5 / 11.2, 8: 11.7 / 11.3, 16: 12.9 / 11.5; a 512-token
// prefill chunk, one sequence 11.7 / 11.3, two 12.9 / 11.5.
Plan make_plan(const swa_dims *d, int32_t window, int num_sms, bool pairs_ok) {
    const int force = forced_kernel();
    Plan p = make_plan_with(d, window, num_sms, force, pairs_ok);
    if (force == 0 && p.kernel >= 3) {
        const Plan k = make_plan_with(d, window, num_sms, 2, pairs_ok);
        const bool small_items = k.rows_per_tile <= 16;
        const bool one_wave = k.items <= (long long)num_sms;
        if (k.kernel == 2 && (small_items || (p.kernel == 3 && one_wave))) return k;
    }
    return p;
}

// ------------------------------------------------------------- workspace

struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
    bool owned = false;
};
std::mutex g_ws_mutex;
Workspace g_ws[kMaxDevices];

swa_status ensure_workspace(int dev, size_t need, cudaStream_t stream, void **out) {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace &w = g_ws[dev];
    if (w.bytes >= need) {
        *out = w.ptr;
        return SWA_OK;
    }
    if (!w.owned && w.ptr != nullptr)
        return fail(SWA_ERR_WORKSPACE, "workspace set by the caller holds %zu bytes, %zu needed",
                    w.bytes, need);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cap != cudaStreamCaptureStatusNone)
        return fail(SWA_ERR_WORKSPACE,
                    "stream is capturing and the workspace (%zu bytes) is below the %zu needed; "
                    "run one call outside capture first or set a workspace",
                    w.bytes, need);
    if (w.ptr) {
        e = cudaFree(w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
        if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
    }
    size_t grow = need + need / 4;
    e = cudaMalloc(&w.ptr, grow);
    if (e != cudaSuccess) {
        w.ptr = nullptr;
        return cuda_fail(e, "cudaMalloc(workspace)");
    }
    w.bytes = grow;
    w.owned = true;
    *out = w.ptr;
    return SWA_OK;
}

template <int D, int RPW, int NRG, bool AP>
cudaError_t launch_simt_ap(const swa::AttnParams &P, cudaStream_t stream) {
    using C = swa::SimtCfg<D, RPW, NRG>;
    auto kern = swa::swa_simt_kernel<D, RPW, NRG, AP>;
    static std::atomic<bool> attr_done[kMaxDevices];
    cudaError_t e = swa::raise_smem_limit(kern, C::SMEM_BYTES, attr_done);
    if (e != cudaSuccess) return e;
    dim3 grid(P.splits, P.Hkv * P.row_tiles, P.B);
    return swa::launch_kernel(kern, grid, dim3(swa::kSimtThreads), C::SMEM_BYTES, stream, P);
}

// The plain kernel, or (fused append) its variant.
template <int D, int RPW, int NRG>
cudaError_t launch_simt(const swa::AttnParams &P, cudaStream_t stream) {
    return P.k_new != nullptr ? launch_simt_ap<D, RPW, NRG, true>(P, stream)
                              : launch_simt_ap<D, RPW, NRG, false>(P, stream);
}

template <int D>
cudaError_t launch_simt_d(const Plan &pl, const swa::AttnParams &P, cudaStream_t s) {
    if (pl.rpw == 4) return launch_simt<D, 4, 1>(P, s);
    if (pl.nrg == 1) return launch_simt<D, 8, 1>(P, s);
    if (pl.nrg == 2) return launch_simt<D, 8, 2>(P, s);
    return launch_simt<D, 8, 4>(P, s);
}

template <int D>
cudaError_t launch_merge(const swa::AttnParams &P, cudaStream_t s) {
    const long long blocks = (long long)P.B * P.Hkv * P.R;  // one per packed row
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return swa::launch_kernel(swa::swa_merge_kernel<D>, dim3((unsigned)blocks),
                              dim3(swa::kMergeThreads), 0, s, P);
}

// Launches the attention kernel of `pl` (and the merge kernel when the
// plan splits the keys).  P carries every pointer, including the partials.
swa_status launch_plan(const Plan &pl, const swa_dims *dims, const swa::AttnParams &P,
                       const void *q, const void *k_cache, const void *v_cache, cudaStream_t s,
                       long long cache_rows = -1) {
    cudaError_t e;
    if (pl.kernel >= 2) {
        swa::TcLaunch L{};
        L.T.a = P;
        L.T.rows_per_tile = pl.rows_per_tile;
        L.T.q_rows_per_tile = pl.q_rows_per_tile;
        L.T.items = (int)pl.items;
        // contiguous blocks of items per CTA for the key-major kernel (measured
        // on GB300, stress W188: q8 50.6 -> 48.8 us, q1 41.1 -> 40.0 us); the
        // rows-major kernel deals them round-robin (blocks: W188 q64 127.2 ->
        // 128.6 us, W1024 q64 405.5 -> 440.5 us)
        L.T.items_per_cta = pl.kernel == 2 ? (int)(pl.items / pl.grid) : 0;
        L.T.items_extra = pl.kernel == 2 ? (int)(pl.items % pl.grid) : 0;
        // measured on GB300: single_stream (8 CTAs) 7.86 -> 7.33 us with every
        // first fill issued at once; batched (128 CTAs) 11.6 -> 10.9 us with the
        // first K tile alone ahead (11.4 us with all)
        L.T.early_max = pl.grid * 2 >= pl.sms ? 1 : 8;
        L.D = dims->head_dim;
        L.N = pl.tc_n;
        L.rows_major = pl.kernel >= 3;
        L.pairs = pl.kernel == 4;
        if (L.pairs) {
            // the kernel takes one CTA's share of an item's rows
            L.T.rows_per_tile = pl.rows_per_tile / 2;
            L.T.q_rows_per_tile = pl.q_rows_per_tile / 2;
        }
        L.grid = (int)pl.grid;
        L.cache_rows = cache_rows >= 0 ? cache_rows : (long long)P.B * P.Hkv * P.L;
        L.q = q;
        L.k = k_cache;
        L.v = v_cache;
        char msg[256] = "";
        e = swa::tc_launch(L, s, msg, sizeof msg);
        if (e != cudaSuccess)
            return msg[0] ? fail(SWA_ERR_CUDA, "%s", msg)
                          : cuda_fail(e, "tensor-core kernel launch");
    } else {
        switch (dims->head_dim) {
            case 64: e = launch_simt_d<64>(pl, P, s); break;
            case 128: e = launch_simt_d<128>(pl, P, s); break;
            default: e = launch_simt_d<256>(pl, P, s); break;
        }
        if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
    }
    if (pl.splits > 1) {
        switch (dims->head_dim) {
            case 64: e = launch_merge<64>(P, s); break;
            case 128: e = launch_merge<128>(P, s); break;
            default: e = launch_merge<256>(P, s); break;
        }
        if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
    }
    return SWA_OK;
}

// Per-device caches, filled on first use by whichever host thread gets
// there (a race between threads only resolves the same value twice).
std::atomic<uint32_t *> g_fault_ptr[kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];

uint32_t *fault_word_ptr(int dev) {
    uint32_t *p = g_fault_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_fault_word) != cudaSuccess) return nullptr;
        p = static_cast<uint32_t *>(a);
        g_fault_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

int device_sms(int dev) {
    int n = g_sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
        g_sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Host checks of a paged cache description against dims.
swa_status check_paged(const swa_paged *paged, const swa_dims *dims) {
    if (paged == nullptr || paged->block_table == nullptr)
        return fail(SWA_ERR_INVALID_ARG, "paged cache description or its block table is NULL");
    if (reinterpret_cast<uintptr_t>(paged->block_table) & 3u)
        return fail(SWA_ERR_INVALID_ARG, "block_table must be 4-byte aligned");
    if (paged->page_size < 8 || paged->page_size % 8 != 0)
        return fail(SWA_ERR_INVALID_ARG, "page_size %d is not a positive multiple of 8",
                    paged->page_size);
    if (paged->max_blocks < 1 || paged->num_pages < 1)
        return fail(SWA_ERR_INVALID_ARG, "max_blocks %d and num_pages %d must be >= 1",
                    paged->max_blocks, paged->num_pages);
    if (dims != nullptr && (long long)dims->max_len != (long long)paged->max_blocks * paged->page_size)
        return fail(SWA_ERR_INVALID_ARG, "dims->max_len %d != max_blocks * page_size = %lld",
                    dims->max_len, (long long)paged->max_blocks * paged->page_size);
    if (dims != nullptr &&
        (long long)paged->num_pages * dims->num_kv_heads * paged->page_size >= (1LL << 31))
        return fail(SWA_ERR_UNSUPPORTED, "the page pool holds 2^31 or more rows");
    return SWA_OK;
}

}  // namespace

// ------------------------------------------------- allocation-free scratch
//
// Split partials of swa_verify_attn_noalloc live in this fixed array instead
// of a cudaMalloc'd workspace.  In host code `g_noalloc_scratch` only names
// the symbol; its device address comes from cudaGetSymbolAddress, resolved
// once per device with that device current.

static __device__ __align__(256) unsigned char g_noalloc_scratch[SWA_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on device `dev` (which must be the
// current device), resolved once per device.
swa_status noalloc_scratch(int dev, void **ptr) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return SWA_OK;
}

// The windowed verify attention of swa_verify_attn, on a contiguous cache
// (paged == NULL) or a paged one; with k_new / v_new non-NULL the kernels
// first write the new rows into the cache (swa_append_verify_attn).  With
// `noalloc` the split partials go to the fixed scratch array above
// (swa_verify_attn_noalloc) and nothing is ever allocated.
swa_status verify_impl(const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *seq_lens, const int32_t *q_pos, int32_t window, float scale,
                       void *out, float *lse, const swa_dims *dims, swa_stream_t stream,
                       const swa_paged *paged, const void *k_new = nullptr,
                       const void *v_new = nullptr, bool noalloc = false) {
    swa_status st = validate_dims(dims, window);
    if (st != SWA_OK) return st;
    if (!q || !k_cache || !v_cache || !seq_lens || !q_pos || !out)
        return fail(SWA_ERR_INVALID_ARG, "a required pointer is NULL");
    if ((k_new == nullptr) != (v_new == nullptr))
        return fail(SWA_ERR_INVALID_ARG, "k_new and v_new must both be given");
    if ((k_new && !aligned16(k_new)) || (v_new && !aligned16(v_new)))
        return fail(SWA_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return fail(SWA_ERR_INVALID_ARG, "q, the K and V caches and out must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(seq_lens) & 3u) || (reinterpret_cast<uintptr_t>(q_pos) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(SWA_ERR_INVALID_ARG, "seq_lens, q_pos and lse must be 4-byte aligned");
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
        return fail(SWA_ERR_INVALID_ARG, "scale must be finite");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev >= kMaxDevices) return fail(SWA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);

    uint32_t *fault = fault_word_ptr(dev);
    if (fault == nullptr) return fail(SWA_ERR_CUDA, "cannot resolve the device fault word");
    // the CTA-pair kernel reads a contiguous cache without a fused append
    const Plan pl = make_plan(dims, window, device_sms(dev), paged == nullptr && k_new == nullptr);
    swa::AttnParams P{};
    P.q = static_cast<const __nv_bfloat16 *>(q);
    P.k = static_cast<const __nv_bfloat16 *>(k_cache);
    P.v = static_cast<const __nv_bfloat16 *>(v_cache);
    P.seq_lens = seq_lens;
    P.q_pos = q_pos;
    P.out = static_cast<__nv_bfloat16 *>(out);
    P.lse = lse;
    P.B = dims->batch;
    P.q_len = dims->q_len;
    P.Hq = dims->num_q_heads;
    P.Hkv = dims->num_kv_heads;
    P.G = dims->num_q_heads / dims->num_kv_heads;
    P.L = dims->max_len;
    P.window = window;
    P.R = P.q_len * P.G;
    P.splits = pl.splits;
    P.chunk = pl.chunk;
    P.row_tiles = pl.row_tiles;
    P.rows_per_tile = pl.rows_per_tile;
    P.qk_scale = scale * swa::kLog2e;
    P.fault = fault;
    P.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    P.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    const long long wl = g_opt_wait_limit.load(std::memory_order_relaxed);
    P.wait_limit = wl > 0 ? wl : swa::kWaitLimitCycles;
    P.withhold_fill = g_opt_withhold.load(std::memory_order_relaxed);
    long long cache_rows = (long long)P.B * P.Hkv * P.L;
    if (paged != nullptr) {
        P.block_table = paged->block_table;
        P.page_size = paged->page_size;
        P.max_blocks = paged->max_blocks;
        P.num_pages = paged->num_pages;
        cache_rows = (long long)paged->num_pages * P.Hkv * paged->page_size;
    }

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pl.splits > 1) {
        void *ws = nullptr;
        if (noalloc) {
            if (pl.workspace > (long long)SWA_NOALLOC_SCRATCH_BYTES)
                return fail(SWA_ERR_WORKSPACE,
                            "this call's %d-way split needs %lld bytes of scratch, above the fixed "
                            "%zu-byte maximum of swa_verify_attn_noalloc; pass fewer splits "
                            "(num_splits = 1 needs none)",
                            pl.splits, pl.workspace, (size_t)SWA_NOALLOC_SCRATCH_BYTES);
            st = noalloc_scratch(dev, &ws);
        } else {
            st = ensure_workspace(dev, (size_t)pl.workspace, s, &ws);
        }
        if (st != SWA_OK) return st;
        P.part_acc = static_cast<float *>(ws);
        P.part_ml = P.part_acc + (size_t)P.B * P.Hkv * P.splits * P.R * dims->head_dim;
    }
    st = launch_plan(pl, dims, P, q, k_cache, v_cache, s, cache_rows);
    if (st != SWA_OK) return st;
    t_last_error[0] = '\0';
    return SWA_OK;
}

}  // namespace

extern "C" {

swa_status swa_verify_attn(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *seq_lens, const int32_t *q_pos, int32_t window,
                           float scale, void *out, float *lse, const swa_dims *dims,
                           swa_stream_t stream) {
    return verify_impl(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out, lse, dims, stream,
                       nullptr);
}

swa_status swa_verify_attn_paged(const void *q, const void *k_pages, const void *v_pages,
                                 const swa_paged *paged, const int32_t *seq_lens,
                                 const int32_t *q_pos, int32_t window, float scale, void *out,
                                 float *lse, const swa_dims *dims, swa_stream_t stream) {
    const swa_status st = check_paged(paged, dims);
    if (st != SWA_OK) return st;
    return verify_impl(q, k_pages, v_pages, seq_lens, q_pos, window, scale, out, lse, dims, stream,
                       paged);
}

swa_status swa_append_verify_attn(const void *q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, const swa_paged *paged,
                                  const int32_t *seq_lens, const int32_t *q_pos, int32_t window,
                                  float scale, void *out, float *lse, const swa_dims *dims,
                                  swa_stream_t stream) {
    if (k_new == nullptr || v_new == nullptr)
        return fail(SWA_ERR_INVALID_ARG, "k_new and v_new must not be NULL");
    if (paged != nullptr) {
        const swa_status st = check_paged(paged, dims);
        if (st != SWA_OK) return st;
    }
    return verify_impl(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out, lse, dims, stream,
                       paged, k_new, v_new);
}

size_t swa_workspace_bytes(const swa_dims *dims, int32_t window) {
    if (validate_dims(dims, window) != SWA_OK) return 0;
    // the largest split count any device could get: the plan for a 1-SM part
    // is not larger than kMaxSplits chunks of one tile each
    const int G = dims->num_q_heads / dims->num_kv_heads;
    const long long R = (long long)dims->q_len * G;
    long long span = (long long)window + dims->q_len - 1;
    if (span > dims->max_len) span = dims->max_len;
    long long splits;
    if (dims->num_splits > 0) {
        splits = dims->num_splits > kMaxSplits ? kMaxSplits : dims->num_splits;
    } else {
        splits = (span + swa::kSimtTileKeys - 1) / swa::kSimtTileKeys;
        if (splits > kMaxSplits) splits = kMaxSplits;
    }
    if (splits <= 1) return 0;
    return (size_t)dims->batch * dims->num_kv_heads * splits * R * (dims->head_dim + 2) * 4;
}

swa_status swa_set_workspace(void *dev_ptr, size_t bytes) {
    if ((dev_ptr == nullptr) != (bytes == 0))
        return fail(SWA_ERR_INVALID_ARG, "dev_ptr and bytes must be both set or both zero");
    if (dev_ptr && !aligned16(dev_ptr))
        return fail(SWA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev >= kMaxDevices) return fail(SWA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace &w = g_ws[dev];
    if (w.owned && w.ptr) {
        e = cudaFree(w.ptr);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
    }
    w.ptr = dev_ptr;
    w.bytes = bytes;
    w.owned = false;
    return SWA_OK;
}

swa_status swa_release_workspace(void) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev >= kMaxDevices) return fail(SWA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace &w = g_ws[dev];
    if (w.owned && w.ptr) {
        e = cudaFree(w.ptr);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
        w = Workspace{};
    }
    return SWA_OK;
}

swa_status swa_plan(const swa_dims *dims, int32_t window, int32_t num_sms, swa_plan_info *plan) {
    swa_status st = validate_dims(dims, window);
    if (st != SWA_OK) return st;
    if (plan == nullptr) return fail(SWA_ERR_INVALID_ARG, "plan is NULL");
    if (num_sms < 1) return fail(SWA_ERR_INVALID_ARG, "num_sms %d < 1", num_sms);
    const Plan p = make_plan(dims, window, num_sms, true);
    plan->kernel = p.kernel;
    plan->num_splits = p.splits;
    plan->chunk_keys = p.chunk;
    plan->row_tiles = p.row_tiles;
    plan->rows_per_tile = p.rows_per_tile;
    plan->grid_ctas = (int32_t)p.grid;
    plan->merge = p.splits > 1 ? 1 : 0;
    plan->workspace_bytes = p.workspace;
    return SWA_OK;
}

const char *swa_last_error(void) { return t_last_error; }

swa_status swa_read_device_errors(uint32_t *flags) {
    if (flags == nullptr) return fail(SWA_ERR_INVALID_ARG, "flags is NULL");
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    e = cudaMemcpyFromSymbol(&v, g_fault_word, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e, "read fault word");
    e = cudaMemcpyToSymbol(g_fault_word, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "clear fault word");
    *flags = v;
    return SWA_OK;
}

swa_status swa_read_debug_checks(uint32_t *count) {
    if (count == nullptr) return fail(SWA_ERR_INVALID_ARG, "count is NULL");
    *count = 0;
    if (!swa::kDebugChecks)
        return fail(SWA_ERR_UNSUPPORTED, "the library was built without SWA_DEBUG_CHECKS");
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    e = cudaMemcpyFromSymbol(&v, g_fault_word, sizeof v, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "read debug-check count");
    e = cudaMemcpyToSymbol(g_fault_word, &zero, sizeof zero, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "clear debug-check count");
    *count = v;
    return SWA_OK;
}

const char *swa_version(void) {
    return swa::kDebugChecks ? "swa 0.1.0 sm_103a debug-checks" : "swa 0.1.0 sm_103a";
}

swa_status swa_set_debug_options(const swa_debug_options *opt) {
    swa_debug_options d{0, 1, 0, -1, 0, 0, 0};
    if (opt != nullptr) d = *opt;
    if (d.force_kernel < 0 || d.force_kernel > 4)
        return fail(SWA_ERR_INVALID_ARG, "force_kernel %d outside [0, 4]", d.force_kernel);
    if (d.pdl != 0 && d.pdl != 1) return fail(SWA_ERR_INVALID_ARG, "pdl %d is not 0 or 1", d.pdl);
    if (d.wait_limit_cycles < 0)
        return fail(SWA_ERR_INVALID_ARG, "wait_limit_cycles %lld < 0",
                    (long long)d.wait_limit_cycles);
    if (d.withhold_fill < -1)
        return fail(SWA_ERR_INVALID_ARG, "withhold_fill %d < -1", d.withhold_fill);
    if (d.rows_per_item < 0)
        return fail(SWA_ERR_INVALID_ARG, "rows_per_item %d < 0", d.rows_per_item);
    if (d.fail_launch < 0)
        return fail(SWA_ERR_INVALID_ARG, "fail_launch %d < 0", d.fail_launch);
    if (d.reserved != 0) return fail(SWA_ERR_INVALID_ARG, "reserved %d is not 0", d.reserved);
    g_opt_force.store(d.force_kernel, std::memory_order_relaxed);
    g_opt_pdl.store(d.pdl, std::memory_order_relaxed);
    g_opt_wait_limit.store(d.wait_limit_cycles, std::memory_order_relaxed);
    g_opt_withhold.store(d.withhold_fill, std::memory_order_relaxed);
    g_opt_rows.store(d.rows_per_item, std::memory_order_relaxed);
    g_opt_fail_launch.store(d.fail_launch, std::memory_order_relaxed);
    return SWA_OK;
}

swa_status swa_get_debug_options(swa_debug_options *opt) {
    if (opt == nullptr) return fail(SWA_ERR_INVALID_ARG, "opt is NULL");
    opt->force_kernel = g_opt_force.load(std::memory_order_relaxed);
    opt->pdl = g_opt_pdl.load(std::memory_order_relaxed);
    opt->wait_limit_cycles = g_opt_wait_limit.load(std::memory_order_relaxed);
    opt->withhold_fill = g_opt_withhold.load(std::memory_order_relaxed);
    opt->rows_per_item = g_opt_rows.load(std::memory_order_relaxed);
    opt->fail_launch = g_opt_fail_launch.load(std::memory_order_relaxed);
    opt->reserved = 0;
    return SWA_OK;
}

}  // extern "C"

bool swa::pdl_enabled() { return g_opt_pdl.load(std::memory_order_relaxed) != 0; }

bool swa::launch_fault_due() {
    int n = g_opt_fail_launch.load(std::memory_order_relaxed);
    while (n > 0)
        if (g_opt_fail_launch.compare_exchange_weak(n, n - 1, std::memory_order_relaxed))
            return n == 1;
    return false;
}

// ------------------------------------------------ greedy verification

namespace {

struct AcceptScratch {
    void *ptr = nullptr;
    size_t rows = 0, seqs = 0;  // capacity: best slots, arrival counters
};
std::mutex g_acc_mutex;
AcceptScratch g_acc[kMaxDevices];

// Zero-filled scratch of >= rows 64-bit slots and >= seqs counters; every
// call leaves it zero again.  Grown (and zeroed on `stream`) outside stream
// capture only.
swa_status ensure_accept_scratch(int dev, size_t rows, size_t seqs, cudaStream_t stream,
                                 unsigned long long **best, uint32_t **done) {
    std::lock_guard<std::mutex> lock(g_acc_mutex);
    AcceptScratch &a = g_acc[dev];
    if (a.rows < rows || a.seqs < seqs) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        cudaError_t e = cudaStreamIsCapturing(stream, &cap);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
        if (cap != cudaStreamCaptureStatusNone)
            return fail(SWA_ERR_WORKSPACE,
                        "stream is capturing and the acceptance scratch (%zu rows, %zu sequences) "
                        "is below the %zu rows, %zu sequences needed; run one call outside capture "
                        "first", a.rows, a.seqs, rows, seqs);
        if (a.ptr) {
            e = cudaFree(a.ptr);
            a.ptr = nullptr;
            a.rows = a.seqs = 0;
            if (e != cudaSuccess) return cuda_fail(e, "cudaFree(acceptance scratch)");
        }
        const size_t nr = rows + rows / 4, ns = seqs + seqs / 4;
        const size_t bytes = nr * 8 + ns * 4;
        e = cudaMalloc(&a.ptr, bytes);
        if (e != cudaSuccess) {
            a.ptr = nullptr;
            return cuda_fail(e, "cudaMalloc(acceptance scratch)");
        }
        e = cudaMemsetAsync(a.ptr, 0, bytes, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(acceptance scratch)");
        a.rows = nr;
        a.seqs = ns;
    }
    *best = static_cast<unsigned long long *>(a.ptr);
    *done = reinterpret_cast<uint32_t *>(static_cast<unsigned long long *>(a.ptr) + a.rows);
    return SWA_OK;
}

}  // namespace

extern "C" {

swa_status swa_greedy_accept(const void *logits, const int32_t *keep_ids, const int32_t *draft,
                             int32_t *argmax_out, int32_t *accepted, int32_t batch,
                             int32_t q_len, int32_t vocab, swa_stream_t stream) {
    if (batch < 1 || batch > 65535)
        return fail(SWA_ERR_INVALID_ARG, "batch %d outside [1, 65535]", batch);
    if (q_len < 1 || q_len > kMaxQLen)
        return fail(SWA_ERR_INVALID_ARG, "q_len %d outside [1, %d]", q_len, kMaxQLen);
    if (vocab < 1) return fail(SWA_ERR_INVALID_ARG, "vocab %d < 1", vocab);
    if (!logits || !argmax_out || !accepted || (q_len > 1 && !draft))
        return fail(SWA_ERR_INVALID_ARG, "a required pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(logits) & 1u) || (reinterpret_cast<uintptr_t>(argmax_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(accepted) & 3u) || (reinterpret_cast<uintptr_t>(draft) & 3u) ||
        (reinterpret_cast<uintptr_t>(keep_ids) & 3u))
        return fail(SWA_ERR_INVALID_ARG, "logits must be 2-byte and the int32 arrays 4-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev >= kMaxDevices) return fail(SWA_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    swa::AcceptParams A{};
    swa_status st = ensure_accept_scratch(dev, (size_t)batch * q_len, (size_t)batch, s, &A.best,
                                          &A.done);
    if (st != SWA_OK) return st;
    // about eight CTAs per SM over all rows (so the last CTAs to finish are
    // a small share of the launch), chunks of >= 16384 logits (measured on
    // GB300, us: B=64 q8 V=262144 50.5 -> 45.9, B=16 18.4 -> 16.6, B=1 6.1 ->
    // 5.4 against two CTAs per SM and chunks of >= 4096)
    const long long rows = (long long)batch * q_len;
    long long nsplit = (8LL * device_sms(dev) + rows - 1) / rows;
    const long long by_len = ((long long)vocab + 16383) / 16384;
    if (nsplit > by_len) nsplit = by_len;
    if (nsplit < 1) nsplit = 1;
    long long chunk = ((long long)vocab + nsplit - 1) / nsplit;
    chunk = (chunk + 7) / 8 * 8;
    nsplit = ((long long)vocab + chunk - 1) / chunk;
    A.logits = static_cast<const uint16_t *>(logits);
    A.keep = keep_ids;
    A.draft = draft;
    A.argmax = argmax_out;
    A.accepted = accepted;
    A.B = batch;
    A.q_len = q_len;
    A.V = vocab;
    A.nsplit = (int)nsplit;
    A.chunk = (int)chunk;
    e = swa::launch_kernel(swa::swa_accept_kernel, dim3((unsigned)nsplit, (unsigned)q_len,
                                                        (unsigned)batch),
                           dim3(swa::kAcceptThreads), 0, s, A);
    if (e != cudaSuccess) return cuda_fail(e, "acceptance kernel launch");
    t_last_error[0] = '\0';
    return SWA_OK;
}

}  // extern "C"

// ------------------------------------------------- allocation-free variant

extern "C" swa_status swa_verify_attn_noalloc(const void *q, const void *k_cache,
                                              const void *v_cache, const int32_t *seq_lens,
                                              const int32_t *q_pos, int32_t window, float scale,
                                              void *out, float *lse, const swa_dims *dims,
                                              swa_stream_t stream) {
    return verify_impl(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out, lse, dims, stream,
                       nullptr, nullptr, nullptr, /*noalloc=*/true);
}
