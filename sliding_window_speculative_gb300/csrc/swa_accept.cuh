// Greedy verification of a draft block: a fused argmax over every verify
// row's logits and the longest accepted draft prefix, in one launch.
//
// Grid (vocabulary chunks, q_len rows, sequences).  Each CTA reduces its
// chunk of one row to the best (value, column) pair, packed into 64 bits
// so that one unsigned maximum orders by value and then by the smaller
// column: key = orderable(value) << 32 | (0xffffffff - column), where a NaN
// orders like -inf.  The CTA folds its key into the row's slot with
// atomicMax; the last CTA of a sequence (a per-sequence arrival counter)
// reads and clears the slots, maps the winning columns through the keep
// set, counts the accepted prefix and clears the counter, so the scratch is
// all zero again after every call.
#pragma once

#include "swa_common.cuh"

namespace swa {

constexpr int kAcceptThreads = 256;

struct AcceptParams {
    const uint16_t *logits;  // bf16 bits [B, q_len, V]
    const int32_t *keep;     // [V] or null
    const int32_t *draft;    // [B, q_len - 1] (null when q_len == 1)
    int32_t *argmax;         // [B, q_len]
    int32_t *accepted;       // [B]
    unsigned long long *best;  // scratch [B * q_len], zero on entry and exit
    uint32_t *done;            // scratch [B], zero on entry and exit
    int B, q_len, V, nsplit, chunk;
};

// Total order on float bits for an unsigned maximum; NaN maps to -inf's key.
__device__ __forceinline__ uint32_t accept_key(uint32_t u) {
    if ((u & 0x7fffffffu) > 0x7f800000u) u = 0xff800000u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long accept_pack(uint16_t h, uint32_t j) {
    return ((unsigned long long)accept_key((uint32_t)h << 16) << 32) |
           (unsigned long long)(0xffffffffu - j);
}

__global__ void __launch_bounds__(kAcceptThreads) swa_accept_kernel(const AcceptParams A) {
    __shared__ unsigned long long red[kAcceptThreads / 32];
    __shared__ int32_t toks[64];
    grid_dep_wait();
    grid_dep_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.z, i = blockIdx.y;
    const long long c0 = (long long)blockIdx.x * A.chunk;
    long long c1 = c0 + A.chunk;
    if (c1 > A.V) c1 = A.V;
    const uint16_t *row = A.logits + ((size_t)b * A.q_len + i) * (size_t)A.V;
    unsigned long long best = 0;
    if (c0 < c1) {
        // scalar head up to a 16-byte boundary, 8 logits per 16-byte load, tail
        long long head = (long long)(((16 - (reinterpret_cast<uintptr_t>(row + c0) & 15)) & 15) >> 1);
        if (head > c1 - c0) head = c1 - c0;
        for (long long j = c0 + tid; j < c0 + head; j += kAcceptThreads) {
            const unsigned long long k = accept_pack(row[j], (uint32_t)j);
            best = k > best ? k : best;
        }
        const long long v0 = c0 + head;
        const long long nvec = (c1 - v0) >> 3;
        const uint4 *vrow = reinterpret_cast<const uint4 *>(row + v0);
#pragma unroll 4
        for (long long q = tid; q < nvec; q += kAcceptThreads) {
            const uint4 w = __ldg(vrow + q);
            const uint32_t j = (uint32_t)(v0 + 8 * q);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const unsigned long long k0 = accept_pack((uint16_t)(ws[e] & 0xffffu), j + 2 * e);
                const unsigned long long k1 = accept_pack((uint16_t)(ws[e] >> 16), j + 2 * e + 1);
                best = k0 > best ? k0 : best;
                best = k1 > best ? k1 : best;
            }
        }
        for (long long j = v0 + 8 * nvec + tid; j < c1; j += kAcceptThreads) {
            const unsigned long long k = accept_pack(row[j], (uint32_t)j);
            best = k > best ? k : best;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o > best ? o : best;
    }
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kAcceptThreads / 32; ++w) best = red[w] > best ? red[w] : best;
        atomicMax(&A.best[(size_t)b * A.q_len + i], best);
        __threadfence();
        const uint32_t arrived = atomicAdd(&A.done[b], 1u);
        if (arrived == (uint32_t)(A.nsplit * A.q_len - 1)) {
            // last CTA of sequence b: every row's slot is final
            __threadfence();
            for (int r = 0; r < A.q_len; ++r) {
                const unsigned long long k = atomicExch(&A.best[(size_t)b * A.q_len + r], 0ull);
                const uint32_t j = 0xffffffffu - (uint32_t)(k & 0xffffffffu);
                const int32_t tok = A.keep ? A.keep[j] : (int32_t)j;
                toks[r] = tok;
                A.argmax[(size_t)b * A.q_len + r] = tok;
            }
            int n = 0;
            while (n < A.q_len - 1 && toks[n] == A.draft[(size_t)b * (A.q_len - 1) + n]) ++n;
            A.accepted[b] = n;
            atomicExch(&A.done[b], 0u);
        }
    }
}

}  // namespace swa
