// Greedy verification of a draft block: a fused argmax over every verify
// row's logits and the longest accepted draft prefix, in one launch.
//
// Grid (vocabulary chunks, q_len rows, sequences).  Each thread keeps a
// running (value, column) over its logits (strictly larger wins: a NaN never
// wins, the first of equal maxima stays); the CTA's best pair is packed into
// 64 bits so that one unsigned maximum orders by value and then by the
// smaller column: key = orderable(value) << 32 | (0xffffffff - column).  The CTA folds its key into the row's slot with
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

// Total order on float bits for an unsigned maximum (-inf lowest of the
// values that can win; NaN never reaches here).  -0.0 and +0.0 compare equal
// as floats (the per-thread scan treats them as one value), so both map to
// the key of +0.0: otherwise a later +0.0 column would beat an earlier -0.0
// column across threads or CTAs and break "the first of equal maxima".
__device__ __forceinline__ uint32_t accept_key(float x) {
    const uint32_t u = x == 0.f ? 0u : __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long accept_pack(float x, uint32_t j) {
    return ((unsigned long long)accept_key(x) << 32) | (unsigned long long)(0xffffffffu - j);
}

// One logit into a thread's running (value, column): strictly larger wins,
// so a NaN never wins and, columns coming in increasing order, the first of
// equal maxima stays.
__device__ __forceinline__ void accept_step(float x, uint32_t j, float &bv, uint32_t &bj) {
    const bool gt = x > bv;
    bv = gt ? x : bv;
    bj = gt ? j : bj;
}

__global__ void __launch_bounds__(kAcceptThreads) swa_accept_kernel(const AcceptParams A) {
    __shared__ unsigned long long red[kAcceptThreads / 32];
    __shared__ int32_t match[64];
    __shared__ int last;
    grid_dep_wait();
    grid_dep_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.z, i = blockIdx.y;
    const long long c0 = (long long)blockIdx.x * A.chunk;
    long long c1 = c0 + A.chunk;
    if (c1 > A.V) c1 = A.V;
    const uint16_t *row = A.logits + ((size_t)b * A.q_len + i) * (size_t)A.V;
    // a chunk with nothing above -inf offers its first column: the row's
    // answer is then column 0, the first of all
    float bv = -__int_as_float(0x7f800000);
    uint32_t bj = (uint32_t)c0;
    if (c0 < c1) {
        // scalar head up to a 16-byte boundary, 8 logits per 16-byte load, tail
        long long head = (long long)(((16 - (reinterpret_cast<uintptr_t>(row + c0) & 15)) & 15) >> 1);
        if (head > c1 - c0) head = c1 - c0;
        for (long long j = c0 + tid; j < c0 + head; j += kAcceptThreads)
            accept_step(__uint_as_float((uint32_t)row[j] << 16), (uint32_t)j, bv, bj);
        const long long v0 = c0 + head;
        const long long nvec = (c1 - v0) >> 3;
        const uint4 *vrow = reinterpret_cast<const uint4 *>(row + v0);
#pragma unroll 4
        for (long long q = tid; q < nvec; q += kAcceptThreads) {
            const uint4 w = __ldg(vrow + q);
            const uint32_t j = (uint32_t)(v0 + 8 * q);
            accept_step(__uint_as_float(w.x << 16), j + 0, bv, bj);
            accept_step(__uint_as_float(w.x & 0xffff0000u), j + 1, bv, bj);
            accept_step(__uint_as_float(w.y << 16), j + 2, bv, bj);
            accept_step(__uint_as_float(w.y & 0xffff0000u), j + 3, bv, bj);
            accept_step(__uint_as_float(w.z << 16), j + 4, bv, bj);
            accept_step(__uint_as_float(w.z & 0xffff0000u), j + 5, bv, bj);
            accept_step(__uint_as_float(w.w << 16), j + 6, bv, bj);
            accept_step(__uint_as_float(w.w & 0xffff0000u), j + 7, bv, bj);
        }
        for (long long j = v0 + 8 * nvec + tid; j < c1; j += kAcceptThreads)
            accept_step(__uint_as_float((uint32_t)row[j] << 16), (uint32_t)j, bv, bj);
    }
    unsigned long long best = accept_pack(bv, bj);
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
        last = atomicAdd(&A.done[b], 1u) == (uint32_t)(A.nsplit * A.q_len - 1);
    }
    __syncthreads();
    if (!last) return;
    // last CTA of sequence b: every row's slot is final; one thread per row
    // reads and clears it, maps the column and compares with its draft
    __threadfence();
    if (tid < A.q_len) {
        const unsigned long long k = atomicExch(&A.best[(size_t)b * A.q_len + tid], 0ull);
        const uint32_t j = 0xffffffffu - (uint32_t)(k & 0xffffffffu);
        const int32_t tok = A.keep ? A.keep[j] : (int32_t)j;
        A.argmax[(size_t)b * A.q_len + tid] = tok;
        match[tid] = tid < A.q_len - 1 && tok == A.draft[(size_t)b * (A.q_len - 1) + tid];
    }
    __syncthreads();
    if (tid == 0) {
        int n = 0;
        while (n < A.q_len - 1 && match[n]) ++n;
        A.accepted[b] = n;
        atomicExch(&A.done[b], 0u);
    }
}

}  // namespace swa
