/*
 * Sliding-window verify attention: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code with the CUDA library.
 *
 * What it computes (the definition, written out, no blocking or fusion):
 *   "The Fast Gemma Challenge: our verified-SOTA recipe, in full", section
 *   "What each piece does, and why", bullet "Sliding window
 *   SLIDING_WINDOW=188": each query attends only to the most recent W tokens.
 *   The window edge is read as the half-open interval (p-W, p], i.e. W keys
 *   including the query's own position.
 *
 *   For sequence b, query head h, draft row i (absolute position
 *   p = q_pos[b] + i) and KV head g = floor(h / G), G = Hq / Hkv:
 *     K(p) = { j : max(0, p-W+1) <= j <= p  and  j < seq_len[b] }
 *     s_j  = scale * sum_d q[b,i,h,d] * k[b,g,j,d]                j in K(p)
 *     lse  = ln sum_{j in K(p)} exp(s_j)
 *     out  = sum_{j in K(p)} exp(s_j - lse) * v[b,g,j,:]
 *   An empty K(p) gives out = 0 and lse = -inf.
 *
 *   The split-KV partial of a key range [c_lo, c_hi) and the log-sum-exp
 *   merge of such partials ("split-KV verify kernel", SPLITKV_VERIFY=1, in
 *   the manifest of the same page) are written out below as well, so that
 *   the merge identity can be checked on the CPU.
 *
 * Inputs are doubles (the exact bf16 values widened).  K and V are given as
 * a window slice per sequence: row t of sequence b holds absolute position
 * base[b] + t, t in [0, T).  A key the definition needs that lies outside the
 * slice is an error (return code 2), never silently skipped.
 *
 * Layouts (all contiguous, row-major):
 *   q    [B, q_len, Hq, D]      k, v  [B, Hkv, T, D]
 *   out  [B, q_len, Hq, D]      lse   [B, q_len, Hq]
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v;
    const int64_t *base, *seq_lens, *q_pos;
    int64_t B, q_len, Hq, Hkv, D, T, window;
    double scale;
    /* key range restriction for partials: [c_lo, c_hi) absolute, or none */
    int restrict_range;
    const int64_t *c_lo, *c_hi; /* per sequence */
    /* results */
    double *out, *lse;          /* full attention */
    double *pm, *pl, *pacc;     /* partials: m, l [B,q_len,Hq], acc [B,q_len,Hq,D] */
    int nthreads, tid;
    int status;
} job_t;

/* Valid key interval of one query row, inclusive; empty when lo > hi. */
static void key_interval(int64_t p, int64_t window, int64_t seq_len,
                         int64_t *lo, int64_t *hi)
{
    int64_t a = p - window + 1;
    *lo = a > 0 ? a : 0;
    *hi = p < seq_len - 1 ? p : seq_len - 1;
}

/* One (sequence, query head) pair: every draft row. */
static int one_head(const job_t *J, int64_t b, int64_t h, double *s)
{
    const int64_t G = J->Hq / J->Hkv;
    const int64_t g = h / G;
    const int64_t D = J->D, T = J->T;
    const double *kb = J->k + ((b * J->Hkv + g) * T) * D;
    const double *vb = J->v + ((b * J->Hkv + g) * T) * D;
    for (int64_t i = 0; i < J->q_len; ++i) {
        const int64_t p = J->q_pos[b] + i;
        const double *qr = J->q + ((b * J->q_len + i) * J->Hq + h) * D;
        const int64_t row = (b * J->q_len + i) * J->Hq + h;
        int64_t lo, hi;
        key_interval(p, J->window, J->seq_lens[b], &lo, &hi);
        if (J->restrict_range) {
            if (lo < J->c_lo[b]) lo = J->c_lo[b];
            if (hi > J->c_hi[b] - 1) hi = J->c_hi[b] - 1;
        }
        if (lo > hi) { /* no key: defined result */
            if (J->restrict_range) {
                J->pm[row] = -INFINITY;
                J->pl[row] = 0.0;
                memset(J->pacc + row * D, 0, (size_t)D * sizeof(double));
            } else {
                J->lse[row] = -INFINITY;
                memset(J->out + row * D, 0, (size_t)D * sizeof(double));
            }
            continue;
        }
        if (lo < J->base[b] || hi >= J->base[b] + T) return 2;
        /* scores */
        double m = -INFINITY;
        for (int64_t j = lo; j <= hi; ++j) {
            const double *kr = kb + (j - J->base[b]) * D;
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += qr[d] * kr[d];
            s[j - lo] = J->scale * dot;
            if (s[j - lo] > m) m = s[j - lo];
        }
        /* max-subtracted exponentials */
        double z = 0.0;
        for (int64_t j = lo; j <= hi; ++j) {
            s[j - lo] = exp(s[j - lo] - m);
            z += s[j - lo];
        }
        if (J->restrict_range) {
            double *acc = J->pacc + row * D;
            for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
            for (int64_t j = lo; j <= hi; ++j) {
                const double *vr = vb + (j - J->base[b]) * D;
                for (int64_t d = 0; d < D; ++d) acc[d] += s[j - lo] * vr[d];
            }
            J->pm[row] = m;
            J->pl[row] = z;
        } else {
            double *o = J->out + row * D;
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t j = lo; j <= hi; ++j) {
                const double w = s[j - lo] / z; /* = exp(s_j - lse) */
                const double *vr = vb + (j - J->base[b]) * D;
                for (int64_t d = 0; d < D; ++d) o[d] += w * vr[d];
            }
            J->lse[row] = m + log(z);
        }
    }
    return 0;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const int64_t units = J->B * J->Hq;
    /* a row's keys lie inside the slice (checked before use), so T bounds them */
    double *s = (double *)malloc((size_t)(J->T + 1) * sizeof(double));
    if (!s) { J->status = 3; return NULL; }
    for (int64_t u = J->tid; u < units; u += J->nthreads) {
        int rc = one_head(J, u / J->Hq, u % J->Hq, s);
        if (rc) { J->status = rc; break; }
    }
    free(s);
    return NULL;
}

static int run(job_t *proto)
{
    if (proto->B < 0 || proto->q_len < 0 || proto->Hq < 1 || proto->Hkv < 1 ||
        proto->D < 1 || proto->T < 0 || proto->window < 1 ||
        proto->Hq % proto->Hkv != 0)
        return 1;
    int nt = proto->nthreads > 0 ? proto->nthreads : 1;
    job_t *jobs = (job_t *)calloc((size_t)nt, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 3; }
    for (int t = 0; t < nt; ++t) {
        jobs[t] = *proto;
        jobs[t].nthreads = nt;
        jobs[t].tid = t;
        jobs[t].status = 0;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, worker, &jobs[t]);
    worker(&jobs[0]);
    for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
    int status = 0;
    for (int t = 0; t < nt; ++t) if (jobs[t].status) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}

/* Full windowed attention.  Returns 0, 1 (bad shape), 2 (slice too short)
 * or 3 (out of memory). */
int oracle_swa_attention(const double *q, const double *k, const double *v,
                         const int64_t *base, const int64_t *seq_lens,
                         const int64_t *q_pos, int64_t B, int64_t q_len,
                         int64_t Hq, int64_t Hkv, int64_t D, int64_t T,
                         int64_t window, double scale, double *out, double *lse,
                         int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v;
    J.base = base; J.seq_lens = seq_lens; J.q_pos = q_pos;
    J.B = B; J.q_len = q_len; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.T = T;
    J.window = window; J.scale = scale;
    J.out = out; J.lse = lse;
    J.nthreads = nthreads;
    return run(&J);
}

/* Split-KV partial over the key range [c_lo[b], c_hi[b]) intersected with
 * each row's window: m = max score, l = sum exp(s - m),
 * acc = sum exp(s - m) * v.  An empty range gives m = -inf, l = 0, acc = 0. */
int oracle_swa_partial(const double *q, const double *k, const double *v,
                       const int64_t *base, const int64_t *seq_lens,
                       const int64_t *q_pos, int64_t B, int64_t q_len,
                       int64_t Hq, int64_t Hkv, int64_t D, int64_t T,
                       int64_t window, double scale, const int64_t *c_lo,
                       const int64_t *c_hi, double *m, double *l, double *acc,
                       int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v;
    J.base = base; J.seq_lens = seq_lens; J.q_pos = q_pos;
    J.B = B; J.q_len = q_len; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.T = T;
    J.window = window; J.scale = scale;
    J.restrict_range = 1; J.c_lo = c_lo; J.c_hi = c_hi;
    J.pm = m; J.pl = l; J.pacc = acc;
    J.nthreads = nthreads;
    return run(&J);
}

/* Log-sum-exp merge of n partials for `rows` independent rows:
 *   M = max_k m_k,  Lambda = sum_k l_k exp(m_k - M),
 *   out = sum_k acc_k exp(m_k - M) / Lambda,  lse = M + ln Lambda.
 * Layouts: m, l [n, rows]; acc [n, rows, D]; out [rows, D]; lse [rows].
 * A row whose partials are all empty gives out = 0, lse = -inf. */
int oracle_lse_merge(const double *m, const double *l, const double *acc,
                     int64_t n, int64_t rows, int64_t D, double *out,
                     double *lse)
{
    if (n < 1 || rows < 0 || D < 1) return 1;
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int64_t k = 0; k < n; ++k)
            if (m[k * rows + r] > M) M = m[k * rows + r];
        double *o = out + r * D;
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        if (M == -INFINITY) { lse[r] = -INFINITY; continue; }
        double Lam = 0.0;
        for (int64_t k = 0; k < n; ++k) {
            const double mk = m[k * rows + r];
            if (mk == -INFINITY) continue;
            const double w = exp(mk - M);
            Lam += l[k * rows + r] * w;
            const double *a = acc + (k * rows + r) * D;
            for (int64_t d = 0; d < D; ++d) o[d] += w * a[d];
        }
        for (int64_t d = 0; d < D; ++d) o[d] /= Lam;
        lse[r] = M + log(Lam);
    }
    return 0;
}

/* Greedy verification of a draft block, after the manifest entries
 * FUSED_SPARSE_ARGMAX (argmax sampling over the LM head's logits, possibly a
 * pruned keep set of the vocabulary) and SPECULATIVE_CONFIG (seven drafted
 * tokens per step) of "The Fast Gemma Challenge: our verified-SOTA recipe, in
 * full".  Per sequence b and verify row i (the row at position q_pos + i
 * scores the token that follows it):
 *   argmax[b][i] = keep[j*], j* = the first column j of logits[b][i] whose
 *                  value is the largest (a NaN is never larger; a row with
 *                  no value above -inf gives j* = 0); keep == NULL: j*;
 *   accepted[b]  = the largest n <= q_len - 1 with argmax[b][i] == draft[b][i]
 *                  for every i < n (draft[b][i] is the token fed as row i + 1).
 * Layouts: logits [B, q_len, V]; keep [V] or NULL; draft [B, q_len - 1];
 * argmax [B, q_len]; accepted [B]. */
int oracle_greedy_accept(const double *logits, const int64_t *keep, const int64_t *draft,
                         int64_t B, int64_t q_len, int64_t V, int64_t *argmax,
                         int64_t *accepted)
{
    if (B < 0 || q_len < 1 || V < 1) return 1;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t i = 0; i < q_len; ++i) {
            const double *row = logits + (b * q_len + i) * V;
            double best = -INFINITY;
            int64_t jbest = 0;
            for (int64_t j = 0; j < V; ++j)
                if (row[j] > best) {
                    best = row[j];
                    jbest = j;
                }
            argmax[b * q_len + i] = keep ? keep[jbest] : jbest;
        }
        int64_t n = 0;
        while (n < q_len - 1 && argmax[b * q_len + n] == draft[b * (q_len - 1) + n]) ++n;
        accepted[b] = n;
    }
    return 0;
}

/* Cache write of a verify block's new rows (the step before the attention,
 * done in the same call by the fused append): row i of sequence b's block
 * holds the key / value of position q_pos[b] + i, so for every KV head h
 *   cache[b][h][q_pos[b] + i][:] = rows[b][i][h][:]
 * for each i with 0 <= q_pos[b] + i < min(seq_len[b], L); no other cache
 * entry changes.  In place on `cache`.
 * Layouts: cache [B, Hkv, L, D]; rows [B, q_len, Hkv, D]. */
int oracle_append_rows(double *cache, const double *rows, const int64_t *q_pos,
                       const int64_t *seq_lens, int64_t B, int64_t q_len, int64_t Hkv,
                       int64_t L, int64_t D)
{
    if (B < 0 || q_len < 1 || Hkv < 1 || L < 1 || D < 1) return 1;
    for (int64_t b = 0; b < B; ++b) {
        const int64_t end = seq_lens[b] < L ? seq_lens[b] : L;
        for (int64_t i = 0; i < q_len; ++i) {
            const int64_t pos = q_pos[b] + i;
            if (pos < 0 || pos >= end) continue;
            for (int64_t h = 0; h < Hkv; ++h) {
                const double *src = rows + ((b * q_len + i) * Hkv + h) * D;
                double *dst = cache + ((b * Hkv + h) * L + pos) * D;
                for (int64_t d = 0; d < D; ++d) dst[d] = src[d];
            }
        }
    }
    return 0;
}
