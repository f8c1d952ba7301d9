/*
 * spec_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU restatement of batched speculative-sampling verification.
 * It exists to check the CUDA path; nothing in the product links, loads or calls it.
 * Only the test suite, the smoke check and the CPU-baseline leg of the benchmark use it.
 * It shares no source, header, table or constant with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *  [SpS]  "Speculative Decoding 为什么是 Lossless 的 — 详细证明教程" (speculative decoding lossless
 *         proof tutorial): §2.2 notation (p = target, q = draft, a(x), (p-q)+, Z, p'), §5.1 algorithm
 *         SpecSampleOne, §6.2-§6.4 proof steps, §7 worked examples, §8 Q1/Q2/Q4 pitfalls,
 *         §9.1 gamma-step chain.
 *  [Hedge] "Not-a-Bandit: Provably No-Regret Drafter Selection in Speculative Decoding for LLMs"
 *         (HedgeSpec notes): Key design 1, counterfactual acceptance gamma_{j,i} = 1 - TV(p, q_i);
 *         Key design 3, loss f_t[i] = 1 - gamma_t[i].
 *  [Cactus] "Cactus: Accelerating Auto-Regressive Decoding with Constrained Acceptance Speculative
 *         Sampling" (Cactus notes): Key design 1 (objective min{h_n/p(n),1}), Key design 2 (closed-form
 *         h; gamma* the root of the divergence constraint on [q(n), +inf), clamped to [q(n), 1]), Key
 *         design 3 (gamma* Taylor closed form, KL divergence). NOTE: that page writes q for the verifier
 *         (target) and p for the draft -- the opposite of [SpS]. This file always says target/draft.
 *  Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11),
 *         the counter-based generator; the pages do not fix a uniform source.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - accept iff r * p_draft(t) < p_target(t)  (strict, no division; [SpS] §5.1 gives both forms);
 *  - uniforms: Philox4x32-10, counter (pos, seq, stream, 0), key (seed lo, seed hi), word 0 mapped to
 *    ((w >> 9) + 0.5) * 2^-23, i.e. an odd multiple of 2^-24 below 1 (exact in fp32 and fp64);
 *    stream 0 = accept r, stream 1 = resample / bonus u;
 *  - inverse CDF in ascending token id: the smallest x whose running sum exceeds u * (total mass);
 *  - a reject with Z <= 0 (possible only through rounding) resamples from the target row itself;
 *  - bonus token (all K drafts accepted) is drawn from target row K with u = U(seed, b, K, stream 1);
 *  - Cactus residual g = (h - p_draft)+ / sum (h - p_draft)+ (the page only says phi and g are
 *    "derived back"); Cactus bonus row is the plain target row; p_target(n) = 1 gives gamma* = 1, s = 0.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -fopenmp spec_oracle.c -o libspec_oracle.so -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------------ */
/* Philox4x32-10 (SC'11 paper above): 10 rounds of the 4x32 S-box; the key is bumped by the   */
/* Weyl constants between rounds.                                                             */
/* ------------------------------------------------------------------------------------------ */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void spec_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; round++) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Uniform on the grid (k + 1/2) 2^-23, k in [0, 2^23): strictly inside (0,1), exact in fp32 and fp64. */
double spec_oracle_uniform(uint64_t seed, uint32_t seq, uint32_t pos, uint32_t stream)
{
    uint32_t ctr[4] = {pos, seq, stream, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    spec_oracle_philox4x32_10(ctr, key, out);
    return ((double)(out[0] >> 9) + 0.5) * (1.0 / 8388608.0);
}

/* ------------------------------------------------------------------------------------------ */
/* Row access: bf16 (stored as uint16 bit patterns) or fp32 logits, converted exactly to double. */
/* ------------------------------------------------------------------------------------------ */
enum { ORACLE_BF16 = 0, ORACLE_FP32 = 1 };

static void load_row(int dtype, const void* base, size_t row, int V, double* x)
{
    if (dtype == ORACLE_BF16) {
        const uint16_t* h = (const uint16_t*)base + row * (size_t)V;
        for (int v = 0; v < V; v++) {
            uint32_t bits = (uint32_t)h[v] << 16;
            float f;
            memcpy(&f, &bits, sizeof f);
            x[v] = (double)f;
        }
    } else {
        const float* f = (const float*)base + row * (size_t)V;
        for (int v = 0; v < V; v++) x[v] = (double)f[v];
    }
}

/* Temperature softmax, max-subtracted: p = softmax(x / T). One T for target and draft is the
 * "standardized sampling" rule of [SpS] §8 Q4 (otherwise the ratio compares two different
 * distributions and losslessness is lost). Logits of -inf get probability 0. */
void spec_oracle_softmax(const double* x, int V, double T, double* p)
{
    double M = -INFINITY;
    for (int v = 0; v < V; v++) {
        double z = x[v] / T;
        if (z > M) M = z;
    }
    double S = 0.0;
    for (int v = 0; v < V; v++) {
        p[v] = exp(x[v] / T - M);
        S += p[v];
    }
    for (int v = 0; v < V; v++) p[v] /= S;
}

/* Inverse CDF over a non-negative weight vector in ascending index order: the smallest x with
 * w[0] + ... + w[x] > target. If rounding leaves no such x, the last index with w > 0.
 * *margin = distance (in the same mass units) from target to the nearer of the chosen index's
 * two CDF boundaries. */
int spec_oracle_inverse_cdf(const double* w, int V, double target, double* margin)
{
    double cum = 0.0;
    int last_pos = -1;
    for (int x = 0; x < V; x++) {
        if (w[x] > 0.0) last_pos = x;
        double before = cum;
        cum += w[x];
        if (w[x] > 0.0 && cum > target) {
            if (margin) {
                double a = target - before, b = cum - target;
                *margin = a < b ? a : b;
            }
            return x;
        }
    }
    if (margin) *margin = 0.0;
    return last_pos;
}

/* One verification step, [SpS] §5.1 SpecSampleOne, generalised to any target distribution h
 * (h = p_target for standard speculative sampling; h = the Cactus target for the constrained
 * variant, [Cactus] Key design 1: accept with min{h_n / p_draft(n), 1}).
 *  1. the draft token t was drawn from the draft distribution (an input here);
 *  2. accept iff r * p_draft(t) < h(t), i.e. r < min(1, h(t)/p_draft(t));
 *  3. otherwise draw from p'(x) = (h(x) - p_draft(x))+ / Z with Z = sum_x (h(x) - p_draft(x))+.
 * mutation (tests only, plants the pitfalls of [SpS] §8): 1 = resample from h itself on reject (Q1),
 * 2 = resample from |h - p_draft| (Q2). 0 = the algorithm as written.
 * Outputs: *accepted, *Z (always computed), *accept_margin = |r - h(t)/p_draft(t)|,
 * *cdf_margin (only meaningful when rejected). Returns the emitted token. */
int spec_oracle_sample_one(const double* h, const double* pd, int V, int t, double r, double u,
                           int mutation, int* accepted, double* Z, double* accept_margin,
                           double* cdf_margin, double* scratch)
{
    double z = 0.0;
    for (int x = 0; x < V; x++) {
        double d = h[x] - pd[x];
        z += d > 0.0 ? d : 0.0;
    }
    if (Z) *Z = z;
    if (accept_margin) *accept_margin = pd[t] > 0.0 ? fabs(r - h[t] / pd[t]) : INFINITY;
    if (r * pd[t] < h[t]) {
        *accepted = 1;
        if (cdf_margin) *cdf_margin = INFINITY;
        return t;
    }
    *accepted = 0;
    double* w = scratch;
    double total = 0.0;
    for (int x = 0; x < V; x++) {
        double d = h[x] - pd[x];
        if (mutation == 1) w[x] = h[x];
        else if (mutation == 2) w[x] = fabs(d);
        else w[x] = d > 0.0 ? d : 0.0;
        total += w[x];
    }
    if (!(total > 0.0)) { /* rounding-only reject: fall back to the target row */
        total = 0.0;
        for (int x = 0; x < V; x++) { w[x] = h[x]; total += w[x]; }
    }
    return spec_oracle_inverse_cdf(w, V, u * total, cdf_margin);
}

/* The divergence of the Cactus target from the target row, for candidate probability q = p_target(n) and
 * h_n = g: with h_i = (1 - g) / (1 - q) p_target(i) for i != n, the sum over i != n factors and
 * KL(h || p_target) = g ln(g / q) + (1 - g) ln((1 - g) / (1 - q)), with 0 ln 0 = 0. */
double spec_oracle_cactus_kl(double q, double g)
{
    double a = (g > 0.0) ? g * log(g / q) : 0.0;
    double b = (g < 1.0) ? (1.0 - g) * log((1.0 - g) / (1.0 - q)) : 0.0;
    return a + b;
}

/* gamma* without the Taylor step ([Cactus] Key design 2 with the KL divergence of Key design 3): the root
 * of KL(h || p_target) = delta on [q, +inf), clamped to [q, 1]. The divergence is 0 at g = q and increases
 * on [q, 1] (its derivative ln(g / q) - ln((1 - g) / (1 - q)) is positive there), so the root is found by
 * bisection of [q, 1] down to the spacing of doubles. No root below 1 (ln(1/q) <= delta) gives 1; q = 0
 * gives 0 (every g > 0 has infinite divergence); delta = 0 gives q. */
double spec_oracle_cactus_gamma_kl(double q, double delta)
{
    if (delta <= 0.0 || q <= 0.0) return q;
    if (q >= 1.0) return 1.0;
    if (spec_oracle_cactus_kl(q, 1.0) <= delta) return 1.0;
    double lo = q, hi = 1.0;
    for (int it = 0; it < 200 && hi - lo > 0.0; it++) {
        double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi) break;
        if (spec_oracle_cactus_kl(q, mid) <= delta) lo = mid;
        else hi = mid;
    }
    return lo;
}

/* Cactus target distribution, [Cactus] Key design 2 and 3 (translated: the page's q is the target,
 * its p is the draft). With q = p_target(n) for the candidate n:
 *   gamma* = min(q + sqrt(2 delta q (1 - q)), 1)  (the Taylor closed form, exact = 0), or the root of
 *   the divergence constraint (exact = 1, spec_oracle_cactus_gamma_kl),
 *   h_n = gamma*,  h_i = (1 - gamma*) / (1 - q) * p_target(i) for i != n.
 * q = 1 gives gamma* = 1 and the other entries 0. Returns gamma*. */
double spec_oracle_cactus_h_mode(const double* pt, int V, int n, double delta, int exact, double* h)
{
    double q = pt[n];
    double g;
    if (exact) {
        g = spec_oracle_cactus_gamma_kl(q, delta);
    } else {
        g = q + sqrt(2.0 * delta * q * (1.0 - q));
        if (g > 1.0) g = 1.0;
    }
    double s = (q < 1.0) ? (1.0 - g) / (1.0 - q) : 0.0;
    for (int i = 0; i < V; i++) h[i] = s * pt[i];
    h[n] = g;
    return g;
}

double spec_oracle_cactus_h(const double* pt, int V, int n, double delta, double* h)
{
    return spec_oracle_cactus_h_mode(pt, V, n, delta, 0, h);
}

/* ------------------------------------------------------------------------------------------ */
/* Batched calls.                                                                             */
/* ------------------------------------------------------------------------------------------ */
/* The chain keeps per-position row pointers on the stack. */
#define ORACLE_MAX_K 64

/* The gamma-step chain of [SpS] §9.1 for one sequence: verify draft positions left to right, stop at
 * the first reject and emit the residual draw there; if every draft is accepted, emit one token from
 * target row K. The per-position quantities (diag, margins) are computed for every j, also after the
 * chain stopped, because the batched output reports them for all positions.
 *   hrows[j] : the target distribution used at position j (p_target, or the Cactus h)
 *   drows[j] : the draft distribution at position j
 *   bonus    : target row K (plain softmax). */
static void chain_one(double** hrows, double** drows, const double* bonus, int K, int V,
                      const int32_t* tok, uint64_t seed, uint32_t seq, int mutation,
                      int32_t* accept_len, int32_t* out, double* diag, double* acc_margin,
                      double* cdf_margin, double* scratch)
{
    int L = K, emitted = -1;
    double cm = INFINITY;
    for (int j = 0; j < K; j++) {
        double r = spec_oracle_uniform(seed, seq, (uint32_t)j, 0u);
        double u = spec_oracle_uniform(seed, seq, (uint32_t)j, 1u);
        int acc = 0;
        double Z = 0.0, am = 0.0, c = INFINITY;
        int e = spec_oracle_sample_one(hrows[j], drows[j], V, tok[j], r, u,
                                       (L == K) ? mutation : 0, &acc, &Z, &am, &c, scratch);
        if (diag) {
            diag[4 * j + 0] = hrows[j][tok[j]];
            diag[4 * j + 1] = drows[j][tok[j]];
            diag[4 * j + 2] = Z;
            diag[4 * j + 3] = r;
        }
        if (acc_margin) acc_margin[j] = am;
        if (L == K) {
            if (acc) {
                out[j] = tok[j];
            } else {
                L = j;
                emitted = e;
                cm = c;
            }
        }
    }
    if (L == K) {
        double u = spec_oracle_uniform(seed, seq, (uint32_t)K, 1u);
        double total = 0.0;
        for (int x = 0; x < V; x++) total += bonus[x];
        emitted = spec_oracle_inverse_cdf(bonus, V, u * total, &cm);
    }
    out[L] = emitted;
    for (int j = L + 1; j <= K; j++) out[j] = -1;
    *accept_len = L;
    if (cdf_margin) *cdf_margin = cm;
}

static int nthreads_or_default(int n)
{
#ifdef _OPENMP
    return n > 0 ? n : omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Standard speculative sampling over a batch ([SpS] §5.1 + §9.1).
 * target [B, K+1, V], draft [B, K, V] (dtype: 0 = bf16 bit patterns, 1 = fp32), tokens [B, K],
 * seeds [B]; seq_index [B] (nullable) gives the sequence number used in the Philox counter
 * (identity when NULL). Returns -1 (and computes nothing) unless 1 <= K <= 64 and V >= 1. Outputs: accept_len [B], out_tokens [B, K+1] (-1 padded),
 * diag [B, K, 4] = (p_target(t), p_draft(t), Z, r) (nullable), accept_margin [B, K] (nullable),
 * cdf_margin [B] (nullable). mutation: see spec_oracle_sample_one. Returns 0. */
int spec_oracle_verify(int dtype, const void* target, const void* draft, const int32_t* tokens,
                       const uint64_t* seeds, const int32_t* seq_index, int B, int K, int V,
                       double T, int mutation, int32_t* accept_len, int32_t* out_tokens,
                       double* diag, double* accept_margin, double* cdf_margin, int nthreads)
{
    if (K < 1 || K > ORACLE_MAX_K || V < 1 || B < 0) return -1;
    int nt = nthreads_or_default(nthreads);
#pragma omp parallel for schedule(dynamic) num_threads(nt)
    for (int b = 0; b < B; b++) {
        double* x = (double*)malloc(sizeof(double) * (size_t)V);
        double* scratch = (double*)malloc(sizeof(double) * (size_t)V);
        double* store = (double*)malloc(sizeof(double) * (size_t)V * (size_t)(2 * K + 1));
        double* hrows[ORACLE_MAX_K];
        double* drows[ORACLE_MAX_K];
        for (int j = 0; j < K; j++) {
            hrows[j] = store + (size_t)j * V;
            drows[j] = store + (size_t)(K + j) * V;
            load_row(dtype, target, (size_t)b * (K + 1) + j, V, x);
            spec_oracle_softmax(x, V, T, hrows[j]);
            load_row(dtype, draft, (size_t)b * K + j, V, x);
            spec_oracle_softmax(x, V, T, drows[j]);
        }
        double* bonus = store + (size_t)(2 * K) * V;
        load_row(dtype, target, (size_t)b * (K + 1) + K, V, x);
        spec_oracle_softmax(x, V, T, bonus);
        uint32_t seq = seq_index ? (uint32_t)seq_index[b] : (uint32_t)b;
        chain_one(hrows, drows, bonus, K, V, tokens + (size_t)b * K, seeds[b], seq, mutation,
                  accept_len + b, out_tokens + (size_t)b * (K + 1),
                  diag ? diag + (size_t)b * K * 4 : NULL,
                  accept_margin ? accept_margin + (size_t)b * K : NULL,
                  cdf_margin ? cdf_margin + b : NULL, scratch);
        free(store);
        free(scratch);
        free(x);
    }
    return 0;
}

/* Cactus constrained acceptance over a batch ([Cactus] Key design 1-3 inside the [SpS] §9.1 chain).
 * Same layout as spec_oracle_verify plus delta >= 0, exact (0: the Taylor gamma*, 1: the root of the
 * divergence constraint) and gamma_star [B, K] (nullable). At each position the target distribution of
 * the chain is h built from the target row and the draft token; the bonus row is the plain target row.
 * diag's first entry is h(t) = gamma*. */
int spec_oracle_cactus_ex(int dtype, const void* target, const void* draft, const int32_t* tokens,
                          const uint64_t* seeds, const int32_t* seq_index, int B, int K, int V,
                          double T, double delta, int exact, int32_t* accept_len, int32_t* out_tokens,
                          double* diag, double* gamma_star, double* accept_margin,
                          double* cdf_margin, int nthreads)
{
    if (K < 1 || K > ORACLE_MAX_K || V < 1 || B < 0) return -1;
    int nt = nthreads_or_default(nthreads);
#pragma omp parallel for schedule(dynamic) num_threads(nt)
    for (int b = 0; b < B; b++) {
        double* x = (double*)malloc(sizeof(double) * (size_t)V);
        double* pt = (double*)malloc(sizeof(double) * (size_t)V);
        double* scratch = (double*)malloc(sizeof(double) * (size_t)V);
        double* store = (double*)malloc(sizeof(double) * (size_t)V * (size_t)(2 * K + 1));
        double* hrows[ORACLE_MAX_K];
        double* drows[ORACLE_MAX_K];
        for (int j = 0; j < K; j++) {
            hrows[j] = store + (size_t)j * V;
            drows[j] = store + (size_t)(K + j) * V;
            load_row(dtype, target, (size_t)b * (K + 1) + j, V, x);
            spec_oracle_softmax(x, V, T, pt);
            double g = spec_oracle_cactus_h_mode(pt, V, tokens[(size_t)b * K + j], delta, exact, hrows[j]);
            if (gamma_star) gamma_star[(size_t)b * K + j] = g;
            load_row(dtype, draft, (size_t)b * K + j, V, x);
            spec_oracle_softmax(x, V, T, drows[j]);
        }
        double* bonus = store + (size_t)(2 * K) * V;
        load_row(dtype, target, (size_t)b * (K + 1) + K, V, x);
        spec_oracle_softmax(x, V, T, bonus);
        uint32_t seq = seq_index ? (uint32_t)seq_index[b] : (uint32_t)b;
        chain_one(hrows, drows, bonus, K, V, tokens + (size_t)b * K, seeds[b], seq, 0,
                  accept_len + b, out_tokens + (size_t)b * (K + 1),
                  diag ? diag + (size_t)b * K * 4 : NULL,
                  accept_margin ? accept_margin + (size_t)b * K : NULL,
                  cdf_margin ? cdf_margin + b : NULL, scratch);
        free(store);
        free(scratch);
        free(pt);
        free(x);
    }
    return 0;
}

int spec_oracle_cactus(int dtype, const void* target, const void* draft, const int32_t* tokens,
                       const uint64_t* seeds, const int32_t* seq_index, int B, int K, int V,
                       double T, double delta, int32_t* accept_len, int32_t* out_tokens,
                       double* diag, double* gamma_star, double* accept_margin,
                       double* cdf_margin, int nthreads)
{
    return spec_oracle_cactus_ex(dtype, target, draft, tokens, seeds, seq_index, B, K, V, T, delta, 0, accept_len,
                                 out_tokens, diag, gamma_star, accept_margin, cdf_margin, nthreads);
}

/* Greedy verification: [SpS] §5.1 and the §9.1 chain with the temperature taken to 0. Both rows become
 * one-hot at their largest logit (the smallest index among equal largest logits: the pages fix no tie
 * rule), so p(t) / q(t) is 1 when the draft token t is the target's argmax and 0 otherwise, whatever the
 * uniform: accept iff t = argmax of target row j. At the first reject the residual (p - q)+ is the one-hot
 * p itself, or empty when the draft row has the same argmax, in which case the row is drawn from p; either
 * way the emitted token is the argmax of target row L. All K accepted: the argmax of target row K. The
 * draft logits and the uniforms drop out. Outputs as spec_oracle_verify's accept_len and out_tokens. */
static int argmax_row(const double* x, int V)
{
    int a = 0;
    for (int i = 1; i < V; i++)
        if (x[i] > x[a]) a = i;
    return a;
}

int spec_oracle_greedy(int dtype, const void* target, const int32_t* tokens, int B, int K, int V,
                       int32_t* accept_len, int32_t* out_tokens, int nthreads)
{
    if (K < 1 || K > ORACLE_MAX_K || V < 1 || B < 0) return -1;
    int nt = nthreads_or_default(nthreads);
#pragma omp parallel for schedule(dynamic) num_threads(nt)
    for (int b = 0; b < B; b++) {
        double* x = (double*)malloc(sizeof(double) * (size_t)V);
        int L = K;
        for (int j = 0; j <= K; j++) {
            load_row(dtype, target, (size_t)b * (K + 1) + j, V, x);
            int a = argmax_row(x, V);
            if (j < K && tokens[(size_t)b * K + j] == a) {
                out_tokens[(size_t)b * (K + 1) + j] = a;
                continue;
            }
            L = j;
            out_tokens[(size_t)b * (K + 1) + j] = a;
            break;
        }
        for (int j = L + 1; j <= K; j++) out_tokens[(size_t)b * (K + 1) + j] = -1;
        accept_len[b] = L;
        free(x);
    }
    return 0;
}

/* HedgeSpec accept-length estimate and its loss ([Hedge] Key design 2 and 3). PARITY UNPINNED against the
 * page: its estimator display (Theorem 3) and loss display are missing from the text; what survives is that
 * the estimate lies in [1, K + 1], that gamma_k is the probability of accepting any token at level k, and
 * that the loss measures the accept length still available up to K + 1. Reading taken: the expected
 * number of tokens of a chain whose level k is reached and accepted with probability gamma_k given the
 * levels before it, est = 1 + sum_{k=1..K} prod_{j<=k} gamma_j, and loss = K + 1 - est. gamma [N, B, K],
 * est and loss [N, B] (loss nullable). */
void spec_oracle_accept_length(const double* gamma, int N, int B, int K, double* est, double* loss)
{
    for (long long r = 0; r < (long long)N * B; r++) {
        double run = 1.0, total = 1.0;
        for (int k = 0; k < K; k++) {
            run *= gamma[r * K + k];
            total += run;
        }
        est[r] = total;
        if (loss) loss[r] = (double)(K + 1) - total;
    }
}

/* NormalHedge (Chaudhuri, Freund, Hsu, "A parameter-free hedging algorithm", NIPS 2009), the learner
 * [Hedge] names for drafter selection (the page states no update rule). One round: the learner played
 * weights p over N experts and saw losses l; its regret to expert i grows by (sum_j p_j l_j) - l_i. The next
 * weights are p_i proportional to ([R_i]+ / c) exp([R_i]+^2 / (2 c)), where c > 0 solves
 * (1/N) sum_i exp([R_i]+^2 / (2 c)) = e; when no regret is positive the weights are uniform. c is found by
 * bisection on log c, the mean taken as a log-sum-exp so that no term overflows. R, p: in/out [N]. */
static double nh_log_mean(const double* Rp, int N, double c)
{
    double mx = -INFINITY;
    for (int i = 0; i < N; i++) {
        double a = Rp[i] * Rp[i] / (2.0 * c);
        if (a > mx) mx = a;
    }
    double s = 0.0;
    for (int i = 0; i < N; i++) s += exp(Rp[i] * Rp[i] / (2.0 * c) - mx);
    return mx + log(s / N);
}

double spec_oracle_normalhedge_scale(const double* R, int N)
{
    double Rp[64];
    int any = 0;
    for (int i = 0; i < N; i++) {
        Rp[i] = R[i] > 0.0 ? R[i] : 0.0;
        if (Rp[i] > 0.0) any = 1;
    }
    if (!any) return 0.0;
    /* log-mean is decreasing in c: above 1 for small c, towards 0 for large c */
    double lo = -200.0, hi = 200.0;   /* log c */
    for (int it = 0; it < 400; it++) {
        double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi) break;
        if (nh_log_mean(Rp, N, exp(mid)) > 1.0) lo = mid;
        else hi = mid;
    }
    return exp(0.5 * (lo + hi));
}

int spec_oracle_normalhedge(double* R, const double* loss, double* p, int N)
{
    if (N < 1 || N > 64) return -1;
    double lp = 0.0;
    for (int i = 0; i < N; i++) lp += p[i] * loss[i];
    for (int i = 0; i < N; i++) R[i] += lp - loss[i];
    double c = spec_oracle_normalhedge_scale(R, N);
    if (c == 0.0) {
        for (int i = 0; i < N; i++) p[i] = 1.0 / N;
        return 0;
    }
    /* weights in log space relative to the largest, then normalised */
    double lw[64], mx = -INFINITY;
    for (int i = 0; i < N; i++) {
        double r = R[i] > 0.0 ? R[i] : 0.0;
        lw[i] = r > 0.0 ? log(r / c) + r * r / (2.0 * c) : -INFINITY;
        if (lw[i] > mx) mx = lw[i];
    }
    double s = 0.0;
    for (int i = 0; i < N; i++) {
        p[i] = lw[i] == -INFINITY ? 0.0 : exp(lw[i] - mx);
        s += p[i];
    }
    for (int i = 0; i < N; i++) p[i] /= s;
    return 0;
}

/* NormalHedge under delayed, censored feedback ([Hedge] Key design 3). The notes say that the accepted tokens
 * of a round are revealed as one block when the round ends, that the counterfactual feedback is censored
 * unless the selected drafter fills the chunk, that the loss is either 1 - gamma (the acceptance
 * probability) or the accept length still available up to K + 1, that the delay is at most 2K, and that in
 * practice the learner keeps a queue of feedback and keeps applying the next available one (the stochastic-
 * setting reduction of Joulani, Gyorgy, Szepesvari, "Online learning under delayed feedback", ICML 2013).
 * They give no pseudo-code; the reading taken here, one learner per sequence:
 *  - round t reports gamma_t [N, K] (all drafters, all levels) and the accepted length L_t of the selected
 *    drafter. Levels j < min(L_t + 1, K) have a fully verified context and are revealed, in level order, as
 *    the next feedback items of the sequence; the levels after them are censored and never used;
 *  - objective 0 (acceptance probability): item n's loss is 1 - gamma of item n, available at once;
 *  - objective 1 (accept length): item n's loss is K + 1 minus the accept-length estimate over the window of
 *    items n .. n + K - 1 (spec_oracle_accept_length's reading), available once item n + K - 1 has arrived,
 *    so an item waits for at most the K - 1 items after it and the pending items never exceed 2K - 1;
 *  - after each round every newly available loss is applied, oldest item first, as one NormalHedge round
 *    (spec_oracle_normalhedge). Items whose window never completes are never applied.
 * gamma [T][N][B][K], accept_len [T][B] in [0, K]; outputs after each round: weights [T][B][N] (the
 * distribution for the next round) and applied [T][B] (NormalHedge rounds so far). Returns 0, or -1 for bad
 * sizes or an accepted length outside [0, K]. */
int spec_oracle_hedge_feedback(const double* gamma, const int32_t* accept_len, int T, int N, int B, int K,
                               int objective, double* weights, int32_t* applied)
{
    if (T < 0 || N < 1 || N > 64 || B < 0 || K < 1 || K > 64 || (objective != 0 && objective != 1)) return -1;
    for (long long i = 0; i < (long long)T * B; i++)
        if (accept_len[i] < 0 || accept_len[i] > K) return -1;
    double* items = (double*)malloc(sizeof(double) * ((size_t)T * K + 1) * N);
    if (!items) return -1;
    for (int b = 0; b < B; b++) {
        double R[64], p[64], loss[64];
        for (int i = 0; i < N; i++) {
            R[i] = 0.0;
            p[i] = 1.0 / N;
        }
        long long n_items = 0, next = 0, done = 0;
        for (int t = 0; t < T; t++) {
            const int L = accept_len[(size_t)t * B + b];
            const int valid = L + 1 < K ? L + 1 : K;
            for (int j = 0; j < valid; j++, n_items++)
                for (int i = 0; i < N; i++)
                    items[n_items * N + i] = gamma[(((size_t)t * N + i) * B + b) * K + j];
            while (objective == 0 ? next < n_items : next + K - 1 < n_items) {
                for (int i = 0; i < N; i++) {
                    if (objective == 0) {
                        loss[i] = 1.0 - items[next * N + i];
                    } else {
                        double run = 1.0, total = 1.0;
                        for (int k = 0; k < K; k++) {
                            run *= items[(next + k) * N + i];
                            total += run;
                        }
                        loss[i] = (double)(K + 1) - total;
                    }
                }
                spec_oracle_normalhedge(R, loss, p, N);
                next++;
                done++;
            }
            for (int i = 0; i < N; i++) weights[((size_t)t * B + b) * N + i] = p[i];
            applied[(size_t)t * B + b] = (int32_t)done;
        }
    }
    free(items);
    return 0;
}

/* Standardised sampling ([SpS] §8 Q4: temperature, top-k and top-p are folded into p and q before the
 * ratio, the same transforms for the target and the draft row). For one row of logits x at temperature T:
 * top-k (0 < k < V) keeps the logits at or above the k-th largest; then top-p (0 < top_p < 1) keeps, of what
 * is left, the logits at or above the value v* at which the mass of the renormalised distribution, summed
 * from the largest logit down, first reaches top_p. Readings (the pages give neither rule): ties at either
 * threshold are all kept (the kept set depends on values only), top-k comes before top-p, and the kept
 * logits keep their values while the others become -inf. Writes the filtered row to out and returns the
 * threshold (-inf when nothing is filtered); *margin = the distance from top_p of the partial sums just
 * before and after the block of values that crosses it (in the renormalised mass; +inf without top-p),
 * the near-tie measure of the top-p decision. */
static int cmp_desc(const void* a, const void* b)
{
    double x = *(const double*)a, y = *(const double*)b;
    return (x < y) - (x > y);
}

double spec_oracle_filter_row(const double* x, int V, double T, int top_k, double top_p, double* out,
                              double* margin, double* scratch)
{
    double thr = -INFINITY;
    if (margin) *margin = INFINITY;
    for (int i = 0; i < V; i++) scratch[i] = x[i];
    qsort(scratch, (size_t)V, sizeof(double), cmp_desc);
    if (top_k > 0 && top_k < V) thr = scratch[top_k - 1];
    if (top_p > 0.0 && top_p < 1.0) {
        double m = scratch[0];
        double total = 0.0;
        for (int i = 0; i < V && scratch[i] >= thr; i++) total += exp((scratch[i] - m) / T);
        double run = 0.0;
        int i = 0;
        while (i < V && scratch[i] >= thr) {
            /* every copy of a value enters together */
            double v = scratch[i], block = 0.0;
            int j = i;
            while (j < V && scratch[j] == v) { block += exp((v - m) / T); j++; }
            double before = run / total;
            run += block;
            double after = run / total;
            if (after >= top_p) {   /* the crossing block: its distances from top_p are the decision's margin */
                if (margin) *margin = fmin(fabs(before - top_p), fabs(after - top_p));
                thr = v > thr ? v : thr;
                break;
            }
            i = j;
        }
    }
    for (int i = 0; i < V; i++) out[i] = x[i] >= thr ? x[i] : -INFINITY;
    return thr;
}

/* spec_oracle_verify on the standardised rows: every target and draft row filtered by
 * spec_oracle_filter_row (same T, top_k, top_p), then the ordinary chain. thr: nullable [B*(K+1) + B*K]
 * thresholds (target rows, then draft rows); pmargin: nullable, the same layout, the top-p margins. */
int spec_oracle_verify_filtered(int dtype, const void* target, const void* draft, const int32_t* tokens,
                                const uint64_t* seeds, int B, int K, int V, double T, int top_k, double top_p,
                                int32_t* accept_len, int32_t* out_tokens, double* diag, double* accept_margin,
                                double* cdf_margin, double* thr, double* pmargin)
{
    if (K < 1 || K > ORACLE_MAX_K || V < 1 || B < 0) return -1;
    double* x = (double*)malloc(sizeof(double) * (size_t)V);
    double* scratch = (double*)malloc(sizeof(double) * (size_t)V);
    double* y = (double*)malloc(sizeof(double) * (size_t)V);
    /* the filtered rows hold input values or -inf, so fp32 stores them exactly */
    float* ft = (float*)malloc(sizeof(float) * (size_t)B * (K + 1) * V);
    float* fd = (float*)malloc(sizeof(float) * (size_t)B * K * V);
    for (long long r = 0; r < (long long)B * (K + 1); r++) {
        load_row(dtype, target, (size_t)r, V, x);
        double mg;
        double t = spec_oracle_filter_row(x, V, T, top_k, top_p, y, &mg, scratch);
        for (int v = 0; v < V; v++) ft[r * V + v] = (float)y[v];
        if (thr) thr[r] = t;
        if (pmargin) pmargin[r] = mg;
    }
    for (long long r = 0; r < (long long)B * K; r++) {
        load_row(dtype, draft, (size_t)r, V, x);
        double mg;
        double t = spec_oracle_filter_row(x, V, T, top_k, top_p, y, &mg, scratch);
        for (int v = 0; v < V; v++) fd[r * V + v] = (float)y[v];
        if (thr) thr[(long long)B * (K + 1) + r] = t;
        if (pmargin) pmargin[(long long)B * (K + 1) + r] = mg;
    }
    int rc = spec_oracle_verify(ORACLE_FP32, ft, fd, tokens, seeds, NULL, B, K, V, T, 0, accept_len, out_tokens,
                                diag, accept_margin, cdf_margin, 0);
    free(fd);
    free(ft);
    free(y);
    free(scratch);
    free(x);
    return rc;
}

/* HedgeSpec counterfactual evaluation ([Hedge] Key design 1): for every drafter i, sequence b and
 * level j < K, gamma[i,b,j] = sum_x min(p_target(x), q_i(x)), the acceptance probability of
 * drafter i at that level ([SpS] §6.3: P(accept) = sum_x min(p, q) = 1 - TV). tv[i,b,j] =
 * 1/2 sum_x |p_target(x) - q_i(x)| is computed separately so that a test can check the identity.
 * The loss for the acceptance-probability objective is 1 - gamma ([Hedge] Key design 3); callers
 * form it from gamma.
 * target [B, K+1, V], drafters [N, B, K, V]. If selected >= 0, the chain of drafter `selected` is also
 * verified exactly as spec_oracle_verify would with draft = drafters[selected]; the verify outputs
 * may then not be NULL. */
int spec_oracle_counterfactual(int dtype, const void* target, const void* drafters, int N, int B,
                               int K, int V, double T, double* gamma, double* tv, int selected,
                               const int32_t* tokens, const uint64_t* seeds,
                               const int32_t* seq_index, int32_t* accept_len, int32_t* out_tokens,
                               double* diag, double* accept_margin, double* cdf_margin,
                               int nthreads)
{
    if (K < 1 || K > ORACLE_MAX_K || V < 1 || B < 0) return -1;
    int nt = nthreads_or_default(nthreads);
#pragma omp parallel for schedule(dynamic) num_threads(nt)
    for (int b = 0; b < B; b++) {
        double* x = (double*)malloc(sizeof(double) * (size_t)V);
        double* q = (double*)malloc(sizeof(double) * (size_t)V);
        double* scratch = (double*)malloc(sizeof(double) * (size_t)V);
        double* store = (double*)malloc(sizeof(double) * (size_t)V * (size_t)(2 * K + 1));
        double* hrows[ORACLE_MAX_K];
        double* drows[ORACLE_MAX_K];
        for (int j = 0; j < K; j++) {
            hrows[j] = store + (size_t)j * V;
            drows[j] = store + (size_t)(K + j) * V;
            load_row(dtype, target, (size_t)b * (K + 1) + j, V, x);
            spec_oracle_softmax(x, V, T, hrows[j]);
            for (int i = 0; i < N; i++) {
                size_t row = ((size_t)i * B + b) * K + j;
                load_row(dtype, drafters, row, V, x);
                spec_oracle_softmax(x, V, T, q);
                double overlap = 0.0, dist = 0.0;
                for (int v = 0; v < V; v++) {
                    double pv = hrows[j][v], qv = q[v];
                    overlap += pv < qv ? pv : qv;
                    dist += fabs(pv - qv);
                }
                size_t o = ((size_t)i * B + b) * K + j;
                if (gamma) gamma[o] = overlap;
                if (tv) tv[o] = 0.5 * dist;
                if (i == selected) memcpy(drows[j], q, sizeof(double) * (size_t)V);
            }
        }
        if (selected >= 0 && selected < N) {
            double* bonus = store + (size_t)(2 * K) * V;
            load_row(dtype, target, (size_t)b * (K + 1) + K, V, x);
            spec_oracle_softmax(x, V, T, bonus);
            uint32_t seq = seq_index ? (uint32_t)seq_index[b] : (uint32_t)b;
            chain_one(hrows, drows, bonus, K, V, tokens + (size_t)b * K, seeds[b], seq, 0,
                      accept_len + b, out_tokens + (size_t)b * (K + 1),
                      diag ? diag + (size_t)b * K * 4 : NULL,
                      accept_margin ? accept_margin + (size_t)b * K : NULL,
                      cdf_margin ? cdf_margin + b : NULL, scratch);
        }
        free(store);
        free(scratch);
        free(q);
        free(x);
    }
    return 0;
}
