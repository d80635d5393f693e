/*
 * dspark_oracle.c — plain, slow, single-threaded CPU oracle of the DSpark ragged-verification
 * hot path (confidence scheduler, front-pack, verify, compact scatter).
 *
 * TEST INFRASTRUCTURE ONLY. This is the independent reference the CUDA library is checked
 * against. Only the test suite, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header, table or helper with the CUDA library, and neither includes,
 * links or calls the other. Compile without fast-math and with -ffp-contract=off so every
 * floating-point operation below is one IEEE operation in the order written.
 *
 * Source of the method: "DSpark in SGLang: Speculative Decoding with Confidence-Driven,
 * Variable-Length Verification" (LMSYS blog as summarised by papercache.org) and the lshu.cn
 * article on DSpark in SGLang (sections 2.3 and 3.3, the min(1, p/q) accept rule). Every
 * function names the passage it follows. Readings of silent points are marked READING.
 *
 * Every function is pinned by a test against something other than itself (brute force,
 * library routines, closed forms, a chi-square law); see the header of each test module.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status bits and mode numbers of the C ABI, restated (the ABI fixes these values). */
#define OR_TIER_OVERFLOW 0x01
#define OR_PACK_CAPACITY 0x02
#define OR_BAD_WINDOW    0x04
#define OR_OUT_OVERFLOW  0x08
#define OR_BAD_COST      0x10
#define OR_BAD_ROWS      0x20
#define OR_BAD_TOKEN     0x40
#define OR_BAD_LENGTH    0x80

#define OR_STATIC     0
#define OR_COMPACT    1
#define OR_CAP_ACCEPT 2

#define OR_BF16 0
#define OR_F32  1

/* ------------------------------------------------------------------------------------------
 * Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC'11): ten rounds of two 64x64->128 multiplies with the published multipliers, a
 * Weyl-sequence key bump between rounds. READING: the pages ask for counter-based Philox
 * uniforms keyed (seed, request, position) without fixing the variant; the 4x64 variant is
 * used, keyed (seed, 0), counter (request, position, step, 0).
 * ---------------------------------------------------------------------------------------- */
static void mulhilo64(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo)
{
    unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
    *hi = (uint64_t)(p >> 64);
    *lo = (uint64_t)p;
}

void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ULL, M1 = 0xCA5A826395121157ULL;
    const uint64_t W0 = 0x9E3779B97F4A7C15ULL, W1 = 0xBB67AE8584CAA73BULL;
    uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t hi0, lo0, hi1, lo1;
        if (round > 0) { k0 += W0; k1 += W1; }
        mulhilo64(M0, x0, &hi0, &lo0);
        mulhilo64(M1, x2, &hi1, &lo1);
        uint64_t y0 = hi1 ^ x1 ^ k0;
        uint64_t y1 = lo1;
        uint64_t y2 = hi0 ^ x3 ^ k1;
        uint64_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The two uniforms of block position i of request b at decode step `step`. */
static void position_uniforms(uint64_t seed, uint64_t step, int b, int i, float* u_accept,
                              double* u_bonus)
{
    uint64_t ctr[4] = {(uint64_t)b, (uint64_t)i, step, 0};
    uint64_t key[2] = {seed, 0};
    uint64_t w[4];
    oracle_philox4x64_10(ctr, key, w);
    *u_accept = (float)(w[0] >> 40) * 0x1p-24f;   /* 24-bit uniform in [0,1), exact in fp32 */
    *u_bonus = (double)(w[1] >> 11) * 0x1p-53;    /* 53-bit uniform in [0,1), exact in fp64 */
}

/* ------------------------------------------------------------------------------------------
 * Confidence scheduler. "DSpark in SGLang", A2 method details: the confidence head scores each
 * draft token, and the product of scores along the block is its survival probability; the
 * scheduler reads the additive cost table T(bs,K) = bias + alpha(bs) + theta(M), M = bs + K
 * (cost-table profiling and modelling) and picks the budget that trades expected accepted
 * tokens against the marginal cost (quick read; cost-table section: "argmax").
 * READINGS: bs = B (every live request commits at least one token); expected committed tokens
 * = B + sum of the K largest survivals (each window counts its anchor row, w_b in [1,gamma]);
 * theta is read at M, not at the rounded tier; survivals are fixed-point keys rint(s * 2^32)
 * so every sum is an exact integer; ties in the order go to the lower request, then the lower
 * position; ties in the objective go to the smallest K.
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    uint64_t key;
    int32_t b;
    int32_t j;
} oracle_cand;

static int oracle_cand_cmp(const void* pa, const void* pb)
{
    const oracle_cand* a = (const oracle_cand*)pa;
    const oracle_cand* c = (const oracle_cand*)pb;
    if (a->key != c->key) return a->key > c->key ? -1 : 1;  /* larger survival first */
    if (a->b != c->b) return a->b < c->b ? -1 : 1;
    if (a->j != c->j) return a->j < c->j ? -1 : 1;
    return 0;
}

static float clamp_conf(float x)
{
    if (!(x > 0.0f)) return 0.0f;  /* also NaN */
    if (x > 1.0f) return 1.0f;
    return x;
}

/* Fixed-point survival keys, request-major [B, gamma-1]. */
void oracle_survival_keys(const float* conf, int B, int gamma, uint64_t* keys)
{
    const int L = gamma - 1;
    for (int b = 0; b < B; ++b) {
        float s = 1.0f;
        for (int j = 0; j < L; ++j) {
            s = s * clamp_conf(conf[(size_t)b * L + j]);
            keys[(size_t)b * L + j] = (uint64_t)llrintf(s * 4294967296.0f);
        }
    }
}

/* windows[B], k_star[1], status |= bits. obj[K] (K = 0..n) receives the objective, -inf where
 * T is not finite and positive; both diagnostics may be NULL. Returns 0, or -1 on bad sizes. */
int oracle_schedule(const float* conf, int B, int gamma, double bias, const double* alpha,
                    int alpha_len, const double* theta, int theta_len, int32_t* windows,
                    int32_t* k_star, int32_t* status, double* obj, uint64_t* sorted_keys)
{
    if (B < 0 || gamma < 1) return -1;
    const int L = gamma - 1;
    const int n = B * L;
    if (B == 0) { *k_star = 0; return 0; }
    if (alpha_len < B + 1 || theta_len < B + n + 1) return -1;

    uint64_t* keys = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(n > 0 ? n : 1));
    oracle_cand* cand = (oracle_cand*)malloc(sizeof(oracle_cand) * (size_t)(n > 0 ? n : 1));
    oracle_survival_keys(conf, B, gamma, keys);
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < L; ++j) {
            oracle_cand* c = &cand[(size_t)b * L + j];
            c->key = keys[(size_t)b * L + j];
            c->b = b;
            c->j = j;
        }
    qsort(cand, (size_t)n, sizeof(oracle_cand), oracle_cand_cmp);
    if (sorted_keys)
        for (int k = 0; k < n; ++k) sorted_keys[k] = cand[k].key;

    /* obj(K) for every K: E(K) = B*2^32 + S(K), T(K) = (bias + alpha[B]) + theta[B+K]. */
    uint64_t S = 0;
    int best_k = -1;
    double best = 0.0;
    for (int K = 0; K <= n; ++K) {
        if (K > 0) S += cand[K - 1].key;
        double T = bias + alpha[B];
        T = T + theta[B + K];
        double value = -INFINITY;
        if (T > 0.0 && T < INFINITY) {
            double E = (double)((uint64_t)B * 4294967296ULL + S);
            value = E / T;
            if (best_k < 0 || value > best) { best = value; best_k = K; }
        }
        if (obj) obj[K] = value;
    }
    int32_t st = 0;
    if (best_k < 0) { st |= OR_BAD_COST; best_k = 0; }

    for (int b = 0; b < B; ++b) windows[b] = 1;
    for (int k = 0; k < best_k; ++k) windows[cand[k].b] += 1;
    *k_star = best_k;
    if (status) *status |= st;
    free(keys);
    free(cand);
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * Front-pack. "DSpark in SGLang", A2, ragged verify over full CUDA graphs: variable windows
 * are packed to the front of one compact cu_seqlens-style buffer and only the total is
 * rounded up to the nearest captured tier; padding rows are waste (figure 2 caption).
 * ---------------------------------------------------------------------------------------- */
int oracle_pack(const int32_t* windows, const int32_t* tokens, int B, int gamma,
                const int32_t* tiers, int n_tiers, int32_t* cu, int32_t* packed_ids,
                int32_t* row_req, int32_t* row_pos, int packed_cap, int32_t* meta,
                int32_t* status)
{
    if (B < 0 || gamma < 1 || n_tiers < 1 || packed_cap < 0) return -1;
    int32_t st = 0;
    cu[0] = 0;
    for (int b = 0; b < B; ++b) {
        int w = windows[b];
        if (w < 1 || w > gamma) {
            st |= OR_BAD_WINDOW;
            w = w < 1 ? 1 : gamma;
        }
        cu[b + 1] = cu[b] + w;
    }
    const int M = cu[B];
    int tier = -1;
    for (int t = 0; t < n_tiers; ++t)
        if (tiers[t] >= M && (tier < 0 || tiers[t] < tier)) tier = tiers[t];
    if (tier < 0) { st |= OR_TIER_OVERFLOW; tier = M; }
    if (tier > packed_cap) st |= OR_PACK_CAPACITY;

    for (int b = 0; b < B; ++b) {
        int w = cu[b + 1] - cu[b];
        for (int i = 0; i < w; ++i) {
            int r = cu[b] + i;
            if (r >= packed_cap) continue;
            packed_ids[r] = tokens[(size_t)b * gamma + i];
            if (row_req) row_req[r] = b;
            if (row_pos) row_pos[r] = i;
        }
    }
    for (int r = M; r < tier && r < packed_cap; ++r) {
        packed_ids[r] = 0;
        if (row_req) row_req[r] = -1;
        if (row_pos) row_pos[r] = -1;
    }
    meta[0] = M;
    meta[1] = tier;
    if (status) *status |= st;
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * Row primitives of verify. Logits are bf16 (top 16 bits of an IEEE fp32) or fp32; every
 * value is widened exactly to double.
 * ---------------------------------------------------------------------------------------- */
static double logit_at(const void* base, int dtype, int64_t V, int64_t row, int64_t v)
{
    if (dtype == OR_BF16) {
        uint16_t h = ((const uint16_t*)base)[row * V + v];
        uint32_t bits = (uint32_t)h << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[row * V + v];
}

/* Greedy verify: the row's argmax, the lowest index among equal maxima. */
int oracle_row_argmax(const void* base, int dtype, int V, int64_t row)
{
    int best_v = 0;
    double best = logit_at(base, dtype, V, row, 0);
    for (int v = 1; v < V; ++v) {
        double x = logit_at(base, dtype, V, row, v);
        if (x > best) { best = x; best_v = v; }
    }
    return best_v;
}

/* Softmax statistics of logits/T: m = max logit, Z = sum_v exp((l_v - m) / T). */
void oracle_row_softmax_stats(const void* base, int dtype, int V, int64_t row, double T,
                              double* m_out, double* z_out)
{
    double m = logit_at(base, dtype, V, row, 0);
    for (int v = 1; v < V; ++v) {
        double x = logit_at(base, dtype, V, row, v);
        if (x > m) m = x;
    }
    double z = 0.0;
    for (int v = 0; v < V; ++v) z += exp((logit_at(base, dtype, V, row, v) - m) / T);
    *m_out = m;
    *z_out = z;
}

static double softmax_prob(const void* base, int dtype, int V, int64_t row, int v, double m,
                           double z, double T)
{
    return exp((logit_at(base, dtype, V, row, v) - m) / T) / z;
}

/* Inverse-CDF draw from the (unnormalised) weights r_v in index order: the smallest v whose
 * running sum exceeds u * R. If rounding leaves none, the last v with r_v > 0. `margin` is the
 * distance of u*R to the chosen interval's nearer end, divided by R (0 on the fallback). */
static int inverse_cdf(const double* r, int V, double u, double* margin)
{
    double R = 0.0;
    for (int v = 0; v < V; ++v) R += r[v];
    double t = u * R;
    double cum = 0.0;
    for (int v = 0; v < V; ++v) {
        double prev = cum;
        cum += r[v];
        if (cum > t) {
            double lo = t - prev, hi = cum - t;
            *margin = (lo < hi ? lo : hi) / R;
            return v;
        }
    }
    *margin = 0.0;
    for (int v = V - 1; v >= 0; --v)
        if (r[v] > 0.0) return v;
    return 0;
}

/* Bonus token. After a rejection at position i: the residual max(0, p - q) of that position
 * (standard speculative sampling; READING — the pages name the residual bonus sample but do not
 * print it). With no rejection: p of the last verified position. A residual that sums to zero
 * (p == q everywhere cannot reject, so only rounding gets here) falls back to p. */
static int draw_bonus(const void* target, const void* draft, int dtype, int V, int64_t trow,
                      int64_t drow, int residual, double mp, double zp, double mq, double zq,
                      double T, double u, double* margin, double* work)
{
    double R = 0.0;
    for (int v = 0; v < V; ++v) {
        double p = softmax_prob(target, dtype, V, trow, v, mp, zp, T);
        double r = p;
        if (residual) {
            double q = softmax_prob(draft, dtype, V, drow, v, mq, zq, T);
            r = p - q > 0.0 ? p - q : 0.0;
        }
        work[v] = r;
        R += r;
    }
    if (residual && !(R > 0.0))
        return draw_bonus(target, draft, dtype, V, trow, drow, 0, mp, zp, mq, zq, T, u, margin,
                          work);
    return inverse_cdf(work, V, u, margin);
}

/* ------------------------------------------------------------------------------------------
 * Verify. "DSpark in SGLang", A2, verify-mode design: static verifies the whole block each
 * step; compact verifies only the scheduled window; cap-accept verifies the whole block,
 * commits only up to the window (output identical to compact) and exposes what full
 * verification would have accepted. Greedy: a draft survives iff it equals the target's argmax,
 * the accept length ends at the first divergence (lshu.cn article, 1.2). Stochastic: accept with
 * probability min(1, p(x)/q(x)) (lshu.cn article, 2.3 and 3.3).
 * READINGS: accept length L counts the committed tokens, the accepted drafts plus the one
 * target token after them, so 1 <= L <= w_b; in cap-accept the committed tokens and the bonus
 * depend on positions i < w_b only, which makes them identical to compact by construction.
 *
 * Diagnostics (each may be NULL): diag_ratio[b, i] = float(p/q) of the accept test of draft
 * i+1 (+inf when q(d) = 0), diag_u[b, i] its uniform, NaN where no test ran; diag_margin[b] =
 * inverse-CDF margin of the stochastic bonus draw (NaN in greedy mode).
 * ---------------------------------------------------------------------------------------- */
int oracle_verify(int mode, int stochastic, const void* target, int target_rows,
                  const void* draft, int dtype, int V, const int32_t* cu, const int32_t* windows,
                  const int32_t* tokens, int B, int gamma, float temperature, uint64_t seed,
                  uint64_t step, int32_t* accept_len, int32_t* committed, int32_t* ceiling,
                  float* row_prob, int32_t* status, float* diag_ratio, float* diag_u,
                  double* diag_margin)
{
    if (B < 0 || gamma < 1 || V < 1 || target_rows < 0) return -1;
    if (mode != OR_STATIC && mode != OR_COMPACT && mode != OR_CAP_ACCEPT) return -1;
    if (dtype != OR_BF16 && dtype != OR_F32) return -1;
    if (stochastic && !(temperature > 0.0f)) return -1;
    const int L = gamma - 1;
    const double T = (double)temperature;
    int32_t st = 0;

    if (row_prob)
        for (int64_t r = 0; r < (int64_t)target_rows * 2; ++r) row_prob[r] = -1.0f;
    if (diag_ratio)
        for (int64_t k = 0; k < (int64_t)B * L; ++k) diag_ratio[k] = NAN;
    if (diag_u)
        for (int64_t k = 0; k < (int64_t)B * L; ++k) diag_u[k] = NAN;
    if (diag_margin)
        for (int b = 0; b < B; ++b) diag_margin[b] = NAN;

    int* g = (int*)malloc(sizeof(int) * (size_t)gamma);
    int* acc = (int*)malloc(sizeof(int) * (size_t)gamma);
    double* mp = (double*)malloc(sizeof(double) * (size_t)gamma);
    double* zp = (double*)malloc(sizeof(double) * (size_t)gamma);
    double* mq = (double*)malloc(sizeof(double) * (size_t)gamma);
    double* zq = (double*)malloc(sizeof(double) * (size_t)gamma);
    double* work = stochastic ? (double*)malloc(sizeof(double) * (size_t)V) : NULL;

    /* The rows a call verifies: [0, N) with N = cu[B], the packed total M (COMPACT: the windows
       are packed to the front of the buffer and nothing past M is read, "DSpark in SGLang", A2
       ragged verify over full CUDA graphs, figure 2), or B * gamma (the block); never more than
       the buffer holds, nor more than B * gamma. */
    int64_t n_rows = (mode == OR_COMPACT) ? (int64_t)cu[B] : (int64_t)B * gamma;
    if (n_rows < 0) n_rows = 0;
    if (n_rows > (int64_t)target_rows) n_rows = target_rows;
    if (n_rows > (int64_t)B * gamma) n_rows = (int64_t)B * gamma;

    for (int b = 0; b < B; ++b) {
        int w = gamma;
        if (mode != OR_STATIC) {
            w = windows[b];
            if (w < 1 || w > gamma) { st |= OR_BAD_WINDOW; w = w < 1 ? 1 : gamma; }
        }
        const int nrows = (mode == OR_COMPACT) ? w : gamma;
        const int64_t base = (mode == OR_COMPACT) ? (int64_t)cu[b] : (int64_t)b * gamma;
        /* COMPACT: each packed row is one request's (the last b with cu[b] <= row), so the
           rows that carry this request's accept tests, cu[b] .. cu[b] + w - 2, must lie before
           the next request's first row; its last row may be shared */
        const int shared = mode == OR_COMPACT && b + 1 < B && nrows >= 2 &&
                           (int64_t)cu[b + 1] < base + nrows - 1;
        int32_t* out = committed + (size_t)b * gamma;
        for (int k = 0; k < gamma; ++k) out[k] = -1;
        if (base < 0 || base + nrows > n_rows || shared) {
            st |= OR_BAD_ROWS;
            accept_len[b] = 0;
            if (ceiling) ceiling[b] = (mode == OR_COMPACT) ? -1 : 0;
            continue;
        }
        /* decisions over the positions this mode verifies */
        const int ndec = nrows - 1;
        for (int i = 0; i < ndec; ++i) {
            const int d = tokens[(size_t)b * gamma + i + 1];
            const int64_t row = base + i;
            if (!stochastic) {
                g[i] = oracle_row_argmax(target, dtype, V, row);
                if (d < 0 || d >= V) { st |= OR_BAD_TOKEN; acc[i] = 0; continue; }
                acc[i] = (d == g[i]);
                continue;
            }
            oracle_row_softmax_stats(target, dtype, V, row, T, &mp[i], &zp[i]);
            const int64_t drow = (int64_t)b * L + i;
            oracle_row_softmax_stats(draft, dtype, V, drow, T, &mq[i], &zq[i]);
            if (d < 0 || d >= V) { st |= OR_BAD_TOKEN; acc[i] = 0; continue; }
            const double p = softmax_prob(target, dtype, V, row, d, mp[i], zp[i], T);
            const double q = softmax_prob(draft, dtype, V, drow, d, mq[i], zq[i], T);
            float u;
            double ub;
            position_uniforms(seed, step, b, i, &u, &ub);
            float ratio = INFINITY;
            if (q == 0.0) {
                acc[i] = 1;
            } else {
                ratio = (float)(p / q);
                acc[i] = (u < ratio);
            }
            if (row_prob) {
                row_prob[row * 2 + 0] = (float)p;
                row_prob[row * 2 + 1] = (float)q;
            }
            if (diag_ratio) diag_ratio[(size_t)b * L + i] = ratio;
            if (diag_u) diag_u[(size_t)b * L + i] = u;
        }
        /* the last verified row: greedy argmax, or p's statistics for a bonus drawn there */
        if (!stochastic)
            g[nrows - 1] = oracle_row_argmax(target, dtype, V, base + nrows - 1);
        else
            oracle_row_softmax_stats(target, dtype, V, base + nrows - 1, T, &mp[nrows - 1],
                                     &zp[nrows - 1]);

        /* committed: the window's own walk (identical in compact and cap-accept) */
        int Lc = 1;
        while (Lc - 1 < w - 1 && acc[Lc - 1]) ++Lc;
        int Lf = 1;
        while (Lf - 1 < ndec && acc[Lf - 1]) ++Lf;

        if (!stochastic) {
            for (int k = 0; k < Lc; ++k) out[k] = g[k];
        } else {
            const int pos = Lc - 1;            /* where the bonus is drawn */
            const int rejected = (pos < w - 1); /* a rejection ended the walk */
            /* mp/zp of row `pos` exist in every mode: pos < ndec was a decision row, and
             * pos == nrows - 1 was filled just above. */
            float u_unused;
            double ub;
            position_uniforms(seed, step, b, pos, &u_unused, &ub);
            double margin = 0.0;
            const int bonus = draw_bonus(target, draft, dtype, V, base + pos,
                                         (int64_t)b * L + pos, rejected, mp[pos], zp[pos],
                                         rejected ? mq[pos] : 0.0, rejected ? zq[pos] : 1.0, T,
                                         ub, &margin, work);
            for (int k = 0; k < Lc - 1; ++k) out[k] = tokens[(size_t)b * gamma + k + 1];
            out[Lc - 1] = bonus;
            if (diag_margin) diag_margin[b] = margin;
        }
        accept_len[b] = Lc;
        if (ceiling) ceiling[b] = (mode == OR_COMPACT) ? -1 : Lf;
    }
    if (status) *status |= st;
    free(g); free(acc); free(mp); free(zp); free(mq); free(zq); free(work);
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * Compact scatter. "DSpark in SGLang", A2, performance and zero-overhead scheduling: a fused
 * kernel writes the accepted tokens back into per-request state.
 * ---------------------------------------------------------------------------------------- */
int oracle_scatter(const int32_t* committed, const int32_t* accept_len, int B, int gamma,
                   int32_t* out_tokens, int32_t* out_len, int out_cap, int32_t* status)
{
    if (B < 0 || gamma < 1 || out_cap < 0) return -1;
    int32_t st = 0;
    for (int b = 0; b < B; ++b) {
        int L = accept_len[b];
        int n = out_len[b];
        if (L < 0 || L > gamma) { st |= OR_BAD_LENGTH; L = L < 0 ? 0 : gamma; }
        if (n < 0 || n > out_cap) { st |= OR_BAD_LENGTH; n = n < 0 ? 0 : out_cap; }
        for (int i = 0; i < L; ++i) {
            if (n + i < out_cap)
                out_tokens[(size_t)b * out_cap + n + i] = committed[(size_t)b * gamma + i];
            else
                st |= OR_OUT_OVERFLOW;
        }
        out_len[b] = (n + L < out_cap) ? n + L : out_cap;
    }
    if (status) *status |= st;
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * Observability counters. "DSpark in SGLang", A2 observability: per-request confidence and
 * calibration metrics (ECE) are reported for post-hoc analysis, and cap-accept exposes the
 * acceptance ceiling that truncation hides (utilisation = committed over ceiling).
 * READING: a draft's outcome is observed up to and including the first rejection of the full
 * block (the ceiling); later drafts are censored. Confidence sums are kept in 2^-32 fixed point
 * so every counter is an exact integer.
 * hist [n_bins][3] = (count, sum of rint(x * 2^32), accepted); util [2] = (committed, ceiling).
 * ---------------------------------------------------------------------------------------- */
int oracle_observe(const float* conf, const int32_t* accept_len, const int32_t* ceiling_len,
                   int B, int gamma, int n_bins, uint64_t* hist, uint64_t* util, int32_t* status)
{
    if (B < 0 || gamma < 1 || n_bins < 1) return -1;
    const int L = gamma - 1;
    int32_t st = 0;
    for (int b = 0; b < B; ++b) {
        int c = ceiling_len[b];
        if (c < 1 || c > gamma) { st |= OR_BAD_LENGTH; c = c < 1 ? 1 : gamma; }
        int a = accept_len[b];
        if (a < 0 || a > gamma) { st |= OR_BAD_LENGTH; a = a < 0 ? 0 : gamma; }
        util[0] += (uint64_t)a;
        util[1] += (uint64_t)c;
        for (int j = 0; j < L && j <= c - 1; ++j) {
            const float x = clamp_conf(conf[(size_t)b * L + j]);
            int k = (int)(x * (float)n_bins);
            if (k > n_bins - 1) k = n_bins - 1;
            const uint64_t fx = x >= 1.0f ? (1ULL << 32) : (uint64_t)llrintf(x * 4294967296.0f);
            hist[3 * k + 0] += 1;
            hist[3 * k + 1] += fx;
            if (j < c - 1) hist[3 * k + 2] += 1;
        }
    }
    if (status) *status |= st;
    return 0;
}
