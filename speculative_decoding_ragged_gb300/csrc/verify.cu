// verify.cu — verify over the target logits and reduction to per-request accept lengths.
//
// Greedy: a draft survives iff it equals the target row's argmax; the accept length ends at
// the first divergence (lshu.cn DSpark article, 1.2). Stochastic: accept with probability
// min(1, p(d)/q(d)) (lshu.cn article, 2.3 and 3.3) with the residual bonus sample of standard
// speculative sampling. Modes: "DSpark in SGLang" (LMSYS blog summary), A2 verify-mode design
// (static, compact, cap-accept: full-block verify that commits exactly what compact commits).
//
// Kernels of one call:
// 1. the streaming kernel (verify_stream.cu): one partial per (row, chunk) unit;
// 2. greedy: verify_finalize_kernel — a CTA per request, or per two or four requests when one
//    per request would occupy every SM (the next step's scheduler, one CTA holding a whole SM's
//    registers, then starts on a free SM while this kernel works): combines the chunk partials
//    of each request's rows, tests each draft against its row's argmax, walks to the first
//    rejection, writes accept_len / committed / ceiling (and, fused, appends the committed
//    tokens to the request's history);
//    stochastic: bonus_final_kernel — spread over the grid: every CTA of a request combines its
//    rows' partials and runs the accept tests (Philox4x64-10 uniforms), sums the bonus row's
//    weights over its tiles, and the last CTA of the request draws the bonus token.
#include <math.h>

#include "verify_common.cuh"

namespace dspark {
namespace {

// Greedy finaliser CTA size: 256 threads for large batches; 1024 for small ones, where every
// row's partials are combined at once (a warp per row).
constexpr int kFinalThreadsLarge = 256;
constexpr int kFinalThreadsSmall = 1024;
constexpr int kFinalSmallBatch = 64;
constexpr int kTileThreads = 256;
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kPickThreads = kTileThreads;
constexpr int kPickKeep = 4;              // tile sums a pick thread keeps in registers
constexpr int kMaxVocabStochastic = 1 << 20;

// ---- Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11), device side ---------------------
__device__ __forceinline__ void philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3,
                                              uint64_t k0, uint64_t k1, uint64_t out[4])
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
        const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += W0; k1 += W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// The bonus draw of one request (stochastic verify): decided by warp 0 of each bonus-kernel CTA
// of the request and handed to the CTA's warps through shared memory.
struct BonusJob {
    int64_t trow;   // target row of the bonus position
    int64_t drow;   // draft row of a residual draw; -1 for a draw from p
    float mp, izp;  // target row maximum and 1/Z
    float mq, izq;  // draft row maximum and 1/Z (residual draws)
    uint64_t ubits; // the position's bonus uniform u' = ubits * 2^-53 (53-bit integer)
    int64_t slot;   // committed[] index that receives the bonus; -1: no draw
};

struct FinalArgs {
    const void* target;
    const void* draft;
    const int32_t* cu;
    const int32_t* windows;
    const int32_t* tokens;
    const void* part_t;
    const void* part_d;
    int32_t* accept_len;
    int32_t* committed;
    int32_t* ceiling;
    float* row_prob;
    int32_t* status;
    float* tiles;     // [B][n_tiles][2]: residual and p weight sums per 256-token tile
    unsigned* done;   // [B]: tile CTAs finished per request (zeroed by the streaming kernel)
    WsHead* head;     // the workspace head, left ready for the next call
    int32_t* out_tokens;   // fused compact scatter (nullptr: none)
    int32_t* out_len;
    int out_cap;
    uint64_t seed, step;
    int mode, V, nc, vec, B, gamma, target_rows, n_tiles;
    int64_t rows_max;
    float s;          // log2(e) / temperature
};

// Eight consecutive logits [v0, v0+8) of a row as fp32; positions >= V read as -inf.
template <int DT>
__device__ __forceinline__ void load8(const char* row, int v0, int V, int vec, float (&x)[8])
{
    if (vec && v0 + 8 <= V) {
        const uint4* q = reinterpret_cast<const uint4*>(row + static_cast<int64_t>(v0) * (DT == DSPARK_BF16 ? 2 : 4));
        if (DT == DSPARK_BF16) {
            const uint4 u = __ldg(q);
            x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
            x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
        } else {
            const uint4 a = __ldg(q), b = __ldg(q + 1);
            x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
            x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
            x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
            x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = (v0 + e < V) ? load_logit<DT>(row, v0 + e) : -INFINITY;
    }
}

// A token's probability under a row with maximum m and 1/Z = iz: exp2((x - m) * s) * iz, with
// explicitly rounded operations so that every kernel computing it gets the same bits (the
// tile sums and the in-tile walk must agree).
__device__ __forceinline__ float token_prob(float x, float m, float iz, float s)
{
    return __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(x, m), s)), iz);
}

// A non-negative probability mass (at most about 2) as 2^-52 fixed point, from the float's
// exponent and mantissa with integer shifts (64-bit conversions use the scarce FP64 path):
// exact for x >= 2^-28, truncated below that; zero and subnormals give 0.
__device__ __forceinline__ uint64_t to_fixed(float x)
{
    const uint32_t b = __float_as_uint(x);
    const int e = static_cast<int>(b >> 23);          // biased exponent (x >= 0)
    if (e == 0) return 0;
    const uint64_t m = static_cast<uint64_t>((b & 0x7FFFFFu) | 0x800000u);
    const int sh = e - 98;                            // x * 2^52 = m * 2^(e - 127 - 23 + 52)
    return sh >= 0 ? (m << sh) : (sh > -64 ? (m >> -sh) : 0ull);
}

// Bonus weights of 8 consecutive tokens from their logits: p_v (residual == 0) or
// max(0, p_v - q_v); tokens at or past V weigh 0.
template <int DT>
__device__ __forceinline__ void bonus_weights_of(const float (&xp)[8], const float (&xq)[8], int v0,
                                                 int V, bool residual, float mp, float izp,
                                                 float mq, float izq, float s, float (&w)[8])
{
    if (residual) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float p = (v0 + e < V) ? token_prob(xp[e], mp, izp, s) : 0.0f;
            const float q = (v0 + e < V) ? token_prob(xq[e], mq, izq, s) : 0.0f;
            w[e] = fmaxf(__fsub_rn(p, q), 0.0f);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            w[e] = (v0 + e < V) ? token_prob(xp[e], mp, izp, s) : 0.0f;
    }
}

__device__ __forceinline__ float sum8(const float (&w)[8])
{
    return ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
}

// Combined softmax statistics of one row from its nc chunk partials, by one warp: each lane
// folds chunks lane, lane+32, ... in order (eight loads in flight at a time) with an online
// rescale, then the lanes combine over a fixed shuffle tree — deterministic for a given nc.
__device__ __forceinline__ void combine_soft(const SoftPart* parts, int nc, float s, int lane,
                                             float& m_out, float& z_out)
{
    float m = -INFINITY, z = 0.0f;
    for (int c0 = lane; c0 < nc; c0 += 32 * 8) {
        SoftPart p[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int c = c0 + 32 * k;
            if (c < nc) p[k] = parts[c];
            else { p[k].m = -INFINITY; p[k].z = 0.0f; }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (p[k].m == -INFINITY) continue;
            if (p[k].m > m) {
                z *= ex2_approx((m - p[k].m) * s);
                m = p[k].m;
            }
            z += p[k].z * ex2_approx((p[k].m - m) * s);
        }
    }
    float M = m;
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float zz = m != -INFINITY ? z * ex2_approx((m - M) * s) : 0.0f;
    for (int off = 16; off > 0; off >>= 1) zz += __shfl_xor_sync(0xffffffffu, zz, off);
    m_out = M;
    z_out = zz;
}

// Combined argmax of one row from its nc chunk partials (exact; eight loads in flight).
__device__ __forceinline__ int combine_arg(const ArgPart* parts, int nc, int lane)
{
    float v = -INFINITY;
    int idx = 0x7FFFFFFF;
    for (int c0 = lane; c0 < nc; c0 += 32 * 8) {
        ArgPart p[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int c = c0 + 32 * k;
            if (c < nc) p[k] = parts[c];
            else { p[k].v = -INFINITY; p[k].idx = 0x7FFFFFFF; }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) arg_merge(v, idx, p[k].v, p[k].idx);
    }
    for (int off = 16; off > 0; off >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
        const int i2 = __shfl_xor_sync(0xffffffffu, idx, off);
        arg_merge(v, idx, v2, i2);
    }
    return idx == 0x7FFFFFFF ? 0 : idx;   // a row of -inf only: index 0
}

// Softmax statistics (m, Z) of a request's rows j = first, first + step, ... < nrows + ndec:
// target rows j < nrows (partials at part_t + (base + j) * nc), then draft rows (part_d +
// (base + j - nrows) * nc). RB rows at a time with every partial load of the batch in flight
// (CPL loads per lane and row, nc <= 32 * CPL); each row folds exactly as combine_soft does
// (lane-strided, in chunk order, then the fixed shuffle tree), so every CTA that combines a
// row gets the same bits. Lane 0 stores the results.
template <int RB, int CPL>
__device__ __forceinline__ void combine_soft_rows(const FinalArgs& A, int64_t base, int nrows,
                                                  int ndec, int first, int step, int lane,
                                                  float* m_t, float* z_t, float* m_d, float* z_d)
{
    const int n = nrows + ndec;
    for (int j0 = first; j0 < n; j0 += step * RB) {
        SoftPart p[RB][CPL];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int j = j0 + r * step;
            const SoftPart* parts =
                j < nrows ? static_cast<const SoftPart*>(A.part_t) + (base + j) * A.nc
                          : static_cast<const SoftPart*>(A.part_d) + (base + j - nrows) * A.nc;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int k = lane + 32 * c;
                if (j < n && k < A.nc) {
                    const float2 v = __ldcg(reinterpret_cast<const float2*>(parts + k));
                    p[r][c].m = v.x;
                    p[r][c].z = v.y;
                } else {
                    p[r][c].m = -INFINITY;
                    p[r][c].z = 0.0f;
                }
            }
        }
        // the batch's rows side by side, so that their shuffle trees overlap (each row's own
        // operations keep their order: the same bits as one row at a time)
        float m[RB], z[RB], M[RB], zz[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            m[r] = -INFINITY;
            z[r] = 0.0f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                if (p[r][c].m == -INFINITY) continue;
                if (p[r][c].m > m[r]) {
                    z[r] *= ex2_approx((m[r] - p[r][c].m) * A.s);
                    m[r] = p[r][c].m;
                }
                z[r] += p[r][c].z * ex2_approx((p[r][c].m - m[r]) * A.s);
            }
            M[r] = m[r];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int r = 0; r < RB; ++r) M[r] = fmaxf(M[r], __shfl_xor_sync(0xffffffffu, M[r], off));
#pragma unroll
        for (int r = 0; r < RB; ++r)
            zz[r] = m[r] != -INFINITY ? z[r] * ex2_approx((m[r] - M[r]) * A.s) : 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int r = 0; r < RB; ++r) zz[r] += __shfl_xor_sync(0xffffffffu, zz[r], off);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const int j = j0 + r * step;
                if (j >= n) break;
                if (j < nrows) { m_t[j] = M[r]; z_t[j] = zz[r]; }
                else { m_d[j - nrows] = M[r]; z_d[j - nrows] = zz[r]; }
            }
        }
    }
}

__device__ __forceinline__ void combine_request_rows(const FinalArgs& A, int64_t base, int nrows,
                                                     int ndec, int warp, int warps, int lane,
                                                     float* m_t, float* z_t, float* m_d,
                                                     float* z_d)
{
    // batches of rows as wide as the warps usually hold: few chunks per row come with large
    // batches (B*gamma > 128 rows), whose requests give a warp two rows at gamma = 8; 33-64
    // chunks come with at most 64 rows (batch-1 decoding: four rows per warp at gamma = 16).
    // Shuffle trees of absent rows would only take issue slots, and each variant adds code
    // that a call from cold caches must fetch.
    if (A.nc <= 32) {
        combine_soft_rows<2, 1>(A, base, nrows, ndec, warp, warps, lane, m_t, z_t, m_d, z_d);
    } else if (A.nc <= 64) {
        combine_soft_rows<4, 2>(A, base, nrows, ndec, warp, warps, lane, m_t, z_t, m_d, z_d);
    } else if (A.nc <= 128) {
        combine_soft_rows<2, 4>(A, base, nrows, ndec, warp, warps, lane, m_t, z_t, m_d, z_d);
    } else {                                          // very wide rows: one at a time
        for (int j = warp; j < nrows + ndec; j += warps) {
            const SoftPart* parts =
                j < nrows ? static_cast<const SoftPart*>(A.part_t) + (base + j) * A.nc
                          : static_cast<const SoftPart*>(A.part_d) + (base + j - nrows) * A.nc;
            float m, z;
            combine_soft(parts, A.nc, A.s, lane, m, z);
            if (lane == 0) {
                if (j < nrows) { m_t[j] = m; z_t[j] = z; }
                else { m_d[j - nrows] = m; z_d[j - nrows] = z; }
            }
        }
    }
}

// Whether request b's rows can be verified: they lie in [0, n_t), the rows the streaming
// kernel covered, and (compact) the rows that carry its accept tests, base .. base + nrows - 2,
// lie before the next request's first row. Each packed row is one request's (the streaming
// kernel files a compact draft under the last b with cu[b] <= row); the last row may be shared.
__device__ __forceinline__ bool request_rows_ok(const FinalArgs& A, int b, int64_t base,
                                                int nrows, int64_t n_t)
{
    if (base < 0 || base + nrows > n_t) return false;
    return !(A.mode == DSPARK_COMPACT && b + 1 < A.B && nrows >= 2 &&
             static_cast<int64_t>(__ldg(A.cu + b + 1)) < base + nrows - 1);
}

// Outputs of a request whose rows cannot be verified (outside the verified rows, or sharing
// tested rows with the next request): nothing committed, (-1, -1) on its rows that the buffer
// does hold, BAD_ROWS (with the caller's bits), and the fused scatter checks the history
// length only. Threads tid < nthreads of one CTA; warp 0 scatters.
__device__ __forceinline__ void bad_rows_outputs(const FinalArgs& A, int b, int64_t base,
                                                 int nrows, int tid, int nthreads, int bits,
                                                 int n_hist)
{
    int32_t* out = A.committed + static_cast<int64_t>(b) * A.gamma;
    for (int k = tid; k < A.gamma; k += nthreads) out[k] = -1;
    if (A.row_prob) {
        for (int t = tid; t < nrows; t += nthreads) {
            const int64_t r = base + t;
            if (r >= 0 && r < A.target_rows) {
                A.row_prob[r * 2] = -1.0f;
                A.row_prob[r * 2 + 1] = -1.0f;
            }
        }
    }
    if (tid == 0) {
        A.accept_len[b] = 0;
        if (A.ceiling) A.ceiling[b] = (A.mode == DSPARK_COMPACT) ? -1 : 0;
        raise_status(A.status, bits | DSPARK_STATUS_BAD_ROWS);
    }
    if (A.out_tokens && tid < 32) {
        const int sb = scatter_request(b, 0, A.gamma, -1, tid, A.out_tokens, A.out_len,
                                       A.out_cap, n_hist);
        if (tid == 0) raise_status(A.status, sb);
    }
}

// Greedy verify's finaliser: FT threads per request (RPC requests per CTA) combine the argmax
// partials of the request's rows (one warp per row), then the request's warp 0 runs the accept
// tests, walks to the first rejection and writes the request's outputs (and, fused, appends its
// tokens to the history).
template <int DT, int FT, int RPC>
__global__ void __launch_bounds__(FT * RPC)
verify_finalize_kernel(FinalArgs A)
{
    constexpr int kFinalThreads = FT;                 // threads per request
    constexpr int kFinalWarps = FT / 32;
    __shared__ int g_ss[RPC][DSPARK_MAX_GAMMA];

    // RPC requests per CTA, FT threads each; a request index past B (the last CTA) idles but
    // meets the block barrier
    const int r = RPC == 1 ? 0 : static_cast<int>(threadIdx.x) / FT;
    const bool live = static_cast<int>(blockIdx.x) * RPC + r < A.B;
    const int b = live ? static_cast<int>(blockIdx.x) * RPC + r : 0;
    int* const g_s = g_ss[r];
    const int tid = static_cast<int>(threadIdx.x) - r * FT;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int gamma = A.gamma;
    const int L = gamma - 1;
    int bits = 0;
    // Inputs that no kernel of this call writes (drafts, windows, cu_seqlens) are fetched before
    // waiting for the streaming kernel: they were complete before that kernel started.
    const int d_mine = tid < L ? __ldg(A.tokens + static_cast<int64_t>(b) * gamma + tid + 1) : -1;
    int w = gamma;
    if (A.mode != DSPARK_STATIC) {
        w = __ldg(A.windows + b);
        if (w < 1 || w > gamma) {
            if (tid == 0) bits |= DSPARK_STATUS_BAD_WINDOW;
            w = w < 1 ? 1 : gamma;
        }
    }
    const int nrows = (A.mode == DSPARK_COMPACT) ? w : gamma;
    const int64_t base = (A.mode == DSPARK_COMPACT) ? static_cast<int64_t>(__ldg(A.cu + b))
                                                    : static_cast<int64_t>(b) * gamma;
    const int64_t n_t = target_row_count(A.mode, A.cu, A.B, gamma, A.target_rows, A.rows_max);
    const bool rows_ok = request_rows_ok(A, b, base, nrows, n_t);
    // the history length the fused scatter appends at: the previous call wrote it, and every
    // kernel of this library triggers its dependents only after its own wait, so all kernels
    // before the streaming kernel have completed by the time this one starts
    const int n_hist = (A.out_tokens != nullptr && warp == 0) ? A.out_len[b] : 0;
    pdl_wait_and_trigger();
    reset_ws_head(A.head);
    int32_t* out = A.committed + static_cast<int64_t>(b) * gamma;

    if (live && !rows_ok) bad_rows_outputs(A, b, base, nrows, tid, kFinalThreads, bits, n_hist);
    const bool work = live && rows_ok;
    const int ndec = nrows - 1;   // accept tests this mode runs

    // 1. per-row argmax from the chunk partials, one warp per row
    if (work) {
        for (int t = warp; t < nrows; t += kFinalWarps) {
            const int g = combine_arg(static_cast<const ArgPart*>(A.part_t) + (base + t) * A.nc,
                                      A.nc, lane);
            if (lane == 0) g_s[t] = g;
        }
    }
    __syncthreads();

    // 2. warp 0: accept tests (lane i tests draft d_{i+1} against row i's argmax), the walk to
    //    the first rejection, the outputs and the fused scatter
    if (work && warp == 0) {
        const bool tested = lane < ndec;
        const bool valid = d_mine >= 0 && d_mine < A.V;
        if (tested && !valid) bits |= DSPARK_STATUS_BAD_TOKEN;
        const bool acc = tested && valid && d_mine == g_s[lane];
        if (A.row_prob && lane < nrows) {
            A.row_prob[(base + lane) * 2] = -1.0f;
            A.row_prob[(base + lane) * 2 + 1] = -1.0f;
        }
        const unsigned rej = __ballot_sync(0xffffffffu, !acc);   // ndec <= 31: never zero
        const int lead = __ffs(rej) - 1;                          // leading accepted drafts
        const int Lc = 1 + min(lead, w - 1);
        const int Lf = 1 + lead;
        if (lane == 0) {
            A.accept_len[b] = Lc;
            if (A.ceiling) A.ceiling[b] = (A.mode == DSPARK_COMPACT) ? -1 : Lf;
        }
        if (lane < gamma) out[lane] = (lane < Lc) ? g_s[lane] : -1;
        if (A.out_tokens) {
            const int tok = lane < Lc ? g_s[lane] : -1;
            const int sb = scatter_request(b, Lc, gamma, tok, lane, A.out_tokens, A.out_len,
                                           A.out_cap, n_hist);
            if (lane == 0) bits |= sb;
        }
        const unsigned any = __ballot_sync(0xffffffffu, bits != 0);
        if (any) {
            int all = bits;
            for (int off = 16; off > 0; off >>= 1) all |= __shfl_xor_sync(0xffffffffu, all, off);
            if (lane == 0) raise_status(A.status, all);
        }
    }
}

// Stochastic bonus, step 2, by the last tile CTA of the request: a block scan of the tile sums
// (exact 2^-52 fixed-point running sums) finds the tile where the running sum first exceeds
// u' * R; one warp then walks that tile's tokens in order. The token is the smallest v whose running weight sum
// exceeds u' * R; a residual summing to zero falls back to p; rounding that leaves no crossing
// takes the last token with positive weight in the last candidate tile.
template <int DT>
__device__ void bonus_pick(const FinalArgs& A, int b, const BonusJob& job, int n_hist,
                           const int* drafts)
{
    constexpr int E = (DT == DSPARK_BF16) ? 2 : 4;
    constexpr int kWarps = kPickThreads / 32;
    __shared__ uint64_t warp_incl[kWarps];
    __shared__ int first_s;
    __shared__ int tile_s;
    __shared__ uint64_t before_s;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const float* sums = A.tiles + static_cast<int64_t>(b) * A.n_tiles * 2;
    const int n = A.n_tiles;
    const int per = (n + kPickThreads - 1) / kPickThreads;
    const int t0 = tid * per, t1 = min(t0 + per, n);
    int col = job.drow >= 0 ? 0 : 1;                  // residual sums, or p sums
    // the thread's tile sums (both columns) stay in registers when it has few tiles
    const bool kept = per <= kPickKeep;
    float2 keep[kPickKeep];
#pragma unroll
    for (int k = 0; k < kPickKeep; ++k)
        keep[k] = (kept && t0 + k < t1) ? __ldcg(reinterpret_cast<const float2*>(sums) + t0 + k)
                                        : make_float2(0.0f, 0.0f);
    // running sums are exact 2^-52 fixed point (probability masses are at most about 1, so
    // every sum stays below 2^53); FP64 throughput is scarce on this part
    uint64_t own = 0, incl = 0, R = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        own = 0;
        if (kept) {
#pragma unroll
            for (int k = 0; k < kPickKeep; ++k)
                if (t0 + k < t1) own += to_fixed(col ? keep[k].y : keep[k].x);
        } else {
            for (int t = t0; t < t1; ++t) own += to_fixed(__ldcg(sums + 2 * t + col));
        }
        incl = own;
        for (int off = 1; off < 32; off <<= 1) {
            const uint64_t v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) warp_incl[warp] = incl;
        __syncthreads();
        uint64_t offset = 0;
        R = 0;
#pragma unroll
        for (int k = 0; k < kWarps; ++k) {
            const uint64_t v = warp_incl[k];
            if (k < warp) offset += v;
            R += v;
        }
        incl += offset;
        __syncthreads();
        if (col == 1 || R > 0) break;
        col = 1;                                      // the residual vanished: draw from p
    }
    // smallest running sum above u' * R: thr = floor(u' * R) = (ubits * R) >> 53, exactly, from
    // the 128-bit product (R < 2^54, so the result fits in 64 bits)
    const uint64_t thr = (__umul64hi(job.ubits, R) << 11) | ((job.ubits * R) >> 53);
    if (tid == 0) first_s = kPickThreads;
    __syncthreads();
    if (incl > thr && t0 < t1) atomicMin(&first_s, tid);
    __syncthreads();
    if (tid == first_s) {
        uint64_t cum = incl - own;
        int tile = -1;
        if (kept) {
            uint64_t last = 0;
#pragma unroll
            for (int k = 0; k < kPickKeep; ++k) {
                if (tile < 0 && t0 + k < t1) {
                    const uint64_t v = to_fixed(col ? keep[k].y : keep[k].x);
                    if (cum + v > thr) tile = t0 + k;
                    else cum += v;
                    last = v;
                }
            }
            if (tile < 0) { tile = t1 - 1; cum -= last; }
        } else {
            for (int t = t0; t < t1; ++t) {
                const uint64_t v = to_fixed(__ldcg(sums + 2 * t + col));
                if (cum + v > thr) { tile = t; break; }
                cum += v;
            }
            if (tile < 0) { tile = t1 - 1; cum -= to_fixed(__ldcg(sums + 2 * tile + col)); }
        }
        tile_s = tile;
        before_s = cum;
    }
    if (tid == 0 && first_s == kPickThreads) {       // rounding left no crossing
        tile_s = n - 1;
        before_s = R - to_fixed(__ldcg(sums + 2 * (n - 1) + col));
    }
    __syncthreads();
    if (warp != 0) return;
    const int tile = tile_s;
    const uint64_t before = before_s;
    const bool residual = col == 0;
    const char* trow = static_cast<const char*>(A.target) + job.trow * A.V * E;
    const char* drow = static_cast<const char*>(A.draft) + (job.drow >= 0 ? job.drow : 0) * A.V * E;
    float xp[8], xq[8], wv[8];
    const int v0 = tile * 256 + lane * 8;
    load8<DT>(trow, v0, A.V, A.vec, xp);
    if (residual) load8<DT>(drow, v0, A.V, A.vec, xq);
    bonus_weights_of<DT>(xp, xq, v0, A.V, residual, job.mp, job.izp, job.mq, job.izq, A.s, wv);
    uint64_t wf[8];
    uint64_t own8 = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        wf[e] = to_fixed(wv[e]);
        own8 += wf[e];
    }
    uint64_t inc8 = own8;
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t v = __shfl_up_sync(0xffffffffu, inc8, off);
        if (lane >= off) inc8 += v;
    }
    const unsigned hit8 = __ballot_sync(0xffffffffu, before + inc8 > thr);
    int chosen = -1;
    if (hit8) {
        const int src = __ffs(hit8) - 1;
        if (lane == src) {
            uint64_t cum = before + inc8 - own8;
            for (int e = 0; e < 8; ++e) {
                cum += wf[e];
                if (cum > thr) { chosen = v0 + e; break; }
            }
        }
        chosen = __shfl_sync(0xffffffffu, chosen, src);
    }
    if (chosen < 0) {                                 // rounding fallback
        int cand = -1;
        for (int e = 7; e >= 0; --e)
            if (wv[e] > 0.0f) { cand = v0 + e; break; }
        for (int off = 16; off > 0; off >>= 1) cand = max(cand, __shfl_xor_sync(0xffffffffu, cand, off));
        chosen = cand >= 0 ? cand : min(tile * 256, A.V - 1);
    }
    if (lane == 0) A.committed[job.slot] = chosen;
    if (A.out_tokens) {                               // fused compact scatter of the request
        const int64_t row0 = static_cast<int64_t>(b) * A.gamma;
        const int Lc = static_cast<int>(job.slot - row0) + 1;
        int tok = -1;
        if (lane < Lc - 1) tok = drafts[lane];       // block token lane + 1, loaded before the wait
        else if (lane == Lc - 1) tok = chosen;
        const int sb = scatter_request(b, Lc, A.gamma, tok, lane, A.out_tokens, A.out_len,
                                       A.out_cap, n_hist);
        if (lane == 0) raise_status(A.status, sb);
    }
}

// Stochastic verify after the streaming kernel, in one launch spread over the grid: the CTAs
// of request b (ctas_per_request of them, each with kTilesPerCta 256-token tiles) each
//   1. combine the chunk partials of the request's target and draft rows into (m, Z) per row
//      (rows spread over the CTA's warps; every CTA gets the same bits),
//   2. run the accept tests of its drafts (Philox4x64-10 uniforms, the min(1, p/q) rule) and
//      walk to the first rejection, which fixes the bonus row: the residual max(0, p - q) of
//      the rejecting position, or p of the last verified position after full acceptance,
//   3. sum the bonus weights over their own tiles (a residual draw also records p's sums, for
//      the rare fallback to p when rounding leaves a residual of zero),
// and the last of the request's CTAs to finish (a per-request counter that the streaming kernel
// zeroed; no CTA waits for another) draws the bonus token by the inverse CDF over the tile sums
// and appends the request's tokens when fused. CTA 0 of the request writes accept_len, the
// ceiling, row_prob and every committed slot but the bonus one, which the drawing CTA writes.
template <int DT, int G>
__global__ void __launch_bounds__(kTileThreads)
bonus_final_kernel(FinalArgs A, int ctas_per_request)
{
    constexpr int kBonusGroup = G;            // tiles a warp loads before reducing them
    constexpr int kTilesPerCta = kTileWarps * G;
    constexpr int E = (DT == DSPARK_BF16) ? 2 : 4;
    __shared__ float mp_s[DSPARK_MAX_GAMMA], zp_s[DSPARK_MAX_GAMMA];
    __shared__ float mq_s[DSPARK_MAX_GAMMA], zq_s[DSPARK_MAX_GAMMA];
    __shared__ uint64_t ub_s[DSPARK_MAX_GAMMA];
    __shared__ float u_s[DSPARK_MAX_GAMMA];
    __shared__ int d_s[DSPARK_MAX_GAMMA];             // the drafts, for the fused scatter
    __shared__ BonusJob job_s;
    const int b = blockIdx.x / ctas_per_request;
    const int cta = blockIdx.x - b * ctas_per_request;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int gamma = A.gamma;
    const int L = gamma - 1;
    int bits = 0;
    // Inputs of the call (drafts, windows, cu_seqlens, the tested drafts' two logits, the
    // history length) are fetched before waiting for the streaming kernel: no kernel of this
    // call writes them, and the previous call's kernels have completed by then.
    const int d_mine = (warp == 0 && lane < L)
                           ? __ldg(A.tokens + static_cast<int64_t>(b) * gamma + lane + 1) : -1;
    int w = gamma;
    if (A.mode != DSPARK_STATIC) {
        w = __ldg(A.windows + b);
        if (w < 1 || w > gamma) {
            if (tid == 0 && cta == 0) bits |= DSPARK_STATUS_BAD_WINDOW;
            w = w < 1 ? 1 : gamma;
        }
    }
    const int nrows = (A.mode == DSPARK_COMPACT) ? w : gamma;
    const int ndec = nrows - 1;
    const int64_t base = (A.mode == DSPARK_COMPACT) ? static_cast<int64_t>(__ldg(A.cu + b))
                                                    : static_cast<int64_t>(b) * gamma;
    const int64_t n_t = target_row_count(A.mode, A.cu, A.B, gamma, A.target_rows, A.rows_max);
    const bool rows_ok = request_rows_ok(A, b, base, nrows, n_t);
    const bool tested = warp == 0 && lane < ndec;
    const bool valid = d_mine >= 0 && d_mine < A.V;
    float lp = 0.0f, lq = 0.0f;
    if (rows_ok && tested && valid) {
        lp = load_logit<DT>(static_cast<const char*>(A.target) + (base + lane) * A.V * E, d_mine);
        lq = load_logit<DT>(static_cast<const char*>(A.draft) +
                                (static_cast<int64_t>(b) * L + lane) * A.V * E, d_mine);
    }
    const int n_hist = (A.out_tokens != nullptr && warp == 0) ? A.out_len[b] : 0;
    // the position's uniforms (Philox4x64-10 of request, position, step and seed, all call
    // inputs): word 0 for the accept test, word 1 for a bonus drawn there; kept in shared
    // memory by the lane that reads them back in the walk
    if (warp == 0) d_s[lane] = d_mine;
    if (warp == 0 && lane < nrows) {
        uint64_t rnd[4];
        philox4x64_10(static_cast<uint64_t>(b), static_cast<uint64_t>(lane), A.step, 0ull,
                      A.seed, 0ull, rnd);
        ub_s[lane] = rnd[1] >> 11;                    // u' = ub * 2^-53
        u_s[lane] = static_cast<float>(rnd[0] >> 40) * 0x1p-24f;
    }
    pdl_wait_and_trigger();
    reset_ws_head(A.head);

    if (!rows_ok) {
        if (cta == 0) bad_rows_outputs(A, b, base, nrows, tid, kTileThreads, bits, n_hist);
        return;
    }

    // 1. (m, Z) of the request's target rows and tested draft rows
    combine_request_rows(A, base, nrows, ndec, warp, kTileWarps, lane, mp_s, zp_s, mq_s, zq_s);
    __syncthreads();

    // 2. accept tests, the walk and the bonus job (warp 0); CTA 0 writes the outputs
    if (warp == 0) {
        const bool writer = cta == 0;
        if (tested && !valid) bits |= DSPARK_STATUS_BAD_TOKEN;
        bool acc = false;
        uint64_t ub = 0;
        if (lane < nrows) {
            ub = ub_s[lane];
            float pp = -1.0f, qq = -1.0f;
            if (tested && valid) {
                // fp32 (FP64 is scarce here): exponents relative to each row's maximum, and the
                // ratio as one exp2 of their difference, so p/q neither under- nor overflows
                const float ep = (lp - mp_s[lane]) * A.s;
                const float eq = (lq - mq_s[lane]) * A.s;
                const float u = u_s[lane];
                if (lq == -INFINITY) {
                    acc = true;                     // q(d) = 0
                } else {
                    const float ratio = exp2f(ep - eq) * (zq_s[lane] / zp_s[lane]);
                    acc = u < ratio;
                }
                pp = exp2f(ep) / zp_s[lane];
                qq = exp2f(eq) / zq_s[lane];
            }
            if (writer && A.row_prob) {
                A.row_prob[(base + lane) * 2] = pp;
                A.row_prob[(base + lane) * 2 + 1] = qq;
            }
        }
        const unsigned rej = __ballot_sync(0xffffffffu, !acc);   // ndec <= 31: never zero
        const int lead = __ffs(rej) - 1;
        const int Lc = 1 + min(lead, w - 1);
        const int Lf = 1 + lead;
        const int pos = Lc - 1;
        const uint64_t jub = __shfl_sync(0xffffffffu, ub, pos);
        if (lane == 0) {
            const bool residual = pos < w - 1;
            BonusJob job;
            job.trow = base + pos;
            job.drow = residual ? static_cast<int64_t>(b) * L + pos : -1;
            job.mp = mp_s[pos];
            job.izp = 1.0f / zp_s[pos];
            job.mq = residual ? mq_s[pos] : 0.0f;
            job.izq = residual ? 1.0f / zq_s[pos] : 0.0f;
            job.ubits = jub;
            job.slot = static_cast<int64_t>(b) * gamma + Lc - 1;
            job_s = job;
        }
        if (writer) {
            int32_t* out = A.committed + static_cast<int64_t>(b) * gamma;
            if (lane < gamma && lane != Lc - 1) out[lane] = (lane < Lc - 1) ? d_mine : -1;
            if (lane == 0) {
                A.accept_len[b] = Lc;
                if (A.ceiling) A.ceiling[b] = (A.mode == DSPARK_COMPACT) ? -1 : Lf;
            }
            const unsigned any = __ballot_sync(0xffffffffu, bits != 0);
            if (any) {
                int all = bits;
                for (int off = 16; off > 0; off >>= 1) all |= __shfl_xor_sync(0xffffffffu, all, off);
                if (lane == 0) raise_status(A.status, all);
            }
        }
    }
    __syncthreads();
    const BonusJob job = job_s;

    // 3. this CTA's tile sums of the bonus row(s)
    const bool residual = job.drow >= 0;
    const char* trow = static_cast<const char*>(A.target) + job.trow * A.V * E;
    const char* drow = static_cast<const char*>(A.draft) + (residual ? job.drow : 0) * A.V * E;
    const int t0 = cta * kTilesPerCta + warp * kBonusGroup;
    float xp[kBonusGroup][8], xq[kBonusGroup][8];
#pragma unroll
    for (int g = 0; g < kBonusGroup; ++g) {
        const int v0 = (t0 + g) * 256 + lane * 8;
        load8<DT>(trow, v0, A.V, A.vec, xp[g]);
        if (residual) load8<DT>(drow, v0, A.V, A.vec, xq[g]);
    }
    float* sums = A.tiles + static_cast<int64_t>(b) * A.n_tiles * 2;
#pragma unroll
    for (int g = 0; g < kBonusGroup; ++g) {
        const int t = t0 + g;
        const int v0 = t * 256 + lane * 8;
        // p once (and q): the residual weight max(p - q, 0) and p's own weight reuse it, with
        // the arithmetic of bonus_weights_of
        float wr[8], wp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const bool in_v = v0 + e < A.V;
            wp[e] = in_v ? token_prob(xp[g][e], job.mp, job.izp, A.s) : 0.0f;
            if (residual) {
                const float q = in_v ? token_prob(xq[g][e], job.mq, job.izq, A.s) : 0.0f;
                wr[e] = fmaxf(__fsub_rn(wp[e], q), 0.0f);
            }
        }
        float sp = sum8(wp);
        float sr = residual ? sum8(wr) : sp;
        for (int off = 16; off > 0; off >>= 1) {
            sp += __shfl_xor_sync(0xffffffffu, sp, off);
            sr += __shfl_xor_sync(0xffffffffu, sr, off);
        }
        if (lane == 0 && t < A.n_tiles) {
            sums[2 * t] = sr;
            sums[2 * t + 1] = sp;
        }
    }
    // the request's last CTA to finish draws the token: after the CTA barrier, one thread
    // counts the CTA done with an acquire-release add at device scope (its release covers the
    // tile sums every warp of the CTA stored before the barrier; its acquire, in the last CTA,
    // every other CTA's); the pick reads the sums from L2 (ld.global.cg)
    __shared__ bool last_s;
    __syncthreads();
    if (tid == 0) {
        unsigned old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old)
                     : "l"(A.done + b) : "memory");
        last_s = old == static_cast<unsigned>(ctas_per_request) - 1;
    }
    __syncthreads();
    if (!last_s) return;
    bonus_pick<DT>(A, b, job, n_hist, d_s);
}

template <int DT, bool STOCH>
int run_verify(const VerifyCall& c, const Plan& plan, WsHead* head, void* part_t, void* part_d,
               unsigned* done, void* tiles, cudaStream_t stream)
{
    const int L = c.gamma - 1;
    const double inv_t = STOCH ? 1.0 / static_cast<double>(c.temperature) : 1.0;
    const float s = static_cast<float>(1.4426950408889634 * inv_t);   // log2(e) / T

    StreamArgs sa;
    sa.target = c.target;
    sa.draft = c.draft;
    sa.cu = c.cu;
    sa.windows = c.windows;
    sa.part_t = part_t;
    sa.part_d = part_d;
    sa.status = c.status;
    sa.mode = c.mode;
    sa.V = c.V;
    sa.nc = plan.nc;
    sa.C = plan.C;
    const size_t esz = (DT == DSPARK_BF16) ? 2 : 4;
    // vector path: whole 8-element groups (V % 8 == 0) starting on 16-byte boundaries
    bool vec = c.V % 8 == 0 && (static_cast<size_t>(c.V) * esz) % 16 == 0 &&
               reinterpret_cast<uintptr_t>(c.target) % 16 == 0;
    if (STOCH) vec = vec && reinterpret_cast<uintptr_t>(c.draft) % 16 == 0;
    sa.vec = vec ? 1 : 0;
    sa.B = c.B;
    sa.gamma = c.gamma;
    sa.target_rows = c.target_rows;
    sa.rows_max = plan.rows_max;
    sa.s = s;
    // stochastic: the bonus kernel's per-request counters, zeroed by the streaming kernel
    sa.zero = STOCH ? done : nullptr;
    sa.n_zero = STOCH ? c.B : 0;
    sa.head = head;

    const int64_t max_units = (plan.rows_max + (STOCH ? static_cast<int64_t>(c.B) * L : 0)) * plan.nc;
    int rc = launch_verify_stream(DT, STOCH, sa, max_units, stream);
    if (rc != DSPARK_OK) return rc;

    FinalArgs fa;
    fa.target = c.target;
    fa.draft = c.draft;
    fa.cu = c.cu;
    fa.windows = c.windows;
    fa.tokens = c.tokens;
    fa.part_t = part_t;
    fa.part_d = part_d;
    fa.accept_len = c.accept_len;
    fa.committed = c.committed;
    fa.ceiling = c.ceiling;
    fa.row_prob = c.row_prob;
    fa.status = c.status;
    fa.seed = c.seed;
    fa.step = c.step;
    fa.mode = c.mode;
    fa.V = c.V;
    fa.nc = plan.nc;
    fa.vec = sa.vec;
    fa.B = c.B;
    fa.gamma = c.gamma;
    fa.target_rows = c.target_rows;
    fa.rows_max = plan.rows_max;
    fa.s = s;
    fa.done = done;
    fa.tiles = static_cast<float*>(tiles);
    fa.head = head;
    fa.out_tokens = c.out_tokens;
    fa.out_len = c.out_len;
    fa.out_cap = c.out_cap;
    fa.n_tiles = (c.V + 255) / 256;
    if (!STOCH) {
        if (c.B <= kFinalSmallBatch)
            return launch_pdl("verify (finalize)", verify_finalize_kernel<DT, kFinalThreadsSmall, 1>,
                              dim3(c.B), dim3(kFinalThreadsSmall), 0, stream, fa);
        // two or four requests per CTA when one per CTA would put a CTA on every SM: the next
        // step's scheduler (one CTA holding a whole SM's registers) can then start on a free SM
        // while the finaliser works
        DeviceInfo dev;
        rc = current_device(&dev);
        if (rc != DSPARK_OK) return rc;
        const int room = dev.sm_count - dev.sm_count / 8;
        if (c.B <= room)
            return launch_pdl("verify (finalize)", verify_finalize_kernel<DT, kFinalThreadsLarge, 1>,
                              dim3(c.B), dim3(kFinalThreadsLarge), 0, stream, fa);
        if (c.B <= 2 * room)
            return launch_pdl("verify (finalize)", verify_finalize_kernel<DT, kFinalThreadsLarge, 2>,
                              dim3((c.B + 1) / 2), dim3(2 * kFinalThreadsLarge), 0, stream, fa);
        return launch_pdl("verify (finalize)", verify_finalize_kernel<DT, kFinalThreadsLarge, 4>,
                          dim3((c.B + 3) / 4), dim3(4 * kFinalThreadsLarge), 0, stream, fa);
    }
    // one tile per warp while the batch's bonus rows would not cover the SMs, four otherwise
    DeviceInfo dev;
    rc = current_device(&dev);
    if (rc != DSPARK_OK) return rc;
    const int64_t cpr4 = ceil_div(fa.n_tiles, kTileWarps * 4);
    if (static_cast<int64_t>(c.B) * cpr4 >= dev.sm_count)
        return launch_pdl("verify (bonus)", bonus_final_kernel<DT, 4>,
                          dim3(static_cast<unsigned>(c.B * cpr4)), dim3(kTileThreads), 0, stream,
                          fa, static_cast<int>(cpr4));
    const int64_t cpr1 = ceil_div(fa.n_tiles, kTileWarps);
    return launch_pdl("verify (bonus)", bonus_final_kernel<DT, 1>,
                      dim3(static_cast<unsigned>(c.B * cpr1)), dim3(kTileThreads), 0, stream, fa,
                      static_cast<int>(cpr1));
}

}  // namespace

// Workspace layout: the head (state handed from call to call); target-row partials; then,
// stochastic only, draft-row partials, the bonus kernel's per-request counters [B] and the bonus
// tile sums [B][n_tiles][2].
struct WsLayout {
    size_t part, done, tiles, total;
};

WsLayout ws_layout(int B, int gamma, int V, int stochastic)
{
    WsLayout l = {0, 0, 0, 0};
    if (B <= 0) return l;
    const Plan plan = make_plan(V, B, gamma);
    const size_t per = stochastic ? sizeof(SoftPart) : sizeof(ArgPart);
    l.part = align_up(static_cast<size_t>(plan.rows_max) * plan.nc * per, 256);
    if (!stochastic) {
        l.total = kWsHeadBytes + l.part;
        return l;
    }
    l.done = align_up(sizeof(unsigned) * static_cast<size_t>(B), 256);
    l.tiles = align_up(sizeof(float) * 2 * static_cast<size_t>(B) * ((V + 255) / 256), 256);
    l.total = kWsHeadBytes + 2 * l.part + l.done + l.tiles;
    return l;
}

size_t verify_workspace_bytes(int B, int gamma, int V, int stochastic)
{
    return ws_layout(B, gamma, V, stochastic).total;
}

int launch_verify(const VerifyCall& c, cudaStream_t stream)
{
    if (c.stochastic && c.V > kMaxVocabStochastic)
        return fail(DSPARK_ERR_UNSUPPORTED, "dspark_verify: stochastic verify supports V <= %d, got %d",
                    kMaxVocabStochastic, c.V);
    const Plan plan = make_plan(c.V, c.B, c.gamma);
    const size_t need = verify_workspace_bytes(c.B, c.gamma, c.V, c.stochastic);
    if (c.ws_bytes < need)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: workspace of %zu bytes, %zu needed",
                    c.ws_bytes, need);
    if (need > 0 && (c.ws == nullptr || reinterpret_cast<uintptr_t>(c.ws) % 16 != 0))
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: workspace must be a 16-byte aligned device pointer");
    const WsLayout lay = ws_layout(c.B, c.gamma, c.V, c.stochastic);
    WsHead* head = static_cast<WsHead*>(c.ws);
    char* ws = static_cast<char*>(c.ws) + kWsHeadBytes;
    void* part_t = ws;
    void* part_d = c.stochastic ? ws + lay.part : nullptr;
    unsigned* done = c.stochastic ? reinterpret_cast<unsigned*>(ws + 2 * lay.part) : nullptr;
    void* tiles = c.stochastic ? ws + 2 * lay.part + lay.done : nullptr;
    if (c.dtype == DSPARK_BF16)
        return c.stochastic
                   ? run_verify<DSPARK_BF16, true>(c, plan, head, part_t, part_d, done, tiles, stream)
                   : run_verify<DSPARK_BF16, false>(c, plan, head, part_t, part_d, done, tiles, stream);
    return c.stochastic
               ? run_verify<DSPARK_F32, true>(c, plan, head, part_t, part_d, done, tiles, stream)
               : run_verify<DSPARK_F32, false>(c, plan, head, part_t, part_d, done, tiles, stream);
}

}  // namespace dspark
