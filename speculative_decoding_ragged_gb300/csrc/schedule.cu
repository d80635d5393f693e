// schedule.cu — the confidence scheduler as one single-CTA kernel.
//
// "DSpark in SGLang: Speculative Decoding with Confidence-Driven, Variable-Length Verification"
// (LMSYS blog summary), A2 method details: the confidence head's scores multiply along the
// block into a survival probability; the scheduler reads the additive cost table
// T(bs,K) = bias + alpha(bs) + theta(bs+K) online and picks the verify budget that maximises
// expected committed tokens per unit of step time, which yields a window per request.
//
// Work: n = B*(gamma-1) <= 16384 candidates, all in shared memory of one CTA.
//   1. survivals -> fixed-point keys; request b's keys already descend along j (survivals
//      never grow), so the array starts as B sorted runs in (request, position) order. The
//      theta entries this thread will need are fetched in the same round trip;
//   2. n <= 4096: a counting sort over 4096 order-preserving key buckets, then the exact place
//      inside each (small) bucket by one 64-bit compare per pair, which orders by key
//      descending, then request, then position; it also records every candidate's rank. When
//      a bucket is too big (many equal keys), a stable merge of the runs instead. Larger n: a
//      bitonic sort of 64-bit words key << 31 | (2^31 - 1 - index);
//   3. block-wide inclusive scan of the keys (exact uint64 sums S(K));
//   4. obj(K) = double(B*2^32 + S(K)) / T(K), argmax K*, the smallest K among equal
//      objectives. FP64 latency is long on this part, and K* is an output while the
//      objective is not: a double-float screen (pairs of fp32 values, error below 2^-42
//      relative, as 64-bit keys that order like the objective) gives each K a key, and one
//      block reduction finds the best key, its K and the runner-up. K* is that K when every
//      other key lies more than 2^-37 below and every K was judged; ties, near ties and cost
//      tables the screen cannot judge (negative or out-of-range terms) take the exact fp64
//      objectives of the K within the margin or not judged, and an argmax over those that
//      compares the objectives' bit patterns as integers (they are positive);
//   5. windows w_b = 1 + count of request b among the first K* candidates: with the ranks,
//      the length of the prefix of its run ranked below K*.
// Latency-bound (microseconds); the grid is one CTA by construction of the problem. Every
// two-level reduction publishes per-warp totals behind one barrier and lets each warp combine
// them itself. The kernel runs once per step from a cold instruction cache, so its loops stay
// rolled: code size, not arithmetic, sets much of its time.
#include "common.cuh"

namespace dspark {
namespace {

constexpr int kMergeMax = 4096;          // ping-pong merge buffers up to this many words
constexpr int kBuckets = 4096;           // 128 buckets per power of two of the key (keys 0, 1 share)
constexpr int kSmallBlockMax = 256;      // up to this many candidates: a 256-thread block

// The block kernel's shape: 1024 threads, or 256 for at most 256 candidates (fewer warps for
// the same few items: every reduction, scan and loop bound of the block costs less).
template <int NT>
struct Shape {
    static_assert(NT == 256 || NT == 1024, "the block scheduler runs 256 or 1024 threads");
    static constexpr int kMergeItems = (NT == 256 ? kSmallBlockMax : kMergeMax) / NT;
    static constexpr int kBucketsPerThread = kBuckets / NT;
    static constexpr int kTiersPerThread = (DSPARK_MAX_TIERS + NT - 1) / NT;
};
constexpr int kBucketMax = 64;           // larger buckets (many equal keys): merge instead
// The screened best decides K* alone when every other key lies more than this below it:
// 2^19 key units, at least 2^-37 of the objective, sixteen times the 2^-41 that two screened
// values' errors (each below 2^-42 relative) can add up to.
constexpr uint64_t kKeyMargin = 1ull << 19;

// Objectives are positive doubles (or "none" = 0), whose bit patterns order like the values:
// compare them as integers, the larger objective first, then the smaller K.
__device__ __forceinline__ bool better(uint64_t o1, int k1, uint64_t o2, int k2)
{
    return o1 > o2 || (o1 == o2 && static_cast<unsigned>(k1) < static_cast<unsigned>(k2));
}

// ---- the screen: obj(K) in double-float arithmetic (pairs of fp32 values) ----
// The exact objective is an fp64 division, and FP64 latency on this part is long (one
// division about 660 cycles). K* is an output but the objective is not, so a screen accurate
// to 2^-42 relative decides K* whenever the best screened K beats every other by the margin
// kKeyMargin (at least 2^-37); only ties, near ties and cost tables the screen cannot judge
// take fp64.
struct DF {
    float h, l;     // value h + l, |l| <= ulp(h) / 2 once normalised
};

__device__ __forceinline__ DF fast_two_sum(float a, float b)   // |a| >= |b|: exact split
{
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ DF two_sum(float a, float b)        // any order: exact split
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

// x (bits of a double) as h + l: h its top 24 significand bits, exactly, l the next 29
// rounded once (relative error < 2^-47). False unless x is 0 or in [2^-60, 2^61).
__device__ __forceinline__ bool split_double(uint64_t bits, DF& out)
{
    if (bits == 0) {
        out = {0.0f, 0.0f};
        return true;
    }
    const int e = static_cast<int>(bits >> 52);           // biased exponent, sign bit included
    if (e < 1023 - 60 || e > 1023 + 60) return false;     // negative, tiny, huge, inf or NaN
    const uint64_t m = (bits & ((1ull << 52) - 1)) | (1ull << 52);   // x = m 2^(e - 1075)
    const float sh = __int_as_float((e - 1075 + 29 + 127) << 23);    // 2^(e - 1046)
    const float sl = __int_as_float((e - 1075 + 127) << 23);         // 2^(e - 1075)
    out = fast_two_sum(__fmul_rn(__uint2float_rn(static_cast<uint32_t>(m >> 29)), sh),
                       __fmul_rn(__uint2float_rn(static_cast<uint32_t>(m & 0x1FFFFFFFu)), sl));
    return true;
}

// An integer 1 <= E < 2^53 as h + l (relative error < 2^-47).
__device__ __forceinline__ DF split_u53(uint64_t E)
{
    const int sh = 40 - __clzll(static_cast<long long>(E));   // bits below the top 24
    if (sh <= 0) return {__uint2float_rn(static_cast<uint32_t>(E)), 0.0f};
    const float h = __fmul_rn(__uint2float_rn(static_cast<uint32_t>(E >> sh)),
                              __int_as_float((sh + 127) << 23));
    return fast_two_sum(h, __uint2float_rn(static_cast<uint32_t>(E & ((1ull << sh) - 1))));
}

// A key that grows with the positive value h + l, continuously across h: h's bits above, then
// l in units of 2^-32 ulp(h) added with its sign, so that one step of h is 2^32 units and a key
// difference measures the value difference (a unit is 2^-56 to 2^-55 of the value).
__device__ __forceinline__ uint64_t df_key(DF g)
{
    const uint32_t hb = __float_as_uint(g.h);
    const int eh = static_cast<int>(hb >> 23) - 127;
    const long long lu = __float2ll_rn(__fmul_rn(g.l, __int_as_float((127 + 55 - eh) << 23)));
    return (static_cast<uint64_t>(hb) << 32) + static_cast<uint64_t>(lu);
}

// The screen key of obj(K) = E / (t0 + theta), theta given by its bits, t0 split once by the
// caller (t0_ok false: not judged). Returns 0 when the screen cannot judge this K (t0 or theta
// negative, outside [2^-60, 2^61), or T = 0); the exact fp64 path then decides it. Error
// budget, relative: E and both cost terms 2^-47 each, their sum 2^-46, the quotient (fp32
// estimate, exact residual by fma, fp32 correction) 2^-43, against the fp64 objective's own
// two roundings 2^-52: below 2^-42 in all.
__device__ __forceinline__ uint64_t screen_key(uint64_t E, DF t0d, bool t0_ok, uint64_t theta_bits)
{
    DF thd;
    if (!t0_ok || !split_double(theta_bits, thd)) return 0;
    const DF s = two_sum(t0d.h, thd.h);
    const DF T = fast_two_sum(s.h, __fadd_rn(__fadd_rn(t0d.l, thd.l), s.l));
    if (!(T.h > 0.0f)) return 0;
    const DF e = split_u53(E);
    const float q1 = __fdividef(e.h, T.h);
    const float ph = __fmul_rn(q1, T.h);
    float r = __fsub_rn(e.h, ph);                      // exact: ph is within 2x of e.h
    r = __fsub_rn(r, __fmaf_rn(q1, T.h, -ph));         // the product's rounding error
    r = __fadd_rn(r, e.l);
    r = __fmaf_rn(-q1, T.l, r);
    return df_key(fast_two_sum(q1, __fdividef(r, T.h)));
}

// The largest 64-bit value over the warp.
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t x)
{
    const uint32_t hi = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(x >> 32));
    const uint32_t lo = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(x >> 32) == hi
                                                           ? static_cast<uint32_t>(x) : 0u);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

// The best key of the warp (the smallest K among equal keys), every other key's maximum (the
// runner-up; a tie with the best counts), and whether any K went unjudged; each lane brings
// its own best (k1, K1), second k2 and flag. Key 0 means none; K1 = -1 with key 0.
__device__ __forceinline__ void warp_top2(uint64_t& k1, int& K1, uint64_t& k2, bool& nj)
{
    const uint64_t m = warp_max_u64(k1);
    const int mK = static_cast<int>(__reduce_min_sync(
        0xffffffffu, k1 == m ? static_cast<uint32_t>(K1) : 0xFFFFFFFFu));
    k2 = warp_max_u64((k1 == m && K1 == mK) ? k2 : k1);
    k1 = m;
    K1 = mK;
    nj = __any_sync(0xffffffffu, nj);
}

// The sorted run of request b: fixed-point survival keys. MERGE: 32-bit keys and indices in
// parallel arrays; else 64-bit words key << 31 | (2^31 - 1 - index).
template <bool MERGE>
__device__ __forceinline__ void write_run(const float* __restrict__ conf, int b, int L,
                                          uint64_t* word, uint32_t* key32, int* index)
{
    float s = 1.0f;
#pragma unroll 1
    for (int j0 = 0; j0 < L; j0 += 8) {
        float c[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j0 + j < L) c[j] = __ldg(conf + static_cast<int64_t>(b) * L + j0 + j);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j0 + j < L) {
                s = __fmul_rn(s, fminf(fmaxf(c[j], 0.0f), 1.0f));   // NaN -> 0
                const int idx = b * L + j0 + j;
                const uint32_t k32 = s >= 1.0f ? 0xFFFFFFFFu : __float2uint_rn(__fmul_rn(s, 4294967296.0f));
                if (MERGE) {
                    key32[idx] = k32;
                    index[idx] = idx;
                } else {
                    const uint64_t key = s >= 1.0f ? (1ull << 32) : static_cast<uint64_t>(k32);
                    word[idx] = (key << 31) | static_cast<uint64_t>(0x7FFFFFFF - idx);
                }
            }
        }
    }
}

// Order-preserving bucket of a 32-bit key (equal keys share a bucket): the fp32 exponent and
// top seven mantissa bits of the key truncated to fp32, so a bucket spans under 1 % of its
// keys; keys 0 and 1 share bucket 0.
__device__ __forceinline__ int key_bucket(uint32_t k32)
{
    if (k32 == 0) return 0;
    const uint32_t f = __float_as_uint(__uint2float_rz(k32));
    return static_cast<int>((f >> 16) - (127u << 7));
}

// A key and its candidate index as one word that orders like (key descending, index
// ascending) when compared as an unsigned integer, larger first.
__device__ __forceinline__ uint64_t rank_word(uint32_t k32, int idx)
{
    return (static_cast<uint64_t>(k32) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

__device__ __forceinline__ uint64_t key_value(uint32_t k32)
{
    return k32 == 0xFFFFFFFFu ? (1ull << 32) : static_cast<uint64_t>(k32);
}

// Bits of a double, exactly, from an integer below 2^53 (integer operations only).
__device__ __forceinline__ double u53_to_double(uint64_t x)
{
    if (x == 0) return 0.0;
    const int lz = __clzll(static_cast<long long>(x));          // >= 11
    const uint64_t m = x << (lz - 11);                           // leading one at bit 52
    const uint64_t e = static_cast<uint64_t>(1023 + 63 - lz);
    return __longlong_as_double(static_cast<long long>((e << 52) | (m & ((1ull << 52) - 1))));
}

// The exact objective double(E) / T(K), T = t0 + theta: its bit pattern, or 0 (none) when T is
// not positive and finite.
__device__ __noinline__ uint64_t exact_objective(uint64_t E, double t0, uint64_t theta_bits)
{
    const double T = t0 + __longlong_as_double(static_cast<long long>(theta_bits));
    const uint64_t tb = static_cast<uint64_t>(__double_as_longlong(T));
    if ((tb >> 63) != 0 || tb == 0 || ((tb >> 52) & 0x7FF) == 0x7FF) return 0;
    return static_cast<uint64_t>(__double_as_longlong(u53_to_double(E) / T));
}

// The exact objective for the one-warp kernel: the bits of double(E) / (t0 + theta), or 0
// when the step time is not positive and finite.
__device__ __forceinline__ uint64_t small_objective(uint64_t E, double t0, uint64_t theta_bits)
{
    const double T = t0 + __longlong_as_double(static_cast<long long>(theta_bits));
    if (!(T > 0.0 && T < INFINITY)) return 0;
    return static_cast<uint64_t>(__double_as_longlong(static_cast<double>(E) / T));
}

// Element i of a small register array, by selects (no local memory under a rolled loop).
template <typename T, int N>
__device__ __forceinline__ T get_n(const T (&a)[N], int i)
{
    T v = a[0];
#pragma unroll
    for (int k = 1; k < N; ++k) v = i == k ? a[k] : v;
    return v;
}
// Sum over the warps before this one of a per-warp total, read by every lane of the warp from
// shared memory after the barrier that published the totals (no second barrier).
template <typename T>
__device__ __forceinline__ T warps_before(const T* total, int warp, int lane)
{
    T v = lane < warp ? total[lane] : T(0);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// The front-pack on the scheduler's CTA (dspark_schedule_pack). The windows are valid by
// construction (1 + a count of at most gamma - 1), so M = B + K* is known before any scan and
// the tier is reduced in the same barrier as the scan of the windows. Then each warp writes
// the rows of its own requests: the requests' rows form one contiguous range, which the warp
// fills coalesced from a warp-private stretch of the row-owner map (request << 5 | position),
// after a warp-level sync only; warps past the last request only meet the barrier and write
// padding. win(b) gives request b's window; owner holds M ints and may overlay what win reads
// (every window is read before the block barrier), and win_s (B ints outside the owner map)
// keeps each thread's windows for the pass after it.
template <int NT, typename WinFn>
__device__ __forceinline__ void pack_after_schedule(WinFn win, int B, int gamma, int K_star,
                                                    PackArgs pk,
                                                    const int (&tier_pre)[Shape<NT>::kTiersPerThread],
                                                    const int* tok_stage, int* owner,
                                                    int* tier_s, int* pack_total, int* win_s,
                                                    int32_t* __restrict__ windows,
                                                    int32_t* __restrict__ status)
{
    constexpr int kThreads = NT;
    constexpr int kTiersPerThread = Shape<NT>::kTiersPerThread;
    // the output pointers as plain locals: no store below can be taken to change them
    int32_t* const cu = pk.cu;
    int32_t* const packed_ids = pk.packed_ids;
    int32_t* const row_req = pk.row_req;
    int32_t* const row_pos = pk.row_pos;
    int32_t* const meta = pk.meta;
    const int32_t* const tokens = pk.tokens;
    const int packed_cap = pk.packed_cap;
    const unsigned full = 0xffffffffu;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int M = B + K_star;

    // tier: the smallest tier >= M (tier_pre: the thread's tiers, INT_MAX past n_tiers);
    // warps without tiers skip
    if (warp * 32 < pk.n_tiers) {
        int best = INT_MAX;
#pragma unroll
        for (int k = 0; k < kTiersPerThread; ++k)
            if (tier_pre[k] >= M && tier_pre[k] < best) best = tier_pre[k];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(full, best, off));
        if (lane == 0 && best != INT_MAX) atomicMin(tier_s, best);
    }

    // windows of this thread's consecutive requests (kept in win_s), and their scan; the warps
    // past the last request only meet the barrier and write padding
    const int items = (B + kThreads - 1) / kThreads;
    const int b0 = tid * items;
    const bool active = warp * 32 * items < B;       // uniform across the warp
    int run = 0, incl = 0;
    if (active) {
#pragma unroll 1
        for (int it = 0; it < items; ++it) {
            const int b = b0 + it;
            if (b >= B) break;
            const int w = win(b);
            windows[b] = w;
            win_s[b] = w;
            run += w;
        }
        incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(full, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) pack_total[warp] = incl;
    }
    __syncthreads();
    if (active) {
        const int base = warps_before(pack_total, warp, lane);   // all earlier warps are active
        const int warp_rows = __shfl_sync(full, incl, 31);
        int acc = base + incl - run;
#pragma unroll 1
        for (int it = 0; it < items; ++it) {
            const int b = b0 + it;
            if (b >= B) break;
            const int w = win_s[b];
            cu[b] = acc;
#pragma unroll 1
            for (int i = 0; i < w; ++i) owner[acc + i] = (b << 5) | i;
            acc += w;
        }
        if (tid == 0) cu[B] = M;
        __syncwarp();
        const int r_end = min(base + warp_rows, packed_cap);
#pragma unroll 1
        for (int r = base + lane; r < r_end; r += 32) {
            const int e = owner[r];
            const int b = e >> 5, i = e & 31;
            const int64_t ti = static_cast<int64_t>(b) * gamma + i;
            packed_ids[r] = tok_stage != nullptr ? tok_stage[ti] : __ldg(tokens + ti);
            if (row_req) row_req[r] = b;
            if (row_pos) row_pos[r] = i;
        }
    }
    int tier = *tier_s;
    int bad = 0;
    if (tier == INT_MAX) {
        tier = M;
        bad |= DSPARK_STATUS_TIER_OVERFLOW;
    }
    if (tier > packed_cap) bad |= DSPARK_STATUS_PACK_CAPACITY;
    const int rows_pad = min(tier, packed_cap);
#pragma unroll 1
    for (int r = M + tid; r < rows_pad; r += kThreads) {
        packed_ids[r] = 0;
        if (row_req) row_req[r] = -1;
        if (row_pos) row_pos[r] = -1;
    }
    if (tid == 0) {
        meta[0] = M;
        meta[1] = tier;
        raise_status(status, bad);      // the same bits in every thread
    }
}

// Before the dependency wait, pull this call's inputs into L2: a prefetch returns no data, so
// it is correct even while the previous kernel is still writing them, and once that kernel has
// finished the loads below find them in L2 instead of DRAM. The inputs' 128-byte lines, laid
// end to end, are dealt round-robin to the threads; every address lies inside its buffer.
__device__ __forceinline__ void prefetch_lines(const void* p, int bytes, int& first, int t,
                                               int nthreads)
{
    const int lines = (bytes + 127) / 128;
    int l = (t - first) % nthreads;       // this thread's first line of the buffer
    if (l < 0) l += nthreads;
#pragma unroll 1
    for (; l < lines; l += nthreads)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(p) +
                                                         128 * static_cast<int64_t>(l)));
    first += lines;
}

__device__ __forceinline__ void prefetch_inputs(int t, int nthreads, const float* conf, int B,
                                                int L, const double* alpha,
                                                const double* theta, const int32_t* tokens,
                                                const int32_t* tiers, int n_tiers)
{
    int first = 0;
    prefetch_lines(conf, 4 * B * L, first, t, nthreads);
    prefetch_lines(theta + B, 8 * (B * L + 1), first, t, nthreads);
    prefetch_lines(alpha + B, 8, first, t, nthreads);
    if (tokens != nullptr) prefetch_lines(tokens, 4 * B * (L + 1), first, t, nthreads);
    if (tiers != nullptr) prefetch_lines(tiers, 4 * n_tiers, first, t, nthreads);
}

// PACK: the same CTA then front-packs the windows it computed (dspark_schedule_pack).
template <bool MERGE, bool PACK, int NT>
__global__ void __launch_bounds__(NT, 1)
schedule_kernel(const float* __restrict__ conf, int B, int L, int n, int n_pad, double bias,
                const double* __restrict__ alpha, const double* __restrict__ theta,
                int32_t* __restrict__ windows, int32_t* __restrict__ k_star,
                int32_t* __restrict__ status, PackArgs pk, int tok_stage_off)
{
    constexpr int kThreads = NT;
    constexpr int kWarps = NT / 32;
    constexpr int kMergeItems = Shape<NT>::kMergeItems;
    constexpr int kBucketsPerThread = Shape<NT>::kBucketsPerThread;
    constexpr int kTiersPerThread = Shape<NT>::kTiersPerThread;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // MERGE: keys ksrc [n] (u32), indices isrc [n], then the ping-pong pair kdst, idst (the
    // bucket path uses that second half as n 64-bit rank words); else words [n_pad] (u64).
    // Then count [B]. The pack's row-owner map overlays the start (M <= B + n ints).
    uint64_t* word = reinterpret_cast<uint64_t*>(smem_raw);
    uint32_t* ksrc = reinterpret_cast<uint32_t*>(smem_raw);
    int* isrc = reinterpret_cast<int*>(ksrc + n);
    uint32_t* kdst = reinterpret_cast<uint32_t*>(isrc + n);
    int* idst = reinterpret_cast<int*>(kdst + n);
    uint64_t* rword = reinterpret_cast<uint64_t*>(kdst);   // 8n-byte aligned: offset 8n
    int* count = MERGE ? (idst + n) : reinterpret_cast<int*>(word + n_pad);
    __shared__ uint64_t warp_total[kWarps];
    __shared__ uint64_t red_obj[kWarps];
    __shared__ uint64_t red_sec[kWarps];
    __shared__ int red_k[kWarps];
    __shared__ int red_nj[kWarps];
    __shared__ double t0_s;
    __shared__ __align__(16) int bucket_cnt[MERGE ? kBuckets : 4];
    __shared__ __align__(16) int bucket_start[MERGE ? kBuckets : 4];
    __shared__ int warp_int[kWarps];
    __shared__ int tier_s;

    // Step 1 reads only call inputs that no kernel of this library writes (confidences, the
    // cost tables, block tokens) and writes only shared memory, so it runs before the wait for
    // the previous kernel on the stream; tiers (a caller may hand in a tier that a pack wrote)
    // and every global write come after it.
    prefetch_inputs(threadIdx.x, kThreads, conf, B, L, alpha, theta, PACK ? pk.tokens : nullptr,
                    PACK ? pk.tiers : nullptr, PACK ? pk.n_tiers : 0);
    const unsigned full = 0xffffffffu;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    int tier_pre[kTiersPerThread];
#pragma unroll
    for (int k = 0; k < kTiersPerThread; ++k) tier_pre[k] = INT_MAX;
    int* tok_stage = nullptr;
    if (PACK) {
        // the pack's tokens are read only at the end: copied into shared memory (cp.async,
        // 16-byte pieces) while the scheduler works, when they fit
        if (tid == 0) tier_s = INT_MAX;
        if (tok_stage_off >= 0) {
            tok_stage = reinterpret_cast<int*>(smem_raw + tok_stage_off);
            const int nt = B * (L + 1);
            const int n16 = nt >> 2;
#pragma unroll 1
            for (int c = tid; c < n16; c += kThreads) {
                const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(tok_stage + 4 * c));
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                             "l"(pk.tokens + 4 * c) : "memory");
            }
#pragma unroll 1
            for (int t = 4 * n16 + tid; t < nt; t += kThreads) tok_stage[t] = __ldg(pk.tokens + t);
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
    }
    constexpr int kMaxItems = MERGE ? kMergeItems : DSPARK_MAX_CANDIDATES / kThreads;
    const int items = (n + kThreads - 1) / kThreads;   // positions per thread, contiguous
    const int p0 = tid * items;
    const uint64_t* theta_bits = reinterpret_cast<const uint64_t*>(theta);

    // 1. sorted runs, and this thread's theta entries (K = p + 1 for owned positions p)
    uint64_t th[kMergeItems];
    if (MERGE) {
#pragma unroll
        for (int it = 0; it < kMergeItems; ++it)
            if (it < items && p0 + it < n) th[it] = __ldg(theta_bits + B + p0 + it + 1);
    }
    uint64_t th0 = 0;
    if (tid == 0) {
        th0 = __ldg(theta_bits + B);
        t0_s = bias + __ldg(alpha + B);
    }
#pragma unroll 1
    for (int b = tid; b < B; b += kThreads) {
        write_run<MERGE>(conf, b, L, word, ksrc, isrc);
        if (!MERGE) count[b] = 0;
    }
    if (MERGE) {
        static_assert(kBuckets % (4 * kThreads) == 0, "16-byte zeroing of the bucket counts");
        for (int j = 4 * tid; j < kBuckets; j += 4 * kThreads)
            *reinterpret_cast<int4*>(bucket_cnt + j) = make_int4(0, 0, 0, 0);
    }
    if (!MERGE)
        for (int i = n + tid; i < n_pad; i += kThreads) word[i] = 0;   // sorts after all words
    pdl_wait_and_trigger();
    if (PACK) {
#pragma unroll
        for (int k = 0; k < kTiersPerThread; ++k)
            if (tid + k * kThreads < pk.n_tiers) tier_pre[k] = __ldg(pk.tiers + tid + k * kThreads);
    }
    __syncthreads();

    // 2. sort descending. MERGE also yields rank_of[i]: the sorted position of candidate i
    int* rank_of = isrc;
    bool sorted = false;
    if (MERGE) {
        // 2a. counting sort by key bucket, when every bucket is small
#pragma unroll 1
        for (int p = tid; p < n; p += kThreads) atomicAdd(&bucket_cnt[key_bucket(ksrc[p])], 1);
        __syncthreads();
        // bucket starts in descending bucket order; thread t owns the reversed buckets
        // kBuckets - 1 - (kBucketsPerThread * t + m), m = 0..kBucketsPerThread-1, read and
        // written as 16-byte vectors of four counts
        constexpr int BPT = kBucketsPerThread;
        static_assert(BPT % 4 == 0, "whole 16-byte vectors of counts per thread");
        const int jv = kBuckets - BPT - BPT * tid;        // the thread's buckets [jv, jv + BPT)
        int a[BPT];                                       // descending bucket order
#pragma unroll
        for (int v = 0; v < BPT / 4; ++v) {
            const int4 cv = *reinterpret_cast<const int4*>(bucket_cnt + jv + 4 * v);
            a[BPT - 1 - 4 * v] = cv.x;
            a[BPT - 2 - 4 * v] = cv.y;
            a[BPT - 3 - 4 * v] = cv.z;
            a[BPT - 4 - 4 * v] = cv.w;
        }
        int own = 0, mx = 0;
#pragma unroll
        for (int m = 0; m < BPT; ++m) {
            own += a[m];
            mx = max(mx, a[m]);
        }
        const int big = mx > kBucketMax;
        int incl_b = own;
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(full, incl_b, off);
            if (lane >= off) incl_b += v;
        }
        if (lane == 31) warp_int[warp] = incl_b;
        if (!__syncthreads_or(big)) {
            const int ex = incl_b - own + warps_before(warp_int, warp, lane);
            int st[BPT];                                  // start of the m-th bucket, descending
            int acc = ex;
#pragma unroll
            for (int m = 0; m < BPT; ++m) {
                st[m] = acc;
                acc += a[m];
            }
#pragma unroll
            for (int v = 0; v < BPT / 4; ++v)
                *reinterpret_cast<int4*>(bucket_start + jv + 4 * v) =
                    make_int4(st[BPT - 1 - 4 * v], st[BPT - 2 - 4 * v], st[BPT - 3 - 4 * v],
                              st[BPT - 4 - 4 * v]);
            __syncthreads();
            // scatter rank words into the bucket ranges (any order inside a bucket); afterwards
            // bucket_start[j] holds the end of bucket j
#pragma unroll 1
            for (int p = tid; p < n; p += kThreads) {
                const uint32_t k = ksrc[p];
                const int q = atomicAdd(&bucket_start[key_bucket(k)], 1);
                rword[q] = rank_word(k, p);      // runs start in index order: isrc[p] == p
            }
            __syncthreads();
            // exact place inside the bucket: one unsigned compare orders (key desc, index asc)
#pragma unroll 1
            for (int q = tid; q < n; q += kThreads) {
                const uint64_t x = rword[q];
                const int j = key_bucket(static_cast<uint32_t>(x >> 32));
                const int c = bucket_cnt[j], s0 = bucket_start[j] - c;
                int r = 0;
#pragma unroll 4
                for (int t = s0; t < s0 + c; ++t) r += rword[t] > x;
                ksrc[s0 + r] = static_cast<uint32_t>(x >> 32);
                rank_of[static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(x))] = s0 + r;
            }
            __syncthreads();
            sorted = true;
        }
    }
    if (MERGE && !sorted) {
        // 2b. stable merge of the per-request runs
        for (int R = L; R < n; R <<= 1) {          // run length: one request, two, four, ...
            int o = p0;
            const int o_end = min(p0 + items, n);
#pragma unroll 1
            while (o < o_end) {
                const int aS = o / (2 * R) * (2 * R);
                const int aE = min(aS + R, n), bE = min(aS + 2 * R, n);
                const int lenA = aE - aS, lenB = bE - aE;
                const uint32_t* A = ksrc + aS;
                const uint32_t* Bk = ksrc + aE;
                // co-rank: how many of the first d merged outputs come from run A
                const int d = o - aS;
                int lo = max(0, d - lenB), hi = min(d, lenA);
#pragma unroll 1
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (A[mid] >= Bk[d - mid - 1]) lo = mid + 1; else hi = mid;
                }
                int i = lo, j = d - lo;
#pragma unroll 1
                for (; o < o_end && o < bE; ++o) {
                    const bool takeA = i < lenA && (j >= lenB || A[i] >= Bk[j]);
                    if (takeA) {
                        kdst[o] = A[i];
                        idst[o] = isrc[aS + i];
                        ++i;
                    } else {
                        kdst[o] = Bk[j];
                        idst[o] = isrc[aE + j];
                        ++j;
                    }
                }
            }
            __syncthreads();
            uint32_t* tk = ksrc; ksrc = kdst; kdst = tk;
            int* ti = isrc; isrc = idst; idst = ti;
        }
        // ranks into the free index buffer
#pragma unroll 1
        for (int p = tid; p < n; p += kThreads) idst[isrc[p]] = p;
        rank_of = idst;
        __syncthreads();
    } else if (!MERGE) {
        for (int k = 2; k <= n_pad; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = tid; i < (n_pad >> 1); i += kThreads) {
                    const int a = ((i & ~(j - 1)) << 1) | (i & (j - 1));
                    const int c = a + j;
                    const uint64_t x = word[a], y = word[c];
                    const bool descending = (a & k) == 0;
                    if (descending ? (x < y) : (x > y)) {
                        word[a] = y;
                        word[c] = x;
                    }
                }
                __syncthreads();
            }
        }
    }
    auto key_at = [&](int p) -> uint64_t {
        return MERGE ? key_value(ksrc[p]) : (word[p] >> 31);
    };
    auto theta_at = [&](int it, int p) -> uint64_t {
        if (!MERGE) return __ldg(theta_bits + B + p + 1);
        return get_n(th, it);
    };

    // 3. inclusive scan of keys over each thread's contiguous positions
    uint64_t run = 0;
#pragma unroll 1
    for (int it = 0; it < items; ++it) {
        const int p = p0 + it;
        if (p >= n) break;
        run += key_at(p);
    }
    uint64_t incl = run;
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t v = __shfl_up_sync(full, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_total[warp] = incl;
    __syncthreads();
    const uint64_t S_excl = incl - run + warps_before(warp_total, warp, lane);
    const uint64_t base_E = static_cast<uint64_t>(B) << 32;
    const double t0 = t0_s;
    DF t0d;
    const bool t0_ok = split_double(static_cast<uint64_t>(__double_as_longlong(t0)), t0d);

    // 4a. screen keys of the K this thread owns (thread 0 also K = 0): the thread keeps its
    // two largest keys and the first one's K, and notes any K the screen cannot judge
    uint64_t key1 = 0, key2 = 0;
    int K1 = -1;
    bool unjudged = false;
    auto take = [&](uint64_t key, int K) {
        if (key == 0) {
            unjudged = true;
        } else if (key > key1) {
            key2 = key1;
            key1 = key;
            K1 = K;
        } else if (key > key2) {
            key2 = key;
        }
    };
    if (tid == 0) take(screen_key(base_E, t0d, t0_ok, th0), 0);
    {
        uint64_t S = S_excl;
#pragma unroll 1
        for (int it = 0; it < kMaxItems; ++it) {
            const int p = p0 + it;
            if (it >= items || p >= n) break;
            S += key_at(p);
            take(screen_key(base_E + S, t0d, t0_ok, theta_at(it, p)), p + 1);
        }
    }
    // the block's best key with its K, the runner-up and the unjudged flag: per warp, then
    // every warp combines the 32 warp results itself behind one barrier
    uint64_t bk = key1, b2 = key2;
    int bK = K1;
    bool nj = unjudged;
    warp_top2(bk, bK, b2, nj);
    if (lane == 0) {
        red_obj[warp] = bk;
        red_sec[warp] = b2;
        red_k[warp] = bK;
        red_nj[warp] = nj ? 1 : 0;
    }
    __syncthreads();
    bk = lane < kWarps ? red_obj[lane] : 0;
    b2 = lane < kWarps ? red_sec[lane] : 0;
    bK = lane < kWarps ? red_k[lane] : -1;
    nj = lane < kWarps && red_nj[lane] != 0;
    warp_top2(bk, bK, b2, nj);
    const uint64_t thr = bk > kKeyMargin ? bk - kKeyMargin : 0;

    // 4b. the screened best is K* when every other K lies beyond the margin and every K was
    // judged. Else (ties, near ties, cost tables the screen cannot judge) the exact fp64
    // objective of every K not judged or within the margin, and the argmax over those. The
    // branch is uniform across the block.
    int K_star = bK;
    bool none = false;
    if (nj || bK < 0 || b2 >= thr) {
        uint64_t best_obj = 0;        // bit pattern of a positive double; 0 = none
        int best_k = -1;
        auto consider = [&](uint64_t E, uint64_t tb, int k) {
            const uint64_t key = screen_key(E, t0d, t0_ok, tb);
            if (key != 0 && key < thr) return;
            const uint64_t obj = exact_objective(E, t0, tb);
            if (obj != 0 && better(obj, k, best_obj, best_k)) {
                best_obj = obj;
                best_k = k;
            }
        };
        if (tid == 0) consider(base_E, th0, 0);
        if (unjudged || key1 >= thr) {
            uint64_t S = S_excl;
#pragma unroll 1
            for (int it = 0; it < kMaxItems; ++it) {
                const int p = p0 + it;
                if (it >= items || p >= n) break;
                S += key_at(p);
                consider(base_E + S, theta_at(it, p), p + 1);
            }
        }
        // the best (objective, K) of a warp, then of the block (every warp combines the 32
        // warp results itself)
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            if (pass == 1) {
                if (lane == 0) {
                    red_obj[warp] = best_obj;
                    red_k[warp] = best_k;
                }
                __syncthreads();
                best_obj = lane < kWarps ? red_obj[lane] : 0;
                best_k = lane < kWarps ? red_k[lane] : -1;
            }
            for (int off = 16; off > 0; off >>= 1) {
                const uint64_t o = __shfl_xor_sync(full, best_obj, off);
                const int kk = __shfl_xor_sync(full, best_k, off);
                if (better(o, kk, best_obj, best_k)) {
                    best_obj = o;
                    best_k = kk;
                }
            }
        }
        none = best_k < 0;            // no K with a positive, finite step time
        K_star = none ? 0 : best_k;
    }
    if (tid == 0) {
        if (none) raise_status(status, DSPARK_STATUS_BAD_COST);
        *k_star = K_star;
    }

    // 5. windows: w_b = 1 + the request's candidates among the first K*. Its candidates sit at
    // increasing sorted positions along j, so they are a prefix of its run.
    auto win_rank = [&](int b) -> int {
        int c = 0;
#pragma unroll 1
        for (int j = 0; j < L; ++j) c += rank_of[b * L + j] < K_star;
        return 1 + c;
    };
    if (!MERGE) {
        for (int p = tid; p < K_star; p += kThreads) {
            const int idx = 0x7FFFFFFF - static_cast<int>(word[p] & 0x7FFFFFFFull);
            atomicAdd(&count[idx / L], 1);
        }
        __syncthreads();
    }
    auto win_count = [&](int b) -> int { return 1 + count[b]; };
    if (PACK) {
        // the staged tokens are complete once every thread's copies have landed (the pack's
        // barrier comes before its first read of them)
        if (tok_stage != nullptr) asm volatile("cp.async.wait_all;" ::: "memory");
        __shared__ int pack_total[kWarps];
        int* owner = reinterpret_cast<int*>(smem_raw);   // sort buffers: at least B + n ints
        if (MERGE)
            pack_after_schedule<NT>(win_rank, B, L + 1, K_star, pk, tier_pre, tok_stage, owner,
                                &tier_s, pack_total, count, windows, status);
        else
            pack_after_schedule<NT>(win_count, B, L + 1, K_star, pk, tier_pre, tok_stage, owner,
                                &tier_s, pack_total, count, windows, status);
    } else {
        for (int b = tid; b < B; b += kThreads) windows[b] = MERGE ? win_rank(b) : win_count(b);
    }
}

__global__ void schedule_trivial_kernel(int B, double bias, const double* __restrict__ alpha,
                                        const double* __restrict__ theta,
                                        int32_t* __restrict__ windows,
                                        int32_t* __restrict__ k_star, int32_t* __restrict__ status)
{
    // gamma == 1: no drafts, K* = 0, every window is the anchor row alone
    pdl_wait_and_trigger();
    const int tid = threadIdx.x;
    for (int b = tid; b < B; b += blockDim.x) windows[b] = 1;
    if (tid == 0) {
        const double T = (bias + alpha[B]) + theta[B];
        if (!(T > 0.0 && T < INFINITY)) raise_status(status, DSPARK_STATUS_BAD_COST);
        *k_star = 0;
    }
}

// ---- one warp for at most 32 candidates ---------------------------------------------------
// The same outputs as schedule_kernel (and, with PACK, as the pack body) when n = B*(gamma-1)
// <= 32: lane i holds candidate i; the warp sorts the candidates' rank words with a shuffle
// bitonic network (a single request's are in order already), scans their keys, screens every
// K as the block kernel does (one K per lane, K = 0 on a free lane) and, when the screen does
// not decide, evaluates the undecided K exactly in fp64 side by side and reduces with the same
// comparator; no block barrier anywhere. A batch of one request lives here.
constexpr int kSmallMax = 32;

template <bool PACK>
__global__ void __launch_bounds__(32, 1)
schedule_small_kernel(const float* __restrict__ conf, int B, int L, double bias,
                      const double* __restrict__ alpha, const double* __restrict__ theta,
                      int32_t* __restrict__ windows, int32_t* __restrict__ k_star,
                      int32_t* __restrict__ status, PackArgs pk)
{
    __shared__ int cu_s[kSmallMax];
    prefetch_inputs(threadIdx.x, 32, conf, B, L, alpha, theta, PACK ? pk.tokens : nullptr,
                    PACK ? pk.tiers : nullptr, PACK ? pk.n_tiers : 0);
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x;
    const int n = B * L;
    const int gamma = L + 1;
    // inputs: this lane's confidences (its request's first j_own + 1), theta of K = lane + 1
    const uint64_t* theta_bits = reinterpret_cast<const uint64_t*>(theta);
    const bool mine = lane < n;
    const int b_own = mine ? lane / L : 0;
    const int j_own = mine ? lane - b_own * L : -1;
    float c[DSPARK_MAX_GAMMA - 1];
#pragma unroll
    for (int j = 0; j < DSPARK_MAX_GAMMA - 1; ++j)
        if (j <= j_own) c[j] = __ldg(conf + static_cast<int64_t>(b_own) * L + j);
    const uint64_t th_k = mine ? __ldg(theta_bits + B + lane + 1) : 0;
    const uint64_t th_0 = __ldg(theta_bits + B);
    const double t0 = bias + __ldg(alpha + B);
    // the pack's block tokens, B * gamma <= 64 of them: lane l holds tokens l and l + 32
    const int nt = B * gamma;
    const int tok_lo = (PACK && lane < nt) ? __ldg(pk.tokens + lane) : 0;
    const int tok_hi = (PACK && lane + 32 < nt) ? __ldg(pk.tokens + lane + 32) : 0;
    // everything above reads call inputs that no kernel of this library writes; outputs and
    // the tiers (which a pack of this library may have written) wait for the previous kernel
    pdl_wait_and_trigger();
    // the first 64 tiers, loaded now so that the round trip overlaps the scheduling below
    const int tier_lo = (PACK && lane < pk.n_tiers) ? __ldg(pk.tiers + lane) : INT_MAX;
    const int tier_hi = (PACK && lane + 32 < pk.n_tiers) ? __ldg(pk.tiers + lane + 32) : INT_MAX;

    // 1. survival key and rank word of the lane's candidate
    float sv = 1.0f;
#pragma unroll
    for (int j = 0; j < DSPARK_MAX_GAMMA - 1; ++j)
        if (j <= j_own) sv = __fmul_rn(sv, fminf(fmaxf(c[j], 0.0f), 1.0f));   // NaN -> 0
    const uint32_t k32 = sv >= 1.0f ? 0xFFFFFFFFu : __float2uint_rn(__fmul_rn(sv, 4294967296.0f));
    uint64_t w = mine ? rank_word(k32, lane) : 0ull;   // 0 sorts after every candidate

    // 2. bitonic sort of the 32 words, descending. One request's words are in order already:
    // its survivals never grow along the block and its indices rise, so its keys fall or stay
    // and its words fall, with the empty lanes' zeros after them.
    if (B > 1) {
#pragma unroll
        for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
            for (int j = k >> 1; j > 0; j >>= 1) {
                const uint64_t o = __shfl_xor_sync(full, w, j);
                const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
                w = keep_max ? (w > o ? w : o) : (w < o ? w : o);
            }
        }
    }
    const uint32_t kp = static_cast<uint32_t>(w >> 32);
    const int idx = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(w));

    // 3. S(K) for K = lane + 1: inclusive scan of the sorted keys
    uint64_t S = lane < n ? key_value(kp) : 0ull;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t v = __shfl_up_sync(full, S, off);
        if (lane >= off) S += v;
    }

    // 4. screen keys: lane i < n takes K = i + 1 and lane n, when there is one, K = 0 (lane 0
    // takes K = 0 besides K = 1 when n = 32). The warp's best screened K is K* when every
    // other K lies beyond the margin and all were judged; else the exact fp64 objectives of
    // the K not judged or within the margin decide, side by side, one division per lane.
    const uint64_t base_E = static_cast<uint64_t>(B) << 32;
    DF t0d;
    const bool t0_ok = split_double(static_cast<uint64_t>(__double_as_longlong(t0)), t0d);
    const bool own = lane <= n;
    const bool extra0 = n == 32 && lane == 0;
    const int K_own = lane == n ? 0 : lane + 1;
    const uint64_t E_own = lane == n ? base_E : base_E + S;
    const uint64_t th_own = lane == n ? th_0 : th_k;
    const uint64_t key_own = own ? screen_key(E_own, t0d, t0_ok, th_own) : 0;
    const uint64_t key_x = extra0 ? screen_key(base_E, t0d, t0_ok, th_0) : 0;
    uint64_t bk = key_own, b2 = 0;
    int bK = key_own != 0 ? K_own : -1;
    bool nj = (own && key_own == 0) || (extra0 && key_x == 0);
    if (key_x != 0) {                    // K = 0 first among equal keys
        if (key_x >= bk) {
            b2 = bk;
            bk = key_x;
            bK = 0;
        } else {
            b2 = key_x;
        }
    }
    warp_top2(bk, bK, b2, nj);
    const uint64_t thr = bk > kKeyMargin ? bk - kKeyMargin : 0;
    int bits = 0;
    int K_star = bK;
    if (nj || bK < 0 || b2 >= thr) {     // uniform across the warp
        uint64_t best_obj = 0;
        int best_k = -1;
        if (own && (key_own == 0 || key_own >= thr)) {
            const uint64_t o = small_objective(E_own, t0, th_own);
            if (o != 0) {
                best_obj = o;
                best_k = K_own;
            }
        }
        if (extra0 && (key_x == 0 || key_x >= thr)) {
            const uint64_t o = small_objective(base_E, t0, th_0);
            if (o != 0 && better(o, 0, best_obj, best_k)) {
                best_obj = o;
                best_k = 0;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const uint64_t o = __shfl_xor_sync(full, best_obj, off);
            const int kk = __shfl_xor_sync(full, best_k, off);
            if (better(o, kk, best_obj, best_k)) {
                best_obj = o;
                best_k = kk;
            }
        }
        if (best_k < 0) {
            bits |= DSPARK_STATUS_BAD_COST;
            best_k = 0;
        }
        K_star = best_k;
    }

    // 5. windows: 1 + the request's candidates among the first K*
    const bool in = lane < K_star;
    const int req = in ? idx / L : -1;
    int cnt = 0;
    for (int b = 0; b < B; ++b) {
        const int cb = __popc(__ballot_sync(full, req == b));
        if (lane == b) cnt = cb;
    }
    if (lane < B) windows[lane] = 1 + cnt;
    if (lane == 0) *k_star = K_star;

    if (PACK) {
        // front-pack: cu by a warp scan of the windows, tier, rows, padding (as the pack kernel)
        const int wv = lane < B ? 1 + cnt : 0;
        int incl = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(full, incl, off);
            if (lane >= off) incl += v;
        }
        const int M = __shfl_sync(full, incl, 31);
        const int excl = incl - wv;
        if (lane < B) {
            cu_s[lane] = excl;
            pk.cu[lane] = excl;
        }
        if (lane == 0) pk.cu[B] = M;
        int best = INT_MAX;
        if (tier_lo >= M) best = tier_lo;
        if (tier_hi >= M && tier_hi < best) best = tier_hi;
        for (int t = 64 + lane; t < pk.n_tiers; t += 32) {
            const int tv = __ldg(pk.tiers + t);
            if (tv >= M && tv < best) best = tv;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(full, best, off));
        int tier = best;
        if (tier == INT_MAX) {
            tier = M;
            bits |= DSPARK_STATUS_TIER_OVERFLOW;
        }
        if (tier > pk.packed_cap) bits |= DSPARK_STATUS_PACK_CAPACITY;
        __syncwarp();
        const int rows = min(M, pk.packed_cap);
        for (int r0 = 0; r0 < rows; r0 += 32) {          // uniform trip count: shuffles inside
            const int r = r0 + lane;
            int b = 0;
            while (b + 1 < B && r < rows && cu_s[b + 1] <= r) ++b;
            const int i = r - cu_s[b];
            const int q = b * gamma + i;                  // < B * gamma <= 64 for rows < M
            const int t_lo = __shfl_sync(full, tok_lo, q & 31);
            const int t_hi = __shfl_sync(full, tok_hi, q & 31);
            if (r < rows) {
                pk.packed_ids[r] = q < 32 ? t_lo : t_hi;
                if (pk.row_req) pk.row_req[r] = b;
                if (pk.row_pos) pk.row_pos[r] = i;
            }
        }
        const int rows_pad = min(tier, pk.packed_cap);
        for (int r = M + lane; r < rows_pad; r += 32) {
            pk.packed_ids[r] = 0;
            if (pk.row_req) pk.row_req[r] = -1;
            if (pk.row_pos) pk.row_pos[r] = -1;
        }
        if (lane == 0) {
            pk.meta[0] = M;
            pk.meta[1] = tier;
        }
    }
    if (lane == 0) raise_status(status, bits);
}

}  // namespace

namespace {

inline size_t align_to(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launches schedule_kernel<merge, PACK> with the dynamic shared memory its size needs; the
// opt-in limit (static plus dynamic) is configured once per device and variant.
template <bool PACK>
int launch_schedule_kernel(const char* what, const float* conf, int B, int L,
                           const dspark_cost* cost, int32_t* windows, int32_t* k_star,
                           int32_t* status, const PackArgs& pk, cudaStream_t stream)
{
    const int n = B * L;
    int n_pad = 1;
    while (n_pad < n) n_pad <<= 1;
    const bool merge = n <= kMergeMax;
    const bool small = n <= kSmallBlockMax;
    size_t smem = (merge ? 16 * static_cast<size_t>(n) : 8 * static_cast<size_t>(n_pad)) +
                  sizeof(int) * static_cast<size_t>(B);
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != DSPARK_OK) return rc;
    // variants: 0 bitonic (1024 threads), 1 bucket or merge (1024), 2 bucket or merge (256)
    const void* fns[3] = {reinterpret_cast<const void*>(schedule_kernel<false, PACK, 1024>),
                          reinterpret_cast<const void*>(schedule_kernel<true, PACK, 1024>),
                          reinterpret_cast<const void*>(schedule_kernel<true, PACK, 256>)};
    static thread_local int configured_device = -1;
    static thread_local size_t max_dynamic[3] = {0, 0, 0};
    if (configured_device != dev.device) {
        for (int v = 0; v < 3; ++v) {
            cudaFuncAttributes attr;
            if (cudaFuncGetAttributes(&attr, fns[v]) != cudaSuccess)
                return check_launch("schedule (attributes)");
            max_dynamic[v] = static_cast<size_t>(dev.smem_optin) - attr.sharedSizeBytes;
            if (cudaFuncSetAttribute(fns[v], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(max_dynamic[v])) != cudaSuccess)
                return check_launch("schedule (shared-memory opt-in)");
        }
        configured_device = dev.device;
    }
    const int v = !merge ? 0 : small ? 2 : 1;
    if (smem > max_dynamic[v])
        return fail(DSPARK_ERR_UNSUPPORTED, "%s: %zu bytes of shared memory needed, the device "
                    "allows %zu", what, smem, max_dynamic[v]);
    // the pack's tokens staged behind the scheduler's arrays when they fit (16-byte aligned)
    int stage_off = -1;
    if (PACK && reinterpret_cast<uintptr_t>(pk.tokens) % 16 == 0) {
        const size_t off = align_to(smem, 16);
        const size_t need = off + sizeof(int) * static_cast<size_t>(B) * (L + 1);
        if (need <= max_dynamic[v]) {
            stage_off = static_cast<int>(off);
            smem = need;
        }
    }
    if (v == 2)
        return launch_pdl(what, schedule_kernel<true, PACK, 256>, dim3(1), dim3(256), smem,
                          stream, conf, B, L, n, n_pad, cost->bias, cost->alpha, cost->theta,
                          windows, k_star, status, pk, stage_off);
    if (v == 1)
        return launch_pdl(what, schedule_kernel<true, PACK, 1024>, dim3(1), dim3(1024), smem,
                          stream, conf, B, L, n, n_pad, cost->bias, cost->alpha, cost->theta,
                          windows, k_star, status, pk, stage_off);
    return launch_pdl(what, schedule_kernel<false, PACK, 1024>, dim3(1), dim3(1024), smem,
                      stream, conf, B, L, n, n_pad, cost->bias, cost->alpha, cost->theta,
                      windows, k_star, status, pk, stage_off);
}

}  // namespace

int launch_schedule(const float* conf, int B, int gamma, const dspark_cost* cost,
                    int32_t* windows, int32_t* k_star, int32_t* status, cudaStream_t stream)
{
    const int L = gamma - 1;
    if (B * L == 0) {
        return launch_pdl("schedule", schedule_trivial_kernel, dim3(1), dim3(256), 0, stream, B,
                          cost->bias, cost->alpha, cost->theta, windows, k_star, status);
    }
    const PackArgs none = {};
    if (B * L <= kSmallMax)
        return launch_pdl("schedule", schedule_small_kernel<false>, dim3(1), dim3(32), 0, stream,
                          conf, B, L, cost->bias, cost->alpha, cost->theta, windows, k_star,
                          status, none);
    return launch_schedule_kernel<false>("dspark_schedule", conf, B, L, cost, windows, k_star,
                                         status, none, stream);
}

int launch_schedule_pack(const float* conf, int B, int gamma, const dspark_cost* cost,
                         int32_t* windows, int32_t* k_star, const PackArgs& pk, int32_t* status,
                         cudaStream_t stream)
{
    if (B * (gamma - 1) <= kSmallMax)
        return launch_pdl("schedule_pack", schedule_small_kernel<true>, dim3(1), dim3(32), 0,
                          stream, conf, B, gamma - 1, cost->bias, cost->alpha, cost->theta,
                          windows, k_star, status, pk);
    return launch_schedule_kernel<true>("dspark_schedule_pack", conf, B, gamma - 1, cost,
                                        windows, k_star, status, pk, stream);
}

}  // namespace dspark
