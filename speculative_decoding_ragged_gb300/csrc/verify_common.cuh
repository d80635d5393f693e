// verify_common.cuh — what the two logit-streaming kernels of dspark_verify share: the fixed
// chunk plan, the unit list (row, chunk), the per-group fold of a lane and the chunk partials
// the finaliser combines.
//
// Every logits row is cut into nc chunks at fixed offsets (c * C, C a multiple of 8 elements
// chosen from V and B*gamma only, never from M), so a row's statistics are bit-identical
// wherever the row sits in the buffer: compact and cap-accept see the same numbers for the same
// row. A unit is one chunk of one row; its partial is
//   greedy:     (max value, lowest index of it)
//   stochastic: (max logit m, sum of exp2((l - m) * log2(e)/T)) — an online softmax.
#pragma once
#include <math.h>

#include "common.cuh"

namespace dspark {

constexpr int kStreamThreads = 256;
constexpr int kStreamWarps = kStreamThreads / 32;
#ifndef DSPARK_UNROLL
#define DSPARK_UNROLL 8
#endif
constexpr int kUnroll = DSPARK_UNROLL;  // 16-byte loads in flight per lane
constexpr int kTargetUnits = 4096;    // aim: about one unit per resident warp
// blocks of at most kSmallRows rows (batch-1 decoding) aim lower: fewer, larger units and fewer
// partials per row for the finaliser shortened the batch-1 step by 3-4 % on GB300
constexpr int kSmallRows = 64;
constexpr int kTargetUnitsSmall = 1024;
#ifndef DSPARK_MAX_CHUNK
#define DSPARK_MAX_CHUNK 12288
#endif
constexpr int kMaxChunk = DSPARK_MAX_CHUNK;   // elements per chunk, upper bound (24 KB of bf16)
#ifndef DSPARK_MIN_CHUNK
#define DSPARK_MIN_CHUNK 256
#endif
constexpr int kMinChunk = DSPARK_MIN_CHUNK;   // elements per chunk, lower bound

struct __align__(8) ArgPart {
    float v;
    int idx;
};
struct __align__(8) SoftPart {
    float m;   // chunk maximum of the raw logits
    float z;   // sum over the chunk of exp2((l - m) * log2(e) / T)
};

struct Plan {
    int nc;       // chunks per row
    int C;        // elements per chunk (multiple of 8)
    int64_t rows_max;
};

inline Plan make_plan(int V, int B, int gamma)
{
    Plan p;
    p.rows_max = static_cast<int64_t>(B) * gamma;
    const int64_t nc_min = ceil_div(V, kMaxChunk);
    const int64_t nc_max = V / kMinChunk > 0 ? V / kMinChunk : 1;
    const int64_t target = p.rows_max <= kSmallRows ? kTargetUnitsSmall : kTargetUnits;
    const int64_t nc_want = ceil_div(target, p.rows_max > 0 ? p.rows_max : 1);
    int64_t nc = nc_want < nc_max ? nc_want : nc_max;
    if (nc < nc_min) nc = nc_min;
    int64_t C = ceil_div(ceil_div(V, nc), 8) * 8;
    p.C = static_cast<int>(C);
    p.nc = static_cast<int>(ceil_div(V, C));
    return p;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The first kWsHeadBytes of a verify workspace: state that one call hands to the next. The
// bulk-copy streaming kernel splits half of its units evenly over its CTAs and hands out the
// other half one at a time from a counter here, so CTAs that stream faster take more of the
// tail. The counter is the high half of the head's first 8-byte word; its low half and the
// second word hold tags. The call's last kernel, which starts only after the streaming kernel
// has completed, leaves the counter at 0 with both tags for the next call. A streaming kernel
// that finds either tag missing (a fresh or cleared workspace, or a former workspace whose
// first bytes another tensor has since written) splits all of its units evenly instead: the
// same partials, only the balance of the tail differs. Tickets add 2^32 to the first word, so
// the low tag never changes while a kernel runs and every CTA reaches the same decision.
struct WsHead {
    unsigned long long word;       // low 32 bits: kWsHeadTag32; high 32 bits: units handed out
    unsigned long long tag;        // kWsHeadTag64
};
constexpr size_t kWsHeadBytes = 256;
constexpr unsigned long long kWsHeadTag32 = 0xd2b8f605ull;
constexpr unsigned long long kWsHeadTag64 = 0x7c3a91e44e1f63a9ull;

// The head's two words (read once per CTA after its wait; volatile: another call wrote them),
// and whether they carry both tags, i.e. were left by a call.
__device__ __forceinline__ void ws_head_read(const WsHead* h, unsigned long long& w,
                                             unsigned long long& t)
{
    w = 0;
    t = 0;
    if (h != nullptr) {
        w = *reinterpret_cast<const volatile unsigned long long*>(&h->word);
        t = *reinterpret_cast<const volatile unsigned long long*>(&h->tag);
    }
}
__device__ __forceinline__ bool ws_head_tags_ok(unsigned long long w, unsigned long long t)
{
    return (w & 0xffffffffull) == kWsHeadTag32 && t == kWsHeadTag64;
}

// The next unit ticket of the dynamic half (a relaxed add of one to the counter).
__device__ __forceinline__ unsigned ws_head_ticket(WsHead* h)
{
    return static_cast<unsigned>(atomicAdd(&h->word, 1ull << 32) >> 32);
}

// Leaves the workspace head ready for the next call (one thread of the call's last kernel,
// after that kernel's wait for the streaming kernel).
__device__ __forceinline__ void reset_ws_head(WsHead* h)
{
    if (h != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
        h->word = kWsHeadTag32;
        h->tag = kWsHeadTag64;
    }
}

struct StreamArgs {
    const void* target;
    const void* draft;
    const int32_t* cu;
    const int32_t* windows;
    void* part_t;
    void* part_d;
    int32_t* status;
    unsigned* zero;   // counters of the call's next kernel, zeroed here (nullptr: none)
    int n_zero;
    WsHead* head;     // the workspace head (bulk kernel's unit counter)
    int mode, V, nc, C, vec, B, gamma, target_rows;
    int64_t rows_max;
    float s;   // log2(e) / temperature
};

// Zeroes the counters the call's next kernel counts on: that kernel waits for this one to
// complete before it reads them, and this one waited for the previous call's kernels.
__device__ __forceinline__ void zero_next_counters(const StreamArgs& A)
{
    if (A.zero != nullptr && blockIdx.x == 0)
        for (int i = threadIdx.x; i < A.n_zero; i += blockDim.x) A.zero[i] = 0u;
}

// Rows this call verifies: compact M = cu[B] (bounded by the buffer), else B*gamma.
__device__ __forceinline__ int64_t target_row_count(int mode, const int32_t* cu, int B, int gamma,
                                                    int target_rows, int64_t rows_max)
{
    int64_t n;
    if (mode == DSPARK_COMPACT) n = cu[B];
    else n = static_cast<int64_t>(B) * gamma;
    if (n < 0) n = 0;
    if (n > target_rows) n = target_rows;
    if (n > rows_max) n = rows_max;
    return n;
}

__device__ __forceinline__ void arg_merge(float& v, int& i, float v2, int i2)
{
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

// ---- per-element kernels of a chunk ---------------------------------------------------
template <int DT>
__device__ __forceinline__ void unpack8(const uint4* q, int k, float (&x)[8]);

template <>
__device__ __forceinline__ void unpack8<DSPARK_BF16>(const uint4* q, int k, float (&x)[8])
{
    const uint4 u = q[k];
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x);
    x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z);
    x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

template <>
__device__ __forceinline__ void unpack8<DSPARK_F32>(const uint4* q, int k, float (&x)[8])
{
    const uint4 a = q[2 * k], b = q[2 * k + 1];
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
}

// Packed fp32 pairs for the f32x2 instructions (two round-to-nearest operations in one).
__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float lo2(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo;
}
__device__ __forceinline__ float hi2(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return hi;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Exact maximum of the 8 bf16 logits of a 16-byte vector, widened to fp32 (max.bf16x2 does not
// round; NaN inputs are unsupported).
__device__ __forceinline__ float bf16x2_max_of(const uint4 u)
{
    uint32_t m01, m23, m;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m01) : "r"(u.x), "r"(u.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m23) : "r"(u.z), "r"(u.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m01), "r"(m23));
    return fmaxf(bf16_lo(m), bf16_hi(m));
}

// Index of the first of the 8 bf16 logits of `u` equal to `a`, the vector's maximum.
__device__ __forceinline__ int bf16_first_equal(const uint4 u, float a)
{
    const float x[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                        bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
    int e = 0;
#pragma unroll
    for (int k = 7; k >= 0; --k)
        if (x[k] == a) e = k;
    return e;
}
// One group of 8 consecutive logits (Q 16-byte vectors at q, first index vb) folded into a
// lane's running state: greedy keeps (maximum, index, and for bf16 the vector holding the
// maximum, resolved to an index once per chunk by bf16_first_equal); stochastic keeps (maximum
// m, sum of exp2((l - m) * s)). A lane visits its groups in increasing index order, so a strict
// '>' keeps the lowest index of its maximum. Both streaming kernels fold through this one
// routine in the same order, so their chunk partials are bit-identical.
// The stochastic fold runs its subtractions, scalings and sums on pairs of fp32 values
// (add/mul.rn.f32x2: each half rounds as its scalar operation would) and takes the group's
// maximum with max.bf16x2: a quarter fewer instructions per group, which took the stochastic
// workload's chained verify call from 14.7 to 14.1 us (compact) and 17.8 to 17.1 us
// (cap-accept) on GB300; the workload is latency-bound and its fold runs in bursts as the
// chunks land.
template <int DT, bool STOCH>
__device__ __forceinline__ void group_update(const uint4* q, int vb, float s, float& a, float& b,
                                             int& idx, uint4& best)
{
    float x[8];
    unpack8<DT>(q, 0, x);
    if (!STOCH) {
        if (DT == DSPARK_BF16) {
            // exact packed max of the 8 bf16 values; the index is resolved once per chunk from
            // the first vector holding the lane's maximum
            const uint4 u = q[0];
            const float vm = bf16x2_max_of(u);
            if (vm > a) { a = vm; best = u; idx = vb; }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (x[e] > a) { a = x[e]; idx = vb + e; }
        }
    } else {
        float vm;
        if (DT == DSPARK_BF16) vm = bf16x2_max_of(q[0]);
        else vm = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                        fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
        if (vm > a) {
            b *= ex2_approx((a - vm) * s);
            a = vm;
        }
        if (a != -INFINITY) {
            // (x - a) * s and the sum in packed pairs (add/mul.rn.f32x2): element pairs
            // (0,1) (2,3) (4,5) (6,7); the sum pairs them as ((t0+t2)+(t4+t6)) + ((t1+t3)+(t5+t7))
            const uint64_t na = pack2(-a, -a), s2 = pack2(s, s);
            uint64_t d[4];
            float t[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                d[h] = mul2(add2(pack2(x[2 * h], x[2 * h + 1]), na), s2);
                t[2 * h] = ex2_approx(lo2(d[h]));
                t[2 * h + 1] = ex2_approx(hi2(d[h]));
            }
            const uint64_t r = add2(add2(pack2(t[0], t[1]), pack2(t[2], t[3])),
                                    add2(pack2(t[4], t[5]), pack2(t[6], t[7])));
            b += lo2(r) + hi2(r);
        }
    }
}

// Where unit (job row, chunk c) reads from and where its partial goes; the flat unit index is
// u = job * nc + c, and the kernels walk (job, c) incrementally (64-bit divisions are long
// software sequences). Draft jobs of the last row of a compact request have no draft (skip).
struct UnitSrc {
    const char* row;
    int64_t slot;   // partial index = (paired target row) * nc + c
    int c;
    bool draft;
    bool skip;
};

template <int E>
__device__ __forceinline__ UnitSrc unit_source(const StreamArgs& A, int64_t job, int c, int64_t n_t,
                                               const int32_t* cu, const int32_t* windows)
{
    UnitSrc s;
    s.c = c;
    s.skip = false;
    s.draft = job >= n_t;
    if (!s.draft) {
        s.row = static_cast<const char*>(A.target) + job * A.V * E;
        s.slot = job * A.nc + s.c;
        return s;
    }
    const int L = A.gamma - 1;
    const int64_t k = job - n_t;
    int b, i;
    int64_t r;
    if (A.mode == DSPARK_COMPACT) {
        r = k;                                   // draft job of packed row r
        int lo = 0, hi = A.B;                    // largest b with cu[b] <= r
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu[mid] <= r) lo = mid; else hi = mid;
        }
        b = lo;
        i = static_cast<int>(r - cu[b]);
        int w = windows[b];
        w = w < 1 ? 1 : (w > A.gamma ? A.gamma : w);
        if (i < 0 || i >= w - 1 || i >= L) {     // last row of a request: no draft
            s.skip = true;
            s.row = nullptr;
            s.slot = 0;
            return s;
        }
    } else {
        const int kk = static_cast<int>(k);      // k < B*(gamma-1) < 2^31
        b = kk / L;
        i = kk - b * L;
        r = static_cast<int64_t>(b) * A.gamma + i;
    }
    s.row = static_cast<const char*>(A.draft) + (static_cast<int64_t>(b) * L + i) * A.V * E;
    s.slot = r * A.nc + s.c;
    return s;
}

// Units this call streams: target rows, then (stochastic) the draft jobs.
template <bool STOCH>
__device__ __forceinline__ int64_t unit_count(const StreamArgs& A, int64_t& n_t, const int32_t* cu)
{
    n_t = target_row_count(A.mode, cu, A.B, A.gamma, A.target_rows, A.rows_max);
    int64_t n_d = 0;
    if (STOCH) n_d = (A.mode == DSPARK_COMPACT) ? n_t : static_cast<int64_t>(A.B) * (A.gamma - 1);
    return (n_t + n_d) * A.nc;
}

// Warp-level end of a unit: reduce the lanes' running values and write the unit's partial.
template <bool STOCH>
__device__ __forceinline__ void write_partial(const StreamArgs& A, const UnitSrc& src, int lane,
                                              float a, float bsum, int idx)
{
    if (!STOCH) {
        for (int off = 16; off > 0; off >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, a, off);
            const int i2 = __shfl_xor_sync(0xffffffffu, idx, off);
            arg_merge(a, idx, v2, i2);
        }
        if (lane == 0) {
            ArgPart p;
            p.v = a;
            p.idx = idx;
            static_cast<ArgPart*>(A.part_t)[src.slot] = p;
        }
    } else {
        float m = a;
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        // fp32 tree over the 32 lanes (FP64 throughput is scarce on this part)
        float z = a != -INFINITY ? bsum * ex2_approx((a - m) * A.s) : 0.0f;
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        if (lane == 0) {
            SoftPart p;
            p.m = m;
            p.z = z;
            static_cast<SoftPart*>(src.draft ? A.part_d : A.part_t)[src.slot] = p;
        }
    }
}

// Launches the streaming kernel for these arguments (the register kernel, or the bulk-copy
// kernel when the rows are 16-byte aligned and the chunk fits its shared-memory stages).
// max_units bounds the units of any M (the grid is sized from it, never from M).
int launch_verify_stream(int dtype, bool stochastic, const StreamArgs& sa, int64_t max_units,
                         cudaStream_t stream);

}  // namespace dspark
