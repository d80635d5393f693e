// verify_stream.cu — the HBM-bound part of dspark_verify: one partial per (row, chunk) unit.
//
// Two interchangeable persistent kernels (bit-identical partials: each lane folds its groups in
// the same order through group_update):
//   verify_stream_kernel — register streaming: each warp owns a contiguous run of units and
//     reads each chunk with 16-byte read-only loads, eight in flight per lane (scalar loads
//     when the rows are not 16-byte aligned or V % 8 != 0);
//   verify_bulk_kernel — bulk-copy streaming: one producer warp per CTA moves whole chunks from
//     HBM into a ring of shared-memory stages with cp.async.bulk (the TMA engine), completion
//     counted on an mbarrier per stage; consumer warps fold the staged chunks.
// The default picks the bulk kernel for launches of 64 MB and more at full size, the register
// kernel below that (dspark_set_stream_kernel overrides).
// Verify rules: lshu.cn DSpark article, 1.2 (greedy), 2.3 and 3.3 (min(1, p/q)); modes: "DSpark
// in SGLang" (LMSYS blog summary), A2 verify-mode design.
#include "verify_common.cuh"

namespace dspark {
namespace {

template <int DT, bool STOCH>
__device__ __forceinline__ void chunk_lane(const char* row, int v0, int v1, int vec, float s,
                                           int lane, float& a, float& b, int& idx)
{
    constexpr int E = (DT == DSPARK_BF16) ? 2 : 4;
    constexpr int Q = (DT == DSPARK_BF16) ? 1 : 2;   // uint4 per 8 elements
    uint4 best = make_uint4(0, 0, 0, 0);             // bf16 greedy: vector holding the maximum
    if (vec) {
        const char* base = row + static_cast<int64_t>(v0) * E;
        const int n8 = (v1 - v0) >> 3;               // groups of 8 elements
        for (int g0 = lane; g0 < n8; g0 += 32 * kUnroll) {
            uint4 buf[kUnroll * Q];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int g = g0 + k * 32;
                if (g < n8) {
#pragma unroll
                    for (int h = 0; h < Q; ++h)
                        buf[k * Q + h] = ld_stream16(base + (static_cast<int64_t>(g) * Q + h) * 16);
                }
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int g = g0 + k * 32;
                if (g < n8) group_update<DT, STOCH>(buf + k * Q, v0 + g * 8, s, a, b, idx, best);
            }
        }
        if (!STOCH && DT == DSPARK_BF16 && idx != 0x7FFFFFFF) idx += bf16_first_equal(best, a);
    } else {
        for (int v = v0 + lane; v < v1; v += 32) {
            const float x = load_logit<DT>(row, v);
            if (!STOCH) {
                if (x > a) { a = x; idx = v; }
            } else {
                if (x > a) {
                    b *= ex2_approx((a - x) * s);
                    a = x;
                }
                if (a != -INFINITY) b += ex2_approx((x - a) * s);
            }
        }
    }
}

// Compact batches of fewer requests than this keep cu_seqlens (and the windows) in shared
// memory, so a draft job's owner search costs shared-memory latency, not L2 round trips.
constexpr int kCuCache = 1024;

// Register-streaming variant: any alignment (scalar loads when the rows are not 16-byte
// aligned or V % 8 != 0).
template <int DT, bool STOCH>
__global__ void __launch_bounds__(kStreamThreads)
verify_stream_kernel(StreamArgs A)
{
    constexpr int E = (DT == DSPARK_BF16) ? 2 : 4;
    __shared__ int32_t cu_s[kCuCache];
    __shared__ int32_t w_s[STOCH ? kCuCache : 1];
    pdl_wait_and_trigger();
    zero_next_counters(A);
    const int32_t* cu = A.cu;
    const int32_t* windows = A.windows;
    if (A.mode == DSPARK_COMPACT && A.B < kCuCache) {      // uniform over the CTA
        for (int i = threadIdx.x; i <= A.B; i += kStreamThreads) cu_s[i] = A.cu[i];
        if (STOCH)
            for (int i = threadIdx.x; i < A.B; i += kStreamThreads) w_s[i] = A.windows[i];
        __syncthreads();
        cu = cu_s;
        if (STOCH) windows = w_s;
    }
    const int lane = threadIdx.x & 31;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kStreamWarps + (threadIdx.x >> 5);
    const int64_t GW = static_cast<int64_t>(gridDim.x) * kStreamWarps;
    int64_t n_t;
    const int64_t U = unit_count<STOCH>(A, n_t, cu);

    // At most one unit per warp: warp gw takes unit gw, so whole CTAs are busy and the rest
    // exit at once. Else contiguous runs [gw U / GW, (gw + 1) U / GW), split in 32-bit
    // arithmetic where GW * U fits (the chunk plan keeps U near 4096 units): three 64-bit
    // divisions are long software sequences, most of a warp's work when it holds one unit.
    int64_t u0, u1, job;
    int c;
    if (U <= GW) {
        const uint32_t g = static_cast<uint32_t>(gw);
        const uint32_t q = g / static_cast<uint32_t>(A.nc);
        u0 = gw;
        u1 = gw < U ? gw + 1 : gw;
        job = q;
        c = static_cast<int>(g - q * static_cast<uint32_t>(A.nc));
    } else if (U * GW <= 0x7fffffff) {
        const uint32_t g = static_cast<uint32_t>(gw), W = static_cast<uint32_t>(GW);
        const uint32_t Uu = static_cast<uint32_t>(U);
        const uint32_t a = g * Uu / W, e = (g + 1) * Uu / W;
        const uint32_t q = a / static_cast<uint32_t>(A.nc);
        u0 = a;
        u1 = e;
        job = q;
        c = static_cast<int>(a - q * static_cast<uint32_t>(A.nc));
    } else {
        u0 = gw * U / GW;
        u1 = (gw + 1) * U / GW;
        job = u0 / A.nc;
        c = static_cast<int>(u0 - job * A.nc);
    }
    for (int64_t u = u0; u < u1; ++u) {
        const UnitSrc src = unit_source<E>(A, job, c, n_t, cu, windows);
        if (++c == A.nc) { c = 0; ++job; }
        if (src.skip) continue;
        const int v0 = src.c * A.C;
        const int v1 = min(A.V, v0 + A.C);
        float a = -INFINITY, bsum = 0.0f;
        int idx = 0x7FFFFFFF;
        chunk_lane<DT, STOCH>(src.row, v0, v1, A.vec, A.s, lane, a, bsum, idx);
        write_partial<STOCH>(A, src, lane, a, bsum, idx);
    }
}

// ---- bulk-copy streaming -----------------------------------------------------------------
// A persistent grid (a few CTAs per SM). CTA i streams unit i first; of the remaining units
// the first quarter is split into one contiguous run per CTA and the other three quarters are
// handed out one unit at a time from the counter in the workspace head (an atomic ticket,
// fetched while the previous copy lands), so CTAs on SMs that stream faster, or that started
// later (a step's scheduler holds one SM's registers until it ends), take more of the tail.
// Without a valid head every remaining unit is in the runs. Warp kBulkConsumers is the
// producer: its lane 0, for its k-th unit, waits until stage k % S is free, records the unit
// in the stage's slot, arms the stage's "full" mbarrier with the unit's byte count (the arrive
// publishes the slot) and starts one cp.async.bulk of the whole chunk into the stage; after
// its last unit it posts one end marker per consumer.
// Consumer warp k % kBulkConsumers waits on the full barrier, reads the slot, folds the staged
// chunk with the same per-lane order as the register kernel, releases the stage on its "empty"
// barrier and writes the unit's partial. Every wait is bounded (about a second of SM clock from
// its own start); a wait that gives up sets DSPARK_STATUS_STALL and the producer still waits,
// bounded, for every copy it started before the CTA exits.
// Per-CTA stamps of the large-vocab launch (instrumented copy, L2 flushed) showed why the tail
// is dynamic: with even runs the CTA bodies spanned 46.4 us (the copy peak's rate) but CTAs
// ended between 40.9 and 46.4 us, since SMs stream at rates a few per cent apart. Handing out
// the second half by ticket took the launch from 51.1 to 49.6 us and the high-load cap-accept
// launch from 178 to 170.5 us; a fifth, a third or all of the units by ticket landed within a
// microsecond of that, a tenth or a twentieth gained less (172-174 us at high load); three
// quarters by ticket then shortened the whole large-vocab step by 0.15-0.2 us, all of them
// lengthened it by 0.25 us. Each
// CTA's first unit is fixed so that the head's tag, one L2 or DRAM round trip, is read while
// that unit's copy is in flight instead of before it. (Starting that copy before the PDL wait,
// where the unit is certainly a target row, shortened the bench's chained steps by 0.3-0.6 us
// only by overlapping the schedule-and-pack kernel, which a serving loop separates from verify
// by the target forward; isolated launches did not move. Not kept.)
// Measured on GB300 (whole steps of the large-vocab and high-load workloads): 4 consumer warps,
// chunks of up to 12288 elements and a 96 KB ring (four stages of up to 24 KB, two CTAs per SM,
// eight chunks in flight per SM) beat chunks of 2048-8192 elements in 32-80 KB rings (three or
// four CTAs per SM), chunks of 14336-16384 elements, and 2 or 8 consumers; one CTA per SM
// reached only 4 TB/s.
#ifndef DSPARK_BULK_CONSUMERS
#define DSPARK_BULK_CONSUMERS 4
#endif
constexpr int kBulkConsumers = DSPARK_BULK_CONSUMERS;
constexpr int kBulkThreads = (kBulkConsumers + 1) * 32;
#ifndef DSPARK_BULK_RING_BYTES
#define DSPARK_BULK_RING_BYTES (96 * 1024)
#endif
constexpr int kBulkRingBytes = DSPARK_BULK_RING_BYTES;   // stage ring per CTA
// The bulk kernel serves launches whose full size (B*gamma rows of V logits) reaches this;
// smaller ones are latency-bound and the register kernel starts faster.
constexpr int64_t kBulkMinBytes = 64ll << 20;
constexpr int kBulkMaxStages = 32;
constexpr long long kWaitCycles = 1ll << 31;

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Waits for the completion of the barrier phase of this parity; false once kWaitCycles of SM
// clock have passed since this wait began (each wait has its own limit, so only one phase that
// stalls that long trips it).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    const long long deadline = clock64() + kWaitCycles;
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n"
            " .reg .pred p;\n"
            " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n"
            "}\n"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (clock64() > deadline) return false;
    }
}

// An L2 policy that marks lines for eviction first: the logits are read once, so they should
// not push out of L2 what the step's other kernels use again (their code, the small inputs
// and outputs, the partials).
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Global -> shared copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) by the
// TMA engine under the L2 policy `pol`; completion is counted on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// The producer's source of unit u: the same row as unit_source, with the request of a compact
// draft job tracked by a cursor (units arrive in increasing order) instead of searched per unit.
struct DraftCursor {
    int b = -1;
};

template <int E>
__device__ __forceinline__ const char* bulk_source(const StreamArgs& A, int64_t job, int64_t n_t,
                                                   DraftCursor& cur)
{
    if (job < n_t) return static_cast<const char*>(A.target) + job * A.V * E;
    const int L = A.gamma - 1;
    const int64_t k = job - n_t;
    int b, i;
    if (A.mode == DSPARK_COMPACT) {
        const int64_t r = k;
        if (cur.b < 0) {                          // first draft job: search as unit_source does
            int lo = 0, hi = A.B;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (A.cu[mid] <= r) lo = mid; else hi = mid;
            }
            cur.b = lo;
        }
        while (cur.b + 1 < A.B && A.cu[cur.b + 1] <= r) ++cur.b;
        b = cur.b;
        i = static_cast<int>(r - A.cu[b]);
        int w = A.windows[b];
        w = w < 1 ? 1 : (w > A.gamma ? A.gamma : w);
        if (i < 0 || i >= w - 1 || i >= L) return nullptr;   // last row of a request: no draft
    } else {
        const int kk = static_cast<int>(k);
        b = kk / L;
        i = kk - b * L;
    }
    return static_cast<const char*>(A.draft) + (static_cast<int64_t>(b) * L + i) * A.V * E;
}

template <int DT, bool STOCH>
__global__ void __launch_bounds__(kBulkThreads, 1)
verify_bulk_kernel(StreamArgs A, int stages, int stage_bytes)
{
    constexpr int E = (DT == DSPARK_BF16) ? 2 : 4;
    constexpr int Q = (DT == DSPARK_BF16) ? 1 : 2;   // uint4 per 8 elements
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full_bar[kBulkMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kBulkMaxStages];
    __shared__ int64_t stage_job[kBulkMaxStages];     // the unit each stage holds (row job,
    __shared__ int stage_c[kBulkMaxStages];           // chunk), or job -1: no more units
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_wait_and_trigger();
    zero_next_counters(A);
    int64_t n_t;
    const int64_t U = unit_count<STOCH>(A, n_t, A.cu);

    if (warp == kBulkConsumers) {                     // producer warp: lane 0 issues
        if (lane != 0) return;
        // Units: first unit blockIdx.x, whatever the head says, so the first copy is in flight
        // before the head's tag arrives; then of the rest [G, U) a contiguous run per CTA over
        // the first quarter and tickets for the other three quarters when the head is valid,
        // else runs over all of it. No kernel writes the head while this one runs: every CTA
        // reads one tag.
        const int64_t G = gridDim.x;
        unsigned long long head_w, head_t;            // compared only when first needed
        ws_head_read(A.head, head_w, head_t);
        bool tickets = false;
        int phase = 0;                                // 0: the first unit, 1: the run, 2: tickets
        int64_t u = blockIdx.x, u1 = 0, S = 0;
        unsigned tk = 0;                              // the ticket in flight
        // the next unit into u; false when this CTA has no more
        auto advance = [&]() -> bool {
            if (phase == 0) {
                tickets = ws_head_tags_ok(head_w, head_t);
                const int64_t R = U > G ? U - G : 0;
                S = tickets ? R / 4 : R;
                u = G + static_cast<int64_t>(blockIdx.x) * S / G;
                u1 = G + static_cast<int64_t>(blockIdx.x + 1) * S / G;
                if (tickets) tk = ws_head_ticket(A.head);  // used after the run
                phase = 1;
                if (u < u1) return true;
            } else if (phase == 1) {
                if (++u < u1) return true;
            }
            phase = 2;
            if (!tickets) return false;
            u = G + S + tk;
            if (u >= U) return false;
            tk = ws_head_ticket(A.head);              // travels while this unit's copy lands
            return true;
        };
        bool ok = true;
        DraftCursor cur;
        const uint64_t pol = evict_first_policy();
        int s = 0;
        uint32_t ph = 0;                              // parity of this use of stage s
        int64_t k = 0;
        bool more = u < U || advance();
        for (; more; ++k, more = advance()) {
            int64_t job;
            int c;
            if (u <= 0x7fffffff) {                    // 32-bit division where it fits
                const int q = static_cast<int>(u) / A.nc;
                job = q;
                c = static_cast<int>(u) - q * A.nc;
            } else {
                job = u / A.nc;
                c = static_cast<int>(u - job * A.nc);
            }
            const uint32_t full = smem_addr(&full_bar[s]);
            if (k >= stages && !mbar_wait(smem_addr(&empty_bar[s]), ph ^ 1u)) {
                ok = false;
                break;
            }
            stage_job[s] = job;                       // published by the arrive below
            stage_c[s] = c;
            const char* row = bulk_source<E>(A, job, n_t, cur);
            if (row == nullptr) {
                mbar_arrive(full);                    // a skipped unit: complete the phase
            } else {
                const int v0 = c * A.C;
                const int v1 = min(A.V, v0 + A.C);
                const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * E;
                mbar_arrive_expect_tx(full, bytes);
                bulk_load(smem_addr(ring + static_cast<size_t>(s) * stage_bytes),
                          row + static_cast<int64_t>(v0) * E, bytes, full, pol);
            }
            if (++s == stages) { s = 0; ph ^= 1u; }
        }
        // one end marker per consumer warp (consecutive slots: one for each of them)
        for (int e = 0; ok && e < kBulkConsumers; ++e, ++k) {
            if (k >= stages && !mbar_wait(smem_addr(&empty_bar[s]), ph ^ 1u)) {
                ok = false;
                break;
            }
            stage_job[s] = -1;
            mbar_arrive(smem_addr(&full_bar[s]));
            if (++s == stages) { s = 0; ph ^= 1u; }
        }
        // every started copy must land before this CTA may exit
        const int64_t issued = k;
        for (int s = 0; s < stages && s < issued; ++s) {
            const int64_t uses = (issued - s + stages - 1) / stages;
            if (!mbar_wait(smem_addr(&full_bar[s]), static_cast<uint32_t>((uses - 1) & 1)))
                ok = false;
        }
        if (!ok) raise_status(A.status, DSPARK_STATUS_STALL);
        return;
    }

    int s = warp;                                     // stages % kBulkConsumers == 0
    uint32_t ph = 0;
    while (true) {
        const bool ok = mbar_wait(smem_addr(&full_bar[s]), ph);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) raise_status(A.status, DSPARK_STATUS_STALL);
            break;
        }
        const int64_t job = stage_job[s];
        const int c = stage_c[s];
        if (job < 0) break;                           // the producer's end marker
        const UnitSrc src = unit_source<E>(A, job, c, n_t, A.cu, A.windows);
        float a = -INFINITY, bsum = 0.0f;
        int idx = 0x7FFFFFFF;
        if (!src.skip) {
            const int v0 = src.c * A.C;
            const int n8 = (min(A.V, v0 + A.C) - v0) >> 3;
            const uint4* q = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(s) * stage_bytes);
            uint4 best = make_uint4(0, 0, 0, 0);
            for (int g = lane; g < n8; g += 32) {
                uint4 v[Q];
#pragma unroll
                for (int h = 0; h < Q; ++h) v[h] = q[g * Q + h];
                group_update<DT, STOCH>(v, v0 + g * 8, A.s, a, bsum, idx, best);
            }
            if (!STOCH && DT == DSPARK_BF16 && idx != 0x7FFFFFFF) idx += bf16_first_equal(best, a);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
        if (!src.skip) write_partial<STOCH>(A, src, lane, a, bsum, idx);
        s += kBulkConsumers;
        if (s >= stages) { s -= stages; ph ^= 1u; }
    }
}

}  // namespace

namespace {

int g_stream_kernel = DSPARK_STREAM_AUTO;   // dspark_set_stream_kernel
cudaEvent_t g_ev_start = nullptr;           // dspark_set_stream_events
cudaEvent_t g_ev_stop = nullptr;

template <int DT, bool STOCH>
int launch_stream_t(const StreamArgs& sa, int64_t max_units, cudaStream_t stream)
{
    constexpr int E = (DT == DSPARK_BF16) ? 2 : 4;
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != DSPARK_OK) return rc;
    int which = g_stream_kernel;
    if (which == DSPARK_STREAM_AUTO)
        which = sa.rows_max * sa.V * E >= kBulkMinBytes ? DSPARK_STREAM_BULK : DSPARK_STREAM_REGISTER;
    if (which == DSPARK_STREAM_BULK && sa.vec) {
        const int stage_bytes = static_cast<int>(align_up(static_cast<size_t>(sa.C) * E, 128));
        int stages = (kBulkRingBytes / stage_bytes) / kBulkConsumers * kBulkConsumers;
        if (stages > kBulkMaxStages) stages = kBulkMaxStages;
        if (stages >= kBulkConsumers) {
            const size_t smem = static_cast<size_t>(stages) * stage_bytes;
            static thread_local int bulk_device = -1;
            static thread_local int bulk_occ = 0;
            if (bulk_device != dev.device) {
                if (cudaFuncSetAttribute(verify_bulk_kernel<DT, STOCH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kBulkRingBytes) != cudaSuccess)
                    return check_launch("verify (bulk stream shared-memory opt-in)");
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &bulk_occ, verify_bulk_kernel<DT, STOCH>, kBulkThreads, kBulkRingBytes) !=
                    cudaSuccess)
                    return check_launch("verify (bulk stream occupancy query)");
                if (bulk_occ < 1) bulk_occ = 1;
                bulk_device = dev.device;
            }
            int64_t grid = static_cast<int64_t>(dev.sm_count) * bulk_occ;
            const int64_t need = ceil_div(max_units, kBulkConsumers);
            if (grid > need) grid = need;
            if (grid < 1) grid = 1;
            return launch_pdl("verify (bulk stream)", verify_bulk_kernel<DT, STOCH>,
                              dim3(static_cast<unsigned>(grid)), dim3(kBulkThreads), smem, stream,
                              sa, stages, stage_bytes);
        }
    }
    static thread_local int occ_device = -1;
    static thread_local int occ = 0;
    if (occ_device != dev.device) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, verify_stream_kernel<DT, STOCH>,
                                                          kStreamThreads, 0) != cudaSuccess)
            return check_launch("verify (occupancy query)");
        if (occ < 1) occ = 1;
        occ_device = dev.device;
    }
    int64_t grid = static_cast<int64_t>(dev.sm_count) * occ;
    const int64_t need = ceil_div(max_units, kStreamWarps);
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    return launch_pdl("verify (stream)", verify_stream_kernel<DT, STOCH>,
                      dim3(static_cast<unsigned>(grid)), dim3(kStreamThreads), 0, stream, sa);
}

}  // namespace

int set_stream_kernel(int which)
{
    if (which != DSPARK_STREAM_AUTO && which != DSPARK_STREAM_REGISTER && which != DSPARK_STREAM_BULK)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_set_stream_kernel: unknown kernel %d", which);
    g_stream_kernel = which;
    return DSPARK_OK;
}

void set_stream_events(cudaEvent_t start, cudaEvent_t stop)
{
    g_ev_start = start;
    g_ev_stop = stop;
}

int launch_verify_stream(int dtype, bool stochastic, const StreamArgs& sa, int64_t max_units,
                         cudaStream_t stream)
{
    if (g_ev_start != nullptr && cudaEventRecord(g_ev_start, stream) != cudaSuccess)
        return check_launch("verify (stream start event)");
    int rc;
    if (dtype == DSPARK_BF16)
        rc = stochastic ? launch_stream_t<DSPARK_BF16, true>(sa, max_units, stream)
                        : launch_stream_t<DSPARK_BF16, false>(sa, max_units, stream);
    else
        rc = stochastic ? launch_stream_t<DSPARK_F32, true>(sa, max_units, stream)
                        : launch_stream_t<DSPARK_F32, false>(sa, max_units, stream);
    if (rc == DSPARK_OK && g_ev_stop != nullptr && cudaEventRecord(g_ev_stop, stream) != cudaSuccess)
        return check_launch("verify (stream stop event)");
    return rc;
}

}  // namespace dspark
