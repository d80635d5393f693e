// pack.cu — the ragged front-pack as one single-CTA kernel of 1024 threads.
//
// "DSpark in SGLang" (LMSYS blog summary), A2, ragged verify over full CUDA graphs: the
// variable windows are front-packed into one compact cu_seqlens-style buffer and only the
// total is rounded up to the nearest captured graph tier, so a smaller budget replays a truly
// smaller graph; padding rows up to the tier are waste (figure 2).
//
//   1. every load is issued up front: each thread's windows and one tier per thread
//      (n_tiers <= 1024), so the block pays one memory round trip;
//   2. windows clamped to [1, gamma]; block-wide exclusive scan -> cu_seqlens;
//   3. tier = min over tiers >= M (tiers need not be sorted);
//   4. cu_seqlens into shared memory; then each thread writes whole rows (token, request,
//      position), finding a row's request by binary search over cu, so that the stores of a
//      warp are contiguous; padding rows up to the tier get 0 / -1 / -1.
// (dspark_schedule_pack packs on the scheduler's own CTA instead, in schedule.cu.)
#include "common.cuh"

namespace dspark {
namespace {

constexpr int kPackThreads = 1024;

__device__ __forceinline__ int pack_load_window(const int32_t* __restrict__ windows, int b)
{
    return __ldg(windows + b);
}

__device__ __forceinline__ void pack_block(const int32_t* windows, const int32_t* __restrict__ tokens,
                                           int B, int gamma, const int32_t* __restrict__ tiers,
                                           int n_tiers, int32_t* __restrict__ cu_out,
                                           int32_t* __restrict__ packed_ids,
                                           int32_t* __restrict__ row_req,
                                           int32_t* __restrict__ row_pos, int packed_cap,
                                           int32_t* __restrict__ meta, int32_t* __restrict__ status)
{
    constexpr int kWarps = kPackThreads / 32;
    __shared__ int warp_total[kWarps];
    __shared__ int tier_s;
    __shared__ int cu_s[DSPARK_MAX_BATCH + 1];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    // 1. loads
    const int tier_v = tid < n_tiers ? __ldg(tiers + tid) : INT_MAX;
    const int items = (B + kPackThreads - 1) / kPackThreads;
    const int b0 = tid * items;
    int w_first = 1;
    if (items == 1 && b0 < B) w_first = pack_load_window(windows, b0);
    if (tid == 0) tier_s = INT_MAX;

    // 2. exclusive scan of the clamped windows
    int bad = 0;
    int run = 0;
    for (int it = 0; it < items; ++it) {
        const int b = b0 + it;
        if (b >= B) break;
        int w = items == 1 ? w_first : pack_load_window(windows, b);
        if (w < 1 || w > gamma) {
            bad = DSPARK_STATUS_BAD_WINDOW;
            w = w < 1 ? 1 : gamma;
        }
        run += w;
    }
    int incl = run;
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_total[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int t = warp_total[lane];
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += v;
        }
        warp_total[lane] = t;
    }
    __syncthreads();
    const int M = warp_total[kWarps - 1];
    const int excl = incl - run + (warp > 0 ? warp_total[warp - 1] : 0);

    // 3. tier
    int best = tier_v >= M ? tier_v : INT_MAX;
    for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
    if (lane == 0 && best != INT_MAX) atomicMin(&tier_s, best);
    __syncthreads();
    int tier = tier_s;
    if (tier == INT_MAX) {
        tier = M;
        bad |= DSPARK_STATUS_TIER_OVERFLOW;
    }
    if (tier > packed_cap) bad |= DSPARK_STATUS_PACK_CAPACITY;

    // 4. cu_seqlens, then the rows: row r belongs to the largest b with cu[b] <= r
    int acc = excl;
    for (int it = 0; it < items; ++it) {
        const int b = b0 + it;
        if (b >= B) break;
        int w = items == 1 ? w_first : pack_load_window(windows, b);
        w = w < 1 ? 1 : (w > gamma ? gamma : w);
        cu_s[b] = acc;
        cu_out[b] = acc;
        acc += w;
    }
    if (tid == 0) cu_out[B] = M;
    __syncthreads();
    const int rows = min(M, packed_cap);
    for (int r = tid; r < rows; r += kPackThreads) {
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu_s[mid] <= r) lo = mid; else hi = mid;
        }
        const int i = r - cu_s[lo];
        const int64_t ti = static_cast<int64_t>(lo) * gamma + i;
        packed_ids[r] = __ldg(tokens + ti);
        if (row_req) row_req[r] = lo;
        if (row_pos) row_pos[r] = i;
    }
    const int rows_pad = min(tier, packed_cap);
    for (int r = M + tid; r < rows_pad; r += kPackThreads) {
        packed_ids[r] = 0;
        if (row_req) row_req[r] = -1;
        if (row_pos) row_pos[r] = -1;
    }
    if (tid == 0) {
        meta[0] = M;
        meta[1] = tier;
    }
    // status bits of every thread
    const unsigned any = __ballot_sync(0xffffffffu, bad != 0);
    if (any) {
        int bits = bad;
        for (int off = 16; off > 0; off >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, off);
        if (lane == 0) raise_status(status, bits);
    }
}

__global__ void __launch_bounds__(kPackThreads, 1)
pack_kernel(const int32_t* __restrict__ windows, const int32_t* __restrict__ tokens, int B,
            int gamma, const int32_t* __restrict__ tiers, int n_tiers,
            int32_t* __restrict__ cu_out, int32_t* __restrict__ packed_ids,
            int32_t* __restrict__ row_req, int32_t* __restrict__ row_pos, int packed_cap,
            int32_t* __restrict__ meta, int32_t* __restrict__ status)
{
    pdl_wait_and_trigger();
    pack_block(windows, tokens, B, gamma, tiers, n_tiers, cu_out, packed_ids, row_req,
                     row_pos, packed_cap, meta, status);
}

}  // namespace

int launch_pack(const int32_t* windows, const int32_t* tokens, int B, int gamma,
                const int32_t* tiers, int n_tiers, int32_t* cu, int32_t* packed_ids,
                int32_t* row_req, int32_t* row_pos, int packed_cap, int32_t* meta,
                int32_t* status, cudaStream_t stream)
{
    return launch_pdl("pack", pack_kernel, dim3(1), dim3(kPackThreads), 0, stream, windows, tokens, B,
                      gamma, tiers, n_tiers, cu, packed_ids, row_req, row_pos, packed_cap, meta,
                      status);
}

}  // namespace dspark
