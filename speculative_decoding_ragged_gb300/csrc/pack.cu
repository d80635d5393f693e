// pack.cu — ragged front-pack as one single-CTA kernel.
//
// "DSpark in SGLang" (LMSYS blog summary), A2, ragged verify over full CUDA graphs: the
// variable windows are front-packed into one compact cu_seqlens-style buffer and only the
// total is rounded up to the nearest captured graph tier, so a smaller budget replays a truly
// smaller graph; padding rows up to the tier are waste (figure 2).
//
//   1. windows clamped to [1, gamma]; block-wide exclusive scan -> cu_seqlens (in smem too);
//   2. tier = min over tiers >= M (block min; tiers need not be sorted);
//   3. one thread per packed row: binary search of cu_seqlens gives (b, i); write the token
//      and the row's (request, position); padding rows up to the tier get 0 / -1 / -1.
#include "common.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads, 1)
pack_kernel(const int32_t* __restrict__ windows, const int32_t* __restrict__ tokens, int B,
            int gamma, const int32_t* __restrict__ tiers, int n_tiers,
            int32_t* __restrict__ cu_out, int32_t* __restrict__ packed_ids,
            int32_t* __restrict__ row_req, int32_t* __restrict__ row_pos, int packed_cap,
            int32_t* __restrict__ meta, int32_t* __restrict__ status)
{
    extern __shared__ int cu[];   // [B + 1]
    __shared__ int warp_total[kWarps];
    __shared__ int tier_s;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    if (tid == 0) tier_s = INT_MAX;
    // 1. exclusive scan; thread t owns requests [t*items, (t+1)*items)
    const int items = (B + kThreads - 1) / kThreads;
    const int b0 = tid * items;
    int bad = 0;
    int run = 0;
    for (int it = 0; it < items; ++it) {
        const int b = b0 + it;
        if (b >= B) break;
        int w = windows[b];
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
    int acc = incl - run + (warp > 0 ? warp_total[warp - 1] : 0);
    for (int it = 0; it < items; ++it) {
        const int b = b0 + it;
        if (b >= B) break;
        int w = windows[b];
        w = w < 1 ? 1 : (w > gamma ? gamma : w);
        cu[b] = acc;
        cu_out[b] = acc;
        acc += w;
    }
    const int M = warp_total[kWarps - 1];
    if (tid == 0) {
        cu[B] = M;
        cu_out[B] = M;
    }
    // 2. tier
    int best = INT_MAX;
    for (int t = tid; t < n_tiers; t += kThreads) {
        const int v = tiers[t];
        if (v >= M && v < best) best = v;
    }
    for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
    if (lane == 0 && best != INT_MAX) atomicMin(&tier_s, best);
    __syncthreads();
    int tier = tier_s;
    if (tier == INT_MAX) {
        tier = M;
        bad |= DSPARK_STATUS_TIER_OVERFLOW;
    }
    if (tier > packed_cap) bad |= DSPARK_STATUS_PACK_CAPACITY;

    // 3. packed rows
    const int rows_real = min(M, packed_cap);
    for (int r = tid; r < rows_real; r += kThreads) {
        int lo = 0, hi = B;   // largest b with cu[b] <= r
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu[mid] <= r) lo = mid; else hi = mid;
        }
        const int i = r - cu[lo];
        packed_ids[r] = tokens[static_cast<int64_t>(lo) * gamma + i];
        if (row_req) row_req[r] = lo;
        if (row_pos) row_pos[r] = i;
    }
    const int rows_pad = min(tier, packed_cap);
    for (int r = M + tid; r < rows_pad; r += kThreads) {
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

}  // namespace

int launch_pack(const int32_t* windows, const int32_t* tokens, int B, int gamma,
                const int32_t* tiers, int n_tiers, int32_t* cu, int32_t* packed_ids,
                int32_t* row_req, int32_t* row_pos, int packed_cap, int32_t* meta,
                int32_t* status, cudaStream_t stream)
{
    const size_t smem = sizeof(int) * static_cast<size_t>(B + 1);
    pack_kernel<<<1, kThreads, smem, stream>>>(windows, tokens, B, gamma, tiers, n_tiers, cu,
                                               packed_ids, row_req, row_pos, packed_cap, meta,
                                               status);
    return check_launch("pack");
}

}  // namespace dspark
