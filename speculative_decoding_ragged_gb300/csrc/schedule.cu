// schedule.cu — the confidence scheduler as one single-CTA kernel.
//
// "DSpark in SGLang: Speculative Decoding with Confidence-Driven, Variable-Length Verification"
// (LMSYS blog summary), A2 method details: the confidence head's scores multiply along the
// block into a survival probability; the scheduler reads the additive cost table
// T(bs,K) = bias + alpha(bs) + theta(bs+K) online and picks the verify budget that maximises
// expected committed tokens per unit of step time, which yields a window per request.
//
// Work: n = B*(gamma-1) <= 16384 candidates, all in shared memory of one CTA.
//   1. survivals -> fixed-point keys, packed with their index into unique 64-bit sort words
//      word = key << 31 | (2^31 - 1 - index), so descending words = keys descending, then
//      index ascending (index = b*(gamma-1) + j orders requests, then positions);
//   2. bitonic sort of the padded power-of-two array, descending;
//   3. block-wide inclusive scan of the keys (exact uint64 sums S(K));
//   4. obj(K) = double(B*2^32 + S(K)) / T(K) and a block argmax (smallest K on ties);
//   5. windows w_b = 1 + count of request b among the first K* words.
// Latency-bound (microseconds); the grid is one CTA by construction of the problem.
#include "common.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ bool better(double o1, int k1, double o2, int k2)
{
    // larger objective; on equal objectives the smaller K (k = -1 means "none": loses ties)
    return o1 > o2 || (o1 == o2 && static_cast<unsigned>(k1) < static_cast<unsigned>(k2));
}

__global__ void __launch_bounds__(kThreads, 1)
schedule_kernel(const float* __restrict__ conf, int B, int L, int n, int n_pad, double bias,
                const double* __restrict__ alpha, const double* __restrict__ theta,
                int32_t* __restrict__ windows, int32_t* __restrict__ k_star,
                int32_t* __restrict__ status)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint64_t* word = reinterpret_cast<uint64_t*>(smem_raw);   // [n_pad]
    int* count = reinterpret_cast<int*>(word + n_pad);          // [B]
    __shared__ uint64_t warp_total[kWarps];
    __shared__ double red_obj[kWarps];
    __shared__ int red_k[kWarps];
    __shared__ int k_best;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;

    // 1. survival keys, one request per thread (the product is sequential along j)
    for (int b = tid; b < B; b += kThreads) {
        float s = 1.0f;
        for (int j = 0; j < L; ++j) {
            const int idx = b * L + j;
            const float c = fminf(fmaxf(conf[idx], 0.0f), 1.0f);   // NaN -> 0
            s = __fmul_rn(s, c);
            const uint64_t key = __float2ull_rn(__fmul_rn(s, 4294967296.0f));
            word[idx] = (key << 31) | static_cast<uint64_t>(0x7FFFFFFF - idx);
        }
        count[b] = 0;
    }
    for (int i = n + tid; i < n_pad; i += kThreads) word[i] = 0;   // sorts after every real word
    __syncthreads();

    // 2. bitonic sort, descending
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

    // 3. inclusive scan of keys; thread t owns positions [t*items, (t+1)*items)
    const int items = (n_pad + kThreads - 1) / kThreads;
    const int p0 = tid * items;
    uint64_t run = 0;
    for (int it = 0; it < items; ++it) {
        const int p = p0 + it;
        if (p < n) run += word[p] >> 31;
    }
    uint64_t incl = run;
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_total[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint64_t t = warp_total[lane];
        for (int off = 1; off < 32; off <<= 1) {
            const uint64_t v = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += v;
        }
        warp_total[lane] = t;   // inclusive over warps
    }
    __syncthreads();
    uint64_t S = incl - run + (warp > 0 ? warp_total[warp - 1] : 0);   // exclusive prefix

    // 4. objective and argmax; K = p + 1 for owned position p, K = 0 by thread 0
    const double t0 = bias + alpha[B];
    const uint64_t base_E = static_cast<uint64_t>(B) << 32;
    double best_obj = -INFINITY;
    int best_k = -1;
    if (tid == 0) {
        const double T = t0 + theta[B];
        if (T > 0.0 && T < INFINITY) {
            best_obj = static_cast<double>(base_E) / T;
            best_k = 0;
        }
    }
    for (int it = 0; it < items; ++it) {
        const int p = p0 + it;
        if (p >= n) break;
        S += word[p] >> 31;
        const int K = p + 1;
        const double T = t0 + theta[B + K];
        if (T > 0.0 && T < INFINITY) {
            const double obj = static_cast<double>(base_E + S) / T;
            if (better(obj, K, best_obj, best_k)) {
                best_obj = obj;
                best_k = K;
            }
        }
    }
    for (int off = 16; off > 0; off >>= 1) {
        const double o = __shfl_xor_sync(0xffffffffu, best_obj, off);
        const int kk = __shfl_xor_sync(0xffffffffu, best_k, off);
        if (better(o, kk, best_obj, best_k)) {
            best_obj = o;
            best_k = kk;
        }
    }
    if (lane == 0) {
        red_obj[warp] = best_obj;
        red_k[warp] = best_k;
    }
    __syncthreads();
    if (warp == 0) {
        best_obj = red_obj[lane];
        best_k = red_k[lane];
        for (int off = 16; off > 0; off >>= 1) {
            const double o = __shfl_xor_sync(0xffffffffu, best_obj, off);
            const int kk = __shfl_xor_sync(0xffffffffu, best_k, off);
            if (better(o, kk, best_obj, best_k)) {
                best_obj = o;
                best_k = kk;
            }
        }
        if (lane == 0) {
            if (best_k < 0) {
                raise_status(status, DSPARK_STATUS_BAD_COST);
                best_k = 0;
            }
            k_best = best_k;
            *k_star = best_k;
        }
    }
    __syncthreads();

    // 5. windows
    const int K_star = k_best;
    for (int p = tid; p < K_star; p += kThreads) {
        const int idx = 0x7FFFFFFF - static_cast<int>(word[p] & 0x7FFFFFFFull);
        atomicAdd(&count[idx / L], 1);
    }
    __syncthreads();
    for (int b = tid; b < B; b += kThreads) windows[b] = 1 + count[b];
}

__global__ void schedule_trivial_kernel(int B, double bias, const double* __restrict__ alpha,
                                        const double* __restrict__ theta,
                                        int32_t* __restrict__ windows,
                                        int32_t* __restrict__ k_star, int32_t* __restrict__ status)
{
    // gamma == 1: no drafts, K* = 0, every window is the anchor row alone
    const int tid = threadIdx.x;
    for (int b = tid; b < B; b += blockDim.x) windows[b] = 1;
    if (tid == 0) {
        const double T = (bias + alpha[B]) + theta[B];
        if (!(T > 0.0 && T < INFINITY)) raise_status(status, DSPARK_STATUS_BAD_COST);
        *k_star = 0;
    }
}

}  // namespace

int launch_schedule(const float* conf, int B, int gamma, const dspark_cost* cost,
                    int32_t* windows, int32_t* k_star, int32_t* status, cudaStream_t stream)
{
    const int L = gamma - 1;
    const int n = B * L;
    if (n == 0) {
        schedule_trivial_kernel<<<1, 256, 0, stream>>>(B, cost->bias, cost->alpha, cost->theta,
                                                        windows, k_star, status);
        return check_launch("schedule");
    }
    int n_pad = 1;
    while (n_pad < n) n_pad <<= 1;
    const size_t smem = sizeof(uint64_t) * static_cast<size_t>(n_pad) +
                        sizeof(int) * static_cast<size_t>(B);
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != DSPARK_OK) return rc;
    // the opt-in limit covers static plus dynamic shared memory
    static thread_local int configured_device = -1;
    static thread_local size_t max_dynamic = 0;
    if (configured_device != dev.device) {
        cudaFuncAttributes attr;
        if (cudaFuncGetAttributes(&attr, schedule_kernel) != cudaSuccess)
            return check_launch("schedule (attributes)");
        max_dynamic = static_cast<size_t>(dev.smem_optin) - attr.sharedSizeBytes;
        if (cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(max_dynamic)) != cudaSuccess)
            return check_launch("schedule (shared-memory opt-in)");
        configured_device = dev.device;
    }
    if (smem > max_dynamic)
        return fail(DSPARK_ERR_UNSUPPORTED, "dspark_schedule: %zu bytes of shared memory needed, "
                    "the device allows %zu", smem, max_dynamic);
    schedule_kernel<<<1, kThreads, smem, stream>>>(conf, B, L, n, n_pad, cost->bias, cost->alpha,
                                                   cost->theta, windows, k_star, status);
    return check_launch("schedule");
}

}  // namespace dspark
