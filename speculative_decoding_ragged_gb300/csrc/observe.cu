// observe.cu — calibration histogram and utilisation counters of verify outcomes.
//
// "DSpark in SGLang" (LMSYS blog summary), A2 observability: per-request confidence and
// calibration metrics (ECE) for post-hoc analysis; cap-accept recovers the acceptance ceiling
// that truncation masks, so utilisation = committed / ceiling. One thread per (request, draft);
// each CTA accumulates a shared-memory histogram and adds it to the caller's counters with
// 64-bit atomics. Counters are exact integers (confidence sums in 2^-32 fixed point), so the
// totals do not depend on the order of the additions.
#include "common.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxBins = 1024;

__global__ void __launch_bounds__(kThreads)
observe_kernel(const float* __restrict__ conf, const int32_t* __restrict__ accept_len,
               const int32_t* __restrict__ ceiling_len, int B, int gamma, int n_bins,
               unsigned long long* __restrict__ hist, unsigned long long* __restrict__ util,
               int32_t* __restrict__ status)
{
    __shared__ unsigned long long h[3 * kMaxBins];
    __shared__ unsigned long long u[2];
    pdl_wait_and_trigger();
    const int tid = threadIdx.x;
    for (int k = tid; k < 3 * n_bins; k += kThreads) h[k] = 0;
    if (tid < 2) u[tid] = 0;
    __syncthreads();

    const int L = gamma - 1;
    int bits = 0;
    // thread (b, j): j in [0, gamma) covers the drafts (j < L) and, at j == L, the request's
    // utilisation terms
    const int64_t e = static_cast<int64_t>(blockIdx.x) * kThreads + tid;
    if (e < static_cast<int64_t>(B) * gamma) {
        int b, j;
        if (static_cast<int64_t>(B) * gamma <= 0x7fffffff) {   // a 32-bit division where it fits
            const int ei = static_cast<int>(e);
            b = ei / gamma;
            j = ei - b * gamma;
        } else {
            b = static_cast<int>(e / gamma);
            j = static_cast<int>(e - static_cast<int64_t>(b) * gamma);
        }
        int c = ceiling_len[b];
        if (c < 1 || c > gamma) {
            bits |= DSPARK_STATUS_BAD_LENGTH;
            c = c < 1 ? 1 : gamma;
        }
        if (j < L) {
            if (j <= c - 1) {
                const float x = fminf(fmaxf(conf[static_cast<int64_t>(b) * L + j], 0.0f), 1.0f);
                int k = static_cast<int>(x * static_cast<float>(n_bins));
                k = k < n_bins ? k : n_bins - 1;
                const unsigned long long fx =
                    x >= 1.0f ? (1ull << 32) : static_cast<unsigned long long>(__float2uint_rn(x * 4294967296.0f));
                atomicAdd(&h[3 * k], 1ull);
                atomicAdd(&h[3 * k + 1], fx);
                if (j < c - 1) atomicAdd(&h[3 * k + 2], 1ull);
            }
        } else {
            int a = accept_len[b];
            if (a < 0 || a > gamma) {
                bits |= DSPARK_STATUS_BAD_LENGTH;
                a = a < 0 ? 0 : gamma;
            }
            atomicAdd(&u[0], static_cast<unsigned long long>(a));
            atomicAdd(&u[1], static_cast<unsigned long long>(c));
        }
    }
    __syncthreads();
    for (int k = tid; k < 3 * n_bins; k += kThreads)
        if (h[k] != 0) atomicAdd(&hist[k], h[k]);
    if (tid < 2 && u[tid] != 0) atomicAdd(&util[tid], u[tid]);
    const unsigned any = __ballot_sync(0xffffffffu, bits != 0);
    if (any) {
        for (int off = 16; off > 0; off >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, off);
        if ((tid & 31) == 0) raise_status(status, bits);
    }
}

}  // namespace

int launch_observe(const float* conf, const int32_t* accept_len, const int32_t* ceiling_len,
                   int B, int gamma, int n_bins, uint64_t* hist, uint64_t* util, int32_t* status,
                   cudaStream_t stream)
{
    const int64_t blocks = ceil_div(static_cast<int64_t>(B) * gamma, kThreads);
    return launch_pdl("observe", observe_kernel, dim3(static_cast<unsigned>(blocks)),
                      dim3(kThreads), 0, stream, conf, accept_len, ceiling_len, B, gamma, n_bins,
                      reinterpret_cast<unsigned long long*>(hist),
                      reinterpret_cast<unsigned long long*>(util), status);
}

}  // namespace dspark
