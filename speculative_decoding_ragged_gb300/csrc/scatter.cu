// scatter.cu — compact scatter of committed tokens into per-request output histories.
//
// "DSpark in SGLang" (LMSYS blog summary), A2, performance and zero-overhead scheduling: a
// fused kernel writes the accepted tokens back into per-request state. One warp per request
// (gamma <= 32 committed tokens, one lane each); the history length is read by every lane
// before lane 0 advances it.
#include "common.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
scatter_kernel(const int32_t* __restrict__ committed, const int32_t* __restrict__ accept_len,
               int B, int gamma, int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_len,
               int out_cap, int32_t* __restrict__ status)
{
    pdl_wait_and_trigger();
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (b >= B) return;   // whole warps leave together
    int bits = 0;
    int L = accept_len[b];
    int n = out_len[b];
    if (L < 0 || L > gamma) { bits |= DSPARK_STATUS_BAD_LENGTH; L = L < 0 ? 0 : gamma; }
    if (n < 0 || n > out_cap) { bits |= DSPARK_STATUS_BAD_LENGTH; n = n < 0 ? 0 : out_cap; }
    if (lane < L) {
        if (n + lane < out_cap)
            out_tokens[b * out_cap + n + lane] = committed[b * gamma + lane];
        else
            bits |= DSPARK_STATUS_OUT_OVERFLOW;
    }
    __syncwarp();
    if (lane == 0) out_len[b] = (n + L < out_cap) ? n + L : out_cap;
    for (int off = 16; off > 0; off >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, off);
    if (lane == 0) raise_status(status, bits);
}

}  // namespace

int launch_scatter(const int32_t* committed, const int32_t* accept_len, int B, int gamma,
                   int32_t* out_tokens, int32_t* out_len, int out_cap, int32_t* status,
                   cudaStream_t stream)
{
    const int64_t blocks = ceil_div(static_cast<int64_t>(B) * 32, kThreads);
    return launch_pdl("scatter", scatter_kernel, dim3(static_cast<unsigned>(blocks)),
                      dim3(kThreads), 0, stream, committed, accept_len, B, gamma, out_tokens,
                      out_len, out_cap, status);
}

}  // namespace dspark
