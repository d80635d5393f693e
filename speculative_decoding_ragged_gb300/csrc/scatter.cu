// scatter.cu — compact scatter of committed tokens into per-request output histories.
//
// "DSpark in SGLang" (LMSYS blog summary), A2, performance and zero-overhead scheduling: a
// fused kernel writes the accepted tokens back into per-request state. One warp per request
// (gamma <= 32 committed tokens, one lane each), through the same per-request routine that
// dspark_verify_scatter runs at the end of its verify.
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
    const int L = accept_len[b];
    const int tok = (lane < L && lane < gamma) ? committed[b * gamma + lane] : -1;
    const int bits = scatter_request(b, L, gamma, tok, lane, out_tokens, out_len, out_cap,
                                     out_len[b]);
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
