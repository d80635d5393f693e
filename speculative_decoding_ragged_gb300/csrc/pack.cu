// pack.cu — ragged front-pack as one single-CTA kernel (the body is in pack_block.cuh).
//
// "DSpark in SGLang" (LMSYS blog summary), A2, ragged verify over full CUDA graphs: the
// variable windows are front-packed into one cu_seqlens-style buffer whose total is rounded
// up to the nearest captured graph tier.
#include "pack_block.cuh"

namespace dspark {
namespace {

__global__ void __launch_bounds__(kPackThreads, 1)
pack_kernel(const int32_t* __restrict__ windows, const int32_t* __restrict__ tokens, int B,
            int gamma, const int32_t* __restrict__ tiers, int n_tiers,
            int32_t* __restrict__ cu_out, int32_t* __restrict__ packed_ids,
            int32_t* __restrict__ row_req, int32_t* __restrict__ row_pos, int packed_cap,
            int32_t* __restrict__ meta, int32_t* __restrict__ status)
{
    pdl_wait_and_trigger();
    pack_block<true>(windows, tokens, B, gamma, tiers, n_tiers, cu_out, packed_ids, row_req,
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
