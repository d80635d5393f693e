// verify_noalloc.cu — dspark_verify_noalloc: dspark_verify with its scratch memory in a static
// device array of this library instead of a caller-supplied workspace.
//
// For callers that cannot provide scratch memory: hosts that hand a kernel library only its
// input and output buffers, and serving loops that reserve the device's memory up front and
// must not call cudaMalloc mid-step. This file allocates nothing: the array below is part of
// the library's device image, and each call forwards to dspark_verify with its address.
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = DSPARK_NOALLOC_SCRATCH_BYTES;

// One copy per device that loads the library, kept until the process exits. In host code
// this name is only a host-side stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

// Device address of the scratch array in the current device's context. Looked up on every
// call (after the module's first load this is a host-side table lookup), so a device reset or
// another context current on the device never leaves a stale address behind.
int scratch_address(void** out)
{
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess || p == nullptr) {
        int dev = -1;
        cudaGetDevice(&dev);
        return dspark::fail(DSPARK_ERR_CUDA,
                            "dspark_verify_noalloc: cudaGetSymbolAddress of the scratch array "
                            "failed on device %d: %s", dev, cudaGetErrorString(e));
    }
    *out = p;
    return DSPARK_OK;
}

}  // namespace

extern "C" int dspark_verify_noalloc(dspark_mode mode, int stochastic, const void* target_logits,
                                     int target_rows, const void* draft_logits,
                                     dspark_dtype dtype, int V, const int32_t* cu_seqlens,
                                     const int32_t* windows, const int32_t* block_tokens, int B,
                                     int gamma, float temperature, uint64_t seed, uint64_t step,
                                     int32_t* accept_len, int32_t* committed,
                                     int32_t* ceiling_len, float* row_prob, int32_t* status,
                                     cudaStream_t stream)
{
    if (B < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 1)
        return dspark::fail(DSPARK_ERR_INVALID_ARG,
                            "dspark_verify_noalloc: bad sizes B=%d gamma=%d V=%d", B, gamma, V);
    const size_t need = dspark_verify_workspace_bytes(B, gamma, V, stochastic);
    if (need > kScratchBytes)
        return dspark::fail(DSPARK_ERR_UNSUPPORTED,
                            "dspark_verify_noalloc: these sizes need %zu bytes of scratch, the "
                            "static array holds %zu (B=%d gamma=%d V=%d stochastic=%d); use "
                            "dspark_verify with a caller workspace", need, kScratchBytes, B,
                            gamma, V, stochastic ? 1 : 0);
    void* scratch = nullptr;
    if (B > 0) {
        const int rc = scratch_address(&scratch);
        if (rc != DSPARK_OK) return rc;
    }
    return dspark_verify(mode, stochastic, target_logits, target_rows, draft_logits, dtype, V,
                         cu_seqlens, windows, block_tokens, B, gamma, temperature, seed, step,
                         accept_len, committed, ceiling_len, row_prob, scratch, kScratchBytes,
                         status, stream);
}
