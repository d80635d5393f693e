// common.cuh — internal helpers shared by the CUDA translation units of libdspark.
// Nothing here is part of the public ABI (include/dspark.h).
#pragma once

#include <climits>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "dspark.h"

namespace dspark {

// ---- host side ------------------------------------------------------------------------
// Records a message for dspark_last_error() on this host thread and returns `code`.
int fail(int code, const char* fmt, ...);
const char* last_error();
// Checks the last launch on this thread; DSPARK_OK or DSPARK_ERR_CUDA with a message.
int check_launch(const char* what);

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int smem_optin = 0;  // largest dynamic shared memory a CTA may opt into
};
// Properties of the current device, cached per device. DSPARK_OK or an error code.
int current_device(DeviceInfo* out);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---- launch helpers implemented per translation unit ------------------------------------
int launch_schedule(const float* conf, int B, int gamma, const dspark_cost* cost,
                    int32_t* windows, int32_t* k_star, int32_t* status, cudaStream_t stream);
int launch_pack(const int32_t* windows, const int32_t* tokens, int B, int gamma,
                const int32_t* tiers, int n_tiers, int32_t* cu, int32_t* packed_ids,
                int32_t* row_req, int32_t* row_pos, int packed_cap, int32_t* meta,
                int32_t* status, cudaStream_t stream);
struct PackArgs {
    const int32_t* tokens;
    const int32_t* tiers;
    int n_tiers;
    int32_t* cu;
    int32_t* packed_ids;
    int32_t* row_req;
    int32_t* row_pos;
    int packed_cap;
    int32_t* meta;
};
// The schedule, then the pack of the windows it wrote, in one single-CTA kernel.
int launch_schedule_pack(const float* conf, int B, int gamma, const dspark_cost* cost,
                         int32_t* windows, int32_t* k_star, const PackArgs& pk, int32_t* status,
                         cudaStream_t stream);
struct VerifyCall {
    int mode, stochastic;
    const void* target;
    int target_rows;
    const void* draft;
    int dtype, V;
    const int32_t* cu;
    const int32_t* windows;
    const int32_t* tokens;
    int B, gamma;
    float temperature;
    uint64_t seed, step;
    int32_t* accept_len;
    int32_t* committed;
    int32_t* ceiling;
    float* row_prob;
    void* ws;
    size_t ws_bytes;
    int32_t* status;
    // fused compact scatter (dspark_verify_scatter); out_tokens == nullptr: none
    int32_t* out_tokens;
    int32_t* out_len;
    int out_cap;
};
size_t verify_workspace_bytes(int B, int gamma, int V, int stochastic);
// dspark_set_stream_kernel: DSPARK_STREAM_AUTO / _REGISTER / _BULK for later verify calls.
int set_stream_kernel(int which);
// dspark_set_stream_events: events recorded around the streaming kernel of later verify calls.
void set_stream_events(cudaEvent_t start, cudaEvent_t stop);
int launch_verify(const VerifyCall& c, cudaStream_t stream);
int launch_scatter(const int32_t* committed, const int32_t* accept_len, int B, int gamma,
                   int32_t* out_tokens, int32_t* out_len, int out_cap, int32_t* status,
                   cudaStream_t stream);
int launch_observe(const float* conf, const int32_t* accept_len, const int32_t* ceiling_len,
                   int B, int gamma, int n_bins, uint64_t* hist, uint64_t* util, int32_t* status,
                   cudaStream_t stream);

// Launch with programmatic dependent launch allowed: the grid may start while the previous
// kernel on the stream finishes; every kernel of this library begins with pdl_wait(), which
// returns once the previous grid has completed and its memory is visible, so nothing is read
// early. Without a preceding kernel (or one that never triggers) this is a plain launch.
template <typename... Params, typename... Args>
int launch_pdl(const char* what, void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
               cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(DSPARK_ERR_CUDA, "dspark %s: %s (%s)", what, cudaGetErrorString(e),
                    cudaGetErrorName(e));
    }
    return check_launch(what);
}

// ---- device side ------------------------------------------------------------------------
// Programmatic dependent launch: wait for the previous grid (a no-op when launched plainly),
// then let the next kernel on the stream begin launching.
__device__ __forceinline__ void pdl_wait_and_trigger()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ void raise_status(int32_t* status, int bits)
{
    if (status != nullptr && bits != 0) atomicOr(status, bits);
}

// Compact scatter of one request by one warp: lane i < L holds committed token i, which is
// appended to the request's history at n0 = out_len[b] (read by the caller, the same value on
// every lane) + i, with clamped lengths and overflow dropped and flagged; lane 0 then advances
// out_len[b]. Returns the status bits (the same on every lane).
__device__ __forceinline__ int scatter_request(int64_t b, int L, int gamma, int tok, int lane,
                                               int32_t* out_tokens, int32_t* out_len, int out_cap,
                                               int n0)
{
    int bits = 0;
    int n = n0;
    if (L < 0 || L > gamma) { bits |= DSPARK_STATUS_BAD_LENGTH; L = L < 0 ? 0 : gamma; }
    if (n < 0 || n > out_cap) { bits |= DSPARK_STATUS_BAD_LENGTH; n = n < 0 ? 0 : out_cap; }
    if (lane < L) {
        if (n + lane < out_cap)
            out_tokens[b * out_cap + n + lane] = tok;
        else
            bits |= DSPARK_STATUS_OUT_OVERFLOW;
    }
    __syncwarp();
    if (lane == 0) out_len[b] = (n + L < out_cap) ? n + L : out_cap;
    for (int off = 16; off > 0; off >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, off);
    return bits;
}

// bf16 is the upper half of an IEEE fp32: widening is a shift, exact.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 16-byte read-only streaming load: skips L1 allocation, asks L2 for a 256-byte prefetch.
__device__ __forceinline__ uint4 ld_stream16(const void* p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 2^x on the SFU (PTX ex2.approx.ftz.f32: a few ulp, subnormal results flush to zero).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Logit v of a row as fp32 (exact widening for bf16).
template <int DT>
__device__ __forceinline__ float load_logit(const void* row, int64_t v)
{
    if (DT == DSPARK_BF16) {
        const uint16_t h = __ldg(reinterpret_cast<const unsigned short*>(row) + v);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    } else {
        return __ldg(reinterpret_cast<const float*>(row) + v);
    }
}

}  // namespace dspark
