// abi.cu — the extern "C" entry points of libdspark: host-side argument checks, the per-thread
// error message, the per-device property cache, and dispatch to the kernels' launchers.
// Every check happens before anything is enqueued; see include/dspark.h for the contract.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace dspark {

namespace {
thread_local char g_error[512] = "";

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
}  // namespace

const char* last_error() { return g_error; }

int fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_error, sizeof g_error, fmt, ap);
    va_end(ap);
    return code;
}

int check_launch(const char* what)
{
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "dspark %s: %s (%s)", what, cudaGetErrorString(e),
                    cudaGetErrorName(e));
    return DSPARK_OK;
}

int current_device(DeviceInfo* out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(DSPARK_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(DSPARK_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (d.device != dev) {
        int sms = 0, optin = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess)
            return fail(DSPARK_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        d.sm_count = sms;
        d.smem_optin = optin;
        d.device = dev;
    }
    *out = d;
    return DSPARK_OK;
}

}  // namespace dspark

using dspark::fail;

namespace {

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" {

int dspark_schedule(const float* conf, int B, int gamma, const dspark_cost* cost,
                    int32_t* windows, int32_t* k_star, int32_t* status, cudaStream_t stream)
{
    if (B < 0 || B > DSPARK_MAX_BATCH)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_schedule: B = %d outside [0, %d]", B,
                    DSPARK_MAX_BATCH);
    if (gamma < 1 || gamma > DSPARK_MAX_GAMMA)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_schedule: gamma = %d outside [1, %d]", gamma,
                    DSPARK_MAX_GAMMA);
    if (static_cast<int64_t>(B) * (gamma - 1) > DSPARK_MAX_CANDIDATES)
        return fail(DSPARK_ERR_UNSUPPORTED, "dspark_schedule: B*(gamma-1) = %lld above %d",
                    static_cast<long long>(B) * (gamma - 1), DSPARK_MAX_CANDIDATES);
    if (k_star == nullptr || !aligned4(k_star))
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_schedule: k_star must be a device int32 pointer");
    if (B == 0) {
        const cudaError_t e = cudaMemsetAsync(k_star, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess)
            return fail(DSPARK_ERR_CUDA, "dspark_schedule: %s", cudaGetErrorString(e));
        return DSPARK_OK;
    }
    if (cost == nullptr || cost->alpha == nullptr || cost->theta == nullptr)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_schedule: cost table and its alpha/theta arrays are required");
    if (cost->alpha_len < B + 1)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_schedule: alpha_len = %d, need >= B+1 = %d",
                    cost->alpha_len, B + 1);
    if (static_cast<int64_t>(cost->theta_len) < static_cast<int64_t>(B) * gamma + 1)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_schedule: theta_len = %d, need >= B*gamma+1 = %lld",
                    cost->theta_len, static_cast<long long>(B) * gamma + 1);
    if ((conf == nullptr && gamma > 1) || windows == nullptr || !aligned4(windows))
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_schedule: conf and windows are required");
    return dspark::launch_schedule(conf, B, gamma, cost, windows, k_star, status, stream);
}

int dspark_pack(const int32_t* windows, const int32_t* block_tokens, int B, int gamma,
                const int32_t* tiers, int n_tiers, int32_t* cu_seqlens, int32_t* packed_ids,
                int32_t* row_req, int32_t* row_pos, int packed_cap, int32_t* meta,
                int32_t* status, cudaStream_t stream)
{
    if (B < 0 || B > DSPARK_MAX_BATCH)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_pack: B = %d outside [0, %d]", B,
                    DSPARK_MAX_BATCH);
    if (gamma < 1 || gamma > DSPARK_MAX_GAMMA)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_pack: gamma = %d outside [1, %d]", gamma,
                    DSPARK_MAX_GAMMA);
    if (n_tiers < 1 || n_tiers > DSPARK_MAX_TIERS)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_pack: n_tiers = %d outside [1, %d]", n_tiers,
                    DSPARK_MAX_TIERS);
    if (packed_cap < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_pack: packed_cap = %d is negative", packed_cap);
    if (tiers == nullptr || cu_seqlens == nullptr || meta == nullptr ||
        (B > 0 && (windows == nullptr || block_tokens == nullptr)) ||
        (packed_cap > 0 && packed_ids == nullptr))
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_pack: a required pointer is NULL");
    return dspark::launch_pack(windows, block_tokens, B, gamma, tiers, n_tiers, cu_seqlens,
                               packed_ids, row_req, row_pos, packed_cap, meta, status, stream);
}

size_t dspark_verify_workspace_bytes(int B, int gamma, int V, int stochastic)
{
    if (B < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 1) {
        fail(DSPARK_ERR_INVALID_ARG, "dspark_verify_workspace_bytes: bad sizes B=%d gamma=%d V=%d",
             B, gamma, V);
        return 0;
    }
    return dspark::verify_workspace_bytes(B, gamma, V, stochastic ? 1 : 0);
}

int dspark_verify(dspark_mode mode, int stochastic, const void* target_logits, int target_rows,
                  const void* draft_logits, dspark_dtype dtype, int V, const int32_t* cu_seqlens,
                  const int32_t* windows, const int32_t* block_tokens, int B, int gamma,
                  float temperature, uint64_t seed, uint64_t step, int32_t* accept_len,
                  int32_t* committed, int32_t* ceiling_len, float* row_prob, void* workspace,
                  size_t workspace_bytes, int32_t* status, cudaStream_t stream)
{
    if (mode != DSPARK_STATIC && mode != DSPARK_COMPACT && mode != DSPARK_CAP_ACCEPT)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: unknown mode %d", static_cast<int>(mode));
    if (dtype != DSPARK_BF16 && dtype != DSPARK_F32)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: unknown dtype %d", static_cast<int>(dtype));
    if (B < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 1 || target_rows < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: bad sizes B=%d gamma=%d V=%d rows=%d",
                    B, gamma, V, target_rows);
    if (static_cast<int64_t>(B) * gamma > INT32_MAX)
        return fail(DSPARK_ERR_UNSUPPORTED, "dspark_verify: B*gamma overflows int32");
    if (stochastic && !(temperature > 0.0f && temperature < INFINITY))
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: stochastic verify needs a finite temperature > 0");
    if (B == 0) return DSPARK_OK;
    if (target_logits == nullptr || block_tokens == nullptr || accept_len == nullptr ||
        committed == nullptr)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: logits, tokens, accept_len and committed are required");
    if (mode == DSPARK_COMPACT && cu_seqlens == nullptr)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: compact mode needs cu_seqlens");
    if (mode != DSPARK_STATIC && windows == nullptr)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: compact and cap-accept modes need windows");
    if (stochastic && draft_logits == nullptr && gamma > 1)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: stochastic verify needs draft logits");
    const size_t esz = dtype == DSPARK_BF16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(target_logits) % esz) != 0 ||
        (draft_logits != nullptr && (reinterpret_cast<uintptr_t>(draft_logits) % esz) != 0))
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_verify: logits must be aligned to their element size");
    dspark::VerifyCall c;
    c.mode = static_cast<int>(mode);
    c.stochastic = stochastic ? 1 : 0;
    c.target = target_logits;
    c.target_rows = target_rows;
    c.draft = draft_logits;
    c.dtype = static_cast<int>(dtype);
    c.V = V;
    c.cu = cu_seqlens;
    c.windows = windows;
    c.tokens = block_tokens;
    c.B = B;
    c.gamma = gamma;
    c.temperature = temperature;
    c.seed = seed;
    c.step = step;
    c.accept_len = accept_len;
    c.committed = committed;
    c.ceiling = ceiling_len;
    c.row_prob = row_prob;
    c.ws = workspace;
    c.ws_bytes = workspace_bytes;
    c.status = status;
    return dspark::launch_verify(c, stream);
}

int dspark_scatter(const int32_t* committed, const int32_t* accept_len, int B, int gamma,
                   int32_t* out_tokens, int32_t* out_len, int out_cap, int32_t* status,
                   cudaStream_t stream)
{
    if (B < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || out_cap < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_scatter: bad sizes B=%d gamma=%d out_cap=%d",
                    B, gamma, out_cap);
    if (B == 0) return DSPARK_OK;
    if (committed == nullptr || accept_len == nullptr || out_len == nullptr ||
        (out_cap > 0 && out_tokens == nullptr))
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_scatter: a required pointer is NULL");
    return dspark::launch_scatter(committed, accept_len, B, gamma, out_tokens, out_len, out_cap,
                                  status, stream);
}

int dspark_observe(const float* conf, const int32_t* accept_len, const int32_t* ceiling_len,
                   int B, int gamma, int n_bins, uint64_t* hist, uint64_t* util,
                   int32_t* status, cudaStream_t stream)
{
    if (B < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || n_bins < 1 || n_bins > 1024)
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_observe: bad sizes B=%d gamma=%d n_bins=%d",
                    B, gamma, n_bins);
    if (B == 0) return DSPARK_OK;
    if ((conf == nullptr && gamma > 1) || accept_len == nullptr || ceiling_len == nullptr ||
        hist == nullptr || util == nullptr ||
        (reinterpret_cast<uintptr_t>(hist) & 7u) != 0 || (reinterpret_cast<uintptr_t>(util) & 7u) != 0)
        return fail(DSPARK_ERR_INVALID_ARG,
                    "dspark_observe: conf, lengths and 8-byte aligned counters are required");
    return dspark::launch_observe(conf, accept_len, ceiling_len, B, gamma, n_bins, hist, util,
                                  status, stream);
}

const char* dspark_last_error(void) { return dspark::last_error(); }

int dspark_version(void) { return 100; }

}  // extern "C"
