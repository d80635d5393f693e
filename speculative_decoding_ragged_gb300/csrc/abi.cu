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

// Argument checks shared by the single and the fused entry points; `fn` names the entry
// point in the error message.
int check_schedule(const char* fn, const float* conf, int B, int gamma, const dspark_cost* cost,
                   const int32_t* windows, const int32_t* k_star)
{
    if (B < 0 || B > DSPARK_MAX_BATCH)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: B = %d outside [0, %d]", fn, B, DSPARK_MAX_BATCH);
    if (gamma < 1 || gamma > DSPARK_MAX_GAMMA)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: gamma = %d outside [1, %d]", fn, gamma,
                    DSPARK_MAX_GAMMA);
    if (static_cast<int64_t>(B) * (gamma - 1) > DSPARK_MAX_CANDIDATES)
        return fail(DSPARK_ERR_UNSUPPORTED, "%s: B*(gamma-1) = %lld above %d", fn,
                    static_cast<long long>(B) * (gamma - 1), DSPARK_MAX_CANDIDATES);
    if (k_star == nullptr || !aligned4(k_star))
        return fail(DSPARK_ERR_INVALID_ARG, "%s: k_star must be a device int32 pointer", fn);
    if (B == 0) return DSPARK_OK;
    if (cost == nullptr || cost->alpha == nullptr || cost->theta == nullptr)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: cost table and its alpha/theta arrays are required", fn);
    if (cost->alpha_len < B + 1)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: alpha_len = %d, need >= B+1 = %d", fn,
                    cost->alpha_len, B + 1);
    if (static_cast<int64_t>(cost->theta_len) < static_cast<int64_t>(B) * gamma + 1)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: theta_len = %d, need >= B*gamma+1 = %lld", fn,
                    cost->theta_len, static_cast<long long>(B) * gamma + 1);
    if ((conf == nullptr && gamma > 1) || windows == nullptr || !aligned4(windows))
        return fail(DSPARK_ERR_INVALID_ARG, "%s: conf and windows are required", fn);
    return DSPARK_OK;
}

int schedule_empty(const char* fn, int32_t* k_star, cudaStream_t stream)
{
    const cudaError_t e = cudaMemsetAsync(k_star, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return fail(DSPARK_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    return DSPARK_OK;
}

int check_pack(const char* fn, const int32_t* windows, const int32_t* block_tokens, int B,
               int gamma, const int32_t* tiers, int n_tiers, const int32_t* cu_seqlens,
               const int32_t* packed_ids, int packed_cap, const int32_t* meta)
{
    if (B < 0 || B > DSPARK_MAX_BATCH)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: B = %d outside [0, %d]", fn, B, DSPARK_MAX_BATCH);
    if (gamma < 1 || gamma > DSPARK_MAX_GAMMA)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: gamma = %d outside [1, %d]", fn, gamma,
                    DSPARK_MAX_GAMMA);
    if (n_tiers < 1 || n_tiers > DSPARK_MAX_TIERS)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: n_tiers = %d outside [1, %d]", fn, n_tiers,
                    DSPARK_MAX_TIERS);
    if (packed_cap < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: packed_cap = %d is negative", fn, packed_cap);
    if (tiers == nullptr || cu_seqlens == nullptr || meta == nullptr ||
        (B > 0 && (windows == nullptr || block_tokens == nullptr)) ||
        (packed_cap > 0 && packed_ids == nullptr))
        return fail(DSPARK_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    return DSPARK_OK;
}

int check_verify(const char* fn, dspark_mode mode, int stochastic, const void* target_logits,
                 int target_rows, const void* draft_logits, dspark_dtype dtype, int V,
                 const int32_t* cu_seqlens, const int32_t* windows, const int32_t* block_tokens,
                 int B, int gamma, float temperature, const int32_t* accept_len,
                 const int32_t* committed)
{
    if (mode != DSPARK_STATIC && mode != DSPARK_COMPACT && mode != DSPARK_CAP_ACCEPT)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: unknown mode %d", fn, static_cast<int>(mode));
    if (dtype != DSPARK_BF16 && dtype != DSPARK_F32)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, static_cast<int>(dtype));
    if (B < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 1 || target_rows < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: bad sizes B=%d gamma=%d V=%d rows=%d", fn, B,
                    gamma, V, target_rows);
    if (static_cast<int64_t>(B) * gamma > INT32_MAX)
        return fail(DSPARK_ERR_UNSUPPORTED, "%s: B*gamma overflows int32", fn);
    if (stochastic && !(temperature > 0.0f && temperature < INFINITY))
        return fail(DSPARK_ERR_INVALID_ARG, "%s: stochastic verify needs a finite temperature > 0", fn);
    if (B == 0) return DSPARK_OK;
    if (target_logits == nullptr || block_tokens == nullptr || accept_len == nullptr ||
        committed == nullptr)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: logits, tokens, accept_len and committed are required", fn);
    if (mode == DSPARK_COMPACT && cu_seqlens == nullptr)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: compact mode needs cu_seqlens", fn);
    if (mode != DSPARK_STATIC && windows == nullptr)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: compact and cap-accept modes need windows", fn);
    if (stochastic && draft_logits == nullptr && gamma > 1)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: stochastic verify needs draft logits", fn);
    const size_t esz = dtype == DSPARK_BF16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(target_logits) % esz) != 0 ||
        (draft_logits != nullptr && (reinterpret_cast<uintptr_t>(draft_logits) % esz) != 0))
        return fail(DSPARK_ERR_INVALID_ARG, "%s: logits must be aligned to their element size", fn);
    return DSPARK_OK;
}

int check_scatter(const char* fn, const int32_t* committed, const int32_t* accept_len, int B,
                  int gamma, const int32_t* out_tokens, const int32_t* out_len, int out_cap)
{
    if (B < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || out_cap < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "%s: bad sizes B=%d gamma=%d out_cap=%d", fn, B,
                    gamma, out_cap);
    if (B == 0) return DSPARK_OK;
    if (committed == nullptr || accept_len == nullptr || out_len == nullptr ||
        (out_cap > 0 && out_tokens == nullptr))
        return fail(DSPARK_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
    return DSPARK_OK;
}

dspark::VerifyCall verify_call(dspark_mode mode, int stochastic, const void* target_logits,
                               int target_rows, const void* draft_logits, dspark_dtype dtype,
                               int V, const int32_t* cu_seqlens, const int32_t* windows,
                               const int32_t* block_tokens, int B, int gamma, float temperature,
                               uint64_t seed, uint64_t step, int32_t* accept_len,
                               int32_t* committed, int32_t* ceiling_len, float* row_prob,
                               void* workspace, size_t workspace_bytes, int32_t* status)
{
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
    c.out_tokens = nullptr;
    c.out_len = nullptr;
    c.out_cap = 0;
    return c;
}

}  // namespace

extern "C" {

int dspark_schedule(const float* conf, int B, int gamma, const dspark_cost* cost,
                    int32_t* windows, int32_t* k_star, int32_t* status, cudaStream_t stream)
{
    const char* fn = "dspark_schedule";
    int rc = check_schedule(fn, conf, B, gamma, cost, windows, k_star);
    if (rc != DSPARK_OK) return rc;
    if (B == 0) return schedule_empty(fn, k_star, stream);
    return dspark::launch_schedule(conf, B, gamma, cost, windows, k_star, status, stream);
}

int dspark_pack(const int32_t* windows, const int32_t* block_tokens, int B, int gamma,
                const int32_t* tiers, int n_tiers, int32_t* cu_seqlens, int32_t* packed_ids,
                int32_t* row_req, int32_t* row_pos, int packed_cap, int32_t* meta,
                int32_t* status, cudaStream_t stream)
{
    int rc = check_pack("dspark_pack", windows, block_tokens, B, gamma, tiers, n_tiers,
                        cu_seqlens, packed_ids, packed_cap, meta);
    if (rc != DSPARK_OK) return rc;
    return dspark::launch_pack(windows, block_tokens, B, gamma, tiers, n_tiers, cu_seqlens,
                               packed_ids, row_req, row_pos, packed_cap, meta, status, stream);
}

int dspark_schedule_pack(const float* conf, int B, int gamma, const dspark_cost* cost,
                         const int32_t* block_tokens, const int32_t* tiers, int n_tiers,
                         int32_t* windows, int32_t* k_star, int32_t* cu_seqlens,
                         int32_t* packed_ids, int32_t* row_req, int32_t* row_pos,
                         int packed_cap, int32_t* meta, int32_t* status, cudaStream_t stream)
{
    const char* fn = "dspark_schedule_pack";
    int rc = check_schedule(fn, conf, B, gamma, cost, windows, k_star);
    if (rc != DSPARK_OK) return rc;
    rc = check_pack(fn, windows, block_tokens, B, gamma, tiers, n_tiers, cu_seqlens, packed_ids,
                    packed_cap, meta);
    if (rc != DSPARK_OK) return rc;
    if (B == 0 || gamma == 1) {   // nothing to rank: the two plain kernels
        rc = B == 0 ? schedule_empty(fn, k_star, stream)
                    : dspark::launch_schedule(conf, B, gamma, cost, windows, k_star, status, stream);
        if (rc != DSPARK_OK) return rc;
        return dspark::launch_pack(windows, block_tokens, B, gamma, tiers, n_tiers, cu_seqlens,
                                   packed_ids, row_req, row_pos, packed_cap, meta, status, stream);
    }
    dspark::PackArgs pk;
    pk.tokens = block_tokens;
    pk.tiers = tiers;
    pk.n_tiers = n_tiers;
    pk.cu = cu_seqlens;
    pk.packed_ids = packed_ids;
    pk.row_req = row_req;
    pk.row_pos = row_pos;
    pk.packed_cap = packed_cap;
    pk.meta = meta;
    return dspark::launch_schedule_pack(conf, B, gamma, cost, windows, k_star, pk, status, stream);
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
    int rc = check_verify("dspark_verify", mode, stochastic, target_logits, target_rows,
                          draft_logits, dtype, V, cu_seqlens, windows, block_tokens, B, gamma,
                          temperature, accept_len, committed);
    if (rc != DSPARK_OK || B == 0) return rc;
    const dspark::VerifyCall c = verify_call(
        mode, stochastic, target_logits, target_rows, draft_logits, dtype, V, cu_seqlens, windows,
        block_tokens, B, gamma, temperature, seed, step, accept_len, committed, ceiling_len,
        row_prob, workspace, workspace_bytes, status);
    return dspark::launch_verify(c, stream);
}

int dspark_verify_scatter(dspark_mode mode, int stochastic, const void* target_logits,
                          int target_rows, const void* draft_logits, dspark_dtype dtype, int V,
                          const int32_t* cu_seqlens, const int32_t* windows,
                          const int32_t* block_tokens, int B, int gamma, float temperature,
                          uint64_t seed, uint64_t step, int32_t* accept_len, int32_t* committed,
                          int32_t* ceiling_len, float* row_prob, void* workspace,
                          size_t workspace_bytes, int32_t* out_tokens, int32_t* out_len,
                          int out_cap, int32_t* status, cudaStream_t stream)
{
    const char* fn = "dspark_verify_scatter";
    int rc = check_verify(fn, mode, stochastic, target_logits, target_rows, draft_logits, dtype,
                          V, cu_seqlens, windows, block_tokens, B, gamma, temperature,
                          accept_len, committed);
    if (rc != DSPARK_OK) return rc;
    rc = check_scatter(fn, committed, accept_len, B, gamma, out_tokens, out_len, out_cap);
    if (rc != DSPARK_OK || B == 0) return rc;
    dspark::VerifyCall c = verify_call(
        mode, stochastic, target_logits, target_rows, draft_logits, dtype, V, cu_seqlens, windows,
        block_tokens, B, gamma, temperature, seed, step, accept_len, committed, ceiling_len,
        row_prob, workspace, workspace_bytes, status);
    c.out_tokens = out_tokens;
    c.out_len = out_len;
    c.out_cap = out_cap;
    return dspark::launch_verify(c, stream);
}

int dspark_scatter(const int32_t* committed, const int32_t* accept_len, int B, int gamma,
                   int32_t* out_tokens, int32_t* out_len, int out_cap, int32_t* status,
                   cudaStream_t stream)
{
    int rc = check_scatter("dspark_scatter", committed, accept_len, B, gamma, out_tokens,
                           out_len, out_cap);
    if (rc != DSPARK_OK || B == 0) return rc;
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

int dspark_set_stream_kernel(int which) { return dspark::set_stream_kernel(which); }

int dspark_set_stream_events(cudaEvent_t start, cudaEvent_t stop)
{
    if ((start == nullptr) != (stop == nullptr))
        return fail(DSPARK_ERR_INVALID_ARG, "dspark_set_stream_events: give both events or neither");
    dspark::set_stream_events(start, stop);
    return DSPARK_OK;
}

const char* dspark_last_error(void) { return dspark::last_error(); }

int dspark_version(void) { return 102; }

}  // extern "C"
