/* A plain C caller of libdspark: no Python, no PyTorch. Device buffers come from cudaMalloc,
 * the calls go on the legacy default stream, and every output is compared with the C oracle
 * on the same seeded inputs (bit for bit: greedy verify).
 *
 * One step of a small batch: dspark_schedule_pack (windows, K*, cu_seqlens, packed ids, tier),
 * the packed target rows gathered on the host from the block, then dspark_verify_scatter in
 * compact mode (accept lengths, committed tokens, histories) and dspark_verify in cap-accept
 * mode (the same commits, and the ceiling). Exit status 0 and "ok" when everything matches.
 * Readings as in the library's header: "DSpark in SGLang" (LMSYS blog summary), A2 method
 * details (confidence scheduler, ragged verify over full CUDA graphs, verify-mode design). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "dspark.h"

/* the oracle's entry points (oracle/dspark_oracle.c) */
int oracle_schedule(const float* conf, int B, int gamma, double bias, const double* alpha,
                    int alpha_len, const double* theta, int theta_len, int32_t* windows,
                    int32_t* k_star, int32_t* status, double* obj, uint64_t* sorted_keys);
int oracle_pack(const int32_t* windows, const int32_t* tokens, int B, int gamma,
                const int32_t* tiers, int n_tiers, int32_t* cu, int32_t* packed_ids,
                int32_t* row_req, int32_t* row_pos, int packed_cap, int32_t* meta,
                int32_t* status);
int oracle_verify(int mode, int stochastic, const void* target, int target_rows,
                  const void* draft, int dtype, int V, const int32_t* cu, const int32_t* windows,
                  const int32_t* tokens, int B, int gamma, float temperature, uint64_t seed,
                  uint64_t step, int32_t* accept_len, int32_t* committed, int32_t* ceiling,
                  float* row_prob, int32_t* status, float* diag_ratio, float* diag_u,
                  double* diag_margin);
int oracle_scatter(const int32_t* committed, const int32_t* accept_len, int B, int gamma,
                   int32_t* out_tokens, int32_t* out_len, int out_cap, int32_t* status);

enum { B = 12, GAMMA = 6, V = 3000, N_TIERS = 3, OUT_CAP = 40, CAP = B * GAMMA };

static int failures = 0;

#define CUDA(x)                                                                              \
    do {                                                                                     \
        cudaError_t e_ = (x);                                                                \
        if (e_ != cudaSuccess) {                                                             \
            fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));                  \
            exit(2);                                                                         \
        }                                                                                    \
    } while (0)

#define DSPARK(x)                                                                            \
    do {                                                                                     \
        int r_ = (x);                                                                        \
        if (r_ != DSPARK_OK) {                                                               \
            fprintf(stderr, "%s returned %d: %s\n", #x, r_, dspark_last_error());            \
            exit(3);                                                                         \
        }                                                                                    \
    } while (0)

/* 64-bit linear congruential generator (Knuth's MMIX constants): the inputs' only source */
static uint64_t lcg_state = 0x2545F4914F6CDD1Dull;
static uint32_t rnd32(void)
{
    lcg_state = lcg_state * 6364136223846793005ull + 1442695040888963407ull;
    return (uint32_t)(lcg_state >> 32);
}
static float rnd01(void) { return (float)(rnd32() >> 8) * (1.0f / 16777216.0f); }

/* fp32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static float from_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static void check_i32(const char* what, const int32_t* got, const int32_t* want, int n)
{
    for (int i = 0; i < n; ++i)
        if (got[i] != want[i]) {
            fprintf(stderr, "%s[%d]: library %d, oracle %d\n", what, i, got[i], want[i]);
            ++failures;
            return;
        }
}

static void* dev_copy(const void* host, size_t bytes)
{
    void* d = NULL;
    CUDA(cudaMalloc(&d, bytes > 0 ? bytes : 16));
    if (bytes > 0) CUDA(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice));
    return d;
}

static void dev_fill(void* d, int value, size_t bytes) { CUDA(cudaMemset(d, value, bytes)); }

int main(void)
{
    const int L = GAMMA - 1;
    /* inputs: confidences, the block's target logits (bf16, a spike per row), block tokens whose
       drafts are the previous row's argmax about two times in three, the cost tables, tiers */
    static float conf[B * (GAMMA - 1)];
    static uint16_t block[B * GAMMA * V];
    static int32_t tokens[B * GAMMA];
    static double alpha[B + 1], theta[B * GAMMA + 1];
    const int32_t tiers[N_TIERS] = {16, 40, CAP};
    for (int i = 0; i < B * L; ++i) conf[i] = 0.3f + 0.7f * rnd01();
    for (int r = 0; r < B * GAMMA; ++r) {
        for (int v = 0; v < V; ++v) block[(size_t)r * V + v] = to_bf16(4.0f * (rnd01() - 0.5f));
        block[(size_t)r * V + rnd32() % V] = to_bf16(7.0f);
    }
    for (int b = 0; b < B; ++b) {
        tokens[b * GAMMA] = (int32_t)(rnd32() % V);
        for (int i = 0; i < L; ++i) {
            const uint16_t* row = block + (size_t)(b * GAMMA + i) * V;
            int best = 0;
            for (int v = 1; v < V; ++v)
                if (from_bf16(row[v]) > from_bf16(row[best])) best = v;
            tokens[b * GAMMA + i + 1] = (rnd32() % 3 != 0) ? best : (int32_t)(rnd32() % V);
        }
    }
    for (int bs = 0; bs <= B; ++bs) alpha[bs] = 0.05 * bs;
    for (int m = 0; m <= B * GAMMA; ++m) theta[m] = 0.02 * m;
    const double bias = 1.0;

    /* ---- the library: schedule and pack, on device buffers ---- */
    float* d_conf = (float*)dev_copy(conf, sizeof(conf));
    double* d_alpha = (double*)dev_copy(alpha, sizeof(alpha));
    double* d_theta = (double*)dev_copy(theta, sizeof(theta));
    int32_t* d_tokens = (int32_t*)dev_copy(tokens, sizeof(tokens));
    int32_t* d_tiers = (int32_t*)dev_copy(tiers, sizeof(tiers));
    int32_t *d_windows, *d_kstar, *d_cu, *d_ids, *d_req, *d_pos, *d_meta, *d_status;
    CUDA(cudaMalloc((void**)&d_windows, B * 4));
    CUDA(cudaMalloc((void**)&d_kstar, 4));
    CUDA(cudaMalloc((void**)&d_cu, (B + 1) * 4));
    CUDA(cudaMalloc((void**)&d_ids, CAP * 4));
    CUDA(cudaMalloc((void**)&d_req, CAP * 4));
    CUDA(cudaMalloc((void**)&d_pos, CAP * 4));
    CUDA(cudaMalloc((void**)&d_meta, 2 * 4));
    CUDA(cudaMalloc((void**)&d_status, 4));
    dev_fill(d_status, 0, 4);
    dspark_cost cost = {bias, d_alpha, B + 1, d_theta, B * GAMMA + 1};
    DSPARK(dspark_schedule_pack(d_conf, B, GAMMA, &cost, d_tokens, d_tiers, N_TIERS, d_windows,
                                d_kstar, d_cu, d_ids, d_req, d_pos, CAP, d_meta, d_status, 0));
    CUDA(cudaDeviceSynchronize());
    int32_t windows[B], kstar, cu[B + 1], ids[CAP], req[CAP], pos[CAP], meta[2], status;
    CUDA(cudaMemcpy(windows, d_windows, sizeof(windows), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&kstar, d_kstar, 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(cu, d_cu, sizeof(cu), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(meta, d_meta, sizeof(meta), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(ids, d_ids, sizeof(ids), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(req, d_req, sizeof(req), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(pos, d_pos, sizeof(pos), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));

    /* the oracle on the same inputs */
    int32_t o_windows[B], o_kstar, o_status = 0, o_cu[B + 1], o_ids[CAP], o_req[CAP], o_pos[CAP],
            o_meta[2];
    if (oracle_schedule(conf, B, GAMMA, bias, alpha, B + 1, theta, B * GAMMA + 1, o_windows,
                        &o_kstar, &o_status, NULL, NULL) != 0 ||
        oracle_pack(o_windows, tokens, B, GAMMA, tiers, N_TIERS, o_cu, o_ids, o_req, o_pos, CAP,
                    o_meta, &o_status) != 0) {
        fprintf(stderr, "oracle refused the inputs\n");
        return 4;
    }
    check_i32("windows", windows, o_windows, B);
    check_i32("k_star", &kstar, &o_kstar, 1);
    check_i32("cu_seqlens", cu, o_cu, B + 1);
    check_i32("meta", meta, o_meta, 2);
    check_i32("packed_ids", ids, o_ids, meta[1]);
    check_i32("row_req", req, o_req, meta[1]);
    check_i32("row_pos", pos, o_pos, meta[1]);
    check_i32("schedule status", &status, &o_status, 1);
    if (failures) return 1;

    /* ---- the packed target rows (standing in for the target forward over the packed batch):
       row cu[b] + i holds the block's row b * gamma + i; the padding rows up to the tier are 0 */
    const int M = meta[0], tier = meta[1];
    uint16_t* packed = (uint16_t*)calloc((size_t)tier * V, 2);
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < windows[b]; ++i)
            memcpy(packed + (size_t)(cu[b] + i) * V, block + (size_t)(b * GAMMA + i) * V, V * 2);
    void* d_packed = dev_copy(packed, (size_t)tier * V * 2);
    void* d_block = dev_copy(block, sizeof(block));

    /* ---- the library: compact verify with the fused scatter, then cap-accept verify ---- */
    const size_t ws_bytes = dspark_verify_workspace_bytes(B, GAMMA, V, 0);
    void* d_ws;
    CUDA(cudaMalloc(&d_ws, ws_bytes));
    int32_t *d_acc, *d_com, *d_out, *d_len, *d_acc2, *d_com2, *d_ceil2;
    CUDA(cudaMalloc((void**)&d_acc, B * 4));
    CUDA(cudaMalloc((void**)&d_com, B * GAMMA * 4));
    CUDA(cudaMalloc((void**)&d_out, B * OUT_CAP * 4));
    CUDA(cudaMalloc((void**)&d_len, B * 4));
    CUDA(cudaMalloc((void**)&d_acc2, B * 4));
    CUDA(cudaMalloc((void**)&d_com2, B * GAMMA * 4));
    CUDA(cudaMalloc((void**)&d_ceil2, B * 4));
    dev_fill(d_out, 0xFF, B * OUT_CAP * 4);
    dev_fill(d_len, 0, B * 4);
    dev_fill(d_status, 0, 4);
    DSPARK(dspark_verify_scatter(DSPARK_COMPACT, 0, d_packed, tier, NULL, DSPARK_BF16, V, d_cu,
                                 d_windows, d_tokens, B, GAMMA, 1.0f, 0, 0, d_acc, d_com, NULL,
                                 NULL, d_ws, ws_bytes, d_out, d_len, OUT_CAP, d_status, 0));
    DSPARK(dspark_verify(DSPARK_CAP_ACCEPT, 0, d_block, B * GAMMA, NULL, DSPARK_BF16, V, NULL,
                         d_windows, d_tokens, B, GAMMA, 1.0f, 0, 0, d_acc2, d_com2, d_ceil2,
                         NULL, d_ws, ws_bytes, d_status, 0));
    CUDA(cudaDeviceSynchronize());
    int32_t acc[B], com[B * GAMMA], out[B * OUT_CAP], len[B], acc2[B], com2[B * GAMMA],
        ceil2[B];
    CUDA(cudaMemcpy(acc, d_acc, sizeof(acc), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(com, d_com, sizeof(com), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(out, d_out, sizeof(out), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(len, d_len, sizeof(len), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(acc2, d_acc2, sizeof(acc2), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(com2, d_com2, sizeof(com2), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(ceil2, d_ceil2, sizeof(ceil2), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));

    /* the oracle: compact verify and scatter, cap-accept verify */
    int32_t o_acc[B], o_com[B * GAMMA], o_ceil[B], o_out[B * OUT_CAP], o_len[B] = {0};
    int32_t o_acc2[B], o_com2[B * GAMMA], o_ceil2[B], o_vstatus = 0;
    for (int i = 0; i < B * OUT_CAP; ++i) o_out[i] = -1;
    if (oracle_verify(1, 0, packed, tier, NULL, 0, V, o_cu, o_windows, tokens, B, GAMMA, 1.0f,
                      0, 0, o_acc, o_com, o_ceil, NULL, &o_vstatus, NULL, NULL, NULL) != 0 ||
        oracle_scatter(o_com, o_acc, B, GAMMA, o_out, o_len, OUT_CAP, &o_vstatus) != 0 ||
        oracle_verify(2, 0, block, B * GAMMA, NULL, 0, V, NULL, o_windows, tokens, B, GAMMA,
                      1.0f, 0, 0, o_acc2, o_com2, o_ceil2, NULL, &o_vstatus, NULL, NULL,
                      NULL) != 0) {
        fprintf(stderr, "oracle refused the verify inputs\n");
        return 4;
    }
    check_i32("accept_len", acc, o_acc, B);
    check_i32("committed", com, o_com, B * GAMMA);
    check_i32("out_len", len, o_len, B);
    check_i32("out_tokens", out, o_out, B * OUT_CAP);
    check_i32("cap-accept accept_len", acc2, o_acc2, B);
    check_i32("cap-accept committed", com2, o_com2, B * GAMMA);
    check_i32("cap-accept ceiling", ceil2, o_ceil2, B);
    check_i32("compact == cap-accept", com2, com, B * GAMMA);
    check_i32("verify status", &status, &o_vstatus, 1);

    int accepted = 0;
    for (int b = 0; b < B; ++b) accepted += acc[b];
    printf("M=%d tier=%d K*=%d accepted=%d\n", M, tier, kstar, accepted);
    free(packed);
    if (failures) return 1;
    printf("ok\n");
    return 0;
}
