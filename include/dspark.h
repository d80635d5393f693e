/*
 * dspark.h — C ABI of the DSpark ragged-verification hot path for one GB300 (sm_103a).
 *
 * A decode step of confidence-driven variable-length speculative verification runs four calls,
 * each one asynchronous on the caller's CUDA stream:
 *
 *   dspark_schedule  confidences c[b,j]  -> per-request verify windows w_b and K*
 *   dspark_pack      windows, block tokens -> cu_seqlens, capture tier, packed token buffer
 *   dspark_verify    packed target logits [M,V] (+ draft logits) -> accept lengths, committed tokens
 *   dspark_scatter   committed tokens -> per-request output histories
 *
 * dspark_schedule_pack and dspark_verify_scatter produce the same results as the two pairs of
 * calls with fewer kernel launches; dspark_observe accumulates calibration counters.
 *
 * Source of the method: "DSpark in SGLang: Speculative Decoding with Confidence-Driven,
 * Variable-Length Verification" (LMSYS blog, as summarised by papercache.org), sections
 * "A2 method details" (confidence scheduler, verify modes, ragged verify over full CUDA graphs,
 * cost-table modelling) and the quick-read summary; the min(1, p/q) accept rule as restated in
 * the lshu.cn DSpark/SGLang article, sections 2.3 and 3.3.
 *
 * Conventions shared by every entry point
 *   - Every array pointer is a DEVICE pointer owned by the caller, unless its comment says
 *     "host". The library never allocates, frees or retains caller memory.
 *   - Arrays are dense, row-major, with the shapes given in brackets; int32_t is little-endian
 *     two's complement; "bf16" is IEEE bfloat16 stored in 16 bits.
 *   - B = number of requests, gamma = block width (1 anchor + gamma-1 drafts), V = vocabulary.
 *   - All work is enqueued on `stream` (0 = legacy default stream); nothing synchronises the host.
 *   - Kernels are launched with programmatic dependent launch allowed. A call may read, while
 *     the previous kernel on the stream is still finishing, its read-only inputs that no
 *     kernel of this library is writing at that moment: confidences, cost tables, block
 *     tokens, logits and, in a verify call's second kernel, windows, cu_seqlens and the
 *     history lengths out_len (that kernel starts early only after the call's first kernel,
 *     which writes none of them, has itself waited for everything before it). Tiers and every
 *     output wait for the previous kernel. A kernel of the caller's that precedes a call on
 *     the stream and triggers its dependents early (griddepcontrol.launch_dependents) must
 *     have written those inputs before it triggers; kernels launched without that trigger
 *     need nothing.
 *   - Return value: DSPARK_OK, or a negative DSPARK_ERR_* code when the host-side argument check
 *     or the kernel launch failed. On error nothing was enqueued (argument errors) or the launch
 *     was refused (DSPARK_ERR_CUDA); dspark_last_error() then describes it.
 *   - Data-dependent problems that only the device can see (a total beyond the largest tier,
 *     a window outside [1,gamma], an output history that is full, ...) never fault and never
 *     trap: the kernel ORs a DSPARK_STATUS_* bit into the caller's int32 `status` word, applies
 *     the documented clamp and carries on. The caller zeroes `status` when it wants a fresh
 *     report and reads it whenever convenient.
 *   - No kernel waits on another kernel or a peer. The only waits are inside one CTA (the
 *     bulk-copy verify kernel's shared-memory stages); each is bounded, and one that gives up
 *     sets DSPARK_STATUS_STALL instead of hanging.
 */
#ifndef DSPARK_H_
#define DSPARK_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---------------------------------------------------------------------- */
#define DSPARK_OK                  0
#define DSPARK_ERR_INVALID_ARG   (-1)  /* null pointer, bad size, bad enum, short workspace */
#define DSPARK_ERR_UNSUPPORTED   (-2)  /* valid request beyond the library's limits          */
#define DSPARK_ERR_CUDA          (-3)  /* the CUDA runtime refused a query or a launch       */

/* ---- device status bits (OR-ed into the caller's int32 status word) -------------------- */
#define DSPARK_STATUS_TIER_OVERFLOW  0x01 /* M above every tier: tier := M (pack)                */
#define DSPARK_STATUS_PACK_CAPACITY  0x02 /* tier above packed_cap: rows >= packed_cap unwritten */
#define DSPARK_STATUS_BAD_WINDOW     0x04 /* a window outside [1,gamma]: clamped into it        */
#define DSPARK_STATUS_OUT_OVERFLOW   0x08 /* a history reached out_cap: tokens past it dropped   */
#define DSPARK_STATUS_BAD_COST       0x10 /* no K had a finite positive T: K* := 0               */
#define DSPARK_STATUS_BAD_ROWS       0x20 /* a request's rows lie outside the verified rows      */
#define DSPARK_STATUS_BAD_TOKEN      0x40 /* a draft id outside [0,V): treated as rejected       */
#define DSPARK_STATUS_BAD_LENGTH     0x80 /* accept_len / out_len outside range: clamped         */
#define DSPARK_STATUS_STALL         0x100 /* a bounded in-kernel wait gave up: this call's verify
                                             results are invalid (not expected in operation)   */

/* ---- limits of the library ----------------------------------------------------------- */
#define DSPARK_MAX_GAMMA        32     /* block width                                         */
#define DSPARK_MAX_CANDIDATES   16384  /* B*(gamma-1): the scheduler sorts them in one CTA    */
#define DSPARK_MAX_BATCH        8192   /* B for schedule and pack (single-CTA scans)          */
#define DSPARK_MAX_TIERS        1024

typedef enum { DSPARK_BF16 = 0, DSPARK_F32 = 1 } dspark_dtype;

/* Verify modes ("A2 method details", verify-mode design):
 *   STATIC     verifies the whole block every step: w_b := gamma, commits the full-block accept.
 *   COMPACT    verifies only the scheduled window: logits hold the packed rows of cu_seqlens.
 *   CAP_ACCEPT verifies the whole block but commits exactly what COMPACT would commit; it also
 *              reports the accept length full verification would have given (the ceiling).  */
typedef enum { DSPARK_STATIC = 0, DSPARK_COMPACT = 1, DSPARK_CAP_ACCEPT = 2 } dspark_mode;

/* Additive step-cost model T(bs,K) = bias + alpha(bs) + theta(bs+K) ("A2 method details",
 * cost-table profiling and modelling). Host struct; `alpha` and `theta` are DEVICE arrays of
 * doubles indexed by bs and by M = bs+K. dspark_schedule reads alpha[B] and theta[B..B*gamma],
 * so alpha_len >= B+1 and theta_len >= B*gamma+1. The struct itself is read during the call
 * only and may live on the host stack. */
typedef struct {
    double        bias;
    const double* alpha;
    int32_t       alpha_len;
    const double* theta;
    int32_t       theta_len;
} dspark_cost;

/* ---------------------------------------------------------------------------------------
 * dspark_schedule — confidence scheduler ("A2 method details": the confidence head's scores
 * multiply along the block into a survival probability; the scheduler turns survivals into
 * per-request verify budgets by trading expected accepted tokens against the cost table).
 *
 *   s[b,j]   = prod_{i<=j} clamp(conf[b,i], 0, 1)           fp32, sequential, j = 0..gamma-2
 *   key[b,j] = round_to_nearest_even(s[b,j] * 2^32)         exact uint64 fixed point
 *   order    = keys descending; ties by b ascending, then j ascending
 *   S(K)     = sum of the first K keys in that order          (exact integer)
 *   obj(K)   = double(B*2^32 + S(K)) / T,  T = (bias + alpha[B]) + theta[B+K]
 *   K*       = the smallest K in [0, B*(gamma-1)] with the largest obj among K whose T is finite
 *              and positive (none: K* = 0 and DSPARK_STATUS_BAD_COST)
 *   w_b      = 1 + number of request b's entries among the first K* in the order
 *
 * conf     [B, gamma-1] fp32 (NaN counts as 0)       windows [B] int32 out    k_star [1] int32 out
 * status   [1] int32 in/out (may be NULL: the bits are then dropped)
 * Limits: 0 <= B <= DSPARK_MAX_BATCH, 1 <= gamma <= DSPARK_MAX_GAMMA,
 *         B*(gamma-1) <= DSPARK_MAX_CANDIDATES. B == 0 writes k_star = 0 only.
 * One single-CTA kernel; no workspace.
 * ------------------------------------------------------------------------------------- */
int dspark_schedule(const float* conf, int B, int gamma, const dspark_cost* cost,
                    int32_t* windows, int32_t* k_star, int32_t* status, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * dspark_pack — ragged front-pack ("A2 method details", ragged verify over full CUDA graphs:
 * variable windows are packed to the front of one compact cu_seqlens-style buffer and only the
 * total is rounded up to the nearest captured graph tier).
 *
 *   w_b         = clamp(windows[b], 1, gamma)   (out of range: DSPARK_STATUS_BAD_WINDOW)
 *   cu_seqlens  = exclusive scan of w: cu[0] = 0, cu[b+1] = cu[b] + w_b, M = cu[B]
 *   tier        = min{ tiers[t] : tiers[t] >= M }; none: tier = M, DSPARK_STATUS_TIER_OVERFLOW
 *   rows r < M  : packed_ids[r] = block_tokens[b, i], row_req[r] = b, row_pos[r] = i
 *                 for the unique (b, i < w_b) with r = cu[b] + i
 *   rows M..tier-1 (padding): packed_ids = 0, row_req = -1, row_pos = -1
 *   rows >= packed_cap are never written (DSPARK_STATUS_PACK_CAPACITY if tier > packed_cap)
 *   meta        = { M, tier }
 *
 * windows [B] int32          block_tokens [B, gamma] int32 (column 0 = anchor, 1.. = drafts)
 * tiers [n_tiers] int32 device, any order      cu_seqlens [B+1] int32 out
 * packed_ids, row_req, row_pos [packed_cap] int32 out (row_req/row_pos may be NULL)
 * meta [2] int32 out          status [1] int32 in/out or NULL
 * Limits: 0 <= B <= DSPARK_MAX_BATCH, 1 <= gamma <= DSPARK_MAX_GAMMA,
 *         1 <= n_tiers <= DSPARK_MAX_TIERS, packed_cap >= 0.
 * ------------------------------------------------------------------------------------- */
int dspark_pack(const int32_t* windows, const int32_t* block_tokens, int B, int gamma,
                const int32_t* tiers, int n_tiers, int32_t* cu_seqlens,
                int32_t* packed_ids, int32_t* row_req, int32_t* row_pos, int packed_cap,
                int32_t* meta, int32_t* status, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * dspark_schedule_pack — dspark_schedule followed by dspark_pack of the windows it writes, in
 * one kernel ("A2 method details", performance: the step's small operations fused to cut the
 * per-step cost; the scheduler's verify-length selection and the ragged window pack are two
 * of the kernels the pages list). Every output (windows, k_star, cu_seqlens, packed_ids,
 * row_req, row_pos, meta, status bits) equals what the two calls in sequence produce; the
 * arguments mean what they mean there, with the same limits and the same errors (messages
 * name dspark_schedule_pack). B == 0 or gamma == 1 run the two plain kernels.
 * ------------------------------------------------------------------------------------- */
int dspark_schedule_pack(const float* conf, int B, int gamma, const dspark_cost* cost,
                         const int32_t* block_tokens, const int32_t* tiers, int n_tiers,
                         int32_t* windows, int32_t* k_star, int32_t* cu_seqlens,
                         int32_t* packed_ids, int32_t* row_req, int32_t* row_pos,
                         int packed_cap, int32_t* meta, int32_t* status, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * dspark_verify — verify over the target logits and reduce to per-request accept lengths.
 *
 * Rows. Target row for (request b, block position i):
 *   COMPACT              row cu_seqlens[b] + i, i < w_b         (target_logits = packed [M, V])
 *   STATIC, CAP_ACCEPT   row b*gamma + i,       i < gamma       (target_logits = block [B*gamma, V])
 * The call verifies rows [0, N): N = cu_seqlens[B] (COMPACT: the packed total M) or B*gamma
 * (STATIC, CAP_ACCEPT), capped at target_rows and at B*gamma; no other row is read.
 * target row (b,i) is the target's distribution for block position i+1, which holds the draft
 * d_{i+1} = block_tokens[b, i+1]. Draft row (b,i) of draft_logits [B, gamma-1, V] is the draft
 * distribution that d_{i+1} was sampled from (stochastic only).
 * A request with a row outside [0, N) (outside the buffer, or, COMPACT, at or past
 * cu_seqlens[B]) flags DSPARK_STATUS_BAD_ROWS and commits nothing (accept_len 0, committed
 * all -1). So does, COMPACT, a request whose rows that carry its accept tests reach into the
 * next request's rows (cu_seqlens[b+1] < cu_seqlens[b] + w_b - 1): each packed row is one
 * request's, although a request's last row may be shared. The exclusive scan of the windows
 * that dspark_pack writes meets both rules; with rows shared otherwise, row_prob of a shared
 * row holds either request's values. COMPACT needs cu_seqlens non-decreasing: where it
 * decreases, the requests whose rows it reorders get undefined accept lengths and tokens
 * (every row index is still checked: no fault).
 *
 * Greedy (stochastic == 0): g[b,i] = argmax_v target[row(b,i), v] (lowest v on ties; NaN
 *   unsupported). d_{i+1} is accepted iff d_{i+1} == g[b,i]; L = 1 + number of leading accepts;
 *   committed[b, k] = g[b, k] for k < L (the accepted drafts followed by the target's token).
 *
 * Stochastic (stochastic == 1; the min(1, p/q) rule of the lshu.cn article, sections 2.3/3.3):
 *   p = softmax(target_row / temperature), q = softmax(draft_row / temperature) over all V.
 *   Uniforms come from Philox4x64-10 (Salmon et al., SC'11) with key (seed, 0) and counter
 *   (b, i, step, 0): word 0 gives u = (w0 >> 40) * 2^-24 for the accept test of d_{i+1},
 *   word 1 gives u' = (w1 >> 11) * 2^-53 for a bonus drawn at position i.
 *   d_{i+1} is accepted iff q(d) == 0 or u < float(p(d) / q(d)).
 *   First rejection at position i: the bonus is drawn from the residual max(0, p - q) of row i
 *   (normalised); no rejection among the w_b - 1 drafts: the bonus is drawn from p of row
 *   w_b - 1. Drawing: the smallest v whose running sum (in v order) exceeds u' * total.
 *   committed[b] = d_1 .. d_{L-1}, bonus.
 *
 * Modes: STATIC uses w_b := gamma. CAP_ACCEPT commits exactly what COMPACT commits for the same
 *   windows (its decisions and bonus depend on rows i < w_b only) and writes
 *   ceiling_len[b] = the accept length over all gamma-1 drafts. STATIC writes ceiling_len =
 *   accept_len; COMPACT writes -1 (when ceiling_len != NULL).
 *
 * target_logits [target_rows, V] bf16 or fp32 (dtype); draft_logits [B, gamma-1, V] same dtype
 *   (stochastic only, else NULL). cu_seqlens [B+1] (COMPACT only, else may be NULL).
 * windows [B] int32 (COMPACT/CAP_ACCEPT; clamped to [1,gamma], DSPARK_STATUS_BAD_WINDOW)
 * block_tokens [B, gamma] int32; ids outside [0,V) flag DSPARK_STATUS_BAD_TOKEN and reject.
 * accept_len [B] int32 out; committed [B, gamma] int32 out (-1 after the L committed tokens);
 * ceiling_len [B] int32 out or NULL; row_prob [target_rows, 2] fp32 out or NULL: (p(d), q(d))
 *   of every target row that carries a stochastic accept test, (-1, -1) on the other rows of a
 *   request (always -1 in greedy mode).
 * workspace: device scratch of at least dspark_verify_workspace_bytes(B, gamma, V, stochastic)
 *   bytes, 16-byte aligned, owned by the caller; no clearing needed. Its first 256 bytes carry
 *   state from one call to the next: the bulk-copy streaming kernel hands out most of its
 *   work from a counter there (bytes 4-7), and each call leaves that counter at zero,
 *   between a 32-bit tag (bytes 0-3) and a 64-bit tag (bytes 8-15), for the next call. A call
 *   that finds either tag missing (a fresh or zeroed workspace, or one whose first bytes were
 *   written since) splits its work evenly instead, with identical results. Between two calls
 *   that share a workspace, leave those 256 bytes as the last call left them or zero them;
 *   the rest is rewritten by every call before it is read. Calls that share one workspace must
 *   not overlap on the GPU.
 * Limits: 0 <= B, 1 <= gamma <= DSPARK_MAX_GAMMA, V >= 1, temperature > 0 (stochastic).
 * Kernels: a persistent streaming kernel over fixed row chunks (register or TMA bulk-copy
 * streaming, see dspark_set_stream_kernel), then, greedy: a finaliser (256 threads or more per
 * request, one to four requests per CTA) that combines the chunk results, walks and writes
 * the outputs; stochastic: a bonus kernel spread over the
 * grid whose CTAs each combine their request's chunk results and run its accept tests, sum
 * the bonus row's weights over their tiles; CTA 0 of a request writes its accept length,
 * drafts and ceiling, and the request's last CTA to finish draws the bonus token and, in
 * dspark_verify_scatter, appends the request's tokens.
 * ------------------------------------------------------------------------------------- */
int dspark_verify(dspark_mode mode, int stochastic,
                  const void* target_logits, int target_rows, const void* draft_logits,
                  dspark_dtype dtype, int V,
                  const int32_t* cu_seqlens, const int32_t* windows, const int32_t* block_tokens,
                  int B, int gamma, float temperature, uint64_t seed, uint64_t step,
                  int32_t* accept_len, int32_t* committed, int32_t* ceiling_len, float* row_prob,
                  void* workspace, size_t workspace_bytes, int32_t* status, cudaStream_t stream);

/* Bytes of device workspace dspark_verify needs for these sizes (0 when B == 0); a value
 * that depends on the sizes only. Returns 0 and sets dspark_last_error on invalid sizes. */
size_t dspark_verify_workspace_bytes(int B, int gamma, int V, int stochastic);

/* ---------------------------------------------------------------------------------------
 * dspark_scatter — compact scatter ("A2 method details", performance: the fused kernel that
 * writes accepted tokens back to per-request state).
 *   L = clamp(accept_len[b], 0, gamma), n = clamp(out_len[b], 0, out_cap)
 *   out_tokens[b, n + i] = committed[b, i] for i < L and n + i < out_cap
 *   out_len[b] = min(out_cap, n + L)   (tokens past out_cap: DSPARK_STATUS_OUT_OVERFLOW)
 * committed [B, gamma] int32; accept_len [B] int32; out_tokens [B, out_cap] int32 in/out;
 * out_len [B] int32 in/out; status [1] int32 in/out or NULL. Limits: B >= 0, 1 <= gamma <= 32.
 * ------------------------------------------------------------------------------------- */
int dspark_scatter(const int32_t* committed, const int32_t* accept_len, int B, int gamma,
                   int32_t* out_tokens, int32_t* out_len, int out_cap, int32_t* status,
                   cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * dspark_verify_scatter — dspark_verify followed by dspark_scatter of its committed tokens,
 * without the scatter's own launch ("A2 method details", performance: the compact scatter is
 * one of the fused kernels). Each request's tokens are appended by the CTA that decides them
 * (greedy: the finaliser; stochastic: the CTA that draws the bonus token). Every output,
 * including out_tokens, out_len and the status bits, equals what dspark_verify then
 * dspark_scatter(committed, accept_len, B, gamma, out_tokens, out_len, out_cap) produce; the
 * arguments, limits and errors are those two calls' (messages name dspark_verify_scatter).
 * ------------------------------------------------------------------------------------- */
int dspark_verify_scatter(dspark_mode mode, int stochastic,
                          const void* target_logits, int target_rows, const void* draft_logits,
                          dspark_dtype dtype, int V,
                          const int32_t* cu_seqlens, const int32_t* windows,
                          const int32_t* block_tokens, int B, int gamma, float temperature,
                          uint64_t seed, uint64_t step, int32_t* accept_len, int32_t* committed,
                          int32_t* ceiling_len, float* row_prob, void* workspace,
                          size_t workspace_bytes, int32_t* out_tokens, int32_t* out_len,
                          int out_cap, int32_t* status, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * dspark_set_stream_kernel — which kernel streams the logits inside dspark_verify and
 * dspark_verify_scatter, for every later call in this process:
 *   DSPARK_STREAM_AUTO (0, the default): the library's choice;
 *   DSPARK_STREAM_REGISTER (1): warps stream 16-byte loads into registers;
 *   DSPARK_STREAM_BULK (2): a producer warp per CTA moves whole chunks into shared memory with
 *     the TMA bulk-copy engine (cp.async.bulk, mbarrier completion) and four warps fold them;
 *     used when the logit rows are 16-byte aligned and V % 8 == 0, else the register kernel.
 * AUTO takes the bulk kernel when B*gamma rows of V logits reach 64 MB, else the register one.
 * Both fold every chunk in the same order, so results are bit-identical whichever runs; only
 * speed differs. Not thread-safe against concurrent verify calls. Returns DSPARK_OK or
 * DSPARK_ERR_INVALID_ARG for an unknown value.
 * ------------------------------------------------------------------------------------- */
#define DSPARK_STREAM_AUTO      0
#define DSPARK_STREAM_REGISTER  1
#define DSPARK_STREAM_BULK      2
int dspark_set_stream_kernel(int which);

/* ---------------------------------------------------------------------------------------
 * dspark_set_stream_events — measurement hook: every later dspark_verify /
 * dspark_verify_scatter call records `start` on its stream just before its logit-streaming
 * kernel and `stop` just after it, so that the caller can time that kernel alone
 * (cudaEventElapsedTime). Both NULL switch it off (the default). The events belong to the
 * caller and must outlive the calls that record them. An event between two kernels stops the
 * next one from starting early (programmatic dependent launch), so a timed call runs slightly
 * slower than an untimed one. Not thread-safe against concurrent verify calls. Returns
 * DSPARK_OK, or DSPARK_ERR_INVALID_ARG when exactly one of the two is NULL.
 * ------------------------------------------------------------------------------------- */
int dspark_set_stream_events(cudaEvent_t start, cudaEvent_t stop);

/* ---------------------------------------------------------------------------------------
 * dspark_observe — calibration and utilisation counters ("A2 method details", observability:
 * per-request confidence and calibration metrics such as ECE; cap-accept recovers the
 * acceptance ceiling that truncation hides, and utilisation is committed over ceiling).
 *
 * c_b = clamp(ceiling_len[b], 1, gamma) is request b's accept length over the full block (the
 * ceiling_len of a CAP_ACCEPT or STATIC verify). Draft j (0-based: the draft d_{j+1} scored by
 * conf[b, j]) is observed when j <= c_b - 1 and j <= gamma - 2: accepted (1) if j < c_b - 1,
 * rejected (0) if j == c_b - 1; later drafts are censored. Each observed draft, with
 * x = clamp(conf[b, j], 0, 1) (NaN counts as 0), adds to bin k = min(n_bins - 1, floor(x * n_bins))
 *   hist[3k] += 1,  hist[3k + 1] += round_to_nearest_even(x * 2^32),  hist[3k + 2] += outcome
 * and util[0] += clamp(accept_len[b], 0, gamma), util[1] += c_b. All counters are uint64 and
 * exact, so the result does not depend on the order of the atomic additions. Expected
 * calibration error = sum_k (hist[3k]/N) |hist[3k+2]/hist[3k] - hist[3k+1]/(2^32 hist[3k])|,
 * utilisation = util[0] / util[1]. Counters accumulate across calls; the caller zeroes them.
 * Out-of-range ceiling_len / accept_len are clamped and flag DSPARK_STATUS_BAD_LENGTH.
 *
 * conf [B, gamma-1] fp32; accept_len, ceiling_len [B] int32; hist [3 * n_bins] uint64 in/out;
 * util [2] uint64 in/out; status [1] int32 in/out or NULL.
 * Limits: B >= 0, 1 <= gamma <= DSPARK_MAX_GAMMA, 1 <= n_bins <= 1024.
 * ------------------------------------------------------------------------------------- */
int dspark_observe(const float* conf, const int32_t* accept_len, const int32_t* ceiling_len,
                   int B, int gamma, int n_bins, uint64_t* hist, uint64_t* util,
                   int32_t* status, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * dspark_graph_begin / dspark_graph_end / dspark_graph_launch / dspark_graph_destroy — one or
 * more whole decode steps captured once as a CUDA graph and replayed with a single launch
 * ("A2 method details", ragged verify over full CUDA graphs, figure 2).
 *
 * dspark_graph_begin(stream) starts a stream capture (thread-local mode) on `stream`; every
 * call of this library the caller then issues on that stream (and any other work on it) is
 * recorded instead of run. dspark_graph_end(stream, &graph) ends the capture and instantiates
 * it; *graph receives an opaque handle (host memory owned by the library until
 * dspark_graph_destroy). dspark_graph_launch(graph, stream) replays the whole recording with
 * one cudaGraphLaunch on any stream of the same device. Replays use the pointers and scalars
 * of the captured calls: new inputs are written into the same buffers before a replay. The
 * library's kernels read M, the windows and the tier on the device, so one graph serves every
 * window allocation and every tier. Kernels keep their programmatic-dependent-launch edges in
 * the graph. Make one eager call of each captured entry point on the device before the
 * capture (per-device set-up such as shared-memory opt-ins happens on the first call).
 * Errors: DSPARK_ERR_INVALID_ARG for the legacy default stream or NULL handles,
 * DSPARK_ERR_CUDA when the runtime refuses the capture, its end, the instantiation or the
 * launch (dspark_last_error names which). dspark_graph_destroy(NULL) does nothing.
 * ------------------------------------------------------------------------------------- */
typedef struct dspark_graph_s* dspark_graph;
int dspark_graph_begin(cudaStream_t stream);
int dspark_graph_end(cudaStream_t stream, dspark_graph* graph);
int dspark_graph_launch(dspark_graph graph, cudaStream_t stream);
int dspark_graph_destroy(dspark_graph graph);

/* ---------------------------------------------------------------------------------------
 * dspark_verify_noalloc — the pages have no counterpart to this entry point; it exists for
 * callers that cannot hand the library scratch memory. Some hosts give a kernel library only
 * its input and output buffers (a plugin interface with no workspace argument), and some
 * serving loops reserve nearly all device memory for the KV cache before decoding starts and
 * must not call cudaMalloc in the middle of a step, where the allocation can fail or
 * synchronise the device and stall the overlapped scheduler.
 *
 * Same arguments, outputs and results as dspark_verify, minus the workspace: the scratch is a
 * static device array of DSPARK_NOALLOC_SCRATCH_BYTES inside this library, which every GPU
 * that loads the library keeps until the process exits. The call allocates nothing.
 *   - Sizes whose dspark_verify_workspace_bytes(B, gamma, V, stochastic) exceeds
 *     DSPARK_NOALLOC_SCRATCH_BYTES are rejected with DSPARK_ERR_UNSUPPORTED and a message.
 *   - Each call looks up the array's device address in the current device's context
 *     (cudaGetSymbolAddress: on the first call this loads the library's device code on that
 *     device, so make that first call before any stream capture).
 *   - Every call on a device shares the one array and leaves its contents behind. Nothing in
 *     it needs to start at zero (each call rewrites what it reads), but calls that overlap on
 *     the GPU — on different streams, or from different host threads — race on it: order
 *     them on one stream or synchronise between them.
 * ------------------------------------------------------------------------------------- */
#define DSPARK_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)  /* 4 MiB per device */
int dspark_verify_noalloc(dspark_mode mode, int stochastic,
                          const void* target_logits, int target_rows, const void* draft_logits,
                          dspark_dtype dtype, int V,
                          const int32_t* cu_seqlens, const int32_t* windows,
                          const int32_t* block_tokens, int B, int gamma, float temperature,
                          uint64_t seed, uint64_t step, int32_t* accept_len, int32_t* committed,
                          int32_t* ceiling_len, float* row_prob, int32_t* status,
                          cudaStream_t stream);

/* Message of the last failed call on this host thread ("" if none). Never NULL. */
const char* dspark_last_error(void);

/* ABI version: 100 * major + minor (1.1: the dspark_graph_* capture and replay calls; 1.2: a
 * 256-byte head in the verify workspace, and a stochastic workspace without per-request bonus
 * jobs). */
int dspark_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_H_ */
