/*
 * dspark.h -- C-ABI of libdspark: batched speculative verification and the
 * hardware-aware prefix scheduler of DSpark, on one GB300 GPU (sm_103a).
 *
 * Method: "DSpark: Confidence-Scheduled Speculative Decoding with
 * Semi-Autoregressive Generation" (DeepSeek-AI / Peking University).
 *   - dspark_verify: section 2.1 "Speculative Decoding" (accept x_k with
 *     probability min(1, p_t^k(x_k) / p_d^k(x_k)), left to right, the first
 *     rejection discards the rest of the block), section 1 (append one bonus
 *     token), Appendix 8 (with nothing admitted the target samples a fresh token
 *     from p_t). The residual distribution after a rejection,
 *     max(0, p_t - p_d) renormalised, is the standard rule of the speculative
 *     sampling papers the DSpark paper cites as [1] and [2].
 *   - dspark_schedule: section 3.2.2 "Hardware-Aware Prefix Scheduler" and
 *     Algorithm 1 of the Chinese translation page (prefix survival products,
 *     global descending sort, greedy admission, early stop at the first
 *     Theta <= Theta_best).
 *
 * Conventions for both calls:
 *   - Every pointer is a DEVICE pointer to memory owned by the caller, unless
 *     stated otherwise. The library allocates nothing, never synchronises the
 *     host with the device, and enqueues all its work on `stream`.
 *   - The return value reports errors detectable on the host before any launch
 *     (DSPARK_ERR_INVALID_ARG, DSPARK_ERR_WORKSPACE) and launch failures
 *     (DSPARK_ERR_CUDA). Nothing is enqueued when a host check fails.
 *   - Errors in the data (a token outside [0, V), a verify length outside
 *     [0, gamma], a uniform outside [0, 1), inconsistent row offsets, a
 *     confidence outside [0, 1] or NaN, non-finite row statistics) are found on
 *     the device and written to *device_status (DSPARK_ERR_BAD_DATA); the first
 *     error recorded wins. The caller reads it after its own synchronisation.
 *     Outputs for the affected requests are then unspecified but every write
 *     stays inside the output buffers. A bounded wait that gives up writes
 *     DSPARK_ERR_TIMEOUT. The library never traps or asserts on the device.
 *   - The first call on each device sets kernel attributes (dynamic shared
 *     memory limits); make one call before capturing a CUDA graph.
 *   - Calls that share a workspace must not overlap on the GPU.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t / CUstream */

typedef enum {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = 1,
  DSPARK_ERR_CUDA = 2,
  DSPARK_ERR_WORKSPACE = 3,
  DSPARK_ERR_TIMEOUT = 4,
  DSPARK_ERR_BAD_DATA = 5,
  DSPARK_ERR_TOO_LARGE = 6 /* batch needs more scratch than dspark_verify_static has */
} dspark_status;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

#define DSPARK_MAX_GAMMA 32
/* Bytes of one row that form one work unit (one partial statistic) of the
   row-statistics pass. */
#define DSPARK_TILE_BYTES 16384
/* Tokens per segment of the inverse-CDF (resample) pass. */
#define DSPARK_RESAMPLE_SEG 2048
/* Near-tie windows: |u - ratio| < 1e-6 for a ratio test, |u*Z - C| < 1e-6*Z
   for an inverse-CDF cut, |Theta(n) - Theta(n-1)| <= 1e-9*Theta(n-1) for a
   scheduler comparison. Decisions inside a window are counted in
   *near_tie_count; outside every window the results are exact functions of
   the inputs. */
#define DSPARK_TIE_EPS 1e-6
#define DSPARK_SCHED_TIE_REL 1e-9

#define DSPARK_ALIGN256(x) ((((size_t)(x)) + 255u) & ~(size_t)255u)
#define DSPARK_CEILDIV(a, b) ((((size_t)(a)) + ((size_t)(b)) - 1u) / ((size_t)(b)))
/* Work units per logit row (sized for 4-byte logits, the larger count). */
#define DSPARK_TILES_PER_ROW(V) DSPARK_CEILDIV((V), DSPARK_TILE_BYTES / 4)
#define DSPARK_SEGS_PER_ROW(V) DSPARK_CEILDIV((V), DSPARK_RESAMPLE_SEG)
#define DSPARK_MAX_ROWS(B, gamma) ((size_t)(B) * (2u * (size_t)(gamma) + 1u))

/* Workspace of dspark_verify, in bytes (256-byte aligned regions):
   header, per-request row starts, row list, per-tile row statistics,
   per-request resample descriptors, per-segment residual sums, tickets. */
#define DSPARK_VERIFY_WS_BYTES(B, gamma, V)                                   \
  ((size_t)256 + DSPARK_ALIGN256(((size_t)(B) + 1u) * 4u) +                   \
   DSPARK_ALIGN256(DSPARK_MAX_ROWS(B, gamma) * 8u) +                          \
   DSPARK_ALIGN256(DSPARK_MAX_ROWS(B, gamma) * DSPARK_TILES_PER_ROW(V) * 16u) + \
   DSPARK_ALIGN256((size_t)(B) * 64u) +                                       \
   DSPARK_ALIGN256((size_t)(B) * DSPARK_SEGS_PER_ROW(V) * 8u) +               \
   DSPARK_ALIGN256((size_t)(B) * 4u))

/* Workspace of dspark_acceptance, in bytes: dspark_verify's workspace, then
   one job record per position and its per-segment sums. */
#define DSPARK_ACCEPTANCE_WS_BYTES(B, gamma, V)                               \
  (DSPARK_VERIFY_WS_BYTES(B, gamma, V) +                                      \
   DSPARK_ALIGN256((size_t)(B) * (size_t)(gamma) * 64u) +                     \
   DSPARK_ALIGN256((size_t)(B) * (size_t)(gamma) * DSPARK_SEGS_PER_ROW(V) * 8u))

/* Vocabulary entries per tensor-core tile and per softmax statistic of the
   drafter, and the largest Markov-head rank it takes. */
#define DSPARK_DRAFT_TILE 128
#define DSPARK_DRAFT_MAX_RANK 256
/* Workspace of dspark_draft_markov, in bytes: the gathered embedding rows
   W1[x_{k-1}] of the batch, two buffers of one statistic per (request, tile),
   the grid-barrier words, one ready flag per request (each on a 128-byte line
   of its own), one barrier per request tile (4 KiB) and (2 MiB) the single
   launch's per-range masses: two position parities x 256 CTAs at most x 128
   requests x 2 records of 16 bytes. */
#define DSPARK_DRAFT_WS_BYTES(B, r, V)                                        \
  (DSPARK_ALIGN256((size_t)(B) * (size_t)(r) * 2u) +                          \
   2u * DSPARK_ALIGN256((size_t)(B) * DSPARK_CEILDIV((V), DSPARK_DRAFT_TILE) * 8u) + \
   256u + DSPARK_ALIGN256((size_t)(B) * 128u) + 4096u + ((size_t)2u << 20))

/* Workspace of dspark_schedule, in bytes: two (key, index) buffers for the
   sort, per-request lengths and a header. */
#define DSPARK_SCHEDULE_WS_BYTES(R, gamma)                                    \
  ((size_t)256 + 2u * DSPARK_ALIGN256((size_t)(R) * (size_t)(gamma) * 8u) +     \
   2u * DSPARK_ALIGN256((size_t)(R) * (size_t)(gamma) * 4u) +                   \
   DSPARK_ALIGN256((size_t)(R) * 4u))

/*
 * dspark_verify -- one batched verification step (DSpark paper, section 2.1).
 *
 * For every request r with verify length l_r = verify_len[r] (0 <= l_r <=
 * gamma), position k = 1..l_r is tested with the temperature-scaled softmax of
 * target row k and draft row k at the draft token x_k = draft_tokens[r][k-1]:
 *   p(v) = exp(z_v/T - M) / sum_w exp(z_w/T - M),  M = max_w z_w/T,
 *   accept x_k  iff  uniforms[r][k-1] < p_t^k(x_k) / p_d^k(x_k),
 * scanning left to right; the first rejection ends the block. With m tests
 * passed: if m < l_r the token after the block is drawn from
 * q = max(0, p_t^{m+1} - p_d^{m+1}) / Z, otherwise from p_t^{l_r+1} (the bonus
 * distribution; with l_r = 0 a fresh token from p_t^1), as the smallest token
 * id y whose running sum exceeds uniforms[r][gamma] * Z (Z = 1 for p_t).
 *
 * Arguments
 *   target_logits  [rows_t][V] row-major, dtype; request r's row k-1 holds
 *                  target position k (k = 1..l_r+1). Dense layout
 *                  (target_row_off == NULL): rows_t = B*(gamma+1), request r
 *                  starts at row r*(gamma+1). Ragged: starts at
 *                  target_row_off[r]; needs target_row_off[r+1] -
 *                  target_row_off[r] >= l_r + 1 and the buffer holds
 *                  target_row_off[B] rows.
 *   draft_logits   [rows_d][V]; request r's row k-1 holds draft position k
 *                  (k = 1..l_r). Dense: r*gamma; ragged: draft_row_off[r],
 *                  with draft_row_off[r+1] - draft_row_off[r] >= l_r.
 *   draft_tokens   [B][gamma] int32; only the first l_r of a request are read.
 *   verify_len     [B] int32.
 *   uniforms       [B][gamma+1] float32 in [0, 1): gamma ratio tests, then the
 *                  resample uniform.
 *   temperature    T > 0 and finite; divides target and draft logits alike.
 *   dtype          DSPARK_BF16 or DSPARK_F32 (both logit buffers).
 *   B >= 0, 1 <= gamma <= DSPARK_MAX_GAMMA, V >= 1.
 *   target_row_off, draft_row_off  [B+1] int64, both NULL (dense) or both set.
 *   accepted_len   out [B] int32: m.
 *   emitted_tokens out [B][gamma+1] int32: x_1..x_m, y, then -1.
 *   probs_out      out [B][gamma][2] float32 or NULL: (p_t^k(x_k), p_d^k(x_k))
 *                  for k <= l_r (computed for every verified position), -1 after.
 *   near_tie_count out [1] uint32 or NULL: decisions inside a near-tie window.
 *   device_status  out [1] int32 (required): DSPARK_OK or a data error.
 *   workspace      device scratch of at least DSPARK_VERIFY_WS_BYTES(B, gamma,
 *                  V) bytes, 256-byte aligned; no initial contents needed.
 *   stream         CUDA stream (NULL = legacy default stream).
 * Logit buffers must be 16-byte aligned for the TMA path; with rows whose byte
 * length is not a multiple of 16 a slower load path is used.
 */
int dspark_verify(const void* target_logits, const void* draft_logits,
                  const int32_t* draft_tokens, const int32_t* verify_len,
                  const float* uniforms, float temperature, int32_t dtype,
                  int32_t B, int32_t gamma, int32_t V,
                  const int64_t* target_row_off, const int64_t* draft_row_off,
                  int32_t* accepted_len, int32_t* emitted_tokens,
                  float* probs_out, uint32_t* near_tie_count,
                  int32_t* device_status, void* workspace,
                  size_t workspace_bytes, struct CUstream_st* stream);

/*
 * dspark_schedule -- hardware-aware prefix scheduler (DSpark paper, section
 * 3.2.2; Algorithm 1 of the Chinese translation page).
 *
 * a_{r,j} = prod_{i<=j} c_{r,i} (multiplied left to right in double); the
 * candidates (r, j) with a_{r,j} > 0 are sorted by a descending (equal values
 * keep the flattened order r*gamma + j - 1) and admitted one by one from
 * B = R, tau = R, Theta_best = R / T(R): each admission sets l_r = j,
 * B += 1, tau += a_{r,j}, Theta = tau / T(B) (that is tau * SPS(B) with
 * SPS = 1/T); the loop stops at the first Theta <= Theta_best.
 *
 * Arguments
 *   confidences   [R][gamma] float32, each in [0, 1].
 *   step_time_ms  [n_profile] float64: the profiled step time T(N) of a
 *                 target forward over N tokens, N = 0..n_profile-1; entries
 *                 for N in [R, R*(gamma+1)] must be > 0.
 *   n_profile     >= R*(gamma+1) + 1.
 *   R >= 1, 1 <= gamma <= DSPARK_MAX_GAMMA.
 *   verify_len    out [R] int32: the chosen l_r.
 *   theta_best    out [1] float64 or NULL.
 *   near_tie_count out [1] uint32 or NULL: evaluated comparisons inside the
 *                 1e-9 relative window.
 *   device_status out [1] int32 (required).
 *   workspace     at least DSPARK_SCHEDULE_WS_BYTES(R, gamma) bytes.
 */
int dspark_schedule(const float* confidences, const double* step_time_ms,
                    int64_t n_profile, int32_t R, int32_t gamma,
                    int32_t* verify_len, double* theta_best,
                    uint32_t* near_tie_count, int32_t* device_status,
                    void* workspace, size_t workspace_bytes,
                    struct CUstream_st* stream);

/*
 * dspark_schedule_capacity -- the production scheduler's capacity (DSpark
 * paper, section 5.2, "Hardware-Aware Prefix Scheduler in Practice").
 *
 * The same candidate order and Theta as dspark_schedule, without the
 * early-stopping break: n* = the first n in 0..|E| that maximises
 * Theta(n) = tau(n) / T(R + n), which steps over jagged drops of T. A serving
 * loop computes it from the confidences of two steps before and uses it as
 * the capacity K of dspark_schedule_topk, so that the admission of the current
 * step never waits for the search and the search never sees the current
 * step's tokens.
 *
 * Arguments are those of dspark_schedule, plus
 *   capacity      out [1] int32 (device, required): n*.
 *   verify_len    out [R] int32: the lengths of the best prefix itself.
 *   theta_best    out [1] float64 or NULL: Theta(n*).
 *   near_tie_count out [1] or NULL: admissions whose Theta lies within 1e-9
 *                 (relative) of the best before them.
 * Errors as in dspark_schedule; a NULL capacity is DSPARK_ERR_INVALID_ARG.
 */
int dspark_schedule_capacity(const float* confidences, const double* step_time_ms,
                             int64_t n_profile, int32_t R, int32_t gamma, int32_t* capacity,
                             int32_t* verify_len, double* theta_best,
                             uint32_t* near_tie_count, int32_t* device_status,
                             void* workspace, size_t workspace_bytes,
                             struct CUstream_st* stream);

/*
 * dspark_schedule_topk -- the production scheduler's admission (DSpark paper,
 * section 5.2): the candidates of the current confidences in the order of
 * dspark_schedule, the first min(K, |E|) of them admitted, K = *capacity read
 * on the device (typically written by an earlier dspark_schedule_capacity on
 * the same stream). l_r = the number of admitted positions of request r (a
 * prefix, since a_{r,j} does not increase with j).
 *
 * Arguments
 *   confidences   [R][gamma] float32, each in [0, 1].
 *   capacity      [1] int32 device (required); a negative value sets
 *                 DSPARK_ERR_BAD_DATA and admits nothing.
 *   R, gamma, verify_len, device_status, workspace, workspace_bytes, stream
 *                 as in dspark_schedule (same workspace size).
 */
int dspark_schedule_topk(const float* confidences, const int32_t* capacity, int32_t R,
                         int32_t gamma, int32_t* verify_len, int32_t* device_status,
                         void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * dspark_schedule_threshold -- the static-threshold baseline (DSpark paper,
 * section 4.3.3, "Static Threshold Sweep"): each request verifies its draft
 * tokens while their confidence reaches the threshold; the suffix from the
 * first token below it is pruned. l_r = max{ j : c_{r,i} >= threshold for all
 * i <= j }. It ignores the system load, which is what the prefix scheduler
 * adds; it serves as the comparison point.
 *
 * Arguments
 *   confidences   [R][gamma] float32, each in [0, 1] (else DSPARK_ERR_BAD_DATA
 *                 in *device_status; a NaN stops its request's prefix).
 *   threshold     finite float.
 *   R >= 1, 1 <= gamma <= DSPARK_MAX_GAMMA.
 *   verify_len    out [R] int32.
 *   device_status out [1] int32 (required).
 * No workspace; one launch on `stream`.
 */
int dspark_schedule_threshold(const float* confidences, float threshold, int32_t R,
                              int32_t gamma, int32_t* verify_len, int32_t* device_status,
                              struct CUstream_st* stream);

/*
 * dspark_acceptance -- the acceptance probability of every verified draft
 * position (DSpark paper, equation 8: P(accept x_k) = sum_v min(p_t^k(v),
 * p_d^k(v)) = 1 - TV(p_t^k, p_d^k); section 3.2.1 trains the confidence head
 * on it). For request r and k = 1..l_r: the temperature-scaled softmaxes of
 * target row k and draft row k, as in dspark_verify.
 *
 * Arguments are those of dspark_verify's logits, lengths and layout
 * (target_logits, draft_logits, verify_len, temperature, dtype, B, gamma, V,
 * target_row_off, draft_row_off), plus
 *   rates         out [B][gamma] float32: rates[r][k-1] for k <= l_r, -1
 *                 beyond (and for every position of an invalid request).
 *   device_status out [1] int32 (required), as in dspark_verify.
 *   workspace     at least DSPARK_ACCEPTANCE_WS_BYTES(B, gamma, V) bytes,
 *                 256-byte aligned; no initial contents needed.
 * It reads every verified row pair twice (the statistics pass, then the
 * minima), so it costs about two streaming passes; dspark_verify does not
 * compute it, dspark_verify_rates computes both with one statistics pass.
 */
int dspark_acceptance(const void* target_logits, const void* draft_logits,
                      const int32_t* verify_len, float temperature, int32_t dtype, int32_t B,
                      int32_t gamma, int32_t V, const int64_t* target_row_off,
                      const int64_t* draft_row_off, float* rates, int32_t* device_status,
                      void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * dspark_verify_rates -- dspark_verify and dspark_acceptance on the same
 * inputs in one call: the verification (section 2.1) and then the acceptance
 * probability of every verified position (equation 8) from the same row
 * statistics, so the rows are streamed for statistics once, not twice (the
 * label of section 3.2.1 for the verified positions of a serving step).
 *
 * Arguments are those of dspark_verify, plus
 *   rates         out [B][gamma] float32, as in dspark_acceptance (required
 *                 when B > 0, else DSPARK_ERR_INVALID_ARG).
 *   workspace     at least DSPARK_ACCEPTANCE_WS_BYTES(B, gamma, V) bytes
 *                 (else DSPARK_ERR_WORKSPACE), 256-byte aligned.
 * The verification outputs equal dspark_verify's and the rates equal
 * dspark_acceptance's, bit for bit. Errors as in dspark_verify.
 */
int dspark_verify_rates(const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const int32_t* verify_len,
                        const float* uniforms, float temperature, int32_t dtype, int32_t B,
                        int32_t gamma, int32_t V, const int64_t* target_row_off,
                        const int64_t* draft_row_off, int32_t* accepted_len,
                        int32_t* emitted_tokens, float* probs_out, uint32_t* near_tie_count,
                        float* rates, int32_t* device_status, void* workspace,
                        size_t workspace_bytes, struct CUstream_st* stream);

/* Size of the library-owned scratch array behind dspark_verify_static. */
#define DSPARK_STATIC_WS_BYTES ((size_t)16u << 20)

/*
 * dspark_verify_static -- dspark_verify for callers that cannot allocate
 * device memory. (The DSpark paper has no counterpart: this is a deployment
 * convenience of this library, not part of the method.)
 *
 * Some callers cannot call cudaMalloc: plugins that a host framework hands only
 * their input and output buffers, with no allocator of their own; serving loops
 * that must not call cudaMalloc because it can synchronise the whole device and
 * stall other streams; and processes that run under a device-memory budget
 * reserved up front. This entry point takes the same arguments as
 * dspark_verify minus the workspace, and computes the same results.
 *
 * Scratch: a file-scope device array of DSPARK_STATIC_WS_BYTES (16 MiB) inside
 * libdspark. Every GPU that loads the library holds it until the process exits.
 * The first call on each device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before
 * any stream capture. The address is kept per device and per context: after a
 * device reset (cudaDeviceReset, or another library resetting the primary
 * context) the next call finds a new context and looks the address up again,
 * so make one call outside stream capture after a reset too. No call
 * allocates or frees memory.
 *
 * Limits and sharing: a batch whose DSPARK_VERIFY_WS_BYTES(B, gamma, V)
 * exceeds DSPARK_STATIC_WS_BYTES is rejected with DSPARK_ERR_TOO_LARGE before
 * anything is launched (for example B = 256, gamma = 16, V = 129,280 needs
 * about 4.5 MB). All calls on a device share the one array, which keeps the
 * last call's contents; every call resets the counters that must start at zero
 * itself. Calls whose work overlaps on the GPU (different streams, or host
 * threads without ordering) race on the array: serialise them.
 *
 * Arguments, outputs and error behaviour are those of dspark_verify.
 */
int dspark_verify_static(const void* target_logits, const void* draft_logits,
                         const int32_t* draft_tokens, const int32_t* verify_len,
                         const float* uniforms, float temperature, int32_t dtype,
                         int32_t B, int32_t gamma, int32_t V,
                         const int64_t* target_row_off, const int64_t* draft_row_off,
                         int32_t* accepted_len, int32_t* emitted_tokens,
                         float* probs_out, uint32_t* near_tie_count,
                         int32_t* device_status, struct CUstream_st* stream);

/*
 * dspark_draft_markov -- the sequential stage of the DSpark drafter with the
 * Markov head (DSpark paper, section 3.1 "Sequential stage", equations 4 and
 * 5): gamma draft tokens per request, drawn left to right.
 *
 * For request b and k = 1..gamma, with x_0 = anchors[b]:
 *   bias(v) = sum_j W1[x_{k-1}][j] * W2[j][v]          (equation 5)
 *   L_k(v)  = bf16(fl32(U_k(v) + bias(v)))              (the emitted draft row)
 *   x_k     = smallest v whose running sum of exp(L_k/T - M) exceeds
 *             uniforms[b][k-1] * Z                     (equation 4 at T)
 * The bias is accumulated in binary32 on the tensor cores (exact whenever every
 * partial sum is, e.g. weights on a 2^-8 grid), added to U_k, rounded to
 * binary32, then to bf16 (ties to even). The tokens are drawn from the emitted
 * rows themselves, so a verifier reading draft_logits sees exactly the draft
 * distribution p_d^k the tokens came from.
 *
 * Arguments
 *   base_logits   [B][gamma][V] bf16: U_k of the parallel stage, request b's
 *                 position k at row b*gamma + k-1 (the dense draft-row layout
 *                 of dspark_verify).
 *   w1            [V][r] bf16: the embedding table W1.
 *   w2t           [V][r] bf16: W2 transposed (row v holds W2[0..r-1][v]).
 *   anchors       [B] int32: x_0, the last token of the previous cycle.
 *   uniforms      [B][gamma] float32 in [0, 1): one per position.
 *   temperature   T > 0 and finite.
 *   B >= 0 (B = 0 does nothing), 1 <= gamma <= DSPARK_MAX_GAMMA,
 *   V >= 8 a multiple of 8, r in {64, 128, 192, 256}.
 * Outputs
 *   draft_logits  [B][gamma][V] bf16: L_k. May be the same buffer as
 *                 base_logits (overwritten in place); otherwise disjoint.
 *   draft_tokens  [B][gamma] int32: x_1..x_gamma.
 *   device_status DSPARK_ERR_BAD_DATA for an anchor outside [0, V), a uniform
 *                 outside [0, 1), a NaN or +inf logit, or a row whose logits
 *                 are all -inf (that request's token is then 0).
 *   workspace     at least DSPARK_DRAFT_WS_BYTES(B, r, V) bytes, 256-byte
 *                 aligned; no state is kept in it between calls.
 * base_logits, w1, w2t and draft_logits must be 16-byte aligned (the tensor
 * memory access unit copies 16-byte aligned boxes); otherwise, and for
 * arguments outside the ranges above, DSPARK_ERR_INVALID_ARG.
 */
int dspark_draft_markov(const void* base_logits, const void* w1, const void* w2t,
                        const int32_t* anchors, const float* uniforms,
                        float temperature, int32_t B, int32_t gamma, int64_t V,
                        int32_t r, void* draft_logits, int32_t* draft_tokens,
                        int32_t* device_status, void* workspace,
                        size_t workspace_bytes, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
