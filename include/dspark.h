/*
 * dspark.h — C ABI of the DSpark per-round speculative-decoding hot path on GB300
 * (sm_103a): Markov-head draft -> confidence scheduler -> exact verification, with the
 * recurrent-head draft, verification on a flattened target batch, the fixed-cutoff
 * scheduler, the acceptance-overlap diagnostic and sequential temperature scaling.
 *
 * The method is the one described on the pages about DSpark (Cheng, Yu, Shao et al.,
 * "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
 * Generation", arXiv 2607.05147):
 *   - numb3r33 blog "DSpark: confidence-scheduled speculative decoding" (sections
 *     "One-token exactness", "Prefix survival and accepted length", "Markov sequential
 *     head", "RNN sequential head", "Confidence head", "Total variation label",
 *     "Sequential temperature scaling", "Scheduler objective", "Greedy prefix
 *     allocation", "Async scheduler in practice", "Variable-length verification without
 *     wasting kernels");
 *   - vllmbangkok blog "DSpark: Confidence-Scheduled Speculative Decoding with
 *     Semi-Autoregressive Generation" (§4.1, §4.2.1, §4.2.2);
 *   - edgeai1 knowledge base "DSpark 精读" (§2 proposal law, §4 confidence head and
 *     batch scheduler);
 *   - mkdocs.reaper.mx "3 · DSpark" (§3.1-§3.3).
 *
 * Conventions for every entry point
 *   - All array pointers are DEVICE pointers owned by the caller, C-contiguous,
 *     row-major.  "U[R,gamma,V]" means element U[(r*gamma + k-1)*V + v] for request r,
 *     draft position k (1-based) and vocabulary id v.  The logit and weight arrays (U,
 *     target, W1, W2, h) must start on a 16-byte boundary (they are read with 16-byte
 *     vector loads and the Tensor Memory Accelerator); others need natural alignment.
 *   - The library never allocates device memory: scratch comes from the caller's
 *     `workspace` (at least the size the matching *_workspace_size() returns, 256-byte
 *     aligned).  A workspace may be reused by later calls on the same stream; calls that
 *     run concurrently need separate workspaces.
 *   - Work is enqueued on `stream` and returns without synchronising the host.  No call
 *     reads device data on the host, so a whole round can be captured in a CUDA graph.
 *   - Arguments are validated on the host before anything is enqueued.  On a non-OK
 *     status nothing was launched; dspark_last_error_message() (thread-local) says why.
 *   - Kernels never trap.  A bounded wait that gives up records DSPARK_TIMEOUT in the
 *     workspace's device status word; read it with dspark_workspace_status().
 *   - There is no CPU fallback: every step runs in this library's CUDA kernels.
 *
 * Random numbers: Philox4x32-10 (Salmon et al., SC'11) with key (lo32 seed, hi32 seed)
 * and counter (lo32 req_id[r], lo32 round, stream<<24 | position, v/4); vocabulary
 * element v takes output word v%4; uniform u = ((word>>8) + 0.5) * 2^-24 in (0,1).
 * Streams: 0 draft Gumbel at position k, 1 acceptance uniform at position j (word 0
 * of chunk 0), 2 correction Gumbel (residual or bonus) at position n_acc+1.  The same
 * (seed, req_id, round) always reproduces the same round, whatever the batch layout.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int dspark_status;

#define DSPARK_OK 0
#define DSPARK_INVALID_ARG 1          /* null pointer, negative size, bad enum, T <= 0 */
#define DSPARK_UNSUPPORTED_SHAPE 2    /* size outside the limits stated per call */
#define DSPARK_WORKSPACE_TOO_SMALL 3  /* ws_bytes below *_workspace_size() */
#define DSPARK_CUDA_ERROR 4           /* a CUDA runtime call or launch failed */
#define DSPARK_TIMEOUT 5              /* a device wait gave up (reported via the status word) */

#define DSPARK_F32 0
#define DSPARK_BF16 1

#define DSPARK_EARLY_STOP 0
#define DSPARK_FULL_SEARCH 1
#define DSPARK_CAPACITY_K 2
#define DSPARK_FIXED 3

/* Human-readable name of a status code (static storage). */
DSPARK_API const char* dspark_status_string(int status);

/* Detail of the last non-OK status returned on the calling host thread. */
DSPARK_API const char* dspark_last_error_message(void);

/* Copies the device status word kept at the start of `workspace` (written by kernels
 * whose bounded waits gave up) into *status, synchronising `stream`.  0 = OK,
 * DSPARK_TIMEOUT otherwise.  Resets the word to 0 when reset != 0. */
DSPARK_API dspark_status dspark_workspace_status(void* workspace, int reset, int* status, void* stream);

/* Measurement hook (not part of the method).  While set, dspark_markov_draft records
 * events[2(k-1)] just before and events[2(k-1)+1] just after the launch of draft
 * position k's vocabulary-streaming step kernel, on the call's stream, for
 * k = 1..min(gamma, n_events/2).  (On the CUDA-core path a vocabulary of at most 4096
 * ids runs every position in one launch; events[0] and events[1] then bracket that
 * launch.)  `events` holds cudaEvent_t handles owned by the caller; NULL or n_events = 0
 * turns recording off.  The setting is per host thread.
 * While the stream is being captured into a CUDA graph, the events become external
 * event-record nodes of the graph, so every replay records them. */
DSPARK_API void dspark_set_profile_events(void* const* events, int n_events);

/* Measurement hook (not part of the method), like dspark_set_profile_events for the
 * verification calls (dspark_verify, dspark_verify_ragged, dspark_verify_static,
 * dspark_verify_overlap): events[0] / events[1] are recorded just before / after the
 * target-row statistics pass, events[2] / events[3] just before / after the correction
 * pass (the residual and bonus draws).  n_events < 4 or NULL turns recording off.  The
 * setting is per host thread. */
DSPARK_API void dspark_set_verify_profile_events(void* const* events, int n_events);

/* ------------------------------------------------------------------------------------
 * Stage 1: Markov-head draft loop with the confidence head.
 *
 * Defines (numb3r33 blog "Markov sequential head"; DSpark 精读 §2; vllmbangkok §4.1):
 *   for k = 1..gamma, with x_0 = x0[r]:
 *     z_v     = (U[r,k,v] + sum_i W1[x_{k-1},i] * W2[i,v]) / temperature
 *     x_k     = argmax_v z_v + g_v, g_v = -ln(-ln u_v) from stream 0 at position k
 *               (a Gumbel-max draw of p_k = softmax(z))
 *     lse_k   = ln sum_v exp z_v ;  logq_k = z_{x_k} - lse_k
 *   and the confidence head (DSpark 精读 §4: linear + sigmoid on [h_k ; W1[x_{k-1}]];
 *   numb3r33 blog "Sequential temperature scaling": one temperature per position):
 *     c_k = sigmoid(conf_logit_scale * (w_h . h[r,k,:] + w_e . W1[x_{k-1},:] + conf_b)
 *                   / conf_temp[k-1])
 *
 * Arguments
 *   R, gamma, V, rank, d  sizes: requests, draft length, vocabulary, low-rank factor
 *                         rank, backbone hidden size.
 *   dtype_u   DSPARK_F32 or DSPARK_BF16 for U.
 *   dtype_w   dtype of W1 and W2.  DSPARK_BF16 runs the bias contraction on the
 *             tcgen05 tensor cores (bf16 x bf16 -> fp32); DSPARK_F32 on CUDA cores (fp32).
 *   dtype_h   dtype of h.
 *   U         [R,gamma,V] backbone base logits.
 *   W1        [V,rank] first low-rank factor (row x is the token's embedding).
 *   W2        [rank,V] second low-rank factor.
 *   h         [R,gamma,d] backbone hidden states.
 *   conf_w    [d+rank] fp32 confidence weights: w_h (d entries) then w_e (rank entries).
 *   conf_b, conf_logit_scale   scalar bias and raw-logit scale of the confidence head.
 *   conf_temp [gamma] fp32 per-position temperatures (> 0).
 *   temperature  sampling temperature T > 0.
 *   x0        [R] int32 anchor tokens in [0,V).
 *   req_id    [R] int64 request keys of the random stream.
 *   seed, round  random-stream key and round index.
 * Outputs ([R,gamma] each): x_out int32 tokens; logq_out, lse_out, conf_out fp32.
 * Limits: 1 <= R, 1 <= gamma <= 64, 1 <= V, rank >= 1, d >= 0.  The bf16 tensor-core
 *   path needs rank % 64 == 0 and rank <= 256 and V % 8 == 0; other bf16 shapes run
 *   on CUDA cores.
 * ---------------------------------------------------------------------------------- */
DSPARK_API size_t dspark_markov_draft_workspace_size(int R, int gamma, int V, int rank, int d, int dtype_w);

DSPARK_API dspark_status dspark_markov_draft(
    int R, int gamma, int V, int rank, int d, int dtype_u, int dtype_w, int dtype_h,
    const void* U, const void* W1, const void* W2, const void* h, const float* conf_w,
    float conf_b, float conf_logit_scale, const float* conf_temp, float temperature,
    const int32_t* x0, const int64_t* req_id, uint64_t seed, uint64_t round,
    int32_t* x_out, float* logq_out, float* lse_out, float* conf_out,
    void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Stage 2: confidence scheduler.
 *
 * Defines (DSpark 精读 §4; mkdocs.reaper.mx §3.3; numb3r33 blog "Scheduler objective",
 * "Greedy prefix allocation", "Async scheduler in practice"; vllmbangkok §4.2.2):
 *   a[r,j] = prod_{i<=j} conf[r,i]   (binary64, multiplied left to right)
 *   candidates (r,j) sorted by a desc, then j asc, then r asc; admitting the first n
 *   gives B(n) = R + n verify tokens and tau(n) = R + sum of the first n a's;
 *   Theta(n) = tau(n) * sps[B(n)].
 *   mode DSPARK_EARLY_STOP  n* = first n with Theta(n+1) <= Theta(n) (else R*gamma)
 *        DSPARK_FULL_SEARCH n* = argmax_n Theta(n), smallest n on ties
 *        DSPARK_CAPACITY_K  K = the full-search n* computed on conf_hist (the stale
 *                           confidences); n* = min(K, R*gamma) on the current order
 *        DSPARK_FIXED       ell_r = min(fixed_len, gamma) for every r
 *   ell_out[r] = number of admitted candidates of request r (always a prefix 1..ell_r),
 *   B_out = R + n*, tau_out = tau(n*).
 * Arguments
 *   conf      [R,gamma] fp32 conditional confidences (stage 1's conf_out).
 *   sps       [sps_len] fp64 profiled target steps/s indexed by B; sps_len >= R*(gamma+1)+1.
 *   conf_hist [R,gamma] fp32, required for DSPARK_CAPACITY_K, ignored otherwise.
 *   fixed_len used by DSPARK_FIXED only (clamped to [0,gamma]).
 * Outputs: ell_out [R] int32, B_out [1] int32, tau_out [1] fp64.
 * Limits: 1 <= R, 1 <= gamma <= 64, R*gamma <= 8192.
 * ---------------------------------------------------------------------------------- */
DSPARK_API size_t dspark_schedule_workspace_size(int R, int gamma);

DSPARK_API dspark_status dspark_schedule(
    int R, int gamma, const float* conf, const double* sps, int sps_len, int mode,
    const float* conf_hist, int fixed_len, int32_t* ell_out, int32_t* B_out, double* tau_out,
    void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Stage 2 with a fixed confidence cutoff (vllmbangkok "Verify smarter, not longer: the
 * role of confidence scheduling": drafts whose confidence is below a fixed cutoff are not
 * verified).  Verification needs a prefix, so request r keeps its leading drafts with
 * c >= threshold:
 *   ell[r] = max { j : c[r,i] >= threshold for every i <= j }   (0 if c[r,1] < threshold)
 *   B      = R + sum_r ell[r];   tau = R + sum_r sum_{j <= ell[r]} prod_{i <= j} c[r,i]
 * (products in binary64, left to right).  A NaN confidence ends the prefix.
 * Arguments as dspark_schedule; threshold is a finite double; the workspace is the one
 * dspark_schedule_workspace_size() sizes.  Limits: 1 <= R, 1 <= gamma <= 64.
 * ---------------------------------------------------------------------------------- */
DSPARK_API dspark_status dspark_schedule_threshold(int R, int gamma, const float* conf, double threshold,
                                                   int32_t* ell_out, int32_t* B_out, double* tau_out,
                                                   void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Stage 3: exact speculative-sampling verification.
 *
 * Defines (numb3r33 blog "One-token exactness", "Why only the longest accepted prefix
 * survives", "Prefix survival and accepted length"):
 *   for j = 1..ell[r]: p = softmax(target[r,j,:]/T) (row j-1 of target, 0-based);
 *     accept x_j iff u_j < p(x_j) / q_j(x_j), q_j(x_j) = exp(logq[r,j]), u_j from
 *     stream 1 at position j; stop at the first rejection.  n_acc = accepted count.
 *   if n_acc < ell[r]: j* = n_acc + 1; q = exp(z - lse_q[r,j*]) with z the draft logits
 *     of position j* recomputed from U, W1[x_{j*-1}], W2 (x_0 = x0[r]);
 *     p = softmax(target row j*-1 / T); y = argmax over {v : p_v > q_v} of
 *     ln(p_v - q_v) + g_v (stream 2, position j*): a draw from (p - q)+ normalised.
 *     If no p_v > q_v (possible only through rounding), y = argmax_v ln p_v + g_v.
 *   else: bonus y = argmax_v target[r,ell,v]/T + g_v (stream 2, position ell+1).
 *   tokens_out[r,:] = x_1..x_{n_acc}, y, then -1 padding; n_out[r] = n_acc + 1.
 * Arguments
 *   target    [R,gamma+1,V] target logits (dtype_t).
 *   U, W1, W2 as in stage 1 (for the residual recomputation).
 *   x0 [R], x [R,gamma] int32; logq, lse_q [R,gamma] fp32 (stage 1 outputs);
 *   ell [R] int32 in [0,gamma] (stage 2 output).
 * Outputs: n_acc_out [R] int32, tokens_out [R,gamma+1] int32, n_out [R] int32.
 * Limits: as stage 1, plus target rows of V elements.
 * ---------------------------------------------------------------------------------- */
DSPARK_API size_t dspark_verify_workspace_size(int R, int gamma, int V, int rank, int dtype_w);

DSPARK_API dspark_status dspark_verify(
    int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
    const void* target, const void* U, const void* W1, const void* W2,
    const int32_t* x0, const int32_t* x, const float* logq, const float* lse_q,
    const int32_t* ell, float temperature, const int64_t* req_id, uint64_t seed, uint64_t round,
    int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out,
    void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Stage 3 on a flattened target batch (numb3r33 blog "Variable-length verification
 * without wasting kernels": the verified rows of all requests are packed back to back
 * and metadata, not padding, keeps each request's rows apart).
 *
 * Same computation, results and limits as dspark_verify; only the target layout differs:
 *   target             [n_target_rows, V] logits; request r's verify rows t = 0..ell[r]
 *                      (row t scores draft t+1; row ell[r] gives the bonus token) are
 *                      rows target_row_offset[r] + t.  Rows may be in any order and
 *                      unused rows may exist; sum_r (ell[r] + 1) rows are read.
 *   n_target_rows      number of rows of `target` (>= 1).
 *   target_row_offset  [R] int32 device array, the first row of each request.
 * The workspace is the one dspark_verify_workspace_size() sizes.  A row index outside
 * [0, n_target_rows) is reported through the workspace status word (DSPARK_INVALID_ARG)
 * and row 0 is read instead.
 * ---------------------------------------------------------------------------------- */
DSPARK_API dspark_status dspark_verify_ragged(
    int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
    const void* target, int n_target_rows, const int32_t* target_row_offset,
    const void* U, const void* W1, const void* W2,
    const int32_t* x0, const int32_t* x, const float* logq, const float* lse_q,
    const int32_t* ell, float temperature, const int64_t* req_id, uint64_t seed, uint64_t round,
    int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out,
    void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Stage 3 for callers that cannot allocate device memory.  (The paper has no
 * counterpart: this is a deployment convenience of this library.)
 *
 * Same arguments, results and limits as dspark_verify, without `workspace`/`ws_bytes`:
 * the scratch is an 8 MiB array inside the library (one copy per GPU that loads the
 * library, held until the process exits).  Shapes whose dspark_verify_workspace_size()
 * exceeds 8 MiB are rejected with DSPARK_UNSUPPORTED_SHAPE.  Allocates nothing.
 *   - The first call on a device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.
 *   - All calls share the array: calls that may overlap on the GPU (other streams, other
 *     host threads on the same device) race and must be ordered by the caller.
 *   - The status block that must start at zero is cleared on `stream` at every call, so
 *     device-side input reports of earlier calls are not kept; read the last call's
 *     report with dspark_verify_static_status() before the next call.
 * ---------------------------------------------------------------------------------- */
DSPARK_API dspark_status dspark_verify_static(
    int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
    const void* target, const void* U, const void* W1, const void* W2,
    const int32_t* x0, const int32_t* x, const float* logq, const float* lse_q,
    const int32_t* ell, float temperature, const int64_t* req_id, uint64_t seed, uint64_t round,
    int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out, void* stream);

/* Device status word of dspark_verify_static's scratch on the current device (the paper
 * has no counterpart either).  Copies it into *status after synchronising `stream`:
 * 0 = OK, DSPARK_INVALID_ARG = the last call met a token id, verify length or target row
 * out of range on the device (it clamped the value and carried on),
 * DSPARK_TIMEOUT = a bounded device wait gave up.  reset != 0 clears the word afterwards.
 * Allocates nothing.  Not for use while `stream` is being captured (it synchronises). */
DSPARK_API dspark_status dspark_verify_static_status(int reset, int* status, void* stream);

/* ------------------------------------------------------------------------------------
 * Stage 1 with the recurrent (RNN) draft head.
 *
 * Defines (numb3r33 blog "DSpark: confidence-scheduled speculative decoding", section "RNN
 * sequential head": s_k = f(s_{k-1}, E(x_{k-1}), h_k), z_k = U_k + W_o s_k; DSpark 精读
 * §2: f is a gated update of the concatenated state, previous-token embedding and hidden
 * state).  The gate is the update-gate cell, for k = 1..gamma (x_0 = x0[r], s_0 = 0):
 *   a   = [s_{k-1}; E[x_{k-1},:]] Wse + h[r,k,:] Wh + bgc          (2*ns values)
 *   s_k = (1 - sigmoid(a[0:ns])) * s_{k-1} + sigmoid(a[0:ns]) * tanh(a[ns:2ns])
 *   s_k is stored in dtype_w (bf16: rounded to nearest even) and used as stored;
 *   z = (U[r,k,:] + s_k Wo) / T;  x_k, lse_k, logq_k as in dspark_markov_draft
 *   (Gumbel-max with stream 0 at position k);
 *   c_k = sigmoid(kappa * (conf_w[0:d] . h[r,k,:] + conf_w[d:d+ns] . s_k + conf_b) / T_k).
 * Arguments
 *   ns        state width, a multiple of 32, <= 256 (tensor-core vocabulary pass for bf16
 *             weights with ns a multiple of 64 and V a multiple of 8, V >= 128).
 *   ne        embedding width (0..2048); d hidden width (0 allowed).
 *   U [R,gamma,V] (dtype_u); E [V,ne], Wse [ns+ne, 2*ns] (gate columns first),
 *   Wh [d, 2*ns], Wo [ns,V] (dtype_w); bgc [2*ns] fp32; h [R,gamma,d] (dtype_h).
 *   conf_w [d+ns] fp32; conf_b, conf_logit_scale (kappa), conf_temp [gamma]; T > 0.
 *   x0 [R], req_id [R], seed, round: as in dspark_markov_draft.
 * Outputs: x_out, logq_out, lse_out, conf_out [R,gamma] as in dspark_markov_draft;
 *   state_out [R,gamma,ns] (dtype_w): the stored states s_1..s_gamma, which the
 *   verification of the round needs (dspark_verify_rnn).
 * Workspace: dspark_rnn_draft_workspace_size().  U, Wo and h 16-byte aligned.
 * ---------------------------------------------------------------------------------- */
DSPARK_API size_t dspark_rnn_draft_workspace_size(int R, int gamma, int V, int ns, int d, int dtype_w);

DSPARK_API dspark_status dspark_rnn_draft(
    int R, int gamma, int V, int ns, int ne, int d, int dtype_u, int dtype_w, int dtype_h,
    const void* U, const void* E, const void* Wse, const void* Wh, const float* bgc, const void* Wo,
    const void* h, const float* conf_w, float conf_b, float conf_logit_scale, const float* conf_temp,
    float temperature, const int32_t* x0, const int64_t* req_id, uint64_t seed, uint64_t round,
    int32_t* x_out, float* logq_out, float* lse_out, float* conf_out, void* state_out,
    void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Stage 3 for a block drafted by the recurrent head.
 *
 * dspark_verify with the residual's bias row taken from the drafted state:
 * z = (U[r,j*,:] + state[r,j*,:] Wo) / T instead of W1[x_{j*-1}] W2.  state [R,gamma,ns]
 * (dtype_w) is dspark_rnn_draft's state_out; every other argument, result and limit is
 * dspark_verify's, with rank = ns.  Workspace: dspark_verify_workspace_size(R, gamma, V,
 * ns, dtype_w).
 * ---------------------------------------------------------------------------------- */
DSPARK_API dspark_status dspark_verify_rnn(
    int R, int gamma, int V, int ns, int dtype_t, int dtype_u, int dtype_w,
    const void* target, const void* U, const void* state, const void* Wo,
    const int32_t* x0, const int32_t* x, const float* logq, const float* lse_q,
    const int32_t* ell, float temperature, const int64_t* req_id, uint64_t seed, uint64_t round,
    int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out,
    void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Acceptance-overlap diagnostic of a drafted block.
 *
 * Defines (numb3r33 blog "DSpark: confidence-scheduled speculative decoding", sections
 * "Total variation label" and "Speculative sampling in one picture"): for every request
 * r and drafted position j = 1..n_r,
 *   c*[r,j] = sum_v min(q_j(v), p_j(v)) = 1 - ||q_j - p_j||_1 / 2,
 *   q_j = exp(z - lse_q[r,j]), z = (U[r,j,:] + W1[x_{j-1},:] W2) / T (x_0 = x0[r]),
 *   p_j = softmax(target row j-1 / T)  (0-based row of target[r]),
 * the probability that the draft token of position j is accepted given its prefix (the
 * expectation of min(1, p/q) under q), i.e. the label the confidence head c_j predicts.
 * n_r = ell[r] when ell is given (the verified positions), gamma when ell is NULL.
 * Arguments
 *   target [R,gamma+1,V] (dtype_t), U [R,gamma,V] (dtype_u), W1 [V,rank], W2 [rank,V]
 *     (dtype_w): as in stages 1 and 3; 16-byte aligned.
 *   x0 [R], x [R,gamma] int32: the drafted tokens (stage 1 output).
 *   lse_q [R,gamma] fp32: the draft log-normalisers (stage 1 output).
 *   ell [R] int32 in [0,gamma], or NULL.
 * Output: overlap_out [R,gamma] fp32; NaN at positions j > n_r.
 * Token ids or lengths outside their range are reported through the workspace status
 * word (DSPARK_INVALID_ARG) and clamped.  Workspace: the size
 * dspark_acceptance_overlap_workspace_size() returns (0 for unsupported sizes).
 * Limits: R*gamma <= 2^24, gamma <= 64.
 * ---------------------------------------------------------------------------------- */
DSPARK_API size_t dspark_acceptance_overlap_workspace_size(int R, int gamma, int V, int rank, int dtype_w);

DSPARK_API dspark_status dspark_acceptance_overlap(
    int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
    const void* target, const void* U, const void* W1, const void* W2,
    const int32_t* x0, const int32_t* x, const float* lse_q, const int32_t* ell,
    float temperature, float* overlap_out, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Stage 3 with the acceptance overlap fused in.
 *
 * dspark_verify (same arguments, results and limits), and in the same pass the
 * acceptance overlap of every verified position (numb3r33 blog "DSpark:
 * confidence-scheduled speculative decoding", section "Total variation label"):
 *   overlap_out [R,gamma] fp32, overlap_out[r,j-1] = sum_v min(q_j(v), p_j(v)) for
 *   j = 1..ell[r], NaN for j > ell[r]; q_j and p_j as in dspark_acceptance_overlap.
 * The target rows' log-normalisers come from the verification's own pass over them; the
 * overlap then takes one more bias contraction over the verified positions (which reads
 * their U and target logits again).  The results equal dspark_acceptance_overlap(..., ell,
 * ...) up to the order of fp32 sums.  Workspace: dspark_verify_overlap_workspace_size() (larger
 * than dspark_verify's; 0 for unsupported sizes).  Without the tensor-core path (fp32
 * weights, or rank / V outside its limits) R*gamma <= 262140.
 * ---------------------------------------------------------------------------------- */
DSPARK_API size_t dspark_verify_overlap_workspace_size(int R, int gamma, int V, int rank, int dtype_w);

DSPARK_API dspark_status dspark_verify_overlap(
    int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
    const void* target, const void* U, const void* W1, const void* W2,
    const int32_t* x0, const int32_t* x, const float* logq, const float* lse_q,
    const int32_t* ell, float temperature, const int64_t* req_id, uint64_t seed, uint64_t round,
    int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out, float* overlap_out,
    void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Sequential temperature scaling (STS) of the confidence head on held-out rounds.
 *
 * Defines (numb3r33 blog "DSpark: confidence-scheduled speculative decoding", section
 * "Sequential temperature scaling"; mkdocs.reaper.mx "3 · DSpark" §3.2): one temperature
 * per position, c_k = sigmoid(z_k / T_k), fitted left to right.  For k = 1..gamma, with
 * T_1..T_{k-1} frozen, T_k is the candidate T of `grid` with the smallest
 *   ECE_k(T) = sum_b | sum_{n in bin b} (p_n - o_n) | / N,
 *   p_n = prod_{i<k} sigmoid(z[n,i] / T_i) * sigmoid(z[n,k] / T),  o_n = 1[acc_len[n] >= k],
 * over M equal-width bins of [0,1] (bin of p: min(floor(p M), M-1)); the first candidate
 * wins ties.  ece_out[k] is that smallest ECE.
 * Arguments
 *   z        [N, gamma] fp32: confidence logits of held-out samples before the
 *            per-position temperature (kappa (w . [h; W1[x]] + b) of the confidence head).
 *   acc_len  [N] int32: accepted drafts of each sample when all gamma were verified.
 *   grid     [G] fp32 candidate temperatures (> 0; others are skipped and reported).
 *   M        calibration bins, 1..16.
 * Outputs: T_out [gamma], ece_out [gamma] fp32 (NaN if no candidate is usable).
 * Deterministic (every sum in a fixed order).  Workspace:
 * dspark_sts_fit_workspace_size().  Limits: gamma <= 64, G <= 65535, N*gamma < 2^31.
 * ---------------------------------------------------------------------------------- */
DSPARK_API size_t dspark_sts_fit_workspace_size(int N, int gamma, int G, int M);

DSPARK_API dspark_status dspark_sts_fit(
    int N, int gamma, const float* z, const int32_t* acc_len, const float* grid, int G, int M,
    float* T_out, float* ece_out, void* workspace, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
