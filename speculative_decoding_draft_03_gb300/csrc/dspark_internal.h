// dspark_internal.h — argument blocks, workspace layouts and launcher declarations
// shared by the library's translation units (host and device).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dspark {

struct Partial;
struct DeviceStatus;

constexpr int kSimtThreads = 256;
constexpr int kSimtGroups = 4;   // groups of 4 vocabulary ids per thread per chunk
constexpr int kSimtRB = 4;       // requests per CTA in the CUDA-core draft step

// Everything one draft position needs (passed by value to kernels).
struct DraftArgs {
  int R, gamma, V, rank, d;
  int dtype_u, dtype_w, dtype_h;
  const void* U;
  const void* W1;
  const void* W2;
  const void* h;
  const float* conf_w;
  float conf_b, conf_scale;
  const float* conf_temp;
  float inv_temp;
  const int32_t* x0;
  const int64_t* req_id;
  uint64_t seed, round;
  int32_t* x_out;
  float* logq_out;
  float* lse_out;
  float* conf_out;
  // workspace pieces
  DeviceStatus* status;
  float* s_h;        // [R*gamma]
  void* W1g;         // [Rpad, rank] gathered factor rows (dtype_w)
  Partial* partials; // [gamma, npart, R] (the CUDA-core path uses the first [npart, R])
  int* hint;         // [gamma, R] best Gumbel key published so far per position (ordered int)
  unsigned long long* win;  // [gamma, R] tensor-core path: (key code, ~id) maximum per position
  // recurrent head (rnn != 0; rank is the state width ns, W1 is unused): the factor row of
  // position k is the state s_k, written by the cell kernel into W1g and state_out
  int rnn;
  int ne;              // embedding width
  const void* E;       // [V, ne]
  const void* Wse;     // [ns+ne, 2ns]: gate columns, then candidate columns
  const void* Wh;      // [d, 2ns]
  const float* bgc;    // [2ns]
  void* state_out;     // [R, gamma, ns] (dtype_w)
  float* hpart;        // [nsplit, R*gamma, 2ns] split-K partial sums of h Wh
  int nsplit;
};

struct VerifyArgs {
  int R, gamma, V, rank;
  int dtype_t, dtype_u, dtype_w;
  const void* target;
  const int32_t* t_off;  // flattened target layout: request r's first row (nullptr: padded)
  int n_trows;           // rows of the flattened target
  const void* U;
  const void* W1;
  const void* W2;
  const int32_t* x0;
  const int32_t* x;
  const float* logq;
  const float* lse_q;
  const int32_t* ell;
  float inv_temp;
  const int64_t* req_id;
  uint64_t seed, round;
  PhiloxKeys keys;  // round keys of seed (filled by launch_verify for the row pass)
  int32_t* n_acc_out;
  int32_t* tokens_out;
  int32_t* n_out;
  // workspace pieces
  DeviceStatus* status;
  int* n_rows;        // [1] number of verify rows
  int* row_req;       // [R*(gamma+1)] request of compact row
  int* row_t;         // [R*(gamma+1)] target row index (0-based) of compact row
  int* row_base;      // [R] first compact row of request r
  int* row_order;     // [R*(gamma+1)] processing order: row ell_r of every request, then the others
  int* work_next;     // [1] next (row, chunk) item of verify_rows (a work queue)
  Partial* row_part;  // [R*(gamma+1), nchunk]
  int nchunk;         // vocabulary chunks per row
  int chunk;          // ids per chunk
  float* lse_t;       // [R] target log-normaliser of the residual row
  int* jstar;         // [R] correction position n_acc + 1: positive after a rejection, negative for a bonus draw
  void* W1g;          // [Rpad, rank] gathered factor rows of the residual positions
  const void* state;  // recurrent head: [R, gamma, rank] states, the factor rows (nullptr: W1[x_{j-1}])
  Partial* res_part;  // [npart, R] residual partials: key = ln rho + g
  Partial* res_part2; // [npart, R] fallback partials: key = ln p + g
  // fused acceptance overlap (nullptr: off): verify_accept writes the target log-normaliser
  // of every verified row and the factor row of every verified position
  float* ovl_lse;     // lse of target row j-1 for position j <= ell[r]
  void* ovl_W1g;      // W1[x_{j-1}] for position j <= ell[r]
  int ovl_compact;    // 1: both in the compact row order (row row_base[r] + j - 1, tensor-core
                      // pass); 0: at the flattened position r*gamma + j - 1 (NaN / zero beyond ell)
  // measurement hook (nullptr: off): cudaEvent_t handles recorded around the row-statistics
  // pass ([0] before, [1] after) and the correction pass ([2] before, [3] after)
  void* const* prof;
  // rejected requests in compact slots (tensor-core correction pass): verify_accept takes
  // slot = atomicAdd(n_rej, 1) for each request that rejected a draft, writes its factor
  // row at W1g row `slot` and rej_req[slot] = r; the correction pass runs over the slots
  int* n_rej;         // [1]
  int* rej_req;       // [R]
  int* res_hint;      // [R] per slot: the best residual key published so far (order-preserving code)
  int res_compact;    // 1: compact slots (tensor cores); 0: W1g at the request index (CUDA cores)
  int res_grid;       // CTAs of the compact correction pass (its partial count follows from *n_rej)
  // compact slots whose residual had no positive p - q (only rounding can cause it): drawn
  // from p by the fallback pass
  int* n_fb;          // [1]
  int* fb_req;        // [R]
};

// Acceptance-overlap diagnostic: c*[r, j-1] = sum_v min(q_j(v), p_j(v)) for the drafted
// positions j <= n_r of every request (n_r = ell[r], or gamma without ell).  Row i of
// the flattened [R*gamma] positions is request i / gamma at position i % gamma + 1.
struct OverlapArgs {
  int R, gamma, V, rank;
  int dtype_t, dtype_u, dtype_w;
  const void* target;   // [R, gamma+1, V]
  const void* U;        // [R, gamma, V]
  const void* W1;
  const void* W2;
  const int32_t* x0;
  const int32_t* x;
  const float* lse_q;   // [R, gamma] draft log-normalisers
  const int32_t* ell;   // [R] or nullptr
  float inv_temp;
  float* out;           // [R, gamma]
  // workspace pieces
  DeviceStatus* status;
  void* W1g;            // [round_up_rows(R*gamma), rank] factor rows W1[x_{j-1}] (zero where unused)
  float* lse_t;         // [R*gamma] target log-normaliser of row j-1 (/T)
  float2* lse_part;     // [R*gamma, nchunk] per-chunk (max, sum exp) of those rows
  int nchunk;
  float* part;          // [npart, R*gamma] partial sums of min(q, p)
  int npart;
  // tensor-core path with lengths: the bias pass runs over compact rows (request
  // row_req[q], target row row_t[q], *n_rows of them, at most rows_max): the verify plan's
  // rows when fused with verification, else the evaluated positions only
  // (overlap_plan_kernel); W1g and lse_t are in that row order and part is [grid, rows_max]
  int* row_req;   // nullptr: the flattened R*gamma positions
  int* row_t;
  int* row_base;  // [R] first compact row of request r
  int* n_rows;
  int rows_max;
};

// Sequential temperature scaling on held-out data (N samples, gamma positions, G grid
// candidates, M <= kStsMaxBins calibration bins).
constexpr int kStsMaxBins = 16;
struct StsArgs {
  int N, gamma, G, M;
  const float* z;          // [N, gamma] confidence logits
  const int32_t* acc_len;  // [N]
  const float* grid;       // [G]
  float* T_out;            // [gamma]
  float* ece_out;          // [gamma]
  // workspace pieces
  DeviceStatus* status;
  float* zt;               // [gamma, N]
  float* prefix;           // [N] prod_{i<k} sigmoid(z_i / T_i)
  float* part;             // [G, S, M] per-chunk bin sums of p - o
  double* ece_g;           // [G]
  int S;                   // sample chunks
};

// Launch with programmatic stream serialization (the kernel must call griddep_wait()
// before its first dependent memory access).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Workspace layout: a 256-byte status block, then 256-byte aligned pieces.
__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Sets the thread's dspark_last_error_message() and returns `code`.
int record_error(int code, const char* msg);

// Records a caller's timing event on `s` (an external event node while `s` is captured).
cudaError_t record_profile_event(void* ev, cudaStream_t s);

int simt_num_chunks(int V);
int tc_supported(int V, int rank, int dtype_w);
int tc_num_partials(int R);
int tc_block_rows(int R);  // rows per request block of a tensor-core launch over R rows
// the same on the device: 32, 64 or 128 rows
__host__ __device__ inline int tc_rows_per_block(int R) { return R <= 32 ? 32 : (R <= 64 ? 64 : 128); }
// The compact correction pass takes at most 64 slots per block: every thread then holds
// two 8-id runs per tile instead of four, so a block's tile time halves, and the pass's
// CTAs split more evenly between the blocks that the device-side slot count needs (with
// 128-slot blocks, 129 rejecting requests already doubled every CTA's tile count).
__host__ __device__ inline int tc_residual_rows_per_block(int R) {
  return tc_rows_per_block(R) < 64 ? tc_rows_per_block(R) : 64;
}
int tc_grid_ctas(int R);   // CTAs of the compact overlap pass over at most R rows
int tc_residual_grid(int R);  // CTAs of the compact correction pass for R requests
// the compact overlap pass is used only when its request blocks fit on the SMs (then it
// launches one CTA per SM and its partials take SMs x R floats)
int tc_compact_ok(int R);
int draft_num_partials(int R, int V, int rank, int dtype_w);
int round_up_rows(int R);

// reset_bounds: also empty every position's published bound and winner (tensor-core path)
cudaError_t launch_conf_hdot(const DraftArgs& a, bool reset_bounds, cudaStream_t s);
cudaError_t launch_draft_prepare(const DraftArgs& a, int k, cudaStream_t s);
cudaError_t launch_draft_step_simt(const DraftArgs& a, int k, cudaStream_t s);
cudaError_t launch_draft_combine(const DraftArgs& a, int k, int npart, cudaStream_t s);
int simt_whole_round(int V);  // the CUDA-core draft fits one vocabulary chunk: one launch per round
cudaError_t launch_draft_round_simt(const DraftArgs& a, cudaStream_t s);
cudaError_t launch_draft_step_tc(const DraftArgs& a, int k, cudaStream_t s);
cudaError_t launch_rnn_step_tc(const DraftArgs& a, int k, cudaStream_t s);
// Recurrent head: h Wh for every position (before the loop), the cell of position k
// (after position k-1's draw), and the confidences from the states (after the loop).
int rnn_hproj_on_tc(int d, int ns, int dtype_w, int dtype_h);
int rnn_num_splits(int R, int gamma, int d, int ns, int dtype_w, int dtype_h);
cudaError_t launch_rnn_hproj(const DraftArgs& a, cudaStream_t s);
cudaError_t launch_rnn_hproj_tc(const DraftArgs& a, cudaStream_t s);
cudaError_t launch_rnn_cell(const DraftArgs& a, int k, bool tc, cudaStream_t s);
cudaError_t launch_rnn_conf(const DraftArgs& a, cudaStream_t s);
// After the last tensor-core position: every position's partial records -> x, lse, logq.
cudaError_t launch_draft_finalize(const DraftArgs& a, int npart, cudaStream_t s);

cudaError_t launch_schedule_threshold(int R, int gamma, const float* conf, double threshold, int32_t* ell_out,
                                      int32_t* B_out, double* tau_out, cudaStream_t s);
cudaError_t launch_schedule(int R, int gamma, const float* conf, const double* sps, int mode,
                            const float* conf_hist, int fixed_len, int32_t* ell_out, int32_t* B_out,
                            double* tau_out, DeviceStatus* status, cudaStream_t s);
size_t schedule_smem_bytes(int R, int gamma);

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s);
cudaError_t launch_residual_tc(const VerifyArgs& a, cudaStream_t s);
size_t residual_partial_entries(int R, int V, int rank, int dtype_w);

cudaError_t launch_overlap(const OverlapArgs& a, cudaStream_t s);
// the bias pass and the combine only, on lse_t and W1g already in place
cudaError_t launch_overlap_pass(const OverlapArgs& a, cudaStream_t s);
cudaError_t launch_overlap_tc(const OverlapArgs& a, cudaStream_t s);
int overlap_num_partials(int R, int gamma, int V, int rank, int dtype_w);
int overlap_num_chunks(int V);

int sts_num_chunks(int N);
cudaError_t launch_sts_fit(const StsArgs& a, cudaStream_t s);

}  // namespace dspark
