// dspark_api.cu — the C ABI: argument validation, workspace layout, stream-ordered
// launches.  No device memory is allocated here; no call synchronises the host except
// dspark_workspace_status().
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace {

thread_local char g_msg[512] = "";
thread_local void* const* g_prof_events = nullptr;
thread_local int g_prof_n = 0;
thread_local void* const* g_vprof_events = nullptr;

dspark_status fail(dspark_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

dspark_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DSPARK_CUDA_ERROR, "%s: %s", what, cudaGetErrorString(e));
}

size_t elem_size(int dtype) { return dtype == DSPARK_BF16 ? 2 : 4; }
bool valid_dtype(int d) { return d == DSPARK_F32 || d == DSPARK_BF16; }

constexpr int kMaxGamma = 64;
constexpr int kVerifyChunk = 8192;

struct DraftLayout {
  size_t s_h, W1g, partials, hint, win, total;
  int npart;
};

DraftLayout draft_layout(int R, int gamma, int V, int rank, int dtype_w) {
  using namespace dspark;
  DraftLayout L;
  size_t off = 256;  // status block
  L.s_h = off;
  off += align256(sizeof(float) * (size_t)R * gamma);
  L.W1g = off;
  off += align256(elem_size(dtype_w) * (size_t)round_up_rows(R) * rank);
  L.npart = draft_num_partials(R, V, rank, dtype_w);
  L.partials = off;
  off += align256((size_t)32 * L.npart * R * gamma);  // one set per draft position
  L.hint = off;
  off += align256(sizeof(int) * (size_t)R * gamma);
  L.win = off;
  off += align256(sizeof(unsigned long long) * (size_t)R * gamma);
  L.total = off;
  return L;
}

struct RnnLayout {
  DraftLayout draft;
  size_t hpart, total;
  int nsplit;
};

// The partial sums are sized for the larger of the two projection splits (the hidden
// state's type decides which projection runs).
RnnLayout rnn_layout(int R, int gamma, int V, int ns, int d, int dtype_w) {
  RnnLayout L;
  L.draft = draft_layout(R, gamma, V, ns, dtype_w);
  L.nsplit = std::max(dspark::rnn_num_splits(R, gamma, d, ns, dtype_w, DSPARK_BF16),
                      dspark::rnn_num_splits(R, gamma, d, ns, dtype_w, DSPARK_F32));
  L.hpart = L.draft.total;
  L.total = L.hpart + dspark::align256(sizeof(float) * (size_t)L.nsplit * R * gamma * 2 * ns);
  return L;
}

struct VerifyLayout {
  size_t counters, row_req, row_t, row_base, row_order, row_part, lse_t, jstar, rej_req, fb_req, res_hint, W1g,
      res_part, res_part2, total;
  int nchunk;
};

VerifyLayout verify_layout(int R, int gamma, int V, int rank, int dtype_w) {
  using namespace dspark;
  VerifyLayout L;
  const size_t rows = (size_t)R * (gamma + 1);
  L.nchunk = (V + kVerifyChunk - 1) / kVerifyChunk;
  const size_t res_entries = residual_partial_entries(R, V, rank, dtype_w);
  size_t off = 256;
  L.counters = off;
  off += 256;
  L.row_req = off;
  off += align256(4 * rows);
  L.row_t = off;
  off += align256(4 * rows);
  L.row_base = off;
  off += align256(4 * (size_t)R);
  L.row_order = off;
  off += align256(4 * rows);
  L.row_part = off;
  off += align256(32 * rows * L.nchunk);
  L.lse_t = off;
  off += align256(4 * (size_t)R);
  L.jstar = off;
  off += align256(4 * (size_t)R);
  L.rej_req = off;
  off += align256(4 * (size_t)R);
  L.fb_req = off;
  off += align256(4 * (size_t)R);
  L.res_hint = off;
  off += align256(4 * (size_t)R);
  L.W1g = off;
  off += align256(elem_size(dtype_w) * (size_t)round_up_rows(R) * rank);
  L.res_part = off;
  off += align256((size_t)32 * res_entries);
  L.res_part2 = off;
  off += align256((size_t)32 * res_entries);
  L.total = off;
  return L;
}

struct OverlapLayout {
  size_t W1g, lse_t, lse_part, part, row_req, row_t, row_base, n_rows, total;
  int npart, nchunk;
};

// Sized for either row order: the flattened positions, or the compact rows of the
// evaluated positions (tensor-core path with lengths: one partial per CTA of its grid).
OverlapLayout overlap_layout(int R, int gamma, int V, int rank, int dtype_w) {
  using namespace dspark;
  OverlapLayout L;
  const size_t rows = (size_t)R * gamma;
  L.npart = overlap_num_partials(R, gamma, V, rank, dtype_w);
  if (tc_supported(V, rank, dtype_w) && tc_compact_ok((int)rows) && tc_grid_ctas((int)rows) > L.npart)
    L.npart = tc_grid_ctas((int)rows);
  size_t off = 256;
  L.W1g = off;
  off += align256(elem_size(dtype_w) * (size_t)round_up_rows((int)rows) * rank);
  L.lse_t = off;
  off += align256(4 * rows);
  L.nchunk = overlap_num_chunks(V);
  L.lse_part = off;
  off += align256(8 * rows * (size_t)L.nchunk);
  L.part = off;
  off += align256(4 * rows * (size_t)L.npart);
  L.row_req = off;
  off += align256(4 * rows);
  L.row_t = off;
  off += align256(4 * rows);
  L.row_base = off;
  off += align256(4 * (size_t)R);
  L.n_rows = off;
  off += 256;
  L.total = off;
  return L;
}

#define CHECK_PTR(p)                                                              \
  do {                                                                            \
    if ((p) == nullptr) return fail(DSPARK_INVALID_ARG, "null pointer: %s", #p); \
  } while (0)

// logit and weight arrays are read with 16-byte vector loads and the TMA
#define CHECK_ALIGN16(p)                                                                     \
  do {                                                                                       \
    if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0)                                         \
      return fail(DSPARK_INVALID_ARG, "%s must start on a 16-byte boundary", #p);            \
  } while (0)

bool aligned256(const void* p) { return ((uintptr_t)p & 255u) == 0; }

}  // namespace

namespace dspark {

dspark_status record_error(dspark_status code, const char* msg) { return fail(code, "%s", msg); }

int round_up_rows(int R) { return ((R + 127) / 128) * 128; }

int draft_num_partials(int R, int V, int rank, int dtype_w) {
  const int simt = simt_num_chunks(V);
  if (tc_supported(V, rank, dtype_w)) {
    const int tc = tc_num_partials(R);
    return simt > tc ? simt : tc;
  }
  return simt;
}

}  // namespace dspark

extern "C" {

const char* dspark_status_string(int status) {
  switch (status) {
    case DSPARK_OK: return "DSPARK_OK";
    case DSPARK_INVALID_ARG: return "DSPARK_INVALID_ARG";
    case DSPARK_UNSUPPORTED_SHAPE: return "DSPARK_UNSUPPORTED_SHAPE";
    case DSPARK_WORKSPACE_TOO_SMALL: return "DSPARK_WORKSPACE_TOO_SMALL";
    case DSPARK_CUDA_ERROR: return "DSPARK_CUDA_ERROR";
    case DSPARK_TIMEOUT: return "DSPARK_TIMEOUT";
    default: return "DSPARK_UNKNOWN_STATUS";
  }
}

const char* dspark_last_error_message(void) { return g_msg; }

// A profiling event recorded while the stream is being captured must become an event
// record node of the graph (not only a capture-ordering marker), so that replays time it.
extern "C++" {
namespace dspark {
cudaError_t record_profile_event(void* ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags((cudaEvent_t)ev, s, cudaEventRecordExternal)
                                             : cudaEventRecord((cudaEvent_t)ev, s);
}
}  // namespace dspark
}
using dspark::record_profile_event;

void dspark_set_profile_events(void* const* events, int n_events) {
  g_prof_events = (events != nullptr && n_events > 0) ? events : nullptr;
  g_prof_n = g_prof_events ? n_events : 0;
}

void dspark_set_verify_profile_events(void* const* events, int n_events) {
  g_vprof_events = (events != nullptr && n_events >= 4) ? events : nullptr;
}

dspark_status dspark_workspace_status(void* workspace, int reset, int* status, void* stream) {
  CHECK_PTR(workspace);
  CHECK_PTR(status);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  dspark::DeviceStatus host;
  cudaError_t e = cudaMemcpyAsync(&host, workspace, sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  *status = host.code;
  if (reset) {
    e = cudaMemsetAsync(workspace, 0, sizeof host, s);
    if (e != cudaSuccess) return cuda_fail(e, "resetting the device status word");
  }
  return DSPARK_OK;
}

size_t dspark_markov_draft_workspace_size(int R, int gamma, int V, int rank, int d, int dtype_w) {
  (void)d;
  if (R < 1 || gamma < 1 || V < 1 || rank < 1) return 0;
  return draft_layout(R, gamma, V, rank, dtype_w).total;
}

dspark_status dspark_markov_draft(int R, int gamma, int V, int rank, int d, int dtype_u, int dtype_w, int dtype_h,
                                  const void* U, const void* W1, const void* W2, const void* h,
                                  const float* conf_w, float conf_b, float conf_logit_scale,
                                  const float* conf_temp, float temperature, const int32_t* x0,
                                  const int64_t* req_id, uint64_t seed, uint64_t round, int32_t* x_out,
                                  float* logq_out, float* lse_out, float* conf_out, void* workspace,
                                  size_t ws_bytes, void* stream) {
  if (R < 1 || gamma < 1 || V < 1 || rank < 1 || d < 0)
    return fail(DSPARK_INVALID_ARG, "sizes must be positive (R=%d gamma=%d V=%d rank=%d d=%d)", R, gamma, V, rank, d);
  if (gamma > kMaxGamma) return fail(DSPARK_UNSUPPORTED_SHAPE, "gamma=%d exceeds %d", gamma, kMaxGamma);
  if ((long long)V > (1ll << 30)) return fail(DSPARK_UNSUPPORTED_SHAPE, "V=%d too large", V);
  if (!valid_dtype(dtype_u) || !valid_dtype(dtype_w) || !valid_dtype(dtype_h))
    return fail(DSPARK_INVALID_ARG, "dtype codes must be DSPARK_F32 or DSPARK_BF16");
  if (!(temperature > 0.f) || !isfinite(temperature))
    return fail(DSPARK_INVALID_ARG, "temperature must be finite and > 0");
  CHECK_PTR(U);
  CHECK_PTR(W1);
  CHECK_PTR(W2);
  if (d > 0) CHECK_PTR(h);
  CHECK_PTR(conf_w);
  CHECK_PTR(conf_temp);
  CHECK_PTR(x0);
  CHECK_PTR(req_id);
  CHECK_PTR(x_out);
  CHECK_PTR(logq_out);
  CHECK_PTR(lse_out);
  CHECK_PTR(conf_out);
  CHECK_PTR(workspace);
  CHECK_ALIGN16(U);
  CHECK_ALIGN16(W1);
  CHECK_ALIGN16(W2);
  if (d > 0) CHECK_ALIGN16(h);
  if (!aligned256(workspace)) return fail(DSPARK_INVALID_ARG, "workspace must be 256-byte aligned");
  const DraftLayout L = draft_layout(R, gamma, V, rank, dtype_w);
  if (ws_bytes < L.total)
    return fail(DSPARK_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, L.total);

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  dspark::DraftArgs a = {};
  a.R = R; a.gamma = gamma; a.V = V; a.rank = rank; a.d = d;
  a.dtype_u = dtype_u; a.dtype_w = dtype_w; a.dtype_h = dtype_h;
  a.U = U; a.W1 = W1; a.W2 = W2; a.h = h;
  a.conf_w = conf_w; a.conf_b = conf_b; a.conf_scale = conf_logit_scale; a.conf_temp = conf_temp;
  a.inv_temp = 1.0f / temperature;
  a.x0 = x0; a.req_id = req_id; a.seed = seed; a.round = round;
  a.x_out = x_out; a.logq_out = logq_out; a.lse_out = lse_out; a.conf_out = conf_out;
  a.status = reinterpret_cast<dspark::DeviceStatus*>(ws);
  a.s_h = reinterpret_cast<float*>(ws + L.s_h);
  a.W1g = ws + L.W1g;
  a.partials = reinterpret_cast<dspark::Partial*>(ws + L.partials);
  a.hint = reinterpret_cast<int*>(ws + L.hint);
  a.win = reinterpret_cast<unsigned long long*>(ws + L.win);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  const bool tc = dspark::tc_supported(V, rank, dtype_w) != 0;
  // Tensor-core path: the step of position 1 gathers its own factor rows (from x0) and
  // writes c_1; conf_hdot empties the bounds and winners.  Otherwise (CUDA-core path, or
  // no hidden state) draft_prepare gathers position 1's factor rows, writes c_1 and
  // empties them.
  const bool prepare = !tc || d == 0;
  if (d > 0) {
    if ((e = dspark::launch_conf_hdot(a, !prepare, s)) != cudaSuccess) return cuda_fail(e, "conf_hdot");
  } else {
    if ((e = cudaMemsetAsync(a.s_h, 0, sizeof(float) * (size_t)R * gamma, s)) != cudaSuccess)
      return cuda_fail(e, "s_h clear");
  }
  if (!tc && dspark::simt_whole_round(V)) {
    // one vocabulary chunk: the whole draft loop in one launch (the profiling events, if
    // set, bracket that launch)
    const bool prof = g_prof_n >= 2;
    if (prof && (e = record_profile_event(g_prof_events[0], s)) != cudaSuccess) return cuda_fail(e, "profile event");
    if ((e = dspark::launch_draft_round_simt(a, s)) != cudaSuccess) return cuda_fail(e, "draft_round_simt");
    if (prof && (e = record_profile_event(g_prof_events[1], s)) != cudaSuccess) return cuda_fail(e, "profile event");
    return DSPARK_OK;
  }
  if (prepare && (e = dspark::launch_draft_prepare(a, 1, s)) != cudaSuccess) return cuda_fail(e, "draft_prepare");
  for (int k = 1; k <= gamma; ++k) {
    int npart;
    const bool prof = 2 * k <= g_prof_n;
    if (prof && (e = record_profile_event(g_prof_events[2 * (k - 1)], s)) != cudaSuccess)
      return cuda_fail(e, "profile event");
    if (tc) {
      if ((e = dspark::launch_draft_step_tc(a, k, s)) != cudaSuccess) return cuda_fail(e, "draft_step_tc");
      npart = dspark::tc_num_partials(R);
    } else {
      if ((e = dspark::launch_draft_step_simt(a, k, s)) != cudaSuccess) return cuda_fail(e, "draft_step_simt");
      npart = dspark::simt_num_chunks(V);
    }
    if (prof && (e = record_profile_event(g_prof_events[2 * (k - 1) + 1], s)) != cudaSuccess)
      return cuda_fail(e, "profile event");
    // Tensor-core path: each step publishes its per-request winner (one 64-bit maximum),
    // from which the next step gathers its own factor rows, so the partial records are
    // merged once, after the last position.  CUDA-core path: a merge kernel per position.
    if (!tc && (e = dspark::launch_draft_combine(a, k, npart, s)) != cudaSuccess)
      return cuda_fail(e, "draft_combine");
  }
  if (tc && (e = dspark::launch_draft_finalize(a, dspark::tc_num_partials(R), s)) != cudaSuccess)
    return cuda_fail(e, "draft_finalize");
  return DSPARK_OK;
}

size_t dspark_schedule_workspace_size(int R, int gamma) {
  (void)R;
  (void)gamma;
  return 256;
}

dspark_status dspark_schedule(int R, int gamma, const float* conf, const double* sps, int sps_len, int mode,
                              const float* conf_hist, int fixed_len, int32_t* ell_out, int32_t* B_out,
                              double* tau_out, void* workspace, size_t ws_bytes, void* stream) {
  if (R < 1 || gamma < 1) return fail(DSPARK_INVALID_ARG, "sizes must be positive (R=%d gamma=%d)", R, gamma);
  if (gamma > kMaxGamma) return fail(DSPARK_UNSUPPORTED_SHAPE, "gamma=%d exceeds %d", gamma, kMaxGamma);
  if ((long long)R * gamma > 8192)
    return fail(DSPARK_UNSUPPORTED_SHAPE, "R*gamma=%lld exceeds 8192 candidates", (long long)R * gamma);
  if (mode < DSPARK_EARLY_STOP || mode > DSPARK_FIXED) return fail(DSPARK_INVALID_ARG, "unknown mode %d", mode);
  CHECK_PTR(conf);
  CHECK_PTR(ell_out);
  CHECK_PTR(B_out);
  CHECK_PTR(tau_out);
  CHECK_PTR(workspace);
  if (mode != DSPARK_FIXED) CHECK_PTR(sps);
  if (mode == DSPARK_CAPACITY_K) CHECK_PTR(conf_hist);
  if (mode != DSPARK_FIXED && (long long)sps_len < (long long)R * (gamma + 1) + 1)
    return fail(DSPARK_INVALID_ARG, "sps_len=%d below R*(gamma+1)+1=%d", sps_len, R * (gamma + 1) + 1);
  if (!aligned256(workspace)) return fail(DSPARK_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < dspark_schedule_workspace_size(R, gamma))
    return fail(DSPARK_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes,
                dspark_schedule_workspace_size(R, gamma));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = dspark::launch_schedule(R, gamma, conf, sps, mode, conf_hist, fixed_len, ell_out, B_out, tau_out,
                                          reinterpret_cast<dspark::DeviceStatus*>(workspace), s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule");
  return DSPARK_OK;
}

dspark_status dspark_schedule_threshold(int R, int gamma, const float* conf, double threshold, int32_t* ell_out,
                                        int32_t* B_out, double* tau_out, void* workspace, size_t ws_bytes,
                                        void* stream) {
  if (R < 1 || gamma < 1) return fail(DSPARK_INVALID_ARG, "sizes must be positive (R=%d gamma=%d)", R, gamma);
  if (gamma > kMaxGamma) return fail(DSPARK_UNSUPPORTED_SHAPE, "gamma=%d exceeds %d", gamma, kMaxGamma);
  if ((long long)R * gamma > (1ll << 24)) return fail(DSPARK_UNSUPPORTED_SHAPE, "R*gamma too large");
  if (!isfinite(threshold)) return fail(DSPARK_INVALID_ARG, "threshold must be finite");
  CHECK_PTR(conf);
  CHECK_PTR(ell_out);
  CHECK_PTR(B_out);
  CHECK_PTR(tau_out);
  CHECK_PTR(workspace);
  if (!aligned256(workspace)) return fail(DSPARK_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < dspark_schedule_workspace_size(R, gamma))
    return fail(DSPARK_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes,
                dspark_schedule_workspace_size(R, gamma));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = dspark::launch_schedule_threshold(R, gamma, conf, threshold, ell_out, B_out, tau_out, s);
  if (e != cudaSuccess) return cuda_fail(e, "schedule_threshold");
  return DSPARK_OK;
}

// dspark_verify_overlap: the verify workspace followed by the overlap pass's pieces.  The
// tensor-core pass runs over the verify plan's compact rows (at most R*(gamma+1), one
// partial per CTA of its grid); the CUDA-core pass over the R*gamma flattened positions.
struct VerifyOverlapLayout {
  VerifyLayout v;
  size_t W1g, lse, part, total;
  int npart, rows;
  bool compact;
};

VerifyOverlapLayout verify_overlap_layout(int R, int gamma, int V, int rank, int dtype_w) {
  using namespace dspark;
  VerifyOverlapLayout L;
  L.v = verify_layout(R, gamma, V, rank, dtype_w);
  L.compact = tc_supported(V, rank, dtype_w) && tc_compact_ok(R * (gamma + 1));
  L.rows = L.compact ? R * (gamma + 1) : R * gamma;
  const size_t rows = (size_t)L.rows;
  L.npart = L.compact ? tc_grid_ctas(L.rows) : overlap_num_partials(R, gamma, V, rank, dtype_w);
  size_t off = L.v.total;
  L.W1g = off;
  off += align256(elem_size(dtype_w) * (size_t)round_up_rows((int)rows) * rank);
  L.lse = off;
  off += align256(4 * rows);
  L.part = off;
  off += align256(4 * rows * (size_t)L.npart);
  L.total = off;
  return L;
}

size_t dspark_verify_workspace_size(int R, int gamma, int V, int rank, int dtype_w) {
  if (R < 1 || gamma < 1 || V < 1 || rank < 1) return 0;
  return verify_layout(R, gamma, V, rank, dtype_w).total;
}

// dspark_verify and dspark_verify_ragged: t_off == nullptr selects the padded target.
static dspark_status verify_impl(int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
                                 const void* target, const int32_t* t_off, int n_trows, const void* U,
                                 const void* W1, const void* state, const void* W2, const int32_t* x0,
                                 const int32_t* x,
                                 const float* logq, const float* lse_q, const int32_t* ell, float temperature,
                                 const int64_t* req_id, uint64_t seed, uint64_t round, int32_t* n_acc_out,
                                 int32_t* tokens_out, int32_t* n_out, void* workspace, size_t ws_bytes,
                                 void* stream, float* overlap_out = nullptr) {
  if (R < 1 || gamma < 1 || V < 1 || rank < 1)
    return fail(DSPARK_INVALID_ARG, "sizes must be positive (R=%d gamma=%d V=%d rank=%d)", R, gamma, V, rank);
  if (gamma > kMaxGamma) return fail(DSPARK_UNSUPPORTED_SHAPE, "gamma=%d exceeds %d", gamma, kMaxGamma);
  if ((long long)V > (1ll << 30)) return fail(DSPARK_UNSUPPORTED_SHAPE, "V=%d too large", V);
  if ((long long)R * (gamma + 1) > (1ll << 24)) return fail(DSPARK_UNSUPPORTED_SHAPE, "R*(gamma+1) too large");
  // the fused overlap's CUDA-core bias pass takes blocks of 4 positions along the grid's y
  if (overlap_out != nullptr && !dspark::tc_supported(V, rank, dtype_w) && ((long long)R * gamma + 3) / 4 > 65535)
    return fail(DSPARK_UNSUPPORTED_SHAPE, "R*gamma=%lld exceeds 262140 without the tensor-core path",
                (long long)R * gamma);
  if (!valid_dtype(dtype_t) || !valid_dtype(dtype_u) || !valid_dtype(dtype_w))
    return fail(DSPARK_INVALID_ARG, "dtype codes must be DSPARK_F32 or DSPARK_BF16");
  if (!(temperature > 0.f) || !isfinite(temperature))
    return fail(DSPARK_INVALID_ARG, "temperature must be finite and > 0");
  CHECK_PTR(target);
  CHECK_PTR(U);
  if (state == nullptr) CHECK_PTR(W1);
  CHECK_PTR(W2);
  CHECK_PTR(x0);
  CHECK_PTR(x);
  CHECK_PTR(logq);
  CHECK_PTR(lse_q);
  CHECK_PTR(ell);
  CHECK_PTR(req_id);
  CHECK_PTR(n_acc_out);
  CHECK_PTR(tokens_out);
  CHECK_PTR(n_out);
  CHECK_PTR(workspace);
  CHECK_ALIGN16(target);
  CHECK_ALIGN16(U);
  if (state == nullptr) CHECK_ALIGN16(W1);
  CHECK_ALIGN16(W2);
  if (!aligned256(workspace)) return fail(DSPARK_INVALID_ARG, "workspace must be 256-byte aligned");
  const VerifyOverlapLayout LO = verify_overlap_layout(R, gamma, V, rank, dtype_w);
  const VerifyLayout& L = LO.v;
  const size_t need = overlap_out != nullptr ? LO.total : L.total;
  if (ws_bytes < need) return fail(DSPARK_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, need);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  dspark::VerifyArgs a = {};
  a.R = R; a.gamma = gamma; a.V = V; a.rank = rank;
  a.dtype_t = dtype_t; a.dtype_u = dtype_u; a.dtype_w = dtype_w;
  a.target = target; a.U = U; a.W1 = W1; a.W2 = W2; a.state = state;
  a.t_off = t_off; a.n_trows = n_trows;
  a.x0 = x0; a.x = x; a.logq = logq; a.lse_q = lse_q; a.ell = ell;
  a.inv_temp = 1.0f / temperature;
  a.req_id = req_id; a.seed = seed; a.round = round;
  a.n_acc_out = n_acc_out; a.tokens_out = tokens_out; a.n_out = n_out;
  a.status = reinterpret_cast<dspark::DeviceStatus*>(ws);
  int* counters = reinterpret_cast<int*>(ws + L.counters);
  a.n_rows = counters;
  a.row_req = reinterpret_cast<int*>(ws + L.row_req);
  a.row_t = reinterpret_cast<int*>(ws + L.row_t);
  a.row_base = reinterpret_cast<int*>(ws + L.row_base);
  a.row_order = reinterpret_cast<int*>(ws + L.row_order);
  a.work_next = counters + 2;
  a.n_rej = counters + 3;
  a.rej_req = reinterpret_cast<int*>(ws + L.rej_req);
  a.n_fb = counters + 4;
  a.fb_req = reinterpret_cast<int*>(ws + L.fb_req);
  a.res_hint = reinterpret_cast<int*>(ws + L.res_hint);
  a.res_compact = dspark::tc_supported(V, rank, dtype_w);
  a.res_grid = dspark::tc_residual_grid(R);
  a.row_part = reinterpret_cast<dspark::Partial*>(ws + L.row_part);
  a.nchunk = L.nchunk;
  a.chunk = kVerifyChunk;
  a.lse_t = reinterpret_cast<float*>(ws + L.lse_t);
  a.jstar = reinterpret_cast<int*>(ws + L.jstar);
  a.W1g = ws + L.W1g;
  a.res_part = reinterpret_cast<dspark::Partial*>(ws + L.res_part);
  a.res_part2 = reinterpret_cast<dspark::Partial*>(ws + L.res_part2);
  a.prof = g_vprof_events;
  if (overlap_out != nullptr) {
    a.ovl_lse = reinterpret_cast<float*>(ws + LO.lse);
    a.ovl_W1g = ws + LO.W1g;
    a.ovl_compact = LO.compact ? 1 : 0;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = dspark::launch_verify(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "verify");
  if (overlap_out != nullptr) {
    // the acceptance overlap on the verify pass's row statistics and factor rows
    dspark::OverlapArgs o = {};
    o.R = R; o.gamma = gamma; o.V = V; o.rank = rank;
    o.dtype_t = dtype_t; o.dtype_u = dtype_u; o.dtype_w = dtype_w;
    o.target = target; o.U = U; o.W1 = W1; o.W2 = W2;
    o.x0 = x0; o.x = x; o.lse_q = lse_q; o.ell = ell;
    o.inv_temp = a.inv_temp;
    o.out = overlap_out;
    o.status = a.status;
    o.W1g = a.ovl_W1g;
    o.lse_t = a.ovl_lse;
    o.part = reinterpret_cast<float*>(ws + LO.part);
    o.npart = LO.npart;
    if (LO.compact) {
      o.row_req = a.row_req;
      o.row_t = a.row_t;
      o.row_base = a.row_base;
      o.n_rows = a.n_rows;
      o.rows_max = LO.rows;
    }
    if ((e = dspark::launch_overlap_pass(o, s)) != cudaSuccess) return cuda_fail(e, "verify_overlap");
  }
  return DSPARK_OK;
}

dspark_status dspark_verify(int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
                            const void* target, const void* U, const void* W1, const void* W2, const int32_t* x0,
                            const int32_t* x, const float* logq, const float* lse_q, const int32_t* ell,
                            float temperature, const int64_t* req_id, uint64_t seed, uint64_t round,
                            int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out, void* workspace,
                            size_t ws_bytes, void* stream) {
  return verify_impl(R, gamma, V, rank, dtype_t, dtype_u, dtype_w, target, nullptr, 0, U, W1, nullptr, W2, x0, x,
                     logq, lse_q, ell, temperature, req_id, seed, round, n_acc_out, tokens_out, n_out, workspace,
                     ws_bytes, stream);
}

dspark_status dspark_verify_ragged(int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
                                   const void* target, int n_target_rows, const int32_t* target_row_offset,
                                   const void* U, const void* W1, const void* W2, const int32_t* x0,
                                   const int32_t* x, const float* logq, const float* lse_q, const int32_t* ell,
                                   float temperature, const int64_t* req_id, uint64_t seed, uint64_t round,
                                   int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out, void* workspace,
                                   size_t ws_bytes, void* stream) {
  if (n_target_rows < 1) return fail(DSPARK_INVALID_ARG, "n_target_rows must be positive (%d)", n_target_rows);
  CHECK_PTR(target_row_offset);
  return verify_impl(R, gamma, V, rank, dtype_t, dtype_u, dtype_w, target, target_row_offset, n_target_rows, U, W1,
                     nullptr, W2, x0, x, logq, lse_q, ell, temperature, req_id, seed, round, n_acc_out, tokens_out,
                     n_out, workspace, ws_bytes, stream);
}

size_t dspark_verify_overlap_workspace_size(int R, int gamma, int V, int rank, int dtype_w) {
  if (R < 1 || gamma < 1 || V < 1 || rank < 1) return 0;
  if ((long long)R * (gamma + 1) > (1ll << 24)) return 0;
  return verify_overlap_layout(R, gamma, V, rank, dtype_w).total;
}

dspark_status dspark_verify_overlap(int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
                                    const void* target, const void* U, const void* W1, const void* W2,
                                    const int32_t* x0, const int32_t* x, const float* logq, const float* lse_q,
                                    const int32_t* ell, float temperature, const int64_t* req_id, uint64_t seed,
                                    uint64_t round, int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out,
                                    float* overlap_out, void* workspace, size_t ws_bytes, void* stream) {
  CHECK_PTR(overlap_out);
  return verify_impl(R, gamma, V, rank, dtype_t, dtype_u, dtype_w, target, nullptr, 0, U, W1, nullptr, W2, x0, x,
                     logq, lse_q, ell, temperature, req_id, seed, round, n_acc_out, tokens_out, n_out, workspace,
                     ws_bytes, stream, overlap_out);
}

size_t dspark_acceptance_overlap_workspace_size(int R, int gamma, int V, int rank, int dtype_w) {
  if (R < 1 || gamma < 1 || V < 1 || rank < 1) return 0;
  if ((long long)R * gamma > (1ll << 24)) return 0;
  return overlap_layout(R, gamma, V, rank, dtype_w).total;
}

dspark_status dspark_acceptance_overlap(int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
                                        const void* target, const void* U, const void* W1, const void* W2,
                                        const int32_t* x0, const int32_t* x, const float* lse_q, const int32_t* ell,
                                        float temperature, float* overlap_out, void* workspace, size_t ws_bytes,
                                        void* stream) {
  if (R < 1 || gamma < 1 || V < 1 || rank < 1)
    return fail(DSPARK_INVALID_ARG, "sizes must be positive (R=%d gamma=%d V=%d rank=%d)", R, gamma, V, rank);
  if (gamma > kMaxGamma) return fail(DSPARK_UNSUPPORTED_SHAPE, "gamma=%d exceeds %d", gamma, kMaxGamma);
  if ((long long)V > (1ll << 30)) return fail(DSPARK_UNSUPPORTED_SHAPE, "V=%d too large", V);
  if ((long long)R * gamma > (1ll << 24)) return fail(DSPARK_UNSUPPORTED_SHAPE, "R*gamma too large");
  if ((long long)R * gamma * dspark::overlap_num_chunks(V) > (1ll << 31) - 1)
    return fail(DSPARK_UNSUPPORTED_SHAPE, "R*gamma*ceil(V/8192) exceeds 2^31-1");
  // the CUDA-core bias pass takes blocks of 4 positions along the grid's y dimension
  if (!dspark::tc_supported(V, rank, dtype_w) && ((long long)R * gamma + 3) / 4 > 65535)
    return fail(DSPARK_UNSUPPORTED_SHAPE, "R*gamma=%lld exceeds 262140 without the tensor-core path",
                (long long)R * gamma);
  if (!valid_dtype(dtype_t) || !valid_dtype(dtype_u) || !valid_dtype(dtype_w))
    return fail(DSPARK_INVALID_ARG, "dtype codes must be DSPARK_F32 or DSPARK_BF16");
  if (!(temperature > 0.f) || !isfinite(temperature))
    return fail(DSPARK_INVALID_ARG, "temperature must be finite and > 0");
  CHECK_PTR(target);
  CHECK_PTR(U);
  CHECK_PTR(W1);
  CHECK_PTR(W2);
  CHECK_PTR(x0);
  CHECK_PTR(x);
  CHECK_PTR(lse_q);
  CHECK_PTR(overlap_out);
  CHECK_PTR(workspace);
  CHECK_ALIGN16(target);
  CHECK_ALIGN16(U);
  CHECK_ALIGN16(W1);
  CHECK_ALIGN16(W2);
  if (!aligned256(workspace)) return fail(DSPARK_INVALID_ARG, "workspace must be 256-byte aligned");
  const OverlapLayout L = overlap_layout(R, gamma, V, rank, dtype_w);
  if (ws_bytes < L.total) return fail(DSPARK_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, L.total);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  dspark::OverlapArgs a = {};
  a.R = R; a.gamma = gamma; a.V = V; a.rank = rank;
  a.dtype_t = dtype_t; a.dtype_u = dtype_u; a.dtype_w = dtype_w;
  a.target = target; a.U = U; a.W1 = W1; a.W2 = W2;
  a.x0 = x0; a.x = x; a.lse_q = lse_q; a.ell = ell;
  a.inv_temp = 1.0f / temperature;
  a.out = overlap_out;
  a.status = reinterpret_cast<dspark::DeviceStatus*>(ws);
  a.W1g = ws + L.W1g;
  a.lse_t = reinterpret_cast<float*>(ws + L.lse_t);
  a.lse_part = reinterpret_cast<float2*>(ws + L.lse_part);
  a.nchunk = L.nchunk;
  a.part = reinterpret_cast<float*>(ws + L.part);
  a.npart = L.npart;
  if (ell != nullptr && dspark::tc_supported(V, rank, dtype_w) && dspark::tc_compact_ok(R * gamma)) {
    // only the evaluated positions go through the tensor-core pass
    a.row_req = reinterpret_cast<int*>(ws + L.row_req);
    a.row_t = reinterpret_cast<int*>(ws + L.row_t);
    a.row_base = reinterpret_cast<int*>(ws + L.row_base);
    a.n_rows = reinterpret_cast<int*>(ws + L.n_rows);
    a.rows_max = R * gamma;
  }
  cudaError_t e = dspark::launch_overlap(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "acceptance_overlap");
  return DSPARK_OK;
}

size_t dspark_rnn_draft_workspace_size(int R, int gamma, int V, int ns, int d, int dtype_w) {
  if (R < 1 || gamma < 1 || V < 1 || ns < 1 || d < 0) return 0;
  return rnn_layout(R, gamma, V, ns, d, dtype_w).total;
}

dspark_status dspark_rnn_draft(int R, int gamma, int V, int ns, int ne, int d, int dtype_u, int dtype_w, int dtype_h,
                               const void* U, const void* E, const void* Wse, const void* Wh, const float* bgc,
                               const void* Wo, const void* h, const float* conf_w, float conf_b,
                               float conf_logit_scale, const float* conf_temp, float temperature, const int32_t* x0,
                               const int64_t* req_id, uint64_t seed, uint64_t round, int32_t* x_out,
                               float* logq_out, float* lse_out, float* conf_out, void* state_out, void* workspace,
                               size_t ws_bytes, void* stream) {
  if (R < 1 || gamma < 1 || V < 1 || ns < 1 || ne < 0 || d < 0)
    return fail(DSPARK_INVALID_ARG, "sizes must be positive (R=%d gamma=%d V=%d ns=%d ne=%d d=%d)", R, gamma, V, ns,
                ne, d);
  if (gamma > kMaxGamma) return fail(DSPARK_UNSUPPORTED_SHAPE, "gamma=%d exceeds %d", gamma, kMaxGamma);
  if ((long long)V > (1ll << 30)) return fail(DSPARK_UNSUPPORTED_SHAPE, "V=%d too large", V);
  if ((long long)R * gamma > (1ll << 24)) return fail(DSPARK_UNSUPPORTED_SHAPE, "R*gamma too large");
  if (ns % 32 != 0 || ns > 256) return fail(DSPARK_UNSUPPORTED_SHAPE, "ns=%d must be a multiple of 32, <= 256", ns);
  if (ne > 2048) return fail(DSPARK_UNSUPPORTED_SHAPE, "ne=%d exceeds 2048", ne);
  if (!valid_dtype(dtype_u) || !valid_dtype(dtype_w) || !valid_dtype(dtype_h))
    return fail(DSPARK_INVALID_ARG, "dtype codes must be DSPARK_F32 or DSPARK_BF16");
  if (!(temperature > 0.f) || !isfinite(temperature))
    return fail(DSPARK_INVALID_ARG, "temperature must be finite and > 0");
  CHECK_PTR(U);
  if (ne > 0) CHECK_PTR(E);
  CHECK_PTR(Wse);
  if (d > 0) CHECK_PTR(Wh);
  CHECK_PTR(bgc);
  CHECK_PTR(Wo);
  if (d > 0) CHECK_PTR(h);
  CHECK_PTR(conf_w);
  CHECK_PTR(conf_temp);
  CHECK_PTR(x0);
  CHECK_PTR(req_id);
  CHECK_PTR(x_out);
  CHECK_PTR(logq_out);
  CHECK_PTR(lse_out);
  CHECK_PTR(conf_out);
  CHECK_PTR(state_out);
  CHECK_PTR(workspace);
  CHECK_ALIGN16(U);
  CHECK_ALIGN16(Wo);
  if (d > 0) CHECK_ALIGN16(h);
  if (d > 0) CHECK_ALIGN16(Wh);
  if (!aligned256(workspace)) return fail(DSPARK_INVALID_ARG, "workspace must be 256-byte aligned");
  const RnnLayout L = rnn_layout(R, gamma, V, ns, d, dtype_w);
  if (ws_bytes < L.total) return fail(DSPARK_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, L.total);

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  dspark::DraftArgs a = {};
  a.R = R; a.gamma = gamma; a.V = V; a.rank = ns; a.d = d;
  a.dtype_u = dtype_u; a.dtype_w = dtype_w; a.dtype_h = dtype_h;
  a.U = U; a.W1 = nullptr; a.W2 = Wo; a.h = h;
  a.conf_w = conf_w; a.conf_b = conf_b; a.conf_scale = conf_logit_scale; a.conf_temp = conf_temp;
  a.inv_temp = 1.0f / temperature;
  a.x0 = x0; a.req_id = req_id; a.seed = seed; a.round = round;
  a.x_out = x_out; a.logq_out = logq_out; a.lse_out = lse_out; a.conf_out = conf_out;
  a.status = reinterpret_cast<dspark::DeviceStatus*>(ws);
  a.s_h = reinterpret_cast<float*>(ws + L.draft.s_h);
  a.W1g = ws + L.draft.W1g;
  a.partials = reinterpret_cast<dspark::Partial*>(ws + L.draft.partials);
  a.hint = reinterpret_cast<int*>(ws + L.draft.hint);
  a.win = reinterpret_cast<unsigned long long*>(ws + L.draft.win);
  a.rnn = 1;
  a.ne = ne; a.E = E; a.Wse = Wse; a.Wh = Wh; a.bgc = bgc;
  a.state_out = state_out;
  a.hpart = reinterpret_cast<float*>(ws + L.hpart);
  a.nsplit = dspark::rnn_num_splits(R, gamma, d, ns, dtype_w, dtype_h);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (d > 0) {
    if ((e = dspark::launch_conf_hdot(a, false, s)) != cudaSuccess) return cuda_fail(e, "conf_hdot");
    if ((e = dspark::launch_rnn_hproj(a, s)) != cudaSuccess) return cuda_fail(e, "rnn_hproj");
  } else {
    if ((e = cudaMemsetAsync(a.s_h, 0, sizeof(float) * (size_t)R * gamma, s)) != cudaSuccess)
      return cuda_fail(e, "s_h clear");
  }
  const bool tc = dspark::tc_supported(V, ns, dtype_w) != 0;
  for (int k = 1; k <= gamma; ++k) {
    if ((e = dspark::launch_rnn_cell(a, k, tc, s)) != cudaSuccess) return cuda_fail(e, "rnn_cell");
    const bool prof = 2 * k <= g_prof_n;
    if (prof && (e = record_profile_event(g_prof_events[2 * (k - 1)], s)) != cudaSuccess)
      return cuda_fail(e, "profile event");
    if (tc) {
      if ((e = dspark::launch_rnn_step_tc(a, k, s)) != cudaSuccess) return cuda_fail(e, "rnn_step_tc");
    } else {
      if ((e = dspark::launch_draft_step_simt(a, k, s)) != cudaSuccess) return cuda_fail(e, "draft_step_simt");
    }
    if (prof && (e = record_profile_event(g_prof_events[2 * (k - 1) + 1], s)) != cudaSuccess)
      return cuda_fail(e, "profile event");
    if (!tc && (e = dspark::launch_draft_combine(a, k, dspark::simt_num_chunks(V), s)) != cudaSuccess)
      return cuda_fail(e, "draft_combine");
  }
  if (tc && (e = dspark::launch_draft_finalize(a, dspark::tc_num_partials(R), s)) != cudaSuccess)
    return cuda_fail(e, "draft_finalize");
  if ((e = dspark::launch_rnn_conf(a, s)) != cudaSuccess) return cuda_fail(e, "rnn_conf");
  return DSPARK_OK;
}

dspark_status dspark_verify_rnn(int R, int gamma, int V, int ns, int dtype_t, int dtype_u, int dtype_w,
                                const void* target, const void* U, const void* state, const void* Wo,
                                const int32_t* x0, const int32_t* x, const float* logq, const float* lse_q,
                                const int32_t* ell, float temperature, const int64_t* req_id, uint64_t seed,
                                uint64_t round, int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out,
                                void* workspace, size_t ws_bytes, void* stream) {
  CHECK_PTR(state);
  return verify_impl(R, gamma, V, ns, dtype_t, dtype_u, dtype_w, target, nullptr, 0, U, nullptr, state, Wo, x0, x,
                     logq, lse_q, ell, temperature, req_id, seed, round, n_acc_out, tokens_out, n_out, workspace,
                     ws_bytes, stream);
}

namespace {
struct StsLayout {
  size_t zt, prefix, part, ece_g, total;
  int S;
};
StsLayout sts_layout(int N, int gamma, int G, int M) {
  StsLayout L;
  L.S = dspark::sts_num_chunks(N);
  size_t off = 256;
  L.zt = off;
  off += dspark::align256(sizeof(float) * (size_t)N * gamma);
  L.prefix = off;
  off += dspark::align256(sizeof(float) * (size_t)N);
  L.part = off;
  off += dspark::align256(sizeof(float) * (size_t)G * L.S * M);
  L.ece_g = off;
  off += dspark::align256(sizeof(double) * (size_t)G);
  L.total = off;
  return L;
}
}  // namespace

size_t dspark_sts_fit_workspace_size(int N, int gamma, int G, int M) {
  if (N < 1 || gamma < 1 || G < 1 || M < 1) return 0;
  return sts_layout(N, gamma, G, M).total;
}

dspark_status dspark_sts_fit(int N, int gamma, const float* z, const int32_t* acc_len, const float* grid, int G,
                             int M, float* T_out, float* ece_out, void* workspace, size_t ws_bytes, void* stream) {
  if (N < 1 || gamma < 1 || G < 1 || M < 1)
    return fail(DSPARK_INVALID_ARG, "sizes must be positive (N=%d gamma=%d G=%d M=%d)", N, gamma, G, M);
  if (gamma > kMaxGamma) return fail(DSPARK_UNSUPPORTED_SHAPE, "gamma=%d exceeds %d", gamma, kMaxGamma);
  if (M > dspark::kStsMaxBins) return fail(DSPARK_UNSUPPORTED_SHAPE, "M=%d bins exceed %d", M, dspark::kStsMaxBins);
  if (G > 65535) return fail(DSPARK_UNSUPPORTED_SHAPE, "G=%d candidates exceed 65535", G);
  if ((long long)N * gamma > (1ll << 31) - 1) return fail(DSPARK_UNSUPPORTED_SHAPE, "N*gamma too large");
  CHECK_PTR(z);
  CHECK_PTR(acc_len);
  CHECK_PTR(grid);
  CHECK_PTR(T_out);
  CHECK_PTR(ece_out);
  CHECK_PTR(workspace);
  if (!aligned256(workspace)) return fail(DSPARK_INVALID_ARG, "workspace must be 256-byte aligned");
  const StsLayout L = sts_layout(N, gamma, G, M);
  if (ws_bytes < L.total) return fail(DSPARK_WORKSPACE_TOO_SMALL, "workspace %zu bytes, need %zu", ws_bytes, L.total);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  dspark::StsArgs a = {};
  a.N = N; a.gamma = gamma; a.G = G; a.M = M;
  a.z = z; a.acc_len = acc_len; a.grid = grid; a.T_out = T_out; a.ece_out = ece_out;
  a.status = reinterpret_cast<dspark::DeviceStatus*>(ws);
  a.zt = reinterpret_cast<float*>(ws + L.zt);
  a.prefix = reinterpret_cast<float*>(ws + L.prefix);
  a.part = reinterpret_cast<float*>(ws + L.part);
  a.ece_g = reinterpret_cast<double*>(ws + L.ece_g);
  a.S = L.S;
  cudaError_t e = dspark::launch_sts_fit(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sts_fit");
  return DSPARK_OK;
}

}  // extern "C"
