// rnn.cu — the recurrent draft head: the parts that run on CUDA cores.
//
// The head keeps a running state over the block instead of only the previous token
// (numb3r33 blog "DSpark: confidence-scheduled speculative decoding", section "RNN
// sequential head": s_k = f(s_{k-1}, E(x_{k-1}), h_k), z_k = U_k + W_o s_k; DSpark 精读
// §2: f is a gated update of the concatenation of the state, the previous token's
// embedding and the position's hidden state).  The gate is read as the update-gate cell
//   a   = [s_{k-1}; E[x_{k-1}]] Wse + h_k Wh + b   (2*ns pre-activations: gate, candidate)
//   s_k = (1 - sigmoid(a_gate)) * s_{k-1} + sigmoid(a_gate) * tanh(a_cand),  s_0 = 0,
// and the state is stored in the weights' type (bf16 rounded to nearest even, or fp32),
// which makes it the A operand of the bias contraction s_k W_o.
//
//   rnn_hproj   h Wh for every (request, position) before the loop (it does not depend
//               on the drafted tokens): split over the hidden dimension, partial sums;
//               a tensor-core GEMM (hproj_tc_kernel) for bf16 operands, else CUDA cores
//   rnn_cell    position k: x_{k-1} (anchor, or position k-1's winner) -> s_k, written
//               to the state output and to the factor-row buffer the draft step reads
//   rnn_conf    after the loop: c_k = sigmoid(kappa (w_h . h_k + w_s . s_k + b) / T_k)
//
// The vocabulary pass of each position is the Markov head's (tensor cores or CUDA
// cores) with the state in place of the gathered factor row W1[x_{k-1}].
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kHRows = 8;        // hidden-state rows per CTA of the CUDA-core projection
constexpr int kHSplit = 512;     // hidden dimensions per split (CUDA-core projection)
constexpr int kCellReq = 4;      // requests per CTA of rnn_cell
constexpr int kCellCols = 8;     // state columns per CTA of rnn_cell (x2: gate and candidate)
constexpr int kCellSlices = 16;  // slices of the input vector per column
constexpr int kCellThreads = 2 * kCellCols * kCellSlices;

// hpart[split][row][c] = sum over the split's hidden dimensions i of h[row][i] Wh[i][c].
// Thread t owns the gate column t and the candidate column ns + t for kHRows rows.
__global__ void rnn_hproj_kernel(DraftArgs a) {
  griddep_allow_next();
  griddep_wait();
  __shared__ float hs[kHRows][kHSplit];
  const int ns = a.rank, n2 = 2 * ns;
  const int rows = a.R * a.gamma;
  const int row0 = blockIdx.x * kHRows;
  const int i0 = blockIdx.y * kHSplit;
  const int len = min(kHSplit, a.d - i0);
  for (int e = threadIdx.x; e < kHRows * kHSplit; e += blockDim.x) {
    const int rr = e / kHSplit, i = e % kHSplit;
    const int row = row0 + rr;
    hs[rr][i] = (row < rows && i < len) ? load_elem(a.h, a.dtype_h, (size_t)row * a.d + i0 + i) : 0.f;
  }
  __syncthreads();
  const int t = threadIdx.x;
  float ag[kHRows], ac[kHRows];
#pragma unroll
  for (int rr = 0; rr < kHRows; ++rr) ag[rr] = ac[rr] = 0.f;
  // four hidden dimensions per step: their eight weights are loaded before any is used
  int i = 0;
  for (; i + 4 <= len; i += 4) {
    float wg[4], wc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const size_t w = (size_t)(i0 + i + q) * n2;
      wg[q] = load_elem(a.Wh, a.dtype_w, w + t);
      wc[q] = load_elem(a.Wh, a.dtype_w, w + ns + t);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int rr = 0; rr < kHRows; ++rr) {
        ag[rr] = fmaf(hs[rr][i + q], wg[q], ag[rr]);
        ac[rr] = fmaf(hs[rr][i + q], wc[q], ac[rr]);
      }
  }
  for (; i < len; ++i) {
    const size_t w = (size_t)(i0 + i) * n2;
    const float wg = load_elem(a.Wh, a.dtype_w, w + t);
    const float wc = load_elem(a.Wh, a.dtype_w, w + ns + t);
#pragma unroll
    for (int rr = 0; rr < kHRows; ++rr) {
      ag[rr] = fmaf(hs[rr][i], wg, ag[rr]);
      ac[rr] = fmaf(hs[rr][i], wc, ac[rr]);
    }
  }
#pragma unroll
  for (int rr = 0; rr < kHRows; ++rr) {
    const int row = row0 + rr;
    if (row >= rows) break;
    float* out = a.hpart + ((size_t)blockIdx.y * rows + row) * n2;
    out[t] = ag[rr];
    out[ns + t] = ac[rr];
  }
}

// Sum of the projection's splits into split 0, in split order (before the position loop,
// so that each cell reads one value per pre-activation).
__global__ void rnn_hsum_kernel(DraftArgs a) {
  griddep_allow_next();
  griddep_wait();
  const size_t n = (size_t)a.R * a.gamma * 2 * a.rank;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float v = a.hpart[i];
  for (int sp = 1; sp < a.nsplit; ++sp) v += a.hpart[(size_t)sp * n + i];
  a.hpart[i] = v;
}

__device__ __forceinline__ void store_state(void* base, int dtype, size_t idx, float v) {
  if (dtype == DSPARK_BF16)
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(base)[idx] = v;
}

// Position k: CTA (block of kCellReq requests, block of kCellCols state columns).  Thread
// (pre-activation column j, slice q) accumulates column j (the first kCellCols are gate
// columns, the others the matching candidate columns) over the input entries q,
// q + kCellSlices, ... for all the CTA's requests, so each weight is loaded once per
// CTA; the slices are then added in a fixed order and kCellCols x kCellReq threads
// finish the update.
// BATCH: weights loaded per thread before any is used; STAGE: input entries per thread and
// step.  Small batches issue every load at once (the cell is a chain of L2 round trips);
// large batches use fewer registers across their thousands of CTAs.
template <int BATCH, int STAGE>
__global__ void __launch_bounds__(kCellThreads) rnn_cell_kernel(DraftArgs a, int k, int tc) {
  extern __shared__ float us[];  // [kCellReq][ns + ne]: s_{k-1}; E[x_{k-1}]
  __shared__ int xs[kCellReq];
  __shared__ float red[kCellSlices][2 * kCellCols][kCellReq];
  const int ns = a.rank, n2 = 2 * ns, nu = ns + a.ne;
  const int r0 = blockIdx.x * kCellReq;
  const int c0 = blockIdx.y * kCellCols;
  const int j = threadIdx.x % (2 * kCellCols);  // pre-activation column within the CTA
  const int q = threadIdx.x / (2 * kCellCols);  // input slice
  const int cj = j < kCellCols ? c0 + j : ns + c0 + (j - kCellCols);  // column of Wse
  const bool col_ok = c0 + (j % kCellCols) < ns;
  griddep_allow_next();
  griddep_wait();
  // the finishing threads' bias and hidden-state projection, loaded ahead of the rest
  float hb_g = 0.f, hb_c = 0.f;
  {
    const int cc = threadIdx.x % kCellCols, rr = threadIdx.x / kCellCols;
    if (threadIdx.x < kCellCols * kCellReq && r0 + rr < a.R && c0 + cc < ns) {
      hb_g = __ldg(a.bgc + c0 + cc);
      hb_c = __ldg(a.bgc + ns + c0 + cc);
      if (a.nsplit > 0) {  // split 0 holds the sum of all splits
        const float* hp = a.hpart + (size_t)((r0 + rr) * a.gamma + (k - 1)) * n2;
        hb_g += hp[c0 + cc];
        hb_c += hp[ns + c0 + cc];
      }
    }
  }
  if (threadIdx.x < kCellReq) {
    const int r = r0 + threadIdx.x;
    int x = 0;
    if (r < a.R) {
      int raw;
      if (k == 1)
        raw = __ldg(a.x0 + r);
      else if (tc)
        raw = (int)~(uint32_t)(a.win[(size_t)(k - 2) * a.R + r] & 0xFFFFFFFFull);
      else
        raw = a.x_out[(size_t)r * a.gamma + (k - 2)];
      x = checked_token(raw, a.V, a.status, 4);
    }
    xs[threadIdx.x] = x;
  }
  // tensor-core path: every position's bound and winner start empty
  if (k == 1 && tc && blockIdx.y == 0)
    for (int i = threadIdx.x; i < kCellReq * a.gamma; i += blockDim.x) {
      const int r = r0 + i / a.gamma, pos = i % a.gamma;
      if (r < a.R) {
        a.hint[(size_t)pos * a.R + r] = __float_as_int(-INFINITY) ^ 0x7FFFFFFF;
        a.win[(size_t)pos * a.R + r] = 0ull;
      }
    }
  __syncthreads();
  // STAGE entries per thread and step, loaded before they are stored
  for (int e0 = threadIdx.x; e0 < kCellReq * nu; e0 += STAGE * blockDim.x) {
    float v[STAGE];
#pragma unroll
    for (int u4 = 0; u4 < STAGE; ++u4) {
      const int e = e0 + u4 * blockDim.x;
      v[u4] = 0.f;
      if (e >= kCellReq * nu) continue;
      const int rr = e / nu, j = e % nu;
      const int r = r0 + rr;
      if (r < a.R) {
        if (j < ns)
          v[u4] = k == 1 ? 0.f : load_elem(a.state_out, a.dtype_w, ((size_t)r * a.gamma + (k - 2)) * ns + j);
        else
          v[u4] = load_elem(a.E, a.dtype_w, (size_t)xs[rr] * a.ne + (j - ns));
      }
    }
#pragma unroll
    for (int u4 = 0; u4 < STAGE; ++u4)
      if (e0 + u4 * blockDim.x < kCellReq * nu) us[e0 + u4 * blockDim.x] = v[u4];
  }
  __syncthreads();
  float acc[kCellReq];
#pragma unroll
  for (int rr = 0; rr < kCellReq; ++rr) acc[rr] = 0.f;
  if (col_ok) {
    int i = q;
    // BATCH input entries per step: their weights are loaded before any is used
    for (; i + (BATCH - 1) * kCellSlices < nu; i += BATCH * kCellSlices) {
      float w[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) w[u] = load_elem(a.Wse, a.dtype_w, (size_t)(i + u * kCellSlices) * n2 + cj);
#pragma unroll
      for (int u = 0; u < BATCH; ++u)
#pragma unroll
        for (int rr = 0; rr < kCellReq; ++rr) acc[rr] = fmaf(us[rr * nu + i + u * kCellSlices], w[u], acc[rr]);
    }
    for (; i < nu; i += kCellSlices) {
      const float w = load_elem(a.Wse, a.dtype_w, (size_t)i * n2 + cj);
#pragma unroll
      for (int rr = 0; rr < kCellReq; ++rr) acc[rr] = fmaf(us[rr * nu + i], w, acc[rr]);
    }
  }
#pragma unroll
  for (int rr = 0; rr < kCellReq; ++rr) red[q][j][rr] = acc[rr];
  __syncthreads();
  if (threadIdx.x >= kCellCols * kCellReq) return;
  const int cc = threadIdx.x % kCellCols, rr = threadIdx.x / kCellCols;
  const int c = c0 + cc;
  const int r = r0 + rr;
  if (r >= a.R || c >= ns) return;
  const int row = r * a.gamma + (k - 1);
  float ag = hb_g, ac = hb_c;
#pragma unroll
  for (int qq = 0; qq < kCellSlices; ++qq) {
    ag += red[qq][cc][rr];
    ac += red[qq][kCellCols + cc][rr];
  }
  const float g = 1.f / (1.f + __expf(-ag));
  const float s = (1.f - g) * us[rr * nu + c] + g * tanhf(ac);
  store_state(a.state_out, a.dtype_w, (size_t)row * ns + c, s);
  store_state(a.W1g, a.dtype_w, (size_t)r * ns + c, s);
}

// One warp per (request, position): the confidence from the hidden-state part and the
// stored state.
__global__ void rnn_conf_kernel(DraftArgs a) {
  griddep_allow_next();
  griddep_wait();
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= a.R * a.gamma) return;
  const int k = wid % a.gamma + 1;
  const float* w_s = a.conf_w + a.d;
  float acc = 0.f;
  for (int i = lane; i < a.rank; i += 32)
    acc = fmaf(__ldg(w_s + i), load_elem(a.state_out, a.dtype_w, (size_t)wid * a.rank + i), acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    const float logit = a.conf_scale * (a.s_h[wid] + acc + a.conf_b);
    a.conf_out[wid] = sigmoidf_dev(logit / __ldg(a.conf_temp + (k - 1)));
  }
}

cudaError_t launch_rnn_hproj(const DraftArgs& a, cudaStream_t s) {
  cudaError_t e;
  const int rows = a.R * a.gamma;
  if (rnn_hproj_on_tc(a.d, a.rank, a.dtype_w, a.dtype_h)) {
    e = launch_rnn_hproj_tc(a, s);
  } else {
    if (a.nsplit != (a.d + kHSplit - 1) / kHSplit) return cudaErrorInvalidValue;
    dim3 grid((rows + kHRows - 1) / kHRows, a.nsplit);
    e = launch_pdl(rnn_hproj_kernel, grid, dim3(a.rank), 0, s, a);
  }
  if (e != cudaSuccess || a.nsplit <= 1) return e;
  const size_t n = (size_t)rows * 2 * a.rank;
  return launch_pdl(rnn_hsum_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, a);
}

cudaError_t launch_rnn_cell(const DraftArgs& a, int k, bool tc, cudaStream_t s) {
  dim3 grid((a.R + kCellReq - 1) / kCellReq, (a.rank + kCellCols - 1) / kCellCols);
  const size_t smem = sizeof(float) * kCellReq * (a.rank + a.ne);
  // few requests: every weight load at once; many: smaller batches (measured both ways)
  if (a.R <= 64) return launch_pdl(rnn_cell_kernel<32, 8>, grid, dim3(kCellThreads), smem, s, a, k, tc ? 1 : 0);
  return launch_pdl(rnn_cell_kernel<8, 4>, grid, dim3(kCellThreads), smem, s, a, k, tc ? 1 : 0);
}

cudaError_t launch_rnn_conf(const DraftArgs& a, cudaStream_t s) {
  const int warps = a.R * a.gamma;
  return launch_pdl(rnn_conf_kernel, dim3((warps * 32 + 255) / 256), dim3(256), 0, s, a);
}

}  // namespace dspark
