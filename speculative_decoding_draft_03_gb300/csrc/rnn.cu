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
//               on the drafted tokens): split over the hidden dimension, partial sums
//   rnn_cell    position k: x_{k-1} (anchor, or position k-1's winner) -> s_k, written
//               to the state output and to the factor-row buffer the draft step reads
//   rnn_conf    after the loop: c_k = sigmoid(kappa (w_h . h_k + w_s . s_k + b) / T_k)
//
// The vocabulary pass of each position is the Markov head's (tensor cores or CUDA
// cores) with the state in place of the gathered factor row W1[x_{k-1}].
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kHRows = 8;        // hidden-state rows per CTA of rnn_hproj
constexpr int kHSplit = 512;     // hidden dimensions per split
constexpr int kCellReq = 4;      // requests per CTA of rnn_cell
constexpr int kCellCols = 64;    // state columns per CTA of rnn_cell

int rnn_num_splits(int d) { return (d + kHSplit - 1) / kHSplit; }

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
  for (int i = 0; i < len; ++i) {
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

__device__ __forceinline__ void store_state(void* base, int dtype, size_t idx, float v) {
  if (dtype == DSPARK_BF16)
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(base)[idx] = v;
}

// Position k: CTA (block of kCellReq requests, block of kCellCols state columns); thread
// (request rr, column c) forms the gate and candidate pre-activations of column c.
__global__ void __launch_bounds__(kCellReq * kCellCols) rnn_cell_kernel(DraftArgs a, int k, int tc) {
  griddep_allow_next();
  griddep_wait();
  extern __shared__ float us[];  // [kCellReq][ns + ne]: s_{k-1}; E[x_{k-1}]
  __shared__ int xs[kCellReq];
  const int ns = a.rank, n2 = 2 * ns, nu = ns + a.ne;
  const int r0 = blockIdx.x * kCellReq;
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
  for (int e = threadIdx.x; e < kCellReq * nu; e += blockDim.x) {
    const int rr = e / nu, j = e % nu;
    const int r = r0 + rr;
    float v = 0.f;
    if (r < a.R) {
      if (j < ns)
        v = k == 1 ? 0.f : load_elem(a.state_out, a.dtype_w, ((size_t)r * a.gamma + (k - 2)) * ns + j);
      else
        v = load_elem(a.E, a.dtype_w, (size_t)xs[rr] * a.ne + (j - ns));
    }
    us[e] = v;
  }
  __syncthreads();
  const int rr = threadIdx.x / kCellCols;
  const int c = blockIdx.y * kCellCols + threadIdx.x % kCellCols;
  const int r = r0 + rr;
  if (r >= a.R || c >= ns) return;
  const int row = r * a.gamma + (k - 1);
  const int rows = a.R * a.gamma;
  float ag = __ldg(a.bgc + c), ac = __ldg(a.bgc + ns + c);
  for (int sp = 0; sp < a.nsplit; ++sp) {
    const float* hp = a.hpart + ((size_t)sp * rows + row) * n2;
    ag += hp[c];
    ac += hp[ns + c];
  }
  const float* u = us + rr * nu;
  for (int j = 0; j < nu; ++j) {
    ag = fmaf(u[j], load_elem(a.Wse, a.dtype_w, (size_t)j * n2 + c), ag);
    ac = fmaf(u[j], load_elem(a.Wse, a.dtype_w, (size_t)j * n2 + ns + c), ac);
  }
  const float g = 1.f / (1.f + __expf(-ag));
  const float s = (1.f - g) * u[c] + g * tanhf(ac);
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
  const int rows = a.R * a.gamma;
  dim3 grid((rows + kHRows - 1) / kHRows, a.nsplit);
  return launch_pdl(rnn_hproj_kernel, grid, dim3(a.rank), 0, s, a);
}

cudaError_t launch_rnn_cell(const DraftArgs& a, int k, bool tc, cudaStream_t s) {
  dim3 grid((a.R + kCellReq - 1) / kCellReq, (a.rank + kCellCols - 1) / kCellCols);
  const size_t smem = sizeof(float) * kCellReq * (a.rank + a.ne);
  return launch_pdl(rnn_cell_kernel, grid, dim3(kCellReq * kCellCols), smem, s, a, k, tc ? 1 : 0);
}

cudaError_t launch_rnn_conf(const DraftArgs& a, cudaStream_t s) {
  const int warps = a.R * a.gamma;
  return launch_pdl(rnn_conf_kernel, dim3((warps * 32 + 255) / 256), dim3(256), 0, s, a);
}

}  // namespace dspark
