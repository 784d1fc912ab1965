// draft_simt.cu — Markov-head draft stage: the parts that run on CUDA cores.
//
//   conf_hdot      s_h[r,k] = w_h . h[r,k,:]        (confidence head, hidden-state part)
//   draft_prepare  for position k: x_{k-1} -> gathered factor row W1[x_{k-1},:] (the
//                  A operand of the bias contraction) and the confidence
//                  c_k = sigmoid(kappa (s_h + w_e . W1[x_{k-1}] + b) / T_k)
//   draft_step_simt  fp32 (or small bf16) path of one draft position: bias row
//                  W1[x_{k-1}] W2 on CUDA cores, z = (U_k + bias)/T, online softmax
//                  statistics and Gumbel-max draw, one partial record per
//                  (vocabulary chunk, request)
//   draft_combine  merges the partials of a position into x_k, lse_k, logq_k and
//                  prepares position k+1 (one CTA per request).
//   draft_round_simt  the three above for every position in one launch, when the
//                  vocabulary is a single chunk (small vocabularies).
//
// Method: numb3r33 blog "DSpark: confidence-scheduled speculative decoding", sections
// "Markov sequential head" (p_k(v|x_{k-1}) = softmax(U_k(v) + W1[x_{k-1}] W2)) and
// "Confidence head"; DSpark 精读 §2 and §4 (confidence on [h_k ; W1[x_{k-1}]]).
//
// Every kernel is launched with programmatic dependent launch and waits for its
// predecessor (griddep_wait) before its first dependent access.
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kCombineThreads = 128;

// s_h[row] = w_h . h[row,:] for the R*gamma rows of h.  A CTA of 256 threads takes two
// rows, four warps per row; each lane issues all of its 16-byte loads of an iteration
// before using them, and the four warp sums are added in a fixed order (deterministic).
constexpr int kHdotThreads = 256;
constexpr int kHdotWarpsPerRow = 4;
constexpr int kHdotRowsPerCta = kHdotThreads / 32 / kHdotWarpsPerRow;
constexpr int kHdotUnroll = 4;

// With n_reset > 0 it also empties the tensor-core path's per-position bounds and winners
// (hint, win: n_reset = gamma * R entries each), so that position 1 needs no prepare launch.
__global__ void __launch_bounds__(kHdotThreads) conf_hdot_kernel(int rows, int d, int dtype_h,
                                                                 const void* __restrict__ h,
                                                                 const float* __restrict__ w_h,
                                                                 float* __restrict__ s_h, int* hint,
                                                                 unsigned long long* win, int n_reset) {
  griddep_allow_next();
  griddep_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_reset; i += gridDim.x * blockDim.x) {
    hint[i] = __float_as_int(-INFINITY) ^ 0x7FFFFFFF;  // order-preserving code of -inf
    win[i] = 0ull;
  }
  __shared__ float part[kHdotRowsPerCta][kHdotWarpsPerRow];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int local = warp / kHdotWarpsPerRow, sub = warp % kHdotWarpsPerRow;
  const int row = blockIdx.x * kHdotRowsPerCta + local;
  constexpr int kStride = 32 * kHdotWarpsPerRow;  // lanes per row
  float acc = 0.f;
  if (row < rows) {
    const size_t base = (size_t)row * d;
    const bool vec = dtype_h == DSPARK_BF16 && (d % 8) == 0 && (reinterpret_cast<uintptr_t>(h) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(w_h) & 15u) == 0;
    if (vec) {
      const int n8 = d / 8;
      const uint4* hp = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(h) + base);
      for (int c0 = sub * 32 + lane; c0 < n8; c0 += kHdotUnroll * kStride) {
        uint4 q[kHdotUnroll];
#pragma unroll
        for (int u = 0; u < kHdotUnroll; ++u) {
          const int c = c0 + u * kStride;
          q[u] = (c < n8) ? __ldg(hp + c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kHdotUnroll; ++u) {
          const int c = c0 + u * kStride;
          if (c >= n8) break;
          const uint32_t wd[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
          // the 8 weights of the chunk in two 16-byte loads (L1/L2 hits: w_h is 4d bytes)
          const float4 w0 = __ldg(reinterpret_cast<const float4*>(w_h) + 2 * c);
          const float4 w1 = __ldg(reinterpret_cast<const float4*>(w_h) + 2 * c + 1);
          const float we[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc = fmaf(we[2 * e], bf16_bits_to_float(wd[e] & 0xFFFFu), acc);
            acc = fmaf(we[2 * e + 1], bf16_bits_to_float(wd[e] >> 16), acc);
          }
        }
      }
    } else {
      for (int i = sub * 32 + lane; i < d; i += kStride) acc = fmaf(__ldg(w_h + i), load_elem(h, dtype_h, base + i), acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) part[local][sub] = acc;
  __syncthreads();
  if (threadIdx.x < kHdotRowsPerCta) {
    const int rr = blockIdx.x * kHdotRowsPerCta + threadIdx.x;
    if (rr < rows) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kHdotWarpsPerRow; ++w) t += part[threadIdx.x][w];
      s_h[rr] = t;
    }
  }
}

// Gather W1[x_prev] into W1g[r] and write c_k; executed by one warp.  Lane l covers the
// factor ids [8l, 8l+8) with one 16-byte load (bf16 rows of rank <= 256), so the whole
// row arrives after one memory latency.
__device__ void prepare_position_warp(const DraftArgs& a, int r, int k, int x_prev, int lane) {
  const size_t src = (size_t)x_prev * a.rank;
  const size_t dst = (size_t)r * a.rank;
  const float* w_e = a.conf_w + a.d;
  float acc = 0.f;
  if (a.dtype_w == DSPARK_BF16 && (a.rank % 8) == 0) {
    const uint4* w1 = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(a.W1) + src);
    uint4* g = reinterpret_cast<uint4*>(reinterpret_cast<unsigned short*>(a.W1g) + dst);
    for (int c = lane; c < a.rank / 8; c += 32) {
      const uint4 q = __ldg(w1 + c);
      g[c] = q;
      const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__ldg(w_e + 8 * c + 2 * e), bf16_bits_to_float(wd[e] & 0xFFFFu), acc);
        acc = fmaf(__ldg(w_e + 8 * c + 2 * e + 1), bf16_bits_to_float(wd[e] >> 16), acc);
      }
    }
  } else if (a.dtype_w == DSPARK_BF16) {
    const unsigned short* w1 = reinterpret_cast<const unsigned short*>(a.W1);
    unsigned short* g = reinterpret_cast<unsigned short*>(a.W1g);
    for (int i = lane; i < a.rank; i += 32) {
      const unsigned short bits = __ldg(w1 + src + i);
      g[dst + i] = bits;
      acc = fmaf(__ldg(w_e + i), bf16_bits_to_float(bits), acc);
    }
  } else {
    const float* w1 = reinterpret_cast<const float*>(a.W1);
    float* g = reinterpret_cast<float*>(a.W1g);
    for (int i = lane; i < a.rank; i += 32) {
      const float v = __ldg(w1 + src + i);
      g[dst + i] = v;
      acc = fmaf(__ldg(w_e + i), v, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    const size_t row = (size_t)r * a.gamma + (k - 1);
    const float logit = a.conf_scale * (a.s_h[row] + acc + a.conf_b);
    a.conf_out[row] = sigmoidf_dev(logit / __ldg(a.conf_temp + (k - 1)));
    // no Gumbel key of position k has been seen yet: the running bound starts at -inf
    // (the order-preserving int code of -inf)
    a.hint[r] = __float_as_int(-INFINITY) ^ 0x7FFFFFFF;
  }
  // tensor-core path: every position's bound and winner start empty
  if (k == 1)
    for (int i = lane; i < a.gamma; i += 32) {
      a.hint[(size_t)i * a.R + r] = __float_as_int(-INFINITY) ^ 0x7FFFFFFF;
      a.win[(size_t)i * a.R + r] = 0ull;
    }
}

// Position 1: one warp per request.
__global__ void __launch_bounds__(32) draft_prepare_kernel(DraftArgs a, int k) {
  griddep_allow_next();
  griddep_wait();
  const int r = blockIdx.x;
  const int raw = (k == 1) ? __ldg(a.x0 + r) : a.x_out[(size_t)r * a.gamma + (k - 2)];
  const int x_prev = checked_token(raw, a.V, a.status, 1);
  prepare_position_warp(a, r, k, x_prev, threadIdx.x & 31);
}

// ---------------------------------------------------------------------------------
// CUDA-core draft step.  blockIdx.x: vocabulary chunk of kSimtGroups*4*blockDim.x ids;
// blockIdx.y: block of RB requests.  Each thread owns groups of 4 consecutive ids so
// that one Philox block serves its 4 elements of a request row.
// ---------------------------------------------------------------------------------
// One draft position for request block r0 .. r0+RB-1 over vocabulary chunk `chunk`
// (the caller has synchronised after writing the block's factor rows W1g).  Writes the
// chunk's partial record per request, or, when the chunk is the whole vocabulary
// (final), the position's x_k, lse_k and logq_k directly (the merge of one record).
template <int RB>
__device__ __forceinline__ void simt_step_block(const DraftArgs& a, int k, int chunk, int r0, bool final,
                                                float* w1s) {
  for (int i = threadIdx.x; i < RB * a.rank; i += blockDim.x) {
    const int rr = i / a.rank, c = i % a.rank;
    const int r = r0 + rr;
    w1s[i] = (r < a.R) ? load_elem(a.W1g, a.dtype_w, (size_t)r * a.rank + c) : 0.f;
  }
  __syncthreads();

  Stats st[RB];
  RngRow rng[RB];
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) {
    st[rr] = stats_empty();
    const int r = min(r0 + rr, a.R - 1);
    rng[rr] = rng_row(a.seed, __ldg(a.req_id + r), a.round, kStreamDraft, (uint32_t)k);
  }
  const int groups_total = (a.V + 3) / 4;
  const int g0 = chunk * kSimtGroups * blockDim.x;
  for (int t = 0; t < kSimtGroups; ++t) {
    const int g = g0 + t * blockDim.x + threadIdx.x;
    if (g >= groups_total) break;
    float acc[RB][4];
#pragma unroll
    for (int rr = 0; rr < RB; ++rr)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rr][e] = 0.f;
    // unrolled so that several rank rows' W2 loads are in flight before their products
#pragma unroll 8
    for (int i = 0; i < a.rank; ++i) {
      float w2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = 4 * g + e;
        w2[e] = (v < a.V) ? load_elem(a.W2, a.dtype_w, (size_t)i * a.V + v) : 0.f;
      }
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) {
        const float w1 = w1s[rr * a.rank + i];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[rr][e] = fmaf(w1, w2[e], acc[rr][e]);
      }
    }
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      const int r = r0 + rr;
      if (r >= a.R) break;
      const Philox4 bits = rng_chunk(rng[rr], (uint32_t)g);
      const uint32_t wd[4] = {bits.x, bits.y, bits.z, bits.w};
      const size_t urow = ((size_t)r * a.gamma + (k - 1)) * a.V;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = 4 * g + e;
        if (v >= a.V) break;
        const float z = (load_elem(a.U, a.dtype_u, urow + v) + acc[rr][e]) * a.inv_temp;
        // online softmax statistics
        if (z > st[rr].m) {
          st[rr].s = st[rr].s * __expf(st[rr].m - z) + 1.f;
          st[rr].m = z;
        } else {
          st[rr].s += __expf(z - st[rr].m);
        }
        // Gumbel-max: skip the draw when even the largest Gumbel cannot win
        if (z + kGumbelMax >= st[rr].key || st[rr].idx < 0) {
          const float key = z + gumbel_fast_from_bits(wd[e]);
          if (key > st[rr].key || st[rr].idx < 0) {
            st[rr].key = key;
            st[rr].idx = v;
            st[rr].zsel = z;
          }
        }
      }
    }
  }
  // block reduction per request: warp shuffle, then across warps through shared memory
  __shared__ Partial red[kSimtThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) {
    const int r = r0 + rr;
    Stats w = warp_reduce_stats(st[rr]);
    if (lane == 0) red[warp] = to_partial(w);
    __syncthreads();
    if (warp == 0) {
      Stats b = (lane < (int)(blockDim.x >> 5)) ? from_partial(red[lane]) : stats_empty();
      b = warp_reduce_stats(b);
      if (lane == 0 && r < a.R) {
        if (final) {
          // the merge of this single record, as the combine kernel computes it
          Stats m = stats_empty();
          stats_merge(m, b);
          const size_t row = (size_t)r * a.gamma + (k - 1);
          const float lse = m.m + logf(m.s);
          a.x_out[row] = m.idx;
          a.lse_out[row] = lse;
          a.logq_out[row] = m.zsel - lse;
        } else {
          a.partials[(size_t)chunk * a.R + r] = to_partial(b);
        }
      }
    }
    __syncthreads();
  }
}

template <int RB>
__global__ void __launch_bounds__(kSimtThreads) draft_step_simt_kernel(DraftArgs a, int k) {
  griddep_wait();
  extern __shared__ float w1s[];  // [RB][rank]
  simt_step_block<RB>(a, k, blockIdx.x, blockIdx.y * RB, false, w1s);
}

// The whole draft loop of one request block when the vocabulary is one chunk: for
// k = 1..gamma, warps 0..RB-1 gather their request's factor row W1[x_{k-1}] and c_k
// (x_0 = the anchor, then the previous position's draw), then the block runs the position
// and writes x_k, lse_k, logq_k itself.  The same arithmetic as the per-position kernels
// (step, combine, prepare) in one launch.
template <int RB>
__global__ void __launch_bounds__(kSimtThreads) draft_round_simt_kernel(DraftArgs a) {
  griddep_allow_next();
  griddep_wait();
  extern __shared__ float w1s[];  // [RB][rank]
  const int r0 = blockIdx.x * RB;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int k = 1; k <= a.gamma; ++k) {
    if (warp < RB && r0 + warp < a.R) {
      const int r = r0 + warp;
      const int raw = (k == 1) ? __ldg(a.x0 + r) : a.x_out[(size_t)r * a.gamma + (k - 2)];
      prepare_position_warp(a, r, k, checked_token(raw, a.V, a.status, 1), lane);
    }
    __syncthreads();
    simt_step_block<RB>(a, k, 0, r0, true, w1s);
  }
}

// One CTA per request: merge npart partials of position k; then prepare position k+1.
__global__ void __launch_bounds__(kCombineThreads) draft_combine_kernel(DraftArgs a, int k, int npart) {
  griddep_allow_next();
  griddep_wait();
  constexpr int kBatch = 4;
  __shared__ Partial red[kCombineThreads / 32];
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Stats st = stats_empty();
  // every thread's partial records are loaded before any is merged
  for (int p0 = threadIdx.x; p0 < npart; p0 += kBatch * kCombineThreads) {
    Partial rec[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int p = p0 + u * kCombineThreads;
      if (p < npart) rec[u] = a.partials[(size_t)p * a.R + r];
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (p0 + u * kCombineThreads < npart) stats_merge(st, from_partial(rec[u]));
  }
  st = warp_reduce_stats(st);
  if (lane == 0) red[warp] = to_partial(st);
  __syncthreads();
  if (warp != 0) return;
  Stats b = (lane < kCombineThreads / 32) ? from_partial(red[lane]) : stats_empty();
  b = warp_reduce_stats(b);
  const size_t row = (size_t)r * a.gamma + (k - 1);
  if (lane == 0) {
    const float lse = b.m + logf(b.s);
    a.x_out[row] = b.idx;
    a.lse_out[row] = lse;
    a.logq_out[row] = b.zsel - lse;
  }
  // Markov head: gather position k+1's factor row (the recurrent head's cell does its own)
  if (k < a.gamma && !a.rnn) prepare_position_warp(a, r, k + 1, checked_token(b.idx, a.V, a.status, 2), lane);
}

// After the last tensor-core position: one warp per (request, position) merges that
// position's partial records into x_k, lse_k and logq_k (the same merge the per-position
// combine does; the steps themselves only needed the winner).
__global__ void __launch_bounds__(256) draft_finalize_kernel(DraftArgs a, int npart) {
  griddep_allow_next();
  griddep_wait();
  constexpr int kRecs = 5;  // records per lane and batch
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= a.R * a.gamma) return;
  const int r = wid / a.gamma, k = wid % a.gamma + 1;
  const Partial* part = a.partials + (size_t)(k - 1) * npart * a.R;
  Stats st = stats_empty();
  for (int g0 = lane; g0 < npart; g0 += 32 * kRecs) {
    Partial rec[kRecs];
#pragma unroll
    for (int q = 0; q < kRecs; ++q)
      if (g0 + 32 * q < npart) rec[q] = part[(size_t)(g0 + 32 * q) * a.R + r];
#pragma unroll
    for (int q = 0; q < kRecs; ++q)
      if (g0 + 32 * q < npart) stats_merge(st, from_partial(rec[q]));
  }
  st = warp_reduce_stats(st);
  if (lane == 0) {
    const size_t row = (size_t)r * a.gamma + (k - 1);
    const float lse = st.m + logf(st.s);
    a.x_out[row] = st.idx;
    a.lse_out[row] = lse;
    a.logq_out[row] = st.zsel - lse;
  }
}

// ---------------------------------------------------------------------------------
// Host-side launchers
// ---------------------------------------------------------------------------------
cudaError_t launch_conf_hdot(const DraftArgs& a, bool reset_bounds, cudaStream_t s) {
  const int rows = a.R * a.gamma;
  const int blocks = (rows + kHdotRowsPerCta - 1) / kHdotRowsPerCta;
  return launch_pdl(conf_hdot_kernel, dim3(blocks), dim3(kHdotThreads), 0, s, rows, a.d, a.dtype_h, a.h, a.conf_w,
                    a.s_h, a.hint, a.win, reset_bounds ? rows : 0);
}

cudaError_t launch_draft_prepare(const DraftArgs& a, int k, cudaStream_t s) {
  return launch_pdl(draft_prepare_kernel, dim3(a.R), dim3(32), 0, s, a, k);
}

int simt_num_chunks(int V) {
  const int groups = (V + 3) / 4;
  const int per = kSimtGroups * kSimtThreads;
  return (groups + per - 1) / per;
}

cudaError_t launch_draft_step_simt(const DraftArgs& a, int k, cudaStream_t s) {
  dim3 grid(simt_num_chunks(a.V), (a.R + kSimtRB - 1) / kSimtRB);
  const size_t smem = sizeof(float) * kSimtRB * a.rank;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(draft_step_simt_kernel<kSimtRB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(draft_step_simt_kernel<kSimtRB>, grid, dim3(kSimtThreads), smem, s, a, k);
}

int simt_whole_round(int V) { return simt_num_chunks(V) == 1; }

cudaError_t launch_draft_round_simt(const DraftArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * kSimtRB * a.rank;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(draft_round_simt_kernel<kSimtRB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(draft_round_simt_kernel<kSimtRB>, dim3((a.R + kSimtRB - 1) / kSimtRB), dim3(kSimtThreads), smem,
                    s, a);
}

cudaError_t launch_draft_finalize(const DraftArgs& a, int npart, cudaStream_t s) {
  const int warps = a.R * a.gamma;
  return launch_pdl(draft_finalize_kernel, dim3((warps * 32 + 255) / 256), dim3(256), 0, s, a, npart);
}

cudaError_t launch_draft_combine(const DraftArgs& a, int k, int npart, cudaStream_t s) {
  return launch_pdl(draft_combine_kernel, dim3(a.R), dim3(kCombineThreads), 0, s, a, k, npart);
}

}  // namespace dspark
