// sts.cu — sequential temperature scaling (STS) of the confidence head on held-out data.
//
// Each position k gets its own temperature, c_k = sigmoid(z_k / T_k), fitted left to
// right: position 1 first, then, with T_1 frozen, the cumulative survival through
// position 2, and so on (numb3r33 blog "DSpark: confidence-scheduled speculative
// decoding", section "Sequential temperature scaling"; mkdocs.reaper.mx "3 · DSpark"
// §3.2: a per-position temperature search minimising the expected calibration error of
// the cumulative product prod_{i<=k} c_i on held-out data).
//
// For held-out sample n (confidence logits z[n,1..gamma], accepted drafts L_n when the
// whole block was verified) and candidate T of the grid, the prediction at position k is
//   p_n = prod_{i<k} sigmoid(z[n,i] / T_i) * sigmoid(z[n,k] / T),  outcome o_n = 1[L_n >= k],
// and ECE(T) = sum_b |sum_{n in bin b} (p_n - o_n)| / N over M equal-width bins of
// [0, 1].  T_k is the grid point with the smallest ECE (the first one on ties).
//
//   sts_prepare   z -> position-major copy (coalesced reads per position)
//   sts_eval      CTA (4 candidates, chunk of 4096 samples): per-bin sums of p - o
//   sts_ece       warp per candidate: ECE (chunk sums in fp32, bins added in binary64)
//   sts_update    argmin over the candidates (every CTA), T_k recorded, and
//                 prefix[n] *= sigmoid(z[n,k] / T_k) for the next position
// All sums run in a fixed order, so the fit is deterministic.
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kStsThreads = 128;
constexpr int kStsPerThread = 32;
constexpr int kStsChunk = kStsThreads * kStsPerThread;
constexpr int kStsCands = 4;  // candidates per CTA: each sample is loaded once for all four

int sts_num_chunks(int N) { return (N + kStsChunk - 1) / kStsChunk; }

__device__ __forceinline__ float sts_sigmoid(float x) { return 1.f / (1.f + expf(-x)); }

__global__ void sts_prepare_kernel(StsArgs a) {
  griddep_allow_next();
  griddep_wait();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)a.N * a.gamma) return;
  const int n = (int)(i / a.gamma), k = (int)(i % a.gamma);
  a.zt[(size_t)k * a.N + n] = __ldg(a.z + i);
}

// CTA (group of kStsCands candidates, chunk of kStsChunk samples): per candidate and bin,
// the sum of p - o over the chunk.  The sigmoid here takes the fast exponential and
// reciprocal (a few units of 1e-7 relative): that moves a prediction across a bin edge
// only when it lies within that distance of the edge.
__global__ void __launch_bounds__(kStsThreads) sts_eval_kernel(StsArgs a, int k) {
  griddep_allow_next();
  griddep_wait();
  const int g0 = blockIdx.x * kStsCands, s = blockIdx.y;
  float inv[kStsCands];
  bool ok[kStsCands];
#pragma unroll
  for (int c = 0; c < kStsCands; ++c) {
    const int g = g0 + c;
    const float T = g < a.G ? __ldg(a.grid + g) : 1.f;
    ok[c] = g < a.G && T > 0.f && isfinite(T);
    if (g < a.G && !ok[c] && threadIdx.x == 0 && s == 0) report_bad_input(a.status, 40);
    inv[c] = ok[c] ? 1.f / T : 0.f;
  }
  const float* zk = a.zt + (size_t)(k - 1) * a.N;
  // thread-private bin sums in shared memory ([candidate][bin][thread]: no two lanes of a
  // warp share a bank), then per bin a fixed-order sum over the threads
  __shared__ float gap[kStsCands][kStsMaxBins][kStsThreads];
#pragma unroll
  for (int c = 0; c < kStsCands; ++c)
#pragma unroll
    for (int b = 0; b < kStsMaxBins; ++b) gap[c][b][threadIdx.x] = 0.f;
  const float fM = (float)a.M;
  // kStsBatch samples per step: their loads are issued before any is used
  constexpr int kStsBatch = 8;
  for (int u0 = 0; u0 < kStsPerThread; u0 += kStsBatch) {
    float pre[kStsBatch], zn[kStsBatch], o[kStsBatch];
    bool in[kStsBatch];
#pragma unroll
    for (int u = 0; u < kStsBatch; ++u) {
      const int n = s * kStsChunk + (u0 + u) * kStsThreads + threadIdx.x;
      in[u] = n < a.N;
      pre[u] = (k == 1 || !in[u]) ? 1.f : a.prefix[n];
      zn[u] = in[u] ? zk[n] : 0.f;
      o[u] = (in[u] && __ldg(a.acc_len + n) >= k) ? 1.f : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kStsBatch; ++u) {
      if (!in[u]) continue;
#pragma unroll
      for (int c = 0; c < kStsCands; ++c) {
        const float p = pre[u] * __frcp_rn(1.f + __expf(-zn[u] * inv[c]));
        const int bin = min((int)(p * fM), a.M - 1);
        gap[c][bin][threadIdx.x] += p - o[u];
      }
    }
  }
  __shared__ float red[kStsCands][kStsThreads / 32][kStsMaxBins];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int c = 0; c < kStsCands; ++c)
    for (int b = 0; b < a.M; ++b) {
      float v = gap[c][b][threadIdx.x];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[c][warp][b] = v;
    }
  __syncthreads();
  for (int i = threadIdx.x; i < kStsCands * a.M; i += kStsThreads) {
    const int c = i / a.M, b = i % a.M;
    const int g = g0 + c;
    if (g >= a.G) continue;
    float v = 0.f;
    for (int w = 0; w < kStsThreads / 32; ++w) v += red[c][w][b];
    a.part[((size_t)g * a.S + s) * a.M + b] = ok[c] ? v : 0.f;
  }
}

// One warp per candidate: ECE = sum over bins of |sum over chunks of the bin sums| / N.
// Lanes take the chunks (fp32), the lane sums are added by a fixed shuffle tree, and the
// bins are added in binary64.
__global__ void __launch_bounds__(kStsThreads) sts_ece_kernel(StsArgs a) {
  griddep_allow_next();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x * (kStsThreads / 32) + (threadIdx.x >> 5);
  if (g >= a.G) return;
  const float T = __ldg(a.grid + g);
  float v[kStsMaxBins];
#pragma unroll
  for (int b = 0; b < kStsMaxBins; ++b) v[b] = 0.f;
  for (int s = lane; s < a.S; s += 32) {
    const float* pp = a.part + ((size_t)g * a.S + s) * a.M;
#pragma unroll
    for (int b = 0; b < kStsMaxBins; ++b)
      if (b < a.M) v[b] += pp[b];
  }
  double e = 0.0;
#pragma unroll
  for (int b = 0; b < kStsMaxBins; ++b) {
    float x = v[b];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    e += fabs((double)x);
  }
  if (lane == 0) a.ece_g[g] = (T > 0.f && isfinite(T)) ? e / (double)a.N : INFINITY;
}

// Every CTA picks the candidate with the smallest ECE (the first on ties); CTA 0 records
// T_k and its ECE; with `advance`, the CTAs then fold sigmoid(z_k / T_k) into the prefix.
__global__ void __launch_bounds__(kStsThreads) sts_update_kernel(StsArgs a, int k, int advance) {
  griddep_allow_next();
  griddep_wait();
  double best = INFINITY;
  int best_g = 0x7fffffff;
  for (int g = threadIdx.x; g < a.G; g += kStsThreads) {
    const double e = a.ece_g[g];
    if (e < best) {  // g ascends within the thread: the first minimum stays
      best = e;
      best_g = g;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double e2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int g2 = __shfl_xor_sync(0xffffffffu, best_g, o);
    if (e2 < best || (e2 == best && g2 < best_g)) {
      best = e2;
      best_g = g2;
    }
  }
  __shared__ double we[kStsThreads / 32];
  __shared__ int wg[kStsThreads / 32];
  __shared__ float t_sel;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    we[warp] = best;
    wg[warp] = best_g;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kStsThreads / 32; ++w)
      if (we[w] < best || (we[w] == best && wg[w] < best_g)) {
        best = we[w];
        best_g = wg[w];
      }
    const bool found = best_g != 0x7fffffff;  // at least one usable candidate
    t_sel = found ? __ldg(a.grid + best_g) : NAN;
    if (blockIdx.x == 0) {
      a.T_out[k - 1] = t_sel;
      a.ece_out[k - 1] = found ? (float)best : NAN;
    }
  }
  __syncthreads();
  if (!advance) return;
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= a.N) return;
  const float pre = k == 1 ? 1.f : a.prefix[n];
  a.prefix[n] = pre * sts_sigmoid(a.zt[(size_t)(k - 1) * a.N + n] / t_sel);
}

cudaError_t launch_sts_fit(const StsArgs& a, cudaStream_t s) {
  const size_t nz = (size_t)a.N * a.gamma;
  cudaError_t e = launch_pdl(sts_prepare_kernel, dim3((unsigned)((nz + 255) / 256)), dim3(256), 0, s, a);
  if (e != cudaSuccess) return e;
  const int warps = kStsThreads / 32;
  for (int k = 1; k <= a.gamma; ++k) {
    const dim3 grid_eval((a.G + kStsCands - 1) / kStsCands, a.S);
    if ((e = launch_pdl(sts_eval_kernel, grid_eval, dim3(kStsThreads), 0, s, a, k)) != cudaSuccess) return e;
    if ((e = launch_pdl(sts_ece_kernel, dim3((a.G + warps - 1) / warps), dim3(kStsThreads), 0, s, a)) != cudaSuccess)
      return e;
    const bool advance = k < a.gamma;
    const int blocks = advance ? (a.N + kStsThreads - 1) / kStsThreads : 1;
    if ((e = launch_pdl(sts_update_kernel, dim3(blocks), dim3(kStsThreads), 0, s, a, k, advance ? 1 : 0)) !=
        cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

}  // namespace dspark
