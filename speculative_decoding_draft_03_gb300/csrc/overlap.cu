// overlap.cu — acceptance-overlap diagnostic of a drafted block.
//
//   c*_j = sum_v min(q_j(v), p_j(v)) = 1 - ||q_j - p_j||_1 / 2
//
// for every drafted position j <= n_r of request r, with q_j = softmax((U_j +
// W1[x_{j-1}] W2)/T) the draft distribution of position j and p_j = softmax(target row
// j-1 / T) the target distribution that verifies it.  It is the probability that the
// draft token of position j is accepted given its prefix: the expectation of
// min(1, p/q) under q (numb3r33 blog "DSpark: confidence-scheduled speculative
// decoding", sections "Total variation label" and "Speculative sampling in one
// picture").  The confidence head is trained against this label; evaluating it on
// verified rounds measures how well c_j is calibrated.
//
//   overlap_plan      (tensor-core path with lengths) compact rows of the evaluated
//                     positions: an exclusive prefix over the lengths
//   overlap_prepare   CTA (flattened position, 8192-id chunk): the chunk's softmax
//                     statistics of target row j-1 / T, and the factor row W1[x_{j-1}]
//                     (the A operand of the bias contraction)
//   overlap_lse       the chunks' statistics -> lse of each position's target row
//   bias pass         the bias rows W1[x_{j-1}] W2 for all positions at once, on the
//                     tensor cores (draft_step_tc_kernel in overlap mode) or on CUDA
//                     cores (overlap_step_simt below); each CTA writes one partial sum
//                     of min(q, p) per position
//   overlap_combine   partial sums -> c*, in a fixed order (deterministic); NaN for the
//                     positions that are not evaluated
// Fused with verification (dspark_verify_overlap), the verify pass supplies the target
// rows' log-normalisers and the factor rows, and only the bias pass and the combine run.
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kOvlThreads = 256;
constexpr int kOvlChunk = 8192;  // vocabulary ids per CTA of the lse pass (4 runs of 8 per thread)

int overlap_num_chunks(int V) { return (V + kOvlChunk - 1) / kOvlChunk; }

// 8 consecutive entries of a logit row as fp32 (V % 8 == 0: the run is inside the row).
__device__ __forceinline__ void load8(const void* base, int dtype, size_t idx, float (&x)[8]) {
  if (dtype == DSPARK_F32) {
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(base) + idx);
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y); x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y); x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
  } else {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(base) + idx));
    const uint32_t wd[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = bf16_bits_to_float(wd[e] & 0xFFFFu);
      x[2 * e + 1] = bf16_bits_to_float(wd[e] >> 16);
    }
  }
}

// Verify length of request r for this diagnostic: ell[r] clamped to [0, gamma] (gamma
// without ell).  An out-of-range length is reported by overlap_prepare.
__device__ __forceinline__ int overlap_len(const OverlapArgs& a, int r) {
  if (a.ell == nullptr) return a.gamma;
  return min(max(__ldg(a.ell + r), 0), a.gamma);
}

__device__ __forceinline__ void online_add(float& m, float& s, float x) {
  if (x > m) {
    s = s * __expf(m - x) + 1.f;
    m = x;
  } else {
    s += __expf(x - m);
  }
}

// Compact rows (tensor-core path with lengths): the evaluated positions of request r are
// rows row_base[r] .. row_base[r] + n_r - 1 (row_req = r, row_t = j - 1), n_rows in all.
// One CTA: an exclusive prefix sum over the clamped lengths.
constexpr int kOvlPlanThreads = 1024;
__global__ void __launch_bounds__(kOvlPlanThreads) overlap_plan_kernel(OverlapArgs a) {
  griddep_allow_next();
  griddep_wait();
  __shared__ int wsum[32];
  const int per = (a.R + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * per, hi = min(lo + per, a.R);
  int run = 0;
  for (int r = lo; r < hi; ++r) run += overlap_len(a, r);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  int base = (incl - run) + (warp > 0 ? wsum[warp - 1] : 0);
  for (int r = lo; r < hi; ++r) {
    const int n = overlap_len(a, r);
    a.row_base[r] = base;
    for (int t = 0; t < n; ++t) {
      a.row_req[base + t] = r;
      a.row_t[base + t] = t;
    }
    base += n;
  }
  if (threadIdx.x == blockDim.x - 1) *a.n_rows = base;
}

// Row of position (r, j) in the prepared arrays: compact row, or the flattened position.
__device__ __forceinline__ size_t overlap_row(const OverlapArgs& a, int r, int j) {
  return a.row_req != nullptr ? (size_t)a.row_base[r] + (j - 1) : (size_t)r * a.gamma + (j - 1);
}

// CTA (position i, vocabulary chunk c): chunk c's (max, sum exp) of target row j-1 / T,
// and for c = 0 the position's factor row (flattened rows: zero where the position is not
// evaluated; compact rows hold only evaluated positions).
__global__ void __launch_bounds__(kOvlThreads) overlap_prepare_kernel(OverlapArgs a) {
  griddep_allow_next();
  griddep_wait();
  const int i = blockIdx.x / a.nchunk, c = blockIdx.x % a.nchunk;
  const int r = i / a.gamma, j = i % a.gamma + 1;
  if (a.ell != nullptr && j == 1 && c == 0 && threadIdx.x == 0) {
    const int l = __ldg(a.ell + r);
    if (l < 0 || l > a.gamma) report_bad_input(a.status, 31);
  }
  const bool valid = j <= overlap_len(a, r);
  if (!valid && a.row_req != nullptr) return;  // compact: no row for this position
  const size_t row = valid ? overlap_row(a, r, j) : (size_t)i;
  if (c == 0 && threadIdx.x < 32) {
    int xp = 0;
    if (valid) {
      const int raw = j == 1 ? __ldg(a.x0 + r) : __ldg(a.x + (size_t)r * a.gamma + (j - 2));
      xp = checked_token(raw, a.V, a.status, 30);
    }
    const size_t src = (size_t)xp * a.rank, dst = row * a.rank;
    if (a.dtype_w == DSPARK_F32) {
      const float* w1 = reinterpret_cast<const float*>(a.W1);
      float* g = reinterpret_cast<float*>(a.W1g);
      for (int e = threadIdx.x; e < a.rank; e += 32) g[dst + e] = valid ? __ldg(w1 + src + e) : 0.f;
    } else {
      const unsigned short* w1 = reinterpret_cast<const unsigned short*>(a.W1);
      unsigned short* g = reinterpret_cast<unsigned short*>(a.W1g);
      for (int e = threadIdx.x; e < a.rank; e += 32) g[dst + e] = valid ? __ldg(w1 + src + e) : (unsigned short)0;
    }
  }
  if (!valid) {
    if (threadIdx.x == 0) a.lse_part[row * a.nchunk + c] = make_float2(-INFINITY, 0.f);
    return;  // uniform across the CTA
  }
  const size_t trow = ((size_t)r * (a.gamma + 1) + (j - 1)) * (size_t)a.V;
  const int v0 = c * kOvlChunk, v1 = min(v0 + kOvlChunk, a.V);
  float m = -INFINITY, s = 0.f;
  if (a.V % 8 == 0) {
    // kOvlChunk / (8 * kOvlThreads) runs of 8 per thread, all loaded before use
    constexpr int kRuns = kOvlChunk / (8 * kOvlThreads);
    float x[kRuns][8];
#pragma unroll
    for (int u = 0; u < kRuns; ++u) {
      const int v = v0 + (u * kOvlThreads + threadIdx.x) * 8;
      if (v < v1) {
        load8(a.target, a.dtype_t, trow + v, x[u]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[u][e] = -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < kRuns; ++u)
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, x[u][e] * a.inv_temp);
    if (m > -INFINITY)
#pragma unroll
      for (int u = 0; u < kRuns; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) s += __expf(x[u][e] * a.inv_temp - m);
  } else {
    for (int v = v0 + threadIdx.x; v < v1; v += kOvlThreads)
      online_add(m, s, load_elem(a.target, a.dtype_t, trow + v) * a.inv_temp);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
  __shared__ float wm[kOvlThreads / 32], ws[kOvlThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    wm[warp] = m;
    ws[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < kOvlThreads / 32 ? wm[lane] : -INFINITY;
    s = lane < kOvlThreads / 32 ? ws[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_merge(m, s, m2, s2);
    }
    if (lane == 0) a.lse_part[row * a.nchunk + c] = make_float2(m, s);
  }
}

// One warp per position: lse of target row j-1 / T from the chunks (lanes take the
// chunks, merged by a fixed shuffle tree); NaN where the position is not evaluated.
__global__ void overlap_lse_kernel(OverlapArgs a) {
  griddep_allow_next();
  griddep_wait();
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= a.R * a.gamma) return;
  const int r = i / a.gamma, j = i % a.gamma + 1;
  if (j > overlap_len(a, r)) {
    if (lane == 0 && a.row_req == nullptr) a.lse_t[i] = NAN;
    return;
  }
  const size_t row = overlap_row(a, r, j);
  float m = -INFINITY, s = 0.f;
  for (int c = lane; c < a.nchunk; c += 32) {
    const float2 p = a.lse_part[row * a.nchunk + c];
    lse_merge(m, s, p.x, p.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
  if (lane == 0) a.lse_t[row] = m + logf(s);
}

// CUDA-core bias pass (fp32 weights or shapes the tensor-core path does not take).
// blockIdx.x: vocabulary chunk; blockIdx.y: block of RB flattened positions.
template <int RB>
__global__ void __launch_bounds__(kSimtThreads) overlap_step_simt_kernel(OverlapArgs a) {
  griddep_allow_next();
  griddep_wait();
  extern __shared__ float w1s[];  // [RB][rank]
  const int rows = a.R * a.gamma;
  const int i0 = blockIdx.y * RB;
  bool ok[RB];
  float lq[RB], lt[RB];
  bool any = false;
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) {
    const int i = i0 + rr;
    ok[rr] = i < rows && (i % a.gamma) + 1 <= overlap_len(a, i / a.gamma);
    lq[rr] = ok[rr] ? __ldg(a.lse_q + i) : 0.f;
    lt[rr] = ok[rr] ? a.lse_t[i] : 0.f;
    any |= ok[rr];
  }
  if (!any) {
    if (threadIdx.x < RB && i0 + (int)threadIdx.x < rows) a.part[(size_t)blockIdx.x * rows + i0 + threadIdx.x] = 0.f;
    return;
  }
  for (int e = threadIdx.x; e < RB * a.rank; e += blockDim.x) {
    const int rr = e / a.rank, c = e % a.rank;
    w1s[e] = ok[rr] ? load_elem(a.W1g, a.dtype_w, (size_t)(i0 + rr) * a.rank + c) : 0.f;
  }
  __syncthreads();
  float sum[RB];
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) sum[rr] = 0.f;
  const int groups_total = (a.V + 3) / 4;
  const int g0 = blockIdx.x * kSimtGroups * blockDim.x;
  for (int t = 0; t < kSimtGroups; ++t) {
    const int g = g0 + t * blockDim.x + threadIdx.x;
    if (g >= groups_total) break;
    float acc[RB][4];
#pragma unroll
    for (int rr = 0; rr < RB; ++rr)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rr][e] = 0.f;
    for (int k = 0; k < a.rank; ++k) {
      float w2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = 4 * g + e;
        w2[e] = (v < a.V) ? load_elem(a.W2, a.dtype_w, (size_t)k * a.V + v) : 0.f;
      }
#pragma unroll
      for (int rr = 0; rr < RB; ++rr) {
        const float w1 = w1s[rr * a.rank + k];
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[rr][e] = fmaf(w1, w2[e], acc[rr][e]);
      }
    }
#pragma unroll
    for (int rr = 0; rr < RB; ++rr) {
      if (!ok[rr]) continue;
      const int i = i0 + rr;
      const int r = i / a.gamma, j = i % a.gamma + 1;
      const size_t urow = (size_t)i * a.V;
      const size_t trow = ((size_t)r * (a.gamma + 1) + (j - 1)) * (size_t)a.V;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = 4 * g + e;
        if (v >= a.V) break;
        const float z = (load_elem(a.U, a.dtype_u, urow + v) + acc[rr][e]) * a.inv_temp;
        const float lp = load_elem(a.target, a.dtype_t, trow + v) * a.inv_temp - lt[rr];
        sum[rr] += fminf(__expf(lp), __expf(z - lq[rr]));
      }
    }
  }
  // block sums per position, added in a fixed order
  __shared__ float red[kSimtThreads / 32][RB];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum[rr] += __shfl_xor_sync(0xffffffffu, sum[rr], o);
    if (lane == 0) red[warp][rr] = sum[rr];
  }
  __syncthreads();
  if (threadIdx.x < RB && i0 + (int)threadIdx.x < rows) {
    float t = 0.f;
    for (int w = 0; w < kSimtThreads / 32; ++w) t += red[w][threadIdx.x];
    a.part[(size_t)blockIdx.x * rows + i0 + threadIdx.x] = t;
  }
}

// One warp per flattened position: c* = sum of the npart partial sums.
__global__ void overlap_combine_kernel(OverlapArgs a, int npart) {
  griddep_allow_next();
  griddep_wait();
  const int rows = a.R * a.gamma;
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= rows) return;
  const bool ok = (i % a.gamma) + 1 <= overlap_len(a, i / a.gamma);
  float t = 0.f;
  if (ok)
    for (int q = lane; q < npart; q += 32) t += a.part[(size_t)q * rows + i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if (lane == 0) a.out[i] = ok ? t : NAN;
}

// Compact rows (fused with verification): one warp per flattened position (r, j), the
// partial sums of compact row row_base[r] + j - 1 over the vocabulary groups the bias pass
// used.  The pass derived its request blocks and groups from the row count exactly as
// here: blocks of rb_rows rows, grid / blocks groups.
__global__ void overlap_combine_compact_kernel(OverlapArgs a, int rb_rows, int grid) {
  griddep_allow_next();
  griddep_wait();
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= a.R * a.gamma) return;
  const int r = i / a.gamma, j = i % a.gamma + 1;
  const bool ok = j <= overlap_len(a, r);
  const int n = max(*a.n_rows, 0);
  const int blocks = (n + rb_rows - 1) / rb_rows;
  const int groups = blocks > 0 ? max(1, grid / blocks) : 0;
  const size_t q = (size_t)a.row_base[r] + (j - 1);
  float t = 0.f;
  if (ok && q < (size_t)n)
    for (int g = lane; g < groups; g += 32) t += a.part[(size_t)g * a.rows_max + q];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if (lane == 0) a.out[i] = ok ? t : NAN;
}

int tc_compact_ok(int R) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 148;
  const int Rb = tc_block_rows(R);
  return (R + Rb - 1) / Rb <= sms;
}

int overlap_num_partials(int R, int gamma, int V, int rank, int dtype_w) {
  const int simt = simt_num_chunks(V);
  if (!tc_supported(V, rank, dtype_w)) return simt;
  const int tc = tc_num_partials(R * gamma);
  return simt > tc ? simt : tc;
}

cudaError_t launch_overlap(const OverlapArgs& a, cudaStream_t s) {
  const int rows = a.R * a.gamma;
  cudaError_t e;
  if (a.row_req != nullptr &&
      (e = launch_pdl(overlap_plan_kernel, dim3(1), dim3(kOvlPlanThreads), 0, s, a)) != cudaSuccess)
    return e;
  e = launch_pdl(overlap_prepare_kernel, dim3((unsigned)((size_t)rows * a.nchunk)), dim3(kOvlThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  if ((e = launch_pdl(overlap_lse_kernel, dim3((unsigned)(((size_t)rows * 32 + 255) / 256)), dim3(256), 0, s, a)) !=
      cudaSuccess)
    return e;
  return launch_overlap_pass(a, s);
}

cudaError_t launch_overlap_pass(const OverlapArgs& a, cudaStream_t s) {
  const int rows = a.R * a.gamma;
  cudaError_t e;
  if (a.row_req != nullptr) {
    // compact rows (tensor-core path only)
    if (!tc_supported(a.V, a.rank, a.dtype_w) || tc_grid_ctas(a.rows_max) > a.npart) return cudaErrorInvalidValue;
    if ((e = launch_overlap_tc(a, s)) != cudaSuccess) return e;
    return launch_pdl(overlap_combine_compact_kernel, dim3((rows * 32 + 255) / 256), dim3(256), 0, s, a,
                      tc_block_rows(a.rows_max), tc_grid_ctas(a.rows_max));
  }
  int npart;
  if (tc_supported(a.V, a.rank, a.dtype_w)) {
    if ((e = launch_overlap_tc(a, s)) != cudaSuccess) return e;
    npart = tc_num_partials(rows);
  } else {
    dim3 grid(simt_num_chunks(a.V), (rows + kSimtRB - 1) / kSimtRB);
    const size_t smem = sizeof(float) * kSimtRB * a.rank;
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(overlap_step_simt_kernel<kSimtRB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e != cudaSuccess) return e;
    }
    if ((e = launch_pdl(overlap_step_simt_kernel<kSimtRB>, grid, dim3(kSimtThreads), smem, s, a)) != cudaSuccess)
      return e;
    npart = (int)grid.x;
  }
  if (npart > a.npart) return cudaErrorInvalidValue;
  return launch_pdl(overlap_combine_kernel, dim3((rows * 32 + 255) / 256), dim3(256), 0, s, a, npart);
}

}  // namespace dspark
