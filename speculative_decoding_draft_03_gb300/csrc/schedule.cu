// schedule.cu — the confidence scheduler in one CTA.
//
// Method (DSpark 精读 §4; mkdocs.reaper.mx "3 · DSpark" §3.3; numb3r33 blog "DSpark:
// confidence-scheduled speculative decoding", sections "Scheduler objective", "Greedy
// prefix allocation", "Losslessness and non-anticipation", "Async scheduler in
// practice"; vllmbangkok §4.2.2):
//   a[r,j] = prod_{i<=j} c[r,i]; sort all (r,j) by a (desc), depth (asc), request (asc);
//   walk the sorted path with tau(n) = R + sum of the first n a's and
//   Theta(n) = tau(n) * SPS(R + n); pick n* per mode; ell_r = admitted count of r.
//
// GB300 layout: R*gamma <= 8192 candidates fit one SM's shared memory.  a is formed
// in binary64 by the same left-to-right products as the method states, so the sort
// keys (the binary64 bit patterns of a, which order like the values for a >= 0) and
// hence the admission order do not depend on rounding.  Each request's chain of a's is
// already sorted, so the global order is a merge of R sorted lists: rounds of pairwise
// merge-path merges; the scan and the mode's pick are block reductions.
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kSchedThreads = 1024;  // one CTA; R*gamma <= 8192 candidates (host-checked)
constexpr int kSchedLaunchThreads = 512;  // threads the confidence scheduler runs with

size_t schedule_smem_bytes(int R, int gamma) {
  const size_t N = (size_t)R * gamma;
  return align256(N * 8) + 2 * align256(N * 2) + align256((size_t)R * 4) + align256(sizeof(double) * 64) + 256;
}

// Shared memory (N = R*gamma <= 8192 candidates, 161 KB at most):
//   key   [N] binary64 bits of a, indexed by candidate id; after the scan the same array
//         holds the prefix sums in sorted order
//   ids   two [N] buffers of candidate ids (the merge ping-pongs between them); before the
//         sort they stage the confidences (N fp32 fill both exactly)
struct SchedSmem {
  unsigned long long* key;
  unsigned short* idA;
  unsigned short* idB;
  unsigned short* sorted;  // the buffer that holds the final order
  int* ell;                // [R]
  double* red;             // [64] reduction scratch
  int* misc;               // [8]
};

// does candidate x come before candidate y?  a desc, then id asc; the id (j-1)*R + r
// orders by depth first, then request.
__device__ __forceinline__ bool before(const SchedSmem& sm, unsigned x, unsigned y) {
  const unsigned long long kx = sm.key[x], ky = sm.key[y];
  return (kx > ky) || (kx == ky && x < y);
}

// a = prod c along each chain (binary64, left to right), keyed by candidate id.  Each
// request's chain is already in sorted order: c <= 1 makes a non-increasing in j, and
// on equal a the smaller depth comes first.  A confidence outside [0,1] (or NaN) is
// reported and clamped, which keeps the chains sorted.
__device__ void build_candidates(SchedSmem& sm, const float* conf, int R, int gamma, DeviceStatus* status) {
  const int N = R * gamma;
  float* cf = reinterpret_cast<float*>(sm.idA);  // spans idA and idB
  for (int i = threadIdx.x; i < N; i += blockDim.x) cf[i] = __ldg(conf + i);
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    double a = 1.0;
    for (int j = 1; j <= gamma; ++j) {
      float c = cf[r * gamma + (j - 1)];
      if (!(c >= 0.f && c <= 1.f)) {
        report_bad_input(status, 20);
        c = (c > 1.f) ? 1.f : 0.f;
      }
      a = __dmul_rn(a, (double)c);
      sm.key[(j - 1) * R + r] = (unsigned long long)__double_as_longlong(a);
    }
  }
  __syncthreads();
  // round-0 lists: chain r at positions [r*gamma, (r+1)*gamma)
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const int r = i / gamma, j = i % gamma;
    sm.idA[i] = (unsigned short)(j * R + r);
  }
  __syncthreads();
}

// Sorts the R chains into one list by rounds of pairwise merges (lists of gamma, 2 gamma,
// 4 gamma, ... ids).  Each thread produces a contiguous run of E = ceil(N / threads)
// outputs: a merge-path binary search finds where its run starts in the two input
// lists, then it merges E elements sequentially.  ceil(log2 R) rounds, one barrier each.
__device__ void merge_sort_chains(SchedSmem& sm, int N, int gamma) {
  unsigned short* src = sm.idA;
  unsigned short* dst = sm.idB;
  const int E = (N + blockDim.x - 1) / blockDim.x;
  for (int L = gamma; L < N; L <<= 1) {
    const int p_begin = threadIdx.x * E, p_end = min(p_begin + E, N);
    int p = p_begin;
    while (p < p_end) {
      const int m0 = (p / (2 * L)) * (2 * L);  // start of this pair
      const int a0 = m0, a_len = min(L, N - m0);
      const int b0 = m0 + a_len, b_len = max(0, min(L, N - b0));
      const int seg_end = min(p_end, m0 + a_len + b_len);
      const int d = p - m0;
      // merge path: i elements of A and d - i of B make up the first d outputs
      int lo = max(0, d - b_len), hi = min(d, a_len);
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (before(sm, src[a0 + mid], src[b0 + d - mid - 1]))
          lo = mid + 1;
        else
          hi = mid;
      }
      int i = lo, j = d - lo;
      for (; p < seg_end; ++p) {
        const bool take_a = (j >= b_len) || (i < a_len && before(sm, src[a0 + i], src[b0 + j]));
        dst[p] = take_a ? src[a0 + i++] : src[b0 + j++];
      }
    }
    __syncthreads();
    unsigned short* t = src;
    src = dst;
    dst = t;
  }
  sm.sorted = src;
}

// Inclusive prefix sums of the sorted a's, written over key[] in sorted order.  Each
// thread gathers its run (at most 8 values) into registers before any is overwritten.
constexpr int kScanPer = 16;  // 8192 candidates / 512 threads

__device__ void scan_sorted(SchedSmem& sm, int N) {
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * per;
  const int hi = min(lo + per, N);
  // binary64 arithmetic is a narrow pipe on this GPU: warps without candidates skip it
  // (per and the warp's first index are uniform, so every branch below is too)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool active = (warp * 32) * per < N;
  double v[kScanPer];
  double run = 0.0;
  double excl = 0.0;
  if (active) {
#pragma unroll
    for (int q = 0; q < kScanPer; ++q) {
      if (q >= per) break;
      v[q] = (lo + q < hi) ? __longlong_as_double((long long)sm.key[sm.sorted[lo + q]]) : 0.0;
      run += v[q];
    }
    // exclusive scan of run totals within the warp
    double incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.0;
    if (lane == 31) sm.red[warp] = incl;
  }
  __syncthreads();
  const int nactive = min((int)(blockDim.x >> 5), (N + 32 * per - 1) / (32 * per));
  if (warp == 0) {
    double w = (lane < nactive) ? sm.red[lane] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    sm.red[32 + lane] = w;  // inclusive warp-total prefix
  }
  __syncthreads();
  if (active) {
    double base = excl + (warp > 0 ? sm.red[32 + warp - 1] : 0.0);
#pragma unroll
    for (int q = 0; q < kScanPer; ++q) {
      if (q >= per) break;
      if (lo + q < hi) {
        base += v[q];
        sm.key[lo + q] = (unsigned long long)__double_as_longlong(base);
      }
    }
  }
  __syncthreads();
}

__device__ __forceinline__ double tau_at(const SchedSmem& sm, int R, int n) {
  return (double)R + (n > 0 ? __longlong_as_double((long long)sm.key[n - 1]) : 0.0);
}

// argmax_n Theta(n) over n = 0..N, smallest n on ties.
__device__ int full_search(SchedSmem& sm, int R, int N, const double* sps) {
  double best = -INFINITY;
  int bn = 0x7FFFFFFF;
  for (int n = threadIdx.x; n <= N; n += blockDim.x) {
    const double th = tau_at(sm, R, n) * __ldg(sps + R + n);
    if (th > best || (th == best && n < bn)) {
      best = th;
      bn = n;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int on = __shfl_xor_sync(0xffffffffu, bn, o);
    if (ob > best || (ob == best && on < bn)) {
      best = ob;
      bn = on;
    }
  }
  __syncthreads();
  if (lane == 0) sm.red[warp] = best;
  int* wn = reinterpret_cast<int*>(sm.red + 32);
  if (lane == 0) wn[warp] = bn;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    best = lane < nw ? sm.red[lane] : -INFINITY;
    bn = lane < nw ? wn[lane] : 0x7FFFFFFF;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int on = __shfl_xor_sync(0xffffffffu, bn, o);
      if (ob > best || (ob == best && on < bn)) {
        best = ob;
        bn = on;
      }
    }
    if (lane == 0) sm.misc[1] = bn;
  }
  __syncthreads();
  const int r = sm.misc[1];
  __syncthreads();
  return r;
}

// first n in [0,N) with Theta(n+1) <= Theta(n), else N.
__device__ int early_stop(SchedSmem& sm, int R, int N, const double* sps) {
  if (threadIdx.x == 0) sm.misc[2] = N;
  __syncthreads();
  int first = N;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    const double t0 = tau_at(sm, R, n) * __ldg(sps + R + n);
    const double t1 = tau_at(sm, R, n + 1) * __ldg(sps + R + n + 1);
    if (t1 <= t0) {
      first = n;
      break;  // n increases along the thread's stride
    }
  }
  if (first < N) atomicMin(&sm.misc[2], first);
  __syncthreads();
  const int r = sm.misc[2];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kSchedThreads, 1)
    schedule_kernel(int R, int gamma, const float* __restrict__ conf, const double* __restrict__ sps, int mode,
                    const float* __restrict__ conf_hist, int fixed_len, int32_t* __restrict__ ell_out,
                    int32_t* __restrict__ B_out, double* __restrict__ tau_out, DeviceStatus* status) {
  griddep_allow_next();
  griddep_wait();
  extern __shared__ __align__(256) unsigned char smem[];
  const int N = R * gamma;
  SchedSmem sm;
  size_t off = 0;
  sm.key = reinterpret_cast<unsigned long long*>(smem + off);
  off += align256((size_t)N * 8);
  sm.idA = reinterpret_cast<unsigned short*>(smem + off);
  off += align256((size_t)N * 2);
  sm.idB = reinterpret_cast<unsigned short*>(smem + off);
  off += align256((size_t)N * 2);
  sm.sorted = sm.idA;
  sm.ell = reinterpret_cast<int*>(smem + off);
  off += align256((size_t)R * 4);
  sm.red = reinterpret_cast<double*>(smem + off);
  off += align256(sizeof(double) * 64);
  sm.misc = reinterpret_cast<int*>(smem + off);

  for (int r = threadIdx.x; r < R; r += blockDim.x) sm.ell[r] = 0;

  if (mode == DSPARK_FIXED) {
    const int L = max(0, min(fixed_len, gamma));
    double part = 0.0;
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
      double a = 1.0, s = 0.0;
      for (int j = 1; j <= L; ++j) {
        a = __dmul_rn(a, (double)__ldg(conf + (size_t)r * gamma + (j - 1)));
        s += a;
      }
      part += s;
      ell_out[r] = L;
    }
    // block sum of the per-thread totals
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) sm.red[warp] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = (double)R;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += sm.red[w];
      *B_out = R + R * L;
      *tau_out = t;
    }
    return;
  }

  int nstar;
  if (mode == DSPARK_CAPACITY_K) {
    build_candidates(sm, conf_hist, R, gamma, status);
    merge_sort_chains(sm, N, gamma);
    scan_sorted(sm, N);
    const int K = full_search(sm, R, N, sps);
    nstar = min(K, N);
  }
  build_candidates(sm, conf, R, gamma, status);
  merge_sort_chains(sm, N, gamma);
  // admitted candidates -> per-request counts (before the scan overwrites the keys)
  if (mode == DSPARK_CAPACITY_K) {
    for (int n = threadIdx.x; n < nstar; n += blockDim.x) atomicAdd(&sm.ell[sm.sorted[n] % R], 1);
    __syncthreads();
  }
  scan_sorted(sm, N);
  if (mode == DSPARK_EARLY_STOP) {
    nstar = early_stop(sm, R, N, sps);
  } else if (mode == DSPARK_FULL_SEARCH) {
    nstar = full_search(sm, R, N, sps);
  }
  if (mode != DSPARK_CAPACITY_K) {
    for (int n = threadIdx.x; n < nstar; n += blockDim.x) atomicAdd(&sm.ell[sm.sorted[n] % R], 1);
  }
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += blockDim.x) ell_out[r] = sm.ell[r];
  if (threadIdx.x == 0) {
    *B_out = R + nstar;
    *tau_out = tau_at(sm, R, nstar);
  }
}

cudaError_t launch_schedule(int R, int gamma, const float* conf, const double* sps, int mode,
                            const float* conf_hist, int fixed_len, int32_t* ell_out, int32_t* B_out,
                            double* tau_out, DeviceStatus* status, cudaStream_t s) {
  const size_t smem = schedule_smem_bytes(R, gamma);
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // 512 threads (at most 16 candidates each, as the scan needs): half as many merge-path
  // searches per merge round as 1024 threads, against the same shared-memory traffic for
  // the merges themselves (the rounds are bound by shared-memory bank conflicts); 68 ->
  // 59 us at 7680 candidates
  const int threads = kSchedLaunchThreads;
  return launch_pdl(schedule_kernel, dim3(1), dim3(threads), smem, s, R, gamma, conf, sps, mode, conf_hist,
                    fixed_len, ell_out, B_out, tau_out, status);
}

// Fixed confidence cutoff (vllmbangkok "Verify smarter, not longer: the role of
// confidence scheduling": drafts below a fixed confidence cutoff are not verified).
// Verification needs a prefix, so request r keeps its leading drafts with c >= threshold.
// B and tau as in the other modes; a is the same left-to-right binary64 product.
__global__ void __launch_bounds__(kSchedThreads) schedule_threshold_kernel(int R, int gamma,
                                                                           const float* __restrict__ conf,
                                                                           double threshold,
                                                                           int32_t* __restrict__ ell_out,
                                                                           int32_t* __restrict__ B_out,
                                                                           double* __restrict__ tau_out) {
  griddep_allow_next();
  griddep_wait();
  __shared__ double red_t[kSchedThreads / 32];
  __shared__ long long red_b[kSchedThreads / 32];
  double part = 0.0;
  long long bsum = 0;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    double a = 1.0;
    int l = 0;
    while (l < gamma) {
      const double c = (double)__ldg(conf + (size_t)r * gamma + l);
      if (!(c >= threshold)) break;
      a = __dmul_rn(a, c);
      part += a;
      ++l;
    }
    ell_out[r] = l;
    bsum += l;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    part += __shfl_xor_sync(0xffffffffu, part, o);
    bsum += __shfl_xor_sync(0xffffffffu, bsum, o);
  }
  if (lane == 0) {
    red_t[warp] = part;
    red_b[warp] = bsum;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = (double)R;
    long long b = R;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      t += red_t[w];
      b += red_b[w];
    }
    *B_out = (int32_t)b;
    *tau_out = t;
  }
}

cudaError_t launch_schedule_threshold(int R, int gamma, const float* conf, double threshold, int32_t* ell_out,
                                      int32_t* B_out, double* tau_out, cudaStream_t s) {
  return launch_pdl(schedule_threshold_kernel, dim3(1), dim3(kSchedThreads), 0, s, R, gamma, conf, threshold, ell_out,
                    B_out, tau_out);
}

}  // namespace dspark
