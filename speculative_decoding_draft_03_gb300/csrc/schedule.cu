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
// hence the admission order do not depend on rounding.  The sort is a bitonic network
// over (key, candidate id) pairs; the scan and the mode's pick are block reductions.
#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kSchedThreads = 1024;  // one CTA; R*gamma <= 8192 candidates (host-checked)

static int next_pow2(int n) {
  int p = 2;
  while (p < n) p <<= 1;
  return p;
}

size_t schedule_smem_bytes(int R, int gamma) {
  const int npad = next_pow2(R * gamma);
  return align256((size_t)npad * 8) + align256((size_t)npad * 2) + align256((size_t)R * 4) +
         align256(sizeof(double) * 64) + 256;
}

struct SchedSmem {
  unsigned long long* key;  // [npad] binary64 bits of a (0 for padding)
  unsigned short* id;       // [npad] candidate id (j-1)*R + r (0xFFFF for padding)
  int* ell;                 // [R]
  double* red;              // [64] reduction scratch
  int* misc;                // [8]
};

// does candidate (ka, ia) come before (kb, ib)?  a desc, then id asc; the id
// (j-1)*R + r orders by depth first, then request.
__device__ __forceinline__ bool before(unsigned long long ka, unsigned ia, unsigned long long kb, unsigned ib) {
  return (ka > kb) || (ka == kb && ia < ib);
}

__device__ void bitonic_sort(SchedSmem& sm, int npad) {
  for (int k = 2; k <= npad; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int p = threadIdx.x; p < (npad >> 1); p += blockDim.x) {
        const int i = 2 * j * (p / j) + (p % j);
        const int l = i + j;
        const unsigned long long ki = sm.key[i], kl = sm.key[l];
        const unsigned ii = sm.id[i], il = sm.id[l];
        const bool up = (i & k) == 0;
        const bool swap = up ? before(kl, il, ki, ii) : before(ki, ii, kl, il);
        if (swap) {
          sm.key[i] = kl;
          sm.key[l] = ki;
          sm.id[i] = (unsigned short)il;
          sm.id[l] = (unsigned short)ii;
        }
      }
      __syncthreads();
    }
  }
}

// a = prod c along each chain, into (key, id); padding sorts last.
__device__ void build_candidates(SchedSmem& sm, const float* conf, int R, int gamma, int npad) {
  const int N = R * gamma;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    double a = 1.0;
    for (int j = 1; j <= gamma; ++j) {
      a = __dmul_rn(a, (double)__ldg(conf + (size_t)r * gamma + (j - 1)));
      const int id = (j - 1) * R + r;
      sm.key[id] = (unsigned long long)__double_as_longlong(a);
      sm.id[id] = (unsigned short)id;
    }
  }
  for (int i = N + threadIdx.x; i < npad; i += blockDim.x) {
    sm.key[i] = 0ull;
    sm.id[i] = 0xFFFFu;
  }
  __syncthreads();
}

// Inclusive prefix sums of the sorted a's, in place into key[] as binary64 bits.
// Each thread scans a contiguous run, then the run totals are scanned across the block.
__device__ void scan_sorted(SchedSmem& sm, int N) {
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * per;
  const int hi = min(lo + per, N);
  double run = 0.0;
  for (int i = lo; i < hi; ++i) run += __longlong_as_double((long long)sm.key[i]);
  // exclusive scan of run totals: warp shuffles, then the 32 warp totals
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  double excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.0;
  if (lane == 31) sm.red[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    double w = (lane < (int)(blockDim.x >> 5)) ? sm.red[lane] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    sm.red[32 + lane] = w;  // inclusive warp-total prefix
  }
  __syncthreads();
  double base = excl + (warp > 0 ? sm.red[32 + warp - 1] : 0.0);
  for (int i = lo; i < hi; ++i) {
    base += __longlong_as_double((long long)sm.key[i]);
    sm.key[i] = (unsigned long long)__double_as_longlong(base);
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
                    int32_t* __restrict__ B_out, double* __restrict__ tau_out) {
  griddep_allow_next();
  griddep_wait();
  extern __shared__ __align__(256) unsigned char smem[];
  const int N = R * gamma;
  int npad = 2;
  while (npad < N) npad <<= 1;
  SchedSmem sm;
  size_t off = 0;
  sm.key = reinterpret_cast<unsigned long long*>(smem + off);
  off += align256((size_t)npad * 8);
  sm.id = reinterpret_cast<unsigned short*>(smem + off);
  off += align256((size_t)npad * 2);
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
    build_candidates(sm, conf_hist, R, gamma, npad);
    bitonic_sort(sm, npad);
    scan_sorted(sm, N);
    const int K = full_search(sm, R, N, sps);
    nstar = min(K, N);
  }
  build_candidates(sm, conf, R, gamma, npad);
  bitonic_sort(sm, npad);
  // admitted candidates -> per-request counts (before the scan overwrites the keys)
  if (mode == DSPARK_CAPACITY_K) {
    for (int n = threadIdx.x; n < nstar; n += blockDim.x) atomicAdd(&sm.ell[sm.id[n] % R], 1);
    __syncthreads();
  }
  scan_sorted(sm, N);
  if (mode == DSPARK_EARLY_STOP) {
    nstar = early_stop(sm, R, N, sps);
  } else if (mode == DSPARK_FULL_SEARCH) {
    nstar = full_search(sm, R, N, sps);
  }
  if (mode != DSPARK_CAPACITY_K) {
    for (int n = threadIdx.x; n < nstar; n += blockDim.x) atomicAdd(&sm.ell[sm.id[n] % R], 1);
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
  (void)status;
  const size_t smem = schedule_smem_bytes(R, gamma);
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(schedule_kernel, dim3(1), dim3(kSchedThreads), smem, s, R, gamma, conf, sps, mode, conf_hist,
                    fixed_len, ell_out, B_out, tau_out);
}

}  // namespace dspark
