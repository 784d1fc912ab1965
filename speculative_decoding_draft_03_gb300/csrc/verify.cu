// verify.cu — exact speculative-sampling verification.
//
// Method (numb3r33 blog "DSpark: confidence-scheduled speculative decoding", sections
// "One-token exactness", "Why only the longest accepted prefix survives", "Prefix
// survival and accepted length"):
//   accept x_j with probability min(1, p(x_j)/q(x_j)), stop at the first rejection,
//   resample that position from (p - q)+ normalised, or emit a bonus token from the
//   next target row when every verified draft survives.
//
// Kernels (one round, stream-ordered, no host synchronisation):
//   verify_plan      ell -> compact list of the target rows that must be read:
//                    rows 0..ell_r of request r (sum_r (ell_r + 1) rows)
//   verify_rows      streams those rows once, coalesced and vectorised, per (row,
//                    vocabulary chunk) item taken from a work queue: for rows
//                    0..ell_r - 1 the (max, sum exp) of t/T (their log-normalisers, which
//                    the acceptance tests need); for row ell_r the bonus draw's
//                    Gumbel-max of t/T + g (stream 2 at position ell_r + 1), which needs
//                    no normaliser
//   verify_accept    per request: row log-normalisers, the acceptance scan; every
//                    verified draft accepted -> the bonus token (merged from row ell_r's
//                    race); a rejection at j* = n_acc + 1 -> a compact slot for the
//                    correction pass, with the factor row of position j*
//   residual_step    per rejected request: recompute the draft logits of position j*
//                    (U + W1[x_{j*-1}] W2), q = exp(z - lse_q), p = exp(t/T - lse_t) from
//                    target row n_acc, Gumbel-max of ln(p - q)+ (and of ln p, the rounding
//                    fallback), stream 2 at position j*
//   residual_combine merges the correction partials into the emitted token.
#include <climits>

#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {

constexpr int kPlanThreads = 1024;
constexpr int kRowThreads = 256;
constexpr int kRowCtasPerSm = 4;  // resident row-pass CTAs per SM (the grid is that many per SM)

// verify length of request r, clamped to [0,gamma] (out-of-range values are reported)
__device__ __forceinline__ int clamp_ell(const VerifyArgs& a, int r) {
  const int l = __ldg(a.ell + r);
  if (l < 0 || l > a.gamma) {
    report_bad_input(a.status, 10);
    return l < 0 ? 0 : a.gamma;
  }
  return l;
}

__global__ void __launch_bounds__(kPlanThreads) verify_plan_kernel(VerifyArgs a) {
  griddep_allow_next();
  griddep_wait();
  __shared__ int wsum[32];
  const int per = (a.R + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * per, hi = min(lo + per, a.R);
  int run = 0;
  for (int r = lo; r < hi; ++r) run += clamp_ell(a, r) + 1;
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
    const int n = clamp_ell(a, r) + 1;
    a.row_base[r] = base;
    for (int t = 0; t < n; ++t) {
      a.row_req[base + t] = r;
      a.row_t[base + t] = t;
    }
    // processing order: row t = ell of every request first (the bonus draw's race, the
    // longest items), then rows 0..ell-1
    a.row_order[r] = base + n - 1;
    for (int t = 0; t + 1 < n; ++t) a.row_order[a.R + (base - r) + t] = base + t;
    a.jstar[r] = 0;
    base += n;
  }
  if (threadIdx.x == blockDim.x - 1) *a.n_rows = base;
  if (threadIdx.x == 0) {
    *a.work_next = 0;
    *a.n_rej = 0;
    *a.n_fb = 0;
  }
}

// Per (row, chunk): (max, sum exp) of t/T.  Every thread keeps its kRowPer ids in
// registers, so the chunk's maximum M is known before any exponential.
constexpr int kRowPer = 32;

__device__ __forceinline__ float block_max(float v, float* sm) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = sm[0];
#pragma unroll
  for (int w = 1; w < kRowThreads / 32; ++w) r = fmaxf(r, sm[w]);
  __syncthreads();
  return r;
}

// The bonus draw's race over one chunk of target row t = ell of request r: the Gumbel-max
// of t/T + g with g from stream 2 at position ell + 1 (the normaliser of that row is a
// constant shift of every key, so it is not needed).  z holds the thread's kRowPer logits
// (already divided by T; -inf past the row), thread ids v0 + (threadIdx.x + i kRowThreads)
// EPV + e for vector i, element e; m is their maximum.  Each thread keys its largest logit
// first; the warp's best such key (an actual element's key) bounds every lane's race, so
// ids are rejected without logarithms when 1 - u >= exp(z - best) (the conversion-free
// form of the draft step), and only survivors evaluate their key.  The chunk's winner is
// written as a partial record (key, id) of the row.
template <int EPV>
__device__ __forceinline__ void bonus_race(const VerifyArgs& a, const float (&z)[kRowPer], float m, int r, int t,
                                           int v0, int row, int c, Partial* sm_red) {
  constexpr int NV = kRowPer / EPV;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const PhiloxRowWords prow =
      philox_row_words(rng_row(a.seed, __ldg(a.req_id + r), a.round, kStreamCorrect, (uint32_t)(t + 1)));
  auto id_of = [&](int k) { return v0 + (threadIdx.x + (k / EPV) * kRowThreads) * EPV + (k % EPV); };
  Stats own = stats_empty();
  if (m > -INFINITY) {
    int km = 0;
#pragma unroll
    for (int k = kRowPer - 1; k >= 0; --k)
      if (z[k] == m) km = k;  // the lowest id among equal maxima
    const int vm = id_of(km);
    const Philox4 b = prow.block((uint32_t)(vm >> 2), a.keys);
    const uint32_t w = (vm & 3) == 0 ? b.x : ((vm & 3) == 1 ? b.y : ((vm & 3) == 2 ? b.z : b.w));
    own.key = m + gumbel_fast_from_bits(w);
    own.idx = vm;
  }
  float thr = own.key;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) thr = fmaxf(thr, __shfl_xor_sync(0xffffffffu, thr, o));
  if (m > -INFINITY && thr > -INFINITY) {
    constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
#pragma unroll
      for (int g4 = 0; g4 < EPV / 4; ++g4) {
        const int k0 = i * EPV + 4 * g4;
        const float gm = fmaxf(fmaxf(z[k0], z[k0 + 1]), fmaxf(z[k0 + 2], z[k0 + 3]));
        if (gm + kGumbelMax < thr) continue;  // no id of the group can reach the bound
        const int vb = id_of(k0);
        const Philox4 b = prow.block((uint32_t)(vb >> 2), a.keys);
        const uint32_t wd[4] = {b.x, b.y, b.z, b.w};
        const float s = -thr * kLog2e;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // 1 - u >= exp(z - best) rejects; v > edge marks the ids that may beat it
          const float term = exp2f_approx(fmaf(z[k0 + e], kLog2e, s)) * kRejectSlack;
          if (!(fmaf(term, 1.f, uniform_mantissa(wd[e])) > kRejectEdge)) continue;
          if (vb + e == own.idx) continue;  // keyed above
          const float key = z[k0 + e] + gumbel_fast_from_bits(wd[e]);
          if (key_better(key, vb + e, own.key, own.idx)) {
            own.key = key;
            own.idx = vb + e;
            thr = fmaxf(thr, key);
          }
        }
      }
    }
  }
  own = warp_reduce_stats(own);
  if (lane == 0) sm_red[warp] = to_partial(own);
  __syncthreads();
  if (threadIdx.x == 0) {
    Stats b = from_partial(sm_red[0]);
#pragma unroll
    for (int w2 = 1; w2 < kRowThreads / 32; ++w2) stats_merge(b, from_partial(sm_red[w2]));
    b.m = -INFINITY;
    b.s = 0.f;
    a.row_part[(size_t)row * a.nchunk + c] = to_partial(b);
  }
  __syncthreads();
}

// Work items are (row position, chunk) pairs taken from a queue in row_order.  Per item
// the CTA needs the chunk maximum M (block max; every thread then sums exp(z - M) against
// the same M, so the partial sums add without rescaling).  The next item's index is taken
// from the queue while the current one is processed, so the atomic's round trip is off
// the critical path.
template <int DT>
__global__ void __launch_bounds__(kRowThreads, kRowCtasPerSm) verify_rows_kernel(VerifyArgs a) {
  griddep_allow_next();
  griddep_wait();
  constexpr int EPV = DT == DSPARK_F32 ? 4 : 8;  // ids per 16-byte vector
  constexpr int NV = kRowPer / EPV;              // vectors per thread per item
  constexpr int kWarps = kRowThreads / 32;
  __shared__ float sm_f[kWarps];
  __shared__ Partial sm_red[kWarps];
  __shared__ int item_s[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_items = (*a.n_rows) * a.nchunk;
  const bool vec_ok = (a.V % EPV) == 0 && (reinterpret_cast<uintptr_t>(a.target) & 15u) == 0;
  if (threadIdx.x == 0) item_s[0] = atomicAdd(a.work_next, 1);
  __syncthreads();
  // every item ends with a block barrier, after which item_s[cur] holds the next index
  for (int cur = 0;; cur ^= 1) {
    const int item = item_s[cur];
    if (item >= n_items) break;
    if (threadIdx.x == 0) item_s[cur ^ 1] = atomicAdd(a.work_next, 1);
    const int pos = item / a.nchunk, c = item % a.nchunk;
    const int row = a.row_order[pos];
    const int r = a.row_req[row], t = a.row_t[row];
    const size_t rbase = target_row_index(a.t_off, a.n_trows, a.gamma, r, t, a.status) * a.V;
    const int v0 = c * a.chunk, v1 = min(v0 + a.chunk, a.V);
    // thread's ids: vector i covers v0 + (threadIdx.x + i*kRowThreads)*EPV + [0, EPV)
    float z[kRowPer];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int vb = v0 + (threadIdx.x + i * kRowThreads) * EPV;
      if (vec_ok && vb + EPV <= v1) {
        if constexpr (DT == DSPARK_F32) {
          const float4 q = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.target) + rbase + vb));
          z[i * 4 + 0] = q.x;
          z[i * 4 + 1] = q.y;
          z[i * 4 + 2] = q.z;
          z[i * 4 + 3] = q.w;
        } else {
          const uint4 q =
              __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(a.target) + rbase + vb));
          const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            z[i * 8 + 2 * e] = bf16_bits_to_float(wd[e] & 0xFFFFu);
            z[i * 8 + 2 * e + 1] = bf16_bits_to_float(wd[e] >> 16);
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) z[i * EPV + e] = (vb + e < v1) ? load_elem(a.target, DT, rbase + vb + e) : -INFINITY;
      }
    }
    if (pos < a.R) {
      // row ell of request r (the first R processing positions): the bonus draw's race
      float m = -INFINITY;
#pragma unroll
      for (int k = 0; k < kRowPer; ++k) {
        z[k] *= a.inv_temp;
        m = fmaxf(m, z[k]);
      }
      bonus_race<EPV>(a, z, m, r, t, v0, row, c, sm_red);
      continue;
    }
    // statistics in base 2: y = t log2(e) / T, two ids per packed instruction; each term
    // 2^(y - M) is one ex2, and the chunk maximum goes back to natural units once
    constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
    const float ys = a.inv_temp * kLog2e;
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < kRowPer; k += 2) {
      mul2f(z[k], z[k + 1], ys, ys);
      m = max3f_(m, z[k], z[k + 1]);
    }
    const float M2 = block_max(m, sm_f);
    const float M = M2 * kLn2;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int k = 0; k < kRowPer; k += 2) {
      sub2f(z[k], z[k + 1], M2, M2);
      z[k] = exp2f_approx(z[k]);
      z[k + 1] = exp2f_approx(z[k + 1]);
      add2f(s0, s1, z[k], z[k + 1]);
    }
    float ssum = s0 + s1;
    // sum of exp(z - M) (one common M: no rescaling): warp reductions, then the warps in
    // a fixed order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    if (lane == 0) sm_f[warp] = ssum;
    __syncthreads();
    if (threadIdx.x == 0) {
      Partial out;
      out.m = M;
      out.s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) out.s += sm_f[w];
      out.key = -INFINITY;
      out.zsel = 0.f;
      out.idx = -1;
      out.pad0 = out.pad1 = out.pad2 = 0;
      a.row_part[(size_t)row * a.nchunk + c] = out;
    }
    __syncthreads();
  }
}

// One warp per request.  Row t = lane + 32 s (s = 0..2, gamma <= 64) is owned by one
// lane: its log-normaliser comes from a warp reduction over the row's
// chunk partials, then every verified draft j = t+1 is tested by its own lane (all loads
// of the request are issued together), and a ballot finds the first rejection.
constexpr int kRowSlots = 3;  // rows per lane: (gamma + 1) <= 96

__global__ void verify_accept_kernel(VerifyArgs a) {
  griddep_allow_next();
  griddep_wait();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= a.R) return;
  const int ell = clamp_ell(a, r);
  const int base = a.row_base[r];
  const int nch = a.nchunk;
  float lse_own[kRowSlots];
#pragma unroll
  for (int s = 0; s < kRowSlots; ++s) lse_own[s] = 0.f;
  // rows 0..ell-1 (log-normalisers), eight at a time, and row ell (the bonus race), all
  // merged the same way: each lane merges chunks lane, lane+32, ... of each row
  int bonus_id = -1;
  for (int t0 = 0; t0 <= ell; t0 += 8) {
    Stats acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = stats_empty();
    for (int c = lane; c < nch; c += 32) {
      Partial rec[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (t0 + q <= ell) rec[q] = a.row_part[(size_t)(base + t0 + q) * nch + c];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (t0 + q <= ell) stats_merge(acc[q], from_partial(rec[q]));
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int t = t0 + q;
      if (t > ell) break;  // uniform across the warp
      if (t == ell) {
        bonus_id = warp_reduce_stats(acc[q]).idx;
        break;
      }
      const Stats st = warp_reduce_stats(acc[q]);
#pragma unroll
      for (int s = 0; s < kRowSlots; ++s)
        if (t == lane + 32 * s) lse_own[s] = st.m + logf(st.s);
    }
  }
  // acceptance test of draft j+1 (lane-owned row j < ell) against target row j
  uint32_t rej[kRowSlots];
  const RngRow acc_rng = rng_row(a.seed, __ldg(a.req_id + r), a.round, kStreamAccept, 0u);
#pragma unroll
  for (int s = 0; s < kRowSlots; ++s) {
    const int j = lane + 32 * s;
    bool reject = false;
    if (j < ell) {
      const int xj = checked_token(__ldg(a.x + (size_t)r * a.gamma + j), a.V, a.status, 11);
      const float tx =
          load_elem(a.target, a.dtype_t, target_row_index(a.t_off, a.n_trows, a.gamma, r, j, a.status) * a.V + xj) *
          a.inv_temp;
      const double lp = (double)tx - (double)lse_own[s];
      const double ratio = exp(lp - (double)__ldg(a.logq + (size_t)r * a.gamma + j));
      RngRow rr = acc_rng;
      rr.c2 = (kStreamAccept << 24) | (uint32_t)(j + 1);
      const double u = uniform_from_bits_f64(rng_chunk(rr, 0u).x);
      reject = !(u < ratio);
    }
    rej[s] = __ballot_sync(0xffffffffu, reject);
  }
  int n_acc = ell;
#pragma unroll
  for (int s = kRowSlots - 1; s >= 0; --s)
    if (rej[s]) n_acc = 32 * s + __ffs(rej[s]) - 1;
  // the row that decides the correction draw: row n_acc (its log-normaliser)
  const int src_lane = n_acc & 31, src_slot = n_acc >> 5;
  float lse_stop = 0.f;
#pragma unroll
  for (int s = 0; s < kRowSlots; ++s) {
    const float l = __shfl_sync(0xffffffffu, lse_own[s], src_lane);
    if (s == src_slot) lse_stop = l;
  }
  const size_t orow = (size_t)r * (a.gamma + 1);
  for (int j = lane; j <= a.gamma; j += 32) {
    if (j < n_acc) a.tokens_out[orow + j] = __ldg(a.x + (size_t)r * a.gamma + j);
    else if (j > n_acc) a.tokens_out[orow + j] = -1;
  }
  if (lane == 0) {
    a.n_acc_out[r] = n_acc;
    a.n_out[r] = n_acc + 1;
  }
  // fused acceptance overlap: target row j's log-normaliser for position j + 1 (j < ell),
  // and the factor row W1[x_{j-1}] of every verified position j; in the compact row order
  // (row base + j - 1) for the tensor-core pass, else at the flattened position (NaN and
  // zero rows beyond ell)
  if (a.ovl_lse != nullptr) {
    const size_t obase = a.ovl_compact ? (size_t)base : (size_t)r * a.gamma;
#pragma unroll
    for (int s = 0; s < kRowSlots; ++s) {
      const int j = lane + 32 * s;
      if (j < ell)
        a.ovl_lse[obase + j] = lse_own[s];
      else if (!a.ovl_compact && j < a.gamma)
        a.ovl_lse[obase + j] = NAN;
    }
    const int jmax = a.ovl_compact ? ell : a.gamma;
    for (int j = 1; j <= jmax; ++j) {
      const bool on = j <= ell;
      int xp = 0;
      if (on)
        xp = checked_token((j == 1) ? __ldg(a.x0 + r) : __ldg(a.x + (size_t)r * a.gamma + (j - 2)), a.V, a.status, 13);
      const size_t src = (size_t)xp * a.rank, dst = (obase + (j - 1)) * a.rank;
      if (a.dtype_w == DSPARK_BF16) {
        const unsigned short* w1 = reinterpret_cast<const unsigned short*>(a.W1);
        unsigned short* g = reinterpret_cast<unsigned short*>(a.ovl_W1g);
        for (int i = lane; i < a.rank; i += 32) g[dst + i] = on ? __ldg(w1 + src + i) : (unsigned short)0;
      } else {
        const float* w1 = reinterpret_cast<const float*>(a.W1);
        float* g = reinterpret_cast<float*>(a.ovl_W1g);
        for (int i = lane; i < a.rank; i += 32) g[dst + i] = on ? __ldg(w1 + src + i) : 0.f;
      }
    }
  }
  // every verified draft accepted: the bonus token is row ell's race winner (position
  // ell + 1, stream 2).  A rejection: the residual draw at position n_acc + 1 from target
  // row n_acc, in the correction pass (jstar = n_acc + 1, a compact slot on the tensor-core
  // path)
  if (lane == 0) {
    a.jstar[r] = n_acc < ell ? n_acc + 1 : 0;
    a.lse_t[r] = lse_stop;
    if (n_acc == ell) a.tokens_out[orow + ell] = bonus_id >= 0 ? bonus_id : 0;
  }
  if (n_acc < ell) {
    const int js = n_acc + 1;
    int slot = r;
    if (a.res_compact) {
      if (lane == 0) slot = atomicAdd(a.n_rej, 1);
      slot = __shfl_sync(0xffffffffu, slot, 0);
      if (lane == 0) {
        a.rej_req[slot] = r;
        a.res_hint[slot] = __float_as_int(-INFINITY) ^ 0x7FFFFFFF;  // no key published yet
      }
    }
    // gather the factor row of position j* for the bias recomputation: W1[x_{j*-1}], or
    // the recurrent head's state s_{j*}
    size_t src;
    const void* rows = a.state != nullptr ? a.state : a.W1;
    if (a.state != nullptr) {
      src = ((size_t)r * a.gamma + (js - 1)) * a.rank;
    } else {
      const int xprev = checked_token((js == 1) ? __ldg(a.x0 + r) : __ldg(a.x + (size_t)r * a.gamma + (js - 2)),
                                      a.V, a.status, 12);
      src = (size_t)xprev * a.rank;
    }
    const size_t dst = (size_t)slot * a.rank;
    if (a.dtype_w == DSPARK_BF16) {
      const unsigned short* w1 = reinterpret_cast<const unsigned short*>(rows);
      unsigned short* g = reinterpret_cast<unsigned short*>(a.W1g);
      for (int i = lane; i < a.rank; i += 32) g[dst + i] = __ldg(w1 + src + i);
    } else {
      const float* w1 = reinterpret_cast<const float*>(rows);
      float* g = reinterpret_cast<float*>(a.W1g);
      for (int i = lane; i < a.rank; i += 32) g[dst + i] = __ldg(w1 + src + i);
    }
  }
}

// CUDA-core residual pass.  blockIdx.x: vocabulary chunk; blockIdx.y: request block.
template <int RB>
__global__ void __launch_bounds__(kSimtThreads) residual_step_simt_kernel(VerifyArgs a) {
  griddep_allow_next();
  griddep_wait();
  extern __shared__ float w1s[];  // [RB][rank]
  const int r0 = blockIdx.y * RB;
  // correction position of each request (0 = none: every verified draft was accepted)
  int js[RB];
  bool any = false;
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) {
    const int r = r0 + rr;
    js[rr] = (r < a.R) ? a.jstar[r] : 0;
    any |= js[rr] > 0;
  }
  if (!any) {
    if (threadIdx.x < RB) {
      const int r = r0 + threadIdx.x;
      if (r < a.R) {
        a.res_part[(size_t)blockIdx.x * a.R + r] = to_partial(stats_empty());
        a.res_part2[(size_t)blockIdx.x * a.R + r] = to_partial(stats_empty());
      }
    }
    return;
  }
  for (int i = threadIdx.x; i < RB * a.rank; i += blockDim.x) {
    const int rr = i / a.rank, c = i % a.rank;
    const int r = r0 + rr;
    w1s[i] = (r < a.R && js[rr] > 0) ? load_elem(a.W1g, a.dtype_w, (size_t)r * a.rank + c) : 0.f;
  }
  __syncthreads();
  Stats st[RB], fb[RB];
  RngRow rng[RB];
  float lq[RB], lt[RB];
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) {
    st[rr] = stats_empty();
    fb[rr] = stats_empty();
    const int r = min(r0 + rr, a.R - 1);
    const int j = max(js[rr], 1);
    rng[rr] = rng_row(a.seed, __ldg(a.req_id + r), a.round, kStreamCorrect, (uint32_t)j);
    lq[rr] = __ldg(a.lse_q + (size_t)r * a.gamma + (j - 1));
    lt[rr] = a.lse_t[r];
  }
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
      if (r >= a.R || js[rr] == 0) continue;
      const Philox4 bits = rng_chunk(rng[rr], (uint32_t)g);
      const uint32_t wd[4] = {bits.x, bits.y, bits.z, bits.w};
      const size_t urow = ((size_t)r * a.gamma + (js[rr] - 1)) * a.V;
      const size_t trow = target_row_index(a.t_off, a.n_trows, a.gamma, r, js[rr] - 1, a.status) * a.V;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = 4 * g + e;
        if (v >= a.V) break;
        const float lp = load_elem(a.target, a.dtype_t, trow + v) * a.inv_temp - lt[rr];
        const float p = __expf(lp);
        const float z = (load_elem(a.U, a.dtype_u, urow + v) + acc[rr][e]) * a.inv_temp;
        const float rho = p - __expf(z - lq[rr]);
        const float g_ = gumbel_fast_from_bits(wd[e]);
        if (rho > 0.f) {
          const float key = __logf(rho) + g_;
          if (key > st[rr].key || st[rr].idx < 0) {
            st[rr].key = key;
            st[rr].idx = v;
          }
        }
        const float k2 = lp + g_;
        if (k2 > fb[rr].key || fb[rr].idx < 0) {
          fb[rr].key = k2;
          fb[rr].idx = v;
        }
      }
    }
  }
  __shared__ Partial red[kSimtThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int rr = 0; rr < RB; ++rr) {
    const int r = r0 + rr;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      Stats w = warp_reduce_stats(which ? fb[rr] : st[rr]);
      if (lane == 0) red[warp] = to_partial(w);
      __syncthreads();
      if (warp == 0) {
        Stats b = (lane < (int)(blockDim.x >> 5)) ? from_partial(red[lane]) : stats_empty();
        b = warp_reduce_stats(b);
        if (lane == 0 && r < a.R) (which ? a.res_part2 : a.res_part)[(size_t)blockIdx.x * a.R + r] = to_partial(b);
      }
      __syncthreads();
    }
  }
}

__global__ void residual_combine_kernel(VerifyArgs a, int npart) {
  griddep_allow_next();
  griddep_wait();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= a.R) return;
  // CUDA-core pass: warp r merges request r's chunk partials ([chunk, R]).  Compact
  // tensor-core pass: warp q merges slot q's group partials ([group, rblocks * RB]), with the
  // kernel's own split of its grid into groups
  int req = r, slot = r;
  size_t stride = (size_t)a.R;
  if (a.res_compact) {
    const int n = *reinterpret_cast<const volatile int*>(a.n_rej);
    if (r >= n) return;
    req = a.rej_req[r];
    const int rb_rows = tc_residual_rows_per_block(a.R);
    const int rblocks = (n + rb_rows - 1) / rb_rows;
    npart = max(1, a.res_grid / rblocks);
    stride = (size_t)rblocks * rb_rows;
  }
  const int js = a.jstar[req];
  if (js <= 0) return;  // no rejection: the bonus token is already written
  Stats st = stats_empty(), fb = stats_empty();
  for (int p = lane; p < npart; p += 32) {
    stats_merge(st, from_partial(a.res_part[(size_t)p * stride + slot]));
    if (!a.res_compact) stats_merge(fb, from_partial(a.res_part2[(size_t)p * stride + slot]));
  }
  st = warp_reduce_stats(st);
  fb = warp_reduce_stats(fb);
  if (lane != 0) return;
  if (st.idx >= 0) {
    a.tokens_out[(size_t)req * (a.gamma + 1) + (js - 1)] = st.idx;
  } else if (!a.res_compact) {
    // no p - q was positive (rounding): the CUDA-core pass kept the ln p draw as well
    a.tokens_out[(size_t)req * (a.gamma + 1) + (js - 1)] = fb.idx;
  } else {
    // the compact pass ran the (p - q)+ race only: the fallback pass draws from p
    a.fb_req[atomicAdd(a.n_fb, 1)] = req;
  }
}

// The rounding fallback of the compact correction pass: for each request whose residual
// had no positive p - q (which exact arithmetic rules out), the draw from p instead, with the
// residual's random numbers (stream 2 at position j*): the Gumbel-max of t/T + g over target
// row j* - 1 (the row's normaliser shifts every key alike).  One CTA per such request; the
// queue is normally empty and every CTA leaves at once.
__global__ void __launch_bounds__(kRowThreads) residual_fallback_kernel(VerifyArgs a) {
  griddep_allow_next();
  griddep_wait();
  __shared__ Partial red[kRowThreads / 32];
  const int n = *reinterpret_cast<const volatile int*>(a.n_fb);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int q = blockIdx.x; q < n; q += gridDim.x) {
    const int req = a.fb_req[q];
    const int js = a.jstar[req];
    const size_t rbase = target_row_index(a.t_off, a.n_trows, a.gamma, req, js - 1, a.status) * a.V;
    const RngRow rr = rng_row(a.seed, __ldg(a.req_id + req), a.round, kStreamCorrect, (uint32_t)js);
    Stats own = stats_empty();
    for (int g = threadIdx.x; g < (a.V + 3) / 4; g += blockDim.x) {
      const Philox4 b = rng_chunk(rr, (uint32_t)g);
      const uint32_t wd[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = 4 * g + e;
        if (v >= a.V) break;
        const float key = load_elem(a.target, a.dtype_t, rbase + v) * a.inv_temp + gumbel_from_bits(wd[e]);
        if (key_better(key, v, own.key, own.idx)) {
          own.key = key;
          own.idx = v;
        }
      }
    }
    own = warp_reduce_stats(own);
    if (lane == 0) red[warp] = to_partial(own);
    __syncthreads();
    if (threadIdx.x == 0) {
      Stats b = from_partial(red[0]);
      for (int w = 1; w < kRowThreads / 32; ++w) stats_merge(b, from_partial(red[w]));
      a.tokens_out[(size_t)req * (a.gamma + 1) + (js - 1)] = b.idx >= 0 ? b.idx : 0;
    }
    __syncthreads();
  }
}

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s) {
  cudaError_t e = launch_pdl(verify_plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int max_items = a.R * (a.gamma + 1) * a.nchunk;
  const int grid = min(max_items, sms * kRowCtasPerSm);  // work queue: CTAs take items until none is left
  if (a.chunk != kRowThreads * kRowPer) return cudaErrorInvalidValue;
  if (a.prof != nullptr && (e = record_profile_event(a.prof[0], s)) != cudaSuccess) return e;
  VerifyArgs ra = a;
  ra.keys = philox_keys(a.seed);
  e = a.dtype_t == DSPARK_F32 ? launch_pdl(verify_rows_kernel<DSPARK_F32>, dim3(grid), dim3(kRowThreads), 0, s, ra)
                              : launch_pdl(verify_rows_kernel<DSPARK_BF16>, dim3(grid), dim3(kRowThreads), 0, s, ra);
  if (e != cudaSuccess) return e;
  if (a.prof != nullptr && (e = record_profile_event(a.prof[1], s)) != cudaSuccess) return e;
  const int wblocks = (a.R * 32 + 255) / 256;
  if ((e = launch_pdl(verify_accept_kernel, dim3(wblocks), dim3(256), 0, s, a)) != cudaSuccess) return e;
  int npart;
  if (a.prof != nullptr && (e = record_profile_event(a.prof[2], s)) != cudaSuccess) return e;
  if (a.res_compact) {
    // the residual recomputes one bias row per rejected request on the tensor cores, over
    // the compact slots (the partial count is derived on the device from their number)
    if ((e = launch_residual_tc(a, s)) != cudaSuccess) return e;
    npart = 0;
  } else {
    dim3 rgrid(simt_num_chunks(a.V), (a.R + kSimtRB - 1) / kSimtRB);
    const size_t smem = sizeof(float) * kSimtRB * a.rank;
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(residual_step_simt_kernel<kSimtRB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e != cudaSuccess) return e;
    }
    if ((e = launch_pdl(residual_step_simt_kernel<kSimtRB>, rgrid, dim3(kSimtThreads), smem, s, a)) != cudaSuccess)
      return e;
    npart = (int)rgrid.x;
  }
  if (a.prof != nullptr && (e = record_profile_event(a.prof[3], s)) != cudaSuccess) return e;
  if ((e = launch_pdl(residual_combine_kernel, dim3(wblocks), dim3(256), 0, s, a, npart)) != cudaSuccess) return e;
  if (!a.res_compact) return cudaSuccess;
  return launch_pdl(residual_fallback_kernel, dim3(32), dim3(kRowThreads), 0, s, a);
}

// Partial records of the correction pass: the CUDA-core pass keeps one per (vocabulary
// chunk, request); the compact tensor-core pass one per (vocabulary group, slot), at most
// its grid times the rows of a block (every CTA covers one block of slots), which stays
// linear in R.
size_t residual_partial_entries(int R, int V, int rank, int dtype_w) {
  if (!tc_supported(V, rank, dtype_w)) return (size_t)simt_num_chunks(V) * R;
  return (size_t)tc_residual_grid(R) * tc_residual_rows_per_block(R);
}

}  // namespace dspark
