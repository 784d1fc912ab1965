// dspark_common.cuh — device helpers shared by the DSpark kernels (sm_103a).
//
// Counter-based random numbers, dtype loads, numerically careful Gumbel draws,
// online softmax / argmax records and their merges, bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

constexpr uint32_t kStreamDraft = 0u;
constexpr uint32_t kStreamAccept = 1u;
constexpr uint32_t kStreamCorrect = 2u;

// Largest value the device Gumbel below can return: -ln(-ln(1 - 2^-25)) = 25 ln 2
// (17.33) plus a margin for rounding.  An element whose logit plus this bound falls
// below the best key found so far can never win a Gumbel-max draw.
constexpr float kGumbelMax = 17.5f;

// ---------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC'11): ten rounds of two 32x32->64 products; the key is bumped by the
// Weyl constants between rounds.
// ---------------------------------------------------------------------------------
struct Philox4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo_a = 0xD2511F53u * c0;
    const uint32_t hi_a = __umulhi(0xD2511F53u, c0);
    const uint32_t lo_b = 0xCD9E8D57u * c2;
    const uint32_t hi_b = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi_b ^ c1 ^ k0;
    const uint32_t n2 = hi_a ^ c3 ^ k1;
    c0 = n0;
    c1 = lo_b;
    c2 = n2;
    c3 = lo_a;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return Philox4{c0, c1, c2, c3};
}

// Key and the two per-row counter words of the method's draws.
struct RngRow {
  uint32_t k0, k1;  // seed
  uint32_t c0, c1;  // lo32(req_id), lo32(round)
  uint32_t c2;      // stream << 24 | position
};

__device__ __forceinline__ RngRow rng_row(uint64_t seed, int64_t req_id, uint64_t round, uint32_t stream,
                                          uint32_t position) {
  RngRow r;
  r.k0 = (uint32_t)seed;
  r.k1 = (uint32_t)(seed >> 32);
  r.c0 = (uint32_t)(uint64_t)req_id;
  r.c1 = (uint32_t)round;
  r.c2 = (stream << 24) | position;
  return r;
}

__device__ __forceinline__ Philox4 rng_chunk(const RngRow& r, uint32_t chunk) {
  return philox4x32_10(r.c0, r.c1, r.c2, chunk, r.k0, r.k1);
}

// u = ((bits >> 8) + 0.5) * 2^-24 = (2b+1) * 2^-25 with b = bits >> 8, strictly inside
// (0,1).  binary64 holds it exactly; binary32 holds u exactly for b < 2^23 (u < 1/2)
// and 1-u = (2^25-2b-1) * 2^-25 exactly for b >= 2^23.
__device__ __forceinline__ double uniform_from_bits_f64(uint32_t bits) {
  return ((double)(bits >> 8) + 0.5) * 0x1.0p-24;
}

// E = -ln u from the exact binary32 piece: ln u itself below 1/2 (E >= ln 2, where a
// few ulps of relative error are harmless), log1p(-(1-u)) above, so that E keeps full
// relative accuracy as u -> 1 (E -> 2^-25), where the winning Gumbel draws live.
__device__ __forceinline__ float neg_log_uniform(uint32_t bits) {
  const uint32_t b = bits >> 8;
  if (b < (1u << 23)) {
    const float u = __uint2float_rn(2u * b + 1u) * 0x1.0p-25f;
    return -logf(u);
  }
  const float w = __uint2float_rn((1u << 25) - 2u * b - 1u) * 0x1.0p-25f;
  return -log1pf(-w);
}

// Standard Gumbel g = -ln(-ln u) = -ln E.
__device__ __forceinline__ float gumbel_from_bits(uint32_t bits) { return -logf(neg_log_uniform(bits)); }

// ---------------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------------
__device__ __forceinline__ float load_elem(const void* base, int dtype, size_t idx) {
  if (dtype == DSPARK_F32) return __ldg(reinterpret_cast<const float*>(base) + idx);
  const unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(base) + idx);
  return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

// ---------------------------------------------------------------------------------
// Online softmax statistics and Gumbel-max records
// ---------------------------------------------------------------------------------
// (m, s): s = sum exp(z - m) over the elements seen.  Empty: m = -inf, s = 0.
// (key, idx, zsel): best Gumbel key, its vocabulary id (lowest id on equal keys) and
// the value selected alongside it (the winner's logit).  Empty: key = -inf, idx = -1.
struct Stats {
  float m, s;
  float key, zsel;
  int idx;
};

__device__ __forceinline__ Stats stats_empty() {
  Stats st;
  st.m = -INFINITY;
  st.s = 0.f;
  st.key = -INFINITY;
  st.zsel = 0.f;
  st.idx = -1;
  return st;
}

__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = s * __expf(m - M) + s2 * __expf(m2 - M);
  m = M;
}

__device__ __forceinline__ bool key_better(float k1, int i1, float k2, int i2) {
  // does (k1,i1) beat (k2,i2)?  Higher key wins; on equal keys the lower id wins.
  if (i1 < 0) return false;
  if (i2 < 0) return true;
  return (k1 > k2) || (k1 == k2 && i1 < i2);
}

__device__ __forceinline__ void stats_merge(Stats& a, const Stats& b) {
  lse_merge(a.m, a.s, b.m, b.s);
  if (key_better(b.key, b.idx, a.key, a.idx)) {
    a.key = b.key;
    a.idx = b.idx;
    a.zsel = b.zsel;
  }
}

__device__ __forceinline__ Stats stats_shfl_xor(const Stats& a, int lane_mask) {
  Stats b;
  b.m = __shfl_xor_sync(0xffffffffu, a.m, lane_mask);
  b.s = __shfl_xor_sync(0xffffffffu, a.s, lane_mask);
  b.key = __shfl_xor_sync(0xffffffffu, a.key, lane_mask);
  b.zsel = __shfl_xor_sync(0xffffffffu, a.zsel, lane_mask);
  b.idx = __shfl_xor_sync(0xffffffffu, a.idx, lane_mask);
  return b;
}

__device__ __forceinline__ Stats warp_reduce_stats(Stats a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Stats b = stats_shfl_xor(a, o);
    stats_merge(a, b);
  }
  return a;
}

// Partial record written per (CTA or chunk, request) and merged by a combine kernel.
struct __align__(16) Partial {
  float m, s, key, zsel;
  int idx, pad0, pad1, pad2;
};

__device__ __forceinline__ Partial to_partial(const Stats& st) {
  Partial p;
  p.m = st.m;
  p.s = st.s;
  p.key = st.key;
  p.zsel = st.zsel;
  p.idx = st.idx;
  p.pad0 = p.pad1 = p.pad2 = 0;
  return p;
}

__device__ __forceinline__ Stats from_partial(const Partial& p) {
  Stats st;
  st.m = p.m;
  st.s = p.s;
  st.key = p.key;
  st.zsel = p.zsel;
  st.idx = p.idx;
  return st;
}

// ---------------------------------------------------------------------------------
// Device status word (first 16 bytes of every workspace)
// ---------------------------------------------------------------------------------
struct DeviceStatus {
  int code;      // 0 OK, DSPARK_TIMEOUT
  int where;     // which wait gave up
  int pad0, pad1;
};

__device__ __forceinline__ void report_timeout(DeviceStatus* st, int where) {
  if (st) {
    atomicExch(&st->code, DSPARK_TIMEOUT);
    atomicExch(&st->where, where);
  }
}

// Device data that the host could not validate (token ids, verify lengths) outside
// its range: recorded as DSPARK_INVALID_ARG; the kernel clamps the value so that every
// access stays in bounds.
__device__ __forceinline__ void report_bad_input(DeviceStatus* st, int where) {
  if (st && atomicCAS(&st->code, 0, DSPARK_INVALID_ARG) == 0) atomicExch(&st->where, where);
}

__device__ __forceinline__ int checked_token(int x, int V, DeviceStatus* st, int where) {
  if (x < 0 || x >= V) {
    report_bad_input(st, where);
    return 0;
  }
  return x;
}

__device__ __forceinline__ float sigmoidf_dev(float x) { return 1.0f / (1.0f + __expf(-x)); }

}  // namespace dspark
