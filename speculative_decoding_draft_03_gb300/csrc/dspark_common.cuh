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
    // one 32x32->64 product each (a single wide multiply), then the xor mix
    const unsigned long long pa = 0xD2511F53ull * (unsigned long long)c0;
    const unsigned long long pb = 0xCD9E8D57ull * (unsigned long long)c2;
    const uint32_t n0 = (uint32_t)(pb >> 32) ^ c1 ^ k0;
    const uint32_t n2 = (uint32_t)(pa >> 32) ^ c3 ^ k1;
    c0 = n0;
    c1 = (uint32_t)pb;
    c2 = n2;
    c3 = (uint32_t)pa;
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

// The same generator specialised to one row: only the 4th counter word (the chunk)
// varies, so the first round's products, half of the second round's and half of the
// third round's are per-row constants, and so are the round keys of rounds 4..10 (kept
// per row rather than re-derived in every block).
// philox_row(...).block(chunk) == rng_chunk(row, chunk) bit for bit.
struct PhiloxRow {
  uint32_t p;       // round 1 input word 2 without the chunk:  hi(M_A c0) ^ k1
  uint32_t g;       // round 2 output word 0 partial:          lo(M_B c2) ^ (k0 + W_A)
  uint32_t h3, l3;  // round 3: hi(M_B e) ^ (k0 + 2 W_A) and lo(M_B e), e = round 2 output word 2
  uint32_t f3;      // round 3: f ^ (k1 + 2 W_B), f = round 2 output word 3
  uint32_t ka[7], kb[7];  // round keys of rounds 4..10

  __device__ __forceinline__ Philox4 block(uint32_t chunk) const {
    const uint32_t x2 = p ^ chunk;
    const unsigned long long pb = 0xCD9E8D57ull * (unsigned long long)x2;
    // round 2 output: (hi(pb) ^ g, lo(pb), e, f); round 3 on it, whose B product M_B e
    // is a per-row constant
    const uint32_t c0r2 = (uint32_t)(pb >> 32) ^ g;
    const unsigned long long qa3 = 0xD2511F53ull * (unsigned long long)c0r2;
    uint32_t c0 = (uint32_t)pb ^ h3, c1 = l3, c2 = (uint32_t)(qa3 >> 32) ^ f3, c3 = (uint32_t)qa3;
#pragma unroll
    for (int i = 3; i < 10; ++i) {
      const unsigned long long qa = 0xD2511F53ull * (unsigned long long)c0;
      const unsigned long long qb = 0xCD9E8D57ull * (unsigned long long)c2;
      const uint32_t n0 = (uint32_t)(qb >> 32) ^ c1 ^ ka[i - 3];
      const uint32_t n2 = (uint32_t)(qa >> 32) ^ c3 ^ kb[i - 3];
      c0 = n0;
      c1 = (uint32_t)qb;
      c2 = n2;
      c3 = (uint32_t)qa;
    }
    return Philox4{c0, c1, c2, c3};
  }
};

__device__ __forceinline__ PhiloxRow philox_row(const RngRow& r) {
  // round 1 with (c0, c1, c2, chunk): outputs (hi(pb)^c1^k0, lo(pb), hi(pa)^chunk^k1, lo(pa))
  const unsigned long long pa = 0xD2511F53ull * (unsigned long long)r.c0;
  const unsigned long long pb = 0xCD9E8D57ull * (unsigned long long)r.c2;
  const uint32_t y0 = (uint32_t)(pb >> 32) ^ r.c1 ^ r.k0;
  const uint32_t y1 = (uint32_t)pb;
  const uint32_t y3 = (uint32_t)pa;
  // round 2 (key + W): its A-product uses y0 only, a per-row constant
  const uint32_t ka = r.k0 + 0x9E3779B9u, kb = r.k1 + 0xBB67AE85u;
  const unsigned long long qa = 0xD2511F53ull * (unsigned long long)y0;
  const uint32_t e = (uint32_t)(qa >> 32) ^ y3 ^ kb;  // round 2 output word 2
  const uint32_t f = (uint32_t)qa;                    // round 2 output word 3
  // round 3 (key + 2W): its B-product uses e only
  const unsigned long long qb3 = 0xCD9E8D57ull * (unsigned long long)e;
  PhiloxRow o;
  o.p = (uint32_t)(pa >> 32) ^ r.k1;
  o.g = y1 ^ ka;
  o.h3 = (uint32_t)(qb3 >> 32) ^ (r.k0 + 2u * 0x9E3779B9u);
  o.l3 = (uint32_t)qb3;
  o.f3 = f ^ (r.k1 + 2u * 0xBB67AE85u);
#pragma unroll
  for (int i = 3; i < 10; ++i) {
    o.ka[i - 3] = r.k0 + (uint32_t)i * 0x9E3779B9u;
    o.kb[i - 3] = r.k1 + (uint32_t)i * 0xBB67AE85u;
  }
  return o;
}

// The round keys of rounds 4..10 depend on the seed alone, which every row of a launch
// shares: a kernel that carries them in its parameters (constant memory, read as
// instruction operands) holds only the five per-row words of PhiloxRowWords in
// registers.  PhiloxRowWords::block(chunk, keys) == PhiloxRow::block(chunk) bit for bit.
struct PhiloxKeys {
  uint32_t ka[7], kb[7];
};

__host__ __device__ inline PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys k;
  for (int i = 3; i < 10; ++i) {
    k.ka[i - 3] = (uint32_t)seed + (uint32_t)i * 0x9E3779B9u;
    k.kb[i - 3] = (uint32_t)(seed >> 32) + (uint32_t)i * 0xBB67AE85u;
  }
  return k;
}

struct PhiloxRowWords {
  uint32_t p, g, h3, l3, f3;  // as in PhiloxRow

  __device__ __forceinline__ Philox4 block(uint32_t chunk, const PhiloxKeys& k) const {
    const uint32_t x2 = p ^ chunk;
    const unsigned long long pb = 0xCD9E8D57ull * (unsigned long long)x2;
    const uint32_t c0r2 = (uint32_t)(pb >> 32) ^ g;
    const unsigned long long qa3 = 0xD2511F53ull * (unsigned long long)c0r2;
    uint32_t c0 = (uint32_t)pb ^ h3, c1 = l3, c2 = (uint32_t)(qa3 >> 32) ^ f3, c3 = (uint32_t)qa3;
#pragma unroll
    for (int i = 3; i < 10; ++i) {
      const unsigned long long qa = 0xD2511F53ull * (unsigned long long)c0;
      const unsigned long long qb = 0xCD9E8D57ull * (unsigned long long)c2;
      const uint32_t n0 = (uint32_t)(qb >> 32) ^ c1 ^ k.ka[i - 3];
      const uint32_t n2 = (uint32_t)(qa >> 32) ^ c3 ^ k.kb[i - 3];
      c0 = n0;
      c1 = (uint32_t)qb;
      c2 = n2;
      c3 = (uint32_t)qa;
    }
    return Philox4{c0, c1, c2, c3};
  }
};

__device__ __forceinline__ PhiloxRowWords philox_row_words(const RngRow& r) {
  const PhiloxRow f = philox_row(r);
  return PhiloxRowWords{f.p, f.g, f.h3, f.l3, f.f3};
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

// Packed fp32 pairs (the f32x2 arithmetic of sm_100 and later): one instruction for two
// independent adds / subtracts / multiplies, each rounded exactly like its scalar
// counterpart; and the three-input maximum (a NaN operand is ignored, as by fmaxf).
__device__ __forceinline__ void add2f(float& a, float& b, float c, float d) {
  asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "add.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a), "+f"(b)
      : "f"(c), "f"(d));
}
__device__ __forceinline__ void sub2f(float& a, float& b, float c, float d) {
  asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "sub.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a), "+f"(b)
      : "f"(c), "f"(d));
}
__device__ __forceinline__ void mul2f(float& a, float& b, float c, float d) {
  asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "mul.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a), "+f"(b)
      : "f"(c), "f"(d));
}
__device__ __forceinline__ float max3f_(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float exp2f_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Standard Gumbel g = -ln(-ln u) from special-function approximations and a short series,
// for the draws that survive the rejection test of a Gumbel-max race.  Its absolute error
// stays far inside the 1e-5 boundary window (checked on the GPU against binary64 over every
// 256th 24-bit uniform code and both tails):
//   u < 1/2:  E = -ln u = -log2(u) ln 2, where |log2 u| >= 1 keeps the approximation's
//             error relative;
//   u >= 1/2: E = -ln(1 - w) = 2 atanh(s) with s = w / (2 - w) in (0, 1/3] (w = 1 - u, exact),
//             the odd series of atanh through s^13 (truncation below 2e-8 relative), so E
//             keeps full relative accuracy as u -> 1, where the winning draws live;
//   g = -ln E with E = 2^e m, m in [1, 2): -(e ln 2 + log2(m) ln 2), e exact.
__device__ __forceinline__ float gumbel_fast_from_bits(uint32_t bits) {
  constexpr float kLn2 = 0.6931471805599453f;
  const uint32_t b = bits >> 8;
  float E;
  if (b < (1u << 23)) {
    const float u = __uint2float_rn(2u * b + 1u) * 0x1.0p-25f;
    E = -lg2_approx(u) * kLn2;
  } else {
    const float w = __uint2float_rn((1u << 25) - 2u * b - 1u) * 0x1.0p-25f;
    const float sv = w * rcp_approx(2.f - w);
    const float t = sv * sv;
    float q = fmaf(t, 1.f / 13.f, 1.f / 11.f);
    q = fmaf(t, q, 1.f / 9.f);
    q = fmaf(t, q, 1.f / 7.f);
    q = fmaf(t, q, 1.f / 5.f);
    q = fmaf(t, q, 1.f / 3.f);
    q = fmaf(t, q, 1.f);
    E = 2.f * sv * q;
  }
  // E is a positive normal number (at least 2^-25): split off its exponent exactly
  const uint32_t eb = __float_as_uint(E);
  const float m = __uint_as_float((eb & 0x007FFFFFu) | 0x3F800000u);
  // the unbiased exponent as a float, without a conversion: 1.5 * 2^23 + e, minus 1.5 * 2^23
  const float e = __int_as_float(0x4B400000 + (int)(eb >> 23) - 127) - 12582912.f;
  return -fmaf(e, kLn2, lg2_approx(m) * kLn2);
}

// Natural logarithm of a positive normal float from its exact exponent and the
// special-function log2 of its mantissa in [1, 2) (absolute error a few 1e-7); values below
// the normal range count as 2^-126 (they never decide a draw: their keys lie ~87 below).
__device__ __forceinline__ float ln_fast(float x) {
  constexpr float kLn2 = 0.6931471805599453f;
  const uint32_t b = __float_as_uint(fmaxf(x, 0x1.0p-126f));
  const float m = __uint_as_float((b & 0x007FFFFFu) | 0x3F800000u);
  const float e = __int_as_float(0x4B400000 + (int)(b >> 23) - 127) - 12582912.f;
  return fmaf(e, kLn2, lg2_approx(m) * kLn2);
}

// 1 - u in binary32 (exact for u >= 1/2, within one rounding below).  Since
// E = -ln u = -ln(1 - w) >= w, an element with w >= t has E >= t.
__device__ __forceinline__ float one_minus_uniform(uint32_t bits) {
  return __uint2float_rn((1u << 25) - 2u * (bits >> 8) - 1u) * 0x1.0p-25f;
}

// Exact rejection test of the Gumbel-max race.  key = z + g beats `best` only if
// E < exp(z - best).  `t` must be an upper bound of exp(z - best); callers inflate
// it by a small factor to cover the rounding of exp and of w.  Returns true when the
// element certainly cannot beat `best`, without evaluating any logarithm.
__device__ __forceinline__ bool gumbel_cannot_win(uint32_t bits, float t) { return one_minus_uniform(bits) >= t; }

// Relative inflation of exp(z - best) in the rejection test: covers the error of the
// fast exponential (a few ulp), the rounding of w, and leaves a wide margin (e^0.002).
constexpr float kRejectSlack = 1.002f;

// The same test without an integer-to-float conversion, for callers that test many
// elements.  f = 1 + floor(b / 2) * 2^-23 (b = bits >> 8; the word's top 23 bits as a
// mantissa) satisfies u - (f - 1) < 2^-23, so 1 - u > 2 - f - 2^-23.  f + t <= 2 - 2^-22
// (evaluated as one FMA, whose rounding stays below 2^-24 in [1, 2)) therefore implies
// 1 - u >= t: the element is rejected only when the exact test would reject it too.
__device__ __forceinline__ float uniform_mantissa(uint32_t bits) { return __uint_as_float(0x3F800000u | (bits >> 9)); }
constexpr float kRejectEdge = 2.f - 0x1.0p-22f;

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

// Row of the target logits holding request r's verify row t: the padded layout
// [R, gamma+1, V] (t_off == nullptr), or the flattened layout with request r's rows at
// t_off[r], t_off[r]+1, ... of n_trows rows.  An offset outside the array is reported
// and row 0 is used instead (every access stays in bounds).
__device__ __forceinline__ size_t target_row_index(const int32_t* t_off, int n_trows, int gamma, int r, int t,
                                                   DeviceStatus* st) {
  if (t_off == nullptr) return (size_t)r * (gamma + 1) + t;
  const long long row = (long long)__ldg(t_off + r) + t;
  if (row < 0 || row >= n_trows) {
    report_bad_input(st, 14);
    return 0;
  }
  return (size_t)row;
}

// Programmatic dependent launch: every kernel of the round is launched so that it may
// start while its predecessor drains.  griddep_wait() returns once the preceding grid
// has completed and its memory is visible; a kernel calls it before touching anything
// a predecessor writes or reads.  griddep_allow_next() lets the next grid start its own
// prologue early (it will still wait before its first dependent access).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_allow_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace dspark
