// draft_tc.cu — the fused draft step on the 5th-generation tensor cores (sm_103a).
//
// One launch per draft position k computes, for every request r and vocabulary id v,
//   z[r,v] = (U[r,k,v] + (W1[x_{k-1}(r),:] . W2[:,v])) / T
// and reduces each request's row to (max, sum exp, Gumbel-max key/id) partials, so the
// vocabulary row is streamed exactly once per position (numb3r33 blog "DSpark:
// confidence-scheduled speculative decoding", section "Markov sequential head";
// DSpark 精读 §2: p_k = softmax(U_k + W1[x_{k-1}] W2), sampled left to right).  Other
// epilogue modes of the same pipeline: verification's correction draw (the rejected
// position's row for the (p - q)+ residual, or the bonus draw from the target row), the
// recurrent head's draft step (factor rows = the states), and the acceptance-overlap
// diagnostic (sum min(q, p) per drafted position).  The file also holds the recurrent
// head's hidden-state projection, a plain tcgen05 GEMM.
//
// GB300 mapping
//   * The bias is an [R x rank] x [rank x V] contraction: tcgen05.mma kind::f16
//     (bf16 x bf16 -> fp32), M = 128 requests (TMEM lanes), N = 128 vocabulary ids per
//     tile (TMEM columns), K = rank.  The gathered factor rows W1[x_{k-1}] (A, K-major)
//     stay resident in shared memory; W2 tiles (B, read in its natural [rank, V] layout,
//     i.e. MN-major) stream through a TMA ring with 128-byte swizzle, marked to stay in
//     L2 across the draft positions of a round.
//   * Accumulators live in TMEM, double-buffered (2 x 128 columns) so the MMA of tile
//     t+1 overlaps the epilogue of tile t.
//   * Epilogue (16 warps, 4 per TMEM lane quarter): each thread owns one request (its
//     TMEM lane) and runs of 8 consecutive vocabulary ids, so softmax statistics and the
//     Gumbel-max draw are thread-local and one Philox block serves 4 consecutive ids.
//     Random words are only turned into Gumbel keys for elements that survive an exact
//     log-free rejection test against the best key known so far.
//   * Few requests (R <= 64): the request rows are replicated across the 4 TMEM lane
//     quarters and each quarter takes a different part of the tile's columns, so all
//     epilogue warps stay busy.
//   * Many requests (R > 128): CTAs are grouped by request block; the CTAs of a group
//     walk the same W2 tiles at the same time, so W2 comes from HBM once per position
//     and from L2 for the other request blocks.
//   * U (draft mode) also arrives by TMA: 128-byte-wide boxes of request rows at the
//     current position, 128B-swizzled so that each thread's row reads are bank-conflict
//     free, several tiles ahead of the epilogue.  Epilogue threads issue no global loads.
//   * Warp roles: warp 0 W2/A TMA producer, warp 1 TMEM allocator + MMA issuer, warp 2 U
//     TMA producer, warps 3..18 epilogue.  Every mbarrier wait is bounded; a wait that
//     gives up records DSPARK_TIMEOUT in the workspace status word and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>

#include "dspark_common.cuh"
#include "dspark_internal.h"

namespace dspark {
namespace tc {

constexpr int kM = 128;           // MMA rows (requests, replicated for small batches)
constexpr int kN = 128;           // vocabulary ids per tile
constexpr int kKAtom = 64;        // bf16 elements per 128-byte swizzle row
constexpr int kStageBytes = kN * kKAtom * 2;  // 16 KB per W2 ring stage (one 64-deep K slice)
constexpr int kMaxUBoxes = 16;
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kFirstEpiWarp = 3;  // warps 0..2: W2/A producer, MMA issuer, U producer
constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
constexpr int kCols = 8;          // vocabulary ids per epilogue pass
constexpr int kTmemCols = 2 * kN;
constexpr int kMaxRank = 256;
#ifdef DSPARK_TEST_WAIT_LIMIT
// Test builds only (never the shipped library): a short wait limit, and a draft call
// with round index kTestStallRound has its U producer issue nothing, so the epilogue's
// first bounded wait gives up and the abort path runs.
constexpr long long kWaitCycles = DSPARK_TEST_WAIT_LIMIT;
constexpr uint64_t kTestStallRound = 0x5EEDull;
#else
constexpr long long kWaitCycles = 4000000000ll;  // ~2 s at 2 GHz
#endif
// Tiles after which a CTA publishes its best keys: one for 32-request blocks (eight
// tiles per CTA, where each publication is a visible share of the step), two otherwise.
template <int RB>
constexpr int publish_tiles() { return RB == 32 ? 1 : 2; }

// Shared-memory plan per request-block size RB.  The U ring (draft mode) holds boxes of
// 128 bytes x RB request rows (32 fp32 or 64 bf16 vocabulary ids); the kernel uses a
// whole number of tiles' worth of them (four fp32 or two bf16 boxes per tile), so it
// needs room for at least four.  RB = 64 and 128 trade one W2 stage for a 64 KB ring.
template <int RB>
struct Smem {
  static constexpr int stages = RB == 32 ? 6 : 5;                 // W2 ring stages
  static constexpr int ubytes = RB == 32 ? 56 * 1024 : 64 * 1024;  // U ring
  static constexpr int uboxes = ubytes / (RB * 128);
  // offsets from the 1024-byte aligned base
  static constexpr int a = 0;                                  // [rank/64][128 rows][128 B]
  static constexpr int b = a + kM * kMaxRank * 2;              // [stages][2][64 rows][128 B]
  static constexpr int u = b + stages * kStageBytes;           // [boxes][rows][128 B]
  static constexpr int pub = u + ubytes;                       // [16 warps][32] float
  static constexpr int bars = pub + kEpiWarps * 32 * 4;        // mbarriers
  static constexpr int total = bars + 512;
  // the final merge ([16 warps][32] Partial = 16 KB) reuses the idle W2 ring
  static constexpr int red = b;
  static_assert(kEpiWarps * 32 * 32 <= stages * kStageBytes, "merge scratch must fit in the W2 ring");
  static_assert(uboxes >= 4 && uboxes <= kMaxUBoxes, "U ring must hold one tile of fp32 boxes");
  static_assert(total + 1024 <= 232448, "shared memory plan exceeds 227 KB");
  static_assert(8 * (2 * stages + 7 + 2 * kMaxUBoxes) + 16 <= 512,
                "barriers, TMEM slot and abort flag fit in 512 B");
};

// ------------------------------------------------------------------------------------
// PTX wrappers
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test, but a thread whose phase is still open is suspended until the phase
// completes or kSuspendNs nanoseconds pass (the PTX suspend-time hint), instead of
// returning at once: a waiting warp then takes no issue slots from the warps that
// share its scheduler, which a tight polling loop does.
constexpr uint32_t kSuspendNs = 1u << 18;  // 262 us, well inside every wait bound

__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up when another role aborted or after kWaitCycles.
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, DeviceStatus* st, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_suspend(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      report_timeout(st, where);
      return false;
    }
  }
}

// Bounded wait on the abort path: returns once the phase completed or after kWaitCycles,
// whatever the abort flag says (used to let copies and MMAs already in flight land
// before the CTA exits).
__device__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait_suspend(bar, parity))
    if (clock64() - t0 > kWaitCycles) return;
}

// 2-D tensor load with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// 3-D tensor load (U viewed as [R][gamma][V]: a box of request rows at one position).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// The W2 factor is re-read at every draft position of a round: keep it resident.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Order-preserving int encoding of a float (for atomicMax on keys of any sign).
__device__ __forceinline__ int ordered_key(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float key_from_ordered(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7FFFFFFF); }

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// The epilogue carries its logits in base 2 (y = z log2(e)), so that each exponential is
// one ex2 instruction; keys and the selected logit are converted back to natural units.
constexpr float kLog2ef = 1.4426950408889634f, kLn2f = 0.6931471805599453f;
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed fused multiply-add of two fp32 pairs (sm_100 f32x2), rounded as fmaf:
// (a, b) <- (fmaf(x0, y0, a), fmaf(x1, y1, b))
__device__ __forceinline__ void fma2(float& a, float& b, float x0, float x1, float y0, float y1) {
  asm("{\n\t.reg .b64 x, y, c;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mov.b64 c, {%0, %1};\n\tfma.rn.f32x2 c, x, y, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "+f"(a), "+f"(b)
      : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 8 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[kCols]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 descriptor format:
// start >> 4 in [0,14), leading byte offset >> 4 in [16,30), stride byte offset >> 4
// in [32,46), version 1 in [46,48), swizzle mode 2 = 128B in [61,64)).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor kind::f16: D fp32, A bf16 K-major, B bf16 MN-major, M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

struct TcParams {
  int R, gamma, V, rank;
  int dtype_u;
  int Rb;          // requests per block: 32, 64 or 128
  int rblocks;     // ceil(R / Rb)
  int ngroups;     // CTAs per request block (= partial records per request)
  int ntiles;      // ceil(V / 128)
  int k;           // draft position (1-based)
  int ubox_cols;   // draft mode: vocabulary ids per 128-byte U box (32 fp32, 64 bf16)
  float inv_temp;
  const void* U;
  const int64_t* req_id;
  uint64_t seed, round;
  PhiloxKeys keys;  // round keys of the seed (uniform over the launch)
  Partial* partials;  // [ngroups, R]
  int* hint;          // [R] published best keys (draft mode; residual mode: per slot)
  DeviceStatus* status;
  // residual mode
  const void* target;
  const int32_t* t_off;  // flattened target rows (nullptr: padded [R, gamma+1, V])
  int n_trows;
  int dtype_t;
  const int* jstar;     // [R] correction position (0 none; negative: a bonus draw)
  const float* lse_q;   // [R, gamma]
  const float* lse_t;   // [R]
  Partial* partials2;   // [ngroups, R] fallback draw
  // draft mode: the factor rows of position k come from the previous position's winner
  // (x0 at k = 1); each CTA publishes its per-request winner into win (64-bit maximum of
  // (key code, ~id)); group-0 CTAs write the confidence c_k for k >= 2
  const int32_t* x0;
  const unsigned long long* win_prev;  // [R] winners of position k-1 (k >= 2)
  unsigned long long* win;             // [R] winners of position k
  const void* W1;                      // [V, rank] bf16
  const float* w_e;                    // [rank]
  const float* s_h;                    // [R, gamma]
  const float* conf_temp;              // [gamma]
  float* conf_out;                     // [R, gamma]
  float conf_b, conf_scale;
  // residual mode: row q is compact slot q, request res_req[q] (*res_nrows slots, known on
  // the device only, so request blocks and vocabulary groups are derived from it)
  const int* res_req;
  const int* res_nrows;
  // overlap mode: rows are the flattened [R*gamma] positions (R above counts rows);
  // row i is request i / gamma at position i % gamma + 1, evaluated when that position
  // is at most ell[request] (every position without ell)
  const int32_t* ell;
  float* ovl_part;  // [ngroups, rows] partial sums of min(q, p)
  // overlap mode on the verify plan's compact rows (nullptr: the flattened positions):
  // row q is target row ovl_t[q] of request ovl_req[q] and evaluates position
  // ovl_t[q] + 1 when ovl_t[q] < ell[request]; *ovl_nrows rows exist (known on the device
  // only), so request blocks and vocabulary groups are derived from it in the kernel;
  // lse_t is in row order
  const int* ovl_req;
  const int* ovl_t;
  const int* ovl_nrows;
  int grid;  // CTAs to launch (0: ngroups * rblocks)
};

constexpr int kModeDraft = 0;
constexpr int kModeResidual = 1;
constexpr int kModeOverlap = 2;
constexpr int kModeRnn = 3;

// 8 consecutive ids of U (fp32 or bf16) as fp32; ids at or beyond V read as 0 (V % 8 == 0,
// so a run of 8 is either entirely inside the row or entirely outside).
__device__ __forceinline__ void load_run8(const void* base, int dtype, size_t row, int v, int V, bool valid,
                                          uint4 (&raw)[2]) {
  if (!valid || v >= V) {
    raw[0] = raw[1] = make_uint4(0u, 0u, 0u, 0u);
  } else if (dtype == DSPARK_F32) {
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(base) + row + v);
    raw[0] = __ldg(src);
    raw[1] = __ldg(src + 1);
  } else {
    raw[0] = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(base) + row + v));
    raw[1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ void decode_run8(int dtype, const uint4 (&raw)[2], float (&x)[kCols]) {
  if (dtype == DSPARK_F32) {
    x[0] = __uint_as_float(raw[0].x); x[1] = __uint_as_float(raw[0].y);
    x[2] = __uint_as_float(raw[0].z); x[3] = __uint_as_float(raw[0].w);
    x[4] = __uint_as_float(raw[1].x); x[5] = __uint_as_float(raw[1].y);
    x[6] = __uint_as_float(raw[1].z); x[7] = __uint_as_float(raw[1].w);
  } else {
    const uint32_t wd[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = bf16_bits_to_float(wd[e] & 0xFFFFu);
      x[2 * e + 1] = bf16_bits_to_float(wd[e] >> 16);
    }
  }
}

// The 8 ids' random words of one run: Philox blocks (v0 / 4) and (v0 / 4 + 1).
__device__ __forceinline__ void philox_run(const PhiloxRowWords& prow, const PhiloxKeys& keys, int v0,
                                           uint32_t (&wd)[kCols]) {
#pragma unroll
  for (int g4 = 0; g4 < 2; ++g4) {
    const Philox4 bits = prow.block((uint32_t)((v0 >> 2) + g4), keys);
    wd[4 * g4 + 0] = bits.x;
    wd[4 * g4 + 1] = bits.y;
    wd[4 * g4 + 2] = bits.z;
    wd[4 * g4 + 3] = bits.w;
  }
}

// Draft modes, one tile of one request row: the thread's KP runs of 8 ids (vocabulary ids
// v0 + 8 ps + i; U in ucur, the bias in TMEM at taddr + 8 ps).  All logits of the tile
// come first, so the online softmax is rescaled once per tile; then the Gumbel-max race
// runs run by run against the best key known so far (own record or published bound).
// (Generating the next run's Philox words while the current run is tested measured
// slower: the extra live registers at 128-row blocks cost more than the overlap gained.)  An id is
// rejected without logarithms when 1 - u >= exp(z - best) = term * exp(m - best) (the
// conversion-free form v = term * scale + f > edge marks the ids that may beat it; the
// run is done when even the largest v is not); survivors evaluate their key.  Without any
// known key, the tile's largest logit is keyed first so that the others are tested
// against it.  Runs at or beyond V, and rows beyond R, contribute nothing.
template <int KP>
__device__ __forceinline__ void draft_tile(const TcParams& p, Stats& st, const PhiloxRowWords& prow,
                                           const uint4 (&ucur)[KP][2], uint32_t taddr, bool acc_ready, bool valid,
                                           int v0, float zscale, float bound, uint32_t bar_acc_empty, int lane) {
  float y[KP][kCols];
  float tmax = -INFINITY;
#pragma unroll
  for (int ps = 0; ps < KP; ++ps) {
    if (acc_ready) {
      float bias[kCols];
      tmem_ld8(taddr + ps * kCols, bias);
      if (ps == KP - 1) {
        // all of this warp's columns are in registers: hand the accumulator back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acc_empty);
      }
      decode_run8(p.dtype_u, ucur[ps], y[ps]);
      // y = (u + bias) * zscale, two ids per packed instruction (rounded as the scalar ops)
#pragma unroll
      for (int i = 0; i < kCols; i += 2) {
        add2f(y[ps][i], y[ps][i + 1], bias[i], bias[i + 1]);
        mul2f(y[ps][i], y[ps][i + 1], zscale, zscale);
      }
    }
    if (!(acc_ready && valid && v0 + ps * kCols < p.V)) {
#pragma unroll
      for (int i = 0; i < kCols; ++i) y[ps][i] = -INFINITY;
    }
    tmax = max3f_(tmax, max3f_(max3f_(y[ps][0], y[ps][1], y[ps][2]), max3f_(y[ps][3], y[ps][4], y[ps][5]), y[ps][6]),
                 y[ps][7]);
  }
  if (!(tmax > -INFINITY)) return;  // nothing of this row in the tile
  // online softmax statistics, one rescale per tile; term_i = 2^(y_i - m) = e^(z_i - m ln 2)
  const float mnew = fmaxf(st.m, tmax);
  float acc = (st.m == -INFINITY) ? 0.f : st.s * ex2_approx(st.m - mnew);
  st.m = mnew;
  float thr = fmaxf(st.idx >= 0 ? st.key : -INFINITY, bound);
  // no id of the tile can reach the best key even with the largest possible Gumbel: no
  // random words are needed
  const bool race = !(thr > -INFINITY && fmaf(tmax, kLn2f, kGumbelMax) < thr);
  if (race && thr == -INFINITY) {
    // no key known yet (this thread's first tile, no bound published): key the tile's
    // largest logit first, the strongest threshold a single draw can give, so that the
    // other ids are tested against it (the lowest id among equal maxima)
    int kb = 0;
#pragma unroll
    for (int q = KP * kCols - 1; q >= 0; --q)
      if (y[q / kCols][q % kCols] == tmax) kb = q;
    const int vm = v0 + kb;
    const Philox4 b4 = prow.block((uint32_t)(vm >> 2), p.keys);
    const uint32_t w = (vm & 3) == 0 ? b4.x : ((vm & 3) == 1 ? b4.y : ((vm & 3) == 2 ? b4.z : b4.w));
    const float cn = tmax * kLn2f;
    st.key = cn + gumbel_fast_from_bits(w);
    st.idx = vm;
    st.zsel = cn;
    thr = st.key;
  }
#pragma unroll
  for (int ps = 0; ps < KP; ++ps) {
    const int vb = v0 + ps * kCols;
    float term[kCols];
#pragma unroll
    for (int i = 0; i < kCols; i += 2) {
      term[i] = y[ps][i];
      term[i + 1] = y[ps][i + 1];
      sub2f(term[i], term[i + 1], mnew, mnew);
    }
#pragma unroll
    for (int i = 0; i < kCols; ++i) term[i] = ex2_approx(term[i]);
    {
      // pairwise sum of the 8 terms
      float a0 = term[0], a1 = term[1], a4 = term[4], a5 = term[5];
      add2f(a0, a1, term[2], term[3]);
      add2f(a4, a5, term[6], term[7]);
      add2f(a0, a1, a4, a5);
      acc += a0 + a1;
    }
    // (no per-run skip test: the tile's test above covers the common case, and a run at or
    // beyond V has only -inf logits, whose keys can never win)
    if (race) {
      uint32_t wd[kCols];
      philox_run(prow, p.keys, vb, wd);
      // the scale e^(m ln 2 - best) is 2^(m - best log2 e)
      const float scale = ex2_approx(fmaf(-thr, kLog2ef, mnew)) * kRejectSlack;
      float v[kCols];
#pragma unroll
      for (int i = 0; i < kCols; ++i) v[i] = uniform_mantissa(wd[i]);
#pragma unroll
      for (int i = 0; i < kCols; i += 2) fma2(v[i], v[i + 1], term[i], term[i + 1], scale, scale);
      const float vmax = fmaxf(max3f_(max3f_(v[0], v[1], v[2]), max3f_(v[3], v[4], v[5]), v[6]), v[7]);
      if (vmax > kRejectEdge) {
        uint32_t cand = 0;
#pragma unroll
        for (int i = 0; i < kCols; ++i)
          if (v[i] > kRejectEdge) cand |= 1u << i;
        while (cand) {
          const int i = __ffs(cand) - 1;
          cand &= cand - 1;
          float zi = 0.f;
          uint32_t wi = 0u;
#pragma unroll
          for (int j = 0; j < kCols; ++j)  // static register selection (no local memory)
            if (j == i) {
              zi = y[ps][j];
              wi = wd[j];
            }
          if (vb + i == st.idx) continue;  // already keyed above
          zi *= kLn2f;
          const float key = zi + gumbel_fast_from_bits(wi);
          if (key > st.key || (key == st.key && vb + i < st.idx)) {
            st.key = key;
            st.idx = vb + i;
            st.zsel = zi;
            thr = fmaxf(thr, key);
          }
        }
      }
    }
  }
  st.s = acc;
}

// RB: requests per block (32, 64 or 128); the 128 MMA rows hold 128/RB copies of it.
// MODE: kModeDraft (one draft position for every request; the factor rows W1[x_{k-1}]
// are gathered by the epilogue), kModeRnn (one draft position with the factor rows
// given: the recurrent head's states), kModeResidual (each request's correction draw:
// the residual at the rejected position j*, or the bonus draw) or kModeOverlap (every drafted position: sum_v min(q, p), the
// expected acceptance).
template <int RB, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    draft_step_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                         const __grid_constant__ CUtensorMap map_u, TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  using SM = Smem<RB>;
  constexpr int kStages = SM::stages;
  // draft positions: U through the TMA ring, online softmax + Gumbel-max, winners published
  constexpr bool kDraftMath = MODE == kModeDraft || MODE == kModeRnn;
  int rblocks = p.rblocks, ngroups = p.ngroups;
  if constexpr (MODE == kModeResidual) {
    // the rejected requests' compact slots: their number comes from the preceding verify
    // pass; CTAs beyond the blocks in use leave before touching any barrier or tensor memory
    griddep_wait();
    const int n = *reinterpret_cast<const volatile int*>(p.res_nrows);
    rblocks = (max(n, 0) + RB - 1) / RB;
    if (rblocks == 0 || rblocks > p.rblocks) return;
    ngroups = max(1, (int)gridDim.x / rblocks);
    if ((int)blockIdx.x >= rblocks * ngroups) return;
  }
  if constexpr (MODE == kModeOverlap) {
    if (p.ovl_nrows != nullptr) {
      // compact rows: their number comes from the preceding verify pass; CTAs beyond the
      // blocks in use leave before touching any barrier or tensor memory
      griddep_wait();
      const int n = *reinterpret_cast<const volatile int*>(p.ovl_nrows);
      rblocks = (max(n, 0) + RB - 1) / RB;
      if (rblocks == 0 || rblocks > p.rblocks) return;
      ngroups = max(1, (int)gridDim.x / rblocks);
      if ((int)blockIdx.x >= rblocks * ngroups) return;
    }
  }
  const int rb = blockIdx.x % rblocks;        // request block of this CTA
  const int group = blockIdx.x / rblocks;     // vocabulary-tile group
  const int katoms = p.rank / kKAtom;

  uint32_t bar_full = sbase + SM::bars;              // [kStages]
  uint32_t bar_empty = bar_full + 8 * kStages;         // [kStages]
  uint32_t bar_acc_full = bar_empty + 8 * kStages;     // [2]
  uint32_t bar_acc_empty = bar_acc_full + 16;          // [2]
  uint32_t bar_a = bar_acc_empty + 16;                 // [1] A rows landed (residual: TMA)
  uint32_t bar_a2 = bar_a + 8;                         // [1] A rows written (draft: epilogue)
  uint32_t bar_ufull = bar_a2 + 8;                     // [kMaxUBoxes]
  uint32_t bar_uempty = bar_ufull + 8 * kMaxUBoxes;    // [kMaxUBoxes]
  uint32_t bar_mma_drain = bar_uempty + 8 * kMaxUBoxes;  // [1] abort path: issued MMAs done
  constexpr int kBarBytes = 8 * (2 * kStages + 7 + 2 * kMaxUBoxes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::bars + kBarBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::bars + kBarBytes + 8);
  // U boxes of a tile: 128/ubox_cols of them, each read by the 16/(128/ubox_cols) warps
  // whose columns fall inside it
  const int uboxes_per_tile = kN / p.ubox_cols;
  const int warps_per_ubox = kEpiWarps / uboxes_per_tile;
  // Ring capacity: a whole number of tiles, so that slot i % n_uboxes is always read by
  // the same warps.  Each of them has consumed the slot's previous fill before it waits
  // for the next one, which keeps every parity wait at most one phase ahead.
  const int n_uboxes = (SM::uboxes / uboxes_per_tile) * uboxes_per_tile;
  const int ubox_bytes = RB * 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full + 8 * b, 1);
      mbar_init(bar_acc_empty + 8 * b, kEpiWarps);
    }
    mbar_init(bar_a, 1);
    mbar_init(bar_a2, 1);
    mbar_init(bar_mma_drain, 1);
    for (int s = 0; s < kMaxUBoxes; ++s) {
      mbar_init(bar_ufull + 8 * s, 1);
      mbar_init(bar_uempty + 8 * s, warps_per_ubox);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // tiles of this CTA: group, group + ngroups, ...
  const int my_tiles = (p.ntiles > group) ? (p.ntiles - group + ngroups - 1) / ngroups : 0;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      // The factor rows (A) are written by the preceding kernel; W2 (B) is an input.
      // So the first ring's worth of W2 stages is issued before waiting for the
      // predecessor, and A right after.
      const uint64_t w2_policy = policy_evict_last();
      const uint64_t a_policy = policy_evict_normal();
      auto load_a = [&]() {
        griddep_wait();
        constexpr int rep = kM / RB;
        mbar_arrive_expect_tx(bar_a, (uint32_t)(kM * p.rank * 2));
        for (int j = 0; j < rep; ++j)
          for (int ka = 0; ka < katoms; ++ka)
            tma_load_2d(sbase + SM::a + ka * (kM * 128) + j * RB * 128, &map_a, bar_a, ka * kKAtom, rb * RB,
                        a_policy);
      };
      const int total = my_tiles * katoms;
      bool a_issued = false;
      bool a_loaded = false;  // an A copy was issued (it must land before the CTA exits)
      int issued = 0;
      int stage = 0;
      uint32_t phase = 0;
      if (MODE == kModeDraft) a_issued = true;  // draft: the epilogue writes A itself
      for (int it = 0; it < total && !*abort_flag; ++it) {
        if (it == kStages && !a_issued) {
          load_a();
          a_issued = a_loaded = true;
        }
        const int t = it / katoms, ka = it % katoms;
        const int v0 = (group + t * ngroups) * kN;
        if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.status, 100)) break;
        if (*abort_flag) break;  // a role gave up while this stage was being released
        const uint32_t dst = sbase + SM::b + stage * kStageBytes;
        mbar_arrive_expect_tx(bar_full + 8 * stage, kStageBytes);
        tma_load_2d(dst, &map_b, bar_full + 8 * stage, v0, ka * kKAtom, w2_policy);
        tma_load_2d(dst + kStageBytes / 2, &map_b, bar_full + 8 * stage, v0 + 64, ka * kKAtom, w2_policy);
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!a_issued && !*abort_flag) {
        load_a();
        a_loaded = true;
      }
      if (*abort_flag) {
        // abort path: the last kStages copies may still be in flight (earlier ones landed
        // before their stage was refilled); let them land before the CTA exits
        for (int i = max(0, issued - kStages); i < issued; ++i)
          mbar_drain(bar_full + 8 * (i % kStages), (uint32_t)(i / kStages) & 1u);
        if (a_loaded) mbar_drain(bar_a, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kM, kN);
      bool ok = mbar_wait(MODE == kModeDraft ? bar_a2 : bar_a, 0, abort_flag, p.status, 200);
      int stage = 0;
      uint32_t phase = 0;
      for (int t = 0; t < my_tiles && ok; ++t) {
        const int buf = t & 1;
        const uint32_t use = (uint32_t)(t >> 1) & 1u;
        if (!mbar_wait(bar_acc_empty + 8 * buf, use ^ 1, abort_flag, p.status, 201)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kN;
        for (int ka = 0; ka < katoms; ++ka) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.status, 202)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_atom = sbase + SM::a + ka * (kM * 128);
          const uint32_t b_stage = sbase + SM::b + stage * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kKAtom / 16; ++kk) {
            // A: K-major rows of 128 B; a 16-deep K step is 32 B further along the row.
            const uint64_t adesc = sw128_desc(a_atom + kk * 32, 16, 1024);
            // B: MN-major; a 16-deep K step is 16 rows (2 KB) further; the two 64-id
            // halves of the tile are 8 KB apart (leading byte offset), 8-row groups of
            // K are 1 KB apart (stride byte offset).
            const uint64_t bdesc = sw128_desc(b_stage + kk * 2048, kStageBytes / 2, 1024);
            mma_bf16(d_tmem, adesc, bdesc, idesc, (ka > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar_empty + 8 * stage);  // frees the ring slot once these MMAs finish
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(bar_acc_full + 8 * buf);
      }
      if (*abort_flag) {
        // abort path: every MMA this thread issued completes before TMEM is released
        mma_commit(bar_mma_drain);
        mbar_drain(bar_mma_drain, 0);
      }
    }
  } else if (warp == 2) {
    // ------------------------------ U producer (draft mode) -------------------
    // U is an input of the round: its boxes stream ahead of the epilogue through a
    // ring of n_uboxes slots, read once (evict-first in L2).
    if (kDraftMath && lane == 0) {
      const uint64_t u_policy = policy_evict_first();
      int total = my_tiles * uboxes_per_tile;
#ifdef DSPARK_TEST_WAIT_LIMIT
      if (p.round == kTestStallRound) total = 0;
#endif
      int issued = 0;
      for (int i = 0; i < total && !*abort_flag; ++i) {
        const int slot = i % n_uboxes;
        const uint32_t ph = (uint32_t)(i / n_uboxes) & 1u;
        if (!mbar_wait(bar_uempty + 8 * slot, ph ^ 1, abort_flag, p.status, 400)) break;
        // an epilogue warp whose wait gave up still releases its slot, possibly with the
        // slot's last copy in flight: never refill after an abort
        if (*abort_flag) break;
        const int t = i / uboxes_per_tile, bx = i % uboxes_per_tile;
        const int v0 = (group + t * ngroups) * kN + bx * p.ubox_cols;
        mbar_arrive_expect_tx(bar_ufull + 8 * slot, (uint32_t)ubox_bytes);
        tma_load_3d(sbase + SM::u + slot * ubox_bytes, &map_u, bar_ufull + 8 * slot, v0, p.k - 1, rb * RB,
                    u_policy);
        ++issued;
      }
      if (*abort_flag)  // abort path: the last ring's worth of boxes may still be in flight
        for (int i = max(0, issued - n_uboxes); i < issued; ++i)
          mbar_drain(bar_ufull + 8 * (i % n_uboxes), (uint32_t)(i / n_uboxes) & 1u);
    }
  } else {
    // ------------------------------ epilogue ----------------------------------
    const int ew = warp - kFirstEpiWarp;   // 0..15
    const int quarter = warp & 3;          // TMEM lane quarter this warp may access
    const int sub = ew >> 2;               // 0..3: which quarter of the replica's columns
    const int row0 = (quarter * 32) % RB;
    const int replica = (quarter * 32) / RB;
    const int r = rb * RB + row0 + lane;
    bool valid = r < p.R;
    constexpr int kPass = RB / 32;         // 8-column passes per tile: 1, 2 or 4
    const int col0 = replica * RB + sub * (RB / 4);  // RB columns per replica, a quarter per warp

    // the residual's positions and normalisers come from the preceding kernel
    if constexpr (MODE != kModeDraft) griddep_wait();
    // draft: position k of every request; residual: row r is compact slot r, request
    // res_req[r] at its rejected position j*; overlap: row r is position r % gamma + 1 of
    // request r / gamma
    int pos = p.k;
    int req = r;
    float lse_q = 0.f, lse_t = 0.f;
    if constexpr (MODE == kModeResidual) {
      valid = valid && r < *reinterpret_cast<const volatile int*>(p.res_nrows);
      req = valid ? p.res_req[r] : 0;
      pos = valid ? p.jstar[req] : 0;
      valid = valid && pos > 0 && pos <= p.gamma;
      if (valid) {
        lse_q = __ldg(p.lse_q + (size_t)req * p.gamma + (pos - 1));
        lse_t = p.lse_t[req];
      }
    }
    int ovl_flat = r;  // overlap: the position's flattened index (its U row and lse_q)
    if constexpr (MODE == kModeOverlap) {
      if (p.ovl_nrows != nullptr) {
        // compact rows: target row t of request req evaluates position t + 1 (t < ell)
        valid = valid && r < *reinterpret_cast<const volatile int*>(p.ovl_nrows);
        req = valid ? __ldg(p.ovl_req + r) : 0;
        const int t = valid ? __ldg(p.ovl_t + r) : 0;
        pos = t + 1;
        valid = valid && t < min(max(__ldg(p.ell + req), 0), p.gamma);
        ovl_flat = req * p.gamma + t;
      } else {
        req = r / p.gamma;
        pos = r % p.gamma + 1;
        if (valid && p.ell != nullptr) valid = pos <= min(max(__ldg(p.ell + req), 0), p.gamma);
      }
      if (valid) {
        lse_q = __ldg(p.lse_q + ovl_flat);
        lse_t = p.lse_t[r];
      }
    }
    Stats st = stats_empty();  // draft: softmax stats + Gumbel-max; residual: ln(p-q)+ + g
    // every mode scales its logits into base 2 (y = z log2(e)): the draft modes keep st.m
    // in base 2 until the merge below, the correction and overlap modes take their
    // normalisers in base 2 too; keys (st.key, fb.key) and st.zsel are natural throughout
    const float zscale = p.inv_temp * kLog2ef;
    const float lse_q2 = lse_q * kLog2ef, lse_t2 = lse_t * kLog2ef;
    float ovl = 0.f;           // overlap only: this thread's sum of min(q, p)
    const PhiloxRowWords prow =
        philox_row_words(rng_row(p.seed, (MODE != kModeOverlap && valid) ? __ldg(p.req_id + req) : 0, p.round,
                           kDraftMath ? kStreamDraft : kStreamCorrect, (uint32_t)pos));
    const bool u_valid = valid;
    const size_t urow = MODE == kModeOverlap
                            ? (size_t)(valid ? ovl_flat : 0) * (size_t)p.V
                            : ((size_t)(u_valid ? req : 0) * p.gamma + (u_valid ? pos - 1 : 0)) * (size_t)p.V;
    const size_t trow =
        (valid ? target_row_index(p.t_off, p.n_trows, p.gamma, req, pos - 1, p.status) : 0) * (size_t)p.V;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;

    // Residual and overlap modes: U of the next tile is loaded into registers while the
    // current one is processed (each request reads its own position), and with 32-request
    // blocks the target run too (larger blocks have no registers to spare for it).  Draft
    // mode: U arrives through the TMA ring; this warp reads box my_box of each tile, from
    // column box_col on.
    uint4 unext[kPass][2];
    constexpr bool kTPref = !kDraftMath && RB == 32;
    uint4 tnext[kPass][2];
    auto load_t = [&](int t, uint4 (&dst)[kPass][2]) {
      const int vt = (group + t * ngroups) * kN;
#pragma unroll
      for (int ps = 0; ps < kPass; ++ps)
        load_run8(p.target, p.dtype_t, trow, vt + col0 + ps * kCols, p.V, valid && t < my_tiles, dst[ps]);
    };
    auto load_u = [&](int t, uint4 (&dst)[kPass][2]) {
      const int vt = (group + t * ngroups) * kN;
#pragma unroll
      for (int ps = 0; ps < kPass; ++ps)
        load_run8(p.U, p.dtype_u, urow, vt + col0 + ps * kCols, p.V, u_valid && t < my_tiles, dst[ps]);
    };
    // Residual mode with 64- and 128-request blocks: the U and target runs of this thread
    // (run k = pass k % kPass of tile k / kPass) stream through a two-run register ring,
    // each loaded two runs ahead of its use
    constexpr bool kRing = MODE == kModeResidual && kPass % 2 == 0;
    uint4 ring_u[2][2], ring_t[2][2];
    auto load_run = [&](int k, uint4 (&du)[2], uint4 (&dt)[2]) {
      const int tk = k / kPass, pk = k % kPass;
      const int vk = (group + tk * ngroups) * kN + col0 + pk * kCols;
      const bool ok = valid && tk < my_tiles;
      load_run8(p.U, p.dtype_u, urow, vk, p.V, ok, du);
      load_run8(p.target, p.dtype_t, trow, vk, p.V, ok, dt);
    };
    const int my_box = col0 / p.ubox_cols;
    const int box_col = col0 % p.ubox_cols;
    const int box_row = row0 + lane;
    const bool u_f32 = p.dtype_u == DSPARK_F32;
    if constexpr (kRing) {
      load_run(0, ring_u[0], ring_t[0]);
      load_run(1, ring_u[1], ring_t[1]);
    } else if constexpr (!kDraftMath) {
      load_u(0, unext);
    }
    if constexpr (kTPref) load_t(0, tnext);
    // the predecessor still reads the partial records this kernel overwrites at the end
    if constexpr (MODE == kModeDraft) {
      griddep_wait();
      // A rows of this position: W1[x_{k-1}] for the request block, x_{k-1} from x0 or
      // the previous position's winner.  Warp ew takes rows ew, ew + 16, ...: lane i loads
      // row i's token, then every lane loads its 16-byte chunk of every row at once (two
      // dependent loads per warp, not two per row), and moves it into the 128-byte
      // swizzled K-atom rows of every replica (lane l: chunk l, rank <= 256).  Group-0
      // CTAs also write c_k.
      const int et0 = threadIdx.x - 32 * kFirstEpiWarp;
      constexpr int kRowsW = RB / kEpiWarps;  // 2, 4 or 8 rows per warp
      int tok = 0;
      if (lane < kRowsW) {
        const int rq = rb * RB + ew + lane * kEpiWarps;
        if (rq < p.R) {
          const int raw = p.k == 1 ? __ldg(p.x0 + rq) : (int)~(uint32_t)(__ldcg(p.win_prev + rq) & 0xFFFFFFFFull);
          tok = checked_token(raw, p.V, p.status, 3);
        }
      }
      const bool has = lane * 8 < p.rank;
      uint4 qa[kRowsW];
#pragma unroll
      for (int i = 0; i < kRowsW; ++i) {
        const int xp = __shfl_sync(0xffffffffu, tok, i);
        const int rq = rb * RB + ew + i * kEpiWarps;
        qa[i] = make_uint4(0u, 0u, 0u, 0u);
        if (rq < p.R && has)
          qa[i] = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(p.W1) +
                                                        (size_t)xp * p.rank) + lane);
      }
      float we[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) we[e] = (group == 0 && has) ? __ldg(p.w_e + lane * 8 + e) : 0.f;
#pragma unroll
      for (int i = 0; i < kRowsW; ++i) {
        const int rr = ew + i * kEpiWarps;
        const int rq = rb * RB + rr;
        const uint4 q = qa[i];
        if (has) {
          const int ka = lane >> 3, c = lane & 7;
          const uint32_t dst = sbase + SM::a + ka * (kM * 128) + rr * 128 + ((c ^ (rr & 7)) << 4);
#pragma unroll
          for (int j = 0; j < kM / RB; ++j)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + j * RB * 128), "r"(q.x), "r"(q.y),
                         "r"(q.z), "r"(q.w)
                         : "memory");
        }
        if (group == 0 && rq < p.R) {
          const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc = fmaf(we[2 * e], bf16_bits_to_float(wd[e] & 0xFFFFu), acc);
            acc = fmaf(we[2 * e + 1], bf16_bits_to_float(wd[e] >> 16), acc);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
          if (lane == 0) {
            const size_t row = (size_t)rq * p.gamma + (p.k - 1);
            const float logit = p.conf_scale * (p.s_h[row] + acc + p.conf_b);
            p.conf_out[row] = sigmoidf_dev(logit / __ldg(p.conf_temp + (p.k - 1)));
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // read next by the tensor cores
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      if (et0 == 0) mbar_arrive(bar_a2);
    }

    // Draft mode: the best key any CTA has published for this request at this position.
    // Every published value is the key of an actual element, so it is a lower bound of
    // the final winner's key and elements that cannot reach it can be skipped.
    float published = -INFINITY;
    float bound = -INFINITY;

    for (int t = 0; t < my_tiles; ++t) {
      const int buf = t & 1;
      const uint32_t use = (uint32_t)(t >> 1) & 1u;
      const int vt = (group + t * ngroups) * kN;
      // the best key published for this request so far (an order-preserving int code)
      const int hint_pref =
          ((kDraftMath || MODE == kModeResidual) && valid) ? __ldcg(p.hint + r) : (int)(0xFF800000u ^ 0x7FFFFFFFu);
      // residual mode: the race's bound for this tile (own record aside)
      const float tile_bound = fmaxf(bound, key_from_ordered(hint_pref));
      uint4 ucur[kPass][2];
      uint4 tcur[kPass][2];
      int uslot = 0;
      bool u_ready = true;
      if constexpr (kRing) {
        // runs come from the ring, pass by pass
      } else if constexpr (!kDraftMath) {
#pragma unroll
        for (int ps = 0; ps < kPass; ++ps) {
          ucur[ps][0] = unext[ps][0];
          ucur[ps][1] = unext[ps][1];
        }
        load_u(t + 1, unext);
        if constexpr (kTPref) {
#pragma unroll
          for (int ps = 0; ps < kPass; ++ps) {
            tcur[ps][0] = tnext[ps][0];
            tcur[ps][1] = tnext[ps][1];
          }
          load_t(t + 1, tnext);
        }
      } else {
        const int i = t * uboxes_per_tile + my_box;
        uslot = i % n_uboxes;
        u_ready = mbar_wait(bar_ufull + 8 * uslot, (uint32_t)(i / n_uboxes) & 1u, abort_flag, p.status, 301);
        // this thread's 8-id runs from its request row of the 128B-swizzled box
        const uint32_t row_addr = sbase + SM::u + uslot * ubox_bytes + box_row * 128;
#pragma unroll
        for (int ps = 0; ps < kPass; ++ps) {
          const int cb = box_col + ps * kCols;
          if (!u_ready) {
            ucur[ps][0] = ucur[ps][1] = make_uint4(0u, 0u, 0u, 0u);
          } else if (u_f32) {
            const int c0 = cb >> 2;  // two 16-byte chunks
            ucur[ps][0] = lds128(row_addr + ((c0 ^ (box_row & 7)) << 4));
            ucur[ps][1] = lds128(row_addr + (((c0 + 1) ^ (box_row & 7)) << 4));
          } else {
            const int c0 = cb >> 3;  // one 16-byte chunk
            ucur[ps][0] = lds128(row_addr + ((c0 ^ (box_row & 7)) << 4));
            ucur[ps][1] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        // the box slot can be refilled once every reader has its values in registers
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_uempty + 8 * uslot);
      }
      // On an abandoned wait the warp keeps iterating without touching TMEM, so that
      // every epilogue warp still meets the same named barriers.
      const bool acc_ready = mbar_wait(bar_acc_full + 8 * buf, use, abort_flag, p.status, 300) && u_ready;
      if (acc_ready) tc_fence_after();
      // the bound published so far, read at the start of this tile (its latency hides
      // behind the tile's logits; it is first needed by the race)
      if constexpr (kDraftMath) draft_tile(p, st, prow, ucur, tmem_base + lane_addr + buf * kN + col0, acc_ready, valid,
                                           vt + col0, zscale, fmaxf(bound, key_from_ordered(hint_pref)),
                                           bar_acc_empty + 8 * buf, lane);
#pragma unroll
      for (int ps = 0; ps < kPass; ++ps) {
        if (kDraftMath || !acc_ready) break;
        const int c = col0 + ps * kCols;
        float bias[kCols];
        tmem_ld8(tmem_base + lane_addr + buf * kN + c, bias);
        if (ps == kPass - 1) {
          // all of this warp's columns are in registers: hand the accumulator back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acc_empty + 8 * buf);
        }
        const int vb = vt + c;
        float z[kCols];
        float tl[kCols];  // ring: this run's target logits, decoded before the slot is refilled
        if constexpr (kRing) {
          decode_run8(p.dtype_u, ring_u[ps & 1], z);
          decode_run8(p.dtype_t, ring_t[ps & 1], tl);
          load_run(t * kPass + ps + 2, ring_u[ps & 1], ring_t[ps & 1]);
        } else {
          decode_run8(p.dtype_u, ucur[ps], z);
        }
        if (!valid || vb >= p.V) continue;
#pragma unroll
        for (int i = 0; i < kCols; ++i) z[i] = (z[i] + bias[i]) * zscale;
        if constexpr (MODE == kModeOverlap) {
          // overlap: min(q, p) with q = exp(z - lse_q), p = exp(t/T - lse_t) (as powers of 2)
          uint4 traw[2];
          if constexpr (kTPref) {
            traw[0] = tcur[ps][0];
            traw[1] = tcur[ps][1];
          } else {
            load_run8(p.target, p.dtype_t, trow, vb, p.V, true, traw);
          }
          float tl[kCols];
          decode_run8(p.dtype_t, traw, tl);
#pragma unroll
          for (int i = 0; i < kCols; ++i)
            ovl += fminf(ex2_approx(fmaf(tl[i], zscale, -lse_t2)), ex2_approx(z[i] - lse_q2));
        } else {
          // residual: q = exp(z - lse_q), p = exp(t/T - lse_t); draw from (p - q)+ by
          // Gumbel-max over ln(p - q) where positive.  (A row with no positive p - q, which
          // only rounding can produce, is drawn from p by the fallback pass.)
          float lp[kCols];
          if constexpr (kRing) {
#pragma unroll
            for (int i = 0; i < kCols; ++i) lp[i] = tl[i];
          } else {
            uint4 traw[2];
            if constexpr (kTPref) {
              traw[0] = tcur[ps][0];
              traw[1] = tcur[ps][1];
            } else {
              load_run8(p.target, p.dtype_t, trow, vb, p.V, true, traw);
            }
            decode_run8(p.dtype_t, traw, lp);
          }
          float gmax = -INFINITY;
#pragma unroll
          for (int i = 0; i < kCols; ++i) {
            lp[i] = fmaf(lp[i], zscale, -lse_t2);
            gmax = fmaxf(gmax, lp[i]);
          }
          const float gtop = fmaf(gmax, kLn2f, kGumbelMax);
          // the best key known: own record, or the best any CTA has published for this slot
          const float thr = fmaxf(st.idx >= 0 ? st.key : -INFINITY, tile_bound);
          // ln(p - q) <= ln p: no draw of the run can improve once ln p + G_max is below it
          if (thr > -INFINITY && gtop < thr) continue;
          // rejection scale: a key ln rho + g beats best only if 1-u < rho e^{-best}; the test
          // in its conversion-free form (without any key yet the scale is infinite and every
          // id with rho > 0 is keyed)
          const float s1 = (thr > -INFINITY) ? __expf(-thr) * kRejectSlack : INFINITY;
          uint32_t wd[kCols];
          float rho[kCols];
          uint32_t cand = 0;
#pragma unroll
          for (int g4 = 0; g4 < 2; ++g4) {
            const Philox4 bits = prow.block((uint32_t)((vb >> 2) + g4), p.keys);
            wd[4 * g4 + 0] = bits.x;
            wd[4 * g4 + 1] = bits.y;
            wd[4 * g4 + 2] = bits.z;
            wd[4 * g4 + 3] = bits.w;
          }
#pragma unroll
          for (int i = 0; i < kCols; ++i) {
            rho[i] = ex2_approx(lp[i]) - ex2_approx(z[i] - lse_q2);
            if (rho[i] > 0.f && fmaf(rho[i], s1, uniform_mantissa(wd[i])) > kRejectEdge) cand |= 1u << i;
          }
          while (cand) {
            const int i = __ffs(cand) - 1;
            cand &= cand - 1;
            float ri = 0.f;
            uint32_t wi = 0u;
#pragma unroll
            for (int j = 0; j < kCols; ++j)  // static register selection (no local memory)
              if (j == i) {
                ri = rho[j];
                wi = wd[j];
              }
            const float k1 = ln_fast(ri) + gumbel_fast_from_bits(wi);
            if (st.idx < 0 || k1 > st.key) {
              st.key = k1;
              st.idx = vb + i;
            }
          }
        }
      }
      if constexpr (kDraftMath || MODE == kModeResidual) {
        // After the first tiles, publish the CTA's best key per request (residual mode: per
        // slot), one atomic per request per CTA, so that CTAs still streaming can reject more
        // of their draws without evaluating them.
        if (t < publish_tiles<RB>()) {
          float* pub = reinterpret_cast<float*>(smem + SM::pub);
          pub[ew * 32 + lane] = (valid && st.idx >= 0) ? st.key : -INFINITY;
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
          const int et = threadIdx.x - 32 * kFirstEpiWarp;
          if (et < RB && rb * RB + et < p.R) {
            float best = -INFINITY;
            for (int w2 = 0; w2 < kEpiWarps; ++w2) {
              const int r0 = (((w2 + kFirstEpiWarp) & 3) * 32) % RB;
              if (et >= r0 && et < r0 + 32) best = fmaxf(best, pub[w2 * 32 + (et - r0)]);
            }
            if (best > published) {
              atomicMax(p.hint + rb * RB + et, ordered_key(best));
              published = best;
            }
          }
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
        }
        // the bound for the next tile
        if (valid) bound = key_from_ordered(hint_pref);
      }
    }
    if constexpr (kDraftMath) st.m *= kLn2f;  // back to natural units
    // merge the threads that share a request: smem slots [ew][lane]
    Partial* red = reinterpret_cast<Partial*>(smem + SM::red);
    const int et = threadIdx.x - 32 * kFirstEpiWarp;  // 0..511
    if constexpr (MODE == kModeOverlap) {
      // the warps holding a row add their sums in a fixed order (deterministic)
      float* redf = reinterpret_cast<float*>(smem + SM::red);
      redf[ew * 32 + lane] = ovl;
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      if (et < RB) {
        float sum = 0.f;
        for (int w2 = 0; w2 < kEpiWarps; ++w2) {
          const int r0 = (((w2 + kFirstEpiWarp) & 3) * 32) % RB;
          if (et >= r0 && et < r0 + 32) sum += redf[w2 * 32 + (et - r0)];
        }
        const int rr = rb * RB + et;
        if (rr < p.R) p.ovl_part[(size_t)group * p.R + rr] = sum;
      }
    }
#pragma unroll
    for (int which = 0; which < ((kDraftMath || MODE == kModeResidual) ? 1 : 0); ++which) {
      red[ew * 32 + lane] = to_partial(st);
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      if (et < RB) {
        Stats m = stats_empty();
        for (int w2 = 0; w2 < kEpiWarps; ++w2) {
          const int q2 = (w2 + kFirstEpiWarp) & 3;
          const int r0 = (q2 * 32) % RB;
          if (et >= r0 && et < r0 + 32) stats_merge(m, from_partial(red[w2 * 32 + (et - r0)]));
        }
        const int rr = rb * RB + et;
        if constexpr (MODE == kModeResidual) {
          // [group, rblocks * RB] over the slots
          if (rr < *reinterpret_cast<const volatile int*>(p.res_nrows))
            p.partials[(size_t)group * rblocks * RB + rr] = to_partial(m);
        } else if (rr < p.R) {
          p.partials[(size_t)group * p.R + rr] = to_partial(m);
        }
        // draft: this CTA's winner for the request, as one 64-bit maximum (key code in the
        // high half, sign-flipped so that the order is unsigned; ~id in the low half, so the
        // lowest id wins equal keys)
        if (kDraftMath && rr < p.R && m.idx >= 0) {
          const unsigned long long packed =
              ((unsigned long long)((uint32_t)ordered_key(m.key) ^ 0x80000000u) << 32) | (uint32_t)~(uint32_t)m.idx;
          atomicMax(p.win + rr, packed);
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------------------------
// Recurrent head: the hidden-state projection h Wh ([R*gamma, d] x [d, 2*ns]) for every
// position at once, as a plain tensor-core GEMM split over the hidden dimension.
// CTA = (128-row tile, 128-column tile, split); A = h rows (K-major, TMA boxes of 64
// hidden dimensions x 128 rows), B = Wh [d, 2*ns] (MN-major, loaded like W2); the
// fp32 accumulator tile goes from TMEM straight to the split's partial-sum slice.
// Warp 0: TMA producer; warp 1: TMEM allocation + MMA issue; warps 4..7: epilogue
// (warp w reads TMEM lane quarter w % 4).
// ------------------------------------------------------------------------------------
constexpr int kGemmStages = 4;
constexpr int kGemmStageBytes = kM * 128 + kStageBytes;  // A atom (16 KB) + B slice (16 KB)
constexpr int kGemmThreads = 256;
constexpr int kGemmSmem = kGemmStages * kGemmStageBytes + 256 + 1024;

struct GemmParams {
  int rows, d, n2;
  int katoms;        // ceil(d / 64)
  int per_split;     // K atoms per split
  float* out;        // [nsplit, rows, n2]
  DeviceStatus* status;
};

__global__ void __launch_bounds__(kGemmThreads, 1)
    hproj_tc_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                    GemmParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x, nt = blockIdx.y, sp = blockIdx.z;
  const int ka0 = sp * p.per_split;
  const int nk = max(0, min(p.per_split, p.katoms - ka0));
  const uint32_t bar_full = sbase + kGemmStages * kGemmStageBytes;
  const uint32_t bar_empty = bar_full + 8 * kGemmStages;
  const uint32_t bar_acc = bar_empty + 8 * kGemmStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kGemmStages * kGemmStageBytes + 8 * (2 * kGemmStages + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kN);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_allow_next();

  if (warp == 0) {
    if (lane == 0) {
      // h and Wh are inputs of the call: nothing earlier in the stream writes them
      const uint64_t pol = policy_evict_normal();
      for (int i = 0; i < nk && !*abort_flag; ++i) {
        const int s = i % kGemmStages;
        const uint32_t ph = (uint32_t)(i / kGemmStages) & 1u;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort_flag, p.status, 500)) break;
        const uint32_t dst = sbase + s * kGemmStageBytes;
        mbar_arrive_expect_tx(bar_full + 8 * s, (uint32_t)kGemmStageBytes);
        const int k0 = (ka0 + i) * kKAtom;
        tma_load_2d(dst, &map_h, bar_full + 8 * s, k0, mt * kM, pol);
        tma_load_2d(dst + kM * 128, &map_w, bar_full + 8 * s, nt * kN, k0, pol);
        tma_load_2d(dst + kM * 128 + kStageBytes / 2, &map_w, bar_full + 8 * s, nt * kN + 64, k0, pol);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kM, kN);
      bool ok = true;
      for (int i = 0; i < nk; ++i) {
        const int s = i % kGemmStages;
        const uint32_t ph = (uint32_t)(i / kGemmStages) & 1u;
        if (!mbar_wait(bar_full + 8 * s, ph, abort_flag, p.status, 501)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_st = sbase + s * kGemmStageBytes;
        const uint32_t b_st = a_st + kM * 128;
#pragma unroll
        for (int kk = 0; kk < kKAtom / 16; ++kk) {
          const uint64_t adesc = sw128_desc(a_st + kk * 32, 16, 1024);
          const uint64_t bdesc = sw128_desc(b_st + kk * 2048, kStageBytes / 2, 1024);
          mma_bf16(tmem_base, adesc, bdesc, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar_empty + 8 * s);
      }
      if (ok) mma_commit(bar_acc);
    }
  } else if (warp >= 4) {
    const int quarter = warp & 3;
    const bool ready = nk > 0 && mbar_wait(bar_acc, 0, abort_flag, p.status, 502);
    if (ready) tc_fence_after();
    // the partial sums overwrite what the previous call's cells read
    griddep_wait();
    const int row = mt * kM + quarter * 32 + lane;
    float* out = p.out + ((size_t)sp * p.rows + row) * p.n2 + nt * kN;
    for (int c = 0; c < kN; c += kCols) {
      float v[kCols];
      if (ready) {
        tmem_ld8(tmem_base + ((uint32_t)(quarter * 32) << 16) + c, v);
      } else {
#pragma unroll
        for (int e = 0; e < kCols; ++e) v[e] = 0.f;
      }
      if (row < p.rows) {
        reinterpret_cast<float4*>(out + c)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(out + c)[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kN);
  }
}

// ------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

static bool make_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                        uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// U as a 3-D tensor [R][gamma][V] (fp32 or bf16): boxes of 128 bytes of ids by `rows`
// request rows at one position.
static bool make_map_u(CUtensorMap* map, const void* base, int dtype, uint64_t V, uint64_t gamma, uint64_t R,
                       uint32_t rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const uint64_t es = dtype == DSPARK_F32 ? 4 : 2;
  cuuint64_t dims[3] = {V, gamma, R};
  cuuint64_t strides[2] = {V * es, gamma * V * es};
  cuuint32_t box[3] = {(cuuint32_t)(128 / es), 1, rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype == DSPARK_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int num_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
  return sms;
}

static int block_rows(int R) { return R <= 32 ? 32 : (R <= 64 ? 64 : 128); }

}  // namespace tc

int tc_supported(int V, int rank, int dtype_w) {
  return dtype_w == DSPARK_BF16 && rank % tc::kKAtom == 0 && rank >= tc::kKAtom && rank <= tc::kMaxRank &&
         V % 8 == 0 && V >= tc::kN;
}

int tc_num_partials(int R) {
  const int Rb = tc::block_rows(R);
  const int rblocks = (R + Rb - 1) / Rb;
  const int groups = tc::num_sms() / rblocks;
  return groups > 0 ? groups : 1;
}

int tc_block_rows(int R) { return tc::block_rows(R); }

int tc_residual_grid(int R) {
  // the compact correction pass: every SM, or one CTA per slot block if there are more
  // blocks than SMs (the kernel derives its blocks and groups from the device-side count)
  const int Rb = tc_residual_rows_per_block(R);
  const int rblocks = (R + Rb - 1) / Rb;
  return rblocks > tc::num_sms() ? rblocks : tc::num_sms();
}

int tc_grid_ctas(int R) {
  // compact overlap rows: every SM (the kernel derives its blocks and groups from the row
  // count), or one CTA per request block if there are more blocks than SMs
  const int Rb = tc::block_rows(R);
  const int rblocks = (R + Rb - 1) / Rb;
  return rblocks > tc::num_sms() ? rblocks : tc::num_sms();
}

namespace tc {

static TcParams base_params(int R, int gamma, int V, int rank, int dtype_u, float inv_temp, const void* U,
                            const int64_t* req_id, uint64_t seed, uint64_t round, DeviceStatus* status) {
  TcParams p;
  memset(&p, 0, sizeof p);
  p.R = R;
  p.gamma = gamma;
  p.V = V;
  p.rank = rank;
  p.dtype_u = dtype_u;
  p.Rb = block_rows(R);
  p.rblocks = (R + p.Rb - 1) / p.Rb;
  p.ngroups = tc_num_partials(R);
  p.ntiles = (V + kN - 1) / kN;
  p.inv_temp = inv_temp;
  p.U = U;
  p.req_id = req_id;
  p.seed = seed;
  p.keys = philox_keys(seed);
  p.round = round;
  p.status = status;
  return p;
}

template <int MODE>
static cudaError_t launch(TcParams p, const void* W1g, const void* W2, cudaStream_t s) {
  CUtensorMap map_a, map_b, map_u;
  if (!make_map_2d(&map_a, W1g, (uint64_t)p.rank, (uint64_t)round_up_rows(p.R), kKAtom, (uint32_t)p.Rb))
    return cudaErrorInvalidValue;
  if (!make_map_2d(&map_b, W2, (uint64_t)p.V, (uint64_t)p.rank, 64, kKAtom)) return cudaErrorInvalidValue;
  p.ubox_cols = p.dtype_u == DSPARK_F32 ? 32 : 64;
  if (MODE == kModeDraft || MODE == kModeRnn) {
    if (!make_map_u(&map_u, p.U, p.dtype_u, (uint64_t)p.V, (uint64_t)p.gamma, (uint64_t)p.R, (uint32_t)p.Rb))
      return cudaErrorInvalidValue;
  } else {
    map_u = map_b;  // unused: the residual reads each request's own position directly
  }
  const int smem = (p.Rb == 32 ? Smem<32>::total : (p.Rb == 64 ? Smem<64>::total : Smem<128>::total)) + 1024;
  auto kern = p.Rb == 32 ? draft_step_tc_kernel<32, MODE>
                         : (p.Rb == 64 ? draft_step_tc_kernel<64, MODE> : draft_step_tc_kernel<128, MODE>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = p.grid > 0 ? p.grid : p.ngroups * p.rblocks;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), (size_t)smem, s, map_a, map_b, map_u, p);
}

}  // namespace tc

cudaError_t launch_draft_step_tc(const DraftArgs& a, int k, cudaStream_t s) {
  tc::TcParams p = tc::base_params(a.R, a.gamma, a.V, a.rank, a.dtype_u, a.inv_temp, a.U, a.req_id, a.seed,
                                   a.round, a.status);
  p.k = k;
  p.partials = a.partials + (size_t)(k - 1) * tc_num_partials(a.R) * a.R;
  p.hint = a.hint + (size_t)(k - 1) * a.R;
  p.x0 = a.x0;
  p.win_prev = k >= 2 ? a.win + (size_t)(k - 2) * a.R : nullptr;
  p.win = a.win + (size_t)(k - 1) * a.R;
  p.W1 = a.W1;
  p.w_e = a.conf_w + a.d;
  p.s_h = a.s_h;
  p.conf_temp = a.conf_temp;
  p.conf_out = a.conf_out;
  p.conf_b = a.conf_b;
  p.conf_scale = a.conf_scale;
  return tc::launch<tc::kModeDraft>(p, a.W1g, a.W2, s);
}

// Recurrent head: position k with the factor rows (the states s_k) already in a.W1g.
cudaError_t launch_rnn_step_tc(const DraftArgs& a, int k, cudaStream_t s) {
  tc::TcParams p = tc::base_params(a.R, a.gamma, a.V, a.rank, a.dtype_u, a.inv_temp, a.U, a.req_id, a.seed,
                                   a.round, a.status);
  p.k = k;
  p.partials = a.partials + (size_t)(k - 1) * tc_num_partials(a.R) * a.R;
  p.hint = a.hint + (size_t)(k - 1) * a.R;
  p.win = a.win + (size_t)(k - 1) * a.R;
  return tc::launch<tc::kModeRnn>(p, a.W1g, a.W2, s);
}

// The hidden-state projection of the recurrent head takes the tensor cores for bf16 h and
// weights with 2*ns a multiple of 128 and d a multiple of 8 (16-byte TMA rows).
int rnn_hproj_on_tc(int d, int ns, int dtype_w, int dtype_h) {
  return d > 0 && d % 8 == 0 && ns % 64 == 0 && dtype_w == DSPARK_BF16 && dtype_h == DSPARK_BF16;
}

// Splits of the hidden dimension: enough CTAs to cover the GPU (tensor cores), or one per
// 512 hidden dimensions (CUDA cores).
int rnn_num_splits(int R, int gamma, int d, int ns, int dtype_w, int dtype_h) {
  if (d <= 0) return 0;
  if (!rnn_hproj_on_tc(d, ns, dtype_w, dtype_h)) return (d + 511) / 512;
  const int katoms = (d + tc::kKAtom - 1) / tc::kKAtom;
  const int tiles = ((R * gamma + tc::kM - 1) / tc::kM) * (2 * ns / tc::kN);
  const int want = std::max(1, std::min(katoms, (tc::num_sms() + tiles - 1) / tiles));
  const int per = (katoms + want - 1) / want;
  return (katoms + per - 1) / per;
}

cudaError_t launch_rnn_hproj_tc(const DraftArgs& a, cudaStream_t s) {
  const int rows = a.R * a.gamma, n2 = 2 * a.rank;
  CUtensorMap map_h, map_w;
  if (!tc::make_map_2d(&map_h, a.h, (uint64_t)a.d, (uint64_t)rows, tc::kKAtom, tc::kM)) return cudaErrorInvalidValue;
  if (!tc::make_map_2d(&map_w, a.Wh, (uint64_t)n2, (uint64_t)a.d, 64, tc::kKAtom)) return cudaErrorInvalidValue;
  tc::GemmParams p;
  p.rows = rows;
  p.d = a.d;
  p.n2 = n2;
  p.katoms = (a.d + tc::kKAtom - 1) / tc::kKAtom;
  const int nsplit = rnn_num_splits(a.R, a.gamma, a.d, a.rank, a.dtype_w, a.dtype_h);
  if (nsplit != a.nsplit) return cudaErrorInvalidValue;
  p.per_split = (p.katoms + nsplit - 1) / nsplit;
  p.out = a.hpart;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(tc::hproj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       tc::kGemmSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((rows + tc::kM - 1) / tc::kM, n2 / tc::kN, nsplit);
  return launch_pdl(tc::hproj_tc_kernel, grid, dim3(tc::kGemmThreads), (size_t)tc::kGemmSmem, s, map_h, map_w, p);
}

cudaError_t launch_overlap_tc(const OverlapArgs& a, cudaStream_t s) {
  const int rows = a.row_req != nullptr ? a.rows_max : a.R * a.gamma;
  tc::TcParams p = tc::base_params(rows, a.gamma, a.V, a.rank, a.dtype_u, a.inv_temp, a.U, nullptr, 0, 0, a.status);
  p.k = 1;
  p.target = a.target;
  p.dtype_t = a.dtype_t;
  p.lse_q = a.lse_q;
  p.lse_t = a.lse_t;
  p.ell = a.ell;
  p.ovl_part = a.part;
  if (a.row_req != nullptr) {
    p.ovl_req = a.row_req;
    p.ovl_t = a.row_t;
    p.ovl_nrows = a.n_rows;
    p.grid = tc_grid_ctas(rows);
  }
  return tc::launch<tc::kModeOverlap>(p, a.W1g, a.W2, s);
}

cudaError_t launch_residual_tc(const VerifyArgs& a, cudaStream_t s) {
  tc::TcParams p = tc::base_params(a.R, a.gamma, a.V, a.rank, a.dtype_u, a.inv_temp, a.U, a.req_id, a.seed,
                                   a.round, a.status);
  p.k = 1;
  p.partials = a.res_part;
  p.partials2 = a.res_part2;
  p.target = a.target;
  p.t_off = a.t_off;
  p.n_trows = a.n_trows;
  p.dtype_t = a.dtype_t;
  p.jstar = a.jstar;
  p.lse_q = a.lse_q;
  p.lse_t = a.lse_t;
  p.res_req = a.rej_req;
  p.res_nrows = a.n_rej;
  p.hint = a.res_hint;
  p.grid = a.res_grid;
  p.Rb = tc_residual_rows_per_block(a.R);
  p.rblocks = (a.R + p.Rb - 1) / p.Rb;
  return tc::launch<tc::kModeResidual>(p, a.W1g, a.W2, s);
}

}  // namespace dspark
