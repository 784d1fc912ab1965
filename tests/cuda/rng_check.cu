// Test-only CUDA library: evaluates the device random-number helpers of the DSpark
// kernels next to CUDA's own Philox4x32-10 (curand_Philox4x32_10, a library routine),
// so the tests can compare them bit for bit and check the Gumbel helpers against
// binary64 references.  Not part of the product library.
#include <curand_kernel.h>

#include "../../speculative_decoding_draft_03_gb300/csrc/dspark_common.cuh"

using namespace dspark;

// For each i: counter (c0[i], c1[i], c2[i], c3[i]), key (k0, k1).  Writes 4 words per
// implementation: out[12*i + 0..3] generic rounds, [4..7] row-specialised, [8..11] curand.
__global__ void philox_kernel(int n, const uint32_t* c0, const uint32_t* c1, const uint32_t* c2, const uint32_t* c3,
                              uint32_t k0, uint32_t k1, uint32_t* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const Philox4 a = philox4x32_10(c0[i], c1[i], c2[i], c3[i], k0, k1);
  RngRow row;
  row.k0 = k0;
  row.k1 = k1;
  row.c0 = c0[i];
  row.c1 = c1[i];
  row.c2 = c2[i];
  const Philox4 b = philox_row(row).block(c3[i]);
  const uint4 c = curand_Philox4x32_10(make_uint4(c0[i], c1[i], c2[i], c3[i]), make_uint2(k0, k1));
  uint32_t* o = out + 12 * (size_t)i;
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
  o[8] = c.x; o[9] = c.y; o[10] = c.z; o[11] = c.w;
}

// Gumbel of raw words; and the rejection test for (bits, t).
__global__ void gumbel_kernel(int n, const uint32_t* bits, const float* t, float* g, int* reject) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  g[i] = gumbel_from_bits(bits[i]);
  reject[i] = gumbel_cannot_win(bits[i], t[i]) ? 1 : 0;
}

// The fast Gumbel of the draft epilogue's survivors.
__global__ void gumbel_fast_kernel(int n, const uint32_t* bits, float* g) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  g[i] = gumbel_fast_from_bits(bits[i]);
}

// The draft step's conversion-free rejection test for (bits, t * scale), as the draft
// epilogue evaluates it.
__global__ void reject_fast_kernel(int n, const uint32_t* bits, const float* t, float scale, int* reject) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  reject[i] = (fmaf(t[i], scale, uniform_mantissa(bits[i])) <= kRejectEdge) ? 1 : 0;
}

extern "C" int rng_check_philox(int n, const uint32_t* c0, const uint32_t* c1, const uint32_t* c2, const uint32_t* c3,
                                uint32_t k0, uint32_t k1, uint32_t* out) {
  philox_kernel<<<(n + 255) / 256, 256>>>(n, c0, c1, c2, c3, k0, k1, out);
  return (int)cudaDeviceSynchronize();
}

extern "C" int rng_check_gumbel(int n, const uint32_t* bits, const float* t, float* g, int* reject) {
  gumbel_kernel<<<(n + 255) / 256, 256>>>(n, bits, t, g, reject);
  return (int)cudaDeviceSynchronize();
}

extern "C" int rng_check_reject_fast(int n, const uint32_t* bits, const float* t, float scale, int* reject) {
  reject_fast_kernel<<<(n + 255) / 256, 256>>>(n, bits, t, scale, reject);
  return (int)cudaDeviceSynchronize();
}

extern "C" int rng_check_gumbel_fast(int n, const uint32_t* bits, float* g) {
  gumbel_fast_kernel<<<(n + 255) / 256, 256>>>(n, bits, g);
  return (int)cudaDeviceSynchronize();
}
