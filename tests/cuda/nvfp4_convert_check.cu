// Exhaustive GPU check of the NVFP4 encode helpers used by the kernels (bit_kv_cache_03_gb300/
// csrc/nvfp4_device.cuh) against encoders written here from the format definitions.
//
// Source of the formats: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)":
// E2M1 values {0, 0.5, 1, 1.5, 2, 3, 4, 6} with sign, one E4M3 scale per 16 elements equal to
// amax / 6 rounded, codes = x / scale rounded; rounding to nearest, ties to even, saturating.
//
// Checked, each over every input where the result can differ:
//   1. e2m1x2_from_f32 (hardware converter) against compare-based E2M1 rounding, all 2^32 inputs
//      except NaN, both nibble positions, sign of zero included;
//   2. e4m3x2_from_f32 against compare-based E4M3 rounding, every non-negative non-NaN input;
//   3. the scale code through div_rn_by(amax, 6, 1/6) against the code of __fdiv_rn(amax, 6), every
//      non-negative finite amax;
//   4. div_rn_by(x, s, 1/s) against __fdiv_rn(x, s) (bits and E2M1 code) for all 126 positive
//      E4M3 scales s and every x in [s / 16, 32 s), plus signed zeros and tiny values;
//   5. nvfp4_encode_rows<4> against four calls of nvfp4_encode_rows<1> on random rows;
//   6. quot_rn(x, s, 1/s), the quotient that keeps the sign of x, against __fdiv_rn(x, s) for x and
//      -x over the inputs of check 4, and its E2M1 code for signed zeros and tiny values.
// Prints one "name mismatches N" line per check; exit status 0 when the checks ran.
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

using namespace kvnvfp4;

namespace {

// E4M3 of t >= 0 by the definition: the nearest value of the grid (ties to the even code),
// saturating at 448; subnormal step 2^-9.
__device__ uint32_t e4m3_by_definition(float t) {
  if (!(t > 0.0f)) return 0u;
  if (t >= 448.0f) return 0x7Eu;
  if (t < 0.015625f) return (uint32_t)__float2int_rn(__fmul_rn(t, 512.0f));
  const uint32_t b = __float_as_uint(t);
  const int e = (int)(b >> 23) - 127;
  uint32_t r = (b >> 20) & 7u;
  const uint32_t rem = b & 0xFFFFFu;
  if (rem > 0x80000u || (rem == 0x80000u && (r & 1u))) ++r;
  const uint32_t code = (uint32_t)((e + 7) << 3) + r;
  return code > 0x7Eu ? 0x7Eu : code;
}

// E2M1 of x by the definition: midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5; at a midpoint the
// even code wins; saturating at 6; sign bit of x kept.
__device__ uint32_t e2m1_by_definition(float x) {
  const float a = fabsf(x);
  const uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                     (a >= 3.5f) + (a > 5.0f);
  return c | ((__float_as_uint(x) >> 28) & 8u);
}

constexpr int kChecks = 11;
__device__ unsigned long long g_bad[kChecks];
__device__ unsigned long long g_first[kChecks];

__device__ void bad(int slot, unsigned long long v) {
  if (atomicAdd(&g_bad[slot], 1ull) == 0ull) g_first[slot] = v;
}

__global__ void check_e2m1(unsigned long long n) {
  for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n;
       i += (unsigned long long)gridDim.x * blockDim.x) {
    const float f = __uint_as_float((uint32_t)i);
    if (f != f) continue;
    const uint32_t ref = e2m1_by_definition(f);
    if ((e2m1x2_from_f32(f, 0.0f) >> 4) != ref) bad(0, i);
    if ((e2m1x2_from_f32(0.0f, f) & 15u) != ref) bad(1, i);
  }
}

__global__ void check_e4m3(unsigned long long n) {
  for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n;
       i += (unsigned long long)gridDim.x * blockDim.x) {
    const float f = __uint_as_float((uint32_t)i);  // i < 2^31: sign bit clear
    if (f != f) continue;
    const uint32_t ref = e4m3_by_definition(f);
    if ((e4m3x2_from_f32(f, 0.0f) >> 8) != ref) bad(2, i);
    if ((e4m3x2_from_f32(0.0f, f) & 255u) != ref) bad(3, i);
  }
}

__global__ void check_scale(unsigned long long n) {
  const float r6 = __frcp_rn(6.0f);
  for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n;
       i += (unsigned long long)gridDim.x * blockDim.x) {
    const float amax = __uint_as_float((uint32_t)i);
    if (!(amax <= 3.4028235e38f)) continue;
    const uint32_t ref = e4m3_by_definition(__fdiv_rn(amax, 6.0f));
    if ((e4m3x2_from_f32(0.0f, div_rn_by(amax, 6.0f, r6)) & 255u) != ref) bad(4, i);
  }
}

__global__ void check_quotient(unsigned long long per_scale) {
  const unsigned long long n = per_scale * 126ull;
  for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n;
       i += (unsigned long long)gridDim.x * blockDim.x) {
    const uint32_t code = 1u + (uint32_t)(i / per_scale);
    const float s = e4m3_decode_pos(code);
    const uint32_t b = __float_as_uint(__fmul_rn(s, 0.0625f)) + (uint32_t)(i % per_scale);
    const float x = __uint_as_float(b);
    if (!(x < __fmul_rn(s, 32.0f))) continue;
    const float ref = __fdiv_rn(x, s), got = div_rn_by(x, s, __frcp_rn(s));
    const unsigned long long tag = ((unsigned long long)code << 32) | b;
    if (__float_as_uint(ref) != __float_as_uint(got)) bad(5, tag);
    if (e2m1_by_definition(ref) != (e2m1x2_from_f32(got, 0.0f) >> 4)) bad(6, tag);
    const float rs = __frcp_rn(s);
    if (__float_as_uint(quot_rn(x, s, rs)) != __float_as_uint(ref) ||
        __float_as_uint(quot_rn(-x, s, rs)) != __float_as_uint(__fdiv_rn(-x, s)))
      bad(9, tag);
  }
}

__global__ void check_zeros() {
  const float xs[6] = {0.0f, -0.0f, 1e-45f, -1e-45f, 1e-30f, -1e-30f};
  for (uint32_t code = 1; code <= 126; ++code) {
    const float s = e4m3_decode_pos(code), r = __frcp_rn(s);
    for (int k = 0; k < 6; ++k) {
      const float q = copysignf(div_rn_by(xs[k], s, r), xs[k]);
      if (e2m1_by_definition(__fdiv_rn(xs[k], s)) != (e2m1x2_from_f32(q, 0.0f) >> 4))
        bad(7, code * 8 + k);
      if (e2m1_by_definition(__fdiv_rn(xs[k], s)) !=
          (e2m1x2_from_f32(quot_rn(xs[k], s, r), 0.0f) >> 4))
        bad(10, code * 8 + k);
    }
  }
}

// one warp per 4 rows: rows<4> against rows<1>, rotated with RoPE on 32 dims and unrotated
__global__ void check_rows(const float* in, const float* rope, int nwarps) {
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= nwarps) return;
  for (int rot = 0; rot < 2; ++rot) {
    float x4[4][4];
    float4 c4[4], s4[4];
    for (int r = 0; r < 4; ++r) {
      for (int e = 0; e < 4; ++e) x4[r][e] = in[((w * 4 + r) * 32 + lane) * 4 + e];
      rope_fetch(rope + ((w * 4 + r) & 63) * 32, 32, lane, c4[r], s4[r]);
    }
    uint32_t pk4[4], sc4[4];
    float xc[4][4];
    for (int r = 0; r < 4; ++r)
      for (int e = 0; e < 4; ++e) xc[r][e] = x4[r][e];
    nvfp4_encode_rows<4>(xc, rot != 0, rot != 0, c4, s4, 32, lane, pk4, sc4);
    for (int r = 0; r < 4; ++r) {
      float x1[1][4] = {{x4[r][0], x4[r][1], x4[r][2], x4[r][3]}};
      const float4 c1[1] = {c4[r]}, s1[1] = {s4[r]};
      uint32_t pk1[1], sc1[1];
      nvfp4_encode_rows<1>(x1, rot != 0, rot != 0, c1, s1, 32, lane, pk1, sc1);
      if (pk1[0] != pk4[r] || sc1[0] != sc4[r]) bad(8, (unsigned long long)(w * 4 + r));
    }
  }
}

}  // namespace

int main() {
  const unsigned long long zero[kChecks] = {};
  if (cudaMemcpyToSymbol(g_bad, zero, sizeof(zero)) != cudaSuccess) return 2;
  check_e2m1<<<1216, 256>>>(1ull << 32);
  check_e4m3<<<1216, 256>>>(1ull << 31);
  check_scale<<<1216, 256>>>(1ull << 31);
  check_quotient<<<1216, 256>>>(9ull << 23);
  check_zeros<<<1, 1>>>();
  // random rows (a fixed LCG), values up to +-64 with some exact zeros and negative zeros
  const int nwarps = 1024, nvals = nwarps * 4 * 32 * 4;
  float* h = new float[nvals];
  float* hr = new float[64 * 32];
  uint32_t st = 12345u;
  for (int i = 0; i < nvals; ++i) {
    st = st * 1664525u + 1013904223u;
    const float v = ((float)(st >> 8) / 16777216.0f - 0.5f) * 128.0f;
    h[i] = (i % 97 == 0) ? 0.0f : (i % 89 == 0) ? -0.0f : v;
  }
  for (int i = 0; i < 64 * 32; ++i) {
    st = st * 1664525u + 1013904223u;
    hr[i] = (float)(st >> 8) / 16777216.0f * 2.0f - 1.0f;
  }
  float *d, *dr;
  if (cudaMalloc(&d, nvals * sizeof(float)) != cudaSuccess) return 2;
  if (cudaMalloc(&dr, 64 * 32 * sizeof(float)) != cudaSuccess) return 2;
  cudaMemcpy(d, h, nvals * sizeof(float), cudaMemcpyHostToDevice);
  cudaMemcpy(dr, hr, 64 * 32 * sizeof(float), cudaMemcpyHostToDevice);
  check_rows<<<nwarps / 8, 256>>>(d, dr, nwarps);
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    printf("cuda error %s\n", cudaGetErrorString(e));
    return 2;
  }
  unsigned long long nb[kChecks], fi[kChecks];
  cudaMemcpyFromSymbol(nb, g_bad, sizeof(nb));
  cudaMemcpyFromSymbol(fi, g_first, sizeof(fi));
  const char* names[kChecks] = {"e2m1_hi", "e2m1_lo", "e4m3_hi", "e4m3_lo", "scale_code",
                                "quotient_bits", "quotient_code", "zeros_sign", "rows4_vs_rows1",
                                "signed_quotient_bits", "signed_quotient_zeros"};
  for (int i = 0; i < kChecks; ++i)
    printf("%s mismatches %llu first %#llx\n", names[i], nb[i], nb[i] ? fi[i] : 0ull);
  cudaFree(d);
  cudaFree(dr);
  delete[] h;
  delete[] hr;
  return 0;
}
