// Device helpers shared by the NVFP4 kernels (sm_103a): format encoders/decoders written from
// the E2M1/E4M3 definitions, and thin inline-PTX wrappers (mbarrier, bulk async copy, warp MMA,
// conversions).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kv_nvfp4.h"

namespace kvnvfp4 {

constexpr int kHeadDim = 128;
constexpr int kPage = 64;
constexpr int kCodeBytes = 64;   // 128 x 4 bit
constexpr int kScaleBytes = 8;   // 128 / 16 E4M3 scales

// Byte offset, within a page block of Hkv heads, of the four K block scales of k-half kh (blocks
// 4 kh .. 4 kh + 3, dims 64 kh .. 64 kh + 63) of slot `key` of KV head h. The K scales are kept in
// the order the tensor core's scale-factor copy reads them: for each head pair and k-half, 32
// rows of 16 bytes, row r holding keys r and r + 32 of the pair's first head, then of its second
// head. A last unpaired head (odd head count) has 8-byte rows (keys r and r + 32).
__host__ __device__ __forceinline__ int kscale_offset(int Hkv, int h, int key, int kh) {
  const int pr = h >> 1, r = key & 31, kk = key >> 5;
  const int base = Hkv * 4096 + pr * 1024;
  if (2 * pr + 1 < Hkv) return base + kh * 512 + r * 16 + (h & 1) * 8 + kk * 4;
  return base + kh * 256 + r * 8 + kk * 4;
}

// ---------------------------------------------------------------------------------------------
// Formats. E4M3 ("fn"): bias 7, subnormal step 2^-9, max finite 448 (0x7E). E2M1: bias 1, values
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
// ---------------------------------------------------------------------------------------------

// Exact value of a non-NaN E4M3 code with the sign bit clear.
__device__ __forceinline__ float e4m3_decode_pos(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  if (e == 0u) return __fmul_rn((float)m, 0.001953125f);  // m * 2^-9, exact
  return __uint_as_float(((e + 120u) << 23) | (m << 20));  // 2^(e-7) * (1 + m/8)
}

// Two f32 -> two E2M1 codes with the sm_100-family converter: round to nearest, ties to the even
// code, saturating at 6, sign kept (a negative value that rounds to zero gives the negative-zero
// code 8). a goes to bits 4..7, b to bits 0..3.
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float a, float b) {
  uint32_t r;
  asm("{\n.reg .b8 d;\ncvt.rn.satfinite.e2m1x2.f32 d, %1, %2;\ncvt.u32.u8 %0, d;\n}"
      : "=r"(r)
      : "f"(a), "f"(b));
  return r;
}

// Two f32 >= 0 -> two E4M3 codes with the converter: round to nearest, ties to even, saturating at
// 448 (0x7E). a goes to bits 8..15, b to bits 0..7.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float a, float b) {
  uint32_t r;
  asm("{\n.reg .b16 d;\ncvt.rn.satfinite.e4m3x2.f32 d, %1, %2;\ncvt.u32.u16 %0, d;\n}"
      : "=r"(r)
      : "f"(a), "f"(b));
  return r;
}

// x / b rounded to nearest from r = the correctly rounded 1 / b: q0 = x r, then one correction
// with the exact residual x - q0 b (Markstein's division step). The result is the correctly
// rounded quotient whenever that is a normal number; a subnormal quotient may be off by an ulp,
// which moves no E4M3 or E2M1 code (it is far below their smallest rounding threshold).
__device__ __forceinline__ float div_rn_by(float x, float b, float r) {
  const float q0 = __fmul_rn(x, r);
  const float res = __fmaf_rn(-q0, b, x);
  return __fmaf_rn(res, r, q0);
}

// x / b rounded to nearest, sign of x kept (a negative zero stays negative), from r = the correctly
// rounded 1 / b: the same Markstein step as div_rn_by with the residual's sign flipped,
// q0 = x r, e = q0 b - x (exact), q = q0 - e r. For x = -0 the last step adds -0 to -0, so the
// quotient is -0 and needs no separate sign fix. Correctly rounded whenever the quotient is normal.
__device__ __forceinline__ float quot_rn(float x, float b, float r) {
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(q0, b, -x);
  return __fmaf_rn(-e, r, q0);
}

// Eight f32 -> eight E2M1 codes (element 0 in the low nibble) with the hardware converter, packed
// into one word.
__device__ __forceinline__ uint32_t e2m1x8_from_f32(const float (&q)[8]) {
  uint32_t r;
  asm("{\n.reg .b8 b0, b1, b2, b3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}

// This lane's RoPE factors for a row at angle-table row `rope_row` (cos of its 4 dims, then sin):
// lanes below rot/4 hold dims of a rotated pair, the others (and a null row) get zeros. Kept apart
// from the encode so that a caller can issue the loads of several rows before any arithmetic.
__device__ __forceinline__ void rope_fetch(const float* rope_row, int rot, int lane, float4& c,
                                           float4& s) {
  c = make_float4(0.f, 0.f, 0.f, 0.f);
  s = c;
  const int half_lanes = rot >> 3;  // lanes holding dims [0, rot/2)
  if (rope_row != nullptr && lane < 2 * half_lanes) {
    const int i0 = 4 * (lane < half_lanes ? lane : lane - half_lanes);
    c = *reinterpret_cast<const float4*>(rope_row + i0);
    s = *reinterpret_cast<const float4*>(rope_row + (rot >> 1) + i0);
  }
}

// RoPE on the first rot dims of R rows held by a warp (pairs i, i + rot/2; lane l holds elements
// 4l..4l+3), with this lane's factors from rope_fetch. The products are rounded separately and then
// added, as the definition reads.
template <int R>
__device__ __forceinline__ void rope_rows(float (&x)[R][4], const float4 (&c)[R],
                                          const float4 (&s)[R], int rot, int lane) {
  const int half_lanes = rot >> 3;           // lanes holding dims [0, rot/2)
  const bool lower = lane < half_lanes;
  const bool paired = lane < 2 * half_lanes;
  const int src = lower ? lane + half_lanes : lane - half_lanes;
  const float ysg = lower ? -1.0f : 1.0f;
  float y[R][4];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e) y[r][e] = __shfl_sync(0xffffffffu, x[r][e], src & 31);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float cc[4] = {c[r].x, c[r].y, c[r].z, c[r].w};
    const float ss[4] = {s[r].x, s[r].y, s[r].z, s[r].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      // lower lane holds a = x_i, partner b = x_{i+half}: a c - b s
      // upper lane holds b = x_{i+half}, partner a = x_i:  b c + a s
      // (-b) s = -(b s) exactly, so both are one add of two rounded products
      const float v = __fadd_rn(__fmul_rn(x[r][e], cc[e]), __fmul_rn(ysg * y[r][e], ss[e]));
      x[r][e] = paired ? v : x[r][e];
    }
  }
}

// R rows of nvfp4_encode_row, advanced in lockstep (every step taken for all R rows before the
// next), with the RoPE factors already fetched (rope_fetch). Each row goes through exactly the
// operations of the one-row encode, so its codes and scale do not depend on R; the R independent
// chains of shuffles and divisions hide one another's latency. `rope` says whether the rows take
// RoPE at all.
template <int R>
__device__ __forceinline__ void nvfp4_encode_rows(float (&x)[R][4], bool rotate, bool rope,
                                                  const float4 (&c)[R], const float4 (&s)[R],
                                                  int rot, int lane, uint32_t (&packed)[R],
                                                  uint32_t (&sc)[R]) {
  if (rotate) {
    if (rope) rope_rows<R>(x, c, s, rot, lane);
    // --- Walsh-Hadamard, stages h = 1, 2, 4, ..., 64 ---
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float a = x[r][0], b = x[r][1];
      x[r][0] = __fadd_rn(a, b); x[r][1] = __fsub_rn(a, b);
      a = x[r][2]; b = x[r][3];
      x[r][2] = __fadd_rn(a, b); x[r][3] = __fsub_rn(a, b);
      a = x[r][0]; b = x[r][2];
      x[r][0] = __fadd_rn(a, b); x[r][2] = __fsub_rn(a, b);
      a = x[r][1]; b = x[r][3];
      x[r][1] = __fadd_rn(a, b); x[r][3] = __fsub_rn(a, b);
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const float sgn = (lane & m) != 0 ? -1.0f : 1.0f;
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // upper lane: o - x, lower lane: x + o; (+-1) x is exact, so one fma rounds as they do
          const float o = __shfl_xor_sync(0xffffffffu, x[r][e], m);
          x[r][e] = __fmaf_rn(sgn, x[r][e], o);
        }
    }
    const float kNorm = __uint_as_float(0x3DB504F3u);  // rn(2^-3.5) = rn(1/sqrt(128))
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[r][e] = __fmul_rn(x[r][e], kNorm);
  }

  // --- NVFP4: block of 16 = 4 lanes ---
  float amax[R];
#pragma unroll
  for (int r = 0; r < R; ++r)
    amax[r] = fmaxf(fmaxf(fabsf(x[r][0]), fabsf(x[r][1])), fmaxf(fabsf(x[r][2]), fabsf(x[r][3])));
#pragma unroll
  for (int r = 0; r < R; ++r) amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], 1));
#pragma unroll
  for (int r = 0; r < R; ++r) amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], 2));
  // scale = RNE_sat_E4M3(amax / 6), codes = RNE_sat_E2M1(x / scale), each quotient rounded to
  // fp32 first, exactly as the definition reads
  const float r6 = __frcp_rn(6.0f);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    sc[r] = e4m3x2_from_f32(0.0f, div_rn_by(amax[r], 6.0f, r6)) & 0xFFu;
    const float sd = e4m3_decode_pos(sc[r]);
    const float rs = __frcp_rn(sd);
    float q[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) q[e] = quot_rn(x[r][e], sd, rs);
    const uint32_t pk = e2m1x2_from_f32(q[1], q[0]) | (e2m1x2_from_f32(q[3], q[2]) << 8);
    packed[r] = sd != 0.0f ? pk : 0u;  // an all-zero block: zero scale, zero codes
  }
}

__device__ __forceinline__ uint32_t nvfp4_encode_row_fetched(float (&x)[4], bool rotate, bool rope,
                                                             float4 c, float4 s, int rot, int lane,
                                                             uint32_t& sc) {
  float xr[1][4] = {{x[0], x[1], x[2], x[3]}};
  const float4 cr[1] = {c}, sr[1] = {s};
  uint32_t packed[1], scr[1];
  nvfp4_encode_rows<1>(xr, rotate, rope, cr, sr, rot, lane, packed, scr);
  sc = scr[0];
  return packed[0];
}

// One 128-element row held by a warp, lane l holding elements 4l..4l+3, encoded as the method
// prescribes: for Q and K rows (rotate) RoPE on the first `rot` dims (pairs i, i + rot/2, angle
// table row `rope_row`, skipped when null) and the normalised Walsh-Hadamard rotation; then NVFP4
// (E4M3 scale per 16 elements = RNE of amax / 6, E2M1 codes = RNE of x / scale). Every fp32 step
// rounds once, exactly as written (explicit _rn intrinsics). Returns this lane's 4 codes (element
// 4l + e in bits 4e..4e+3) and sets sc to the scale of its 16-element block.
__device__ __forceinline__ uint32_t nvfp4_encode_row(float (&x)[4], bool rotate,
                                                     const float* rope_row, int rot, int lane,
                                                     uint32_t& sc) {
  float4 c, s;
  rope_fetch(rotate ? rope_row : nullptr, rot, lane, c, s);
  return nvfp4_encode_row_fetched(x, rotate, rope_row != nullptr, c, s, rot, lane, sc);
}

// ---------------------------------------------------------------------------------------------
// Conversions via the hardware converters (PTX cvt, sm_100+ family).
// ---------------------------------------------------------------------------------------------

// Four bytes of packed E2M1 pairs -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void cvt_e2m1x8_f16(uint32_t w, uint32_t& r0, uint32_t& r1,
                                               uint32_t& r2, uint32_t& r3) {
  asm("{\n.reg .b8 b0, b1, b2, b3;\n"
      "mov.b32 {b0, b1, b2, b3}, %4;\n"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) -> f16x2.
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16(uint32_t two_bytes) {
  uint32_t r;
  const uint16_t h = (uint16_t)two_bytes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}

// (lo, hi) fp32 -> f16x2, round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Broadcast the low / high f16 of a pair to both halves.
__device__ __forceinline__ uint32_t dup_lo(uint32_t h2) { return __byte_perm(h2, 0, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi(uint32_t h2) { return __byte_perm(h2, 0, 0x3232); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------------------------
// Warp-level MMA m16n8k16 (f16 inputs, f32 accumulate) and the transposing 8x8 b16 matrix load.
// ---------------------------------------------------------------------------------------------
// D += A B for one m16n8k16 tile. Not volatile, so the compiler may interleave independent MMAs
// with the conversions that feed them.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices from shared memory, each transposed on the way (lane 8 m + r gives the
// address of row r of matrix m).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// ---------------------------------------------------------------------------------------------
// Shared-memory access and mbarrier / bulk-copy wrappers.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void sts16(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((uint16_t)v) : "memory");
}
// 8 bytes from global memory through the read-only path.
__device__ __forceinline__ uint2 ldg_nc_u2(const void* ptr) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
                   bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete asks to be suspended for up to
// hint_ns (it resumes as soon as the phase completes), so that waiting warps do not poll the
// barrier and take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity,
                                                      uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete, for at most ~2 s of wall time. Returns
// false on timeout (the caller records KV_NVFP4_DEV_TIMEOUT and carries on).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > 2000000000ull) return false;
  }
}

// A bounded wait that records a timeout and then stops waiting (later waits only poll once), so
// that a kernel whose peer never arrives still runs to its end and reports KV_NVFP4_DEV_TIMEOUT.
__device__ __forceinline__ void wait_bar(uint32_t bar, uint32_t parity, bool& timed_out) {
  if (timed_out) {
    (void)mbar_try_wait(bar, parity);
    return;
  }
  if (!mbar_wait_bounded(bar, parity)) timed_out = true;
}

// wait_bar whose tries suspend the thread (up to 1 ms each) instead of returning at once.
__device__ __forceinline__ void wait_bar_sleep(uint32_t bar, uint32_t parity, bool& timed_out) {
  if (timed_out) {
    (void)mbar_try_wait(bar, parity);
    return;
  }
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_suspend(bar, parity, 1000000u)) {
    if (global_timer_ns() - t0 > 2000000000ull) {
      timed_out = true;
      return;
    }
  }
}

// Bulk (non-tensor) async copy global -> shared, completing on an mbarrier. Both addresses
// 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// An L2 cache policy that marks the lines it touches first for eviction (for data read once and
// streamed through: the KV pages of a decode call).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// The default L2 policy (lines kept as any other), for copies whose lines may be read again.
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void flag_status(int32_t* status, int32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

}  // namespace kvnvfp4

// ---------------------------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core) wrappers: TMEM allocation, MMA issue, commit, TMEM loads
// and stores, and the fences that order them against thread synchronisation.
// ---------------------------------------------------------------------------------------------
namespace kvnvfp4 {

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes become visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor, no swizzle: start address, leading-dimension byte offset
// (stride between core matrices along K), stride-dimension byte offset (along M or N), and the
// descriptor version bit of the sm_100 family.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// D[tmem] (+)= A * B, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A * B, f16 inputs, f32 accumulate, with A read from tensor memory (M rows in the
// lanes, two consecutive K elements per 32-bit column) and B from shared memory.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A * B with E2M1 operands and E4M3 scales, one scale per 16 elements along K.
__device__ __forceinline__ void mma_nvf4_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Arrive once on an mbarrier when every previously issued tcgen05.mma of this thread completes.
// Shared memory -> TMEM copy of a 32-row x 16-byte tile (row i to lane i, four 32-bit columns),
// replicated to all four lane quadrants; ordered before later MMAs issued by the same thread.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// 32 lanes x 8 / 16 consecutive 32-bit columns; lane = thread's lane within its warp quadrant.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 16 columns of zeros.
__device__ __forceinline__ void tmem_st16_zero(uint32_t taddr) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,"
      "%1};" ::"r"(taddr), "r"(0u)
      : "memory");
}
// Wait for this thread's TMEM loads, tying the 32 loaded registers to the wait.
__device__ __forceinline__ void tmem_wait_ld_regs32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
// Named barrier over nthreads threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_barrier_any(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.or.pred p, %2, %3, q;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}
// Wait for this thread's TMEM loads, tying the loaded registers to the wait so that no use of
// them is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}

// Maximum of a float over the 32 lanes of the warp (finite values and -inf).
__device__ __forceinline__ float warp_max_f32(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

}  // namespace kvnvfp4
