// Comparator KV formats for decode attention, for byte-count and roofline comparison with the
// NVFP4 path at the same workloads: bf16 K and V (512 B per token per KV head), int8 K and V with
// one fp32 scale per row (264 B), and the upstream variant with NVFP4 K (no Hadamard rotation) and
// fp16 V (328 B). Each has an append kernel (RoPE on Q and K, then the format's encoding) and a
// decode kernel; the plan, the (m, l, O) partials and the split-K merge are the NVFP4 path's.
//
// Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)": 144 bytes per
// token per KV head against 264 for int8 and 512 for bf16, and the upstream NVFP4 path that keeps
// V in fp16 without outlier suppression (no rotation). Readings: int8 rows use s = amax / 127 (fp32)
// and codes RNE(x / s) clamped to +-127; Q stays unquantised (bf16 after RoPE) in every format.
//
// Page block: one chunk per KV head, in head order; a chunk holds K then V for the page's 64
// slots (row bytes: bf16 / fp16 256, int8 128 + a 4-byte scale, NVFP4 64 + 8):
//   bf16:  [K 64 x 256][V 64 x 256]
//   int8:  [K codes 64 x 128][K scales 64 x 4][V codes 64 x 128][V scales 64 x 4]
//   k4v16: [K codes 64 x 64][K scales 64 x 8][V 64 x 256]
// Within a row, the 16-byte unit u of slot k is stored at unit u ^ sw(k), so that the decode
// kernel's shared-memory reads of 8 or 16 slots at once fall in distinct banks:
//   bf16 K and V, fp16 V:  sw = k & 7        (ldmatrix of 8 slots at one logical unit)
//   int8 K:                sw = (k & 1) << 2 (a lane reads units t and t + 4 of its slot)
//   int8 V:                sw = ((k >> 1) & 3) << 1 (a lane reads unit g of 4 slots 2t ...)
//   NVFP4 K codes and all scales: no swizzle.
//
// Decode kernel: grid (plan CTAs, KV heads), one head per CTA; warp 0 streams the head's chunk of
// each page (one bulk copy) into a stage ring, warps 1..4 each take 16 keys of every page. Q.K^T
// and P.V run on mma.sync m16n8k16 with f32 accumulation (bf16 operands for the bf16 format, f16
// for the others; int8 and NVFP4 values are exact in f16). P is fed as a hi + lo pair in rows 0..7
// and 8..15 of the A operand, so the 16-row M costs nothing extra. The four warps' (m, l, O) are
// merged in shared memory at the end of a segment and written as the output row or a split-K
// partial.

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

cudaError_t launch_split_merge(const void* groups, const int32_t* split_groups,
                               const float* partials, float* out, int32_t Hq, int32_t Hkv,
                               int32_t G, int32_t q_len, float c2, int32_t num_split,
                               bool late_tables, cudaStream_t stream);

namespace {

constexpr int kFmtBf16 = 0, kFmtInt8 = 1, kFmtK4V16 = 2;
constexpr int kCmpCompute = 4;                        // compute warps (16 keys of a page each)
constexpr int kCmpThreads = 32 * (1 + kCmpCompute);
constexpr int kCmpRows = 8;                           // query rows of a plan group
constexpr int kCmpPartFloats = kCmpRows * 128 + 2 * kCmpRows;
constexpr int kCmpStageBudget = 160 * 1024;

template <int FMT> struct Fmt;
template <> struct Fmt<kFmtBf16> {
  static constexpr int kChunk = 32768, kOffKs = 0, kOffV = 16384, kOffVs = 0;
};
template <> struct Fmt<kFmtInt8> {
  static constexpr int kChunk = 16896, kOffKs = 8192, kOffV = 8448, kOffVs = 16640;
};
template <> struct Fmt<kFmtK4V16> {
  static constexpr int kChunk = 20992, kOffKs = 4096, kOffV = 4608, kOffVs = 0;
};

__host__ __device__ constexpr int chunk_bytes(int fmt) {
  return fmt == kFmtBf16 ? 32768 : fmt == kFmtInt8 ? 16896 : 20992;
}

__device__ __forceinline__ int sw_k(int fmt, int k) {
  return fmt == kFmtBf16 ? (k & 7) : fmt == kFmtInt8 ? ((k & 1) << 2) : 0;
}
__device__ __forceinline__ int sw_v(int fmt, int k) {
  return fmt == kFmtInt8 ? (((k >> 1) & 3) << 1) : (k & 7);
}

// ---------------------------------------------------------------------------------------------
// Append: one warp per row (Q, K or V of one token), lane l holding elements 4l..4l+3.
// ---------------------------------------------------------------------------------------------
struct CmpAppendParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* seq_ids;
  const int32_t* positions;
  int64_t T;
  const float* rope;
  int32_t rope_max_pos, rot_dim;
  const int32_t* block_table;
  int32_t num_seqs, max_pages, num_pages;
  uint8_t* pool;
  uint16_t* q_out;  // bf16 [T][Hq][128], RoPE applied
  int32_t Hq, Hkv;  // Hq = 0 when q is absent
  int32_t* status;
};

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}
__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  return (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
         ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

template <int FMT>
__global__ void __launch_bounds__(256) cmp_append_kernel(const CmpAppendParams p) {
  using F = Fmt<FMT>;
  const int lane = threadIdx.x & 31;
  const int64_t per_tok = p.Hq + 2 * p.Hkv;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= p.T * per_tok) return;  // warp-uniform
  const int64_t t = row / per_tok;
  const int w = (int)(row - t * per_tok);
  const int32_t seq = p.seq_ids[t], pos = p.positions[t];
  if (seq < 0 || seq >= p.num_seqs) {
    if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_SEQ);
    return;
  }
  if (pos < 0 || pos >= p.max_pages * kPage) {
    if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_POS);
    return;
  }
  const int kind = w < p.Hq ? 0 : (w - p.Hq < p.Hkv ? 1 : 2);  // Q, K, V
  const int h = kind == 0 ? w : (kind == 1 ? w - p.Hq : w - p.Hq - p.Hkv);
  const uint16_t* src = (kind == 0 ? p.q + (t * p.Hq + h) * kHeadDim
                                   : (kind == 1 ? p.k : p.v) + (t * p.Hkv + h) * kHeadDim);
  uint8_t* chunk = nullptr;
  if (kind != 0) {
    const int32_t page = p.block_table[(int64_t)seq * p.max_pages + pos / kPage];
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_PAGE);
      return;
    }
    chunk = p.pool + ((int64_t)page * p.Hkv + h) * F::kChunk;
  }
  const bool rotate = kind != 2 && p.rot_dim > 0;
  if (rotate && pos >= p.rope_max_pos) {
    if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_ROPE);
    return;
  }
  const uint2 raw = ldg_nc_u2(src + 4 * lane);
  float x[1][4] = {{__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                    __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)}};
  float4 c[1], s[1];
  rope_fetch(rotate ? p.rope + (int64_t)pos * p.rot_dim : nullptr, p.rot_dim, lane, c[0], s[0]);
  if (rotate) rope_rows<1>(x, c, s, p.rot_dim, lane);
  const int slot = pos % kPage;
  if (kind == 0) {  // Q: bf16 of the rotated row
    *reinterpret_cast<uint2*>(p.q_out + (t * p.Hq + h) * kHeadDim + 4 * lane) =
        make_uint2(bf16x2_bits(x[0][0], x[0][1]), bf16x2_bits(x[0][2], x[0][3]));
    return;
  }
  if (FMT == kFmtBf16 || (FMT == kFmtK4V16 && kind == 2)) {  // 16-bit rows, 8 bytes per lane
    const uint2 v2 = FMT == kFmtBf16
                         ? make_uint2(bf16x2_bits(x[0][0], x[0][1]), bf16x2_bits(x[0][2], x[0][3]))
                         : make_uint2(f16x2_bits(x[0][0], x[0][1]), f16x2_bits(x[0][2], x[0][3]));
    const int sw = kind == 1 ? sw_k(FMT, slot) : sw_v(FMT, slot);
    uint8_t* rowp = chunk + (kind == 1 ? 0 : F::kOffV) + slot * 256;
    *reinterpret_cast<uint2*>(rowp + (((lane >> 1) ^ sw) << 4) + (lane & 1) * 8) = v2;
  } else if (FMT == kFmtInt8) {
    float amax = fmaxf(fmaxf(fabsf(x[0][0]), fabsf(x[0][1])), fmaxf(fabsf(x[0][2]), fabsf(x[0][3])));
    amax = warp_max_f32(amax);
    const float sc = __fdiv_rn(amax, 127.0f);
    uint32_t packed = 0;
    if (sc != 0.0f) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int q = __float2int_rn(__fdiv_rn(x[0][e], sc));  // nearest, ties to even
        q = q > 127 ? 127 : (q < -127 ? -127 : q);
        packed |= ((uint32_t)q & 0xFFu) << (8 * e);
      }
    }
    const int sw = kind == 1 ? sw_k(FMT, slot) : sw_v(FMT, slot);
    uint8_t* rowp = chunk + (kind == 1 ? 0 : F::kOffV) + slot * 128;
    *reinterpret_cast<uint32_t*>(rowp + (((lane >> 2) ^ sw) << 4) + (lane & 3) * 4) = packed;
    if (lane == 0)
      *reinterpret_cast<float*>(chunk + (kind == 1 ? F::kOffKs : F::kOffVs) + slot * 4) = sc;
  } else {  // k4v16 K: NVFP4 of the rotated row (no Hadamard)
    uint32_t pk[1], scb[1];
    nvfp4_encode_rows<1>(x, false, false, c, s, p.rot_dim, lane, pk, scb);
    *reinterpret_cast<uint16_t*>(chunk + slot * 64 + 2 * lane) = (uint16_t)pk[0];
    if ((lane & 3) == 0) chunk[F::kOffKs + slot * 8 + (lane >> 2)] = (uint8_t)scb[0];
  }
}

// ---------------------------------------------------------------------------------------------
// Decode
// ---------------------------------------------------------------------------------------------
struct CmpDecodeParams {
  const uint16_t* q;  // bf16 [tokens][Hq][128], RoPE applied
  const uint8_t* pool;
  const int32_t* block_table;
  int32_t max_pages, num_pages;
  const int4* groups;    // 2 x int4 per group: {seq, 0, rg, len}, {n_seg, first_part, pages, 0}
  const int4* segments;  // {group, page_lo, page_hi, part_slot or -1}
  const int32_t* cta_seg;
  float* partials;       // [num_partials][Hkv][kCmpPartFloats]
  float* out;
  int32_t* status;
  int32_t Hq, Hkv, G, q_len, causal;
  float c2;  // sm_scale * log2(e)
};

struct CmpSeg {
  int seq, rg, len, n_seg, lo, hi, part;
};

__device__ __forceinline__ CmpSeg cmp_load_seg(const CmpDecodeParams& p, int s) {
  const int4 seg = p.segments[s];
  const int4 g0 = p.groups[2 * seg.x];
  const int4 g1 = p.groups[2 * seg.x + 1];
  CmpSeg r;
  r.lo = seg.y; r.hi = seg.z; r.part = seg.w;
  r.seq = g0.x; r.rg = g0.z; r.len = g0.w;
  r.n_seg = g1.x;
  return r;
}

template <int FMT>
struct CmpSmem {
  static constexpr int kStages = kCmpStageBudget / Fmt<FMT>::kChunk;
  static constexpr int kOffMergeO = kStages * Fmt<FMT>::kChunk;          // [4 warps][8][128] f32
  static constexpr int kOffMergeML = kOffMergeO + kCmpCompute * kCmpRows * 128 * 4;  // m, l
  static constexpr int kOffPid = kOffMergeML + kCmpCompute * 2 * kCmpRows * 4;
  static constexpr int kOffBars = (kOffPid + kStages * 4 + 7) & ~7;      // full[S], empty[S]
  static constexpr int kBytes = kOffBars + 2 * kStages * 8;
};

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two int8 values (the bytes that sel puts in bytes 0 and 2) -> f16x2, exactly: 1024 + (c + 128) is an f16 with the
// byte as its low mantissa bits; subtracting 1152 leaves c.
__device__ __forceinline__ uint32_t i8x2_f16(uint32_t x, uint32_t sel) {
  const uint32_t b = __byte_perm(x ^ 0x80808080u, 0x64646464u, sel);
  return hsub2(b, 0x64806480u);
}

// Opaque zero (rows 8..15 of an A operand that carry nothing).
__device__ __forceinline__ uint32_t zero_reg() {
  uint32_t z;
  asm volatile("mov.b32 %0, 0;" : "=r"(z));
  return z;
}

template <int FMT>
__device__ void cmp_producer(const CmpDecodeParams& p, uint8_t* smem, int lane) {
  using SM = CmpSmem<FMT>;
  constexpr int S = SM::kStages;
  constexpr uint32_t kChunk = Fmt<FMT>::kChunk;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full0 = sbase + SM::kOffBars, empty0 = full0 + 8 * S;
  volatile int32_t* stage_pid = reinterpret_cast<volatile int32_t*>(smem + SM::kOffPid);
  const int h = blockIdx.y;
  uint32_t k = 0;
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const CmpSeg sg = cmp_load_seg(p, s);
    for (int p0 = sg.lo; p0 < sg.hi; p0 += 32) {
      const int n = min(32, sg.hi - p0);
      const int32_t mine =
          (lane < n) ? p.block_table[(int64_t)sg.seq * p.max_pages + p0 + lane] : -1;
      for (int j = 0; j < n; ++j, ++k) {
        const int32_t pid = __shfl_sync(0xffffffffu, mine, j);
        if (lane == 0) {
          const uint32_t st = k % S;
          if (k >= (uint32_t)S) wait_bar(empty0 + 8 * st, ((k / S) - 1) & 1, timed_out);
          const bool valid = pid >= 0 && pid < p.num_pages;
          stage_pid[st] = valid ? pid : -1;
          if (valid) {
            mbar_arrive_expect_tx(full0 + 8 * st, kChunk);
            bulk_g2s(sbase + st * kChunk, p.pool + ((int64_t)pid * p.Hkv + h) * kChunk, kChunk,
                     full0 + 8 * st);
          } else {
            flag_status(p.status, KV_NVFP4_DEV_BAD_PAGE);
            mbar_arrive(full0 + 8 * st);
          }
        }
        __syncwarp();
      }
    }
  }
  if (lane == 0) {
    for (uint32_t st = 0; st < (uint32_t)S && st < k; ++st) {  // no copy in flight at exit
      const uint32_t last = k - 1 - ((k - 1 - st) % S);
      wait_bar(full0 + 8 * st, (last / S) & 1, timed_out);
    }
    if (timed_out) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
  }
}

// Dims of the A / B fragment k indices {2t, 2t + 1} (the first pair) of k-step d for lane t; the
// second pair {2t + 8, 2t + 9} is the first pair + 8 (bf16) or + 2 (int8, NVFP4 K). The same
// permutation is applied to Q and K, so Q.K^T is unchanged.
template <int FMT>
__device__ __forceinline__ int qk_dim(int d, int t) {
  if (FMT == kFmtBf16) return 16 * d + 2 * t;
  if (FMT == kFmtInt8) return 16 * (t + 4 * (d >> 2)) + 4 * (d & 3);  // units t, t + 4 of a row
  return 32 * t + 4 * d;                                               // code unit t of a row
}
template <int FMT>
__device__ __forceinline__ int qk_dim2(int d, int t) {
  return qk_dim<FMT>(d, t) + (FMT == kFmtBf16 ? 8 : 2);
}

template <int FMT>
__device__ void cmp_compute(const CmpDecodeParams& p, uint8_t* smem, int w, int lane) {
  using F = Fmt<FMT>;
  using SM = CmpSmem<FMT>;
  constexpr int S = SM::kStages;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full0 = sbase + SM::kOffBars, empty0 = full0 + 8 * S;
  const volatile int32_t* stage_pid = reinterpret_cast<const volatile int32_t*>(smem + SM::kOffPid);
  float* mo = reinterpret_cast<float*>(smem + SM::kOffMergeO);
  float* mml = reinterpret_cast<float*>(smem + SM::kOffMergeML);
  const int h = blockIdx.y;
  const int g = lane >> 2, t = lane & 3;
  const int kb = 16 * w;  // this warp's keys within every page
  const int rows_total = p.G * p.q_len;
  const float c2 = p.c2;
  const uint32_t z = zero_reg();
  uint32_t k = 0;
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const CmpSeg sg = cmp_load_seg(p, s);
    const int r = sg.rg * kCmpRows + g;
    const bool rvalid = r < rows_total;
    const int L0 = sg.len - p.q_len;
    const int lim = rvalid ? (p.causal ? L0 + r / p.G : sg.len - 1) : -1;
    // Q fragments of row g for every k-step (rows g + 8 carry nothing)
    uint32_t qa[8][2];
    {
      const uint16_t* qr =
          p.q + (((int64_t)sg.seq * p.q_len + (rvalid ? r / p.G : 0)) * p.Hq + h * p.G +
                 (rvalid ? r % p.G : 0)) * kHeadDim;
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        uint32_t x0 = 0u, x1 = 0u;
        if (rvalid) {
          x0 = *reinterpret_cast<const uint32_t*>(qr + qk_dim<FMT>(d, t));
          x1 = *reinterpret_cast<const uint32_t*>(qr + qk_dim2<FMT>(d, t));
        }
        if (FMT == kFmtBf16) {
          qa[d][0] = x0;
          qa[d][1] = x1;
        } else {  // bf16 -> f16 (exact for |q| in [2^-14, 65504])
          qa[d][0] = f16x2_bits(__uint_as_float(x0 << 16), __uint_as_float(x0 & 0xFFFF0000u));
          qa[d][1] = f16x2_bits(__uint_as_float(x1 << 16), __uint_as_float(x1 & 0xFFFF0000u));
        }
      }
    }
    float m = -INFINITY, l = 0.f;
    float acc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;

    for (int pg = sg.lo; pg < sg.hi; ++pg, ++k) {
      const uint32_t st = k % S;
      wait_bar(full0 + 8 * st, (k / S) & 1, timed_out);
      const int32_t pid = stage_pid[st];
      const uint32_t stage = sbase + st * F::kChunk;
      const uint8_t* stp = smem + st * F::kChunk;
      if (pid >= 0) {
        // ---- scores: 2 n-tiles of 8 keys (kb + 8 jt + g is this lane's B column) ----
        float sc[2][4];
#pragma unroll
        for (int jt = 0; jt < 2; ++jt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[jt][e] = 0.f;
        if (FMT == kFmtBf16) {
          const int mi = lane >> 3, key = kb + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
          for (int d = 0; d < 8; ++d) {
            uint32_t b[4];
            const int u = 2 * d + (mi & 1);
            ldsm_x4(stage + key * 256 + ((u ^ (key & 7)) << 4), b[0], b[1], b[2], b[3]);
            mma_bf16(sc[0], qa[d][0], z, qa[d][1], z, b[0], b[1]);
            mma_bf16(sc[1], qa[d][0], z, qa[d][1], z, b[2], b[3]);
          }
        } else if (FMT == kFmtInt8) {
#pragma unroll
          for (int jt = 0; jt < 2; ++jt) {
            const int key = kb + 8 * jt + g;
            const int sw = (key & 1) << 2;
            const uint4 u0 = lds128(stage + key * 128 + ((t ^ sw) << 4));
            const uint4 u1 = lds128(stage + key * 128 + (((t + 4) ^ sw) << 4));
            const uint32_t wv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int d = 0; d < 8; ++d)
              mma16816(sc[jt], qa[d][0], z, qa[d][1], z, i8x2_f16(wv[d], 0x4140),
                       i8x2_f16(wv[d], 0x4342));
          }
        } else {
#pragma unroll
          for (int jt = 0; jt < 2; ++jt) {
            const int key = kb + 8 * jt + g;
            const uint4 cu = lds128(stage + key * 64 + t * 16);
            const uint16_t sb = *reinterpret_cast<const uint16_t*>(stp + F::kOffKs + key * 8 + 2 * t);
            const uint32_t s2 = cvt_e4m3x2_f16(sb);  // blocks 2t (low half), 2t + 1 (high)
            const uint32_t slo = dup_lo(s2), shi = dup_hi(s2);
            const uint32_t cw[4] = {cu.x, cu.y, cu.z, cu.w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t e0, e1, e2, e3;  // dims 32t + 8 q4 + (0..1 | 2..3 | 4..5 | 6..7)
              cvt_e2m1x8_f16(cw[q4], e0, e1, e2, e3);
              const uint32_t scl = q4 < 2 ? slo : shi;
              mma16816(sc[jt], qa[2 * q4][0], z, qa[2 * q4][1], z, hmul2(e0, scl), hmul2(e1, scl));
              mma16816(sc[jt], qa[2 * q4 + 1][0], z, qa[2 * q4 + 1][1], z, hmul2(e2, scl),
                       hmul2(e3, scl));
            }
          }
        }
        // ---- scale (int8 K), mask, running max and sum, P as hi + lo ----
        float sv[4];  // this lane's keys: kb + 2t, 2t + 1, 2t + 8, 2t + 9 (row g)
        sv[0] = sc[0][0]; sv[1] = sc[0][1]; sv[2] = sc[1][0]; sv[3] = sc[1][1];
        const int kk[4] = {kb + 2 * t, kb + 2 * t + 1, kb + 8 + 2 * t, kb + 9 + 2 * t};
        if (FMT == kFmtInt8) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sv[e] *= *reinterpret_cast<const float*>(stp + F::kOffKs + kk[e] * 4);
        }
        float pm = -INFINITY;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (pg * kPage + kk[e] > lim) sv[e] = -INFINITY;  // causal, page tail, padding row
          pm = fmaxf(pm, sv[e]);
        }
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
        const float mn = fmaxf(m, pm);
        const float alpha = (mn == m) ? 1.f : fast_exp2((m - mn) * c2);  // 0 when m was -inf
        m = mn;
        float pr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pr[e] = sv[e] == -INFINITY ? 0.f : fast_exp2((sv[e] - mn) * c2);
        l = l * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
        if (alpha != 1.f) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] *= alpha;
        }
        if (FMT == kFmtInt8) {  // the V row scales, folded into P
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pr[e] *= *reinterpret_cast<const float*>(stp + F::kOffVs + kk[e] * 4);
        }
        uint32_t a0, a1, a2, a3;  // rows g: P hi; rows g + 8: P lo
        if (FMT == kFmtBf16) {
          a0 = bf16x2_bits(pr[0], pr[1]);
          a2 = bf16x2_bits(pr[2], pr[3]);
          a1 = bf16x2_bits(pr[0] - __uint_as_float(a0 << 16), pr[1] - __uint_as_float(a0 & 0xFFFF0000u));
          a3 = bf16x2_bits(pr[2] - __uint_as_float(a2 << 16), pr[3] - __uint_as_float(a2 & 0xFFFF0000u));
        } else {
          a0 = f16x2_bits(pr[0], pr[1]);
          a2 = f16x2_bits(pr[2], pr[3]);
          const __half2 h0 = *reinterpret_cast<const __half2*>(&a0);
          const __half2 h2 = *reinterpret_cast<const __half2*>(&a2);
          a1 = f16x2_bits(pr[0] - __low2float(h0), pr[1] - __high2float(h0));
          a3 = f16x2_bits(pr[2] - __low2float(h2), pr[3] - __high2float(h2));
        }
        // ---- O += P V ----
        if (FMT == kFmtInt8) {  // lane g takes dims 16 g .. 16 g + 15: tile jj column n = dim 16 n + jj
          uint4 vw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            vw[e] = lds128(stage + F::kOffV + kk[e] * 128 + ((g ^ sw_v(FMT, kk[e])) << 4));
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const uint32_t x0 = (&vw[0].x)[q4], x1 = (&vw[1].x)[q4];
            const uint32_t x2 = (&vw[2].x)[q4], x3 = (&vw[3].x)[q4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {  // dim 16 g + 4 q4 + e: byte e of each key's word
              // byte e of keys 2t and 2t + 1 into bytes 0 and 2, then to an f16 pair (same for
              // keys 2t + 8 and 2t + 9)
              const uint32_t sel = (uint32_t)e | ((uint32_t)(4 + e) << 8);
              const uint32_t b0 = i8x2_f16(__byte_perm(x0, x1, sel), 0x4240);
              const uint32_t b1 = i8x2_f16(__byte_perm(x2, x3, sel), 0x4240);
              mma16816(acc[4 * q4 + e], a0, a1, a2, a3, b0, b1);
            }
          }
        } else {  // 16-bit V rows through transposing ldmatrix; tile j = dims 8 j .. 8 j + 7
          const int mi = lane >> 3, key = kb + (mi & 1) * 8 + (lane & 7);
#pragma unroll
          for (int jp = 0; jp < 8; ++jp) {
            uint32_t b[4];
            const int u = 2 * jp + (mi >> 1);
            ldsm_x4_t(stage + F::kOffV + key * 256 + ((u ^ (key & 7)) << 4), b[0], b[1], b[2], b[3]);
            if (FMT == kFmtBf16) {
              mma_bf16(acc[2 * jp], a0, a1, a2, a3, b[0], b[1]);
              mma_bf16(acc[2 * jp + 1], a0, a1, a2, a3, b[2], b[3]);
            } else {
              mma16816(acc[2 * jp], a0, a1, a2, a3, b[0], b[1]);
              mma16816(acc[2 * jp + 1], a0, a1, a2, a3, b[2], b[3]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
    }

    // ---- segment end: the four warps' (m, l, O) merged per row ----
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    float* myo = mo + (w * kCmpRows + g) * 128;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int dim = FMT == kFmtInt8 ? 16 * (2 * t + c) + j : 8 * j + 2 * t + c;
        myo[dim] = acc[j][c] + acc[j][c + 2];  // hi and lo rows
      }
    }
    if (t == 0) {
      mml[(w * 2) * kCmpRows + g] = m;
      mml[(w * 2 + 1) * kCmpRows + g] = l;
    }
    named_barrier_sync(1, 32 * kCmpCompute);
    {
      // thread i of the 128: row i / 16, dims 8 (i % 16) .. + 7
      const int i = w * 32 + lane, row = i >> 4, d0 = 8 * (i & 15);
      float M = -INFINITY;
#pragma unroll
      for (int v = 0; v < kCmpCompute; ++v) M = fmaxf(M, mml[(v * 2) * kCmpRows + row]);
      float Lsum = 0.f, o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = 0.f;
#pragma unroll
      for (int v = 0; v < kCmpCompute; ++v) {
        const float mv = mml[(v * 2) * kCmpRows + row];
        const float f = mv == -INFINITY ? 0.f : fast_exp2((mv - M) * c2);
        Lsum += f * mml[(v * 2 + 1) * kCmpRows + row];
        const float* ov = mo + (v * kCmpRows + row) * 128 + d0;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] += f * ov[e];
      }
      const int rr = sg.rg * kCmpRows + row;
      if (sg.n_seg > 1) {
        float* part = p.partials + ((int64_t)sg.part * p.Hkv + h) * kCmpPartFloats;
#pragma unroll
        for (int e = 0; e < 8; ++e) part[row * 128 + d0 + e] = o[e];
        if ((i & 15) == 0) {
          part[kCmpRows * 128 + row] = M;
          part[kCmpRows * 128 + kCmpRows + row] = Lsum;
        }
      } else if (rr < rows_total && Lsum > 0.f) {
        float* dst = p.out + (((int64_t)sg.seq * p.q_len + rr / p.G) * p.Hq + h * p.G + rr % p.G) * 128 + d0;
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e] = o[e] / Lsum;
      }
    }
    named_barrier_sync(1, 32 * kCmpCompute);  // the merge area is free for the next segment
  }
  if (timed_out && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

template <int FMT>
__global__ void __launch_bounds__(kCmpThreads, 1) cmp_decode_kernel(const CmpDecodeParams p) {
  using SM = CmpSmem<FMT>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    const uint32_t full0 = smem_u32(smem + SM::kOffBars);
    for (int s = 0; s < SM::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(full0 + 8 * (SM::kStages + s), kCmpCompute);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0)
    cmp_producer<FMT>(p, smem, lane);
  else
    cmp_compute<FMT>(p, smem, warp - 1, lane);
  __syncthreads();
}

}  // namespace

int cmp_chunk_bytes(int fmt) { return chunk_bytes(fmt); }

cudaError_t launch_cmp_append(int fmt, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                              const int32_t* seq_ids, const int32_t* positions, int64_t T,
                              const float* rope, int32_t rope_max_pos, int32_t rot_dim,
                              const int32_t* block_table, int32_t num_seqs, int32_t max_pages,
                              int32_t num_pages, uint8_t* pool, uint16_t* q_out, int32_t Hq,
                              int32_t Hkv, int32_t* status, cudaStream_t stream) {
  CmpAppendParams p{q,        k,       v,    seq_ids,   positions, T,         rope,
                    rope_max_pos, rot_dim, block_table, num_seqs, max_pages, num_pages, pool,
                    q_out,    q ? Hq : 0, Hkv, status};
  const int64_t rows = T * (int64_t)(p.Hq + 2 * Hkv);
  const int64_t blocks = (rows + 7) / 8;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  if (fmt == kFmtBf16) cmp_append_kernel<kFmtBf16><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else if (fmt == kFmtInt8) cmp_append_kernel<kFmtInt8><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else cmp_append_kernel<kFmtK4V16><<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_cmp_decode(int fmt, const uint16_t* q, const uint8_t* pool,
                              const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                              const void* groups, const void* segments, const int32_t* cta_seg,
                              const int32_t* split_groups, int32_t num_split, float* partials,
                              float* out, int32_t* status, int32_t Hq, int32_t Hkv, int32_t q_len,
                              int32_t causal, float sm_scale, int32_t grid, cudaStream_t stream) {
  CmpDecodeParams p;
  p.q = q; p.pool = pool; p.block_table = block_table; p.max_pages = max_pages;
  p.num_pages = num_pages; p.groups = static_cast<const int4*>(groups);
  p.segments = static_cast<const int4*>(segments); p.cta_seg = cta_seg; p.partials = partials;
  p.out = out; p.status = status; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv; p.q_len = q_len;
  p.causal = causal; p.c2 = sm_scale * 1.4426950408889634f;
  if (grid > 0) {
    const dim3 gd((unsigned)grid, (unsigned)Hkv);
    cudaError_t e;
    if (fmt == kFmtBf16) {
      e = cudaFuncSetAttribute(cmp_decode_kernel<kFmtBf16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, CmpSmem<kFmtBf16>::kBytes);
      if (e != cudaSuccess) return e;
      cmp_decode_kernel<kFmtBf16><<<gd, kCmpThreads, CmpSmem<kFmtBf16>::kBytes, stream>>>(p);
    } else if (fmt == kFmtInt8) {
      e = cudaFuncSetAttribute(cmp_decode_kernel<kFmtInt8>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, CmpSmem<kFmtInt8>::kBytes);
      if (e != cudaSuccess) return e;
      cmp_decode_kernel<kFmtInt8><<<gd, kCmpThreads, CmpSmem<kFmtInt8>::kBytes, stream>>>(p);
    } else {
      e = cudaFuncSetAttribute(cmp_decode_kernel<kFmtK4V16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, CmpSmem<kFmtK4V16>::kBytes);
      if (e != cudaSuccess) return e;
      cmp_decode_kernel<kFmtK4V16><<<gd, kCmpThreads, CmpSmem<kFmtK4V16>::kBytes, stream>>>(p);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_split_merge(groups, split_groups, partials, out, Hq, Hkv, p.G, q_len, p.c2,
                            num_split, false, stream);
}

}  // namespace kvnvfp4
