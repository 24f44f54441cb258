// Fused quantize-append: RoPE -> normalised Walsh-Hadamard rotation -> NVFP4 for Q and K rows,
// NVFP4 only for V rows, stored into the paged pool (K, V) or the Q buffer.
//
// Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)" (Hadamard
// rotation of K and Q before quantisation, V unrotated, E2M1 codes with one E4M3 scale per 16
// elements, row-major scales, current K/V quantised as they are generated) and section "YaRN
// context extension" (theta 1e7, 25 % rotary dims, linear position scaling).
//
// Mapping: one THREAD per 128-element row, all 128 values in registers, so the rotation needs
// no shuffles: the seven butterfly stages (h = 1, 2, ..., 64, in that order) are 896 register
// adds, the per-16 amax is an in-thread max, and the thread writes its row's 64 code bytes as
// four 16-byte pieces. Rows are taken in the flattened order [token][Q heads, K heads, V heads],
// 32 rows (one per lane) per warp-block.
//
// Staging: a warp-block's bf16 rows come into shared memory by cp.async with coalesced 16-byte
// requests (16 lanes per 256-byte row), into rows padded to 272 bytes so that each thread's
// reads of its own row are free of bank conflicts. Every warp keeps two such buffers: the rows
// of its next block are in flight while it computes the current one, and the per-row metadata
// (sequence, position, page, destinations) is resolved when the block's copies are issued.
//
// Every fp32 step that feeds a code is rounded exactly as the definition states (explicit _rn
// intrinsics, no contraction), so codes and scales are bit-identical to a plain CPU evaluation.

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

namespace {

constexpr int kWarps = 4;                         // warps per CTA
constexpr int kRowPitch = 272;                    // staged bf16 row: 256 bytes + 16 of padding
constexpr int kBufBytes = 32 * kRowPitch;         // one warp-block of 32 rows
constexpr int kMetaBytes = 32 * 32;               // RowMeta of 32 rows
constexpr int kWarpSmem = 2 * (kBufBytes + kMetaBytes);
constexpr int kSmemBytes = kWarps * kWarpSmem;    // 73,728 bytes: three CTAs per SM
constexpr int kCtasPerSm = 3;

struct AppendParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* seq_ids;
  const int32_t* positions;
  int32_t T;             // tokens of this launch
  int32_t per_tok;       // rows per token: Hq + 2 Hkv (Hq = 0 without Q)
  const float* rope;
  int32_t rope_max_pos;
  int32_t rot_dim;
  const int32_t* block_table;
  int32_t num_seqs;
  int32_t max_pages;
  int32_t num_pages;
  uint8_t* pool;         // num_pages blocks of Hkv * 9216 bytes
  uint8_t* q_codes;
  uint8_t* q_scales;
  int32_t Hq;            // 0 when q is absent
  int32_t Hkv;
  int32_t* status;
};

// Where one row goes. kind: 0 = nothing to do (padding row, or a row flagged and skipped),
// 1 = rotated row (Q or K: RoPE + Hadamard + NVFP4), 2 = plain row (V: NVFP4 only).
struct RowMeta {
  uint8_t* codes;      // code piece 0; piece p at codes + p * code_step
  uint8_t* scales;     // scales of blocks 0..3; blocks 4..7 at scales + hi_step
  int32_t hi_step;
  int32_t code_step;   // 128 for K (tensor-core tile order), 16 otherwise
  int32_t pos;         // position, for RoPE
  int32_t kind;
};
static_assert(sizeof(RowMeta) == 32, "metadata slot");

// Resolves row `row` of the flattened [token][Q, K, V heads] order: source row and destination,
// with the same checks and status bits as the definition of the call (a bad sequence id or
// position skips every row of the token; a bad page skips the K/V row; a rotated row past the
// RoPE table is skipped).
__device__ __forceinline__ const uint16_t* locate_row(const AppendParams& p, int32_t row,
                                                      RowMeta& m) {
  m.codes = nullptr; m.scales = nullptr; m.hi_step = 4; m.code_step = 16; m.pos = 0; m.kind = 0;
  if (row >= p.T * p.per_tok) return nullptr;
  const int32_t t = row / p.per_tok;
  const int32_t w = row - t * p.per_tok;
  const int32_t seq = p.seq_ids[t];
  const int32_t pos = p.positions[t];
  bool bad = false;
  if (seq < 0 || seq >= p.num_seqs) {
    flag_status(p.status, KV_NVFP4_DEV_BAD_SEQ);
    bad = true;
  }
  if (pos < 0 || pos >= p.max_pages * kPage) {
    flag_status(p.status, KV_NVFP4_DEV_BAD_POS);
    bad = true;
  }
  if (bad) return nullptr;
  m.pos = pos;
  const uint16_t* src;
  bool rotate;
  if (w < p.Hq) {  // Q row
    const int64_t qr = (int64_t)t * p.Hq + w;
    src = p.q + qr * kHeadDim;
    m.codes = p.q_codes + qr * kCodeBytes;
    m.scales = p.q_scales + qr * kScaleBytes;
    rotate = true;
  } else {
    const int32_t kv = w - p.Hq;
    const bool is_k = kv < p.Hkv;
    const int32_t h = is_k ? kv : kv - p.Hkv;
    const int32_t page = p.block_table[(int64_t)seq * p.max_pages + pos / kPage];
    if (page < 0 || page >= p.num_pages) {
      flag_status(p.status, KV_NVFP4_DEV_BAD_PAGE);
      return nullptr;
    }
    // page block: [K codes H*4096 (tile order)][K scales H*512 (scale-copy order)][V codes
    // H*4096][V scales H*512]
    uint8_t* blk = p.pool + (int64_t)page * p.Hkv * 9216;
    const int k = pos % kPage;
    src = (is_k ? p.k : p.v) + ((int64_t)t * p.Hkv + h) * kHeadDim;
    if (is_k) {
      m.codes = blk + h * 4096 + (k >> 3) * 512 + (k & 7) * 16;
      m.code_step = 128;
      m.scales = blk + kscale_offset(p.Hkv, h, k, 0);
      m.hi_step = kscale_offset(p.Hkv, h, k, 1) - kscale_offset(p.Hkv, h, k, 0);
    } else {
      m.codes = blk + p.Hkv * 4608 + h * 4096 + k * 64;
      m.scales = blk + p.Hkv * 8704 + h * 512 + k * 8;
    }
    rotate = is_k;
  }
  if (rotate && p.rot_dim > 0 && pos >= p.rope_max_pos) {
    flag_status(p.status, KV_NVFP4_DEV_BAD_ROPE);
    return nullptr;
  }
  m.kind = rotate ? 1 : 2;
  return src;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Metadata of warp-block `blk` (row blk * 32 + lane for this lane) into slot `u`, and the copies
// of its 32 bf16 rows into buffer `u`: request i moves rows 2i and 2i + 1, 16 lanes per row. A
// row with nothing to do is zero-filled without reading global memory.
__device__ __forceinline__ void issue_block(const AppendParams& p, int32_t blk, uint32_t buf,
                                            RowMeta* meta, int lane) {
  RowMeta m;
  const uint16_t* src = locate_row(p, blk * 32 + lane, m);
  meta[lane] = m;
  const uint64_t s = reinterpret_cast<uint64_t>(src);
  const int half = lane >> 4, c = lane & 15;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = 2 * i + half;
    const uint64_t sr = __shfl_sync(0xffffffffu, s, r);
    const uint16_t* g = sr != 0 ? reinterpret_cast<const uint16_t*>(sr) + 8 * c : p.k;
    cp_async16(buf + r * kRowPitch + c * 16, g, sr != 0 ? 16u : 0u);
  }
  cp_async_commit();
}

// Quantises this lane's row from the staged bf16 copy at `row` (shared address) and stores it.
__device__ __forceinline__ void encode_store_row(const AppendParams& p, uint32_t row,
                                                 const RowMeta& m) {
  float x[128];
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint4 v = lds128(row + c * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[8 * c + 2 * e] = __uint_as_float(w[e] << 16);
      x[8 * c + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
  if (m.kind == 1) {
    // RoPE on the first rot dims: dim j < rot/2 pairs with j + rot/2. The partner's original
    // value is read back from the staged copy, so the rotation can be done in place; each
    // product is rounded on its own, then added (a c - b s and b c + a s, as the definition reads)
    const int rot = p.rot_dim, half = rot >> 1;
    if (rot > 0) {
      const float* trow = p.rope + (int64_t)m.pos * rot;
#pragma unroll
      for (int j0 = 0; j0 < 128; j0 += 4) {
        if (j0 < rot) {
          const bool lower = j0 < half;
          const int i0 = lower ? j0 : j0 - half;          // angle index of dims j0 .. j0 + 3
          const float4 c4 = *reinterpret_cast<const float4*>(trow + i0);
          const float4 s4 = *reinterpret_cast<const float4*>(trow + half + i0);
          const uint2 pb = lds64(row + 2 * (lower ? j0 + half : j0 - half));
          const float part[4] = {__uint_as_float(pb.x << 16), __uint_as_float(pb.x & 0xFFFF0000u),
                                 __uint_as_float(pb.y << 16), __uint_as_float(pb.y & 0xFFFF0000u)};
          const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
          const float ss[4] = {s4.x, s4.y, s4.z, s4.w};
          const float sg = lower ? -1.0f : 1.0f;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            x[j0 + e] = __fadd_rn(__fmul_rn(x[j0 + e], cc[e]), __fmul_rn(sg * part[e], ss[e]));
        }
      }
    }
    // Walsh-Hadamard, Sylvester order, stages h = 1, 2, 4, ..., 64
#pragma unroll
    for (int h = 1; h < 128; h <<= 1) {
#pragma unroll
      for (int j = 0; j < 128; ++j) {
        if ((j & h) == 0) {
          const float a = x[j], b = x[j + h];
          x[j] = __fadd_rn(a, b);
          x[j + h] = __fsub_rn(a, b);
        }
      }
    }
    const float kNorm = __uint_as_float(0x3DB504F3u);  // rn(2^-3.5) = rn(1/sqrt(128))
#pragma unroll
    for (int j = 0; j < 128; ++j) x[j] = __fmul_rn(x[j], kNorm);
  }

  // NVFP4 per 16-element block: scale = RNE_sat_E4M3(amax / 6), codes = RNE_sat_E2M1(x / scale),
  // each quotient rounded to fp32 first, exactly as the definition reads
  const float r6 = __frcp_rn(6.0f);
  uint32_t codes[16];
  uint32_t sc_lo = 0u, sc_hi = 0u;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(x[16 * b + e]));
    const uint32_t sc = e4m3x2_from_f32(0.0f, div_rn_by(amax, 6.0f, r6)) & 0xFFu;
    const float sd = e4m3_decode_pos(sc);
    const float rs = __frcp_rn(sd);
    uint32_t w0 = 0u, w1 = 0u;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float a = x[16 * b + e], bb = x[16 * b + e + 1];
      const uint32_t byte = e2m1x2_from_f32(copysignf(div_rn_by(bb, sd, rs), bb),
                                            copysignf(div_rn_by(a, sd, rs), a));
      w0 |= byte << (4 * e);
    }
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float a = x[16 * b + 8 + e], bb = x[16 * b + 9 + e];
      const uint32_t byte = e2m1x2_from_f32(copysignf(div_rn_by(bb, sd, rs), bb),
                                            copysignf(div_rn_by(a, sd, rs), a));
      w1 |= byte << (4 * e);
    }
    const bool zero = sd == 0.0f;  // an all-zero block: zero scale, zero codes
    codes[2 * b] = zero ? 0u : w0;
    codes[2 * b + 1] = zero ? 0u : w1;
    if (b < 4) sc_lo |= sc << (8 * b);
    else sc_hi |= sc << (8 * (b - 4));
  }
  // 64 code bytes as four 16-byte pieces (piece q = blocks 2q, 2q + 1), then the scales
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(m.codes + q * m.code_step) =
        make_uint4(codes[4 * q], codes[4 * q + 1], codes[4 * q + 2], codes[4 * q + 3]);
  *reinterpret_cast<uint32_t*>(m.scales) = sc_lo;
  *reinterpret_cast<uint32_t*>(m.scales + m.hi_step) = sc_hi;
}

__global__ void __launch_bounds__(kWarps * 32, kCtasPerSm) append_kernel(const AppendParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  // Launched as a programmatic dependent of the previous kernel on the stream (e.g. the attention
  // of the previous step, which reads the pool): wait for it before touching memory, then let the
  // next kernel (the attention of this step) start its launch while this one runs; that kernel
  // waits for this one in turn before reading the pool.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t* wsm = smem + warp * kWarpSmem;
  const uint32_t buf0 = smem_u32(wsm);
  RowMeta* meta0 = reinterpret_cast<RowMeta*>(wsm + 2 * kBufBytes);
  const int32_t nblocks = (p.T * p.per_tok + 31) / 32;
  const int32_t stride = gridDim.x * kWarps;
  int32_t b = blockIdx.x * kWarps + warp;
  if (b < nblocks) issue_block(p, b, buf0, meta0, lane);
  uint32_t u = 0;
  for (; b < nblocks; b += stride, u ^= 1u) {
    const int32_t bn = b + stride;
    if (bn < nblocks) {
      issue_block(p, bn, buf0 + (u ^ 1u) * kBufBytes, meta0 + (u ^ 1u) * 32, lane);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const RowMeta m = meta0[u * 32 + lane];
    if (m.kind != 0) encode_store_row(p, buf0 + u * kBufBytes + lane * kRowPitch, m);
    __syncwarp();  // buffer u is free for the block after next
  }
}

}  // namespace

cudaError_t launch_append(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* seq_ids, const int32_t* positions, int64_t T,
                          const float* rope, int32_t rope_max_pos, int32_t rot_dim,
                          const int32_t* block_table, int32_t num_seqs, int32_t max_pages,
                          int32_t num_pages, uint8_t* pool, uint8_t* q_codes,
                          uint8_t* q_scales, int32_t Hq, int32_t Hkv, int32_t* status,
                          int32_t num_sms, cudaStream_t stream) {
  static bool attr_done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  const int32_t hq = q ? Hq : 0;
  const int32_t per_tok = hq + 2 * Hkv;
  // rows of one launch stay below 2^31 (32-bit row arithmetic in the kernel)
  const int64_t max_tok = (int64_t)0x7FFFFFE0 / per_tok;
  for (int64_t t0 = 0; t0 < T; t0 += max_tok) {
    const int64_t n = T - t0 < max_tok ? T - t0 : max_tok;
    AppendParams p{q ? q + t0 * Hq * kHeadDim : nullptr,
                   k + t0 * Hkv * kHeadDim,
                   v + t0 * Hkv * kHeadDim,
                   seq_ids + t0,
                   positions + t0,
                   (int32_t)n,
                   per_tok,
                   rope,
                   rope_max_pos,
                   rot_dim,
                   block_table,
                   num_seqs,
                   max_pages,
                   num_pages,
                   pool,
                   q ? q_codes + t0 * Hq * kCodeBytes : nullptr,
                   q ? q_scales + t0 * Hq * kScaleBytes : nullptr,
                   hq,
                   Hkv,
                   status};
    const int64_t nblocks = (n * per_tok + 31) / 32;
    const int64_t want = (nblocks + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 1) * kCtasPerSm;
    const int64_t grid = want < cap ? want : cap;
    if (grid <= 0) continue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, append_kernel, p);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvnvfp4
