// Fused quantize-append: RoPE -> normalised Walsh-Hadamard rotation -> NVFP4 for Q and K rows,
// NVFP4 only for V rows, stored into the paged pool (K, V) or the Q buffer.
//
// Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)" (Hadamard
// rotation of K and Q before quantisation, V unrotated, E2M1 codes with one E4M3 scale per 16
// elements, row-major scales, current K/V quantised as they are generated) and section "YaRN
// context extension" (theta 1e7, 25 % rotary dims, linear position scaling).
//
// Rows are taken in the flattened order [token][Q heads, K heads, V heads]. Two kernels:
//
// Bulk batches (prefill chunks, cache population): TWO threads per 128-element row, each holding
// 64 values in registers: thread h owns elements 32 j + 16 h + i (j < 4, i < 16), i.e. the 16-value
// blocks 2 j + h. Of the seven butterfly stages (h = 1, 2, ..., 64, in that order) only the stage
// that pairs elements 16 apart crosses to the partner thread (one shuffle per value); the others
// are register adds. A 16-value scale block lies in one thread, so its amax needs no shuffle, and
// each thread stores 8 bytes of every 16-byte code piece. A warp-block is 16 rows; its bf16 rows
// come into shared memory by cp.async with coalesced 16-byte requests, into rows padded to 272
// bytes (row r = lane % 16, half h = lane / 16 keeps every thread's 16-byte reads free of bank
// conflicts). Each warp keeps two such buffers: the next block's rows are in flight while it
// computes the current one. RoPE reads the partner of a rotated value back from the staged row,
// so any rotary width works without shuffles.
//
// Small batches (a decode step's few new tokens): one warp per row, lane l holding elements
// 4 l .. 4 l + 3 (the encoder shared with the fused decode step), four rows per warp, so that a
// handful of rows spreads over many SMs and finishes with the least latency.
//
// Every fp32 step that feeds a code is rounded exactly as the definition states (explicit _rn
// intrinsics, no contraction), so codes and scales are bit-identical to a plain CPU evaluation.

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

namespace {

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

// Resolves row w (Q heads, then K heads, then V heads) of token t: source row and destination,
// with the checks and status bits of the call's definition (a bad sequence id or position skips
// every row of the token; a bad page skips the K/V row; a rotated row past the RoPE table is
// skipped). Status bits are set only when `report` (one caller per row).
__device__ __forceinline__ const uint16_t* locate_row(const AppendParams& p, int32_t t, int32_t w,
                                                      bool report, RowMeta& m) {
  m.codes = nullptr; m.scales = nullptr; m.hi_step = 4; m.code_step = 16; m.pos = 0; m.kind = 0;
  if (t >= p.T) return nullptr;
  const int32_t seq = p.seq_ids[t];
  const int32_t pos = p.positions[t];
  bool bad = false;
  if (seq < 0 || seq >= p.num_seqs) {
    if (report) flag_status(p.status, KV_NVFP4_DEV_BAD_SEQ);
    bad = true;
  }
  if (pos < 0 || pos >= p.max_pages * kPage) {
    if (report) flag_status(p.status, KV_NVFP4_DEV_BAD_POS);
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
      if (report) flag_status(p.status, KV_NVFP4_DEV_BAD_PAGE);
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
    if (report) flag_status(p.status, KV_NVFP4_DEV_BAD_ROPE);
    return nullptr;
  }
  m.kind = rotate ? 1 : 2;
  return src;
}

// =============================================================================================
// Bulk kernel: two threads per row.
// =============================================================================================
constexpr int kWarps = 4;                         // warps per CTA
constexpr int kRowsPerBlock = 16;                 // rows of a warp-block
constexpr int kRowPitch = 272;                    // staged bf16 row: 256 bytes + 16 of padding
constexpr int kBufBytes = kRowsPerBlock * kRowPitch;
constexpr int kMetaBytes = kRowsPerBlock * 32;    // RowMeta of the block's rows
constexpr int kWarpSmem = 2 * (kBufBytes + kMetaBytes);
constexpr int kSmemBytes = kWarps * kWarpSmem + 128 * 8;  // + the E4M3 scale table: 39,936 B
constexpr int kCtasPerSm = 5;

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

// The bulk kernel's rows come in two spaces, so that a warp-block never mixes rotated and plain
// rows: blocks [0, rot_blocks) hold the rotated rows ([token][Q heads, K heads]), the blocks after
// them the plain rows ([token][V heads]).
__device__ __forceinline__ void block_row(const AppendParams& p, int32_t blk, int32_t rot_blocks,
                                          int r, int32_t& t, int32_t& w) {
  const int32_t nrot = p.Hq + p.Hkv;
  if (blk < rot_blocks) {
    const int32_t row = blk * kRowsPerBlock + r;
    t = row / nrot;
    w = row - t * nrot;
  } else {
    const int32_t row = (blk - rot_blocks) * kRowsPerBlock + r;
    t = row / p.Hkv;
    w = nrot + (row - t * p.Hkv);
  }
}

// Metadata of warp-block `blk` (lane r < 16 resolves the block's row r) into `meta`, and the
// copies of its 16 bf16 rows into buffer `buf`: request i moves rows 2 i and 2 i + 1, 16 lanes
// per row. A row with nothing to do is zero-filled without reading global memory.
__device__ __forceinline__ void issue_block(const AppendParams& p, int32_t blk, int32_t rot_blocks,
                                            uint32_t buf, RowMeta* meta, int lane) {
  uint64_t s = 0;
  if (lane < kRowsPerBlock) {
    RowMeta m;
    int32_t t, w;
    block_row(p, blk, rot_blocks, lane, t, w);
    s = reinterpret_cast<uint64_t>(locate_row(p, t, w, true, m));
    meta[lane] = m;
  }
  const int half = lane >> 4, c = lane & 15;
#pragma unroll
  for (int i = 0; i < kRowsPerBlock / 2; ++i) {
    const int r = 2 * i + half;
    const uint64_t sr = __shfl_sync(0xffffffffu, s, r);
    const uint16_t* g = sr != 0 ? reinterpret_cast<const uint16_t*>(sr) + 8 * c : p.k;
    cp_async16(buf + r * kRowPitch + c * 16, g, sr != 0 ? 16u : 0u);
  }
  cp_async_commit();
}

// max(m, |a|, |b|)
__device__ __forceinline__ float max3_abs(float m, float a, float b) {
  float r;
  asm("{\n.reg .f32 t1, t2;\nabs.f32 t1, %2;\nabs.f32 t2, %3;\nmax.f32 %0, %1, t1, t2;\n}"
      : "=f"(r)
      : "f"(m), "f"(a), "f"(b));
  return r;
}

// Thread h of a row: quantises its 64 values from the staged bf16 row at `row` (shared address)
// and stores its half of the row's codes and scales. Both threads of every row of the block run
// this together: the Hadamard stage that pairs elements 16 apart is a shuffle with lane ^ 16, and
// `rotated` (the block's row space) is the same for the whole warp. sc_tab holds, per E4M3 code,
// the decoded scale and its correctly rounded reciprocal.
__device__ __forceinline__ void encode_half_row(const AppendParams& p, uint32_t row,
                                                const RowMeta& m, int h, bool rotated,
                                                const float2* sc_tab) {
  // x[16 j + i] = element 32 j + 16 h + i
  float x[64];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint4 v = lds128(row + 64 * j + 32 * h + 16 * u);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[16 * j + 8 * u + 2 * e] = __uint_as_float(w[e] << 16);
        x[16 * j + 8 * u + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
  }
  if (rotated) {
    // RoPE on the first rot dims: dim e < rot/2 pairs with e + rot/2. The partner's original
    // value is read back from the staged copy, so the rotation can be done in place; each
    // product is rounded on its own, then added (a c - b s and b c + a s, as the definition
    // reads). Four consecutive dims share one table load (rot/2 is a multiple of 4). A skipped
    // row (kind 0) rotates zeros and stores nothing.
    const int rot = p.rot_dim, half = rot >> 1;
    if (rot > 0 && m.kind != 0) {
      const float* trow = p.rope + (int64_t)m.pos * rot;
#pragma unroll
      for (int k0 = 0; k0 < 64; k0 += 4) {
        if (32 * (k0 >> 4) >= rot) break;  // no rotated dim in this or a later 32-dim chunk
        const int e0 = 32 * (k0 >> 4) + 16 * h + (k0 & 15);
        if (e0 < rot) {
          const bool lower = e0 < half;
          const int i0 = lower ? e0 : e0 - half;          // angle index of dims e0 .. e0 + 3
          const float4 c4 = *reinterpret_cast<const float4*>(trow + i0);
          const float4 s4 = *reinterpret_cast<const float4*>(trow + half + i0);
          const uint2 pb = lds64(row + 2 * (lower ? e0 + half : e0 - half));
          const float part[4] = {__uint_as_float(pb.x << 16), __uint_as_float(pb.x & 0xFFFF0000u),
                                 __uint_as_float(pb.y << 16), __uint_as_float(pb.y & 0xFFFF0000u)};
          const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
          const float ss[4] = {s4.x, s4.y, s4.z, s4.w};
          const float sg = lower ? -1.0f : 1.0f;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            x[k0 + e] = __fadd_rn(__fmul_rn(x[k0 + e], cc[e]), __fmul_rn(sg * part[e], ss[e]));
        }
      }
    }
    // Walsh-Hadamard, Sylvester order: stages 1, 2, 4, 8 (inside a 16-value block), 16 (with the
    // partner thread), 32, 64 (across this thread's blocks)
#pragma unroll
    for (int hs = 1; hs < 16; hs <<= 1) {
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        if ((k & hs) == 0) {
          const float a = x[k], b = x[k + hs];
          x[k] = __fadd_rn(a, b);
          x[k + hs] = __fsub_rn(a, b);
        }
      }
    }
    {
      // the lower element of a pair is in thread 0: thread 0 keeps a + b, thread 1 keeps a - b;
      // (+-1) x is exact, so one fma rounds as the add or subtract does
      const float sgn = h ? -1.0f : 1.0f;
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        const float o = __shfl_xor_sync(0xffffffffu, x[k], 16);
        x[k] = __fmaf_rn(sgn, x[k], o);
      }
    }
#pragma unroll
    for (int hs = 16; hs < 64; hs <<= 1) {
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        if ((k & hs) == 0) {
          const float a = x[k], b = x[k + hs];
          x[k] = __fadd_rn(a, b);
          x[k + hs] = __fsub_rn(a, b);
        }
      }
    }
    const float kNorm = __uint_as_float(0x3DB504F3u);  // rn(2^-3.5) = rn(1/sqrt(128))
#pragma unroll
    for (int k = 0; k < 64; ++k) x[k] = __fmul_rn(x[k], kNorm);
  }

  // NVFP4 per 16-value block (block 2 j + h = x[16 j .. 16 j + 15]): scale = RNE_sat_E4M3(amax / 6),
  // codes = RNE_sat_E2M1(x / scale), each quotient rounded to fp32 first, as the definition reads
  const float r6 = __uint_as_float(0x3E2AAAABu);  // rn(1/6)
  uint32_t codes[8];
  uint32_t sc4 = 0u;  // scales of blocks h, 2 + h, 4 + h, 6 + h
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float amax = fabsf(x[16 * j]);
#pragma unroll
    for (int e = 1; e < 15; e += 2) amax = max3_abs(amax, x[16 * j + e], x[16 * j + e + 1]);
    amax = fmaxf(amax, fabsf(x[16 * j + 15]));  // elements 0 .. 15 of the block
    const uint32_t sc = e4m3x2_from_f32(0.0f, div_rn_by(amax, 6.0f, r6)) & 0xFFu;
    const float2 sr = sc_tab[sc];  // decoded scale, its reciprocal
    float q[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) q[e] = quot_rn(x[16 * j + e], sr.x, sr.y);
    const float(&q0)[8] = *reinterpret_cast<const float(*)[8]>(&q[0]);
    const float(&q1)[8] = *reinterpret_cast<const float(*)[8]>(&q[8]);
    const bool zero = sc == 0u;  // an all-zero block: zero scale, zero codes
    codes[2 * j] = zero ? 0u : e2m1x8_from_f32(q0);
    codes[2 * j + 1] = zero ? 0u : e2m1x8_from_f32(q1);
    sc4 |= sc << (8 * j);
  }
  // 16-byte code piece j = blocks 2 j (thread 0) and 2 j + 1 (thread 1): 8 bytes each
  if (m.kind != 0) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint2*>(m.codes + j * m.code_step + 8 * h) =
          make_uint2(codes[2 * j], codes[2 * j + 1]);
  }
  // scales: thread 0 holds blocks 0, 2, 4, 6 and thread 1 blocks 1, 3, 5, 7; thread 0 stores
  // blocks 0..3, thread 1 blocks 4..7
  const uint32_t other = __shfl_xor_sync(0xffffffffu, sc4, 16);
  const uint32_t s0 = h ? other : sc4, s1 = h ? sc4 : other;
  if (m.kind != 0) {
    const uint32_t word = h ? __byte_perm(s0, s1, 0x7362) : __byte_perm(s0, s1, 0x5140);
    *reinterpret_cast<uint32_t*>(m.scales + (h ? m.hi_step : 0)) = word;
  }
}

__global__ void __launch_bounds__(kWarps * 32, kCtasPerSm) append_rows_kernel(const AppendParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  // decoded E4M3 scale and its correctly rounded reciprocal, per code (0x7F, NaN, never occurs)
  float2* sc_tab = reinterpret_cast<float2*>(smem + kWarps * kWarpSmem);
  if (threadIdx.x < 128) {
    const float sd = e4m3_decode_pos(threadIdx.x);
    sc_tab[threadIdx.x] = make_float2(sd, __frcp_rn(sd));
  }
  __syncthreads();
  // Launched as a programmatic dependent of the previous kernel on the stream (e.g. the attention
  // of the previous step, which reads the pool): wait for it before touching memory, then let the
  // next kernel (the attention of this step) start its launch while this one runs; that kernel
  // waits for this one in turn before reading the pool.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int r = lane & 15, h = lane >> 4;
  uint8_t* wsm = smem + warp * kWarpSmem;
  const uint32_t buf0 = smem_u32(wsm);
  RowMeta* meta0 = reinterpret_cast<RowMeta*>(wsm + 2 * kBufBytes);
  const int32_t rot_blocks = (p.T * (p.Hq + p.Hkv) + kRowsPerBlock - 1) / kRowsPerBlock;
  const int32_t nblocks = rot_blocks + (p.T * p.Hkv + kRowsPerBlock - 1) / kRowsPerBlock;
  const int32_t stride = gridDim.x * kWarps;
  int32_t b = blockIdx.x * kWarps + warp;
  if (b < nblocks) issue_block(p, b, rot_blocks, buf0, meta0, lane);
  uint32_t u = 0;
  for (; b < nblocks; b += stride, u ^= 1u) {
    const int32_t bn = b + stride;
    if (bn < nblocks) {
      issue_block(p, bn, rot_blocks, buf0 + (u ^ 1u) * kBufBytes, meta0 + (u ^ 1u) * kRowsPerBlock,
                  lane);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const RowMeta m = meta0[u * kRowsPerBlock + r];
    // both threads of every row run the encoder (the shuffles need the whole warp)
    encode_half_row(p, buf0 + u * kBufBytes + r * kRowPitch, m, h, b < rot_blocks, sc_tab);
    __syncwarp();  // buffer u is free for the block after next
  }
}

// =============================================================================================
// Small-batch kernel: one warp per row, four rows per warp.
// =============================================================================================
constexpr int kSmallWarps = 8;
constexpr int kSmallRowsPerWarp = 4;

__global__ void __launch_bounds__(kSmallWarps * 32, 4) append_small_kernel(const AppendParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int32_t row0 = (blockIdx.x * kSmallWarps + warp) * kSmallRowsPerWarp;
  RowMeta m[kSmallRowsPerWarp];
  uint2 raw[kSmallRowsPerWarp];
#pragma unroll
  for (int j = 0; j < kSmallRowsPerWarp; ++j) {
    const int32_t row = row0 + j, t = row / p.per_tok;
    const uint16_t* src = locate_row(p, t, row - t * p.per_tok, lane == 0, m[j]);
    raw[j] = src != nullptr ? ldg_nc_u2(src + 4 * lane) : make_uint2(0u, 0u);
  }
#pragma unroll
  for (int j = 0; j < kSmallRowsPerWarp; ++j) {
    if (m[j].kind == 0) continue;  // warp-uniform: every lane resolved the same row
    float x[4] = {__uint_as_float(raw[j].x << 16), __uint_as_float(raw[j].x & 0xFFFF0000u),
                  __uint_as_float(raw[j].y << 16), __uint_as_float(raw[j].y & 0xFFFF0000u)};
    const bool rotate = m[j].kind == 1;
    const float* rope_row = (rotate && p.rot_dim > 0) ? p.rope + (int64_t)m[j].pos * p.rot_dim
                                                      : nullptr;
    uint32_t sc;
    const uint32_t packed = nvfp4_encode_row(x, rotate, rope_row, p.rot_dim, lane, sc);
    // lane l holds code bytes 2 l, 2 l + 1 of the row: 16-byte piece l / 8, offset (2 l) % 16
    *reinterpret_cast<uint16_t*>(m[j].codes + (lane >> 3) * m[j].code_step + ((2 * lane) & 15)) =
        (uint16_t)packed;
    if ((lane & 3) == 0)
      m[j].scales[(lane < 16 ? 0 : m[j].hi_step) + ((lane >> 2) & 3)] = (uint8_t)sc;
  }
}

// Rows up to which the small-batch kernel runs (a decode step's or a verify step's new tokens).
constexpr int64_t kSmallRows = 8192;

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
    const cudaError_t e = cudaFuncSetAttribute(
        append_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  const int32_t hq = q ? Hq : 0;
  const int32_t per_tok = hq + 2 * Hkv;
  // rows of one launch stay below 2^31 (32-bit row arithmetic in the kernels)
  const int64_t max_tok = (int64_t)0x7FFFFFE0 / per_tok;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
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
    const int64_t rows = n * per_tok;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (rows <= kSmallRows) {
      const int64_t per_cta = (int64_t)kSmallWarps * kSmallRowsPerWarp;
      cfg.gridDim = dim3((unsigned)((rows + per_cta - 1) / per_cta));
      cfg.blockDim = dim3(kSmallWarps * 32);
      cfg.dynamicSmemBytes = 0;
      e = cudaLaunchKernelEx(&cfg, append_small_kernel, p);
    } else {
      const int64_t nblocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
      const int64_t want = (nblocks + kWarps - 1) / kWarps;
      const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 1) * kCtasPerSm;
      cfg.gridDim = dim3((unsigned)(want < cap ? want : cap));
      cfg.blockDim = dim3(kWarps * 32);
      cfg.dynamicSmemBytes = kSmemBytes;
      e = cudaLaunchKernelEx(&cfg, append_rows_kernel, p);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvnvfp4
