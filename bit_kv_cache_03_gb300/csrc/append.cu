// Fused quantize-append: RoPE -> normalised Walsh-Hadamard rotation -> NVFP4 for Q and K rows,
// NVFP4 only for V rows, stored into the paged pool (K, V) or the Q buffer.
//
// Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)" (Hadamard
// rotation of K and Q before quantisation, V unrotated, E2M1 codes with one E4M3 scale per 16
// elements, row-major scales, current K/V quantised as they are generated) and section "YaRN
// context extension" (theta 1e7, 25 % rotary dims, linear position scaling).
//
// Mapping: one warp per 128-element row, lane l holds elements 4l..4l+3 (one 8-byte load).
//   RoPE pairs (i, i + rot_dim/2) sit in lanes l and l + rot_dim/8: one shuffle.
//   Hadamard: stages h = 1, 2 inside the lane, h = 4..64 as xor-shuffles over lane bits 0..4.
//   A 16-element scale block is a group of four lanes: two xor-shuffles give its amax.
// Every fp32 step that feeds a code is rounded exactly as the definition states (explicit _rn
// intrinsics, no contraction), so codes and scales are bit-identical to a plain CPU evaluation.
// Each warp handles kRowsPerWarp rows and issues all of their loads before computing, to keep
// enough bytes in flight for an HBM-bound kernel.

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kRowsPerWarp = 4;

struct AppendParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* seq_ids;
  const int32_t* positions;
  int64_t T;
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
  int32_t Hq;   // 0 when q is absent
  int32_t Hkv;
  int32_t* status;
};

struct RowTarget {
  const uint16_t* src;  // bf16 row
  uint8_t* codes;       // code destination, or nullptr to skip the row
  uint8_t* scales;      // scales of blocks 0..3; blocks 4..7 at scales + hi_step
  int32_t hi_step;      // 4, or for K rows the distance to the second 64-dim half's scales
  int32_t pos;          // position, for RoPE
  bool rotate;
  bool tiled;           // K codes: 16-byte pieces 128 bytes apart (tensor-core tile order)
};

__device__ __forceinline__ RowTarget locate_row(const AppendParams& p, int64_t row, int lane) {
  RowTarget r{nullptr, nullptr, nullptr, 4, 0, false, false};
  const int32_t per_tok = p.Hq + 2 * p.Hkv;
  const int64_t t = row / per_tok;
  const int32_t w = (int32_t)(row - t * per_tok);
  const int32_t seq = p.seq_ids[t];
  const int32_t pos = p.positions[t];
  bool bad = false;
  if (seq < 0 || seq >= p.num_seqs) {
    if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_SEQ);
    bad = true;
  }
  if (pos < 0 || pos >= p.max_pages * kPage) {
    if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_POS);
    bad = true;
  }
  if (bad) return r;
  r.pos = pos;
  if (w < p.Hq) {  // Q row
    r.src = p.q + (t * p.Hq + w) * kHeadDim;
    r.codes = p.q_codes + (t * p.Hq + w) * kCodeBytes;
    r.scales = p.q_scales + (t * p.Hq + w) * kScaleBytes;
    r.rotate = true;
  } else {
    const int32_t kv = w - p.Hq;
    const bool is_k = kv < p.Hkv;
    const int32_t h = is_k ? kv : kv - p.Hkv;
    const int32_t page = p.block_table[(int64_t)seq * p.max_pages + pos / kPage];
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_PAGE);
      return r;
    }
    // page block: [K codes H*4096 (tiled)][K scales H*512 (scale-copy order)][V codes H*4096]
    // [V scales H*512]
    uint8_t* blk = p.pool + (int64_t)page * p.Hkv * 9216;
    const int k = pos % kPage;
    r.src = (is_k ? p.k : p.v) + (t * p.Hkv + h) * kHeadDim;
    if (is_k) {
      r.codes = blk + h * 4096 + (k >> 3) * 512 + (k & 7) * 16;  // + chunk * 128 + byte % 16
      r.scales = blk + kscale_offset(p.Hkv, h, k, 0);
      r.hi_step = kscale_offset(p.Hkv, h, k, 1) - kscale_offset(p.Hkv, h, k, 0);
    } else {
      r.codes = blk + p.Hkv * 4608 + h * 4096 + k * 64;
      r.scales = blk + p.Hkv * 8704 + h * 512 + k * 8;
    }
    r.tiled = is_k;
    r.rotate = is_k;
  }
  if (r.rotate && p.rot_dim > 0 && pos >= p.rope_max_pos) {
    if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_ROPE);
    r.codes = nullptr;
  }
  return r;
}

__device__ __forceinline__ void quantize_store_row(float (&x)[4], const RowTarget& r,
                                                   const AppendParams& p, int lane) {
  // a row past the RoPE table is flagged and not stored: do not read the table for it either
  const float* rope_row = (r.rotate && p.rot_dim > 0 && r.codes != nullptr)
                              ? p.rope + (int64_t)r.pos * p.rot_dim : nullptr;
  uint32_t sc;
  const uint32_t packed = nvfp4_encode_row(x, r.rotate, rope_row, p.rot_dim, lane, sc);
  if (r.codes != nullptr) {
    // lane l holds code bytes 2l, 2l+1 of the row: 16-byte piece l / 8, offset (2l) % 16
    uint8_t* dst = r.tiled ? r.codes + (lane >> 3) * 128 + ((2 * lane) & 15) : r.codes + 2 * lane;
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
    if ((lane & 3) == 0) r.scales[(lane < 16 ? 0 : r.hi_step) + ((lane >> 2) & 3)] = (uint8_t)sc;
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32, 4) append_kernel(const AppendParams p) {
  // Launched as a programmatic dependent of the previous kernel on the stream (e.g. the attention
  // of the previous step, which reads the pool): wait for it before touching memory, then let the
  // next kernel (the attention of this step) start its launch while this one runs; that kernel
  // waits for this one in turn before reading the pool.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t rows = p.T * (int64_t)(p.Hq + 2 * p.Hkv);
  const int64_t row0 = ((int64_t)blockIdx.x * kWarpsPerBlock + warp) * kRowsPerWarp;
  RowTarget tg[kRowsPerWarp];
  uint2 raw[kRowsPerWarp];
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    tg[j].codes = nullptr;
    raw[j] = make_uint2(0u, 0u);
    if (row0 + j < rows) {
      tg[j] = locate_row(p, row0 + j, lane);
      if (tg[j].codes != nullptr) raw[j] = ldg_nc_u2(tg[j].src + 4 * lane);
    }
  }
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    if (tg[j].codes == nullptr) continue;  // warp-uniform: every lane saw the same row
    float x[4];
    x[0] = __uint_as_float(raw[j].x << 16);
    x[1] = __uint_as_float(raw[j].x & 0xFFFF0000u);
    x[2] = __uint_as_float(raw[j].y << 16);
    x[3] = __uint_as_float(raw[j].y & 0xFFFF0000u);
    quantize_store_row(x, tg[j], p, lane);
  }
}

}  // namespace

cudaError_t launch_append(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* seq_ids, const int32_t* positions, int64_t T,
                          const float* rope, int32_t rope_max_pos, int32_t rot_dim,
                          const int32_t* block_table, int32_t num_seqs, int32_t max_pages,
                          int32_t num_pages, uint8_t* pool, uint8_t* q_codes,
                          uint8_t* q_scales, int32_t Hq, int32_t Hkv, int32_t* status,
                          cudaStream_t stream) {
  AppendParams p{q,       k,         v,           seq_ids,  positions, T,
                 rope,    rope_max_pos, rot_dim,  block_table, num_seqs, max_pages,
                 num_pages, pool,    q_codes,     q_scales, q ? Hq : 0, Hkv, status};
  const int64_t rows = T * (int64_t)(p.Hq + 2 * Hkv);
  const int64_t per_block = (int64_t)kWarpsPerBlock * kRowsPerWarp;
  const int64_t blocks = (rows + per_block - 1) / per_block;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kWarpsPerBlock * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_kernel, p);
}

}  // namespace kvnvfp4
