// Paged GQA attention over the NVFP4 cache for query tiles of many rows (speculative verify,
// prefill chunks), with both products on the tcgen05 tensor cores.
//
// Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)": the Q.K^T
// product in NVFP4 with E4M3 block scales (both Q and K quantised), V dequantised for the P.V
// product. The tile decomposition, the lazily raised running max and the split-K merge are this
// library's design; the pages say nothing about the kernel's decomposition.
//
// Work decomposition. A group is (sequence, KV-head pair, tile of 64 query rows per head), a row
// being (query token, head in the GQA group) as in the decode kernel. The plan lays the groups'
// pages end to end and gives each persistent CTA a contiguous, page-balanced share (segments); a
// group spread over several CTAs leaves one (m, l, O) partial per segment and head, merged by a
// second launch.
//
// Per page (64 keys of the pair's two heads, 18 KB in four bulk copies):
//   Q.K^T: tcgen05.mma kind::mxf4nvf4 block_scale.scale_vec::4X, M = 128 query rows (64 of head
//     2p, then 64 of head 2p + 1), N = 128 keys (64 of each head), K = 64 per instruction. The
//     cross terms (rows of one head against keys of the other) are computed and ignored; in return
//     the K codes and scales are used exactly as the pool stores them (tensor-core tile order,
//     scale-copy order) and the K scales go to TMEM with one copy per k-half.
//   Softmax: four warps, one query row per thread (TMEM lane = row), fp32 online softmax. The
//     running max m of a row is raised only when a page's max exceeds it by more than 2^8 in the
//     exp2 domain (then the whole O tile is rescaled in TMEM, all rows at once), so
//     P = exp2((s - m) c2) <= 2^8 fits f16 and O, l use the same m; the result O / l is unchanged.
//   V: two warps dequantise the page's V rows (E2M1 x E4M3 is exact in f16), two key rows of one
//     head per thread, into an MN-major f16 tile.
//   P.V: tcgen05.mma kind::f16, transposed per head: O^T[dims][rows] += V^T P^T with M = 128 dims
//     (A = the dequantised V tile), N = 64 rows (B = P, K-major), K = 16 keys per instruction. O^T
//     stays in TMEM for the whole segment.
// Two S buffers, two P tiles and three V tiles: the Q.K^T of page j + 2 and the P.V of page j - 1
// run on the tensor pipe while the softmax of page j runs.
//
// Warp roles (256 threads): warp 0 bulk-copy producer, warp 1 MMA issuer and TMEM owner, warps
// 2..5 softmax and epilogue (TMEM lane quadrants 2, 3, 0, 1), warps 6, 7 V dequantisation. Every
// wait is an mbarrier wait bounded in time; on a timeout the kernel records KV_NVFP4_DEV_TIMEOUT
// and carries on, so it cannot hang.

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

namespace {

constexpr int kTRows = 64;                  // query rows per head in a tile
constexpr int kTStages = 4;
// one page of a head pair in a stage: K codes (both heads, tile order), K scales (scale-copy
// order), V codes, V scales
constexpr int kStK = 0, kStKs = 8192, kStV = 9216, kStVs = 17408;
constexpr int kTStageBytes = 18432;
constexpr int kVtHeadBytes = 16384;         // dequantised V of one head: 64 keys x 128 dims, f16
constexpr int kPHeadBytes = 8192;           // P of one head: 64 rows x 64 keys, f16
constexpr int kTPartHeadFloats = kTRows * 128 + 2 * kTRows;  // O[64][128], m[64], l[64]

constexpr int kTWarpProducer = 0, kTWarpMma = 1, kTWarpSoft0 = 2, kTWarpDeq0 = 6;
constexpr int kTDeqWarps = 2;              // on the sub-partitions without the producer / MMA warp
constexpr int kTVtBufs = 3;                // dequantised V tiles
constexpr int kTThreads = (kTWarpDeq0 + kTDeqWarps) * 32;
constexpr uint32_t kNbSoft = 1;             // named barrier of the four softmax warps
constexpr float kLazyMax = 8.0f;            // raise the running max only past 2^8 (exp2 domain)

// shared memory map
constexpr int kTOffStage = 0;
constexpr int kTOffQ = kTOffStage + kTStages * kTStageBytes;  // [128 rows][64 B], tile order
constexpr int kTOffVt = kTOffQ + 8192;                         // [kTVtBufs][2 heads]
constexpr int kTOffP = kTOffVt + kTVtBufs * 2 * kVtHeadBytes;  // [2 buffers][2 heads]
constexpr int kTOffSfw = kTOffP + 2 * 2 * kPHeadBytes;         // lone head's K scales widened
constexpr int kTOffQsc = kTOffSfw + 2 * 1024;                  // Q scales [128 rows][8]
constexpr int kTOffAlpha = kTOffQsc + 128 * 8;                 // rescale factors [128 rows]
constexpr int kTOffMl = kTOffAlpha + 128 * 4;                  // m [128], l [128]
constexpr int kTOffBars = kTOffMl + 2 * 128 * 4;
// barrier indices
constexpr int kTbStageFull = 0;
constexpr int kTbStageEmpty = kTbStageFull + kTStages;
constexpr int kTbSFull = kTbStageEmpty + kTStages;  // [2]
constexpr int kTbSFree = kTbSFull + 2;              // [2]
constexpr int kTbPFull = kTbSFree + 2;              // [2]
constexpr int kTbVtFull = kTbPFull + 2;             // [kTVtBufs]
constexpr int kTbVtFree = kTbVtFull + kTVtBufs;     // [kTVtBufs]
constexpr int kTbPvDone = kTbVtFree + kTVtBufs;     // [2]
constexpr int kTbQReady = kTbPvDone + 2;
constexpr int kTbOFree = kTbQReady + 1;
constexpr int kTNumBars = kTbOFree + 1;
constexpr int kTOffPid = kTOffBars + kTNumBars * 8;
constexpr int kTOffTmemSlot = kTOffPid + 8 * 4;
constexpr int kTSmemBytes = kTOffTmemSlot + 16;
static_assert(kTStages <= 8, "stage page-id slots");
static_assert(kTSmemBytes <= 227 * 1024, "shared memory budget");

// TMEM columns
constexpr uint32_t kTColS = 0;      // [2 buffers][128 keys]
constexpr uint32_t kTColO = 256;    // O^T: [2 heads][64 rows]
constexpr uint32_t kTColSfa = 384;  // Q scales: [2 k-halves][4]
constexpr uint32_t kTColSfb = 392;  // K scales: [2 buffers][2 k-halves][4]
constexpr uint32_t kTTmemCols = 512;

// instruction descriptors (dense, no negation):
//   Q.K^T: A, B = E2M1 K-major, scale type UE4M3, N = 128, M = 128
//   P.V:   D = f32, A = B = f16, A MN-major, B K-major, N = 64, M = 128
constexpr uint32_t kIdescQKT = (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPVT = (1u << 4) | (1u << 15) | ((64u >> 3) << 17) | ((128u >> 4) << 24);

struct TileParams {
  const uint8_t* q_codes;
  const uint8_t* q_scales;
  const uint8_t* pool;
  const int32_t* block_table;
  int32_t max_pages;
  int32_t num_pages;
  const int4* groups;      // 2 x int4 per group: {seq, pair, rg, len}, {n_seg, first_part, pages, 0}
  const int4* segments;    // {group, page_lo, page_hi, part_slot or -1}
  const int32_t* cta_seg;  // [grid + 1]
  float* partials;         // [num_partials][2][kTPartHeadFloats]
  float* out;
  int32_t* status;
  int32_t Hq, Hkv, G, q_len, causal;
  float c2;                // sm_scale * log2(e)
};

struct TSeg {
  int seq, pair, rg, len, n_seg, first_part, lo, hi, part;
  bool two;  // the pair has both heads (false for the last head of an odd head count)
};

__device__ __forceinline__ TSeg t_load_seg(const TileParams& p, int s) {
  const int4 seg = p.segments[s];
  const int4 g0 = p.groups[2 * seg.x];
  const int4 g1 = p.groups[2 * seg.x + 1];
  TSeg r;
  r.lo = seg.y; r.hi = seg.z; r.part = seg.w;
  r.seq = g0.x; r.pair = g0.y; r.rg = g0.z; r.len = g0.w;
  r.n_seg = g1.x; r.first_part = g1.y;
  r.two = 2 * r.pair + 1 < p.Hkv;
  return r;
}

__device__ __forceinline__ uint32_t tbar(uint32_t bars, int i) { return bars + 8u * (uint32_t)i; }

// --------------------------------------------------------------------------------------------
// Producer warp: lane 0 streams the pair's part of each page (K codes, K scales, V codes, V
// scales: four bulk copies) into a kTStages ring; the other lanes load page ids 32 at a time.
// --------------------------------------------------------------------------------------------
__device__ void t_producer(const TileParams& p, uint8_t* smem, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kTOffBars;
  volatile int32_t* stage_pid = reinterpret_cast<volatile int32_t*>(smem + kTOffPid);
  const int64_t blk = (int64_t)p.Hkv * 9216;
  uint32_t k = 0;
  bool to = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const TSeg sg = t_load_seg(p, s);
    const uint32_t kb = sg.two ? 8192u : 4096u, sb = sg.two ? 1024u : 512u;
    const int64_t offK = (int64_t)sg.pair * 8192, offKs = (int64_t)p.Hkv * 4096 + sg.pair * 1024;
    const int64_t offV = (int64_t)p.Hkv * 4608 + sg.pair * 8192;
    const int64_t offVs = (int64_t)p.Hkv * 8704 + sg.pair * 1024;
    for (int p0 = sg.lo; p0 < sg.hi; p0 += 32) {
      const int n = min(32, sg.hi - p0);
      const int32_t mine =
          (lane < n) ? p.block_table[(int64_t)sg.seq * p.max_pages + p0 + lane] : -1;
      for (int j = 0; j < n; ++j, ++k) {
        const int32_t pid = __shfl_sync(0xffffffffu, mine, j);
        if (lane == 0) {
          const uint32_t st = k % kTStages;
          if (k >= kTStages)
            wait_bar(tbar(bars, kTbStageEmpty + st), ((k / kTStages) - 1) & 1, to);
          const bool valid = pid >= 0 && pid < p.num_pages;
          stage_pid[st] = valid ? pid : -1;
          const uint32_t full = tbar(bars, kTbStageFull + st);
          if (valid) {
            const uint8_t* src = p.pool + (int64_t)pid * blk;
            const uint32_t dst = sbase + kTOffStage + st * kTStageBytes;
            mbar_arrive_expect_tx(full, 2u * (kb + sb));
            bulk_g2s(dst + kStK, src + offK, kb, full);
            bulk_g2s(dst + kStKs, src + offKs, sb, full);
            bulk_g2s(dst + kStV, src + offV, kb, full);
            bulk_g2s(dst + kStVs, src + offVs, sb, full);
          } else {
            flag_status(p.status, KV_NVFP4_DEV_BAD_PAGE);  // the page is skipped (P = 0, V = 0)
            mbar_arrive(full);
          }
        }
        __syncwarp();
      }
    }
  }
  if (lane == 0) {
    // no copy into this CTA's shared memory may still be in flight at exit
    for (uint32_t st = 0; st < kTStages && st < k; ++st) {
      const uint32_t last = k - 1 - ((k - 1 - st) % kTStages);
      wait_bar(tbar(bars, kTbStageFull + st), (last / kTStages) & 1, to);
    }
    if (to) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
  }
}

// --------------------------------------------------------------------------------------------
// MMA warp. A tcgen05 instruction takes this warp tens of cycles to issue, so the Q.K^T of a page
// is issued two pages ahead of its softmax: per segment, Q.K^T of its first two pages, then for
// each page k the Q.K^T of page k + 2 (into the S buffer whose scores the softmax of page k has
// read, first thing) followed by the P.V of page k (it waits for that page's P and V tiles). A segment's first P.V
// overwrites O^T; it waits until the previous segment's epilogue has read O^T. The shared-memory
// descriptors are built once and advanced by adding the byte offset / 16 to the address field.
// --------------------------------------------------------------------------------------------
struct MmaDescs {
  uint64_t q, k, vt, p, sfk, sfw;  // descriptors of offset 0 of each region
};

__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) {
  return d + (uint64_t)(bytes >> 4);  // start-address field: addresses stay below 2^18
}

// Q.K^T of page kq: K scales to TMEM, two MMAs (k-halves) into S buffer kq % 2.
__device__ __forceinline__ void t_issue_qk(const MmaDescs& D, uint32_t sbase, uint32_t bars,
                                           uint32_t tbase, uint32_t kq, bool two, int lane,
                                           bool& to) {
  const uint32_t st = kq % kTStages, b = kq & 1u;
  wait_bar(tbar(bars, kTbStageFull + st), (kq / kTStages) & 1, to);
  // S buffer b free: the softmax warps have read S of page kq - 2
  if (kq >= 2) wait_bar(tbar(bars, kTbSFree + b), ((kq >> 1) - 1) & 1, to);
  const uint32_t soff = kTOffStage + st * kTStageBytes;
  if (!two) {  // a lone head's 8-byte scale rows widened to 16 (the absent head's half 0)
    const uint32_t sfw = sbase + kTOffSfw + b * 1024;
#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
      const uint2 v = lds64(sbase + soff + kStKs + kh * 256 + lane * 8);
      sts128(sfw + kh * 512 + lane * 16, v.x, v.y, 0u, 0u);
    }
    fence_async_smem();
  }
  __syncwarp();
  if (lane == 0) {
    tc_fence_after();
    const uint64_t sf = two ? desc_add(D.sfk, soff) : desc_add(D.sfw, b * 1024);
    tmem_cp_32x128b_x4(tbase + kTColSfb + b * 8, sf);
    tmem_cp_32x128b_x4(tbase + kTColSfb + b * 8 + 4, desc_add(sf, 512));
    const uint64_t kd = desc_add(D.k, soff);
    mma_nvf4_ss(tbase + kTColS + b * 128, D.q, kd, kIdescQKT, tbase + kTColSfa,
                tbase + kTColSfb + b * 8, 0u);
    mma_nvf4_ss(tbase + kTColS + b * 128, desc_add(D.q, 256), desc_add(kd, 256), kIdescQKT,
                tbase + kTColSfa + 4, tbase + kTColSfb + b * 8 + 4, 1u);
    // (the stage's K is released by the softmax warps, which arrive on its empty barrier after
    // S is complete)
    mma_commit(tbar(bars, kTbSFull + b));
  }
  __syncwarp();
}

// P.V of page kk: per head, four MMAs (16 keys each) into O^T.
__device__ __forceinline__ void t_issue_pv(const MmaDescs& D, uint32_t bars, uint32_t tbase,
                                           uint32_t kk, bool first, bool two, int lane,
                                           bool& to) {
  const uint32_t b = kk & 1u, v = kk % kTVtBufs;
  wait_bar(tbar(bars, kTbPFull + b), (kk >> 1) & 1, to);
  wait_bar(tbar(bars, kTbVtFull + v), (kk / kTVtBufs) & 1, to);
  if (lane == 0) {
    tc_fence_after();
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      if (hh == 1 && !two) break;
      const uint64_t ad = desc_add(D.vt, (v * 2 + hh) * kVtHeadBytes);
      const uint64_t bd = desc_add(D.p, (b * 2 + hh) * kPHeadBytes);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)  // 16 keys per instruction
        mma_f16_ss(tbase + kTColO + hh * 64, desc_add(ad, ks * 4096), desc_add(bd, ks * 256),
                   kIdescPVT, (first && ks == 0) ? 0u : 1u);
    }
    mma_commit(tbar(bars, kTbPvDone + b));
    mma_commit(tbar(bars, kTbVtFree + v));
  }
  __syncwarp();
}

__device__ void t_mma(const TileParams& p, uint8_t* smem, uint32_t tbase, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kTOffBars;
  MmaDescs D;
  D.q = smem_desc(sbase + kTOffQ, 128, 512);
  D.k = smem_desc(sbase + kStK, 128, 512);          // + stage offset
  D.sfk = smem_desc(sbase + kStKs, 16, 128);        // + stage offset
  D.sfw = smem_desc(sbase + kTOffSfw, 16, 128);
  D.vt = smem_desc(sbase + kTOffVt, 2048, 128);
  D.p = smem_desc(sbase + kTOffP, 128, 1024);
  uint32_t k = 0, sgi = 0;
  bool to = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s, ++sgi) {
    const TSeg sg = t_load_seg(p, s);
    const int n = sg.hi - sg.lo;
    wait_bar(tbar(bars, kTbQReady), sgi & 1, to);  // this segment's Q tile and its scales
    t_issue_qk(D, sbase, bars, tbase, k, sg.two, lane, to);
    if (n > 1) t_issue_qk(D, sbase, bars, tbase, k + 1, sg.two, lane, to);
    for (int j = 0; j < n; ++j) {
      // S buffer of page k + j + 2 is free once the softmax of page k + j has read its scores,
      // early in that softmax; its P.V waits for the end of it
      if (j + 2 < n) t_issue_qk(D, sbase, bars, tbase, k + j + 2, sg.two, lane, to);
      if (j == 0 && sgi > 0) wait_bar(tbar(bars, kTbOFree), (sgi - 1) & 1, to);
      t_issue_pv(D, bars, tbase, k + j, j == 0, sg.two, lane, to);
    }
    k += n;
  }
  if (to) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// --------------------------------------------------------------------------------------------
// V dequantisation warps: warp hh converts head hh of the pair, lane l the key rows l and l + 32
// (64 code bytes and 8 scales each) into 128 f16 values of the MN-major tile (core matrix = 8 keys
// x 8 dims, dims contiguous); zeros for a key past the sequence end or on a skipped page. The
// 16-byte loads of a row are rotated by key so that the eight keys of a quarter-warp read distinct
// banks. The two warps sit on the sub-partitions that hold neither the producer nor the MMA warp.
// --------------------------------------------------------------------------------------------
// One key row's loads: 64 code bytes (rotated 16-byte pieces) and 8 scales.
struct VRow {
  uint4 cw[4];
  uint2 sc8;
};

__device__ __forceinline__ void t_vrow_load(uint32_t stage, int hh, int key, VRow& r) {
  const int rot = (key >> 1) & 3;
  r.sc8 = lds64(stage + kStVs + hh * 512 + key * 8);
#pragma unroll
  for (int qq = 0; qq < 4; ++qq)
    r.cw[qq] = lds128(stage + kStV + hh * 4096 + key * 64 + 16 * ((qq + rot) & 3));
}

__device__ __forceinline__ void t_vrow_store(const VRow& r, uint32_t dst_tile, int key, bool ok) {
  const uint32_t dst = dst_tile + (key >> 3) * 2048 + (key & 7) * 16;
  const int rot = (key >> 1) & 3;
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    const int q4 = (qq + rot) & 3;  // 16 code bytes = dims 32 q4 .. 32 q4 + 31
    // scales of blocks 2 q4 (dims 32 q4 ..) and 2 q4 + 1 (dims 32 q4 + 16 ..); 0 past the end
    const uint32_t two_sc = ok ? ((q4 < 2 ? r.sc8.x : r.sc8.y) >> (16 * (q4 & 1))) & 0xFFFFu : 0u;
    const uint32_t sh = cvt_e4m3x2_f16(two_sc);
    const uint32_t s0 = dup_lo(sh), s1 = dup_hi(sh);
    const uint32_t words[4] = {r.cw[qq].x, r.cw[qq].y, r.cw[qq].z, r.cw[qq].w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {  // word w: dims 32 q4 + 8 w .. + 7 (byte = dims 2i, 2i + 1)
      uint32_t r0, r1, r2, r3;
      cvt_e2m1x8_f16(words[w], r0, r1, r2, r3);
      const uint32_t sc = w < 2 ? s0 : s1;
      sts128(dst + (4 * q4 + w) * 128, hmul2(r0, sc), hmul2(r1, sc), hmul2(r2, sc),
             hmul2(r3, sc));
    }
  }
}

__device__ void t_dequant(const TileParams& p, uint8_t* smem, int warp, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kTOffBars;
  const volatile int32_t* stage_pid = reinterpret_cast<const volatile int32_t*>(smem + kTOffPid);
  const int hh = warp - kTWarpDeq0;
  uint32_t k = 0;
  bool to = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const TSeg sg = t_load_seg(p, s);
    const bool head_ok = hh == 0 || sg.two;
    for (int page = sg.lo; page < sg.hi; ++page, ++k) {
      const uint32_t st = k % kTStages, v = k % kTVtBufs;
      wait_bar(tbar(bars, kTbStageFull + st), (k / kTStages) & 1, to);
      // V tile v free once the P.V of page k - kTVtBufs is complete
      if (k >= kTVtBufs) wait_bar(tbar(bars, kTbVtFree + v), ((k / kTVtBufs) - 1) & 1, to);
      if (head_ok) {
        const bool pvalid = stage_pid[st] >= 0;
        const uint32_t stage = sbase + kTOffStage + st * kTStageBytes;
        const uint32_t tile = sbase + kTOffVt + (v * 2 + hh) * kVtHeadBytes;
        // both rows' loads first, then the conversions (the stores would otherwise order each
        // load after the previous row piece's stores). A key past the sequence end or on a
        // skipped page gets scale 0: its stale code bytes turn into zeros.
        VRow r0, r1;
        t_vrow_load(stage, hh, lane, r0);
        t_vrow_load(stage, hh, lane + 32, r1);
        t_vrow_store(r0, tile, lane, pvalid && page * kPage + lane < sg.len);
        t_vrow_store(r1, tile, lane + 32, pvalid && page * kPage + lane + 32 < sg.len);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(tbar(bars, kTbVtFull + v));
        mbar_arrive(tbar(bars, kTbStageEmpty + st));
      }
    }
  }
  if (to && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// --------------------------------------------------------------------------------------------
// Softmax warps. Thread (quadrant q, lane) owns tile row r = 32 q + lane (TMEM lane r of S): head
// 2 pair + r / 64, tile row r % 64; in the epilogue and the O rescale the same thread owns head
// dimension r (TMEM lane r of O^T).
// --------------------------------------------------------------------------------------------
// The segment's Q tile: codes into the A operand tile (tile order), scales into TMEM in the
// replicated scale-factor layout (lane i, column w of a k-half: scales of rows 32 w + i).
__device__ __forceinline__ void t_load_q(const TileParams& p, const TSeg& sg, uint8_t* smem,
                                         uint32_t sbase, uint32_t tbase, uint32_t lane_base, int r,
                                         int lane) {
  const int hh = r >> 6, i = r & 63;
  const int head = 2 * sg.pair + hh, gr = sg.rg * kTRows + i;
  uint4 c[4];
  uint2 sc = make_uint2(0u, 0u);
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) c[ch] = make_uint4(0u, 0u, 0u, 0u);
  if (head < p.Hkv && gr < p.G * p.q_len) {
    const int64_t qrow = ((int64_t)sg.seq * p.q_len + gr / p.G) * p.Hq + head * p.G + gr % p.G;
    const uint4* src = reinterpret_cast<const uint4*>(p.q_codes + qrow * kCodeBytes);
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) c[ch] = src[ch];
    sc = *reinterpret_cast<const uint2*>(p.q_scales + qrow * kScaleBytes);
  }
#pragma unroll
  for (int ch = 0; ch < 4; ++ch)
    sts128(sbase + kTOffQ + (r >> 3) * 512 + ch * 128 + (r & 7) * 16, c[ch].x, c[ch].y, c[ch].z,
           c[ch].w);
  *reinterpret_cast<uint2*>(smem + kTOffQsc + r * 8) = sc;
  named_barrier_sync(kNbSoft, 128);
  uint32_t sf[8];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint2 v = *reinterpret_cast<const uint2*>(smem + kTOffQsc + (32 * w + lane) * 8);
    sf[w] = v.x;
    sf[4 + w] = v.y;
  }
  tmem_st8(tbase + lane_base + kTColSfa, sf);
  tmem_wait_st();
  fence_async_smem();
  tc_fence_before();
  __syncwarp();
}

__device__ void t_softmax(const TileParams& p, uint8_t* smem, uint32_t tbase, int warp,
                          int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kTOffBars;
  const volatile int32_t* stage_pid = reinterpret_cast<const volatile int32_t*>(smem + kTOffPid);
  float* alpha_s = reinterpret_cast<float*>(smem + kTOffAlpha);
  float* ml_s = reinterpret_cast<float*>(smem + kTOffMl);
  const int q = warp & 3;
  const int r = 32 * q + lane;
  const int hh = r >> 6, i = r & 63;
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const float c2 = p.c2;
  const int rows_total = p.G * p.q_len;
  uint32_t k = 0, sgi = 0;
  bool to = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  if (s_begin < s_end) {
    t_load_q(p, t_load_seg(p, s_begin), smem, sbase, tbase, lane_base, r, lane);
    if (lane == 0) mbar_arrive(tbar(bars, kTbQReady));
  }
  for (int s = s_begin; s < s_end; ++s, ++sgi) {
    const TSeg sg = t_load_seg(p, s);
    const int n = sg.hi - sg.lo;
    const int head = 2 * sg.pair + hh, gr = sg.rg * kTRows + i;
    const bool row_ok = head < p.Hkv && gr < rows_total;
    // largest visible key position of this row (-1: no key)
    const int limit = row_ok ? (p.causal ? sg.len - p.q_len + gr / p.G : sg.len - 1) : -1;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < n; ++j, ++k) {
      const uint32_t b = k & 1u, st = k % kTStages;
      wait_bar(tbar(bars, kTbSFull + b), (k >> 1) & 1, to);
      tc_fence_after();
      uint32_t s_lo[32], s_hi[32];  // scores of keys 0..31, 32..63 of this row's head
      {
        const uint32_t col = tbase + lane_base + kTColS + b * 128 + hh * 64;
        tmem_ld32(col, s_lo);
        tmem_ld32(col + 32, s_hi);
        tmem_wait_ld_regs32(s_lo);
        tmem_wait_ld_regs32(s_hi);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tbar(bars, kTbSFree + b));
      // the page id, published before the stage's full barrier completed; S complete means the
      // Q.K^T MMAs have read the stage's K, which this warp's arrival releases with the page id
      wait_bar(tbar(bars, kTbStageFull + st), (k / kTStages) & 1, to);
      const bool pvalid = stage_pid[st] >= 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(tbar(bars, kTbStageEmpty + st));
      const int kp0 = (sg.lo + j) * kPage;
      const int nvis = pvalid ? max(0, min(kPage, limit - kp0 + 1)) : 0;  // keys c < nvis visible
      const bool full = nvis == kPage;
      // page max of the row: eight independent chains, then a tree
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
      if (full) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(s_lo[c]));
          mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(s_hi[c]));
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          mx[c & 7] = fmaxf(mx[c & 7], c < nvis ? __uint_as_float(s_lo[c]) : -INFINITY);
          mx[c & 7] = fmaxf(mx[c & 7], c + 32 < nvis ? __uint_as_float(s_hi[c]) : -INFINITY);
        }
      }
      const float pmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float mc = fmaxf(m, pmax);
      if (j == 0) {
        m = mc;  // nothing accumulated yet in this segment
      } else {
        const bool need = mc > m && (m == -INFINITY || (mc - m) * c2 > kLazyMax);
        if (named_barrier_any(kNbSoft, 128, need)) {
          // all P.V MMAs so far complete before O^T is rescaled
          wait_bar(tbar(bars, kTbPvDone + ((k - 1) & 1u)), ((k - 1) >> 1) & 1, to);
          tc_fence_after();
          const float alpha = (mc == m) ? 1.f : fast_exp2((m - mc) * c2);  // 0 when m was -inf
          l *= alpha;
          m = mc;
          alpha_s[r] = alpha;
          named_barrier_sync(kNbSoft, 128);
#pragma unroll 1
          for (int cc = 0; cc < (sg.two ? 4 : 2); ++cc) {  // O^T columns 32 cc .. (rows of the tile)
            uint32_t o[32];
            const uint32_t col = tbase + lane_base + kTColO + cc * 32;
            tmem_ld32(col, o);
            tmem_wait_ld_regs32(o);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 a = *reinterpret_cast<const float4*>(alpha_s + cc * 32 + e);
              o[e] = __float_as_uint(__uint_as_float(o[e]) * a.x);
              o[e + 1] = __float_as_uint(__uint_as_float(o[e + 1]) * a.y);
              o[e + 2] = __float_as_uint(__uint_as_float(o[e + 2]) * a.z);
              o[e + 3] = __float_as_uint(__uint_as_float(o[e + 3]) * a.w);
            }
            tmem_st32(col, o);
          }
          tmem_wait_st();
        }
      }
      // P tile b free once the P.V of page k - 2 is complete
      if (k >= 2) wait_bar(tbar(bars, kTbPvDone + b), ((k >> 1) - 1) & 1, to);
      const float mc2 = m * c2;
      const uint32_t prow = sbase + kTOffP + (b * 2 + hh) * kPHeadBytes + (i >> 3) * 1024 + (i & 7) * 16;
      float ls[8];  // row-sum partials, one per 8 keys
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        float pv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = 8 * c8 + e;
          const float x = __uint_as_float(c < 32 ? s_lo[c & 31] : s_hi[c & 31]);
          const float pe = fast_exp2(fmaf(x, c2, -mc2));
          pv[e] = (full || c < nvis) ? pe : 0.f;
        }
        ls[c8] = ((pv[0] + pv[1]) + (pv[2] + pv[3])) + ((pv[4] + pv[5]) + (pv[6] + pv[7]));
        sts128(prow + c8 * 128, pack_f16x2(pv[0], pv[1]), pack_f16x2(pv[2], pv[3]),
               pack_f16x2(pv[4], pv[5]), pack_f16x2(pv[6], pv[7]));
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tbar(bars, kTbPFull + b));
    }

    // ---- segment end: the next segment's Q tile (every Q.K^T of this one is complete), then
    // the epilogue of this one ----
    if (s + 1 < s_end) {
      t_load_q(p, t_load_seg(p, s + 1), smem, sbase, tbase, lane_base, r, lane);
      if (lane == 0) mbar_arrive(tbar(bars, kTbQReady));
    }
    const uint32_t kl = k - 1;
    wait_bar(tbar(bars, kTbPvDone + (kl & 1u)), (kl >> 1) & 1, to);
    tc_fence_after();
    named_barrier_sync(kNbSoft, 128);  // the previous epilogue's reads of m, l are done
    ml_s[r] = m;
    ml_s[128 + r] = l;
    named_barrier_sync(kNbSoft, 128);
    const bool split = sg.n_seg > 1;
    const int d = r;  // this thread's head dimension in O^T
    float* part = split ? p.partials + (int64_t)sg.part * 2 * kTPartHeadFloats : nullptr;
#pragma unroll 1
    for (int cc = 0; cc < (sg.two ? 4 : 2); ++cc) {
      uint32_t o[32];
      tmem_ld32(tbase + lane_base + kTColO + cc * 32, o);
      tmem_wait_ld_regs32(o);
      const int h2 = cc >> 1;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int i2 = (cc & 1) * 32 + e, g2 = sg.rg * kTRows + i2;
        if (g2 >= rows_total) continue;
        const float v = __uint_as_float(o[e]);
        if (split) {
          part[h2 * kTPartHeadFloats + i2 * 128 + d] = v;
        } else {
          const float l2 = ml_s[128 + h2 * 64 + i2];
          if (l2 > 0.f) {
            const int tok = g2 / p.G, qh = (2 * sg.pair + h2) * p.G + g2 % p.G;
            p.out[(((int64_t)sg.seq * p.q_len + tok) * p.Hq + qh) * 128 + d] = v / l2;
          }
        }
      }
    }
    if (split && row_ok) {
      part[hh * kTPartHeadFloats + kTRows * 128 + i] = m;
      part[hh * kTPartHeadFloats + kTRows * 128 + kTRows + i] = l;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tbar(bars, kTbOFree));
  }
  if (to && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

__global__ void __launch_bounds__(kTThreads, 1) tile_kernel(const TileParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = smem_u32(smem + kTOffBars);
  // the split-K merge launched after this kernel may be scheduled now; it waits for this grid's
  // completion before it reads anything this kernel writes
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(tbar(bars, kTbStageFull + s), 1);
      // dequant warps (V read), softmax warps (S complete, so K read; page id read)
      mbar_init(tbar(bars, kTbStageEmpty + s), kTDeqWarps + 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tbar(bars, kTbSFull + b), 1);
      mbar_init(tbar(bars, kTbSFree + b), 4);
      mbar_init(tbar(bars, kTbPFull + b), 4);
      mbar_init(tbar(bars, kTbPvDone + b), 1);
    }
    for (int v = 0; v < kTVtBufs; ++v) {
      mbar_init(tbar(bars, kTbVtFull + v), kTDeqWarps);
      mbar_init(tbar(bars, kTbVtFree + v), 1);
    }
    mbar_init(tbar(bars, kTbQReady), 4);
    mbar_init(tbar(bars, kTbOFree), 4);
    fence_mbar_init();
  }
  if (warp == kTWarpMma) tmem_alloc(smem_u32(smem + kTOffTmemSlot), kTTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // launched as a programmatic dependent of the previous kernel on the stream (the append that
  // wrote the pool rows and Q, or the previous call's merge, which reads the partials this kernel
  // rewrites): nothing below runs before it completes
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(smem + kTOffTmemSlot);

  if (warp == kTWarpProducer) {
    t_producer(p, smem, lane);
  } else if (warp == kTWarpMma) {
    t_mma(p, smem, tbase, lane);
  } else if (warp >= kTWarpSoft0 && warp < kTWarpDeq0) {
    t_softmax(p, smem, tbase, warp, lane);
  } else {
    t_dequant(p, smem, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTWarpMma) tmem_dealloc(tbase, kTTmemCols);
}

// --------------------------------------------------------------------------------------------
// Split-K merge of the tile kernel's partials (second launch): one CTA per (split group, head of
// the pair, row of the tile); its 256 threads are 8 slices of the group's partials x 32 four-dim
// columns:  M = max_q m_q,  L = sum_q 2^((m_q - M) c2) l_q,  o = sum_q 2^((m_q - M) c2) O_q / L.
// --------------------------------------------------------------------------------------------
struct TMergeParams {
  const int4* groups;
  const int32_t* split;    // [num_split] group indices
  const float* partials;   // [num_partials][2][kTPartHeadFloats]
  float* out;
  int32_t Hq, Hkv, G, q_len;
  float c2;
};

__global__ void __launch_bounds__(256) tile_merge_kernel(const TMergeParams p) {
  __shared__ float s_m[8], s_l[8];
  __shared__ float4 s_o[8][32];
  asm volatile("griddepcontrol.launch_dependents;");
  const int gi = p.split[blockIdx.x];  // plan tables: written before the attention launch
  const int hh = blockIdx.y / kTRows, i = blockIdx.y % kTRows;
  const int4 g0 = p.groups[2 * gi], g1 = p.groups[2 * gi + 1];
  const int r = g0.z * kTRows + i, head = 2 * g0.y + hh;
  // the partials are visible only after the attention grid has completed and flushed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (head >= p.Hkv || r >= p.G * p.q_len) return;  // uniform over the CTA
  const int n_seg = g1.x;
  const int slice = threadIdx.x >> 5, d4 = threadIdx.x & 31;
  const int64_t stride = 2 * (int64_t)kTPartHeadFloats;
  const float* base = p.partials + (int64_t)g1.y * stride + hh * kTPartHeadFloats;
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int q = slice; q < n_seg; q += 8) {
    const float* pq = base + q * stride;
    const float mq = __ldcg(pq + kTRows * 128 + i);
    const float lq = __ldcg(pq + kTRows * 128 + kTRows + i);
    const float4 ov = __ldcg(reinterpret_cast<const float4*>(pq + i * 128) + d4);
    if (mq == -INFINITY) continue;  // a segment with no visible key for this row
    const float mn = fmaxf(M, mq);
    const float a = fast_exp2((M - mn) * p.c2), f = fast_exp2((mq - mn) * p.c2);
    M = mn;
    L = L * a + f * lq;
    O.x = O.x * a + f * ov.x; O.y = O.y * a + f * ov.y;
    O.z = O.z * a + f * ov.z; O.w = O.w * a + f * ov.w;
  }
  s_o[slice][d4] = O;
  if (d4 == 0) { s_m[slice] = M; s_l[slice] = L; }
  __syncthreads();
  if (slice == 0) {
    float Mt = s_m[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) Mt = fmaxf(Mt, s_m[j]);
    float Lt = 0.f;
    float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (s_m[j] == -INFINITY) continue;
      const float f = fast_exp2((s_m[j] - Mt) * p.c2);
      const float4 v = s_o[j][d4];
      Lt += f * s_l[j];
      Ot.x += f * v.x; Ot.y += f * v.y; Ot.z += f * v.z; Ot.w += f * v.w;
    }
    if (Lt > 0.f) {
      const int tok = r / p.G, qh = head * p.G + r % p.G;
      float4* dst = reinterpret_cast<float4*>(
          p.out + (((int64_t)g0.x * p.q_len + tok) * p.Hq + qh) * 128 + 4 * d4);
      *dst = make_float4(Ot.x / Lt, Ot.y / Lt, Ot.z / Lt, Ot.w / Lt);
    }
  }
}

}  // namespace

int tile_smem_bytes() { return kTSmemBytes; }

// Attention for tiles of 64 rows per head of a KV-head pair (see the top of this file), then the
// merge of the split groups' partials; both launched as programmatic dependents on the stream.
cudaError_t launch_tile(const uint8_t* q_codes, const uint8_t* q_scales, const uint8_t* pool,
                        const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                        const void* groups, const void* segments, const int32_t* cta_seg,
                        const int32_t* split_groups, int32_t num_split, float* partials,
                        float* out, int32_t* status, int32_t Hq, int32_t Hkv, int32_t q_len,
                        int32_t causal, int32_t grid, float sm_scale, cudaStream_t stream) {
  // the attribute belongs to each device: set once per device
  static bool attr_done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(tile_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kTSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  if (Hkv < 1) return cudaErrorInvalidValue;
  TileParams p;
  p.q_codes = q_codes; p.q_scales = q_scales; p.pool = pool;
  p.block_table = block_table; p.max_pages = max_pages; p.num_pages = num_pages;
  p.groups = reinterpret_cast<const int4*>(groups);
  p.segments = reinterpret_cast<const int4*>(segments);
  p.cta_seg = cta_seg;
  p.partials = partials; p.out = out; p.status = status;
  p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv; p.q_len = q_len; p.causal = causal;
  p.c2 = sm_scale * 1.4426950408889634f;
  if (grid <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kTThreads);
    cfg.dynamicSmemBytes = kTSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, tile_kernel, p);
    if (le != cudaSuccess) return le;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || num_split <= 0) return e;
  TMergeParams mp;
  mp.groups = p.groups; mp.split = split_groups; mp.partials = partials; mp.out = out;
  mp.Hq = Hq; mp.Hkv = Hkv; mp.G = p.G; mp.q_len = q_len; mp.c2 = p.c2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_split, 2u * kTRows);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tile_merge_kernel, mp);
}

}  // namespace kvnvfp4
