// Paged GQA attention over the NVFP4 cache for query tiles of many rows (speculative verify,
// prefill chunks), with both products on the tcgen05 tensor cores.
//
// Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)": the Q.K^T
// product in NVFP4 with E4M3 block scales (both Q and K quantised), V dequantised for the P.V
// product. The tile decomposition, the lazily raised running max and the split-K merge are this
// library's design; the pages say nothing about the kernel's decomposition.
//
// Work decomposition. A group is (sequence, KV head, tile of 128 query rows of that head), a row
// being (query token, head in the GQA group) as in the decode kernel. The plan lays the groups'
// pages end to end and gives each persistent CTA a contiguous, page-balanced share (segments); a
// group spread over several CTAs leaves one (m, l, O) partial per segment, merged by a second
// launch. Keys are taken in blocks of 128 (two pages of the head; the last block of a segment may
// hold one).
//
// Per block (the head's part of two pages, 19 KB in eight bulk copies):
//   Q.K^T: tcgen05.mma kind::mxf4nvf4 block_scale.scale_vec::4X, M = 128 query rows, N = 128
//     keys, K = 64 per instruction (two per 128-dim row) into one of two S buffers in tensor
//     memory. The K codes are used as the pool stores them (tensor-core tile order); the Q.K^T
//     warp gathers the head's K scales of the two pages into the scale-factor copy's row order
//     ahead of time.
//   Softmax: eight warps, two per tensor-memory lane quadrant: one query row per thread (lane =
//     row) and 64 of the block's 128 keys per warp, fp32 online softmax. The two warps of a
//     quadrant exchange their partial row maxima through shared memory. The running max m of a
//     row is raised only when a block's max exceeds it by more than 2^15 in the exp2 domain (the
//     warps then rescale their halves of the row of O in tensor memory), so P = exp2((s - m) c2)
//     <= 2^15 fits f16 (largest finite value 65504). Each warp writes its 64 P values in f16
//     pairs over the first 32 of its own 64 S columns, where the P.V product reads them as its A
//     operand. Tiles of at most 64 rows (speculative verify) run in split-page mode: the rows are
//     repeated in lanes 64..127 and each lane set takes one page of the block, 32 keys per warp,
//     so that the exponentials run on all four SM sub-partitions (see the softmax warps below).
//   V: four warps dequantise the block's V rows (E2M1 x E4M3 is exact in f16), one key row per
//     thread, into an MN-major f16 tile in shared memory.
//   P.V: tcgen05.mma kind::f16, O[rows][dims] += P V with M = 128 rows (A = P in tensor memory),
//     N = 144 (B = the dequantised V tile: the 128 head dims, a column of ones and 15 of zeros),
//     K = 16 keys per instruction (eight per block). The column of ones makes the tensor core
//     accumulate each row's sum of P (the softmax denominator l) beside O, in fp32, from the very
//     f16 P values the product uses; O and l stay in tensor memory for the whole segment.
// Two S buffers and two V tiles: the Q.K^T and the dequantisation of block j + 1 run while the
// softmax and the P.V of block j do.
//
// Warp roles (480 threads): warp 0 bulk-copy producer, warp 1 Q.K^T issuer and tensor-memory
// owner, warps 2..9 softmax and epilogue (warp w: lane quadrant w mod 4, key half (w - 2) / 4),
// warps 10..13 V dequantisation, warp 14 P.V issuer. The two MMA issuers sit on different SM
// sub-partitions (warp w runs on sub-partition w mod 4), so that issuing one block's P.V and
// the next block's Q.K^T overlap. Every wait is an mbarrier wait bounded in time; on a timeout the kernel
// records KV_NVFP4_DEV_TIMEOUT and carries on, so it cannot hang.
//
// Barriers per block kb (S buffer and V tile b = kb mod 2, stage kb mod 4):
//   StageFull   producer copies landed            -> Q.K^T warp (K scales), V warps
//   SFull[b]    Q.K^T complete (commit)           -> softmax
//   StageEmpty  Q.K^T complete (commit) and V warps done with the stage
//   PFull[b]    softmax wrote P, V warps wrote V  -> P.V warp issues P.V
//   PvDone[b]   P.V complete (commit)             -> S buffer b and V tile b free; O readable

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

namespace {

constexpr int kTRows = 128;                 // query rows of one KV head in a tile
constexpr int kTStages = 4;                 // key blocks in flight
// one block in a stage: the head's K codes of both pages (tile order, adjacent so that the 128
// keys form one B operand), the K scales of the head's pair (or lone head) per page, V codes,
// V scales
constexpr int kStK = 0, kStKs = 8192, kStV = 10240, kStVs = 18432;
constexpr int kTStageBytes = 19456;
constexpr int kVtCols = 144;                // B operand columns: 128 dims, ones, 15 zeros
constexpr int kVtGroupBytes = kVtCols * 16; // one 8-key group of the V tile: 18 chunks of 8 x 8
constexpr int kVtBytes = 16 * kVtGroupBytes;  // dequantised V of a block: 128 keys, f16
constexpr int kTPartFloats = kTRows * 128 + 2 * kTRows;  // a partial: O[rows][128], m[], l[]

constexpr int kTWarpProducer = 0, kTWarpMma = 1, kTWarpSoft0 = 2, kTSoftWarps = 8;
constexpr int kTWarpDeq0 = kTWarpSoft0 + kTSoftWarps, kTDeqWarps = 4;
constexpr int kTWarpPv = kTWarpDeq0 + kTDeqWarps;
constexpr int kTThreads = (kTWarpPv + 1) * 32;
constexpr uint32_t kNbQ = 1;                // named barrier: the four softmax warps that load Q
constexpr uint32_t kNbPair = 2;             // named barriers 2..5: the two warps of a quadrant
constexpr float kLazyMax = 15.0f;           // raise the running max only past 2^15 (exp2 domain)

// shared memory map
constexpr int kTOffStage = 0;
constexpr int kTOffQ = kTOffStage + kTStages * kTStageBytes;  // [128 rows][64 B], tile order
constexpr int kTOffVt = kTOffQ + 8192;                         // [2] V tiles
constexpr int kTOffSfk = kTOffVt + 2 * kVtBytes;               // [kTStages][2 k-halves][512 B]
constexpr int kTOffQsc = kTOffSfk + kTStages * 1024;           // Q scales [128 rows][8]
// row maxima of the softmax warps: [2 parities][2 halves][128 rows] f32, or in split-page mode
// [2 parities][4 warps][64 rows]
constexpr int kTOffRed = kTOffQsc + 128 * 8;
constexpr int kTOffXch = kTOffRed + 2 * 2 * 128 * 4;           // split-page epilogue: O, l of 64 rows
constexpr int kTXchOBytes = 64 * 128 * 4;
constexpr int kTOffBars = kTOffXch + kTXchOBytes + 64 * 4;
// barrier indices
constexpr int kTbStageFull = 0;
constexpr int kTbStageEmpty = kTbStageFull + kTStages;
constexpr int kTbSFull = kTbStageEmpty + kTStages;  // [2]
constexpr int kTbPFull = kTbSFull + 2;              // [2]
constexpr int kTbPvDone = kTbPFull + 2;             // [2]
constexpr int kTbQReady = kTbPvDone + 2;
constexpr int kTbOFree = kTbQReady + 1;
constexpr int kTbDrain = kTbOFree + 1;              // every tcgen05 op of both issuers complete
constexpr int kTNumBars = kTbDrain + 1;
constexpr int kTOffPid = kTOffBars + kTNumBars * 8;            // [kTStages][2] page ids or -1
constexpr int kTOffTmemSlot = kTOffPid + kTStages * 2 * 4;
constexpr int kTSmemBytes = kTOffTmemSlot + 16;
static_assert(kTSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kTOffXch % 16 == 0, "16-byte accesses of the exchange area");

// TMEM columns
constexpr uint32_t kTColS = 0;      // [2 buffers][128 keys]; P (f16 pairs) at 0..31 and 64..95
constexpr uint32_t kTColO = 256;    // O: [128 dims], then l, then 15 zero columns
constexpr uint32_t kTColSfa = 400;  // Q scales: [2 k-halves][4]
constexpr uint32_t kTColSfb = 408;  // K scales: [2 buffers][2 k-halves][4]
constexpr uint32_t kTTmemCols = 512;

// instruction descriptors (dense, no negation):
//   Q.K^T: A, B = E2M1 K-major, scale type UE4M3, N = 128, M = 128
//   P.V:   D = f32, A = B = f16, A K-major (tensor memory), B MN-major, N = 144, M = 128
constexpr uint32_t kIdescQK = (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV =
    (1u << 4) | (1u << 16) | (((uint32_t)kVtCols >> 3) << 17) | ((128u >> 4) << 24);

struct TileParams {
  const uint8_t* q_codes;
  const uint8_t* q_scales;
  const uint8_t* pool;
  const int32_t* block_table;
  int32_t max_pages;
  int32_t num_pages;
  const int4* groups;      // 2 x int4 per group: {seq, kv head, rg, len}, {n_seg, first_part, pages, 0}
  const int4* segments;    // {group, page_lo, page_hi, part_slot or -1}
  const int32_t* cta_seg;  // [grid + 1]
  float* partials;         // [num_partials][kTPartFloats]
  float* out;
  int32_t* status;
  int32_t Hq, Hkv, G, q_len, causal;
  float c2;                // sm_scale * log2(e)
};

struct TSeg {
  int seq, head, rg, len, n_seg, first_part, lo, hi, part;
};

__device__ __forceinline__ TSeg t_load_seg(const TileParams& p, int s) {
  const int4 seg = p.segments[s];
  const int4 g0 = p.groups[2 * seg.x];
  const int4 g1 = p.groups[2 * seg.x + 1];
  TSeg r;
  r.lo = seg.y; r.hi = seg.z; r.part = seg.w;
  r.seq = g0.x; r.head = g0.y; r.rg = g0.z; r.len = g0.w;
  r.n_seg = g1.x; r.first_part = g1.y;
  return r;
}

__device__ __forceinline__ uint32_t tbar(uint32_t bars, int i) { return bars + 8u * (uint32_t)i; }

// key blocks (two pages each) of a segment
__device__ __forceinline__ int seg_blocks(const TSeg& sg) { return (sg.hi - sg.lo + 1) >> 1; }

// --------------------------------------------------------------------------------------------
// Producer warp: lane 0 streams the head's part of each page (K codes, K scales, V codes, V
// scales: four bulk copies per page) into the kTStages ring, two pages per stage; the other lanes
// load page ids 32 at a time.
// --------------------------------------------------------------------------------------------
__device__ void t_producer(const TileParams& p, uint8_t* smem, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kTOffBars;
  volatile int32_t* stage_pid = reinterpret_cast<volatile int32_t*>(smem + kTOffPid);
  const int64_t blk = (int64_t)p.Hkv * 9216;
  // with one row tile per (sequence, KV head) (verify) a page is read once per call: marked first
  // for eviction it leaves the L2 to the split-K partials the merge reads next; with several tiles
  // per head (a prefill chunk) the other tiles read the same pages, so they are kept as usual
  const uint64_t policy =
      p.G * p.q_len <= kTRows ? l2_evict_first_policy() : l2_evict_normal_policy();
  uint32_t k = 0;
  bool to = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const TSeg sg = t_load_seg(p, s);
    const bool lone = (sg.head | 1) >= p.Hkv;  // the last head of an odd count has no partner
    const uint32_t ksb = lone ? 512u : 1024u;
    const int64_t offK = (int64_t)sg.head * 4096;
    const int64_t offKs = (int64_t)p.Hkv * 4096 + (sg.head >> 1) * 1024;
    const int64_t offV = (int64_t)p.Hkv * 4608 + sg.head * 4096;
    const int64_t offVs = (int64_t)p.Hkv * 8704 + sg.head * 512;
    const uint32_t per_page = 4096u + ksb + 4096u + 512u;
    for (int p0 = sg.lo; p0 < sg.hi; p0 += 32) {  // 32 pages: a whole number of blocks
      const int n = min(32, sg.hi - p0);
      const int32_t mine =
          (lane < n) ? p.block_table[(int64_t)sg.seq * p.max_pages + p0 + lane] : -1;
      for (int j = 0; j < n; j += 2, ++k) {
        const int32_t pid0 = __shfl_sync(0xffffffffu, mine, j);
        const int32_t pid1 = __shfl_sync(0xffffffffu, mine, min(j + 1, 31));
        if (lane == 0) {
          const uint32_t st = k % kTStages;
          if (k >= kTStages)
            wait_bar_sleep(tbar(bars, kTbStageEmpty + st), ((k / kTStages) - 1) & 1, to);
          const bool has1 = j + 1 < n;
          const bool v0 = pid0 >= 0 && pid0 < p.num_pages;
          const bool v1 = has1 && pid1 >= 0 && pid1 < p.num_pages;
          if (!v0 || (has1 && !v1)) flag_status(p.status, KV_NVFP4_DEV_BAD_PAGE);  // skipped
          stage_pid[2 * st] = v0 ? pid0 : -1;
          stage_pid[2 * st + 1] = v1 ? pid1 : -1;
          const uint32_t full = tbar(bars, kTbStageFull + st);
          const uint32_t bytes = (v0 ? per_page : 0u) + (v1 ? per_page : 0u);
          if (bytes > 0u) {
            mbar_arrive_expect_tx(full, bytes);
            const uint32_t dst = sbase + kTOffStage + st * kTStageBytes;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              if (!(q == 0 ? v0 : v1)) continue;
              const uint8_t* src = p.pool + (int64_t)(q == 0 ? pid0 : pid1) * blk;
              bulk_g2s_hint(dst + kStK + q * 4096, src + offK, 4096u, full, policy);
              bulk_g2s_hint(dst + kStKs + q * 1024, src + offKs, ksb, full, policy);
              bulk_g2s_hint(dst + kStV + q * 4096, src + offV, 4096u, full, policy);
              bulk_g2s_hint(dst + kStVs + q * 512, src + offVs, 512u, full, policy);
            }
          } else {
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
      wait_bar_sleep(tbar(bars, kTbStageFull + st), (last / kTStages) & 1, to);
    }
    if (to) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
  }
}

// --------------------------------------------------------------------------------------------
// MMA issuers. The Q.K^T warp, per block: gathers the block's K scales (as soon as its stage has
// landed), then, once the P.V of block kb - 2 (which read its P from the S buffer) has completed,
// issues the Q.K^T into that buffer; a segment's first Q.K^T waits for its Q tile. The P.V warp,
// per block: once the block's P and V tile are written, issues its P.V; a segment's first P.V
// overwrites O and waits until the previous segment's epilogue has read O.
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) {
  return d + (uint64_t)(bytes >> 4);  // start-address field: addresses stay below 2^18
}

// The head's K scales of block kb's two pages, gathered by the warp's lanes into the
// scale-factor copy's rows (row r = page 0's keys r and r + 32, then page 1's, per k-half; the
// scale-factor and the key index of the B operand are then 64 page + key), in the ring slot of
// the block's stage. The slot's previous reader, the Q.K^T of block kb - 4, completed before
// this warp issued the Q.K^T of block kb - 2 (it waited for the P.V of block kb - 4).
__device__ __forceinline__ void t_gather_kscales(uint32_t sbase, uint32_t bars, uint32_t kb,
                                                 int head, bool lone, int lane, bool& to) {
  const uint32_t st = kb % kTStages;
  wait_bar_sleep(tbar(bars, kTbStageFull + st), (kb / kTStages) & 1, to);
  const uint32_t stage = sbase + kTOffStage + st * kTStageBytes;
  const uint32_t sfk = sbase + kTOffSfk + st * 1024;
#pragma unroll
  for (int kh = 0; kh < 2; ++kh) {
    uint2 v[2];
#pragma unroll
    for (int q = 0; q < 2; ++q)  // a missing second page leaves stale scales: its keys are masked
      v[q] = lone ? lds64(stage + kStKs + q * 1024 + kh * 256 + lane * 8)
                  : lds64(stage + kStKs + q * 1024 + kh * 512 + lane * 16 + (head & 1) * 8);
    sts128(sfk + kh * 512 + lane * 16, v[0].x, v[0].y, v[1].x, v[1].y);
  }
  fence_async_smem();
  __syncwarp();
}

// Q.K^T of block kb (its K scales gathered, its S buffer free).
__device__ __forceinline__ void t_issue_qk(uint64_t dq, uint64_t dk, uint64_t dsf, uint32_t bars,
                                           uint32_t tbase, uint32_t kb, int lane) {
  const uint32_t st = kb % kTStages, b = kb & 1u;
  if (lane == 0) {
    tc_fence_after();
    tmem_cp_32x128b_x4(tbase + kTColSfb + b * 8, desc_add(dsf, st * 1024));
    tmem_cp_32x128b_x4(tbase + kTColSfb + b * 8 + 4, desc_add(dsf, st * 1024 + 512));
    const uint64_t kd = desc_add(dk, kTOffStage + st * kTStageBytes);
    mma_nvf4_ss(tbase + kTColS + b * 128, dq, kd, kIdescQK, tbase + kTColSfa,
                tbase + kTColSfb + b * 8, 0u);
    mma_nvf4_ss(tbase + kTColS + b * 128, desc_add(dq, 256), desc_add(kd, 256), kIdescQK,
                tbase + kTColSfa + 4, tbase + kTColSfb + b * 8 + 4, 1u);
    mma_commit(tbar(bars, kTbSFull + b));
    mma_commit(tbar(bars, kTbStageEmpty + st));  // K codes and scales consumed
  }
  __syncwarp();
}

__device__ void t_mma_qk(const TileParams& p, uint8_t* smem, uint32_t tbase, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kTOffBars;
  const uint64_t dq = smem_desc(sbase + kTOffQ, 128, 512);
  const uint64_t dk = smem_desc(sbase + kStK, 128, 512);   // + stage offset
  const uint64_t dsf = smem_desc(sbase + kTOffSfk, 16, 128);
  uint32_t kb = 0, sgi = 0;
  bool to = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s, ++sgi) {
    const TSeg sg = t_load_seg(p, s);
    const int n = seg_blocks(sg);
    const bool lone = (sg.head | 1) >= p.Hkv;
    for (int j = 0; j < n; ++j, ++kb) {
      t_gather_kscales(sbase, bars, kb, sg.head, lone, lane, to);
      if (j == 0) wait_bar_sleep(tbar(bars, kTbQReady), sgi & 1, to);  // the segment's Q tile, scales
      // S buffer kb & 1 is free once the P.V of block kb - 2 (which read its P) has completed
      if (kb >= 2) wait_bar_sleep(tbar(bars, kTbPvDone + (kb & 1u)), ((kb - 2) >> 1) & 1, to);
      t_issue_qk(dq, dk, dsf, bars, tbase, kb, lane);
    }
    if (to) break;  // a lost signal: issue nothing more (the drain below still runs)
  }
  if (to) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// P.V of block kb: eight MMAs (16 keys each) into O; A = P in the S buffer (keys 0..63 in
// columns 0..31, keys 64..127 in columns 64..95; in split-page mode keys 32 i .. 32 i + 31 in
// columns 32 i .. 32 i + 15).
__device__ void t_mma_pv(const TileParams& p, uint8_t* smem, uint32_t tbase, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kTOffBars;
  const uint64_t dv = smem_desc(sbase + kTOffVt, kVtGroupBytes, 128);
  const bool dup = p.G * p.q_len <= kTRows / 2;  // split-page mode (see the softmax warps)
  uint32_t kb = 0, sgi = 0;
  bool to = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s, ++sgi) {
    const int n = seg_blocks(t_load_seg(p, s));
    if (sgi > 0) wait_bar_sleep(tbar(bars, kTbOFree), (sgi - 1) & 1, to);
    for (int j = 0; j < n; ++j, ++kb) {
      const uint32_t b = kb & 1u;
      wait_bar_sleep(tbar(bars, kTbPFull + b), (kb >> 1) & 1, to);
      if (lane == 0) {
        tc_fence_after();
        const uint64_t bd = desc_add(dv, b * kVtBytes);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t acol = dup ? 64 * (ks >> 2) + 32 * ((ks >> 1) & 1) + 8 * (ks & 1)
                                    : 64 * (ks >> 2) + 8 * (ks & 3);
          mma_f16_ts(tbase + kTColO, tbase + kTColS + b * 128 + acol,
                     desc_add(bd, ks * 2 * kVtGroupBytes), kIdescPV, (j == 0 && ks == 0) ? 0u : 1u);
        }
        mma_commit(tbar(bars, kTbPvDone + b));
      }
      __syncwarp();
    }
    if (to) break;
  }
  if (to) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// --------------------------------------------------------------------------------------------
// V dequantisation warps: thread t of the four warps converts key t of the block (64 code bytes
// and 8 scales) into 128 f16 values of the MN-major tile (core matrix = 8 keys x 8 dims, dims
// contiguous; per 8-key group 16 chunks of dims, then the chunk holding the column of ones and a
// chunk of zeros, written once at the start); zeros for a key past the sequence end or on a
// skipped page. The 16-byte loads of a row are rotated by key so that the eight keys of a
// quarter-warp read distinct banks.
// --------------------------------------------------------------------------------------------
__device__ void t_dequant(const TileParams& p, uint8_t* smem, int warp, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kTOffBars;
  const volatile int32_t* stage_pid = reinterpret_cast<const volatile int32_t*>(smem + kTOffPid);
  const int key = (warp - kTWarpDeq0) * 32 + lane;  // 0..127 within the block
  const int pg = key >> 6, slot = key & 63;
  const int rot = (key >> 1) & 3;
  // this key's row of the two extra chunks in both tiles: dim 128 = 1, dims 129 .. 143 = 0 (the
  // P.V product then accumulates each row's sum of P in column 128 of O)
#pragma unroll
  for (int v = 0; v < 2; ++v) {
    const uint32_t row = sbase + kTOffVt + v * kVtBytes + (key >> 3) * kVtGroupBytes + (key & 7) * 16;
    sts128(row + 16 * 128, 0x3C00u, 0u, 0u, 0u);  // f16 1.0 in the low half of the first word
    sts128(row + 17 * 128, 0u, 0u, 0u, 0u);
  }
  fence_async_smem();
  uint32_t kb = 0;
  bool to = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const TSeg sg = t_load_seg(p, s);
    const int n = seg_blocks(sg);
    for (int j = 0; j < n; ++j, ++kb) {
      const uint32_t st = kb % kTStages, v = kb & 1u;
      wait_bar_sleep(tbar(bars, kTbStageFull + st), (kb / kTStages) & 1, to);
      // V tile v is free once the P.V of block kb - 2 is complete
      if (kb >= 2) wait_bar_sleep(tbar(bars, kTbPvDone + v), ((kb - 2) >> 1) & 1, to);
      const int page = sg.lo + 2 * j + pg;
      const bool ok = page < sg.hi && stage_pid[2 * st + pg] >= 0 && page * kPage + slot < sg.len;
      const uint32_t stage = sbase + kTOffStage + st * kTStageBytes;
      uint4 cw[4];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
        cw[qq] = lds128(stage + kStV + pg * 4096 + slot * 64 + 16 * ((qq + rot) & 3));
      const uint2 sc8 = lds64(stage + kStVs + pg * 512 + slot * 8);
      const uint32_t dst =
          sbase + kTOffVt + v * kVtBytes + (key >> 3) * kVtGroupBytes + (key & 7) * 16;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const int q4 = (qq + rot) & 3;  // 16 code bytes = dims 32 q4 .. 32 q4 + 31
        // scales of blocks 2 q4 (dims 32 q4 ..) and 2 q4 + 1 (dims 32 q4 + 16 ..); 0 for a key
        // with no data (its stale code bytes turn into zeros)
        const uint32_t two_sc = ok ? ((q4 < 2 ? sc8.x : sc8.y) >> (16 * (q4 & 1))) & 0xFFFFu : 0u;
        const uint32_t sh = cvt_e4m3x2_f16(two_sc);
        const uint32_t s0 = dup_lo(sh), s1 = dup_hi(sh);
        const uint32_t words[4] = {cw[qq].x, cw[qq].y, cw[qq].z, cw[qq].w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {  // word w: dims 32 q4 + 8 w .. + 7 (byte = dims 2i, 2i + 1)
          uint32_t r0, r1, r2, r3;
          cvt_e2m1x8_f16(words[w], r0, r1, r2, r3);
          const uint32_t sc = w < 2 ? s0 : s1;
          sts128(dst + (4 * q4 + w) * 128, hmul2(r0, sc), hmul2(r1, sc), hmul2(r2, sc),
                 hmul2(r3, sc));
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(tbar(bars, kTbPFull + v));
        mbar_arrive(tbar(bars, kTbStageEmpty + st));
      }
    }
  }
  if (to && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// --------------------------------------------------------------------------------------------
// Softmax warps. A tile of more than 64 query rows: thread (quadrant q, lane) owns tile row
// r = 32 q + lane (tensor-memory lane r of S and O); warp half h takes page h of each block (keys
// 64 h .. 64 h + 63) and dims 64 h .. 64 h + 63 of O. A tile of at most 64 rows (split-page mode,
// kDup): tile rows 64..127 repeat rows 0..63, so that every lane quadrant holds scores and the
// exponentials of a block are spread over the four SM sub-partitions (warp w runs on
// sub-partition w mod 4, and only it reads lane quadrant w mod 4). Quadrants 0, 1 take page 0 of
// each block and quadrants 2, 3 page 1, warp half h keys 32 h .. 32 h + 31 of the page; lane r of
// P holds the row's P over its page and zeros over the other, so the P.V accumulates the row's
// sums over page 0 in lanes 0..63 of O and over page 1 in lanes 64..127, which the epilogue adds.
// --------------------------------------------------------------------------------------------
// The segment's Q tile (loaded by the four warps of half 0): codes into the A operand tile (tile
// order), scales into tensor memory in the replicated scale-factor layout (lane i, column w of a
// k-half: scales of rows 32 w + i).
template <bool kDup>
__device__ __forceinline__ void t_load_q(const TileParams& p, const TSeg& sg, uint8_t* smem,
                                         uint32_t sbase, uint32_t tbase, uint32_t lane_base, int r,
                                         int lane) {
  const int gr = sg.rg * kTRows + (kDup ? (r & 63) : r);
  uint4 c[4];
  uint2 sc = make_uint2(0u, 0u);
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) c[ch] = make_uint4(0u, 0u, 0u, 0u);
  if (gr < p.G * p.q_len) {
    const int64_t qrow = ((int64_t)sg.seq * p.q_len + gr / p.G) * p.Hq + sg.head * p.G + gr % p.G;
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
  named_barrier_sync(kNbQ, 128);
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
  named_barrier_sync(kNbQ, 128);  // the staging rows are read before the next tile rewrites them
}

// 32 consecutive tensor-memory columns of this warp's lanes.
__device__ __forceinline__ void ld32_at(uint32_t taddr, uint32_t* dst) {
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(dst));
}

// max(a, b, c)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Multiplies 32 columns of O (this thread's row) by alpha in tensor memory.
__device__ __forceinline__ void t_scale_o32(uint32_t taddr, float alpha) {
  uint32_t o[32];
  tmem_ld32(taddr, o);
  tmem_wait_ld_regs32(o);
#pragma unroll
  for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
  tmem_st32(taddr, o);
}

template <bool kDup>
__device__ void t_softmax(const TileParams& p, uint8_t* smem, uint32_t tbase, int warp,
                          int lane) {
  constexpr int kNc = kDup ? 32 : 64;  // keys of each block that one warp takes
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kTOffBars;
  float* red = reinterpret_cast<float*>(smem + kTOffRed);
  const int q = warp & 3;
  const int h = (warp - kTWarpSoft0) >> 2;
  const int r = 32 * q + lane;              // tensor-memory lane
  const int rr = kDup ? (r & 63) : r;       // tile row
  const int pg = kDup ? (q >> 1) : h;       // page of each block that this warp takes
  const int kofs = kDup ? 32 * h : 0;       // its first key within the page
  // the warps that share this thread's row: the quadrant's pair, or (kDup) the two pairs
  const uint32_t nb_row = kDup ? kNbPair + (q & 1) : kNbPair + q;
  constexpr uint32_t kRowThreads = kDup ? 128 : 64;
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const uint32_t ocol = tbase + lane_base + kTColO;
  const float c2 = p.c2;
  const int rows_total = p.G * p.q_len;
  uint32_t kb = 0, sgi = 0;
  bool to = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  if (h == 0 && s_begin < s_end) {
    t_load_q<kDup>(p, t_load_seg(p, s_begin), smem, sbase, tbase, lane_base, r, lane);
    if (lane == 0) mbar_arrive(tbar(bars, kTbQReady));
  }
  for (int s = s_begin; s < s_end; ++s, ++sgi) {
    const TSeg sg = t_load_seg(p, s);
    const int n = seg_blocks(sg);
    const int gr = sg.rg * kTRows + rr;
    const bool row_ok = gr < rows_total;
    // a quadrant whose 32 rows are all padding computes nothing (its two warps still take part
    // in every mbarrier); its rows of P and O are never read into a result
    const bool warp_live = sg.rg * kTRows + (rr & ~31) < rows_total;
    // largest visible key position of this row (-1: no key)
    const int limit = row_ok ? (p.causal ? sg.len - p.q_len + gr / p.G : sg.len - 1) : -1;
    float m = -INFINITY;
    // this warp's page of each block is skipped (its keys masked) when its id lies outside the
    // pool, as the producer skips it; the id is read from the block table one block ahead, so that
    // the block loop touches no shared-memory barrier but the S-full and P-full ones
    const int32_t* bt = p.block_table + (int64_t)sg.seq * p.max_pages;
    int32_t pid_next = (sg.lo + pg < sg.hi) ? __ldg(bt + sg.lo + pg) : -1;
    for (int j = 0; j < n; ++j, ++kb) {
      const uint32_t b = kb & 1u;
      const int page = sg.lo + 2 * j + pg;
      const int32_t pid = pid_next;
      const bool valid = page < sg.hi && pid >= 0 && pid < p.num_pages;
      if (page + 2 < sg.hi) pid_next = __ldg(bt + page + 2);
      wait_bar_sleep(tbar(bars, kTbSFull + b), (kb >> 1) & 1, to);
      tc_fence_after();
      __syncwarp();
      if (warp_live) {
        const uint32_t sbuf = tbase + lane_base + kTColS + b * 128;
        const uint32_t scol = sbuf + 64 * pg + kofs;
        // keys c < nv of this warp's share of its page are visible to this row; a padding row (no
        // query) is left unmasked: its P and O are never read, and its scores are finite or its own
        const int nv =
            !row_ok ? kNc : valid ? max(0, min(kNc, limit - page * kPage - kofs + 1)) : 0;
        uint32_t sv[kNc];
#pragma unroll
        for (int c = 0; c < kNc; c += 32) ld32_at(scol + c, &sv[c]);
#pragma unroll
        for (int c = 0; c < kNc; c += 32)
          tmem_wait_ld_regs32(*reinterpret_cast<uint32_t(*)[32]>(&sv[c]));
        if (__any_sync(0xffffffffu, nv != kNc)) {
#pragma unroll
          for (int c = 0; c < kNc; ++c) sv[c] = c < nv ? sv[c] : __float_as_uint(-INFINITY);
        }
        // this warp's max of the row: eight chains of three-input maxima, then a tree
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = __uint_as_float(sv[e]);
#pragma unroll
        for (int c = 8; c < kNc - 8; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            mx[e] = fmax3(mx[e], __uint_as_float(sv[c + e]), __uint_as_float(sv[c + 8 + e]));
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], __uint_as_float(sv[kNc - 8 + e]));
        float pmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                           fmaxf(mx[6], mx[7]));
        // the other warps' maxima of the row (buffers alternate by block, so a slow partner still
        // reads this block's values after this warp has moved on)
        if (kDup) {
          red[(b * 4 + 2 * pg + h) * 64 + rr] = pmax;
          named_barrier_sync(nb_row, kRowThreads);
          const float* rb = red + b * 256 + rr;
          pmax = fmaxf(fmax3(rb[0], rb[64], rb[128]), rb[192]);
        } else {
          red[(b * 2 + h) * 128 + r] = pmax;
          named_barrier_sync(nb_row, kRowThreads);
          pmax = fmaxf(pmax, red[(b * 2 + (h ^ 1)) * 128 + r]);
        }
        // every warp of the row holds the same row maxima, so they take the same decisions
        const float mc = fmaxf(m, pmax);
        float alpha = 1.f;
        bool need = false;
        if (j == 0) {
          m = mc;  // nothing accumulated yet in this segment
        } else if (mc > m && (m == -INFINITY || (mc - m) * c2 > kLazyMax)) {
          need = true;
          alpha = m == -INFINITY ? 0.f : fast_exp2((m - mc) * c2);
          m = mc;
        }
        // P = exp2(s c2 - m c2) <= 2^15 in f16 pairs over the first kNc / 2 of this warp's
        // columns; a masked key (-inf) gives 0, also while m is still -inf (then the offset is
        // taken as 0)
        const float mc2 = m == -INFINITY ? 0.f : m * c2;
        uint32_t pk[kNc / 2];
#pragma unroll
        for (int c = 0; c < kNc; c += 2) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(sv[c]), c2, -mc2));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sv[c + 1]), c2, -mc2));
          pk[c >> 1] = pack_f16x2(p0, p1);
        }
        if constexpr (kDup) {
          tmem_st16(scol, pk);
          // zeros over the same keys of the other page (columns no warp of this quadrant reads)
          tmem_st16_zero(sbuf + 64 * (pg ^ 1) + kofs);
        } else {
          tmem_st32(scol, pk);
        }
        // rows whose max was raised: this warp's half of their row of O (half 0 also l) is
        // rescaled once the previous block's P.V has completed (after the P stores, so that the
        // scores are no longer held); the loads and stores are warp-wide
        if (__any_sync(0xffffffffu, need)) {
          wait_bar_sleep(tbar(bars, kTbPvDone + ((kb - 1) & 1u)), ((kb - 1) >> 1) & 1, to);
          tc_fence_after();
          t_scale_o32(ocol + 64 * h, alpha);
          t_scale_o32(ocol + 64 * h + 32, alpha);
          if (h == 0) {
            uint32_t o8[8];
            tmem_ld8(ocol + 128, o8);
            tmem_wait_ld_regs(o8);
            o8[0] = __float_as_uint(__uint_as_float(o8[0]) * alpha);  // l
            tmem_st8(ocol + 128, o8);
          }
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tbar(bars, kTbPFull + b));
    }

    // ---- segment end: the next segment's Q tile (every Q.K^T of this one is complete), then
    // the epilogue of this one ----
    if (h == 0 && s + 1 < s_end) {
      t_load_q<kDup>(p, t_load_seg(p, s + 1), smem, sbase, tbase, lane_base, r, lane);
      if (lane == 0) mbar_arrive(tbar(bars, kTbQReady));
    }
    const uint32_t kl = kb - 1;
    wait_bar_sleep(tbar(bars, kTbPvDone + (kl & 1u)), (kl >> 1) & 1, to);
    tc_fence_after();
    const bool split = sg.n_seg > 1;
    float4* xo = reinterpret_cast<float4*>(smem + kTOffXch);  // [32 dim quads][64 rows]
    float* xl = reinterpret_cast<float*>(smem + kTOffXch + kTXchOBytes);
    if (warp_live) {
      if (kDup) {
        // quadrants 2, 3 hand their rows' sums over page 1 (O and l) to quadrants 0, 1
        if (q >= 2) {
#pragma unroll 1
          for (int cc = 2 * h; cc < 2 * h + 2; ++cc) {
            uint32_t o[32];
            tmem_ld32(ocol + 32 * cc, o);
            tmem_wait_ld_regs32(o);
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              xo[(cc * 8 + (e >> 2)) * 64 + rr] =
                  make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                              __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
          }
          if (h == 0) {
            uint32_t o8[8];
            tmem_ld8(ocol + 128, o8);
            tmem_wait_ld_regs(o8);
            xl[rr] = __uint_as_float(o8[0]);
          }
        }
        named_barrier_sync(nb_row, kRowThreads);
      }
      if (!kDup || q < 2) {
        uint32_t o8[8];
        tmem_ld8(ocol + 128, o8);
        tmem_wait_ld_regs(o8);
        // the row's sum of P, accumulated by the P.V MMAs
        const float l = __uint_as_float(o8[0]) + (kDup ? xl[rr] : 0.f);
        float* part = split ? p.partials + (int64_t)sg.part * kTPartFloats : nullptr;
        const int tok = gr / p.G, qh = sg.head * p.G + gr % p.G;
        float* orow = p.out + (((int64_t)sg.seq * p.q_len + tok) * p.Hq + qh) * 128;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int cc = 2 * h; cc < 2 * h + 2; ++cc) {
          uint32_t o[32];
          tmem_ld32(ocol + 32 * cc, o);
          tmem_wait_ld_regs32(o);
          float ov[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __uint_as_float(o[e]);
          if (kDup) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 x = xo[(cc * 8 + (e >> 2)) * 64 + rr];
              ov[e] += x.x; ov[e + 1] += x.y; ov[e + 2] += x.z; ov[e + 3] += x.w;
            }
          }
          if (row_ok) {
            if (split) {
              float4* dst = reinterpret_cast<float4*>(part + rr * 128 + 32 * cc);
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                dst[e >> 2] = make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
            } else if (l > 0.f) {
              float4* dst = reinterpret_cast<float4*>(orow + 32 * cc);
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                dst[e >> 2] = make_float4(ov[e] * inv, ov[e + 1] * inv, ov[e + 2] * inv,
                                          ov[e + 3] * inv);
            }
          }
        }
        if (row_ok && split && h == 0) {
          part[kTRows * 128 + rr] = m;
          part[kTRows * 128 + kTRows + rr] = l;
        }
      }
      // the exchange area is read before the next segment's epilogue rewrites it
      if (kDup) named_barrier_sync(nb_row, kRowThreads);
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
      // the Q.K^T (K codes and scales read, by its commit) and the V warps
      mbar_init(tbar(bars, kTbStageEmpty + s), 1 + kTDeqWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tbar(bars, kTbSFull + b), 1);
      mbar_init(tbar(bars, kTbPFull + b), kTSoftWarps + kTDeqWarps);
      mbar_init(tbar(bars, kTbPvDone + b), 1);
    }
    mbar_init(tbar(bars, kTbQReady), 4);
    mbar_init(tbar(bars, kTbOFree), kTSoftWarps);
    mbar_init(tbar(bars, kTbDrain), 2);  // one commit per issuer
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
    t_mma_qk(p, smem, tbase, lane);
  } else if (warp >= kTWarpSoft0 && warp < kTWarpDeq0) {
    if (p.G * p.q_len <= kTRows / 2) t_softmax<true>(p, smem, tbase, warp, lane);
    else t_softmax<false>(p, smem, tbase, warp, lane);
  } else if (warp < kTWarpPv) {
    t_dequant(p, smem, warp, lane);
  } else {
    t_mma_pv(p, smem, tbase, lane);
  }

  if (warp == kTWarpMma || warp == kTWarpPv) {
    // tensor memory is freed only once no tcgen05 op of this CTA is in flight (after a timeout
    // some may still be; the wait is bounded like every other)
    if (lane == 0) mma_commit(tbar(bars, kTbDrain));
    __syncwarp();
    bool to = false;
    wait_bar_sleep(tbar(bars, kTbDrain), 0, to);
    if (to && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTWarpMma) tmem_dealloc(tbase, kTTmemCols);
}


// --------------------------------------------------------------------------------------------
// Split-K merge of the tile kernel's partials (second launch): one CTA per (split group, row of
// the tile); its 256 threads are 8 slices of the group's partials x 32 four-dim columns:
//   M = max_q m_q,  L = sum_q 2^((m_q - M) c2) l_q,  o = sum_q 2^((m_q - M) c2) O_q / L.
// --------------------------------------------------------------------------------------------
struct TMergeParams {
  const int4* groups;
  const int32_t* split;    // [num_split] group indices
  const float* partials;   // [num_partials][kTPartFloats]
  float* out;
  int32_t Hq, G, q_len;
  float c2;
};

constexpr int kTMergeSlices = 8;
constexpr int kTMergePerRound = 8;  // partials a slice requests at once (64 per CTA and round)

__global__ void __launch_bounds__(32 * kTMergeSlices, 2) tile_merge_kernel(const TMergeParams p) {
  __shared__ float s_m[kTMergeSlices], s_l[kTMergeSlices];
  __shared__ float4 s_o[kTMergeSlices][32];
  asm volatile("griddepcontrol.launch_dependents;");
  const int gi = p.split[blockIdx.x];  // plan tables: written before the attention launch
  const int i = blockIdx.y;
  const int4 g0 = p.groups[2 * gi], g1 = p.groups[2 * gi + 1];
  const int r = g0.z * kTRows + i, head = g0.y;
  // the partials are visible only after the attention grid has completed and flushed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (r >= p.G * p.q_len) return;  // uniform over the CTA
  const int n_seg = g1.x;
  const int slice = threadIdx.x >> 5, d4 = threadIdx.x & 31;
  const float* base = p.partials + (int64_t)g1.y * kTPartFloats;
  // per round a slice requests its partials q = q0 + 8 u (u < 8) at once (one L2 round trip for a
  // group of up to 64 segments) and combines them with independent weights
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = slice; q0 < n_seg; q0 += kTMergeSlices * kTMergePerRound) {
    float mq[kTMergePerRound], lq[kTMergePerRound];
    float4 ov[kTMergePerRound];
#pragma unroll
    for (int u = 0; u < kTMergePerRound; ++u) {
      const int q = q0 + kTMergeSlices * u;
      mq[u] = -INFINITY;
      lq[u] = 0.f;
      ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (q < n_seg) {
        const float* pq = base + (int64_t)q * kTPartFloats;
        mq[u] = __ldcg(pq + kTRows * 128 + i);
        lq[u] = __ldcg(pq + kTRows * 128 + kTRows + i);
        ov[u] = __ldcg(reinterpret_cast<const float4*>(pq + i * 128) + d4);
      }
    }
    float mn = M;
#pragma unroll
    for (int u = 0; u < kTMergePerRound; ++u) mn = fmaxf(mn, mq[u]);
    if (mn == -INFINITY) continue;  // no visible key for this row in any partial so far
    const float a = fast_exp2((M - mn) * p.c2);  // 0 while M is -inf
    L *= a;
    O.x *= a; O.y *= a; O.z *= a; O.w *= a;
#pragma unroll
    for (int u = 0; u < kTMergePerRound; ++u) {
      if (mq[u] == -INFINITY) continue;  // a segment with no visible key for this row
      const float f = fast_exp2((mq[u] - mn) * p.c2);
      L += f * lq[u];
      O.x += f * ov[u].x; O.y += f * ov[u].y; O.z += f * ov[u].z; O.w += f * ov[u].w;
    }
    M = mn;
  }
  s_o[slice][d4] = O;
  if (d4 == 0) { s_m[slice] = M; s_l[slice] = L; }
  __syncthreads();
  if (slice == 0) {
    float Mt = s_m[0];
#pragma unroll
    for (int j = 1; j < kTMergeSlices; ++j) Mt = fmaxf(Mt, s_m[j]);
    float Lt = 0.f;
    float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kTMergeSlices; ++j) {
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
      const float inv = 1.f / Lt;
      *dst = make_float4(Ot.x * inv, Ot.y * inv, Ot.z * inv, Ot.w * inv);
    }
  }
}

}  // namespace

int tile_smem_bytes() { return kTSmemBytes; }

// Attention for tiles of 128 rows of one KV head (see the top of this file), then the merge of the
// split groups' partials; both launched as programmatic dependents on the stream.
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
  mp.Hq = Hq; mp.G = p.G; mp.q_len = q_len; mp.c2 = p.c2;
  const int rows_total = p.G * q_len;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_split, (unsigned)(rows_total < kTRows ? rows_total : kTRows));
  cfg.blockDim = dim3(32 * kTMergeSlices);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tile_merge_kernel, mp);
}

}  // namespace kvnvfp4
