// Paged GQA decode / speculative-verify attention over the NVFP4 cache, on the tcgen05 tensor
// cores, with split-K.
//
// Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)": the Q.K^T
// product in NVFP4 with E4M3 block scales (both Q and K quantised), V dequantised for the P.V
// product, row-major KV scales. The split-K decomposition and the fp32 log-sum-exp merge are this
// library's design; the pages say nothing about the kernel's decomposition.
//
// Work decomposition. A group is (sequence, tile of 8 query rows) over every KV head; a row is
// (query token, head in the GQA group). The plan lays the groups' pages end to end and gives each
// persistent CTA (one per SM) a contiguous, page-balanced share: one or more segments, each a page
// range of one group. A CTA's softmax state carries across the pages of a segment; a group that
// spans CTAs leaves one (m, l, O) partial per segment and the CTA taking its last ticket merges.
//
// One page = 64 keys of every KV head, a 9216 x H byte block moved by ONE bulk async copy.
//
// Per page, with KV heads taken in pairs (2p, 2p+1):
//   Q.K^T: tcgen05.mma kind::mxf4nvf4, block_scale.scale_vec::4X (E2M1 x E2M1, UE4M3 scale per
//     16 elements), M = 128 = 64 keys of head 2p over 64 keys of head 2p+1, N = 16 = 8 query rows
//     of head 2p then 8 of head 2p+1, K = 64 per instruction (two per 128-dim row). The K codes
//     are stored in the pool in the tensor core's 8-row x 16-byte tile order, so the page lands in
//     shared memory ready for the MMA; scales go to TMEM in the replicated 32-lane x 4-column
//     layout. Cross terms (head 2p keys x head 2p+1 rows) are computed and ignored.
//   softmax: 8 warps read S from TMEM (one key per lane), take the exact page max per (head, row)
//     (warp max reduction + one exchange between the two warps holding a head), keep an fp32
//     running max and row sums, and write P = exp2((s - max) log2e scale) <= 1 to shared memory as
//     f16 hi + lo.
//   P.V: 4 warps dequantise V (E2M1 x E4M3 is exact in f16) into an MN-major shared tile; one
//     thread issues tcgen05.mma kind::f16 with M = 128 dims, N = 16 (P hi in columns 0..7, P lo in
//     8..15), K = 16 keys per instruction, into a per-page TMEM accumulator (4 slots). Two pages
//     later the softmax warps fold that page into the running O^T (O = O * alpha + O_page), so a
//     rising max never stalls the tensor-core pipeline on a rescale.
//
// Warp roles (480 threads): warp 0 TMA producer, warp 1 Q.K^T issuer and TMEM owner, warp 2 P.V
// issuer, warps 3..10 softmax / scale factors / epilogue (two groups of four, one per KV-head pair,
// covering the four TMEM lane quadrants), warps 11..14 V dequant.
// Every wait is an mbarrier wait bounded in time; on a timeout the kernel records
// KV_NVFP4_DEV_TIMEOUT and carries on, so it cannot hang.

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

namespace {

constexpr int kMaxHkv = 4;
constexpr int kStages = 3;
constexpr int kStageBytes = kMaxHkv * 9216;        // one page block of up to 4 heads
constexpr int kVhSlots = 5;                        // dequantised V tiles (one head-page each)
constexpr int kVhBytes = 64 * 128 * 2;             // 64 keys x 128 dims x f16
constexpr int kPBytes = kMaxHkv * 2048;            // per page: per head P hi (1 KB) + lo (1 KB)
constexpr int kQBytes = 2 * 1024;                  // two head pairs x 16 rows x 64 B
constexpr int kRows = 8;                           // query rows per head per group
constexpr int kPartHeadFloats = kRows * 128 + 2 * kRows;  // O[8][128], m[8], l[8]

constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpPv = 2, kWarpSoftmax0 = 3, kWarpDequant0 = 11;
constexpr int kDequantWarps = 4;
constexpr int kThreads = (kWarpDequant0 + kDequantWarps) * 32;

// shared memory map
constexpr int kOffStage = 0;
constexpr int kOffVh = kOffStage + kStages * kStageBytes;
constexpr int kOffP = kOffVh + kVhSlots * kVhBytes;
constexpr int kOffQ = kOffP + 2 * kPBytes;
constexpr int kOffBars = kOffQ + kQBytes;
// barrier indices
constexpr int kBarStageFull = 0;                    // [kStages]
constexpr int kBarStageEmpty = kBarStageFull + kStages;
constexpr int kBarSfaFull = kBarStageEmpty + kStages;  // [2]
constexpr int kBarQkDone = kBarSfaFull + 2;         // [2]
constexpr int kBarSFree = kBarQkDone + 2;           // [2]
constexpr int kBarPFull = kBarSFree + 2;            // [2]
constexpr int kBarPvDone = kBarPFull + 2;           // [2]
constexpr int kBarVhFull = kBarPvDone + 2;          // [kVhSlots]
constexpr int kBarVhFree = kBarVhFull + kVhSlots;   // [kVhSlots]
constexpr int kOSlots = 4;                          // per-page P.V accumulators in TMEM
constexpr int kBarQReady = kBarVhFree + kVhSlots;
constexpr int kBarOFree = kBarQReady + 1;            // [kOSlots]: page accumulator folded
constexpr int kNumBars = kBarOFree + kOSlots;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
// misc: stage page ids, tmem base, flags (need-max per page parity x warp, rescale per
// half, ticket), reduction scratch, per-head alpha / mu / L
constexpr int kOffStagePid = kOffMisc;
constexpr int kOffTmemSlot = kOffStagePid + 4 * kStages;
constexpr int kOffFlags = kOffTmemSlot + 16;
constexpr int kOffRed = kOffFlags + 128;  // float [3][4 quadrants][2 pairs][8 rows]: page max x2, sums
constexpr int kOffAlpha = kOffRed + 3 * 4 * 2 * kRows * 4;  // float [kOSlots][kMaxHkv][8]
constexpr int kOffMu = kOffAlpha + kOSlots * kMaxHkv * kRows * 4;
constexpr int kOffL = kOffMu + kMaxHkv * kRows * 4;
constexpr int kSmemBytes = kOffL + kMaxHkv * kRows * 4 + 64;

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;        // [2 buffers][2 pairs][16]
constexpr uint32_t kColSfa = 64;     // [2 buffers][2 pairs][2 k-halves][4]
constexpr uint32_t kColSfb = 96;     // [2 pairs][2 k-halves][4]
constexpr uint32_t kColOMain = 128;  // running O^T: [4 heads][16] (hi + lo halves)
constexpr uint32_t kColOPage = 192;  // per-page O^T: [kOSlots][4 heads][16]

// instruction descriptors (dense, no negation):
//   QK: A, B = E2M1 (format 1) K-major, scale type UE4M3, N = 16, M = 128
//   PV: D = f32, A, B = f16, both MN-major, N = 16, M = 128
constexpr uint32_t kIdescQK = (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = (1u << 4) | (1u << 15) | (1u << 16) | ((16u >> 3) << 17) |
                              ((128u >> 4) << 24);

struct DecodeParams {
  const uint8_t* q_codes;
  const uint8_t* q_scales;
  const uint8_t* pool;
  const int32_t* block_table;
  int32_t max_pages;
  int32_t num_pages;
  const int4* groups;      // 2 x int4 per group: {seq, 0, rg, len}, {n_seg, first_part, pages, 0}
  const int4* segments;    // {group, page_lo, page_hi, part_slot or -1}
  const int32_t* cta_seg;  // [grid + 1]
  int32_t* counters;       // [num_groups] merge tickets
  float* partials;         // [num_partials][Hkv][kPartHeadFloats]
  float* out;
  int32_t* status;
  int32_t Hq, Hkv, G, q_len, causal;
  float c2;                // sm_scale * log2(e)
};

struct SegInfo {
  int seq, rg, len, n_seg, first_part, lo, hi, part, group;
};

__device__ __forceinline__ SegInfo load_seg(const DecodeParams& p, int s) {
  const int4 seg = p.segments[s];
  const int4 g0 = p.groups[2 * seg.x];
  const int4 g1 = p.groups[2 * seg.x + 1];
  SegInfo r;
  r.group = seg.x; r.lo = seg.y; r.hi = seg.z; r.part = seg.w;
  r.seq = g0.x; r.rg = g0.z; r.len = g0.w;
  r.n_seg = g1.x; r.first_part = g1.y;
  return r;
}

// Bounded wait: after a thread has once hit the time limit its later waits do not block, so a
// kernel whose pipeline lost a signal still ends promptly (with KV_NVFP4_DEV_TIMEOUT set).
__device__ __forceinline__ void wait_bar(uint32_t bar, uint32_t parity, bool& timed_out) {
  if (timed_out) {
    (void)mbar_try_wait(bar, parity);
    return;
  }
  if (!mbar_wait_bounded(bar, parity)) timed_out = true;
}

// --------------------------------------------------------------------------------------------
// Producer warp: lane 0 streams the CTA's pages (all KV heads of a page in one bulk copy) into a
// kStages ring; the other lanes load page ids 32 at a time. The page id (or -1 when it lies
// outside the pool) is published in shared memory before the stage's full barrier is armed.
// --------------------------------------------------------------------------------------------
__device__ void producer(const DecodeParams& p, uint8_t* smem, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBars;
  volatile int32_t* stage_pid = reinterpret_cast<volatile int32_t*>(smem + kOffStagePid);
  const uint32_t blk_bytes = (uint32_t)p.Hkv * 9216u;
  uint32_t k = 0;
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const SegInfo sg = load_seg(p, s);
    for (int p0 = sg.lo; p0 < sg.hi; p0 += 32) {
      const int n = min(32, sg.hi - p0);
      const int32_t mine =
          (lane < n) ? p.block_table[(int64_t)sg.seq * p.max_pages + p0 + lane] : -1;
      for (int j = 0; j < n; ++j, ++k) {
        const int32_t pid = __shfl_sync(0xffffffffu, mine, j);
        if (lane == 0) {
          const uint32_t st = k % kStages;
          if (k >= kStages)
            wait_bar(bars + 8 * (kBarStageEmpty + st), ((k / kStages) - 1) & 1, timed_out);
          const bool valid = pid >= 0 && pid < p.num_pages;
          stage_pid[st] = valid ? pid : -1;
          const uint32_t full = bars + 8 * (kBarStageFull + st);
          if (valid) {
            mbar_arrive_expect_tx(full, blk_bytes);
            bulk_g2s(sbase + kOffStage + st * kStageBytes, p.pool + (int64_t)pid * blk_bytes,
                     blk_bytes, full);
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
    for (uint32_t st = 0; st < kStages && st < k; ++st) {
      const uint32_t last = k - 1 - ((k - 1 - st) % kStages);
      wait_bar(bars + 8 * (kBarStageFull + st), (last / kStages) & 1, timed_out);
    }
    if (timed_out) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
  }
}

// --------------------------------------------------------------------------------------------
// MMA issue (one thread each for Q.K^T and for P.V).
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ void issue_qk(const DecodeParams& p, uint32_t sbase, uint32_t tbase,
                                         uint32_t k, int npairs, bool& timed_out) {
  const uint32_t bars = sbase + kOffBars;
  const uint32_t st = k % kStages, b = k & 1;
  wait_bar(bars + 8 * (kBarStageFull + st), (k / kStages) & 1, timed_out);
  wait_bar(bars + 8 * (kBarSfaFull + b), (k >> 1) & 1, timed_out);
  if (k >= 2) wait_bar(bars + 8 * (kBarSFree + b), ((k >> 1) - 1) & 1, timed_out);
  tc_fence_after();
  const uint32_t kc = sbase + kOffStage + st * kStageBytes;
  const uint32_t qb = sbase + kOffQ;
  for (int pr = 0; pr < npairs; ++pr) {
    for (int kh = 0; kh < 2; ++kh) {
      const uint64_t ad = smem_desc(kc + pr * 8192 + kh * 256, 128, 512);
      const uint64_t bd = smem_desc(qb + pr * 1024 + kh * 256, 128, 512);
      mma_nvf4_ss(tbase + kColS + b * 32 + pr * 16, ad, bd, kIdescQK,
                  tbase + kColSfa + b * 16 + pr * 8 + kh * 4, tbase + kColSfb + pr * 8 + kh * 4,
                  (uint32_t)kh);
    }
  }
  mma_commit(bars + 8 * (kBarQkDone + b));
  mma_commit(bars + 8 * (kBarStageEmpty + st));  // K codes consumed once the QK MMAs complete
}

// Q.K^T issuer: runs ahead of the softmax as far as the stage ring, the scale-factor buffers and
// the two S buffers allow.
__device__ void qk_issuer(const DecodeParams& p, uint8_t* smem, uint32_t tbase) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBars;
  const int npairs = (p.Hkv + 1) >> 1;
  uint32_t k = 0, sgi = 0;
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s, ++sgi) {
    const SegInfo sg = load_seg(p, s);
    wait_bar(bars + 8 * kBarQReady, sgi & 1, timed_out);  // Q tile and its scales for this group
    for (int j = 0; j < sg.hi - sg.lo; ++j, ++k) issue_qk(p, sbase, tbase, k, npairs, timed_out);
  }
  if (timed_out) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// P.V issuer: per page and head, four MMAs (16 keys each) into the page's TMEM accumulator.
__device__ void pv_issuer(const DecodeParams& p, uint8_t* smem, uint32_t tbase) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBars;
  uint32_t k = 0, hp = 0;
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const SegInfo sg = load_seg(p, s);
    for (int j = 0; j < sg.hi - sg.lo; ++j, ++k) {
      const uint32_t b = k & 1, os = k % kOSlots;
      wait_bar(bars + 8 * (kBarPFull + b), (k >> 1) & 1, timed_out);
      if (k >= kOSlots) wait_bar(bars + 8 * (kBarOFree + os), ((k / kOSlots) - 1) & 1, timed_out);
      tc_fence_after();
      for (int h = 0; h < p.Hkv; ++h, ++hp) {
        const uint32_t slot = hp % kVhSlots;
        wait_bar(bars + 8 * (kBarVhFull + slot), (hp / kVhSlots) & 1, timed_out);
        tc_fence_after();
        const uint32_t vh = sbase + kOffVh + slot * kVhBytes;
        const uint32_t pb = sbase + kOffP + b * kPBytes + h * 2048;
        for (int i = 0; i < 4; ++i) {  // 16 keys per instruction
          const uint64_t ad = smem_desc(vh + i * 4096, 2048, 128);
          const uint64_t bd = smem_desc(pb + i * 256, 128, 1024);
          mma_f16_ss(tbase + kColOPage + os * 64 + h * 16, ad, bd, kIdescPV, i > 0 ? 1u : 0u);
        }
        mma_commit(bars + 8 * (kBarVhFree + slot));
      }
      mma_commit(bars + 8 * (kBarPvDone + b));
    }
  }
  if (timed_out) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// --------------------------------------------------------------------------------------------
// Softmax warps: 8 warps, two groups of four. Group pr works on KV-head pair pr; within a group
// the four warps cover the four TMEM lane quadrants (qd = warp % 4). For S a lane holds one key:
// TMEM lane L = 32 qd + lane is key L % 64 of head 2 pr + L / 64. For O a lane holds one head dim.
// --------------------------------------------------------------------------------------------
constexpr int kSoftmaxWarps = 8;

struct SoftmaxCtx {
  const DecodeParams* p;
  uint8_t* smem;
  uint32_t sbase, bars, tbase, lane_base;
  int lane, qd, pr, half, key, head, gt;  // gt: thread index within the pair group (0..127)
  bool active;                            // the pair has a real head for this thread's half
  bool timed_out;
};

// Scale factors of page k's K rows of this warp's pair into TMEM (replicated 32-lane x 4-column
// layout: lane i, column j holds the 4 scales of MMA row 32 j + i); releases the stage's K scales.
__device__ __forceinline__ void write_sfa(SoftmaxCtx& c, uint32_t k, int page, int len) {
  const DecodeParams& p = *c.p;
  const uint32_t st = k % kStages, b = k & 1;
  wait_bar(c.bars + 8 * (kBarStageFull + st), (k / kStages) & 1, c.timed_out);
  if (k >= 2) wait_bar(c.bars + 8 * (kBarQkDone + b), ((k >> 1) - 1) & 1, c.timed_out);
  const bool pvalid = reinterpret_cast<volatile int32_t*>(c.smem + kOffStagePid)[st] >= 0;
  const uint32_t ks = c.sbase + kOffStage + st * kStageBytes + p.Hkv * 4096;
  const int kp0 = page * 64;
  uint32_t sf[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int hh = 2 * c.pr + (j >> 1), kk = 32 * (j & 1) + c.lane;
    uint2 v = make_uint2(0u, 0u);
    if (hh < p.Hkv && pvalid && kp0 + kk < len) v = lds64(ks + hh * 512 + kk * 8);
    sf[j] = v.x;      // k-half 0: scales of dims 0..63
    sf[4 + j] = v.y;  // k-half 1: dims 64..127
  }
  tmem_st8(c.tbase + c.lane_base + kColSfa + b * 16 + c.pr * 8, sf);
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (c.lane == 0) {
    mbar_arrive(c.bars + 8 * (kBarSfaFull + b));
    mbar_arrive(c.bars + 8 * (kBarStageEmpty + st));
  }
}

// Fold page j's P.V accumulator into the running O^T of this warp's pair (one dim per lane):
// O = O * alpha_j + O_page(j), alpha_j = 2^((mu_{j-1} - mu_j) c2) per (head, row). P hi and P lo
// were accumulated in columns 0..7 and 8..15 and are summed here.
__device__ __forceinline__ void fold_page(SoftmaxCtx& c, uint32_t j, bool first) {
  const DecodeParams& p = *c.p;
  const volatile float* alpha = reinterpret_cast<const volatile float*>(c.smem + kOffAlpha) +
                                (j % kOSlots) * kMaxHkv * kRows;
#pragma unroll 1
  for (int e = 0; e < 2; ++e) {
    const int h = 2 * c.pr + e;
    if (h >= p.Hkv) continue;
    uint32_t pg[16], om[8];
    tmem_ld16(c.tbase + c.lane_base + kColOPage + (j % kOSlots) * 64 + h * 16, pg);
    if (!first) tmem_ld8(c.tbase + c.lane_base + kColOMain + h * 16, om);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const float v = __uint_as_float(pg[i]) + __uint_as_float(pg[8 + i]);
      om[i] = __float_as_uint(first ? v : fmaf(__uint_as_float(om[i]), alpha[h * kRows + i], v));
    }
    tmem_st8(c.tbase + c.lane_base + kColOMain + h * 16, om);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (c.lane == 0) mbar_arrive(c.bars + 8 * (kBarOFree + j % kOSlots));
}

__device__ __forceinline__ void store_row(const DecodeParams& p, int seq, int hh, int r, int dim,
                                          float v) {
  const int tok = r / p.G, qh = hh * p.G + r % p.G;
  p.out[(((int64_t)seq * p.q_len + tok) * p.Hq + qh) * 128 + dim] = v;
}

__device__ void softmax_warps(const DecodeParams& p, uint8_t* smem, uint32_t tbase, int warp,
                              int lane) {
  SoftmaxCtx c;
  c.p = &p; c.smem = smem; c.sbase = smem_u32(smem); c.bars = c.sbase + kOffBars;
  c.tbase = tbase; c.lane = lane; c.qd = warp & 3;
  c.pr = (warp - kWarpSoftmax0) >> 2;
  c.lane_base = (uint32_t)(c.qd * 32) << 16;
  c.half = c.qd >> 1;                 // TMEM lanes 64..127 hold the odd head of the pair
  c.key = (c.qd * 32 + lane) & 63;
  c.head = 2 * c.pr + c.half;
  c.active = c.head < p.Hkv;
  c.gt = ((warp - kWarpSoftmax0) & 3) * 32 + lane;
  c.timed_out = false;
  const int dim = c.qd * 32 + lane;   // this thread's head dim in O
  const uint32_t gbar = 1 + c.pr;     // named barrier of this pair group (128 threads)
  const int rows_total = p.G * p.q_len;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + kOffFlags);
  volatile float* red = reinterpret_cast<volatile float*>(smem + kOffRed) + c.pr * 96;
  volatile float* alpha_s = reinterpret_cast<volatile float*>(smem + kOffAlpha);
  volatile float* mu_s = reinterpret_cast<volatile float*>(smem + kOffMu);
  volatile float* l_s = reinterpret_cast<volatile float*>(smem + kOffL);
  const volatile int32_t* stage_pid = reinterpret_cast<const volatile int32_t*>(smem + kOffStagePid);
  uint32_t k = 0;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];

  for (int s = s_begin; s < s_end; ++s) {
    const SegInfo sg = load_seg(p, s);
    const int n = sg.hi - sg.lo;
    const int row0 = sg.rg * kRows;
    const int L0 = sg.len - p.q_len;
    // largest visible key position of row i of the tile (-1 for a padding row)
    auto lim = [&](int i) -> int {
      const int r = row0 + i;
      return (r < rows_total) ? (p.causal ? L0 + r / p.G : sg.len - 1) : -1;
    };
    // ---- this pair's Q tile (B operand of Q.K^T) and its scale factors ----
    if (c.gt < 64) {
      const int nrow = c.gt >> 2, ch = c.gt & 3;
      const int hh = 2 * c.pr + (nrow >> 3), r = row0 + (nrow & 7);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (hh < p.Hkv && r < rows_total) {
        const int64_t qrow = ((int64_t)sg.seq * p.q_len + r / p.G) * p.Hq + hh * p.G + r % p.G;
        v = *reinterpret_cast<const uint4*>(p.q_codes + qrow * 64 + 16 * ch);
      }
      sts128(c.sbase + kOffQ + c.pr * 1024 + (nrow >> 3) * 512 + ch * 128 + (nrow & 7) * 16, v.x,
             v.y, v.z, v.w);
    }
    {
      uint32_t sf[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) sf[q] = 0u;
      if (lane < 16) {
        const int h2 = 2 * c.pr + (lane >> 3), r2 = row0 + (lane & 7);
        if (h2 < p.Hkv && r2 < rows_total) {
          const int64_t qrow = ((int64_t)sg.seq * p.q_len + r2 / p.G) * p.Hq + h2 * p.G + r2 % p.G;
          const uint2 qs = *reinterpret_cast<const uint2*>(p.q_scales + qrow * 8);
          sf[0] = qs.x;
          sf[4] = qs.y;
        }
      }
      tmem_st8(tbase + c.lane_base + kColSfb + c.pr * 8, sf);
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bars + 8 * kBarQReady);
    }
    float mu[kRows], lp[kRows];  // running max (raw score units) and partial row sums, own head
#pragma unroll
    for (int i = 0; i < kRows; ++i) { mu[i] = -INFINITY; lp[i] = 0.f; }

    write_sfa(c, k, sg.lo, sg.len);
    const uint32_t k0 = k;
    for (int j = 0; j < n; ++j, ++k) {
      if (j + 1 < n) write_sfa(c, k + 1, sg.lo + j + 1, sg.len);
      const uint32_t b = k & 1, st = k % kStages;
      wait_bar(c.bars + 8 * (kBarQkDone + b), (k >> 1) & 1, c.timed_out);
      tc_fence_after();
      uint32_t sr[8];
      tmem_ld8(tbase + c.lane_base + kColS + b * 32 + c.pr * 16 + c.half * 8, sr);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bars + 8 * (kBarSFree + b));

      // ---- exact page max per row: warp reduction, then across the two warps of the head ----
      const bool hv = c.active && stage_pid[st] >= 0;
      const int kp = (sg.lo + j) * 64 + c.key;
      uint32_t vmask = 0;  // bit i: key visible to row i
#pragma unroll
      for (int i = 0; i < kRows; ++i)
        if (hv && kp <= lim(i)) vmask |= 1u << i;
      volatile float* rb = red + (k & 1) * 32;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const float x = ((vmask >> i) & 1u) ? __uint_as_float(sr[i]) : -INFINITY;
        const float m = ord2f(__reduce_max_sync(0xffffffffu, f2ord(x)));
        if (lane == 0) rb[c.qd * 8 + i] = m;
      }
      named_barrier_sync(gbar, 128);
      float* alpha_page = const_cast<float*>(alpha_s) + (k % kOSlots) * kMaxHkv * kRows;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const float pm = fmaxf(rb[(2 * c.half) * 8 + i], rb[(2 * c.half + 1) * 8 + i]);
        const float mn = fmaxf(mu[i], pm);
        const float a = (mn == -INFINITY) ? 1.f : fast_exp2((mu[i] - mn) * p.c2);
        mu[i] = mn;
        lp[i] *= a;
        if (lane == 0 && (c.qd & 1) == 0 && c.head < kMaxHkv) alpha_page[c.head * kRows + i] = a;
      }
      // ---- P = exp2((s - mu) c2) <= 1 as f16 hi + lo, B operand of P.V (rows contiguous per key)
      if (k >= 2) wait_bar(c.bars + 8 * (kBarPvDone + b), ((k >> 1) - 1) & 1, c.timed_out);
      if (c.active) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < kRows; i += 2) {
          const float p0 = ((vmask >> i) & 1u) ? fast_exp2((__uint_as_float(sr[i]) - mu[i]) * p.c2) : 0.f;
          const float p1 =
              ((vmask >> (i + 1)) & 1u) ? fast_exp2((__uint_as_float(sr[i + 1]) - mu[i + 1]) * p.c2) : 0.f;
          lp[i] += p0;
          lp[i + 1] += p1;
          hi[i / 2] = pack_f16x2(p0, p1);
          lo[i / 2] = pack_f16x2(p0 - f16_lo_to_f32(hi[i / 2]), p1 - f16_hi_to_f32(hi[i / 2]));
        }
        const uint32_t a = c.sbase + kOffP + b * kPBytes + c.head * 2048 + (c.key >> 3) * 128 +
                           (c.key & 7) * 16;
        sts128(a, hi[0], hi[1], hi[2], hi[3]);
        sts128(a + 1024, lo[0], lo[1], lo[2], lo[3]);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bars + 8 * (kBarPFull + b));
      // ---- fold the page two back (its P.V completed: the wait above covered it) ----
      if (j >= 2) {
        tc_fence_after();
        fold_page(c, k - 2, k - 2 == k0);
      }
    }
    // ---- segment epilogue: fold the last pages, row sums, then O^T (one head dim per lane) ----
    for (uint32_t jj = (n >= 2 ? k - 2 : k0); jj < k; ++jj) {
      wait_bar(c.bars + 8 * (kBarPvDone + (jj & 1)), (jj >> 1) & 1, c.timed_out);
      tc_fence_after();
      fold_page(c, jj, jj == k0);
    }
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      float v = lp[i];
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
      if (lane == 0) red[64 + c.qd * 8 + i] = v;
      if (lane == 0 && (c.qd & 1) == 0 && c.head < kMaxHkv) mu_s[c.head * 8 + i] = mu[i];
    }
    named_barrier_sync(gbar, 128);
    if (c.gt < 16) {
      const int hf = c.gt >> 3, i = c.gt & 7, hh = 2 * c.pr + hf;
      l_s[hh * 8 + i] = red[64 + (2 * hf) * 8 + i] + red[64 + (2 * hf + 1) * 8 + i];
    }
    named_barrier_sync(gbar, 128);
    const bool split = sg.n_seg > 1;
    const int part_stride = p.Hkv * kPartHeadFloats;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = 2 * c.pr + e;
      if (h >= p.Hkv) continue;
      uint32_t o[8];
      tmem_ld8(tbase + c.lane_base + kColOMain + h * 16, o);
      tmem_wait_ld();
      float* part = split ? p.partials + (int64_t)sg.part * part_stride + h * kPartHeadFloats
                          : nullptr;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const int r = row0 + i;
        const float ov = __uint_as_float(o[i]);
        const float Ls = l_s[h * 8 + i];
        if (split) {
          if (r < rows_total) part[i * 128 + dim] = ov;
          if (dim == 0) {
            part[kRows * 128 + i] = mu_s[h * 8 + i];
            part[kRows * 128 + kRows + i] = Ls;
          }
        } else if (r < rows_total && Ls > 0.f) {
          store_row(p, sg.seq, h, r, dim, ov / Ls);
        }
      }
    }
    if (split) {
      // the CTA that completes the group's last segment combines all of its partials
      __threadfence();
      named_barrier_sync(3, 32 * kSoftmaxWarps);
      if (c.pr == 0 && c.gt == 0) {
        __threadfence();
        const int ticket = atomicAdd(p.counters + sg.group, 1);
        const int last = ticket == sg.n_seg - 1;
        if (last) p.counters[sg.group] = 0;  // ready for the next call on this workspace
        flags[24] = last;
      }
      named_barrier_sync(3, 32 * kSoftmaxWarps);
      if (flags[24]) {
        __threadfence();
        const float* pb = p.partials + (int64_t)sg.first_part * part_stride;
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * c.pr + e;
          if (h >= p.Hkv) continue;
          for (int i = 0; i < kRows; ++i) {
            const int r = row0 + i;
            if (r >= rows_total) continue;
            const float* ph = pb + h * kPartHeadFloats;
            float M = -INFINITY;
            for (int q = 0; q < sg.n_seg; ++q)
              M = fmaxf(M, __ldcg(ph + (int64_t)q * part_stride + kRows * 128 + i));
            float Lt = 0.f, Ot = 0.f;
            for (int q = 0; q < sg.n_seg; ++q) {
              const float* pq = ph + (int64_t)q * part_stride;
              const float mq = __ldcg(pq + kRows * 128 + i);
              const float f = (mq == -INFINITY) ? 0.f : fast_exp2((mq - M) * p.c2);
              Lt += f * __ldcg(pq + kRows * 128 + kRows + i);
              Ot += f * __ldcg(pq + i * 128 + dim);
            }
            if (Lt > 0.f) store_row(p, sg.seq, h, r, dim, Ot / Lt);
          }
        }
      }
    }
    named_barrier_sync(3, 32 * kSoftmaxWarps);  // scratch reused by the next segment
  }
  if (c.timed_out && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// --------------------------------------------------------------------------------------------
// Dequant warps: V codes x E4M3 scales -> f16 V^T tile (MN-major: 8 dims x 8 keys core tiles).
// Warp wd takes keys 16 wd .. 16 wd + 15 of every head (two groups of 8), each lane one key and one
// 32-dim quarter per group; the quarter is rotated by key so that shared-memory reads and writes
// are free of bank conflicts.
// --------------------------------------------------------------------------------------------
__device__ void dequant_warps(const DecodeParams& p, uint8_t* smem, int warp, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBars;
  const volatile int32_t* stage_pid = reinterpret_cast<const volatile int32_t*>(smem + kOffStagePid);
  const int wd = warp - kWarpDequant0;
  const int quarter = ((lane >> 3) + ((lane & 7) >> 1)) & 3;
  constexpr int kRounds = 64 / (8 * kDequantWarps);  // 8-key groups per warp and head
  uint32_t k = 0, hp = 0;
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const SegInfo sg = load_seg(p, s);
    for (int page = sg.lo; page < sg.hi; ++page, ++k) {
      const uint32_t st = k % kStages;
      wait_bar(bars + 8 * (kBarStageFull + st), (k / kStages) & 1, timed_out);
      const bool pvalid = stage_pid[st] >= 0;
      const uint32_t stage = sbase + kOffStage + st * kStageBytes;
      for (int h = 0; h < p.Hkv; ++h, ++hp) {
        const uint32_t slot = hp % kVhSlots;
        if (hp >= kVhSlots) wait_bar(bars + 8 * (kBarVhFree + slot), ((hp / kVhSlots) - 1) & 1, timed_out);
#pragma unroll
        for (int rd = 0; rd < kRounds; ++rd) {
          const int key = 8 * (kRounds * wd + rd) + (lane & 7);
          const bool kvalid = pvalid && page * 64 + key < sg.len;
          const uint4 cw = lds128(stage + p.Hkv * 4608 + h * 4096 + key * 64 + 16 * quarter);
          const uint32_t sc = kvalid ? lds16(stage + p.Hkv * 8704 + h * 512 + key * 8 + 2 * quarter) : 0u;
          const uint32_t sh = cvt_e4m3x2_f16(sc);
          const uint32_t s0 = dup_lo(sh), s1 = dup_hi(sh);
          const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
          const uint32_t vh = sbase + kOffVh + slot * kVhBytes + (key >> 3) * 2048 + (key & 7) * 16;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t r0, r1, r2, r3;
            cvt_e2m1x8_f16(words[q], r0, r1, r2, r3);
            const uint32_t sq = q < 2 ? s0 : s1;  // dims 32 quarter + 8 q .. : block 2 quarter + q / 2
            sts128(vh + (4 * quarter + q) * 128, hmul2(r0, sq), hmul2(r1, sq), hmul2(r2, sq),
                   hmul2(r3, sq));
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (kBarVhFull + slot));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * (kBarStageEmpty + st));
    }
  }
  if (timed_out && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = smem_u32(smem + kOffBars);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars + 8 * (kBarStageFull + s), 1);
      mbar_init(bars + 8 * (kBarStageEmpty + s), 8 + kDequantWarps + 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars + 8 * (kBarSfaFull + b), 8);
      mbar_init(bars + 8 * (kBarQkDone + b), 1);
      mbar_init(bars + 8 * (kBarSFree + b), 8);
      mbar_init(bars + 8 * (kBarPFull + b), 8);
      mbar_init(bars + 8 * (kBarPvDone + b), 1);
    }
    for (int v = 0; v < kVhSlots; ++v) {
      mbar_init(bars + 8 * (kBarVhFull + v), kDequantWarps);
      mbar_init(bars + 8 * (kBarVhFree + v), 1);
    }
    mbar_init(bars + 8 * kBarQReady, 8);
    for (int o = 0; o < kOSlots; ++o) mbar_init(bars + 8 * (kBarOFree + o), 8);
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(smem_u32(smem + kOffTmemSlot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);

  if (warp == kWarpProducer) {
    producer(p, smem, lane);
  } else if (warp == kWarpMma) {
    if (lane == 0) qk_issuer(p, smem, tbase);
  } else if (warp == kWarpPv) {
    if (lane == 0) pv_issuer(p, smem, tbase);
  } else if (warp < kWarpDequant0) {
    softmax_warps(p, smem, tbase, warp, lane);
  } else {
    dequant_warps(p, smem, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

int decode_smem_bytes() { return kSmemBytes; }

cudaError_t launch_decode(const uint8_t* q_codes, const uint8_t* q_scales, const uint8_t* pool,
                          const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                          const void* groups, const void* segments, const int32_t* cta_seg,
                          int32_t* counters, float* partials, float* out, int32_t* status,
                          int32_t Hq, int32_t Hkv, int32_t q_len, int32_t causal, int32_t grid,
                          float sm_scale, cudaStream_t stream) {
  static bool attr_done = false;  // the attribute belongs to the function, set once per process
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  if (Hkv < 1 || Hkv > kMaxHkv) return cudaErrorInvalidValue;
  DecodeParams p;
  p.q_codes = q_codes; p.q_scales = q_scales; p.pool = pool;
  p.block_table = block_table; p.max_pages = max_pages; p.num_pages = num_pages;
  p.groups = reinterpret_cast<const int4*>(groups);
  p.segments = reinterpret_cast<const int4*>(segments);
  p.cta_seg = cta_seg;
  p.counters = counters; p.partials = partials; p.out = out; p.status = status;
  p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv; p.q_len = q_len; p.causal = causal;
  p.c2 = sm_scale * 1.4426950408889634f;
  if (grid <= 0) return cudaSuccess;
  decode_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kvnvfp4
