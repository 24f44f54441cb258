// Paged GQA decode / speculative-verify attention over the NVFP4 cache, with split-K.
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
// spans CTAs leaves one (m, l, O) partial per segment, and a second launch merges the partials of
// every split group in parallel.
//
// One page = 64 keys of every KV head, a 9216 x H byte block moved by ONE bulk async copy.
//
// Q.K^T on the tcgen05 tensor cores: kind::mxf4nvf4, block_scale.scale_vec::4X (E2M1 x E2M1 with
// a UE4M3 scale per 16 elements), M = 128 = 64 keys of head 2p over 64 keys of head 2p+1, N = 16 =
// 8 query rows of head 2p then 8 of head 2p+1, K = 64 per instruction (two per 128-dim row). The
// K codes are stored in the pool in the tensor core's 8-row x 16-byte tile order, so the page
// lands in shared memory ready for the MMA; the K scales go to TMEM in the replicated 32-lane x
// 4-column layout. Cross terms (head 2p keys x head 2p+1 rows) are computed and ignored. Four
// MMAs per page for four KV heads.
//
// Softmax and P.V in eight attention warps. Warp (pair p, TMEM lane quadrant q) owns head
// 2p + q / 2 and keys 32 (q % 2) .. 32 (q % 2) + 31 of every page, with its own running max, row
// sums and O accumulator; the two warps of a head merge once, at the end of a segment. Per page a
// warp reads its S slice from TMEM (one key per lane), takes the page max per row with warp
// reductions, rescales its accumulator when a max grows, and writes P = exp2((s - m) log2e scale)
// <= 1 in f16 to a private shared tile (f16 keeps 11 significant bits of P; the method's own P.V
// runs in bf16, with 8). The P.V product runs on the warp-level tensor path (mma.sync m16n8k16,
// f32 accumulate), transposed: O^T += V^T P^T, with 16 head dims as M (a lane's rows g and g + 8
// are two adjacent dims of its 16-dim scale block), 16 keys as K and the 8 query rows as N. P
// comes in with one transposing ldmatrix per page; V goes from its E2M1 codes straight into A
// fragments: the nibbles of two keys are interleaved into one byte per dim, converted with
// cvt.e2m1x2 and multiplied by the two keys' E4M3 scales (E2M1 x E4M3 is exact in f16). Within a
// 16-key step the keys are taken in a fixed permutation, the same for P and V, that keeps the
// shared-memory reads conflict-free.
//
// Warp roles (320 threads): warp 0 bulk-copy producer, warp 1 Q.K^T issuer and TMEM owner, warps
// 2..9 attention. Every wait is an mbarrier wait bounded in time; on a timeout the kernel records
// KV_NVFP4_DEV_TIMEOUT and carries on, so it cannot hang.

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

namespace {

constexpr int kMaxHkv = 4;
constexpr int kStages = 5;
constexpr int kStageBytes = kMaxHkv * 9216;        // one page block of up to 4 heads
constexpr int kSBufs = 4;                          // score (S) buffers in TMEM
constexpr int kQBytes = 2 * 1024;                  // two head pairs x 16 rows x 64 B
constexpr int kRows = 8;                           // query rows per head per group
constexpr int kPartHeadFloats = kRows * 128 + 2 * kRows;  // O[8][128], m[8], l[8]

constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpAttn0 = 2;
constexpr int kAttnWarps = 8;
constexpr int kThreads = (kWarpAttn0 + kAttnWarps) * 32;
// Register bound: three warps share one SM sub-partition's 16K registers, so <= 168 per thread.
constexpr int kBoundThreads = 384;

// Fused step: at the start of each segment the producer fills one stage slot (the step slot) with
// the segment sequence's bf16 Q rows, new K and V rows and RoPE rows, ahead of the segment's pages,
// so the prologue that encodes them reads shared memory only. Offsets within the slot; the sizes
// are bounded by (Hq / Hkv) q_len <= 8: at most 32 Q rows, 32 K and 32 V rows of 256 B, 8 RoPE
// rows of up to 512 B.
constexpr int kStepQ = 0, kStepK = 8192, kStepV = 16384, kStepRope = 24576;
static_assert(kStepRope + 8 * 128 * 4 <= kMaxHkv * 9216, "step slot larger than a stage");

constexpr int kPsBytes = 1024;                     // per attention warp: 32 keys x (hi 16 B, lo 16 B)
constexpr int kMergeHeadBytes = 8 * 32 * 16 + 2 * kRows * 4;  // O: 8 float4 per lane; m[8], l[8]

// shared memory map
constexpr int kOffStage = 0;
constexpr int kOffSfStage = kOffStage + kStages * kStageBytes;  // [kSBufs][pair][k-half][32 x 16 B]
constexpr int kOffPs = kOffSfStage + kSBufs * 2048;
constexpr int kOffQ = kOffPs + kAttnWarps * kPsBytes;
constexpr int kOffMerge = kOffQ + kQBytes;
constexpr int kOffBars = kOffMerge + kMaxHkv * kMergeHeadBytes;
// barrier indices
constexpr int kBarStageFull = 0;                       // [kStages]
constexpr int kBarStageEmpty = kBarStageFull + kStages;  // [kStages]
constexpr int kBarQkDone = kBarStageEmpty + kStages;   // [kSBufs]
constexpr int kBarSFree = kBarQkDone + kSBufs;         // [kSBufs]
constexpr int kBarQReady = kBarSFree + kSBufs;
constexpr int kBarKvReady = kBarQReady + 1;  // fused append: the segment's new K/V rows are written
constexpr int kBarDrain = kBarKvReady + 1;   // every tcgen05 op of the CTA complete
constexpr int kNumBars = kBarDrain + 1;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
// misc: stage page ids, tmem base
constexpr int kOffStagePid = kOffMisc;
constexpr int kOffTmemSlot = kOffStagePid + 4 * 8;
constexpr int kOffQsc = kOffTmemSlot + 16;   // fused append: Q scales [2 pairs][16 rows][8]
constexpr int kSmemBytes = kOffQsc + 2 * 16 * 8;
static_assert(kStages <= 8, "stage page-id slots");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kOffQ % 16 == 0 && kOffQsc % 8 == 0, "Q tile 16-byte, Q scale rows 8-byte aligned");

// TMEM columns
constexpr uint32_t kColS = 0;                 // [kSBufs][2 pairs][16]
constexpr uint32_t kColSfa = 32 * kSBufs;     // [kSBufs][2 pairs][2 k-halves][4]
constexpr uint32_t kColSfb = 48 * kSBufs;     // [2 pairs][2 k-halves][4]
constexpr uint32_t kTmemCols = kColSfb + 16 <= 128 ? 128 : 256;  // a power of two >= 32
static_assert(kColSfb + 16 <= 256, "TMEM columns");

// instruction descriptor (dense, no negation): A, B = E2M1 (format 1) K-major, scale type UE4M3,
// N = 16, M = 128
constexpr uint32_t kIdescQK = (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// named barriers: 3 = the attention warps, 4 + h = the two warps of KV head h
constexpr uint32_t kNbAttn = 3, kNbHead0 = 4;

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
  float* partials;         // [num_partials][Hkv][kPartHeadFloats]
  float* out;
  int32_t* status;
  int32_t Hq, Hkv, G, q_len, causal;
  float c2;                // sm_scale * log2(e)
  // fused append (kv_nvfp4_decode_step): the step's new tokens, bf16, sequence-major
  const uint16_t* q_new;   // [num_seqs * q_len][Hq][128]
  const uint16_t* k_new;   // [num_seqs * q_len][Hkv][128]
  const uint16_t* v_new;
  const float* rope;       // [rope_max_pos][rot_dim]
  int32_t rope_max_pos, rot_dim;
  uint8_t* pool_w;         // the pool, receiving the new K/V rows
  uint8_t* q_codes_out;    // optional copy of the encoded Q rows, or null
  uint8_t* q_scales_out;
  // 1 when the plan tables (cta_seg, segments, groups) were written before the launch (not by the
  // kernel this one depends on), so that they may be read before the dependency wait
  int32_t early_tables;
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

// --------------------------------------------------------------------------------------------
// Producer warp: lane 0 streams the CTA's pages (all KV heads of a page in one bulk copy) into a
// kStages ring; the other lanes load page ids 32 at a time. The page id (or -1 when it lies
// outside the pool) is published in shared memory before the stage's full barrier is armed.
// --------------------------------------------------------------------------------------------
template <bool FUSED>
__device__ void producer(const DecodeParams& p, uint8_t* smem, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBars;
  volatile int32_t* stage_pid = reinterpret_cast<volatile int32_t*>(smem + kOffStagePid);
  const uint32_t blk_bytes = (uint32_t)p.Hkv * 9216u;
  // the pages are read once per call: marked first for eviction, they leave the L2 to what is
  // read again soon (the split-K partials, which the merge reads after this kernel, the plan
  // tables and the block table)
  const uint64_t stream_policy = l2_evict_first_policy();
  uint32_t k = 0, kvr = 0;
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const SegInfo sg = load_seg(p, s);
    if (FUSED) {  // the segment's step slot (bf16 Q, new K/V and RoPE rows of its sequence)
      if (lane == 0) {
        const uint32_t st = k % kStages;
        if (k >= kStages)
          wait_bar(bars + 8 * (kBarStageEmpty + st), ((k / kStages) - 1) & 1, timed_out);
        stage_pid[st] = -1;
        const int first_pos = sg.len - p.q_len;
        const uint32_t qb = (uint32_t)(p.q_len * p.Hq) * 256u, kb = (uint32_t)(p.q_len * p.Hkv) * 256u;
        // RoPE rows that exist in the table (a row past it is flagged by the prologue)
        const int nrope = p.rot_dim > 0 ? max(0, min(p.q_len, p.rope_max_pos - first_pos)) : 0;
        const uint32_t rb = (uint32_t)(nrope * p.rot_dim) * 4u;
        const uint32_t full = bars + 8 * (kBarStageFull + st);
        const uint32_t dst = sbase + kOffStage + st * kStageBytes;
        const int64_t tok0 = (int64_t)sg.seq * p.q_len;
        mbar_arrive_expect_tx(full, qb + 2u * kb + rb);
        bulk_g2s(dst + kStepQ, p.q_new + tok0 * p.Hq * kHeadDim, qb, full);
        bulk_g2s(dst + kStepK, p.k_new + tok0 * p.Hkv * kHeadDim, kb, full);
        bulk_g2s(dst + kStepV, p.v_new + tok0 * p.Hkv * kHeadDim, kb, full);
        if (rb > 0u) bulk_g2s(dst + kStepRope, p.rope + (int64_t)first_pos * p.rot_dim, rb, full);
      }
      ++k;
      __syncwarp();
    }
    // fused append: pages from this one on hold the step's new rows, written by this CTA's
    // attention warps at the segment's start; copy them only after that
    const int first_new_page = FUSED ? (sg.len - p.q_len) / kPage : 0x7fffffff;
    bool new_written = false;
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
          if (FUSED && !new_written && p0 + j >= first_new_page) {
            wait_bar(bars + 8 * kBarKvReady, kvr & 1, timed_out);
            ++kvr;
            new_written = true;
          }
          const bool valid = pid >= 0 && pid < p.num_pages;
          stage_pid[st] = valid ? pid : -1;
          const uint32_t full = bars + 8 * (kBarStageFull + st);
          if (valid) {
            mbar_arrive_expect_tx(full, blk_bytes);
            bulk_g2s_hint(sbase + kOffStage + st * kStageBytes, p.pool + (int64_t)pid * blk_bytes,
                          blk_bytes, full, stream_policy);
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
// Q.K^T warp. Per page the 32 lanes gather the page's K scales into the order of the MMA's scale
// factors (row i of a (pair, k-half) tile holds the 4-byte scale groups of MMA rows i, 32 + i,
// 64 + i, 96 + i) in a shared staging tile; lane 0 copies the tiles into TMEM with tcgen05.cp
// (replicated to the four lane quadrants) and issues the MMAs, which the tensor pipe runs after
// the copies. The warp runs ahead of the attention warps as far as the stage ring and the two S
// buffers allow.
// --------------------------------------------------------------------------------------------
template <bool FUSED>
__device__ void qk_warp(const DecodeParams& p, uint8_t* smem, uint32_t tbase, int lane) {
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBars;
  const int npairs = (p.Hkv + 1) >> 1;
  uint32_t k = 0, ks = 0, sgi = 0;  // pages (S buffers), stage slots, segments
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s, ++sgi) {
    const SegInfo sg = load_seg(p, s);
    if (FUSED) {
      // this warp's share of releasing the step slot; waiting for the slot first orders the
      // arrival after the slot's previous use was released (as for a page slot)
      const uint32_t st = ks % kStages;
      wait_bar(bars + 8 * (kBarStageFull + st), (ks / kStages) & 1, timed_out);
      if (lane == 0) mbar_arrive(bars + 8 * (kBarStageEmpty + st));
      ++ks;
    }
    for (int j = 0; j < sg.hi - sg.lo; ++j, ++k, ++ks) {
      const uint32_t st = ks % kStages, b = k % kSBufs;
      wait_bar(bars + 8 * (kBarStageFull + st), (ks / kStages) & 1, timed_out);
      // S buffer b free: the attention warps have read S of page k - kSBufs, so that page's MMAs
      // and scale copies are complete and staging tile b may be rewritten
      if (k >= kSBufs) wait_bar(bars + 8 * (kBarSFree + b), ((k / kSBufs) - 1) & 1, timed_out);
      const uint32_t stage = sbase + kOffStage + st * kStageBytes;
      const uint32_t sfs = sbase + kOffSfStage + b * 2048;
      // K scales: a full head pair's are already in the page in the scale-copy order (32 rows of
      // 16 bytes per k-half) and are copied straight from the stage; a last unpaired head's
      // 8-byte rows are widened into the staging tile first (the absent head's half is zero)
      const bool half_pair = (p.Hkv & 1) != 0;
      if (half_pair) {
        const int pr = npairs - 1;
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const uint2 v = lds64(stage + p.Hkv * 4096 + pr * 1024 + kh * 256 + lane * 8);
          sts128(sfs + (pr * 2 + kh) * 512 + lane * 16, v.x, v.y, 0u, 0u);
        }
        fence_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        tc_fence_after();
        for (int pr = 0; pr < npairs; ++pr)
          for (int kh = 0; kh < 2; ++kh) {
            const uint32_t src = (half_pair && pr == npairs - 1)
                                     ? sfs + (pr * 2 + kh) * 512
                                     : stage + p.Hkv * 4096 + pr * 1024 + kh * 512;
            tmem_cp_32x128b_x4(tbase + kColSfa + b * 16 + pr * 8 + kh * 4, smem_desc(src, 16, 128));
          }
      }
      if (j == 0) {
        // the segment's Q tile and its scales, awaited only now: the first page's K-scale copies
        // above were issued while the attention warps encoded Q
        __syncwarp();
        wait_bar(bars + 8 * kBarQReady, sgi & 1, timed_out);
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t qb = sbase + kOffQ;
        for (int pr = 0; pr < npairs; ++pr) {
          for (int kh = 0; kh < 2; ++kh) {
            const uint64_t ad = smem_desc(stage + pr * 8192 + kh * 256, 128, 512);
            const uint64_t bd = smem_desc(qb + pr * 1024 + kh * 256, 128, 512);
            mma_nvf4_ss(tbase + kColS + b * 32 + pr * 16, ad, bd, kIdescQK,
                        tbase + kColSfa + b * 16 + pr * 8 + kh * 4,
                        tbase + kColSfb + pr * 8 + kh * 4, (uint32_t)kh);
          }
        }
        mma_commit(bars + 8 * (kBarQkDone + b));
        mma_commit(bars + 8 * (kBarStageEmpty + st));  // K codes consumed once the MMAs complete
      }
      __syncwarp();
    }
    // a segment without pages (the plan makes none) still consumes its Q-ready phase
    if (sg.hi <= sg.lo) wait_bar(bars + 8 * kBarQReady, sgi & 1, timed_out);
  }
  if (timed_out) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// --------------------------------------------------------------------------------------------
// Attention warps: 8 warps, two groups of four. Group pr works on KV-head pair pr; within a group
// the four warps cover the four TMEM lane quadrants (qd = warp % 4). TMEM lane L = 32 qd + lane
// holds key L % 64 of head 2 pr + L / 64, so warp (pr, qd) owns head 2 pr + qd / 2 and keys
// 32 (qd % 2) .. 32 (qd % 2) + 31 of every page.
// --------------------------------------------------------------------------------------------
struct AttnCtx {
  const DecodeParams* p;
  uint8_t* smem;
  uint32_t sbase, bars, tbase, lane_base;
  int lane, qd, pr, half, head, key0, gt;  // gt: thread index within the pair group (0..127)
  bool active;                       // the warp's head exists (Hkv may be odd)
  bool timed_out;
};

// Byte address of the P row (half 0 of a 32-byte slot; half 1 is not used) of warp-local key
// `key` in a warp's P tile: four keys per 128-byte line, the slots and halves permuted by line so
// that both the row stores and the transposing ldmatrix reads are free of bank conflicts.
__device__ __forceinline__ uint32_t p_addr(uint32_t base, int key, int half) {
  const int q = key >> 2;
  return base + q * 128 + 32 * ((key & 3) ^ (q & 3)) + 16 * (half ^ (q & 1));
}

__device__ __forceinline__ float pick8(const float (&v)[kRows], int i) {
  float r = v[0];
#pragma unroll
  for (int j = 1; j < kRows; ++j) r = (i == j) ? v[j] : r;
  return r;
}

// Visibility of keys to the rows of the segment's row tile.
struct RowVis {
  int mylim;           // largest visible key position of row lane % 8 (-1 for a padding row)
  int lim_min;         // the smallest limit over the real rows (that of row 0)
  uint32_t rows_mask;  // bit i: row i is a real row
};

// Wait for page kk's scores and start loading this warp's slice (one key per lane, 8 rows).
__device__ __forceinline__ void s_issue(AttnCtx& c, uint32_t kk, uint32_t (&sr)[8]) {
  const uint32_t b = kk % kSBufs;
  wait_bar(c.bars + 8 * (kBarQkDone + b), (kk / kSBufs) & 1, c.timed_out);
  tc_fence_after();
  tmem_ld8(c.tbase + c.lane_base + kColS + b * 32 + c.pr * 16 + c.half * 8, sr);
}

// Finish loading page kk's scores and turn them into P in the P tile
// at pt: page max per row over the warp's 32 keys (warp reductions), running max and row-sum
// update, P = exp2((s - m) c2) <= 1 in f16. Returns whether a max grew (then alpha_a and
// alpha_b are the factors for rows 2t and 2t + 1 of the accumulator). kv_lim: keys of the page
// below it are real (0 when the page was skipped).
template <int NR>
__device__ __forceinline__ bool s_softmax(AttnCtx& c, uint32_t kk, uint32_t kst, int page, int len,
                                          const RowVis& rv, uint32_t (&sr)[8], float (&m)[kRows],
                                          float (&lp)[kRows], uint32_t pt, int t, float c2,
                                          float& alpha_a, float& alpha_b, int& kv_lim) {
  tmem_wait_ld_regs(sr);
  const uint32_t st = kst % kStages;
  // the Q.K^T warp saw this stage land; waiting here as well makes the V bytes and the page id
  // visible to this warp (the wait returns at once)
  wait_bar(c.bars + 8 * (kBarStageFull + st), (kst / kStages) & 1, c.timed_out);
  const bool pvalid = reinterpret_cast<const volatile int32_t*>(c.smem + kOffStagePid)[st] >= 0;
  kv_lim = pvalid ? len - page * 64 : 0;
  if (!c.active) return false;
  uint32_t vmask = 0;  // bit i: this lane's key is visible to row i
  if (pvalid) {
    if (page * 64 + 63 <= rv.lim_min) {
      vmask = rv.rows_mask;
    } else {
      const int kp = page * 64 + c.key0 + c.lane;
#pragma unroll
      for (int i = 0; i < NR; ++i)
        if (kp <= __shfl_sync(0xffffffffu, rv.mylim, i)) vmask |= 1u << i;
    }
  }
  float pm[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i)
    pm[i] = warp_max_f32(((vmask >> i) & 1u) ? __uint_as_float(sr[i]) : -INFINITY);
  bool grow = false;  // warp-uniform: every lane holds the same maxima
#pragma unroll
  for (int i = 0; i < NR; ++i) grow |= pm[i] > m[i];
  alpha_a = alpha_b = 1.f;
  if (grow) {  // rare once the running maxima have settled
    float alpha[kRows];
#pragma unroll
    for (int i = NR; i < kRows; ++i) alpha[i] = 1.f;
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      const float mn = fmaxf(m[i], pm[i]);
      alpha[i] = (mn == m[i]) ? 1.f : fast_exp2((m[i] - mn) * c2);  // 0 when m was -inf
      lp[i] *= alpha[i];
      m[i] = mn;
    }
    alpha_a = pick8(alpha, 2 * t);
    alpha_b = pick8(alpha, 2 * t + 1);
  }
  uint32_t hi[4];
#pragma unroll
  for (int i = 0; i < kRows; i += 2) {
    const float p0 = (i < NR && ((vmask >> i) & 1u))
                         ? fast_exp2((__uint_as_float(sr[i]) - m[i]) * c2) : 0.f;
    const float p1 = (i + 1 < NR && ((vmask >> (i + 1)) & 1u))
                         ? fast_exp2((__uint_as_float(sr[i + 1]) - m[i + 1]) * c2) : 0.f;
    lp[i] += p0;
    lp[i + 1] += p1;
    hi[i / 2] = pack_f16x2(p0, p1);
  }
  sts128(p_addr(pt, c.lane, 0), hi[0], hi[1], hi[2], hi[3]);
  return grow;
}

// O += P V over the warp's 32 keys of a page, two 16-key steps. P comes from the P tile through
// transposing ldmatrix (lm0, lm1: this lane's row addresses for the two steps); V codes of the
// lane's four keys per step (vk0, vk1, vk0 + 2, vk1 + 2) and dims 16 g .. 16 g + 15 are decoded
// into B fragments: one byte per dim holding the nibbles of two keys (first key low), converted
// by cvt.e2m1x2 and multiplied by the two keys' E4M3 scales. A key at or past kv_lim gets scale 0
// (its code bytes are stale). All shared loads of the page are issued before the arithmetic.
__device__ __forceinline__ void pv_page(const uint8_t* sm, uint32_t lm, uint32_t vco, uint32_t vso,
                                        int key0, int kv_lim, int vk0, int vk1,
                                        float (&acc)[8][4]) {
  // B fragments (P^T, keys x query rows) of both 16-key steps in one transposing ldmatrix
  uint32_t b[2][2];
  ldsm_x4_trans(lm, b[0][0], b[0][1], b[1][0], b[1][1]);
  uint2 wv[2][4];
  uint32_t sc[2][2];
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const int kb = key0 + 16 * ks;
    const int kk[4] = {kb + vk0, kb + vk1, kb + vk0 + 2, kb + vk1 + 2};
    uint32_t s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      wv[ks][e] = *reinterpret_cast<const uint2*>(sm + vco + kk[e] * 64);
      s[e] = kk[e] < kv_lim ? (uint32_t)sm[vso + kk[e] * 8] : 0u;
    }
    sc[ks][0] = cvt_e4m3x2_f16(s[0] | (s[1] << 8));
    sc[ks][1] = cvt_e4m3x2_f16(s[2] | (s[3] << 8));
  }
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const uint32_t x0 = w ? wv[ks][0].y : wv[ks][0].x, x1 = w ? wv[ks][1].y : wv[ks][1].x;
      const uint32_t x2 = w ? wv[ks][2].y : wv[ks][2].x, x3 = w ? wv[ks][3].y : wv[ks][3].x;
      const uint32_t ze01 = (x0 & 0x0F0F0F0Fu) | ((x1 << 4) & 0xF0F0F0F0u);
      const uint32_t zo01 = ((x0 >> 4) & 0x0F0F0F0Fu) | (x1 & 0xF0F0F0F0u);
      const uint32_t ze23 = (x2 & 0x0F0F0F0Fu) | ((x3 << 4) & 0xF0F0F0F0u);
      const uint32_t zo23 = ((x2 >> 4) & 0x0F0F0F0Fu) | (x3 & 0xF0F0F0F0u);
      uint32_t e0[4], o0[4], e2[4], o2[4];
      cvt_e2m1x8_f16(ze01, e0[0], e0[1], e0[2], e0[3]);
      cvt_e2m1x8_f16(zo01, o0[0], o0[1], o0[2], o0[3]);
      cvt_e2m1x8_f16(ze23, e2[0], e2[1], e2[2], e2[3]);
      cvt_e2m1x8_f16(zo23, o2[0], o2[1], o2[2], o2[3]);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)  // A rows g, g + 8: dims 16 g + 2 m, + 1 (m = 4 w + jj)
        mma16816(acc[4 * w + jj], hmul2(e0[jj], sc[ks][0]), hmul2(o0[jj], sc[ks][0]),
                 hmul2(e2[jj], sc[ks][1]), hmul2(o2[jj], sc[ks][1]), b[ks][0], b[ks][1]);
    }
  }
}

// Fused append (kv_nvfp4_decode_step), at the start of a segment: the tile's Q rows are encoded
// from bf16 (RoPE, Hadamard rotation, NVFP4: the append's arithmetic) straight into the Q tile,
// their scales into the staging rows at kOffQsc, and the step's new K/V rows that fall on this
// segment's pages into the pool. After a proxy fence the producer may copy those pages. The new
// tokens of sequence s are rows s * q_len .. s * q_len + q_len - 1 of q, k, v, at positions
// len - q_len .. len - 1; a sequence has one row tile here, so one CTA writes each new row.
// One new K or V row of the step, fetched (bf16 values, RoPE factors, page id) before it is
// encoded and stored.
struct NewKvRow {
  uint2 raw;
  float4 c, s;
  int32_t pid;
  int pos, h;
  bool is_k;
};

__device__ __forceinline__ void new_kv_fetch(const DecodeParams& p, const SegInfo& sg,
                                             const uint8_t* slot, int ri, int t0, int lane,
                                             NewKvRow& r) {
  const int tok = t0 + ri / (2 * p.Hkv), w = ri % (2 * p.Hkv);
  r.is_k = w < p.Hkv;
  r.h = r.is_k ? w : w - p.Hkv;
  r.pos = sg.len - p.q_len + tok;
  r.pid = p.block_table[(int64_t)sg.seq * p.max_pages + r.pos / kPage];
  r.raw = *reinterpret_cast<const uint2*>(slot + (r.is_k ? kStepK : kStepV) +
                                          (tok * p.Hkv + r.h) * 256 + 8 * lane);
  const bool rope = r.is_k && p.rot_dim > 0 && r.pos < p.rope_max_pos;
  rope_fetch(rope ? reinterpret_cast<const float*>(slot + kStepRope) + tok * p.rot_dim : nullptr,
             p.rot_dim, lane, r.c, r.s);
}

__device__ __forceinline__ void new_kv_store(const DecodeParams& p, const NewKvRow& r, int lane) {
  if (r.pid < 0 || r.pid >= p.num_pages) {  // the producer skips (and flags) the page as well
    if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_PAGE);
    return;
  }
  if (r.is_k && p.rot_dim > 0 && r.pos >= p.rope_max_pos) {
    if (lane == 0) flag_status(p.status, KV_NVFP4_DEV_BAD_ROPE);
    return;
  }
  float x[4] = {__uint_as_float(r.raw.x << 16), __uint_as_float(r.raw.x & 0xFFFF0000u),
                __uint_as_float(r.raw.y << 16), __uint_as_float(r.raw.y & 0xFFFF0000u)};
  uint32_t sc;
  const uint32_t packed =
      nvfp4_encode_row_fetched(x, r.is_k, r.is_k && p.rot_dim > 0, r.c, r.s, p.rot_dim, lane, sc);
  // page block: [K codes H*4096 (tile order)][K scales H*512][V codes H*4096][V scales H*512]
  uint8_t* blk = p.pool_w + (int64_t)r.pid * p.Hkv * 9216;
  const int slot = r.pos % kPage;
  uint8_t* codes;
  uint8_t* scales;  // this lane's block (lane / 4) when lane % 4 == 0
  if (r.is_k) {
    codes = blk + r.h * 4096 + (slot >> 3) * 512 + (slot & 7) * 16 + (lane >> 3) * 128 +
            ((2 * lane) & 15);
    scales = blk + kscale_offset(p.Hkv, r.h, slot, lane >> 4) + ((lane >> 2) & 3);
  } else {
    codes = blk + p.Hkv * 4608 + r.h * 4096 + slot * 64 + 2 * lane;
    scales = blk + p.Hkv * 8704 + r.h * 512 + slot * 8 + (lane >> 2);
  }
  *reinterpret_cast<uint16_t*>(codes) = (uint16_t)packed;
  if ((lane & 3) == 0) *scales = (uint8_t)sc;
}

// Fused step, per segment, by the attention warps: the segment's Q tile encoded from the bf16
// rows into shared memory (and, by the first segment of the group, into q_codes_out), and the
// step's new K/V rows that fall on the segment's pages stored into the pool. The bf16 rows and
// RoPE rows come from the step slot, which the producer filled ahead of the segment; the one
// global load left is the page id of a new row (while the other CTAs stream the cache, a global
// load takes about a microsecond, and the segment's first QK waits for this prologue). Inlined:
// out of line, its reads of the kernel parameters and the segment record went through memory and
// the prologue took about twice as long (a decode step of 4 x 128K tokens 1.8 us longer, measured).
// One Q row encoded by eight threads (o = lane % 8 holds the row's 16-value block o: elements
// 16 o .. 16 o + 15), from its bf16 values at `row` in shared memory: RoPE on the first rot dims
// (the partner of a rotated value read back from the staged row, each product rounded on its own,
// then added), the Hadamard stages 1 .. 8 in registers and 16, 32, 64 with lanes o ^ 1, o ^ 2,
// o ^ 4, the normalisation, and NVFP4 of the thread's own block (its amax, scale and codes need
// no exchange). Every step rounds as the definition states, so the codes and the scale equal those
// of the warp-per-row encoder bit for bit. All 32 lanes must call it (the exchanges are warp-wide);
// a lane with `load` false encodes zeros.
__device__ __forceinline__ void encode_q_octet(uint32_t row, bool load, const float* trow, int rot,
                                               int o, uint2& codes, uint32_t& scale) {
  float x[16];
  {
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    if (load) {
      v0 = lds128(row + 32 * o);
      v1 = lds128(row + 32 * o + 16);
    }
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
  if (load && trow != nullptr) {
    const int half = rot >> 1;
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 4) {
      const int e0 = 16 * o + k0;  // dims e0 .. e0 + 3 (rot / 2 is a multiple of 4)
      if (e0 < rot) {
        const bool lower = e0 < half;
        const int i0 = lower ? e0 : e0 - half;
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
#pragma unroll
  for (int hs = 1; hs < 16; hs <<= 1) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if ((k & hs) == 0) {
        const float a = x[k], b = x[k + hs];
        x[k] = __fadd_rn(a, b);
        x[k + hs] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    // the lower element of a pair sits in the thread without bit m: it keeps a + b, the other
    // a - b; (+-1) x is exact, so one fma rounds as the add or subtract does
    const float sgn = (o & m) != 0 ? -1.0f : 1.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float other = __shfl_xor_sync(0xffffffffu, x[k], m);
      x[k] = __fmaf_rn(sgn, x[k], other);
    }
  }
  const float kNorm = __uint_as_float(0x3DB504F3u);  // rn(2^-3.5) = rn(1/sqrt(128))
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    x[k] = __fmul_rn(x[k], kNorm);
    amax = fmaxf(amax, fabsf(x[k]));
  }
  const float r6 = __frcp_rn(6.0f);
  scale = e4m3x2_from_f32(0.0f, div_rn_by(amax, 6.0f, r6)) & 0xFFu;
  const float sd = e4m3_decode_pos(scale);
  const float rs = __frcp_rn(sd);
  float q[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) q[k] = quot_rn(x[k], sd, rs);
  const float(&q0)[8] = *reinterpret_cast<const float(*)[8]>(&q[0]);
  const float(&q1)[8] = *reinterpret_cast<const float(*)[8]>(&q[8]);
  codes = sd != 0.0f ? make_uint2(e2m1x8_from_f32(q0), e2m1x8_from_f32(q1))
                     : make_uint2(0u, 0u);  // an all-zero block: zero scale, zero codes
}

template <int NR>
__device__ __forceinline__ void fused_prologue(const DecodeParams& p, const SegInfo& sg,
                                               uint8_t* smem, const uint8_t* slot, uint32_t sbase,
                                               uint32_t bars, int aw, int lane) {
  const int rows_total = p.G * p.q_len;
  const int row0 = sg.rg * kRows;
  const bool q_out = p.q_codes_out != nullptr && (sg.n_seg == 1 || sg.part == sg.first_part);
  uint8_t* qsc = smem + kOffQsc;
  // the step's new K and V rows on this segment's pages; the first one of this warp fetched now
  // (its page id is a global load), stored after the Q rows are encoded
  const int first_pos = sg.len - p.q_len;
  const int t0 = max(0, sg.lo * kPage - first_pos), t1 = min(p.q_len, sg.hi * kPage - first_pos);
  const int nrows = t1 > t0 ? (t1 - t0) * 2 * p.Hkv : 0;
  NewKvRow kv;
  if (aw < nrows) new_kv_fetch(p, sg, slot, aw, t0, lane, kv);
  // The tile rows that can be real, NR per head (4 NR over the two head pairs), eight threads per
  // row and four rows per warp: row rr = 4 aw + lane / 8. Rows NR .. 7 of a head are never
  // computed; their Q tile rows keep the zeros written at the start.
  {
    const int o = lane & 7;
    const int rr = 4 * aw + (lane >> 3);
    const bool tile_row = rr < 4 * NR;
    const int pr = rr / (2 * NR), hip = (rr % (2 * NR)) / NR;
    const int nrow = 8 * hip + rr % NR;  // tile row of pair pr
    const int hh = 2 * pr + hip, r = row0 + (nrow & 7);
    int state = 0;  // 0: padding row, 1: row past the RoPE table, 2: row to encode
    int64_t qtrow = 0;
    uint32_t rowaddr = 0;
    const float* trow = nullptr;
    if (tile_row && hh < p.Hkv && r < rows_total) {
      const int tok = r / p.G, qh = hh * p.G + r % p.G;
      qtrow = ((int64_t)sg.seq * p.q_len + tok) * p.Hq + qh;
      const int pos = sg.len - p.q_len + tok;
      state = (p.rot_dim == 0 || pos < p.rope_max_pos) ? 2 : 1;
      rowaddr = smem_u32(slot) + kStepQ + (tok * p.Hq + qh) * 256;
      if (p.rot_dim > 0) trow = reinterpret_cast<const float*>(slot + kStepRope) + tok * p.rot_dim;
    }
    uint2 codes;
    uint32_t scale;
    encode_q_octet(rowaddr, state == 2, trow, p.rot_dim, o, codes, scale);
    if (state == 2 && q_out) {
      *reinterpret_cast<uint2*>(p.q_codes_out + qtrow * kCodeBytes + 8 * o) = codes;
      p.q_scales_out[qtrow * kScaleBytes + o] = (uint8_t)scale;
    } else if (state == 1 && o == 0) {  // a position past the RoPE table: flagged, scores zero
      flag_status(p.status, KV_NVFP4_DEV_BAD_ROPE);
    }
    if (tile_row) {
      // tensor-core tile order: the row's code bytes 8 o .. 8 o + 7 sit in 16-byte piece o / 2
      const uint32_t a = sbase + kOffQ + pr * 1024 + (nrow >> 3) * 512 + (o >> 1) * 128 +
                         (nrow & 7) * 16 + 8 * (o & 1);
      asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(codes.x), "r"(codes.y)
                   : "memory");
      qsc[(pr * 16 + nrow) * 8 + o] = (uint8_t)scale;
    }
  }
  if (aw < nrows) new_kv_store(p, kv, lane);
#pragma unroll 1
  for (int ri = aw + kAttnWarps; ri < nrows; ri += kAttnWarps) {  // more than 8 new rows
    new_kv_fetch(p, sg, slot, ri, t0, lane, kv);
    new_kv_store(p, kv, lane);
  }
  // the pool rows visible to this CTA's bulk copies (async proxy) before the producer copies their
  // page: each writer orders its stores before later async-proxy accesses, and the barrier below
  // plus the producer's wait on the KV-ready barrier carry that order to the copy (the only reader
  // of those rows in this kernel; a GPU-scope fence here made these CTAs the step's last by
  // 1-3 us); the Q tile and its staged scales complete before the scale factors are read
  if (nrows > 0) asm volatile("fence.proxy.async.global;" ::: "memory");
  named_barrier_sync(kNbAttn, 32 * kAttnWarps);
  if (nrows > 0 && aw == 0 && lane == 0) mbar_arrive(bars + 8 * kBarKvReady);
}

template <int NR, bool FUSED>
__device__ void attention_warps(const DecodeParams& p, uint8_t* smem, uint32_t tbase, int warp,
                                int lane) {
  AttnCtx c;
  c.p = &p; c.smem = smem; c.sbase = smem_u32(smem); c.bars = c.sbase + kOffBars;
  c.tbase = tbase; c.lane = lane; c.qd = warp & 3;
  const int aw = warp - kWarpAttn0;
  c.pr = aw >> 2;
  c.lane_base = (uint32_t)(c.qd * 32) << 16;
  c.half = c.qd >> 1;                 // TMEM lanes 64..127 hold the odd head of the pair
  c.head = 2 * c.pr + c.half;
  c.key0 = 32 * (c.qd & 1);
  c.active = c.head < p.Hkv;
  c.gt = (aw & 3) * 32 + lane;
  c.timed_out = false;
  const int g = lane >> 2, t = lane & 3;  // mma fragment coordinates
  const uint32_t ps = c.sbase + kOffPs + aw * kPsBytes;
  // ldmatrix rows of this lane: matrix mi = lane / 8 is 16-key step mi / 2, fragment k indices
  // 0..7 or 8..15 (mi % 2); the fragment k index maps to a warp-local key by the permutation
  // below (also used for V)
  uint32_t lm_addr;
  {
    const int mi = lane >> 3, kidx = (mi & 1) * 8 + (lane & 7), tt = (kidx & 7) >> 1;
    const int local = 4 * tt + ((kidx >> 3) << 1) + ((kidx & 1) ^ (tt & 1));
    lm_addr = p_addr(ps, 16 * (mi >> 1) + local, 0);
  }
  // B fragment keys of this lane within a 16-key step: k = 2t, 2t+1, 2t+8, 2t+9 -> keys
  // 4t + {0,1,2,3} with the pair order flipped for odd t (so lanes t and t+1 read different banks)
  const int vk0 = 4 * t + (t & 1), vk1 = 4 * t + 1 - (t & 1);
  const int rows_total = p.G * p.q_len;
  const float c2 = p.c2;
  uint32_t k = 0, ks = 0;  // pages (S buffers), stage slots
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];

  for (int s = s_begin; s < s_end; ++s) {
    const SegInfo sg = load_seg(p, s);
    const int n = sg.hi - sg.lo;
    const int row0 = sg.rg * kRows;
    const int L0 = sg.len - p.q_len;
    // largest visible key position of row lane % 8 of the tile (-1 for a padding row); rows are
    // ordered by token, so row 0 has the smallest limit
    int mylim;
    {
      const int r = row0 + (lane & 7);
      mylim = (r < rows_total) ? (p.causal ? L0 + r / p.G : sg.len - 1) : -1;
    }
    const int lim_min = __shfl_sync(0xffffffffu, mylim, 0);
    const uint32_t rows_mask = __ballot_sync(0xffffffffu, mylim >= 0) & 0xFFu;

    // ---- this pair's Q tile (B operand of Q.K^T) and its scale factors ----
    if (FUSED) {
      const uint32_t st = ks % kStages;
      wait_bar(c.bars + 8 * (kBarStageFull + st), (ks / kStages) & 1, c.timed_out);
      fused_prologue<NR>(p, sg, smem, smem + kOffStage + st * kStageBytes, c.sbase, c.bars, aw,
                         lane);
      if (lane == 0) mbar_arrive(c.bars + 8 * (kBarStageEmpty + st));  // slot read by this warp
      ++ks;
    } else if (c.gt < 64) {
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
      if (FUSED) {  // scales staged by the prologue, rows of pair c.pr in tile order
        if (lane < 16) {
          const uint2 qs = *reinterpret_cast<const uint2*>(smem + kOffQsc + (c.pr * 16 + lane) * 8);
          sf[0] = qs.x;
          sf[4] = qs.y;
        }
      } else if (lane < 16) {
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

    // running max (raw score units) and per-lane partial row sums, replicated per row
    float m[kRows], lp[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) { m[i] = -INFINITY; lp[i] = 0.f; }
    // O accumulator: acc[dd] is the m16n8 tile of dims 16 n + dd (n = fragment column); rows
    // 0..7 are the query rows, rows 8..15 stay zero
    float acc[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[mt][q] = 0.f;

    // Per page: scores -> running max, row sums and P (one P tile), accumulator rescale when a
    // max grew, then two 16-key steps of O += P V.
    const RowVis rv{mylim, lim_min, rows_mask};
    for (int j = 0; j < n; ++j, ++k, ++ks) {
      const uint32_t st = ks % kStages;
      uint32_t sr[8];
      float alpha_a = 1.f, alpha_b = 1.f;
      int kv_lim = 0;
      s_issue(c, k, sr);
      const bool grow = s_softmax<NR>(c, k, ks, sg.lo + j, sg.len, rv, sr, m, lp, ps, t, c2,
                                      alpha_a, alpha_b, kv_lim);
      __syncwarp();
      if (grow) {  // entries 0, 2: row 2t; entries 1, 3: row 2t + 1
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          acc[mt][0] *= alpha_a; acc[mt][2] *= alpha_a;
          acc[mt][1] *= alpha_b; acc[mt][3] *= alpha_b;
        }
      }
      if (c.active) {
        const uint32_t stage = c.sbase + kOffStage + st * kStageBytes;
        const uint32_t vc = stage + p.Hkv * 4608 + c.head * 4096 + 8 * g;  // codes of dims 16 g ..
        const uint32_t vs = stage + p.Hkv * 8704 + c.head * 512 + g;       // scale of block g
        pv_page(smem, lm_addr, vc - c.sbase, vs - c.sbase, c.key0, kv_lim, vk0, vk1, acc);
      }
      // the page's S buffer and stage slot are released together (the Q.K^T warp runs pages
      // ahead, so it seldom waits for an S buffer)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(c.bars + 8 * (kBarSFree + k % kSBufs));
        mbar_arrive(c.bars + 8 * (kBarStageEmpty + st));
      }
    }

    // ---- segment end: row sums, then the two warps of each head merge ----
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      float v = lp[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      lp[i] = v;
    }
    const bool split = sg.n_seg > 1;
    const int part_stride = p.Hkv * kPartHeadFloats;
    if (c.active) {
      // lane (g, t) holds rows 2t and 2t + 1, dims 16 g .. 16 g + 15: acc[m][0 | 2] is row 2t,
      // dims 16 g + 2m | 16 g + 2m + 1; acc[m][1 | 3] the same for row 2t + 1
      const uint32_t mg = c.sbase + kOffMerge + c.head * kMergeHeadBytes;
      volatile float* mml =
          reinterpret_cast<volatile float*>(smem + kOffMerge + c.head * kMergeHeadBytes + 8 * 32 * 16);
      const uint32_t hb = kNbHead0 + c.head;
      if (c.qd & 1) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          sts128(mg + (q * 32 + lane) * 16, __float_as_uint(acc[q][0]), __float_as_uint(acc[q][1]),
                 __float_as_uint(acc[q][2]), __float_as_uint(acc[q][3]));
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < kRows; ++i) { mml[i] = m[i]; mml[kRows + i] = lp[i]; }
        }
        named_barrier_sync(hb, 64);  // state written
        named_barrier_sync(hb, 64);  // state read: the area is free for the next segment
      } else {
        named_barrier_sync(hb, 64);
        float M[2], L[2], f1[2], f2[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = 2 * t + hh;
          const float m1 = pick8(m, i), l1 = pick8(lp, i);
          const float m2 = mml[i], l2 = mml[kRows + i];
          M[hh] = fmaxf(m1, m2);
          f1[hh] = (m1 == -INFINITY) ? 0.f : fast_exp2((m1 - M[hh]) * c2);
          f2[hh] = (m2 == -INFINITY) ? 0.f : fast_exp2((m2 - M[hh]) * c2);
          L[hh] = f1[hh] * l1 + f2[hh] * l2;
        }
        float o[2][16];  // rows 2t, 2t + 1; dims 16 g .. 16 g + 15
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 u = lds128(mg + (q * 32 + lane) * 16);
          o[0][2 * q] = f1[0] * acc[q][0] + f2[0] * __uint_as_float(u.x);
          o[1][2 * q] = f1[1] * acc[q][1] + f2[1] * __uint_as_float(u.y);
          o[0][2 * q + 1] = f1[0] * acc[q][2] + f2[0] * __uint_as_float(u.z);
          o[1][2 * q + 1] = f1[1] * acc[q][3] + f2[1] * __uint_as_float(u.w);
        }
        named_barrier_sync(hb, 64);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = 2 * t + hh, r = row0 + i;
          if (split) {
            float* part = p.partials + (int64_t)sg.part * part_stride + c.head * kPartHeadFloats;
            float4* dst = reinterpret_cast<float4*>(part + i * 128 + 16 * g);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_float4(o[hh][4 * q], o[hh][4 * q + 1], o[hh][4 * q + 2], o[hh][4 * q + 3]);
            if (g == 0) {
              part[kRows * 128 + i] = M[hh];
              part[kRows * 128 + kRows + i] = L[hh];
            }
          } else if (r < rows_total && L[hh] > 0.f) {
            const int tok = r / p.G, qh = c.head * p.G + r % p.G;
            float4* dst = reinterpret_cast<float4*>(
                p.out + (((int64_t)sg.seq * p.q_len + tok) * p.Hq + qh) * 128 + 16 * g);
            const float inv = 1.f / L[hh];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_float4(o[hh][4 * q] * inv, o[hh][4 * q + 1] * inv,
                                   o[hh][4 * q + 2] * inv, o[hh][4 * q + 3] * inv);
          }
        }
      }
    }
  }
  if (c.timed_out && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

// NR: query rows computed per head (6 when no tile has more real rows, else all 8); FUSED: the
// step's append is done in the kernel (kv_nvfp4_decode_step)
template <int NR, bool FUSED>
__global__ void __launch_bounds__(kBoundThreads, 1) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = smem_u32(smem + kOffBars);
  // the split-K merge launched after this kernel may be scheduled now; it waits for this grid's
  // completion before it reads anything this kernel writes
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars + 8 * (kBarStageFull + s), 1);
      mbar_init(bars + 8 * (kBarStageEmpty + s), 1 + kAttnWarps);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(bars + 8 * (kBarQkDone + b), 1);
      mbar_init(bars + 8 * (kBarSFree + b), kAttnWarps);
    }
    mbar_init(bars + 8 * kBarQReady, kAttnWarps);
    mbar_init(bars + 8 * kBarKvReady, 1);
    mbar_init(bars + 8 * kBarDrain, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(smem_u32(smem + kOffTmemSlot), kTmemCols);
  // the fused prologue writes only the rows that can be real: the others stay zero
  for (int i = threadIdx.x; i < kQBytes / 16; i += kThreads)
    sts128(smem_u32(smem + kOffQ) + 16 * i, 0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < 2 * 16; i += kThreads)  // 8-byte rows (the area is 8-aligned)
    *reinterpret_cast<uint2*>(smem + kOffQsc + 8 * i) = make_uint2(0u, 0u);
  if (p.early_tables && lane == 0) {
    // bring this CTA's first segment record into L1 while the previous kernel finishes: every warp
    // starts by reading it, three dependent loads that otherwise take ~1.5 us under the page
    // stream of the other CTAs
    const int s0 = __ldg(p.cta_seg + blockIdx.x), s1 = __ldg(p.cta_seg + blockIdx.x + 1);
    if (s0 < s1) {
      const int4 seg = __ldg(p.segments + s0);
      const int4 g0 = __ldg(p.groups + 2 * seg.x), g1 = __ldg(p.groups + 2 * seg.x + 1);
      asm volatile("" ::"r"(g0.x), "r"(g1.x));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // launched as a programmatic dependent of the previous kernel on the stream (the append that
  // wrote this step's pool rows and Q, or the previous call's merge, which reads the partials this
  // kernel rewrites): everything above overlapped its tail; nothing below runs before it completes
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);

  if (warp == kWarpProducer) {
    producer<FUSED>(p, smem, lane);
  } else if (warp == kWarpMma) {
    qk_warp<FUSED>(p, smem, tbase, lane);
  } else {
    attention_warps<NR, FUSED>(p, smem, tbase, warp, lane);
  }

  if (warp == kWarpMma) {
    // tensor memory is freed only once no tcgen05 op of this CTA is in flight (after a timeout
    // some may still be; the wait is bounded like every other)
    if (lane == 0) mma_commit(bars + 8 * kBarDrain);
    __syncwarp();
    bool to = false;
    wait_bar(bars + 8 * kBarDrain, 0, to);
    if (to && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tbase, kTmemCols);
}

// --------------------------------------------------------------------------------------------
// Split-K merge (second launch). One CTA per (split group, KV head, row of the tile); its 256
// threads are 8 slices of the group's partials x 32 four-dim columns, so the partial reads of all
// groups run in parallel across the GPU:
//   M = max_q m_q,  L = sum_q 2^((m_q - M) c2) l_q,  o = sum_q 2^((m_q - M) c2) O_q / L.
// --------------------------------------------------------------------------------------------
struct MergeParams {
  const int4* groups;
  const int32_t* split;    // [num_split] group indices
  const float* partials;   // [num_partials][Hkv][kPartHeadFloats]
  float* out;
  int32_t Hq, Hkv, G, q_len;
  float c2;
};

constexpr int kMergeSlices = 8;
constexpr int kMergePerRound = 8;  // partials a slice requests at once (64 per CTA and round)

// LATE_TABLES: the plan tables were written by a kernel earlier in the same step (not by a copy
// before the attention launch), so they are read only after the wait as well.
template <bool LATE_TABLES>
__global__ void __launch_bounds__(32 * kMergeSlices, 2) merge_kernel(const MergeParams p) {
  __shared__ float s_m[kMergeSlices], s_l[kMergeSlices];
  __shared__ float4 s_o[kMergeSlices][32];
  asm volatile("griddepcontrol.launch_dependents;");  // the next kernel may begin its launch
  // launched as a programmatic dependent of the attention kernel: its partials are visible only
  // after this wait (which returns when that grid has completed and flushed)
  if (LATE_TABLES) asm volatile("griddepcontrol.wait;" ::: "memory");
  const int gi = p.split[blockIdx.x];  // plan tables: written before the attention launch
  const int h = blockIdx.y / kRows, i = blockIdx.y % kRows;
  const int4 g0 = p.groups[2 * gi], g1 = p.groups[2 * gi + 1];
  const int r = g0.z * kRows + i;
  if (!LATE_TABLES) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (r >= p.G * p.q_len) return;  // padding row of the last tile (uniform over the CTA)
  const int n_seg = g1.x;
  const int slice = threadIdx.x >> 5, d4 = threadIdx.x & 31;
  const int64_t stride = (int64_t)p.Hkv * kPartHeadFloats;
  const float* base = p.partials + (int64_t)g1.y * stride + h * kPartHeadFloats;
  // Per round a slice requests its partials q = q0 + 8 u (u < 8) all at once, so that a round
  // costs one L2 round trip (a group of up to 64 segments takes one round); they are then
  // combined with independent maxima and weights rather than one dependent step per partial.
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = slice; q0 < n_seg; q0 += kMergeSlices * kMergePerRound) {
    float mq[kMergePerRound], lq[kMergePerRound];
    float4 ov[kMergePerRound];
#pragma unroll
    for (int u = 0; u < kMergePerRound; ++u) {
      const int q = q0 + kMergeSlices * u;
      mq[u] = -INFINITY;
      lq[u] = 0.f;
      ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (q < n_seg) {
        const float* pq = base + q * stride;
        mq[u] = __ldcg(pq + kRows * 128 + i);
        lq[u] = __ldcg(pq + kRows * 128 + kRows + i);
        ov[u] = __ldcg(reinterpret_cast<const float4*>(pq + i * 128) + d4);
      }
    }
    float mn = M;
#pragma unroll
    for (int u = 0; u < kMergePerRound; ++u) mn = fmaxf(mn, mq[u]);
    if (mn == -INFINITY) continue;  // no visible key in any partial so far
    const float a = fast_exp2((M - mn) * p.c2);  // 0 while M is -inf
    L *= a;
    O.x *= a; O.y *= a; O.z *= a; O.w *= a;
#pragma unroll
    for (int u = 0; u < kMergePerRound; ++u) {
      if (mq[u] == -INFINITY) continue;  // a segment with no visible key, or none at all
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
    for (int j = 1; j < kMergeSlices; ++j) Mt = fmaxf(Mt, s_m[j]);
    float Lt = 0.f;
    float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMergeSlices; ++j) {
      if (s_m[j] == -INFINITY) continue;
      const float f = fast_exp2((s_m[j] - Mt) * p.c2);
      const float4 v = s_o[j][d4];
      Lt += f * s_l[j];
      Ot.x += f * v.x; Ot.y += f * v.y; Ot.z += f * v.z; Ot.w += f * v.w;
    }
    if (Lt > 0.f) {
      const int tok = r / p.G, qh = h * p.G + r % p.G;
      float4* dst = reinterpret_cast<float4*>(
          p.out + (((int64_t)g0.x * p.q_len + tok) * p.Hq + qh) * 128 + 4 * d4);
      const float inv = 1.f / Lt;
      *dst = make_float4(Ot.x * inv, Ot.y * inv, Ot.z * inv, Ot.w * inv);
    }
  }
}

}  // namespace

int decode_smem_bytes() { return kSmemBytes; }

cudaError_t launch_split_merge(const void* groups, const int32_t* split_groups,
                               const float* partials, float* out, int32_t Hq, int32_t Hkv,
                               int32_t G, int32_t q_len, float c2, int32_t num_split,
                               bool late_tables, cudaStream_t stream);

cudaError_t launch_decode(const uint8_t* q_codes, const uint8_t* q_scales, const uint8_t* pool,
                          const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                          const void* groups, const void* segments, const int32_t* cta_seg,
                          const int32_t* split_groups, int32_t num_split, float* partials,
                          float* out, int32_t* status,
                          int32_t Hq, int32_t Hkv, int32_t q_len, int32_t causal, int32_t grid,
                          float sm_scale, const uint16_t* q_new, const uint16_t* k_new,
                          const uint16_t* v_new, const float* rope, int32_t rope_max_pos,
                          int32_t rot_dim, uint8_t* pool_w, uint8_t* q_codes_out,
                          uint8_t* q_scales_out, bool late_tables, cudaStream_t stream) {
  // the attribute belongs to each instantiation and each device: set once per device
  static bool attr_done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaSuccess;
    const void* kernels[] = {(const void*)decode_kernel<8, false>, (const void*)decode_kernel<6, false>,
                             (const void*)decode_kernel<8, true>, (const void*)decode_kernel<6, true>};
    for (const void* kf : kernels)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  if (Hkv < 1 || Hkv > kMaxHkv) return cudaErrorInvalidValue;
  DecodeParams p;
  p.q_codes = q_codes; p.q_scales = q_scales; p.pool = pool;
  p.block_table = block_table; p.max_pages = max_pages; p.num_pages = num_pages;
  p.groups = reinterpret_cast<const int4*>(groups);
  p.segments = reinterpret_cast<const int4*>(segments);
  p.cta_seg = cta_seg;
  p.partials = partials; p.out = out; p.status = status;
  p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv; p.q_len = q_len; p.causal = causal;
  p.c2 = sm_scale * 1.4426950408889634f;
  p.q_new = q_new; p.k_new = k_new; p.v_new = v_new; p.rope = rope;
  p.rope_max_pos = rope_max_pos; p.rot_dim = rot_dim; p.pool_w = pool_w;
  p.q_codes_out = q_codes_out; p.q_scales_out = q_scales_out;
  p.early_tables = late_tables ? 0 : 1;
  const bool fused = q_new != nullptr;
  if (grid <= 0) return cudaSuccess;
  // programmatic dependent launch: the kernel is set up while the previous kernel on the stream
  // finishes, and waits for it (griddepcontrol.wait) before touching memory
  {
    cudaLaunchConfig_t dc = {};
    dc.gridDim = dim3((unsigned)grid);
    dc.blockDim = dim3(kThreads);
    dc.dynamicSmemBytes = kSmemBytes;
    dc.stream = stream;
    cudaLaunchAttribute da[1];
    da[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    da[0].val.programmaticStreamSerializationAllowed = 1;
    dc.attrs = da;
    dc.numAttrs = 1;
    // every tile has at most G * q_len real rows: with six or fewer, rows 6 and 7 are never computed
    const bool six = p.G * q_len <= 6;
    const cudaError_t le =
        fused ? (six ? cudaLaunchKernelEx(&dc, decode_kernel<6, true>, p)
                     : cudaLaunchKernelEx(&dc, decode_kernel<8, true>, p))
              : (six ? cudaLaunchKernelEx(&dc, decode_kernel<6, false>, p)
                     : cudaLaunchKernelEx(&dc, decode_kernel<8, false>, p));
    if (le != cudaSuccess) return le;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || num_split <= 0) return e;
  return launch_split_merge(p.groups, split_groups, partials, out, Hq, Hkv, p.G, q_len, p.c2,
                            num_split, late_tables, stream);
}

// The split-K merge launch (also used by the comparator decode): one CTA per (split group, KV
// head, row of the tile), as a programmatic dependent of the attention kernel before it on the
// stream (it waits for that grid to complete before reading the partials).
cudaError_t launch_split_merge(const void* groups, const int32_t* split_groups,
                               const float* partials, float* out, int32_t Hq, int32_t Hkv,
                               int32_t G, int32_t q_len, float c2, int32_t num_split,
                               bool late_tables, cudaStream_t stream) {
  if (num_split <= 0) return cudaSuccess;
  MergeParams mp;
  mp.groups = static_cast<const int4*>(groups); mp.split = split_groups; mp.partials = partials;
  mp.out = out; mp.Hq = Hq; mp.Hkv = Hkv; mp.G = G; mp.q_len = q_len; mp.c2 = c2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_split, (unsigned)(Hkv * kRows));
  cfg.blockDim = dim3(32 * kMergeSlices);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return late_tables ? cudaLaunchKernelEx(&cfg, merge_kernel<true>, mp)
                     : cudaLaunchKernelEx(&cfg, merge_kernel<false>, mp);
}

}  // namespace kvnvfp4
