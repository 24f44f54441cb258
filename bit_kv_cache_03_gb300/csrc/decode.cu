// Paged GQA decode / speculative-verify attention over the NVFP4 cache, with split-K.
//
// Source: prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)": Q.K^T from
// NVFP4 Q and K with their E4M3 block scales, V dequantised for the P.V product, row-major KV
// scales. Split-K with an fp32 log-sum-exp merge is this library's design (the pages run long
// contexts from a paged pool and say nothing about the kernel's decomposition).
//
// Work decomposition: a group is (sequence, kv head, tile of 8 query rows); a row is (query token,
// head in the GQA group), row = token * group + head_in_group. The plan lays the groups' pages
// (cut into split-K chunks) end to end and hands every CTA (one persistent CTA per SM) an equal
// share of that page stream; a CTA's share is one or more segments, each a contiguous page
// range of one group. Within a segment the CTA's state carries across chunks (online softmax);
// at the end of a segment it writes either the final rows (the group lies in one CTA) or one
// (m, l, O) partial, and the CTA that takes the group's last ticket combines its partials.
//
// Per CTA: the last warp is the producer; lane 0 streams every page of the CTA's segments into a
// 16-slot shared-memory ring with bulk async copies (K codes 4 KiB, K scales 512 B, V codes
// 4 KiB, V scales 512 B per page and head), each slot guarded by a full and an empty mbarrier.
// Warps 0..11 consume: three groups of four warps take the segment's pages round-robin, and the
// four warps of a group split a page into 16-key sub-tiles (empty barrier count 4).
//
// Per 16-key sub-tile and warp, the product runs on the warp-level tensor path with keys as the M
// dimension (16 keys per MMA) and the 8 query rows as N:
//   S^T[key][row] = sum_d Khat[key][d] Qhat[row][d]        (8 x m16n8k16, k = 16 dims per step)
//   O^T[dim][row] += sum_key Vhat^T[dim][key] P^T[key][row] (8 m-tiles of 16 dims)
// Khat, Vhat and Qhat are the NVFP4 values converted to f16 (E2M1 * E4M3 has at most 6
// significant bits and lies in [2^-10, 2688], so it is exact in f16); products accumulate in
// fp32. P is fed as an f16 hi/lo pair (p = hi + lo to ~2^-22 relative), so the P.V product
// carries fp32-level precision. The dims inside an MMA are a fixed permutation of the head
// dims (the same one for both operands), chosen so that each thread reads contiguous bytes.
//
// Softmax: running max per row, exp2 with log2(e) folded into the scale, rescale of the
// accumulator only when the max grows. At the end of a segment the 12 warps' states are merged
// in shared memory; merging never waits on another CTA.

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

namespace {

constexpr int kGroups = 3;                     // pages processed concurrently per CTA
constexpr int kConsumerWarps = 4 * kGroups;     // four warps (16-key sub-tiles) per page
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kSlots = 16;
constexpr int kKcOff = 0, kKsOff = 4096, kVcOff = 4608, kVsOff = 8704;
constexpr int kSlotBytes = 9216;
constexpr int kRows = 8;                           // query rows per work item
constexpr int kPartFloats = kRows * 128 + 2 * kRows;  // O[8][128], m[8], l[8]
constexpr int kRingBytes = kSlots * kSlotBytes;
constexpr int kBarOff = kRingBytes;                // 2 * kSlots mbarriers
constexpr int kSlotPidOff = kBarOff + 2 * kSlots * 8;   // int32 page id per slot
constexpr int kMergeOff = kSlotPidOff + kSlots * 4;
constexpr int kMergeFloats = kConsumerWarps * kPartFloats;
constexpr int kFlagOff = kMergeOff + kMergeFloats * 4;
constexpr int kSmemBytes = kFlagOff + 16;

struct DecodeParams {
  const uint8_t* q_codes;
  const uint8_t* q_scales;
  const uint8_t* k_codes;
  const uint8_t* k_scales;
  const uint8_t* v_codes;
  const uint8_t* v_scales;
  const int32_t* block_table;
  int32_t max_pages;
  int32_t num_pages;
  const int4* groups;    // 2 x int4 per group: {seq, kvh, rg, len}, {n_seg, first_part, pages, 0}
  const int4* segments;  // {group, page_lo, page_hi, part_slot or -1}
  const int32_t* cta_seg;  // [grid + 1]: segments of CTA b are [cta_seg[b], cta_seg[b+1])
  int32_t* counters;     // [num_groups], merge tickets
  float* partials;       // [num_partials][kPartFloats]
  float* out;
  int32_t* status;
  int32_t Hq, Hkv, G, q_len, causal;
  float c2;              // sm_scale * log2(e)
};

// --------------------------------------------------------------------------------------------
// Producer warp: lane 0 streams the CTA's pages into the ring; the other lanes help load page
// ids 32 at a time. The page id (or -1 for an id outside the pool) is published in shared
// memory before the slot's full barrier is armed, so consumers never read the block table.
// --------------------------------------------------------------------------------------------
__device__ void producer(const DecodeParams& p, uint8_t* smem, int lane) {
  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = smem_u32(smem + kBarOff);
  volatile int32_t* slot_pid = reinterpret_cast<volatile int32_t*>(smem + kSlotPidOff);
  uint32_t k = 0;
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];
  for (int s = s_begin; s < s_end; ++s) {
    const int4 seg = p.segments[s];
    const int4 g0 = p.groups[2 * seg.x];
    const int seq = g0.x, kvh = g0.y;
    for (int p0 = seg.y; p0 < seg.z; p0 += 32) {
      const int n = min(32, seg.z - p0);
      const int32_t mine = (lane < n) ? p.block_table[(int64_t)seq * p.max_pages + p0 + lane] : -1;
      for (int j = 0; j < n; ++j, ++k) {
        const int32_t pid = __shfl_sync(0xffffffffu, mine, j);
        if (lane == 0) {
          const uint32_t slot = k % kSlots;
          const uint32_t full = bars + 8 * slot;
          if (k >= kSlots) {
            if (!mbar_wait_bounded(bars + 8 * (kSlots + slot), ((k / kSlots) - 1) & 1))
              timed_out = true;
          }
          const bool valid = pid >= 0 && pid < p.num_pages;
          slot_pid[slot] = valid ? pid : -1;
          if (valid) {
            const int64_t head = (int64_t)pid * p.Hkv + kvh;
            const uint32_t dst = ring + slot * kSlotBytes;
            mbar_arrive_expect_tx(full, kSlotBytes);
            bulk_g2s(dst + kKcOff, p.k_codes + head * 4096, 4096, full);
            bulk_g2s(dst + kKsOff, p.k_scales + head * 512, 512, full);
            bulk_g2s(dst + kVcOff, p.v_codes + head * 4096, 4096, full);
            bulk_g2s(dst + kVsOff, p.v_scales + head * 512, 512, full);
          } else {
            mbar_arrive(full);  // completes the phase with no data; consumers skip the page
          }
        }
        __syncwarp();
      }
    }
  }
  if (lane == 0) {
    // Drain: no copy into this CTA's shared memory may still be in flight at exit.
    const uint32_t issued = k;
    for (uint32_t s = 0; s < kSlots && s < issued; ++s) {
      const uint32_t last = issued - 1 - ((issued - 1 - s) % kSlots);  // last use of slot s
      if (!mbar_wait_bounded(bars + 8 * (last % kSlots), (last / kSlots) & 1)) timed_out = true;
    }
    if (timed_out) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
  }
}

// --------------------------------------------------------------------------------------------
// Consumer warp: one page (64 keys) against the item's 8 query rows.
// --------------------------------------------------------------------------------------------
struct WarpState {
  float o[8][4];   // O^T fragments: m-tile i -> dims 16g+i (c0,c1) and 16g+8+i (c2,c3)
  float m[2];      // running max (raw dot-product units) of rows 2t, 2t+1
  float l[2];      // per-thread partial sums of p for rows 2t, 2t+1
  uint32_t qf[8][2];  // Q B-fragments for k-steps 0..7
};

__device__ __forceinline__ void process_subtile(WarpState& st, uint32_t slot_addr, int sub, int kp0,
                                                int len, int lim0, int lim1, float c2, int g,
                                                int t) {
  const uint32_t kc = slot_addr + kKcOff, ks = slot_addr + kKsOff;
  const uint32_t vc = slot_addr + kVcOff, vs = slot_addr + kVsOff;

  // ---- scores S^T for keys 16*sub .. 16*sub+15 of the page ----
  float S[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int ka = 16 * sub + g, kb = ka + 8;
    const uint4 ca = lds128(kc + ka * 64 + 16 * t);
    const uint4 cb = lds128(kc + kb * 64 + 16 * t);
    uint32_t sa = lds16(ks + ka * 8 + 2 * t);
    uint32_t sb = lds16(ks + kb * 8 + 2 * t);
    if (kp0 + ka >= len) sa = 0;  // keys past the end may hold stale bytes: force them to 0
    if (kp0 + kb >= len) sb = 0;
    const uint32_t sah = cvt_e4m3x2_f16(sa), sbh = cvt_e4m3x2_f16(sb);
    const uint32_t sa0 = dup_lo(sah), sa1 = dup_hi(sah);
    const uint32_t sb0 = dup_lo(sbh), sb1 = dup_hi(sbh);
    const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w};
    const uint32_t wb[4] = {cb.x, cb.y, cb.z, cb.w};
    // two independent accumulators (even / odd k-steps) halve the MMA dependency chain
    float c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      cvt_e2m1x8_f16(wa[w], a0, a1, a2, a3);
      cvt_e2m1x8_f16(wb[w], b0, b1, b2, b3);
      const uint32_t sA = (w < 2) ? sa0 : sa1;  // bytes 0..7 of the 16 -> block 2t, 8..15 -> 2t+1
      const uint32_t sB = (w < 2) ? sb0 : sb1;
      // step s = 2w uses bytes (0,1) of word w, step 2w+1 bytes (2,3)
      mma_f16_16816(S, hmul2(a0, sA), hmul2(b0, sB), hmul2(a1, sA), hmul2(b1, sB),
                    st.qf[2 * w][0], st.qf[2 * w][1]);
      mma_f16_16816(c1, hmul2(a2, sA), hmul2(b2, sB), hmul2(a3, sA), hmul2(b3, sB),
                    st.qf[2 * w + 1][0], st.qf[2 * w + 1][1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) S[e] += c1[e];
  }

  // ---- online softmax over these 16 keys ----
  const int kpa = kp0 + 16 * sub + g, kpb = kpa + 8;
  float mx0 = -INFINITY, mx1 = -INFINITY;
  if (kpa <= lim0) mx0 = S[0];
  if (kpa <= lim1) mx1 = S[1];
  if (kpb <= lim0) mx0 = fmaxf(mx0, S[2]);
  if (kpb <= lim1) mx1 = fmaxf(mx1, S[3]);
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, m));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, m));
  }
  if (mx0 > st.m[0]) {
    const float alpha = (st.m[0] == -INFINITY) ? 0.f : fast_exp2((st.m[0] - mx0) * c2);
#pragma unroll
    for (int i = 0; i < 8; ++i) { st.o[i][0] *= alpha; st.o[i][2] *= alpha; }
    st.l[0] *= alpha;
    st.m[0] = mx0;
  }
  if (mx1 > st.m[1]) {
    const float alpha = (st.m[1] == -INFINITY) ? 0.f : fast_exp2((st.m[1] - mx1) * c2);
#pragma unroll
    for (int i = 0; i < 8; ++i) { st.o[i][1] *= alpha; st.o[i][3] *= alpha; }
    st.l[1] *= alpha;
    st.m[1] = mx1;
  }
  const float p0 = (kpa <= lim0) ? fast_exp2((S[0] - st.m[0]) * c2) : 0.f;
  const float p1 = (kpa <= lim1) ? fast_exp2((S[1] - st.m[1]) * c2) : 0.f;
  const float p2 = (kpb <= lim0) ? fast_exp2((S[2] - st.m[0]) * c2) : 0.f;
  const float p3 = (kpb <= lim1) ? fast_exp2((S[3] - st.m[1]) * c2) : 0.f;
  st.l[0] += p0 + p2;
  st.l[1] += p1 + p3;
  // P as f16 hi + lo, transposed into the B layout (keys along k)
  const uint32_t h01 = pack_f16x2(p0, p1);
  const uint32_t h23 = pack_f16x2(p2, p3);
  const uint32_t l01 = pack_f16x2(p0 - f16_lo_to_f32(h01), p1 - f16_hi_to_f32(h01));
  const uint32_t l23 = pack_f16x2(p2 - f16_lo_to_f32(h23), p3 - f16_hi_to_f32(h23));
  const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
  const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);

  // ---- V^T fragments: keys (2t, 2t+1) and (2t+8, 2t+9) of the sub-tile, dims of block g ----
  const int v0 = 16 * sub + 2 * t;
  const uint2 w0 = lds64(vc + v0 * 64 + 8 * g);
  const uint2 w1 = lds64(vc + (v0 + 1) * 64 + 8 * g);
  const uint2 w2 = lds64(vc + (v0 + 8) * 64 + 8 * g);
  const uint2 w3 = lds64(vc + (v0 + 9) * 64 + 8 * g);
  uint32_t s0 = lds8(vs + v0 * 8 + g), s1 = lds8(vs + (v0 + 1) * 8 + g);
  uint32_t s2 = lds8(vs + (v0 + 8) * 8 + g), s3 = lds8(vs + (v0 + 9) * 8 + g);
  if (kp0 + v0 >= len) s0 = 0;
  if (kp0 + v0 + 1 >= len) s1 = 0;
  if (kp0 + v0 + 8 >= len) s2 = 0;
  if (kp0 + v0 + 9 >= len) s3 = 0;
  const uint32_t sp01 = cvt_e4m3x2_f16(s0 | (s1 << 8));
  const uint32_t sp23 = cvt_e4m3x2_f16(s2 | (s3 << 8));
  // interleave the nibbles of two keys: byte k of `e` = (dim 2k of key b) << 4 | (dim 2k of
  // key a); `o` likewise for dim 2k+1
  const uint32_t e0 = (w0.x & 0x0F0F0F0Fu) | ((w1.x & 0x0F0F0F0Fu) << 4);
  const uint32_t o0 = ((w0.x >> 4) & 0x0F0F0F0Fu) | (w1.x & 0xF0F0F0F0u);
  const uint32_t e1 = (w0.y & 0x0F0F0F0Fu) | ((w1.y & 0x0F0F0F0Fu) << 4);
  const uint32_t o1 = ((w0.y >> 4) & 0x0F0F0F0Fu) | (w1.y & 0xF0F0F0F0u);
  const uint32_t e2 = (w2.x & 0x0F0F0F0Fu) | ((w3.x & 0x0F0F0F0Fu) << 4);
  const uint32_t o2 = ((w2.x >> 4) & 0x0F0F0F0Fu) | (w3.x & 0xF0F0F0F0u);
  const uint32_t e3 = (w2.y & 0x0F0F0F0Fu) | ((w3.y & 0x0F0F0F0Fu) << 4);
  const uint32_t o3 = ((w2.y >> 4) & 0x0F0F0F0Fu) | (w3.y & 0xF0F0F0F0u);
  // D01[j] = (Vhat[key v0][16g+j], Vhat[key v0+1][16g+j]) for j = 0..15, likewise D23
  uint32_t D01[16], D23[16];
  cvt_e2m1x8_f16(e0, D01[0], D01[2], D01[4], D01[6]);
  cvt_e2m1x8_f16(o0, D01[1], D01[3], D01[5], D01[7]);
  cvt_e2m1x8_f16(e1, D01[8], D01[10], D01[12], D01[14]);
  cvt_e2m1x8_f16(o1, D01[9], D01[11], D01[13], D01[15]);
  cvt_e2m1x8_f16(e2, D23[0], D23[2], D23[4], D23[6]);
  cvt_e2m1x8_f16(o2, D23[1], D23[3], D23[5], D23[7]);
  cvt_e2m1x8_f16(e3, D23[8], D23[10], D23[12], D23[14]);
  cvt_e2m1x8_f16(o3, D23[9], D23[11], D23[13], D23[15]);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a0 = hmul2(D01[i], sp01), a1 = hmul2(D01[8 + i], sp01);
    const uint32_t a2 = hmul2(D23[i], sp23), a3 = hmul2(D23[8 + i], sp23);
    mma_f16_16816(st.o[i], a0, a1, a2, a3, bh0, bh1);
    mma_f16_16816(st.o[i], a0, a1, a2, a3, bl0, bl1);
  }
}

__device__ __forceinline__ void store_out(const DecodeParams& p, int seq, int kvh, int r, int dim,
                                          float v) {
  const int tok = r / p.G, hq = kvh * p.G + r % p.G;
  p.out[(((int64_t)seq * p.q_len + tok) * p.Hq + hq) * 128 + dim] = v;
}

__device__ void consumer(const DecodeParams& p, uint8_t* smem, int warp, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = smem_u32(smem + kBarOff);
  const volatile int32_t* slot_pid = reinterpret_cast<const volatile int32_t*>(smem + kSlotPidOff);
  float* mrg = reinterpret_cast<float*>(smem + kMergeOff);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + kFlagOff);
  const int ctid = warp * 32 + lane;  // consumer thread index
  const int rows_total = p.G * p.q_len;
  uint32_t kbase = 0;
  bool timed_out = false;
  const int s_begin = p.cta_seg[blockIdx.x], s_end = p.cta_seg[blockIdx.x + 1];

  for (int s = s_begin; s < s_end; ++s) {
    const int4 seg = p.segments[s];
    const int4 g0 = p.groups[2 * seg.x];
    const int4 g1 = p.groups[2 * seg.x + 1];
    const int seq = g0.x, kvh = g0.y, rg = g0.z, len = g0.w;
    const int n_seg = g1.x, first_part = g1.y;
    const int row0 = rg * kRows;
    const int L0 = len - p.q_len;
    // visibility limit (largest visible key position) of rows 2t, 2t+1; -1 for padding rows
    int lim[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = row0 + 2 * t + e;
      lim[e] = (r < rows_total) ? (p.causal ? L0 + r / p.G : len - 1) : -1;
    }
    WarpState st;
#pragma unroll
    for (int i = 0; i < 8; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
    {
      // Q fragments of row g: dims 32t + 4s + {0,1} and + {2,3} for k-step s
      const int r = row0 + g;
      uint4 qc = make_uint4(0u, 0u, 0u, 0u);
      uint32_t qs = 0;
      if (r < rows_total) {
        const int tok = r / p.G, hq = kvh * p.G + r % p.G;
        const int64_t qrow = ((int64_t)seq * p.q_len + tok) * p.Hq + hq;
        qc = *reinterpret_cast<const uint4*>(p.q_codes + qrow * 64 + 16 * t);
        qs = *reinterpret_cast<const uint16_t*>(p.q_scales + qrow * 8 + 2 * t);
      }
      const uint32_t sh = cvt_e4m3x2_f16(qs);
      const uint32_t s0 = dup_lo(sh), s1 = dup_hi(sh);
      const uint32_t wq[4] = {qc.x, qc.y, qc.z, qc.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t a0, a1, a2, a3;
        cvt_e2m1x8_f16(wq[w], a0, a1, a2, a3);
        const uint32_t sc = (w < 2) ? s0 : s1;
        st.qf[2 * w][0] = hmul2(a0, sc);
        st.qf[2 * w][1] = hmul2(a1, sc);
        st.qf[2 * w + 1][0] = hmul2(a2, sc);
        st.qf[2 * w + 1][1] = hmul2(a3, sc);
      }
    }
    // pages of this segment: warp group q = warp / 4 takes pages q, q + kGroups, ...; the four
    // warps of a group split each page into four 16-key sub-tiles
    const int n_pages = seg.z - seg.y;
    const int grp = warp >> 2, sub = warp & 3;
    for (int j = grp; j < n_pages; j += kGroups) {
      const uint32_t k = kbase + j;
      const uint32_t slot = k % kSlots;
      if (!mbar_wait_bounded(bars + 8 * slot, (k / kSlots) & 1)) timed_out = true;
      if (slot_pid[slot] >= 0) {
        const int kp0 = (seg.y + j) * kPage;
        process_subtile(st, ring + slot * kSlotBytes, sub, kp0, len, lim[0], lim[1], p.c2, g, t);
      } else if (lane == 0 && sub == 0) {
        flag_status(p.status, KV_NVFP4_DEV_BAD_PAGE);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * (kSlots + slot));
    }
    kbase += n_pages;

    // ---- merge the consumer warps' states in shared memory ----
    float l0 = st.l[0], l1 = st.l[1];
#pragma unroll
    for (int m = 4; m < 32; m <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, m);
      l1 += __shfl_xor_sync(0xffffffffu, l1, m);
    }
    float* Ow = mrg + warp * kPartFloats;  // [dim][8 rows], then m[8], l[8]
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int dA = 16 * g + i, dB = dA + 8;
      *reinterpret_cast<float2*>(Ow + dA * kRows + 2 * t) = make_float2(st.o[i][0], st.o[i][1]);
      *reinterpret_cast<float2*>(Ow + dB * kRows + 2 * t) = make_float2(st.o[i][2], st.o[i][3]);
    }
    if (g == 0) {
      Ow[kRows * 128 + 2 * t] = st.m[0];
      Ow[kRows * 128 + 2 * t + 1] = st.m[1];
      Ow[kRows * 128 + kRows + 2 * t] = l0;
      Ow[kRows * 128 + kRows + 2 * t + 1] = l1;
    }
    named_barrier_sync(1, kConsumerWarps * 32);

    const bool split = n_seg > 1;
    float* part = split ? p.partials + (int64_t)seg.w * kPartFloats : nullptr;
    for (int idx = ctid; idx < kRows * 128; idx += kConsumerWarps * 32) {  // (row, dim)
      const int row = idx >> 7, dim = idx & 127;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mrg[w * kPartFloats + kRows * 128 + row]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float* base = mrg + w * kPartFloats;
          const float mw = base[kRows * 128 + row];
          const float f = (mw == -INFINITY) ? 0.f : fast_exp2((mw - M) * p.c2);
          L += f * base[kRows * 128 + kRows + row];
          O += f * base[dim * kRows + row];
        }
      }
      const int r = row0 + row;
      if (split) {
        part[row * 128 + dim] = O;
        if (dim == 0) {
          part[kRows * 128 + row] = M;
          part[kRows * 128 + kRows + row] = L;
        }
      } else if (r < rows_total && L > 0.f) {
        store_out(p, seq, kvh, r, dim, O / L);
      }
    }
    if (split) {
      // ---- ticket: the CTA that finishes the group's last segment combines all partials ----
      __threadfence();  // this thread's partial writes, visible device-wide before the ticket
      named_barrier_sync(1, kConsumerWarps * 32);
      if (ctid == 0) {
        __threadfence();
        int32_t* ctr = p.counters + seg.x;
        const int ticket = atomicAdd(ctr, 1);
        const int last = (ticket == n_seg - 1);
        if (last) *ctr = 0;  // ready for the next call on this workspace
        *flag = last;
      }
      named_barrier_sync(1, kConsumerWarps * 32);
      if (*flag) {
        __threadfence();
        const float* pb = p.partials + (int64_t)first_part * kPartFloats;
        for (int idx = ctid; idx < kRows * 128; idx += kConsumerWarps * 32) {
          const int row = idx >> 7, dim = idx & 127;
          const int r = row0 + row;
          if (r >= rows_total) continue;
          float M = -INFINITY;
          for (int c = 0; c < n_seg; ++c) M = fmaxf(M, __ldcg(pb + c * kPartFloats + kRows * 128 + row));
          float L = 0.f, O = 0.f;
          for (int c = 0; c < n_seg; ++c) {
            const float* q = pb + c * kPartFloats;
            const float mc = __ldcg(q + kRows * 128 + row);
            const float f = (mc == -INFINITY) ? 0.f : fast_exp2((mc - M) * p.c2);
            L += f * __ldcg(q + kRows * 128 + kRows + row);
            O += f * __ldcg(q + row * 128 + dim);
          }
          if (L > 0.f) store_out(p, seq, kvh, r, dim, O / L);
        }
      }
    }
    named_barrier_sync(1, kConsumerWarps * 32);  // merge area reused by the next segment
  }
  if (timed_out && lane == 0) flag_status(p.status, KV_NVFP4_DEV_TIMEOUT);
}

__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    const uint32_t bars = smem_u32(smem + kBarOff);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bars + 8 * s, 1);
      mbar_init(bars + 8 * (kSlots + s), 4);  // released by the page's four warps
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kConsumerWarps) {
    producer(p, smem, lane);
    return;
  }
  consumer(p, smem, warp, lane);
}

}  // namespace

int decode_smem_bytes() { return kSmemBytes; }

cudaError_t launch_decode(const uint8_t* q_codes, const uint8_t* q_scales, const uint8_t* k_codes,
                          const uint8_t* k_scales, const uint8_t* v_codes,
                          const uint8_t* v_scales, const int32_t* block_table, int32_t max_pages,
                          int32_t num_pages, const void* groups, const void* segments,
                          const int32_t* cta_seg, int32_t* counters, float* partials, float* out,
                          int32_t* status, int32_t Hq, int32_t Hkv, int32_t q_len, int32_t causal,
                          int32_t grid, float sm_scale, cudaStream_t stream) {
  static bool attr_done = false;  // the attribute belongs to the function, set once per process
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  DecodeParams p;
  p.q_codes = q_codes; p.q_scales = q_scales;
  p.k_codes = k_codes; p.k_scales = k_scales; p.v_codes = v_codes; p.v_scales = v_scales;
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
