// C ABI of the NVFP4 KV-cache library: argument validation, the RoPE table, the split-K plan,
// and the kernel launches. Declarations and contracts are in include/kv_nvfp4.h.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "kv_nvfp4.h"

namespace kvnvfp4 {
cudaError_t launch_append(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* seq_ids, const int32_t* positions, int64_t T,
                          const float* rope, int32_t rope_max_pos, int32_t rot_dim,
                          const int32_t* block_table, int32_t num_seqs, int32_t max_pages,
                          int32_t num_pages, uint8_t* pool, uint8_t* q_codes,
                          uint8_t* q_scales, int32_t Hq, int32_t Hkv, int32_t* status,
                          int32_t num_sms, cudaStream_t stream);
cudaError_t launch_decode(const uint8_t* q_codes, const uint8_t* q_scales, const uint8_t* pool,
                          const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                          const void* groups, const void* segments, const int32_t* cta_seg,
                          const int32_t* split_groups, int32_t num_split, float* partials,
                          float* out, int32_t* status,
                          int32_t Hq, int32_t Hkv, int32_t q_len, int32_t causal, int32_t grid,
                          float sm_scale, const uint16_t* q_new, const uint16_t* k_new,
                          const uint16_t* v_new, const float* rope, int32_t rope_max_pos,
                          int32_t rot_dim, uint8_t* pool_w, uint8_t* q_codes_out,
                          uint8_t* q_scales_out, bool late_tables, cudaStream_t stream);
int cmp_chunk_bytes(int fmt);
cudaError_t launch_cmp_append(int fmt, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                              const int32_t* seq_ids, const int32_t* positions, int64_t T,
                              const float* rope, int32_t rope_max_pos, int32_t rot_dim,
                              const int32_t* block_table, int32_t num_seqs, int32_t max_pages,
                              int32_t num_pages, uint8_t* pool, uint16_t* q_out, int32_t Hq,
                              int32_t Hkv, int32_t* status, cudaStream_t stream);
cudaError_t launch_cmp_decode(int fmt, const uint16_t* q, const uint8_t* pool,
                              const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                              const void* groups, const void* segments, const int32_t* cta_seg,
                              const int32_t* split_groups, int32_t num_split, float* partials,
                              float* out, int32_t* status, int32_t Hq, int32_t Hkv, int32_t q_len,
                              int32_t causal, float sm_scale, int32_t grid, cudaStream_t stream);
cudaError_t launch_tile(const uint8_t* q_codes, const uint8_t* q_scales, const uint8_t* pool,
                        const int32_t* block_table, int32_t max_pages, int32_t num_pages,
                        const void* groups, const void* segments, const int32_t* cta_seg,
                        const int32_t* split_groups, int32_t num_split, float* partials,
                        float* out, int32_t* status, int32_t Hq, int32_t Hkv, int32_t q_len,
                        int32_t causal, int32_t grid, float sm_scale, cudaStream_t stream);
cudaError_t launch_page_copy(bool spill, const uint8_t* src, uint8_t* dst, const int32_t* ids,
                             int32_t n, int32_t num_pages, uint32_t page_bytes, int sms,
                             int32_t* status, cudaStream_t stream);
cudaError_t launch_step_inputs(const void* const src[3], void* const dst[3],
                               const uint32_t n16[3], const void* plan, uint32_t plan_bytes,
                               void* workspace, cudaStream_t stream);
int inline_plan_bytes();
}  // namespace kvnvfp4

namespace {

constexpr int kRowsPerItem = 8;   // query rows per KV head in one decode work group
constexpr int kPartHeadFloats = kRowsPerItem * 128 + 2 * kRowsPerItem;  // O[8][128], m[8], l[8]
// Tiles of more rows (speculative verify, prefill chunks) go to the tile kernel: groups of one
// KV head and 128 rows, one partial (O, m, l of the tile's rows) per segment.
constexpr int kTileRows = 128;
constexpr int kTailCharge = 2;    // extra pages charged for a decode group's last page
constexpr int kTileSegCharge = 10;  // pages charged for each segment of the tile kernel
constexpr int kTilePartFloats = kTileRows * 128 + 2 * kTileRows;

constexpr int kMaxAttnKvHeads = 4;  // the decode kernel stages every head of a page

// The attention kernel a (layout, q_len) pair runs on: more than 8 rows per KV head, or more KV
// heads than the decode kernel stages per page, -> the tile kernel (which works per KV head).
bool tile_mode(const kv_nvfp4_layout* L, int32_t q_len) {
  return (int64_t)(L->num_q_heads / L->num_kv_heads) * q_len > kRowsPerItem ||
         L->num_kv_heads > kMaxAttnKvHeads;
}
constexpr int kMaxGridForSizing = 1024;  // workspace sizing when no device is visible

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

kv_nvfp4_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return KV_NVFP4_OK;
  g_last_cuda_error = e;
  return KV_NVFP4_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int num_sms_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cached[64] = {0};
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// The split-K work list. Groups are (sequence, 8-row query tile) over every KV head for the
// decode kernel, or (sequence, KV head, 128-row tile) for the tile kernel, in that order; each
// group's visited pages are cut into chunks of chunk_pages, and the chunk stream of all groups is
// dealt out to `grid` CTAs in contiguous ranges of about total_pages / grid pages each. For the
// decode kernel a group's last page is charged kTailCharge pages more: in the fused decode step
// the CTA holding it also encodes and stores the step's new K/V rows (measured ~1-2 us, two
// pages' time), so it gets that many fewer pages. For the tile kernel each segment costs
// kTileSegCharge pages on top of its pages (its Q load, pipeline start and epilogue take ~5 us,
// about ten pages' time): a CTA whose range crosses a group boundary runs two segments, and with
// page-balanced ranges such CTAs ended ~7 us after the median one on the verify workload. The
// tile plan therefore takes the smallest per-CTA cost cap for which a greedy fill of the chunk
// stream needs at most `grid` CTAs (a binary search, each probe linear in the groups).
struct PlanBuild {
  kv_nvfp4_plan_info info;
  std::vector<int32_t> groups;    // 8 ints per group
  std::vector<int32_t> segments;  // 4 ints per segment
  std::vector<int32_t> cta_seg;   // grid + 1
  std::vector<int32_t> split;     // indices of the groups with more than one segment
};

// Greedy fill of the chunk stream (groups in order, each cut into chunks of chunk_pages, a
// group's last chunk possibly shorter) into CTAs of cost at most cap, a segment costing charge
// plus its pages. Returns the CTAs needed (INT64_MAX when one chunk and a charge exceed the cap);
// with `out` it also records the segments {group, lo, hi} and each CTA's first segment.
static int64_t tile_fill(const std::vector<int32_t>& gpages, int32_t chunk_pages, int64_t charge,
                         int64_t cap, std::vector<int32_t>* segs, std::vector<int32_t>* cta_first) {
  int64_t ctas = 1, used = 0;
  if (cta_first) cta_first->assign(1, 0);
  for (size_t gi = 0; gi < gpages.size(); ++gi) {
    const int32_t pages = gpages[gi];
    int32_t lo = 0;
    while (lo < pages) {
      const int64_t first = std::min<int64_t>(chunk_pages, pages - lo);
      if (used + charge + first > cap) {
        if (used == 0) return INT64_MAX;  // a chunk and its charge alone exceed the cap
        ++ctas;
        used = 0;
        if (cta_first) cta_first->push_back((int32_t)(segs->size() / 4));
      }
      used += charge;
      const int64_t room = cap - used;
      int64_t take = (int64_t)(pages - lo) <= room ? (int64_t)(pages - lo)
                                                  : room / chunk_pages * chunk_pages;
      if (take < first) take = first;
      const int32_t hi = lo + (int32_t)take;
      used += take;
      if (segs) {
        segs->push_back((int32_t)gi);
        segs->push_back(lo);
        segs->push_back(hi);
        segs->push_back(-1);
      }
      lo = hi;
      if (lo < pages) {  // the CTA is full: the group continues on the next one
        ++ctas;
        used = 0;
        if (cta_first) cta_first->push_back((int32_t)(segs->size() / 4));
      }
    }
  }
  return ctas;
}

kv_nvfp4_status plan_build(const kv_nvfp4_layout* L, const int32_t* h_seq_lens, int32_t num_seqs,
                           int32_t q_len, int32_t causal, int32_t chunk_tokens, int32_t num_sms,
                           bool tile, PlanBuild* pb) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return KV_NVFP4_EINVAL;
  if (h_seq_lens == nullptr || num_seqs <= 0 || q_len <= 0 || num_sms <= 0) return KV_NVFP4_EINVAL;
  if (chunk_tokens <= 0 || chunk_tokens % L->page_size != 0) return KV_NVFP4_EINVAL;
  const int32_t P = L->page_size;
  const int32_t G = L->num_q_heads / L->num_kv_heads;
  const int64_t rows = (int64_t)G * q_len;
  const int64_t tile_rows = tile ? kTileRows : kRowsPerItem;
  const int64_t n_rg = (rows + tile_rows - 1) / tile_rows;
  const int64_t n_pairs = tile ? L->num_kv_heads : 1;  // groups per (sequence, row tile)
  const int32_t chunk_pages = chunk_tokens / P;
  const int64_t n_groups = (int64_t)num_seqs * n_pairs * n_rg;
  if (n_groups > (1 << 26)) return KV_NVFP4_EINVAL;
  int64_t total_pages = 0, total_chunks = 0, total_tok = 0, max_len = 0;
  std::vector<int32_t> gpages((size_t)n_groups);
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t len = h_seq_lens[s];
    if (len < q_len || len < 1) return KV_NVFP4_EINVAL;
    total_tok += len;
    if (len > max_len) max_len = len;
    for (int64_t pr = 0; pr < n_pairs; ++pr)
      for (int64_t rg = 0; rg < n_rg; ++rg) {
        int64_t vis = len;  // keys any row of the tile can see
        if (causal) {
          const int64_t last_row = std::min<int64_t>(rows - 1, rg * tile_rows + tile_rows - 1);
          vis = (int64_t)(len - q_len) + last_row / G + 1;
        }
        const int64_t pages = (vis + P - 1) / P;
        gpages[(size_t)(((int64_t)s * n_pairs + pr) * n_rg + rg)] = (int32_t)pages;
        total_pages += pages;
        total_chunks += (pages + chunk_pages - 1) / chunk_pages;
      }
  }
  const int64_t grid = std::min<int64_t>(num_sms, total_chunks);
  const int64_t tail = tile ? 0 : kTailCharge;  // cost of a group's last page beyond one page
  const int64_t total_cost = total_pages + tail * n_groups;
  pb->groups.assign((size_t)n_groups * 8, 0);
  pb->segments.clear();
  pb->cta_seg.assign((size_t)grid + 1, 0);
  std::vector<int32_t> seg_count((size_t)n_groups, 0);
  if (tile) {
    // the smallest cost cap whose greedy fill needs at most `grid` CTAs
    const int64_t charge = kTileSegCharge;
    int64_t lo_cap = (total_pages + charge * grid + grid - 1) / grid;
    int64_t hi_cap = lo_cap;
    while (tile_fill(gpages, chunk_pages, charge, hi_cap, nullptr, nullptr) > grid) hi_cap *= 2;
    while (lo_cap < hi_cap) {
      const int64_t mid = lo_cap + (hi_cap - lo_cap) / 2;
      if (tile_fill(gpages, chunk_pages, charge, mid, nullptr, nullptr) <= grid) hi_cap = mid;
      else lo_cap = mid + 1;
    }
    std::vector<int32_t> first;
    tile_fill(gpages, chunk_pages, charge, hi_cap, &pb->segments, &first);
    for (size_t c = 0; c < first.size() && c <= (size_t)grid; ++c) pb->cta_seg[c] = first[c];
    const int32_t nseg_t = (int32_t)(pb->segments.size() / 4);
    for (size_t c = first.size(); c <= (size_t)grid; ++c) pb->cta_seg[c] = nseg_t;
    for (int32_t si = 0; si < nseg_t; ++si) seg_count[(size_t)pb->segments[(size_t)si * 4]] += 1;
  }
  // deal chunks to CTAs: CTA c closes once the pages dealt so far reach (c+1) * total / grid
  int64_t cta = 0, dealt = 0;
  for (int64_t gi = 0; !tile && gi < n_groups; ++gi) {
    const int32_t pages = gpages[(size_t)gi];
    int32_t lo = 0;
    while (lo < pages) {
      // extend this segment chunk by chunk while the CTA is below its quota
      int32_t hi = lo;
      while (hi < pages) {
        hi = std::min(pages, hi + chunk_pages);
        const int64_t quota = (cta + 1) * total_cost / grid;
        if (cta < grid - 1 && dealt + (hi - lo) + (hi == pages ? tail : 0) >= quota) break;
      }
      pb->segments.push_back((int32_t)gi);
      pb->segments.push_back(lo);
      pb->segments.push_back(hi);
      pb->segments.push_back(-1);
      seg_count[(size_t)gi] += 1;
      dealt += hi - lo + (hi == pages ? tail : 0);
      lo = hi;
      const int64_t quota = (cta + 1) * total_cost / grid;
      if (cta < grid - 1 && dealt >= quota) {
        ++cta;
        pb->cta_seg[(size_t)cta] = (int32_t)(pb->segments.size() / 4);
      }
    }
  }
  const int64_t n_seg = (int64_t)pb->segments.size() / 4;
  if (!tile)
    for (int64_t c = cta + 1; c <= grid; ++c) pb->cta_seg[(size_t)c] = (int32_t)n_seg;
  // partial slots, contiguous per group in segment order; the split groups, in group order, are
  // the work list of the merge launch
  int64_t parts = 0;
  std::vector<int32_t> first_part((size_t)n_groups, -1);
  for (int64_t si = 0; si < n_seg; ++si) {
    const int32_t gi = pb->segments[(size_t)si * 4];
    if (seg_count[(size_t)gi] > 1) {
      if (first_part[(size_t)gi] < 0) first_part[(size_t)gi] = (int32_t)parts;
      pb->segments[(size_t)si * 4 + 3] = (int32_t)parts++;
    }
  }
  pb->split.clear();
  for (int64_t gi = 0; gi < n_groups; ++gi)
    if (seg_count[(size_t)gi] > 1) pb->split.push_back((int32_t)gi);
  for (int64_t gi = 0; gi < n_groups; ++gi) {
    const int64_t rg = gi % n_rg, pr = (gi / n_rg) % n_pairs, s = gi / (n_rg * n_pairs);
    int32_t* g = &pb->groups[(size_t)gi * 8];
    g[0] = (int32_t)s; g[1] = (int32_t)pr; g[2] = (int32_t)rg; g[3] = h_seq_lens[s];
    g[4] = seg_count[(size_t)gi]; g[5] = first_part[(size_t)gi]; g[6] = gpages[(size_t)gi]; g[7] = 0;
  }
  kv_nvfp4_plan_info* info = &pb->info;
  std::memset(info, 0, sizeof(*info));
  info->num_seqs = num_seqs;
  info->q_len = q_len;
  info->causal = causal ? 1 : 0;
  info->chunk_pages = chunk_pages;
  info->num_kv_heads = L->num_kv_heads;
  info->num_row_groups = (int32_t)n_rg;
  info->num_groups = (int32_t)n_groups;
  info->num_segments = (int32_t)n_seg;
  info->num_partials = (int32_t)parts;
  info->num_split_groups = (int32_t)pb->split.size();
  info->grid = (int32_t)grid;
  info->max_seq_len = (int32_t)max_len;
  info->total_kv_tokens = total_tok;
  info->total_pages = total_pages;
  uint64_t off = 0;
  info->off_groups = off;
  off = align_up(off + 32ull * n_groups, 256);
  info->off_segments = off;
  off = align_up(off + 16ull * n_seg, 256);
  info->off_cta = off;
  off = align_up(off + 4ull * (grid + 1), 256);
  info->off_split = off;
  off = align_up(off + 4ull * pb->split.size(), 256);
  info->off_partials = off;
  const uint64_t part_floats =
      tile ? (uint64_t)kTilePartFloats : (uint64_t)kPartHeadFloats * L->num_kv_heads;
  off = align_up(off + 4ull * part_floats * parts, 256);
  info->workspace_bytes = off;
  return KV_NVFP4_OK;
}

// RoPE table on the host: [max_pos][rot_dim], cos then sin, angle (pos / pos_scale) * inv_freq.
void rope_fill(float* t, int32_t max_pos, int32_t rot_dim, double theta, double pos_scale) {
  const int half = rot_dim / 2;
  std::vector<double> inv_freq(half);
  for (int i = 0; i < half; ++i) inv_freq[i] = std::pow(theta, -(2.0 * i) / (double)rot_dim);
  for (int32_t p = 0; p < max_pos; ++p) {
    float* row = t + (int64_t)p * rot_dim;
    const double pp = (double)p / pos_scale;
    for (int i = 0; i < half; ++i) {
      const double a = pp * inv_freq[i];
      row[i] = (float)std::cos(a);
      row[half + i] = (float)std::sin(a);
    }
  }
}

}  // namespace

// ---- page spill / restore ----------------------------------------------------------------------
namespace {

// Build the plan for num_ctas CTAs and upload its tables (everything before the partials) into
// the device workspace with one copy on the stream.
// The host image of a plan's tables (groups, segments, per-CTA segment ranges, split-group list;
// everything before info.off_partials), as the workspace holds them.
std::vector<int32_t> plan_image(const PlanBuild& pb) {
  const kv_nvfp4_plan_info& pi = pb.info;
  std::vector<int32_t> host((size_t)(pi.off_partials / 4), 0);
  std::memcpy(host.data() + pi.off_groups / 4, pb.groups.data(), pb.groups.size() * 4);
  std::memcpy(host.data() + pi.off_segments / 4, pb.segments.data(), pb.segments.size() * 4);
  std::memcpy(host.data() + pi.off_cta / 4, pb.cta_seg.data(), pb.cta_seg.size() * 4);
  std::memcpy(host.data() + pi.off_split / 4, pb.split.data(), pb.split.size() * 4);
  return host;
}

// Build the plan for num_ctas CTAs and upload its tables (everything before the partials) into
// the device workspace with one copy on the stream.
kv_nvfp4_status plan_upload(const kv_nvfp4_layout* L, const int32_t* h_seq_lens, int32_t num_seqs,
                            int32_t q_len, int32_t causal, int32_t chunk_tokens, int num_ctas,
                            bool tile, void* d_workspace, size_t ws_bytes,
                            kv_nvfp4_plan_info* info, void* stream) {
  PlanBuild pb;
  const kv_nvfp4_status s =
      plan_build(L, h_seq_lens, num_seqs, q_len, causal, chunk_tokens, num_ctas, tile, &pb);
  if (s != KV_NVFP4_OK) return s;
  const kv_nvfp4_plan_info& pi = pb.info;
  if (ws_bytes < pi.workspace_bytes) return KV_NVFP4_ENOSPACE;
  const std::vector<int32_t> host = plan_image(pb);
  const cudaError_t e = cudaMemcpyAsync(d_workspace, host.data(), host.size() * 4,
                                        cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e);
  *info = pi;
  return KV_NVFP4_OK;
}

// Device address of page-locked host memory (its mapping into the GPU's address space), or null
// for any other kind of memory. Clears the error a failed query leaves behind.
const void* mapped_host_address(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Device address of an arena: page-locked host memory (its mapped device address) or device
// memory. Pageable host memory, which the GPU cannot address on every system, is refused.
kv_nvfp4_status arena_device_address(const void* arena, const void** dev) {
  cudaPointerAttributes a{};
  const cudaError_t e = cudaPointerGetAttributes(&a, arena);
  if (e != cudaSuccess) {
    cudaGetLastError();  // the query's error is not a launch error: do not leave it set
    return e == cudaErrorInvalidValue ? KV_NVFP4_EINVAL : cuda_status(e);
  }
  if (a.type == cudaMemoryTypeHost) {
    if (a.devicePointer == nullptr) return KV_NVFP4_EINVAL;
    *dev = a.devicePointer;
    return KV_NVFP4_OK;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *dev = arena;
    return KV_NVFP4_OK;
  }
  return KV_NVFP4_EINVAL;  // cudaMemoryTypeUnregistered: pageable host memory
}

kv_nvfp4_status page_copy(const kv_nvfp4_layout* L, bool spill, const uint8_t* pool,
                          int32_t num_pages, const int32_t* d_page_ids, int32_t n,
                          const uint8_t* arena, int32_t* d_status, void* stream) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || n < 0) return KV_NVFP4_EINVAL;
  if (n == 0) return KV_NVFP4_OK;
  if (!pool || !arena || !d_page_ids || num_pages <= 0 || !aligned16(pool) || !aligned16(arena))
    return KV_NVFP4_EINVAL;
  const void* arena_dev = nullptr;
  const kv_nvfp4_status s = arena_device_address(arena, &arena_dev);
  if (s != KV_NVFP4_OK) return s;
  const int sms = num_sms_current_device();
  if (sms <= 0) return cuda_status(cudaErrorNoDevice);
  const uint32_t pb = (uint32_t)kv_nvfp4_page_bytes(L);
  const uint8_t* a = static_cast<const uint8_t*>(arena_dev);
  return cuda_status(kvnvfp4::launch_page_copy(
      spill, spill ? pool : a, spill ? const_cast<uint8_t*>(a) : const_cast<uint8_t*>(pool),
      d_page_ids, n, num_pages, pb, sms, d_status, (cudaStream_t)stream));
}

}  // namespace

// The fused decode step; late_tables: the plan tables are written by a kernel of the same step
// (the merge reads them only after its wait).
static kv_nvfp4_status decode_step_impl(const kv_nvfp4_layout* L, const kv_nvfp4_plan_info* plan,
                                     void* d_workspace, const void* q, const void* k,
                                     const void* v, const float* d_rope_table,
                                     int32_t rope_max_pos, const int32_t* d_block_table,
                                     int32_t max_pages, int32_t num_pages, uint8_t* pool,
                                     uint8_t* q_codes_out, uint8_t* q_scales_out, float sm_scale,
                                     float* out, int32_t* d_status, bool late_tables,
                                     void* stream) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || plan == nullptr) return KV_NVFP4_EINVAL;
  if (L->num_kv_heads > kMaxAttnKvHeads) return KV_NVFP4_EINVAL;
  if (plan->num_kv_heads != L->num_kv_heads || plan->num_seqs <= 0 || plan->q_len <= 0 ||
      plan->grid <= 0)
    return KV_NVFP4_EINVAL;
  // one row tile per sequence: each new row is encoded and stored by exactly one CTA
  if ((int64_t)(L->num_q_heads / L->num_kv_heads) * plan->q_len > kRowsPerItem)
    return KV_NVFP4_EINVAL;
  if (!d_workspace || !q || !k || !v || !pool || !d_block_table || !out || num_pages <= 0 ||
      max_pages <= 0)
    return KV_NVFP4_EINVAL;
  if ((q_codes_out == nullptr) != (q_scales_out == nullptr)) return KV_NVFP4_EINVAL;
  if (q_codes_out != nullptr && !aligned16(q_codes_out)) return KV_NVFP4_EINVAL;
  if (L->rot_dim > 0 && (!d_rope_table || rope_max_pos <= 0 || !aligned16(d_rope_table)))
    return KV_NVFP4_EINVAL;
  if ((int64_t)plan->max_seq_len > (int64_t)max_pages * L->page_size) return KV_NVFP4_EINVAL;
  const void* ptrs[] = {d_workspace, q, k, v, pool, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return KV_NVFP4_EINVAL;
  if (!(sm_scale > 0.0f)) sm_scale = 1.0f / std::sqrt((float)L->head_dim);
  char* ws = (char*)d_workspace;
  const cudaError_t e = kvnvfp4::launch_decode(
      nullptr, nullptr, pool, d_block_table, max_pages, num_pages, ws + plan->off_groups,
      ws + plan->off_segments, (const int32_t*)(ws + plan->off_cta),
      (const int32_t*)(ws + plan->off_split), plan->num_split_groups,
      (float*)(ws + plan->off_partials), out, d_status,
      L->num_q_heads, L->num_kv_heads, plan->q_len, plan->causal, plan->grid, sm_scale,
      (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, d_rope_table, rope_max_pos,
      L->rot_dim, pool, q_codes_out, q_scales_out, late_tables, (cudaStream_t)stream);
  return cuda_status(e);
}



extern "C" {

const char* kv_nvfp4_status_string(kv_nvfp4_status s) {
  switch (s) {
    case KV_NVFP4_OK: return "ok";
    case KV_NVFP4_EINVAL: return "invalid argument";
    case KV_NVFP4_ECUDA: return "CUDA launch or copy failed";
    case KV_NVFP4_ENOSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int32_t kv_nvfp4_version(void) { return 10000; }

const char* kv_nvfp4_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

// ---- page spill / restore ----------------------------------------------------------------------
kv_nvfp4_status kv_nvfp4_spill_pages(const kv_nvfp4_layout* layout, const uint8_t* pool,
                                     int32_t num_pages, const int32_t* d_page_ids, int32_t n,
                                     uint8_t* arena, int32_t* d_status, void* stream) {
  return page_copy(layout, true, pool, num_pages, d_page_ids, n, arena, d_status, stream);
}

kv_nvfp4_status kv_nvfp4_restore_pages(const kv_nvfp4_layout* layout, const uint8_t* arena,
                                       const int32_t* d_page_ids, int32_t n, uint8_t* pool,
                                       int32_t num_pages, int32_t* d_status, void* stream) {
  return page_copy(layout, false, pool, num_pages, d_page_ids, n, arena, d_status, stream);
}

kv_nvfp4_status kv_nvfp4_layout_check(const kv_nvfp4_layout* L) {
  if (L == nullptr) return KV_NVFP4_EINVAL;
  if (L->head_dim != 128 || L->page_size != 64) return KV_NVFP4_EINVAL;
  if (L->num_kv_heads <= 0 || L->num_q_heads <= 0) return KV_NVFP4_EINVAL;
  if (L->num_q_heads % L->num_kv_heads != 0) return KV_NVFP4_EINVAL;
  if (L->num_q_heads > 4096) return KV_NVFP4_EINVAL;
  if (L->rot_dim < 0 || L->rot_dim > 128 || L->rot_dim % 8 != 0) return KV_NVFP4_EINVAL;
  return KV_NVFP4_OK;
}

size_t kv_nvfp4_page_bytes(const kv_nvfp4_layout* L) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return 0;
  return (size_t)L->page_size * 2 * (64 + 8) * (size_t)L->num_kv_heads;
}

kv_nvfp4_status kv_nvfp4_pool_bytes(const kv_nvfp4_layout* L, int32_t num_pages,
                                    size_t* bytes) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || num_pages < 0 || bytes == nullptr)
    return KV_NVFP4_EINVAL;
  *bytes = (size_t)num_pages * kv_nvfp4_page_bytes(L);
  return KV_NVFP4_OK;
}

size_t kv_nvfp4_rope_table_bytes(int32_t max_pos, int32_t rot_dim) {
  if (max_pos < 0 || rot_dim < 0) return 0;
  return (size_t)max_pos * (size_t)rot_dim * sizeof(float);
}

kv_nvfp4_status kv_nvfp4_rope_table_fill_host(float* h_table, int32_t max_pos, int32_t rot_dim,
                                              double theta, double pos_scale) {
  if (h_table == nullptr || max_pos <= 0 || rot_dim <= 0 || rot_dim % 8 != 0 || rot_dim > 128 ||
      !(theta > 0.0) || !(pos_scale > 0.0))
    return KV_NVFP4_EINVAL;
  rope_fill(h_table, max_pos, rot_dim, theta, pos_scale);
  return KV_NVFP4_OK;
}

kv_nvfp4_status kv_nvfp4_rope_table_init(float* d_table, int32_t max_pos, int32_t rot_dim,
                                         double theta, double pos_scale, void* stream) {
  if (d_table == nullptr || max_pos <= 0 || rot_dim <= 0 || rot_dim % 8 != 0 || rot_dim > 128 ||
      !(theta > 0.0) || !(pos_scale > 0.0) || !aligned16(d_table))
    return KV_NVFP4_EINVAL;
  std::vector<float> h((size_t)max_pos * rot_dim);
  rope_fill(h.data(), max_pos, rot_dim, theta, pos_scale);
  // pageable source: the runtime stages it before returning, so `h` may be freed afterwards
  cudaError_t e = cudaMemcpyAsync(d_table, h.data(), h.size() * sizeof(float),
                                  cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e);
  return KV_NVFP4_OK;
}

kv_nvfp4_status kv_nvfp4_append(const kv_nvfp4_layout* L, const void* q, const void* k,
                                const void* v, const int32_t* d_seq_ids,
                                const int32_t* d_positions, int32_t T, const float* d_rope_table,
                                int32_t rope_max_pos, const int32_t* d_block_table,
                                int32_t num_seqs, int32_t max_pages, int32_t num_pages,
                                uint8_t* pool, uint8_t* q_codes, uint8_t* q_scales,
                                int32_t* d_status, void* stream) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return KV_NVFP4_EINVAL;
  if (T < 0 || num_seqs <= 0 || max_pages <= 0 || num_pages <= 0) return KV_NVFP4_EINVAL;
  if (T == 0) return KV_NVFP4_OK;
  if (!k || !v || !d_seq_ids || !d_positions || !d_block_table || !pool) return KV_NVFP4_EINVAL;
  if (q && (!q_codes || !q_scales)) return KV_NVFP4_EINVAL;
  if (L->rot_dim > 0 && (!d_rope_table || rope_max_pos <= 0 || !aligned16(d_rope_table)))
    return KV_NVFP4_EINVAL;
  if (!aligned16(k) || !aligned16(v) || (q && !aligned16(q)) || !aligned16(pool))
    return KV_NVFP4_EINVAL;
  const cudaError_t e = kvnvfp4::launch_append(
      (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, d_seq_ids, d_positions, T,
      d_rope_table, rope_max_pos, L->rot_dim, d_block_table, num_seqs, max_pages, num_pages,
      pool, q_codes, q_scales, L->num_q_heads, L->num_kv_heads,
      d_status, num_sms_current_device(), (cudaStream_t)stream);
  return cuda_status(e);
}

kv_nvfp4_status kv_nvfp4_plan_workspace_bytes(const kv_nvfp4_layout* L, const int32_t* h_seq_lens,
                                              int32_t num_seqs, int32_t q_len, int32_t causal,
                                              int32_t chunk_tokens, size_t* bytes) {
  if (bytes == nullptr) return KV_NVFP4_EINVAL;
  int num_sms = num_sms_current_device();
  if (num_sms <= 0) num_sms = kMaxGridForSizing;  // no device: size for the largest grid
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return KV_NVFP4_EINVAL;
  PlanBuild pb;
  const kv_nvfp4_status s = plan_build(L, h_seq_lens, num_seqs, q_len, causal, chunk_tokens,
                                       num_sms, tile_mode(L, q_len), &pb);
  if (s != KV_NVFP4_OK) return s;
  *bytes = (size_t)pb.info.workspace_bytes;
  return KV_NVFP4_OK;
}

kv_nvfp4_status kv_nvfp4_plan_host(const kv_nvfp4_layout* L, const int32_t* h_seq_lens,
                                   int32_t num_seqs, int32_t q_len, int32_t causal,
                                   int32_t chunk_tokens, int32_t num_ctas, void* h_workspace,
                                   size_t ws_bytes, kv_nvfp4_plan_info* info) {
  if (info == nullptr || h_workspace == nullptr || num_ctas <= 0) return KV_NVFP4_EINVAL;
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return KV_NVFP4_EINVAL;
  PlanBuild pb;
  const kv_nvfp4_status s = plan_build(L, h_seq_lens, num_seqs, q_len, causal, chunk_tokens,
                                       num_ctas, tile_mode(L, q_len), &pb);
  if (s != KV_NVFP4_OK) return s;
  const kv_nvfp4_plan_info& pi = pb.info;
  if (ws_bytes < pi.workspace_bytes) return KV_NVFP4_ENOSPACE;
  char* h = (char*)h_workspace;
  std::memset(h, 0, (size_t)pi.off_partials);
  std::memcpy(h + pi.off_groups, pb.groups.data(), pb.groups.size() * 4);
  std::memcpy(h + pi.off_segments, pb.segments.data(), pb.segments.size() * 4);
  std::memcpy(h + pi.off_cta, pb.cta_seg.data(), pb.cta_seg.size() * 4);
  std::memcpy(h + pi.off_split, pb.split.data(), pb.split.size() * 4);
  *info = pi;
  return KV_NVFP4_OK;
}

kv_nvfp4_status kv_nvfp4_plan(const kv_nvfp4_layout* L, const int32_t* h_seq_lens,
                              int32_t num_seqs, int32_t q_len, int32_t causal,
                              int32_t chunk_tokens, void* d_workspace, size_t ws_bytes,
                              kv_nvfp4_plan_info* info, void* stream) {
  if (info == nullptr || d_workspace == nullptr || !aligned16(d_workspace)) return KV_NVFP4_EINVAL;
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return KV_NVFP4_EINVAL;
  const int num_sms = num_sms_current_device();
  if (num_sms <= 0) return cuda_status(cudaErrorNoDevice);
  return plan_upload(L, h_seq_lens, num_seqs, q_len, causal, chunk_tokens, num_sms,
                     tile_mode(L, q_len), d_workspace, ws_bytes, info, stream);
}

kv_nvfp4_status kv_nvfp4_decode_attn(const kv_nvfp4_layout* L, const kv_nvfp4_plan_info* plan,
                                     void* d_workspace, const uint8_t* q_codes,
                                     const uint8_t* q_scales, float sm_scale, const uint8_t* pool,
                                     int32_t num_pages, const int32_t* d_block_table,
                                     int32_t max_pages, float* out, int32_t* d_status,
                                     void* stream) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || plan == nullptr) return KV_NVFP4_EINVAL;
  if (plan->num_kv_heads != L->num_kv_heads || plan->num_seqs <= 0 || plan->q_len <= 0 ||
      plan->grid <= 0)
    return KV_NVFP4_EINVAL;
  if (!d_workspace || !q_codes || !q_scales || !pool || !d_block_table || !out ||
      num_pages <= 0 || max_pages <= 0)
    return KV_NVFP4_EINVAL;
  // every page index the work list touches must lie inside the block table's rows
  if ((int64_t)plan->max_seq_len > (int64_t)max_pages * L->page_size) return KV_NVFP4_EINVAL;
  const void* ptrs[] = {d_workspace, q_codes, q_scales, pool, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return KV_NVFP4_EINVAL;
  if (!(sm_scale > 0.0f)) sm_scale = 1.0f / std::sqrt((float)L->head_dim);
  // the plan's tiling must be the one this layout and q_len run on
  const bool tile = tile_mode(L, plan->q_len);
  const int64_t rows = (int64_t)(L->num_q_heads / L->num_kv_heads) * plan->q_len;
  const int64_t tile_rows = tile ? kTileRows : kRowsPerItem;
  if (plan->num_row_groups != (rows + tile_rows - 1) / tile_rows) return KV_NVFP4_EINVAL;
  char* ws = (char*)d_workspace;
  cudaError_t e;
  if (tile) {
    e = kvnvfp4::launch_tile(q_codes, q_scales, pool, d_block_table, max_pages, num_pages,
                             ws + plan->off_groups, ws + plan->off_segments,
                             (const int32_t*)(ws + plan->off_cta),
                             (const int32_t*)(ws + plan->off_split), plan->num_split_groups,
                             (float*)(ws + plan->off_partials), out, d_status, L->num_q_heads,
                             L->num_kv_heads, plan->q_len, plan->causal, plan->grid, sm_scale,
                             (cudaStream_t)stream);
  } else {
    e = kvnvfp4::launch_decode(
        q_codes, q_scales, pool, d_block_table, max_pages, num_pages, ws + plan->off_groups,
        ws + plan->off_segments, (const int32_t*)(ws + plan->off_cta),
        (const int32_t*)(ws + plan->off_split), plan->num_split_groups,
        (float*)(ws + plan->off_partials), out, d_status,
        L->num_q_heads, L->num_kv_heads, plan->q_len, plan->causal, plan->grid, sm_scale,
        nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, nullptr, nullptr, false,
        (cudaStream_t)stream);
  }
  return cuda_status(e);
}

kv_nvfp4_status kv_nvfp4_decode_step(const kv_nvfp4_layout* L, const kv_nvfp4_plan_info* plan,
                                     void* d_workspace, const void* q, const void* k,
                                     const void* v, const float* d_rope_table,
                                     int32_t rope_max_pos, const int32_t* d_block_table,
                                     int32_t max_pages, int32_t num_pages, uint8_t* pool,
                                     uint8_t* q_codes_out, uint8_t* q_scales_out, float sm_scale,
                                     float* out, int32_t* d_status, void* stream) {
  return decode_step_impl(L, plan, d_workspace, q, k, v, d_rope_table, rope_max_pos,
                          d_block_table, max_pages, num_pages, pool, q_codes_out, q_scales_out,
                          sm_scale, out, d_status, false, stream);
}

kv_nvfp4_status kv_nvfp4_decode_step_host(
    const kv_nvfp4_layout* L, const int32_t* h_seq_lens, int32_t num_seqs, int32_t q_len,
    int32_t causal, int32_t chunk_tokens, void* d_workspace, size_t ws_bytes, const void* h_q,
    const void* h_k, const void* h_v, void* d_q, void* d_k, void* d_v, const float* d_rope_table,
    int32_t rope_max_pos, const int32_t* d_block_table, int32_t max_pages, int32_t num_pages,
    uint8_t* pool, float sm_scale, float* d_out, float* h_out, int32_t* d_status,
    kv_nvfp4_plan_info* plan_out, void* stream) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || h_seq_lens == nullptr || num_seqs <= 0 ||
      q_len <= 0)
    return KV_NVFP4_EINVAL;
  if (!h_q || !h_k || !h_v || !d_q || !d_k || !d_v || !h_out || !d_out || !d_workspace ||
      !aligned16(d_workspace))
    return KV_NVFP4_EINVAL;
  // the same checks as the fused step, before anything is enqueued
  if (L->num_kv_heads > kMaxAttnKvHeads ||
      (int64_t)(L->num_q_heads / L->num_kv_heads) * q_len > kRowsPerItem)
    return KV_NVFP4_EINVAL;
  const int num_sms = num_sms_current_device();
  if (num_sms <= 0) return cuda_status(cudaErrorNoDevice);
  const cudaStream_t st = (cudaStream_t)stream;
  const size_t rows = (size_t)num_seqs * (size_t)q_len;
  const size_t qb = rows * (size_t)L->num_q_heads * 256, kb = rows * (size_t)L->num_kv_heads * 256;
  const size_t ob = rows * (size_t)L->num_q_heads * 128 * 4;
  PlanBuild pb;
  kv_nvfp4_status s = plan_build(L, h_seq_lens, num_seqs, q_len, causal, chunk_tokens, num_sms,
                                 false, &pb);
  if (s != KV_NVFP4_OK) return s;
  const kv_nvfp4_plan_info& info = pb.info;
  if (ws_bytes < info.workspace_bytes) return KV_NVFP4_ENOSPACE;
  const std::vector<int32_t> image = plan_image(pb);
  // Page-locked host buffers (16-byte aligned): the GPU reads the new rows and writes the output
  // over the host link itself, with no copy-engine operation in the step. Otherwise: copies.
  const void* mq = aligned16(h_q) ? mapped_host_address(h_q) : nullptr;
  const void* mk = aligned16(h_k) ? mapped_host_address(h_k) : nullptr;
  const void* mv = aligned16(h_v) ? mapped_host_address(h_v) : nullptr;
  const void* mo = aligned16(h_out) ? mapped_host_address(h_out) : nullptr;
  const bool zero_copy = mq && mk && mv && mo && aligned16(d_q) && aligned16(d_k) &&
                         aligned16(d_v) && qb / 16 <= 0xFFFFFFFFull;
  cudaError_t e = cudaSuccess;
  if (zero_copy) {
    const size_t img_bytes = image.size() * 4;
    const bool inline_plan = img_bytes <= (size_t)kvnvfp4::inline_plan_bytes();
    if (!inline_plan)
      e = cudaMemcpyAsync(d_workspace, image.data(), img_bytes, cudaMemcpyHostToDevice, st);
    const void* src[3] = {mq, mk, mv};
    void* dst[3] = {d_q, d_k, d_v};
    const uint32_t n16[3] = {(uint32_t)(qb / 16), (uint32_t)(kb / 16), (uint32_t)(kb / 16)};
    if (e == cudaSuccess)
      e = kvnvfp4::launch_step_inputs(src, dst, n16, inline_plan ? image.data() : nullptr,
                                      inline_plan ? (uint32_t)img_bytes : 0u, d_workspace, st);
    if (e != cudaSuccess) return cuda_status(e);
  } else {
    e = cudaMemcpyAsync(d_q, h_q, qb, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_k, h_k, kb, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_v, h_v, kb, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(d_workspace, image.data(), image.size() * 4, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  float* out = zero_copy ? static_cast<float*>(const_cast<void*>(mo)) : d_out;
  s = decode_step_impl(L, &info, d_workspace, d_q, d_k, d_v, d_rope_table, rope_max_pos,
                       d_block_table, max_pages, num_pages, pool, nullptr, nullptr, sm_scale, out,
                       d_status, zero_copy, stream);
  if (s != KV_NVFP4_OK) return s;
  if (!zero_copy) {
    e = cudaMemcpyAsync(h_out, d_out, ob, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (plan_out != nullptr) *plan_out = info;
  return KV_NVFP4_OK;
}

// ---- comparator formats -----------------------------------------------------------------------
size_t kv_cmp_page_bytes(const kv_nvfp4_layout* L, int32_t fmt) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || fmt < KV_CMP_BF16 || fmt > KV_CMP_K4V16) return 0;
  return (size_t)L->num_kv_heads * (size_t)kvnvfp4::cmp_chunk_bytes(fmt);
}

kv_nvfp4_status kv_cmp_append(const kv_nvfp4_layout* L, int32_t fmt, const void* q, const void* k,
                              const void* v, const int32_t* d_seq_ids, const int32_t* d_positions,
                              int32_t T, const float* d_rope_table, int32_t rope_max_pos,
                              const int32_t* d_block_table, int32_t num_seqs, int32_t max_pages,
                              int32_t num_pages, uint8_t* pool, void* q_out, int32_t* d_status,
                              void* stream) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || fmt < KV_CMP_BF16 || fmt > KV_CMP_K4V16)
    return KV_NVFP4_EINVAL;
  if (T < 0 || num_seqs <= 0 || max_pages <= 0 || num_pages <= 0) return KV_NVFP4_EINVAL;
  if (T == 0) return KV_NVFP4_OK;
  if (!k || !v || !d_seq_ids || !d_positions || !d_block_table || !pool) return KV_NVFP4_EINVAL;
  if (q && !q_out) return KV_NVFP4_EINVAL;
  if (L->rot_dim > 0 && (!d_rope_table || rope_max_pos <= 0 || !aligned16(d_rope_table)))
    return KV_NVFP4_EINVAL;
  if (!aligned16(k) || !aligned16(v) || (q && (!aligned16(q) || !aligned16(q_out))) ||
      !aligned16(pool))
    return KV_NVFP4_EINVAL;
  return cuda_status(kvnvfp4::launch_cmp_append(
      fmt, (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, d_seq_ids, d_positions, T,
      d_rope_table, rope_max_pos, L->rot_dim, d_block_table, num_seqs, max_pages, num_pages, pool,
      (uint16_t*)q_out, L->num_q_heads, L->num_kv_heads, d_status, (cudaStream_t)stream));
}

kv_nvfp4_status kv_cmp_plan_workspace_bytes(const kv_nvfp4_layout* L, const int32_t* h_seq_lens,
                                            int32_t num_seqs, int32_t q_len, int32_t causal,
                                            int32_t chunk_tokens, size_t* bytes) {
  if (bytes == nullptr || kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return KV_NVFP4_EINVAL;
  int num_sms = num_sms_current_device();
  if (num_sms <= 0) num_sms = kMaxGridForSizing;
  const int ctas = num_sms / L->num_kv_heads > 0 ? num_sms / L->num_kv_heads : 1;
  PlanBuild pb;
  const kv_nvfp4_status s =
      plan_build(L, h_seq_lens, num_seqs, q_len, causal, chunk_tokens, ctas, false, &pb);
  if (s != KV_NVFP4_OK) return s;
  *bytes = (size_t)pb.info.workspace_bytes;
  return KV_NVFP4_OK;
}

kv_nvfp4_status kv_cmp_plan(const kv_nvfp4_layout* L, const int32_t* h_seq_lens, int32_t num_seqs,
                            int32_t q_len, int32_t causal, int32_t chunk_tokens,
                            void* d_workspace, size_t ws_bytes, kv_nvfp4_plan_info* info,
                            void* stream) {
  if (info == nullptr || d_workspace == nullptr || !aligned16(d_workspace) ||
      kv_nvfp4_layout_check(L) != KV_NVFP4_OK)
    return KV_NVFP4_EINVAL;
  const int num_sms = num_sms_current_device();
  if (num_sms <= 0) return cuda_status(cudaErrorNoDevice);
  const int ctas = num_sms / L->num_kv_heads > 0 ? num_sms / L->num_kv_heads : 1;
  return plan_upload(L, h_seq_lens, num_seqs, q_len, causal, chunk_tokens, ctas, false,
                     d_workspace, ws_bytes, info, stream);
}

kv_nvfp4_status kv_cmp_decode_attn(const kv_nvfp4_layout* L, int32_t fmt,
                                   const kv_nvfp4_plan_info* plan, void* d_workspace,
                                   const void* q_rot, float sm_scale, const uint8_t* pool,
                                   int32_t num_pages, const int32_t* d_block_table,
                                   int32_t max_pages, float* out, int32_t* d_status,
                                   void* stream) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || plan == nullptr || fmt < KV_CMP_BF16 ||
      fmt > KV_CMP_K4V16)
    return KV_NVFP4_EINVAL;
  if (plan->num_kv_heads != L->num_kv_heads || plan->num_seqs <= 0 || plan->q_len <= 0 ||
      plan->grid <= 0 || L->num_kv_heads > 65535)
    return KV_NVFP4_EINVAL;
  if (!d_workspace || !q_rot || !pool || !d_block_table || !out || num_pages <= 0 ||
      max_pages <= 0)
    return KV_NVFP4_EINVAL;
  if ((int64_t)plan->max_seq_len > (int64_t)max_pages * L->page_size) return KV_NVFP4_EINVAL;
  const void* ptrs[] = {d_workspace, q_rot, pool, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return KV_NVFP4_EINVAL;
  if (!(sm_scale > 0.0f)) sm_scale = 1.0f / std::sqrt((float)L->head_dim);
  char* ws = (char*)d_workspace;
  return cuda_status(kvnvfp4::launch_cmp_decode(
      fmt, (const uint16_t*)q_rot, pool, d_block_table, max_pages, num_pages,
      ws + plan->off_groups, ws + plan->off_segments, (const int32_t*)(ws + plan->off_cta),
      (const int32_t*)(ws + plan->off_split), plan->num_split_groups,
      (float*)(ws + plan->off_partials), out, d_status, L->num_q_heads, L->num_kv_heads,
      plan->q_len, plan->causal, sm_scale, plan->grid, (cudaStream_t)stream));
}

}  // extern "C"
