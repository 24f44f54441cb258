// C ABI of the NVFP4 KV-cache library: argument validation, the RoPE table, the split-K plan,
// and the kernel launches. Declarations and contracts are in include/kv_nvfp4.h.

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
                          int32_t num_pages, uint8_t* k_codes, uint8_t* k_scales,
                          uint8_t* v_codes, uint8_t* v_scales, uint8_t* q_codes,
                          uint8_t* q_scales, int32_t Hq, int32_t Hkv, int32_t* status,
                          cudaStream_t stream);
cudaError_t launch_decode(const uint8_t* q_codes, const uint8_t* q_scales, const uint8_t* k_codes,
                          const uint8_t* k_scales, const uint8_t* v_codes,
                          const uint8_t* v_scales, const int32_t* block_table, int32_t max_pages,
                          int32_t num_pages, const void* seqinfo, const void* items,
                          int32_t* counters, float* partials, float* out, int32_t* status,
                          int32_t Hq, int32_t Hkv, int32_t q_len, int32_t causal, int32_t n_rg,
                          int32_t total_items, float sm_scale, int num_sms, cudaStream_t stream);
}  // namespace kvnvfp4

namespace {

constexpr int kRowsPerItem = 8;   // query rows per decode work item
constexpr int kPartFloats = kRowsPerItem * 128 + 2 * kRowsPerItem;

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

// Layout of a plan workspace for the given lengths; also validates them.
kv_nvfp4_status plan_layout(const kv_nvfp4_layout* L, const int32_t* h_seq_lens, int32_t num_seqs,
                            int32_t q_len, int32_t chunk_tokens, kv_nvfp4_plan_info* info) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return KV_NVFP4_EINVAL;
  if (h_seq_lens == nullptr || num_seqs <= 0 || q_len <= 0) return KV_NVFP4_EINVAL;
  if (chunk_tokens <= 0 || chunk_tokens % L->page_size != 0) return KV_NVFP4_EINVAL;
  const int32_t G = L->num_q_heads / L->num_kv_heads;
  const int64_t rows = (int64_t)G * q_len;
  const int64_t n_rg = (rows + kRowsPerItem - 1) / kRowsPerItem;
  if (n_rg > (1 << 20)) return KV_NVFP4_EINVAL;
  const int32_t chunk_pages = chunk_tokens / L->page_size;
  int64_t chunks = 0, partials = 0, max_chunks = 0, total = 0, max_len = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t len = h_seq_lens[s];
    if (len < q_len || len < 1) return KV_NVFP4_EINVAL;
    const int64_t pages = (len + L->page_size - 1) / L->page_size;
    const int64_t nc = (pages + chunk_pages - 1) / chunk_pages;
    chunks += nc;
    if (nc > 1) partials += nc * L->num_kv_heads * n_rg;
    if (nc > max_chunks) max_chunks = nc;
    total += len;
    if (len > max_len) max_len = len;
  }
  if (chunks * L->num_kv_heads * n_rg > 0x7FFFFFFF || partials > 0x7FFFFFFF)
    return KV_NVFP4_EINVAL;
  std::memset(info, 0, sizeof(*info));
  info->num_seqs = num_seqs;
  info->q_len = q_len;
  info->chunk_pages = chunk_pages;
  info->num_chunks = (int32_t)chunks;
  info->num_row_groups = (int32_t)n_rg;
  info->num_kv_heads = L->num_kv_heads;
  info->num_partials = (int32_t)partials;
  info->max_chunks = (int32_t)max_chunks;
  info->total_kv_tokens = total;
  info->max_seq_len = (int32_t)max_len;
  uint64_t off = 0;
  info->off_seqinfo = off;
  off = align_up(off + 16ull * num_seqs, 256);
  info->off_items = off;
  off = align_up(off + 16ull * chunks, 256);
  info->off_counters = off;
  off = align_up(off + 4ull * num_seqs * L->num_kv_heads * n_rg, 256);
  info->off_partials = off;
  off = align_up(off + 4ull * kPartFloats * partials, 256);
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

kv_nvfp4_status kv_nvfp4_layout_check(const kv_nvfp4_layout* L) {
  if (L == nullptr) return KV_NVFP4_EINVAL;
  if (L->head_dim != 128 || L->page_size != 64) return KV_NVFP4_EINVAL;
  if (L->num_kv_heads <= 0 || L->num_q_heads <= 0) return KV_NVFP4_EINVAL;
  if (L->num_q_heads % L->num_kv_heads != 0) return KV_NVFP4_EINVAL;
  if (L->num_q_heads / L->num_kv_heads > 8) return KV_NVFP4_EINVAL;
  if (L->rot_dim < 0 || L->rot_dim > 128 || L->rot_dim % 8 != 0) return KV_NVFP4_EINVAL;
  return KV_NVFP4_OK;
}

size_t kv_nvfp4_page_bytes(const kv_nvfp4_layout* L) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return 0;
  return (size_t)L->page_size * 2 * (64 + 8) * (size_t)L->num_kv_heads;
}

kv_nvfp4_status kv_nvfp4_pool_plane_bytes(const kv_nvfp4_layout* L, int32_t num_pages,
                                          size_t* code_bytes, size_t* scale_bytes) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || num_pages < 0) return KV_NVFP4_EINVAL;
  const size_t slots = (size_t)num_pages * L->num_kv_heads * L->page_size;
  if (code_bytes) *code_bytes = slots * 64;
  if (scale_bytes) *scale_bytes = slots * 8;
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
  if (cudaMemcpyAsync(d_table, h.data(), h.size() * sizeof(float), cudaMemcpyHostToDevice,
                      (cudaStream_t)stream) != cudaSuccess)
    return KV_NVFP4_ECUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return KV_NVFP4_ECUDA;
  return KV_NVFP4_OK;
}

kv_nvfp4_status kv_nvfp4_append(const kv_nvfp4_layout* L, const void* q, const void* k,
                                const void* v, const int32_t* d_seq_ids,
                                const int32_t* d_positions, int32_t T, const float* d_rope_table,
                                int32_t rope_max_pos, const int32_t* d_block_table,
                                int32_t num_seqs, int32_t max_pages, int32_t num_pages,
                                uint8_t* k_codes, uint8_t* k_scales, uint8_t* v_codes,
                                uint8_t* v_scales, uint8_t* q_codes, uint8_t* q_scales,
                                int32_t* d_status, void* stream) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK) return KV_NVFP4_EINVAL;
  if (T < 0 || num_seqs <= 0 || max_pages <= 0 || num_pages <= 0) return KV_NVFP4_EINVAL;
  if (T == 0) return KV_NVFP4_OK;
  if (!k || !v || !d_seq_ids || !d_positions || !d_block_table || !k_codes || !k_scales ||
      !v_codes || !v_scales)
    return KV_NVFP4_EINVAL;
  if (q && (!q_codes || !q_scales)) return KV_NVFP4_EINVAL;
  if (L->rot_dim > 0 && (!d_rope_table || rope_max_pos <= 0 || !aligned16(d_rope_table)))
    return KV_NVFP4_EINVAL;
  if (!aligned16(k) || !aligned16(v) || (q && !aligned16(q))) return KV_NVFP4_EINVAL;
  const cudaError_t e = kvnvfp4::launch_append(
      (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, d_seq_ids, d_positions, T,
      d_rope_table, rope_max_pos, L->rot_dim, d_block_table, num_seqs, max_pages, num_pages,
      k_codes, k_scales, v_codes, v_scales, q_codes, q_scales, L->num_q_heads, L->num_kv_heads,
      d_status, (cudaStream_t)stream);
  return e == cudaSuccess ? KV_NVFP4_OK : KV_NVFP4_ECUDA;
}

kv_nvfp4_status kv_nvfp4_plan_workspace_bytes(const kv_nvfp4_layout* L, const int32_t* h_seq_lens,
                                              int32_t num_seqs, int32_t q_len,
                                              int32_t chunk_tokens, size_t* bytes) {
  if (bytes == nullptr) return KV_NVFP4_EINVAL;
  kv_nvfp4_plan_info info;
  const kv_nvfp4_status s = plan_layout(L, h_seq_lens, num_seqs, q_len, chunk_tokens, &info);
  if (s != KV_NVFP4_OK) return s;
  *bytes = (size_t)info.workspace_bytes;
  return KV_NVFP4_OK;
}

kv_nvfp4_status kv_nvfp4_plan(const kv_nvfp4_layout* L, const int32_t* h_seq_lens,
                              int32_t num_seqs, int32_t q_len, int32_t chunk_tokens,
                              void* d_workspace, size_t ws_bytes, kv_nvfp4_plan_info* info,
                              void* stream) {
  if (info == nullptr || d_workspace == nullptr || !aligned16(d_workspace)) return KV_NVFP4_EINVAL;
  kv_nvfp4_plan_info pi;
  const kv_nvfp4_status s = plan_layout(L, h_seq_lens, num_seqs, q_len, chunk_tokens, &pi);
  if (s != KV_NVFP4_OK) return s;
  if (ws_bytes < pi.workspace_bytes) return KV_NVFP4_ENOSPACE;
  // host image of the seqinfo + items region
  std::vector<int32_t> host((size_t)(pi.off_counters / 4), 0);
  int32_t* seqinfo = host.data() + pi.off_seqinfo / 4;
  int32_t* items = host.data() + pi.off_items / 4;
  int64_t ci = 0, part = 0;
  const int32_t P = L->page_size;
  for (int32_t sq = 0; sq < num_seqs; ++sq) {
    const int32_t len = h_seq_lens[sq];
    const int32_t pages = (len + P - 1) / P;
    const int32_t nc = (pages + pi.chunk_pages - 1) / pi.chunk_pages;
    seqinfo[4 * sq + 0] = len;
    seqinfo[4 * sq + 1] = nc;
    seqinfo[4 * sq + 2] = (int32_t)part;
    seqinfo[4 * sq + 3] = 0;
    if (nc > 1) part += (int64_t)nc * L->num_kv_heads * pi.num_row_groups;
    for (int32_t c = 0; c < nc; ++c, ++ci) {
      const int32_t pb = c * pi.chunk_pages;
      const int32_t np = (pages - pb < pi.chunk_pages) ? pages - pb : pi.chunk_pages;
      items[4 * ci + 0] = sq;
      items[4 * ci + 1] = pb;
      items[4 * ci + 2] = np;
      items[4 * ci + 3] = c;
    }
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(d_workspace, host.data(), host.size() * 4, cudaMemcpyHostToDevice, st) !=
      cudaSuccess)
    return KV_NVFP4_ECUDA;
  const size_t ctr_bytes = (size_t)(pi.off_partials - pi.off_counters);
  if (cudaMemsetAsync((char*)d_workspace + pi.off_counters, 0, ctr_bytes, st) != cudaSuccess)
    return KV_NVFP4_ECUDA;
  *info = pi;
  return KV_NVFP4_OK;
}

kv_nvfp4_status kv_nvfp4_decode_attn(const kv_nvfp4_layout* L, const kv_nvfp4_plan_info* plan,
                                     void* d_workspace, const uint8_t* q_codes,
                                     const uint8_t* q_scales, int32_t causal, float sm_scale,
                                     const uint8_t* k_codes, const uint8_t* k_scales,
                                     const uint8_t* v_codes, const uint8_t* v_scales,
                                     int32_t num_pages, const int32_t* d_block_table,
                                     int32_t max_pages, float* out, int32_t* d_status,
                                     void* stream) {
  if (kv_nvfp4_layout_check(L) != KV_NVFP4_OK || plan == nullptr) return KV_NVFP4_EINVAL;
  if (plan->num_kv_heads != L->num_kv_heads || plan->num_seqs <= 0 || plan->q_len <= 0)
    return KV_NVFP4_EINVAL;
  if (!d_workspace || !q_codes || !q_scales || !k_codes || !k_scales || !v_codes || !v_scales ||
      !d_block_table || !out || num_pages <= 0 || max_pages <= 0)
    return KV_NVFP4_EINVAL;
  // every page index the work list touches must lie inside the block table's rows
  if ((int64_t)plan->max_seq_len > (int64_t)max_pages * L->page_size) return KV_NVFP4_EINVAL;
  const void* ptrs[] = {d_workspace, q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return KV_NVFP4_EINVAL;
  const int num_sms = num_sms_current_device();
  if (num_sms <= 0) return KV_NVFP4_ECUDA;
  if (!(sm_scale > 0.0f)) sm_scale = 1.0f / std::sqrt((float)L->head_dim);
  char* ws = (char*)d_workspace;
  const int64_t total = (int64_t)plan->num_chunks * plan->num_kv_heads * plan->num_row_groups;
  const cudaError_t e = kvnvfp4::launch_decode(
      q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, d_block_table, max_pages,
      num_pages, ws + plan->off_seqinfo, ws + plan->off_items,
      (int32_t*)(ws + plan->off_counters), (float*)(ws + plan->off_partials), out, d_status,
      L->num_q_heads, L->num_kv_heads, plan->q_len, causal ? 1 : 0, plan->num_row_groups,
      (int32_t)total, sm_scale, num_sms, (cudaStream_t)stream);
  return e == cudaSuccess ? KV_NVFP4_OK : KV_NVFP4_ECUDA;
}

}  // extern "C"
