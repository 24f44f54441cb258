// Decode attention for callers that cannot allocate device memory.
//
// kv_nvfp4_decode_attn needs a workspace (the split-K work list and the (m, l, O) partials of the
// groups split over several CTAs) that the caller allocates. Some callers cannot do that: an
// inference engine that reserves all of the GPU's memory for its own arena at start-up and hands
// a layer only its input and output buffers, or a plug-in running under an allocator it does not
// control, where a cudaMalloc either fails or stalls every stream on the device while it runs.
// For them kv_nvfp4_decode_attn_noalloc keeps the workspace in a fixed buffer compiled into this
// library: the same plan and the same two kernels, with nothing allocated on the device.
//
// The buffer is shared by every call in the process, on every stream. Each call rewrites the
// tables it needs before its kernels read them, and every partial is written before it is
// merged, so nothing in it has to start at zero; but two calls whose kernels overlap on the GPU
// (different streams, or different host threads) overwrite each other's work list and partials.
// Such calls must be serialised by the caller.

#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "kv_nvfp4.h"

namespace {

// Work list and partials of kv_nvfp4_decode_attn_noalloc. Every GPU that loads the library holds
// these KV_NVFP4_NOALLOC_SCRATCH_BYTES until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KV_NVFP4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the buffer on the current device. In host code the array's name is only a
// host-side stand-in, so the address is looked up once per device (with that device current)
// and kept.
cudaError_t scratch_on_current_device(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kv_nvfp4_status kv_nvfp4_decode_attn_noalloc(
    const kv_nvfp4_layout* layout, const int32_t* h_seq_lens, int32_t num_seqs, int32_t q_len,
    int32_t causal, int32_t chunk_tokens, const uint8_t* q_codes, const uint8_t* q_scales,
    float sm_scale, const uint8_t* pool, int32_t num_pages, const int32_t* d_block_table,
    int32_t max_pages, float* out, int32_t* d_status, void* stream) {
  // the plan this call needs, checked against the fixed buffer before anything touches the GPU
  size_t need = 0;
  kv_nvfp4_status s = kv_nvfp4_plan_workspace_bytes(layout, h_seq_lens, num_seqs, q_len, causal,
                                                    chunk_tokens, &need);
  if (s != KV_NVFP4_OK) return s;
  if (need > (size_t)KV_NVFP4_NOALLOC_SCRATCH_BYTES) return KV_NVFP4_ENOSPACE;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return KV_NVFP4_ECUDA;
  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return KV_NVFP4_ECUDA;
  // host image of the work list for this device's CTA count, then one copy into the buffer (a
  // pageable source is staged by the runtime before the copy call returns)
  thread_local std::vector<uint8_t> image;
  image.resize(need);
  kv_nvfp4_plan_info info;
  s = kv_nvfp4_plan_host(layout, h_seq_lens, num_seqs, q_len, causal, chunk_tokens, sms,
                         image.data(), need, &info);
  if (s != KV_NVFP4_OK) return s;
  if (info.workspace_bytes > (uint64_t)KV_NVFP4_NOALLOC_SCRATCH_BYTES) return KV_NVFP4_ENOSPACE;
  if (cudaMemcpyAsync(scratch, image.data(), (size_t)info.off_partials, cudaMemcpyHostToDevice,
                      (cudaStream_t)stream) != cudaSuccess)
    return KV_NVFP4_ECUDA;
  return kv_nvfp4_decode_attn(layout, &info, scratch, q_codes, q_scales, sm_scale, pool, num_pages,
                              d_block_table, max_pages, out, d_status, stream);
}
