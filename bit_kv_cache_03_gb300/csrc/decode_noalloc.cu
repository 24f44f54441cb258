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
//
// The work list is uploaded from host memory built by each call, so a call cannot be recorded
// into a CUDA graph (a replay would read whatever that host memory holds by then): while the
// stream is capturing, the call is refused before anything is enqueued.

#include <cstdint>
#include <memory>
#include <mutex>
#include <new>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kv_nvfp4.h"

namespace {

// Work list and partials of kv_nvfp4_decode_attn_noalloc. Every GPU that loads the library holds
// these KV_NVFP4_NOALLOC_SCRATCH_BYTES until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KV_NVFP4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// The buffer's device address, looked up once per device and context: after cudaDeviceReset the
// device gets a new primary context, the module is loaded again and the array moves, so an entry
// is only used while the context it was looked up in is still the current one.
struct ScratchEntry {
  CUcontext ctx;
  void* addr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point query (no link against libcuda).
CtxGetCurrentFn ctx_get_current() {
  static const CtxGetCurrentFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  return fn;
}

CUcontext current_context() {
  CUcontext c = nullptr;
  const CtxGetCurrentFn fn = ctx_get_current();
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the buffer on the current device. In host code the array's name is only a
// host-side stand-in, so the address is looked up (with the device current) on the first call in
// each context and kept for later calls in that context.
cudaError_t scratch_on_current_device(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const CUcontext ctx = current_context();
  ScratchEntry& ent = g_scratch[dev];
  if (ctx == nullptr || ent.addr == nullptr || ent.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    ent.addr = p;
    ent.ctx = current_context();  // the lookup makes the device's primary context current
  }
  *addr = ent.addr;
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
  // not into a graph: the upload below reads host memory that is gone once this call returns
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing((cudaStream_t)stream, &cap) != cudaSuccess) return KV_NVFP4_ECUDA;
  if (cap != cudaStreamCaptureStatusNone) return KV_NVFP4_EINVAL;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return KV_NVFP4_ECUDA;
  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return KV_NVFP4_ECUDA;
  // host image of the work list for this device's CTA count, then one copy into the buffer; the
  // source is pageable, so the runtime stages it before the copy call returns and the image is
  // freed on return (only its tables, below info.off_partials, are written and copied)
  const std::unique_ptr<uint8_t[]> image(new (std::nothrow) uint8_t[need]);
  if (!image) return KV_NVFP4_ENOSPACE;
  kv_nvfp4_plan_info info;
  s = kv_nvfp4_plan_host(layout, h_seq_lens, num_seqs, q_len, causal, chunk_tokens, sms,
                         image.get(), need, &info);
  if (s != KV_NVFP4_OK) return s;
  if (info.workspace_bytes > (uint64_t)KV_NVFP4_NOALLOC_SCRATCH_BYTES) return KV_NVFP4_ENOSPACE;
  if (cudaMemcpyAsync(scratch, image.get(), (size_t)info.off_partials, cudaMemcpyHostToDevice,
                      (cudaStream_t)stream) != cudaSuccess)
    return KV_NVFP4_ECUDA;
  return kv_nvfp4_decode_attn(layout, &info, scratch, q_codes, q_scales, sm_scale, pool, num_pages,
                              d_block_table, max_pages, out, d_status, stream);
}
