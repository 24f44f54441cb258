// Page spill and restore: whole page blocks copied between the pool (device memory) and an arena
// (page-locked host memory, reached by the GPU's own loads and stores over the host link, or
// device memory), following a device list of page ids.
//
// Source: prismix.dev/news/833001997676, section "Multi-level prefix reuse with host-KV safety
// net": cache pages moved out to host memory and restored from it. A page block holds every KV
// head's K and V codes and scales for its 64 slots, so a page moves as one contiguous block.
//
// One CTA per page at a time (grid-stride over the id list, a few CTAs per SM): the CTA reads the
// page id once, then its 256 threads move the page's 16-byte words, each thread issuing all of
// its loads before its stores, so that a whole 4-head page (36,864 B) is in flight per CTA. The
// copy is bound by the host link, not by HBM; no shared memory is involved.

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace kvnvfp4 {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kWordsPerThread = 9;  // 9 x 256 x 16 B = 36,864 B
constexpr int kCopyCtasPerSm = 4;

// kSpill: arena slot i <- pool page ids[i]; otherwise pool page ids[i] <- arena slot i.
template <bool kSpill>
__global__ void __launch_bounds__(kCopyThreads) page_copy_kernel(
    const uint4* __restrict__ src, uint4* __restrict__ dst, const int32_t* __restrict__ ids,
    int32_t n, int32_t num_pages, int32_t words, int32_t* status) {
  for (int32_t i = blockIdx.x; i < n; i += gridDim.x) {
    const int32_t id = ids[i];
    if (id < 0 || id >= num_pages) {  // uniform over the CTA: the page is skipped
      if (threadIdx.x == 0) flag_status(status, KV_NVFP4_DEV_BAD_PAGE);
      continue;
    }
    const uint4* s = src + (int64_t)(kSpill ? id : i) * words;
    uint4* d = dst + (int64_t)(kSpill ? i : id) * words;
    for (int32_t w0 = 0; w0 < words; w0 += kWordsPerThread * kCopyThreads) {
      uint4 v[kWordsPerThread];
#pragma unroll
      for (int j = 0; j < kWordsPerThread; ++j) {
        const int32_t w = w0 + j * kCopyThreads + (int32_t)threadIdx.x;
        if (w < words) v[j] = s[w];
      }
#pragma unroll
      for (int j = 0; j < kWordsPerThread; ++j) {
        const int32_t w = w0 + j * kCopyThreads + (int32_t)threadIdx.x;
        if (w < words) d[w] = v[j];
      }
    }
  }
}

}  // namespace

cudaError_t launch_page_copy(bool spill, const uint8_t* src, uint8_t* dst, const int32_t* ids,
                             int32_t n, int32_t num_pages, uint32_t page_bytes, int sms,
                             int32_t* status, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int grid = n < sms * kCopyCtasPerSm ? n : sms * kCopyCtasPerSm;
  const int32_t words = (int32_t)(page_bytes / 16u);
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  if (spill)
    page_copy_kernel<true><<<grid, kCopyThreads, 0, stream>>>(s, d, ids, n, num_pages, words,
                                                                status);
  else
    page_copy_kernel<false><<<grid, kCopyThreads, 0, stream>>>(s, d, ids, n, num_pages, words,
                                                                 status);
  return cudaGetLastError();
}

}  // namespace kvnvfp4
