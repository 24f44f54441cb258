// Inputs of a decode step taken straight from page-locked host memory.
//
// kv_nvfp4_decode_step_host drives one decode step from host buffers. When those buffers are
// page-locked (so the GPU can address them over the host link), no copy-engine operation is
// needed: this kernel reads the step's new Q/K/V rows from host memory into the caller's device
// buffers and writes the split-K work list, passed inline in its parameters, into the workspace;
// the attention and merge kernels that follow write the output rows straight into the host
// output buffer. The step is then a chain of three kernels, each launched as a programmatic
// dependent of the one before, with no copy operation between them to serialise on.

#include <cstdint>
#include <cuda_runtime.h>

namespace kvnvfp4 {

constexpr int kInlinePlanBytes = 8192;  // work lists up to this size travel in the parameters

namespace {

struct StepInputParams {
  const uint4* src[3];   // host-mapped q, k, v rows
  uint4* dst[3];         // the caller's device buffers
  uint32_t n16[3];       // 16-byte units of each
  uint32_t plan_n16;     // 16-byte units of the inline work list (0: none)
  uint4* plan_dst;       // workspace offset 0
  uint4 plan[kInlinePlanBytes / 16];
};

__global__ void __launch_bounds__(256) step_inputs_kernel(const __grid_constant__ StepInputParams p) {
  // the attention kernel of this step may be scheduled now; it waits for this grid to complete
  // before it reads the work list or the new rows
  asm volatile("griddepcontrol.launch_dependents;");
  const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t nt = gridDim.x * blockDim.x;
  // this thread's first unit of each buffer is read from host memory before the wait, so the
  // host-link latency overlaps the previous kernel's tail (the host wrote the rows before the call)
  uint4 first[3];
#pragma unroll
  for (int b = 0; b < 3; ++b)
    if (tid < p.n16[b]) first[b] = p.src[b][tid];
  // the previous kernel on the stream (the last step's attention or merge) reads the workspace
  // and the device row buffers: overwrite them only after it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (uint32_t i = tid; i < p.plan_n16; i += nt) p.plan_dst[i] = p.plan[i];
#pragma unroll
  for (int b = 0; b < 3; ++b) {
    if (tid < p.n16[b]) p.dst[b][tid] = first[b];
    for (uint32_t i = tid + nt; i < p.n16[b]; i += nt) p.dst[b][i] = p.src[b][i];
  }
}

}  // namespace

// Copies n16 16-byte units of q, k, v from host-mapped memory to device memory and, when
// plan_bytes > 0, the work-list image (at most kInlinePlanBytes, a multiple of 16) to
// workspace offset 0. One launch, a programmatic dependent of the previous kernel on the stream.
cudaError_t launch_step_inputs(const void* const src[3], void* const dst[3],
                               const uint32_t n16[3], const void* plan, uint32_t plan_bytes,
                               void* workspace, cudaStream_t stream) {
  if (plan_bytes > (uint32_t)kInlinePlanBytes || (plan_bytes & 15u) != 0) return cudaErrorInvalidValue;
  StepInputParams p;
  uint32_t total = plan_bytes / 16;
  for (int b = 0; b < 3; ++b) {
    p.src[b] = static_cast<const uint4*>(src[b]);
    p.dst[b] = static_cast<uint4*>(dst[b]);
    p.n16[b] = n16[b];
    total = total > n16[b] ? total : n16[b];
  }
  p.plan_n16 = plan_bytes / 16;
  p.plan_dst = static_cast<uint4*>(workspace);
  const uint4* pl = static_cast<const uint4*>(plan);
  for (uint32_t i = 0; i < p.plan_n16; ++i) p.plan[i] = pl[i];
  // one 16-byte unit per thread of the largest buffer (up to 256 KB): every load is in flight at
  // once, and before the wait
  uint32_t grid = (total + 255) / 256;
  grid = grid < 1 ? 1 : (grid > 64 ? 64 : grid);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_inputs_kernel, p);
}

int inline_plan_bytes() { return kInlinePlanBytes; }

}  // namespace kvnvfp4
