// stage.cu — copy of the query block from pinned host memory into the decode
// workspace, once per call.
//
// The decode kernel reads q in fragments: every CTA reads the query rows of its
// heads, in 4-byte pieces.  From device memory that is cheap; from pinned host
// memory it is ~150 CTAs x the whole block in small reads over the host link,
// which measured 10 us a 32K batch-1 call.  When q is host memory, this kernel
// copies it once (16-byte loads) into the workspace and the decode reads that
// copy.  It is launched as a programmatic dependent: it reads the host block
// while the preceding kernel is still running, and writes the copy only after
// that kernel has completed (an earlier call's decode may still read the copy).
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kStageThreads = 256;
constexpr int kStageUnroll = 4;  // 16-byte loads in flight a thread

__global__ void __launch_bounds__(kStageThreads) q_stage_kernel(const uint4* src, uint4* dst, size_t n16) {
  // the decode that follows may be scheduled now; it waits for this grid before reading q
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t i0 = (size_t)blockIdx.x * kStageThreads * kStageUnroll + threadIdx.x;
  uint4 v[kStageUnroll];
#pragma unroll
  for (int u = 0; u < kStageUnroll; ++u) {
    const size_t i = i0 + (size_t)u * kStageThreads;
    v[u] = i < n16 ? src[i] : make_uint4(0, 0, 0, 0);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
  for (int u = 0; u < kStageUnroll; ++u) {
    const size_t i = i0 + (size_t)u * kStageThreads;
    if (i < n16) dst[i] = v[u];
  }
}

}  // namespace

cudaError_t launch_q_stage(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  const size_t per_cta = (size_t)kStageThreads * kStageUnroll;
  const size_t grid = (n16 + per_cta - 1) / per_cta;
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kStageThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, q_stage_kernel, reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst),
                            n16);
}

}  // namespace kvq
