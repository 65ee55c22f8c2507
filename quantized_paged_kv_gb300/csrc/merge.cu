// merge.cu — the merge kernel: the log-sum-exp combine of split partials (see
// merge.cuh) as a kernel of its own, for kvq_split_merge and for decode calls
// whose decode kernel did not merge itself.  A persistent grid (at most two CTAs
// per SM) of 8-warp CTAs.  The kernel is launched as a programmatic dependent of
// the preceding kernel (it may start while that grid drains) and waits for it
// with griddepcontrol.wait before reading any partial.
#include <algorithm>

#include "merge.cuh"

namespace kvq {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

__global__ void __launch_bounds__(kMergeThreads)
    merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                 const int32_t* __restrict__ offs, int uniform, int batch, int num_q_heads, int D, void* out,
                 int out_bf16, float* lse_out, int offs_ready) {
  // a following decode may be scheduled now (it waits for this grid before it
  // writes anything this kernel reads)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The split offsets may be read before the preceding kernel completes when the
  // caller says so (they come from the plan, which the decode kernel never
  // writes); the partials only after it.
  if (!offs_ready) asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float4 red_o[kMergeWarps][32];
  __shared__ float red_w[kMergeWarps];
  __shared__ float red_m[kMergeWarps];
  __shared__ int red_s[kMergeWarps];
  auto sync = [] { __syncthreads(); };
  const int smax = merge_max_splits<kMergeWarps>(offs, uniform, batch, red_s, sync);
  if (smax <= 1) return;  // nothing to merge
  if (offs_ready) asm volatile("griddepcontrol.wait;" ::: "memory");
  merge_all<kMergeWarps>(o_part, lse_part, offs, uniform, batch, num_q_heads, D, out, out_bf16, lse_out, smax, red_o, red_w,
                         red_m, sync);
}

int merge_grid_limit() {
  static int limit = 0;
  if (limit == 0) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      limit = 2 * sms;
    else
      limit = 256;
  }
  return limit;
}

}  // namespace

cudaError_t launch_merge(const float* o_part, const float* lse_part, const int32_t* offsets, int uniform_splits,
                         int batch, int num_q_heads, int head_dim, void* out, int out_bf16, float* lse_out,
                         bool offsets_ready, cudaStream_t stream) {
  const int64_t tasks = (int64_t)batch * num_q_heads * (head_dim / kMinSliceCols);  // most tasks of any shape
  if (tasks <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>(tasks, merge_grid_limit());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel, o_part, lse_part, offsets, uniform_splits, batch, num_q_heads,
                            head_dim, out, out_bf16, lse_out, offsets_ready ? 1 : 0);
}

}  // namespace kvq
