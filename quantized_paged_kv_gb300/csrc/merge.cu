// merge.cu — log-sum-exp combine of split partials ("long-context-attention-and-
// lessons", section "Give more GPU workers a piece of the attention calculation":
// each piece produces a weighted value sum and the information needed to
// normalise it; averaging the partial outputs would be incorrect).
//
//   M = max_s lse_s,  w_s = exp(lse_s - M),  out = sum_s w_s o_s / sum_s w_s,
//   lse = M + log(sum_s w_s);  a split with lse = -inf (no tokens) has weight 0.
//
// A persistent grid (at most two CTAs per SM) walks the (sequence, query head,
// 64-column slice of D) tuples; sequences with a single split are skipped at the
// cost of one load.  A CTA's 256 threads are 16 float4 columns x 16 split lanes,
// each split lane summing every 16th split with four partial rows in flight,
// then a shared-memory reduction over the split lanes.  The kernel is launched as a programmatic dependent of the decode
// kernel (it may start while the decode grid drains) and waits for the decode
// grid's results with griddepcontrol.wait before reading any partial.
#include <algorithm>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kCols = 16;                          // float4 columns per CTA (64 elements)
constexpr int kLanes = kMergeThreads / kCols;      // split lanes

__global__ void __launch_bounds__(kMergeThreads)
    merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                 const int32_t* __restrict__ offs, int batch, int num_q_heads, int D, void* out, int out_bf16,
                 float* lse_out) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float red_m[kMergeThreads / 32];
  __shared__ float4 red_o[kLanes][kCols];
  __shared__ float red_w[kLanes];
  const int tid = threadIdx.x;
  const int col = tid % kCols;
  const int lane = tid / kCols;
  const int slices = D / (4 * kCols);
  const int64_t tuples = (int64_t)batch * num_q_heads * slices;
  for (int64_t t = blockIdx.x; t < tuples; t += gridDim.x) {
    const int bg = static_cast<int>(t / slices);
    const int slice = static_cast<int>(t - (int64_t)bg * slices);
    const int b = bg / num_q_heads;
    const int g = bg - b * num_q_heads;
    const int base = offs[b];
    const int S = offs[b + 1] - base;
    if (S <= 1) continue;  // written directly by the decode kernel (uniform across the CTA)
    const float* lrow = lse_part + (size_t)base * num_q_heads + g;  // stride num_q_heads

    // max of the split lse values
    float m = -INFINITY;
    for (int s = tid; s < S; s += kMergeThreads) m = fmaxf(m, lrow[(size_t)s * num_q_heads]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) red_m[tid >> 5] = m;
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) M = fmaxf(M, red_m[w]);

    const int d = slice * 4 * kCols + col * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M != -INFINITY) {
      const float* orow = o_part + (size_t)base * num_q_heads * D + (size_t)g * D + d;
      const size_t ostride = (size_t)num_q_heads * D;
      int s = lane;
      for (; s + 3 * kLanes < S; s += 4 * kLanes) {  // four rows in flight
        float l[4];
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          l[u] = lrow[(size_t)(s + u * kLanes) * num_q_heads];
          v[u] = *reinterpret_cast<const float4*>(orow + (size_t)(s + u * kLanes) * ostride);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float w = l[u] == -INFINITY ? 0.f : expf(l[u] - M);
          wsum += w;
          acc.x += w * v[u].x;
          acc.y += w * v[u].y;
          acc.z += w * v[u].z;
          acc.w += w * v[u].w;
        }
      }
      for (; s < S; s += kLanes) {
        const float l = lrow[(size_t)s * num_q_heads];
        if (l == -INFINITY) continue;
        const float w = expf(l - M);
        const float4 v = *reinterpret_cast<const float4*>(orow + (size_t)s * ostride);
        wsum += w;
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
    }
    red_o[lane][col] = acc;
    if (col == 0) red_w[lane] = wsum;
    __syncthreads();
    if (lane == 0) {
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float W = 0.f;
#pragma unroll
      for (int j = 0; j < kLanes; ++j) {
        const float4 v = red_o[j][col];
        o.x += v.x;
        o.y += v.y;
        o.z += v.z;
        o.w += v.w;
        W += red_w[j];
      }
      float lse = -INFINITY;
      if (M != -INFINITY && W > 0.f) {
        const float inv = 1.f / W;
        o.x *= inv;
        o.y *= inv;
        o.z *= inv;
        o.w *= inv;
        lse = M + logf(W);
      } else {
        o = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const size_t off = ((size_t)b * num_q_heads + g) * D + d;
      if (out_bf16) {
        __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(out) + off);
        ob[0] = __floats2bfloat162_rn(o.x, o.y);
        ob[1] = __floats2bfloat162_rn(o.z, o.w);
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + off) = o;
      }
      if (d == 0 && lse_out) lse_out[(size_t)b * num_q_heads + g] = lse;
    }
    __syncthreads();  // shared buffers are reused by the next tuple
  }
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

cudaError_t launch_merge(const float* o_part, const float* lse_part, const int32_t* offsets, int batch,
                         int num_q_heads, int head_dim, void* out, int out_bf16, float* lse_out,
                         cudaStream_t stream) {
  const int64_t tuples = (int64_t)batch * num_q_heads * (head_dim / (4 * kCols));
  if (tuples <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>(tuples, merge_grid_limit());
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
  return cudaLaunchKernelEx(&cfg, merge_kernel, o_part, lse_part, offsets, batch, num_q_heads, head_dim, out,
                            out_bf16, lse_out);
}

}  // namespace kvq
