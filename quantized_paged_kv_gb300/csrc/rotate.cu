// rotate.cu — rotation of K/V/q rows before quantization ("Smaller KV cache,
// faster first token", section "Lever one: 4-bit KV with TurboQuant": the K and
// V vectors are rotated before they are quantized, so that outliers spread over
// all dimensions).
//
// R(x) = D^(-1/2) H_D (s * x) with H_D the Sylvester Hadamard matrix and the
// fixed signs s_i = -1 iff bit 31 of (i + 1) * 2654435761 mod 2^32 is set (Knuth's
// multiplicative hash); R^-1(y) = s * (D^(-1/2) H_D y).  R preserves dot
// products, so attention over rotated q and K gives the same scores, and over
// rotated V gives R(o), undone by R^-1.  Arithmetic (it fixes the stored bits):
// fp32 butterflies in stage order h = 1, 2, 4, ..., D/2, each pair (a, b) at
// positions (i, i + h), bit h of i clear, becoming (a + b, a - b); one multiply
// by fp32(D^(-1/2)); rounding to the output type (bf16: nearest, ties to even).
//
// One warp a row: lane l holds elements EPL l .. EPL l + EPL - 1; stages h < EPL
// run inside the lane, the others pair lane l with lane l ^ (h / EPL).
#include <cuda_bf16.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kRotWarps = 8;

__device__ __forceinline__ float rot_sign(int i) {
  const uint32_t h = static_cast<uint32_t>(i + 1) * 2654435761u;
  return (h >> 31) ? -1.f : 1.f;
}

template <int D>
__device__ __forceinline__ float rot_norm() {
  return D == 256 ? __uint_as_float(0x3d800000u) : __uint_as_float(0x3db504f3u);  // fp32(D^-1/2)
}

// 16-byte pieces of EPL contiguous elements (EPL = 4 or 8; bf16 or fp32)
template <int EPL, bool BF16>
__device__ __forceinline__ void load_row_part(const void* p, float (&x)[EPL]) {
  if constexpr (BF16) {
    uint32_t w[EPL / 2];
    if constexpr (EPL == 8) {
      const uint4 v = *static_cast<const uint4*>(p);
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
      const uint2 v = *static_cast<const uint2*>(p);
      w[0] = v.x; w[1] = v.y;
    }
#pragma unroll
    for (int i = 0; i < EPL / 2; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL / 4; ++i) {
      const float4 v = static_cast<const float4*>(p)[i];
      x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
    }
  }
}

template <int EPL, bool BF16>
__device__ __forceinline__ void store_row_part(void* p, const float (&x)[EPL]) {
  if constexpr (BF16) {
    uint32_t w[EPL / 2];
#pragma unroll
    for (int i = 0; i < EPL / 2; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    if constexpr (EPL == 8) *static_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else *static_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int i = 0; i < EPL / 4; ++i)
      static_cast<float4*>(p)[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
  }
}

// Launched as a programmatic dependent: the kernels after it may be scheduled at
// once (they wait for this grid before reading its output), and it reads its
// input only after the preceding kernel (which may have written it) completed.
template <int D, bool IN_BF16, bool OUT_BF16, bool INVERSE>
__global__ void __launch_bounds__(kRotWarps * 32) rotate_kernel(const void* in, void* out, int64_t n_rows) {
  constexpr int EPL = D / 32;  // elements a lane
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRotWarps + (threadIdx.x >> 5);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (row >= n_rows) return;  // the whole warp leaves together
  float x[EPL];
  const int64_t base = row * D + lane * EPL;
  load_row_part<EPL, IN_BF16>(IN_BF16 ? static_cast<const void*>(static_cast<const __nv_bfloat16*>(in) + base)
                                      : static_cast<const void*>(static_cast<const float*>(in) + base),
                              x);
  if constexpr (!INVERSE) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) x[e] *= rot_sign(lane * EPL + e);  // exact
  }
  // butterflies inside the lane
#pragma unroll
  for (int h = 1; h < EPL; h <<= 1) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      if (e & h) continue;
      const float a = x[e], b = x[e + h];
      x[e] = a + b;
      x[e + h] = a - b;
    }
  }
  // butterflies across lanes
#pragma unroll
  for (int h = EPL; h < D; h <<= 1) {
    const int m = h / EPL;
    const bool upper = lane & m;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float w = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = upper ? w - x[e] : x[e] + w;
    }
  }
  const float norm = rot_norm<D>();
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    x[e] *= norm;
    if constexpr (INVERSE) x[e] *= rot_sign(lane * EPL + e);  // exact
  }
  store_row_part<EPL, OUT_BF16>(OUT_BF16 ? static_cast<void*>(static_cast<__nv_bfloat16*>(out) + base)
                                        : static_cast<void*>(static_cast<float*>(out) + base),
                                x);
}

template <int D, bool IN_BF16, bool OUT_BF16>
cudaError_t launch_rot_t(const void* in, void* out, int64_t n_rows, bool inverse, cudaStream_t stream) {
  const int64_t grid = (n_rows + kRotWarps - 1) / kRotWarps;
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kRotWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return inverse ? cudaLaunchKernelEx(&cfg, rotate_kernel<D, IN_BF16, OUT_BF16, true>, in, out, n_rows)
                 : cudaLaunchKernelEx(&cfg, rotate_kernel<D, IN_BF16, OUT_BF16, false>, in, out, n_rows);
}

template <int D>
cudaError_t launch_rot_d(const void* in, bool in_bf16, void* out, bool out_bf16, int64_t n_rows, bool inverse,
                         cudaStream_t stream) {
  if (in_bf16 && out_bf16) return launch_rot_t<D, true, true>(in, out, n_rows, inverse, stream);
  if (in_bf16) return launch_rot_t<D, true, false>(in, out, n_rows, inverse, stream);
  if (out_bf16) return launch_rot_t<D, false, true>(in, out, n_rows, inverse, stream);
  return launch_rot_t<D, false, false>(in, out, n_rows, inverse, stream);
}

}  // namespace

cudaError_t launch_rotate(const void* in, bool in_bf16, void* out, bool out_bf16, int64_t n_rows, int head_dim,
                          bool inverse, cudaStream_t stream) {
  if (n_rows <= 0) return cudaSuccess;
  if (head_dim == 256) return launch_rot_d<256>(in, in_bf16, out, out_bf16, n_rows, inverse, stream);
  if (head_dim == 128) return launch_rot_d<128>(in, in_bf16, out, out_bf16, n_rows, inverse, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
