// append.cu — kv_quant_append: quantize new K/V rows and scatter them into slots.
//
// INT8 ("half-the-memory-int8-kv-cache", section "An 8-bit cache was already
// available"): per (token, KV head) row, scale = fp32(absmax / 127) and
// code = clamp(rne(fp32(x / scale)), -127, 127) (the symmetric clamp and
// round-to-nearest follow the gllm page, section "Quantization Design").
// NVFP4 ("Building an NVFP4 KV cache for a hybrid Qwen model", sections "How 2,048
// bytes became 576" and "Writing and reading the packed cache"): group maxima over
// 16 elements, an E4M3 scale per group, E2M1 rounding, pairs packed low nibble
// first; invalid (negative) slots do not write.
//
// One thread handles 8 consecutive elements of one row (16-byte loads); D/8
// threads share a row and reduce its maxima with shuffles.  A row is one
// (token, KV head, K-or-V) triple.  Coalesced stores: codes 8 (INT8) / 4 (NVFP4) /
// 16 (BF16) bytes per thread, contiguous across the row.
#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kAppendThreads = 256;

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// E2M1 code (sign in bit 3) of y: nearest of {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to
// the even code, saturating at 6.  The thresholds are the midpoints between grid
// neighbours; at a midpoint the comparison is strict where the lower neighbour
// has the even code and inclusive where the upper one does.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  const uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
                     (a > 5.0f);
  return m | ((__float_as_uint(y) >> 31) << 3);
}

template <int FMT, int D>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendParams p) {
  // a following decode (a programmatic dependent) may be scheduled now; it waits
  // for this grid to complete before it reads the cache
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int TPR = D / 8;
  constexpr int ROWS = kAppendThreads / TPR;
  const int64_t row = (int64_t)blockIdx.x * ROWS + threadIdx.x / TPR;
  const int t = threadIdx.x % TPR;
  const int64_t nrows = p.n_tokens * p.num_kv_heads * 2;
  const bool in_range = row < nrows;
  const int64_t r = in_range ? row : 0;
  const int which = static_cast<int>(r & 1);  // 0: K, 1: V
  const int64_t nh = r >> 1;
  const int Hkv = p.num_kv_heads;
  const int64_t n = nh / Hkv;
  const int h = static_cast<int>(nh - n * Hkv);
  const int64_t slot = p.slots[n];
  bool write = in_range && slot >= 0;
  if (write && slot >= p.capacity) {
    if (t == 0 && which == 0 && p.status) atomicOr(p.status, KVQ_DEV_BAD_SLOT);
    write = false;
  }

  const uint16_t* src = (which ? p.v_new : p.k_new) + nh * D + t * 8;
  const uint4 raw = *reinterpret_cast<const uint4*>(src);
  float x[8];
  unpack_bf16x8(raw, x);
  if (p.check_finite && in_range) {
    bool fin = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) fin &= isfinite(x[i]);
    if (!fin && p.status) atomicOr(p.status, KVQ_DEV_NONFINITE);
  }

  const int64_t page = write ? slot / 16 : 0;
  const int prow = write ? static_cast<int>(slot % 16) : 0;
  const int64_t drow = (page * Hkv + h) * 16 + prow;  // row index in [num_pages][Hkv][16]
  uint8_t* codes = which ? p.v_codes : p.k_codes;
  uint8_t* scales = which ? p.v_scales : p.k_scales;

  if constexpr (FMT == KVQ_FMT_BF16) {
    if (write) *reinterpret_cast<uint4*>(codes + drow * (2 * D) + t * 16) = raw;
  } else if constexpr (FMT == KVQ_FMT_INT8) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 127.0f);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int ci = 0;
      if (s > 0.f) ci = min(127, max(-127, __float2int_rn(__fdiv_rn(x[i], s))));
      const uint32_t byte = static_cast<uint32_t>(ci) & 0xFFu;
      if (i < 4) lo |= byte << (8 * i);
      else hi |= byte << (8 * (i - 4));
    }
    if (write) {
      *reinterpret_cast<uint2*>(codes + drow * D + t * 8) = make_uint2(lo, hi);
      if (t == 0) reinterpret_cast<float*>(scales)[drow] = s;
    }
  } else {  // NVFP4: a group of 16 elements = threads (2k, 2k+1)
    const float gs = which ? p.v_gs : p.k_gs;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const float t2 = __fmul_rn(__fdiv_rn(amax, 6.0f), gs);
    const uint32_t sf = f32_to_e4m3_satfinite(t2);
    const float sd = __low2float(u32_as_h2(e4m3x2_to_h2(sf)));
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t ci = 0;
      if (sd > 0.f) ci = e2m1_code(__fdiv_rn(__fmul_rn(x[i], gs), sd));
      packed |= ci << (4 * i);  // element 2j in the low nibble of byte j
    }
    if (write) {
      *reinterpret_cast<uint32_t*>(codes + drow * (D / 2) + t * 4) = packed;
      if ((t & 1) == 0) scales[drow * (D / 16) + t / 2] = static_cast<uint8_t>(sf);
    }
  }
}

template <int FMT, int D>
cudaError_t launch_append_t(const AppendParams& p, cudaStream_t stream) {
  constexpr int ROWS = kAppendThreads / (D / 8);
  const int64_t nrows = p.n_tokens * p.num_kv_heads * 2;
  const int64_t blocks = (nrows + ROWS - 1) / ROWS;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  append_kernel<FMT, D><<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(int format, int head_dim, const AppendParams& p, cudaStream_t stream) {
  switch (format) {
    case KVQ_FMT_INT8:
      return head_dim == 256 ? launch_append_t<KVQ_FMT_INT8, 256>(p, stream)
                             : launch_append_t<KVQ_FMT_INT8, 128>(p, stream);
    case KVQ_FMT_BF16:
      return head_dim == 256 ? launch_append_t<KVQ_FMT_BF16, 256>(p, stream)
                             : launch_append_t<KVQ_FMT_BF16, 128>(p, stream);
    case KVQ_FMT_NVFP4:
      return launch_append_t<KVQ_FMT_NVFP4, 256>(p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
