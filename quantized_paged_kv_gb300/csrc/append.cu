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
// INT8 with one scale per 32 values (the same page, section "Is 8 bits
// enough?"): the INT8 codec applied to each group of 32 consecutive elements; the
// scales are stored group-major in each (page, KV head) block, [D/32][16].
//
// With rotation ("Smaller KV cache, faster first token", section "Lever one:
// 4-bit KV with TurboQuant": K and V are rotated before they are quantized), each
// row is first replaced by R(x) = D^(-1/2) H_D (s * x) rounded to bf16, with the
// same fp32 butterfly arithmetic as the rotation kernel (stages h = 1 .. D/2,
// pairs (a, b) -> (a + b, a - b), one multiply by fp32(D^(-1/2)), nearest-even
// bf16), so the stored codes equal those of a rotation pass followed by a plain
// append, without the rotated rows' round trip through memory.
//
// A thread handles EPT consecutive elements of a row (one or two 16-byte loads):
// 16 for NVFP4 (a thread holds one whole scale group) and INT8, 8 for the others;
// D/EPT threads share a row and reduce its maxima with shuffles, and each thread
// carries append_rows<FMT>() rows whose loads go out together.  A row is one (token, KV
// head, K-or-V) triple; a block's rows share the KV head and K-or-V.  Coalesced
// stores: codes EPT (INT8) / EPT/2 (NVFP4) / 2 EPT (BF16) bytes per thread,
// contiguous across the row.
#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kAppendThreads = 256;

// Elements a thread, per format.  Measured on 8,192 tokens (D = 256), 8 against
// 16 (two rows a thread group): INT8 14.7 / 14.7 us, INT8 per 32 values 19.1 /
// 22.1, BF16 12.7 / 12.9, NVFP4 20.9 / 19.7.  INT8 with 16 elements and one row a
// thread group (two rows a warp share each warp instruction of the row-scale
// arithmetic): 13.99 against 14.18 us for 8 elements and two rows (same run).
template <int FMT>
__host__ __device__ constexpr int append_ept() {
  return FMT == KVQ_FMT_NVFP4 || FMT == KVQ_FMT_INT8 ? 16 : 8;
}

template <int EPT>
struct Piece {  // a thread's EPT bf16 elements
  uint4 q[EPT / 8];
};

template <int EPT>
__device__ __forceinline__ void unpack_piece(const Piece<EPT>& v, float (&x)[EPT]) {
#pragma unroll
  for (int k = 0; k < EPT / 8; ++k) {
    const uint32_t w[4] = {v.q[k].x, v.q[k].y, v.q[k].z, v.q[k].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[8 * k + 2 * i] = __uint_as_float(w[i] << 16);
      x[8 * k + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

// Packed fp32 pairs (add/sub/mul .rn.f32x2: two IEEE round-to-nearest operations
// in one instruction, the same results as the scalar ones).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Sign flips of the rotation for this thread's elements EPT t .. EPT t + EPT - 1,
// as XOR masks on the bf16x2 words of its piece: s_i = -1 iff bit 31 of (i + 1) *
// 2654435761 mod 2^32 is set (Knuth's multiplicative hash).
template <int EPT>
__device__ __forceinline__ Piece<EPT> rot_sign_masks(int t) {
  Piece<EPT> m;
#pragma unroll
  for (int k = 0; k < EPT / 8; ++k) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t i = static_cast<uint32_t>(EPT * t + 8 * k + 2 * j);
      const uint32_t lo = ((i + 1u) * 2654435761u) >> 31, hi = ((i + 2u) * 2654435761u) >> 31;
      w[j] = (lo << 15) | (hi << 31);
    }
    m.q[k] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return m;
}

// raw (this thread's EPT bf16 elements EPT t .. EPT t + EPT - 1 of a row spread
// over D/EPT consecutive lanes, signs already applied) <- bf16(R(x)).  fp32
// butterflies in stage order; across lanes, fma(x, -1, w) = w - x and fma(x, 1, w)
// = x + w with one rounding, as the plain sums.  Every lane of the warp takes part
// (shuffles).
template <int D, int EPT>
__device__ __forceinline__ Piece<EPT> rotate_piece_bf16(const Piece<EPT>& raw, int t) {
  float x[EPT];
  unpack_piece<EPT>(raw, x);
#pragma unroll
  for (int h = 1; h < EPT; h <<= 1) {  // butterflies inside the lane
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      if (e & h) continue;
      const float a = x[e], b = x[e + h];
      x[e] = a + b;
      x[e + h] = a - b;
    }
  }
#pragma unroll
  for (int h = EPT; h < D; h <<= 1) {  // across the row's lanes: lane t pairs with t ^ (h / EPT)
    const int m = h / EPT;
    const float sg = (t & m) ? -1.f : 1.f;  // upper lane: w - x; lower lane: x + w
#pragma unroll
    for (int e = 0; e < EPT; ++e) x[e] = fmaf(x[e], sg, __shfl_xor_sync(0xffffffffu, x[e], m));
  }
  const float norm = D == 256 ? __uint_as_float(0x3d800000u) : __uint_as_float(0x3db504f3u);  // fp32(D^-1/2)
  Piece<EPT> out;
#pragma unroll
  for (int k = 0; k < EPT / 8; ++k) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(x[8 * k + 2 * j] * norm, x[8 * k + 2 * j + 1] * norm);
      w[j] = *reinterpret_cast<const uint32_t*>(&b);
    }
    out.q[k] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return out;
}

// Quantize one row (D/EPT threads, this thread's EPT elements in `raw`): token n,
// KV head h, K (which = 0) or V (1); write it to `slot`.  ROT: rotate it first
// (sgn: rot_sign_masks(t)).
template <int FMT, int D, bool ROT, int EPT = append_ept<FMT>()>
__device__ __forceinline__ void append_row(const AppendParams& p, int h, int which, bool in_range, int64_t slot,
                                           Piece<EPT> raw, int t, const Piece<EPT>& sgn) {
  const int Hkv = p.num_kv_heads;
  bool write = in_range && slot >= 0;
  if (write && slot >= p.capacity) {
    if (t == 0 && which == 0 && p.status) atomicOr(p.status, KVQ_DEV_BAD_SLOT);
    write = false;
  }
  if (p.check_finite && in_range) {
    float x[EPT];
    unpack_piece<EPT>(raw, x);
    bool fin = true;
#pragma unroll
    for (int i = 0; i < EPT; ++i) fin &= isfinite(x[i]);
    if (!fin && p.status) atomicOr(p.status, KVQ_DEV_NONFINITE);
  }
  if constexpr (ROT) {
#pragma unroll
    for (int k = 0; k < EPT / 8; ++k)
      raw.q[k] = make_uint4(raw.q[k].x ^ sgn.q[k].x, raw.q[k].y ^ sgn.q[k].y, raw.q[k].z ^ sgn.q[k].z,
                            raw.q[k].w ^ sgn.q[k].w);
    raw = rotate_piece_bf16<D, EPT>(raw, t);
  }
  float x[EPT];
  unpack_piece<EPT>(raw, x);

  const int64_t page = write ? slot / 16 : 0;
  const int prow = write ? static_cast<int>(slot % 16) : 0;
  const int64_t drow = (page * Hkv + h) * 16 + prow;  // row index in [num_pages][Hkv][16]
  uint8_t* codes = which ? p.v_codes : p.k_codes;
  uint8_t* scales = which ? p.v_scales : p.k_scales;

  if constexpr (FMT == KVQ_FMT_BF16) {
    if (write) {
      uint4* dst = reinterpret_cast<uint4*>(codes + drow * (2 * D) + t * (2 * EPT));
#pragma unroll
      for (int k = 0; k < EPT / 8; ++k) dst[k] = raw.q[k];
    }
  } else if constexpr (FMT == KVQ_FMT_INT8 || FMT == KVQ_FMT_INT8_G32) {
    // threads sharing one scale: the row, or a group of 32 elements
    constexpr int TPG = FMT == KVQ_FMT_INT8 ? D / EPT : 32 / EPT;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) amax = fmaxf(amax, fabsf(x[i]));
    if constexpr (TPG == 32) {  // one row a warp: the bit patterns of |x| order like the values
      amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
    } else {
#pragma unroll
      for (int o = 1; o < TPG; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    }
    const float s = __fdiv_rn(amax, 127.0f);
    // code = rne(fp32(x / s)).  Adding 1.5 * 2^23 rounds a float with |v| < 2^22
    // to an integer (ties to even) and leaves that integer's two's-complement low
    // byte in the low byte of the sum's bits.  For a normal, finite s, q = fp32(x
    // * fp32(1 / s)) is within 2^-23 relative (1.6e-5 absolute, |x / s| <= 127.0001)
    // of x / s and fp32(x / s) within 2^-18 of it, so both round to the same
    // integer unless q lies within 2^-14 of a half-integer; then, as for a
    // subnormal, zero or non-finite s, the row takes the exact quotients.
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    const bool fast = s >= 1.17549435e-38f && s <= 3.40282347e+38f;
    float y[EPT];
    bool exact = !fast;
    if (fast) {
      const float rs = __frcp_rn(s);
      const uint64_t rs2 = f2(rs, rs), mg2 = f2(kMagic, kMagic);
#pragma unroll
      for (int i = 0; i < EPT; i += 2) {  // q, q + magic, q - rne(q) for two elements at once
        const uint64_t q2 = mul2(f2(x[i], x[i + 1]), rs2);
        const uint64_t y2 = add2(q2, mg2);
        float d0, d1;
        f2_split(sub2(q2, sub2(y2, mg2)), d0, d1);
        f2_split(y2, y[i], y[i + 1]);
        exact |= fmaxf(fabsf(d0), fabsf(d1)) > 0.5f - 0x1p-14f;
      }
    }
    if (__any_sync(0xffffffffu, exact)) {  // rare: the warp's rows (all lanes) take the exact path
#pragma unroll
      for (int i = 0; i < EPT; ++i) {
        const float q = s > 0.f ? fminf(127.f, fmaxf(-127.f, __fdiv_rn(x[i], s))) : 0.f;
        y[i] = q + kMagic;
      }
    }
    uint32_t b[EPT];
#pragma unroll
    for (int i = 0; i < EPT; ++i) b[i] = __float_as_uint(y[i]);
    uint32_t c[EPT / 4];
#pragma unroll
    for (int j = 0; j < EPT / 4; ++j)
      c[j] = prmt(prmt(b[4 * j], b[4 * j + 1], 0x0040u), prmt(b[4 * j + 2], b[4 * j + 3], 0x0040u), 0x5410u);
    if (write) {
      if constexpr (EPT == 16)
        *reinterpret_cast<uint4*>(codes + drow * D + t * EPT) = make_uint4(c[0], c[1], c[2], c[3]);
      else
        *reinterpret_cast<uint2*>(codes + drow * D + t * EPT) = make_uint2(c[0], c[1]);
      if constexpr (FMT == KVQ_FMT_INT8) {
        if (t == 0) reinterpret_cast<float*>(scales)[drow] = s;
      } else if (t % TPG == 0) {  // group t / TPG of the row: [page][head][group][16 rows]
        reinterpret_cast<float*>(scales)[((page * Hkv + h) * (D / 32) + t / TPG) * 16 + prow] = s;
      }
    }
  } else {  // NVFP4: a group of 16 elements = one thread
    static_assert(FMT != KVQ_FMT_NVFP4 || EPT == 16, "an NVFP4 thread holds one scale group");
    const float gs = which ? p.v_gs : p.k_gs;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const float t2 = __fmul_rn(__fdiv_rn(amax, 6.0f), gs);
    const uint32_t sf = f32_to_e4m3_satfinite(t2);
    const float sd = __low2float(u32_as_h2(e4m3x2_to_h2(sf)));
    // y = fp32(fp32(x * gs) / sd) is rounded to E2M1 (ties to even, saturating),
    // whose rounding thresholds 0.25 .. 5 are integers in 4 y.  With r = fp32(1 /
    // sd) (sd >= 2^-9 or 0), v = fp32(fp32(x * gs) * r) is within 2^-23 relative of
    // x gs / sd and y within 2^-24; |4 y| <= 26, so unless 4 v lies within 2^-16
    // of an integer both round to the same code.  Otherwise the row takes the
    // exact quotients.
    // On packed pairs: xg = x gs, y = xg r, u = 4 y (exact) and u - rne(u), with
    // rne(u) = (u + 1.5 * 2^23) - 1.5 * 2^23 for |u| < 2^22 (a larger |u| means a
    // saturated code either way).
    float xg[EPT], y[EPT];
    bool near = false;
    const float r = sd > 0.f ? __frcp_rn(sd) : 0.f;
    const uint64_t gs2 = f2(gs, gs), r2 = f2(r, r), four2 = f2(4.f, 4.f), mg2 = f2(12582912.0f, 12582912.0f);
#pragma unroll
    for (int i = 0; i < EPT; i += 2) {
      const uint64_t xg2 = mul2(f2(x[i], x[i + 1]), gs2);
      const uint64_t y2 = mul2(xg2, r2);  // sd = 0: every code 0 (y = 0, or NaN for a non-finite input)
      const uint64_t u2 = mul2(y2, four2);
      float d0, d1;
      f2_split(sub2(u2, sub2(add2(u2, mg2), mg2)), d0, d1);
      f2_split(xg2, xg[i], xg[i + 1]);
      f2_split(y2, y[i], y[i + 1]);
      near |= fminf(fabsf(d0), fabsf(d1)) < 0x1p-16f;
    }
    const bool exact = sd > 0.f && near;
    if (__any_sync(0xffffffffu, exact)) {
#pragma unroll
      for (int i = 0; i < EPT; ++i) y[i] = sd > 0.f ? __fdiv_rn(xg[i], sd) : 0.f;
    }
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j)
      packed[j / 4] |= (sd > 0.f ? f32x2_to_e2m1x2(y[2 * j], y[2 * j + 1]) : 0u) << (8 * (j % 4));
    if (write) {
      *reinterpret_cast<uint2*>(codes + drow * (D / 2) + t * 8) = make_uint2(packed[0], packed[1]);
      scales[drow * (D / 16) + t] = static_cast<uint8_t>(sf);
    }
  }
}

// Rows a thread group carries: their loads (rows and slot ids) are all issued
// before the first row is quantized, so each thread keeps EPT/8 x append_rows
// 16-byte loads in flight (two for every format).  Measured on 8,192 tokens
// (D = 256, 16 elements a thread, INT8): 2 rows 14.7 us, 3 rows 15.8, 4 rows 16.7
// (fewer resident blocks), 1 row 14.0.
template <int FMT>
__host__ __device__ constexpr int append_rows() {
  return FMT == KVQ_FMT_INT8 ? 1 : 2;
}

// Grid: x over token blocks, y over (KV head, K or V) = 2 h + which, so that no
// index needs a division.
template <int FMT, int D, bool ROT>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendParams p) {
  // a following decode (a programmatic dependent) may be scheduled now; it waits
  // for this grid to complete before it reads the cache
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int EPT = append_ept<FMT>();
  constexpr int TPR = D / EPT;
  constexpr int ROWS = kAppendThreads / TPR;  // tokens a block handles side by side
  const int t = threadIdx.x % TPR;
  const int which = blockIdx.y & 1;
  const int h = blockIdx.y >> 1;
  const int64_t n0 = (int64_t)blockIdx.x * ROWS * append_rows<FMT>() + threadIdx.x / TPR;
  const uint16_t* src = (which ? p.v_new : p.k_new) + (int64_t)h * D + t * EPT;
  const int64_t stride = (int64_t)p.num_kv_heads * D;  // elements between tokens
  Piece<EPT> raw[append_rows<FMT>()];
  int64_t slot[append_rows<FMT>()];
#pragma unroll
  for (int u = 0; u < append_rows<FMT>(); ++u) {
    const int64_t n = n0 + (int64_t)u * ROWS;
    const int64_t nn = n < p.n_tokens ? n : 0;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + nn * stride);
#pragma unroll
    for (int k = 0; k < EPT / 8; ++k) raw[u].q[k] = s4[k];
    slot[u] = p.slots[nn];
  }
  Piece<EPT> sgn{};
  if constexpr (ROT) sgn = rot_sign_masks<EPT>(t);
#pragma unroll
  for (int u = 0; u < append_rows<FMT>(); ++u) {
    const int64_t n = n0 + (int64_t)u * ROWS;
    append_row<FMT, D, ROT>(p, h, which, n < p.n_tokens, slot[u], raw[u], t, sgn);
  }
}

template <int FMT, int D>
cudaError_t launch_append_t(const AppendParams& p, cudaStream_t stream) {
  constexpr int TOKENS = kAppendThreads / (D / append_ept<FMT>()) * append_rows<FMT>();  // tokens a block covers
  const int64_t blocks = (p.n_tokens + TOKENS - 1) / TOKENS;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF || 2 * p.num_kv_heads > 65535) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(2 * p.num_kv_heads));
  if (p.rotate)
    append_kernel<FMT, D, true><<<grid, kAppendThreads, 0, stream>>>(p);
  else
    append_kernel<FMT, D, false><<<grid, kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(int format, int head_dim, const AppendParams& p, cudaStream_t stream) {
  switch (format) {
    case KVQ_FMT_INT8:
      return head_dim == 256 ? launch_append_t<KVQ_FMT_INT8, 256>(p, stream)
                             : launch_append_t<KVQ_FMT_INT8, 128>(p, stream);
    case KVQ_FMT_INT8_G32:
      return head_dim == 256 ? launch_append_t<KVQ_FMT_INT8_G32, 256>(p, stream)
                             : launch_append_t<KVQ_FMT_INT8_G32, 128>(p, stream);
    case KVQ_FMT_BF16:
      return head_dim == 256 ? launch_append_t<KVQ_FMT_BF16, 256>(p, stream)
                             : launch_append_t<KVQ_FMT_BF16, 128>(p, stream);
    case KVQ_FMT_NVFP4:
      return head_dim == 256 ? launch_append_t<KVQ_FMT_NVFP4, 256>(p, stream)
                             : launch_append_t<KVQ_FMT_NVFP4, 128>(p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
