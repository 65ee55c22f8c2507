// prefill.cu — causal attention of a prompt chunk over a paged INT8 / BF16 cache
// ("half-the-memory-int8-kv-cache", section "Read the prompt using a small
// temporary buffer": a chunk of prompt tokens does enough work per key that it
// pays to read each converted key for many queries; the cached history is read
// in sections whose partial results are combined with the attention weights, as
// for a generated token).
//
// The chunk's T tokens are the last T entries of one sequence's cache (L tokens
// in all); query token i sits at position L - T + i and sees tokens 0 .. L-T+i.
// Here the cache is not converted into a temporary copy: like the decode kernel,
// every page is read once per CTA and its codes enter the tensor cores as exact
// f16 integers (per-token INT8 scales applied to the logits and folded into P).
//
// Work item (one CTA): 128 query rows (token, query head) of one KV head — 16 a
// consumer warp, so every mma.m16n8k16 tile is full — against one range of the
// keys those rows can see (a key split; splits are merged by the merge kernel).
//   * warps 8..11: producers (the first two issue): page j of the range goes to
//     stage j % NST by producer j % 2; one TMA box each for K and V (one head) and
//     a bulk copy each for their scales.
//   * warps 0..7: consumers, each over every page of the range: S = Q K^T for its
//     16 rows, the online softmax with a causal limit per row, O^T += V^T P'^T
//     (two 8-row column tiles; P' split hi + lo for fp32 output, as in the decode
//     kernel).
//   * registers: the producer warpgroup gives registers back, the consumers take
//     them (setmaxnreg), as in the decode kernel.
// All waits are bounded (%globaltimer); a timeout sets KVQ_DEV_TIMEOUT and stops.
#include "decode.cuh"

namespace kvq {
namespace {

constexpr int kPreCW = 8;            // consumer warps
constexpr int kPreRows = kPreCW * 16;  // query rows of an item
constexpr int kPreNP = 2;            // issuing producer warps

template <int FMT, int D>
struct PrefillLayout {
  using T = DecodeTraits<FMT, D>;
  static constexpr int kThreads = (kPreCW + 4) * 32;
  static constexpr int kLaunchRegs = 65536 / kThreads / 8 * 8;
  static constexpr int kProducerRegs = 56;
  static constexpr int kConsumerRegs = (kLaunchRegs * kThreads - kProducerRegs * 128) / (kPreCW * 32) / 8 * 8;
  static_assert(kConsumerRegs * kPreCW * 32 + kProducerRegs * 128 <= kLaunchRegs * kThreads, "register split");
  static constexpr int kHeadCode = kPage * T::kRow;
  static constexpr int kHeadScale = kPage * T::kScaleRow;
  static constexpr int kStageCode = 2 * kHeadCode;
  static constexpr int kStageScale = 2 * kHeadScale;
  static constexpr int kStage = kStageCode + kStageScale;
  static constexpr int kQTile = 16 * D * 2;  // a warp's 16 query rows, f16 / bf16
  static constexpr int kAvail = (227 * 1024 - 1024 - 2 * kMaxStages * 8) / 1024 * 1024;
  static constexpr int kRing = kAvail - kPreCW * kQTile;
  static constexpr int kNST = (kRing / kStage < kMaxStages ? kRing / kStage : kMaxStages) / kPreNP * kPreNP;
  static_assert(kNST >= 2, "ring");
  static constexpr int kSmemBytes = 1024 + kAvail + 2 * kMaxStages * 8;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// position (byte offset) of element (row, k) of a warp's q tile: rows of D f16,
// 16-byte chunks XOR-swizzled by the row; within a k-step (16 elements) the
// elements are stored in the order the K fragments use (see the q tile loop)
__device__ __forceinline__ uint32_t qtile_off(int row, int chunk, int D) {
  return row * D * 2 + (((chunk ^ (row & 7))) << 4);
}

template <int FMT, int D>
__global__ void __launch_bounds__(PrefillLayout<FMT, D>::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const PrefillParams p) {
  using T = DecodeTraits<FMT, D>;
  using Lo = PrefillLayout<FMT, D>;
  constexpr int KS = D / 16;
  constexpr int MT = D / 16;
  constexpr int NST = Lo::kNST;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* codes = smem;                          // NST x [K][V]
  uint8_t* scales = smem + NST * Lo::kStageCode;  // NST x [K][V]
  uint8_t* qtiles = smem + Lo::kRing;             // kPreCW x kQTile
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lo::kAvail);
  uint64_t* empty = full + kMaxStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.num_q_heads / p.num_kv_heads;
  const int TG = p.q_len * G;  // query rows of a KV head
  // item: heaviest row blocks first (they see the most keys)
  const int it = blockIdx.x;
  const int s = it % p.splits;
  const int rest = it / p.splits;
  const int h = rest % p.num_kv_heads;
  const int rb = p.row_blocks - 1 - rest / p.num_kv_heads;
  const int row0 = rb * kPreRows;
  // keys the block's last row can see, and this split's share of their pages
  const int last_tok = min(p.q_len - 1, (row0 + kPreRows - 1) / G);
  const int kmax = p.seq_len - p.q_len + last_tok + 1;
  const int np_all = (kmax + kPage - 1) / kPage;
  const int pg0 = (int)((int64_t)s * np_all / p.splits);
  const int n = (int)((int64_t)(s + 1) * np_all / p.splits) - pg0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kPreCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp >= kPreCW) {
    // ================================================================ producers
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Lo::kProducerRegs));
    const int pi = warp - kPreCW;
    if (pi >= kPreNP || lane != 0) return;
    int last = -1;  // last page this producer issued
    for (int j = pi; j < n; j += kPreNP) {
      const int st = j % NST, rnd = j / NST;
      if (rnd > 0 && !mbar_wait(&empty[st], (rnd - 1) & 1, kWaitLimitNs)) {
        atomicOr(p.status, KVQ_DEV_TIMEOUT);
        break;
      }
      int pg = p.block_table[pg0 + j];
      if (pg < 0 || pg >= p.num_pages) {
        atomicOr(p.status, KVQ_DEV_BAD_PAGE);
        mbar_arrive(&full[st]);  // nothing to load; the stage keeps stale bytes (status flagged)
        last = j;
        continue;
      }
      uint8_t* kc = codes + st * Lo::kStageCode;
      mbar_arrive_expect_tx(&full[st], Lo::kStage);
      tma_load_5d(kc, &tm_k, 0, 0, 0, h, pg, &full[st]);
      tma_load_5d(kc + Lo::kHeadCode, &tm_v, 0, 0, 0, h, pg, &full[st]);
      if constexpr (T::kScaleRow > 0) {
        uint8_t* ks = scales + st * Lo::kStageScale;
        const size_t off = ((size_t)pg * p.num_kv_heads + h) * Lo::kHeadScale;
        bulk_load(ks, p.k_scales + off, Lo::kHeadScale, &full[st]);
        bulk_load(ks + Lo::kHeadScale, p.v_scales + off, Lo::kHeadScale, &full[st]);
      }
      last = j;
    }
    // every copy this producer issued lands before it (and so the CTA) may exit
    for (int j = last; j >= 0 && j > last - NST; j -= kPreNP)
      if (!mbar_wait(&full[j % NST], (j / NST) & 1, kWaitLimitNs)) {
        atomicOr(p.status, KVQ_DEV_TIMEOUT);
        break;
      }
    return;
  }

  // ================================================================== consumers
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Lo::kConsumerRegs));
  const int r = lane >> 2, c = lane & 3;
  const int wrow0 = row0 + warp * 16;  // this warp's first query row
  uint8_t* qt = qtiles + warp * Lo::kQTile;

  // ---- q tile: rows wrow0 .. +15 (token i = row / G, head g = row % G), each
  // scaled by a power of two so its largest |q| is in [2^14, 2^15) and exact in
  // f16 (INT8: f16 MMA); the powers of two are undone on the logits.  Element k
  // of k-step j is stored at tile column kcol(j, k) in the order of the K
  // fragments: INT8 k (2c, 2c+1) <- d 16j+4c+{0,1}, (2c+8, 2c+9) <- d 16j+4c+{2,3};
  // BF16 in natural order.  Lane pairs (lane, lane ^ 16) share a row.
  float row_scale[2] = {1.f, 1.f};  // 2^-k of rows r and r + 8
  {
    for (int rr = 0; rr < 16; ++rr) {
      const int row = wrow0 + rr;
      const bool ok = row < TG;
      const int ti = ok ? row / G : 0, g = ok ? row - (row / G) * G : 0;
      const __nv_bfloat16* qrow =
          reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t)ti * p.num_q_heads + h * G + g) * D;
      // 32 lanes x (D / 32) elements
      constexpr int EPL = D / 32;
      float v[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[e] = ok ? __bfloat162float(qrow[lane * EPL + e]) : 0.f;
      float up = 1.f;
      if constexpr (!T::kBf16Mma) {
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        int k = 0;
        if (amax > 0.f) {
          int ex;
          frexpf(amax, &ex);
          k = min(126, max(-126, 15 - ex));
        }
        up = pow2f(k);
        if (rr == r) row_scale[0] = pow2f(-k);
        if (rr == r + 8) row_scale[1] = pow2f(-k);
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const int d = lane * EPL + e;
        const int j = d >> 4, dd = d & 15;  // k-step, position within its 16 d's
        int kk;                              // k index of d within k-step j
        if constexpr (FMT == KVQ_FMT_INT8) {
          const int cc = dd >> 2, q2 = dd & 3;  // d = 16j + 4cc + q2
          kk = q2 < 2 ? 2 * cc + q2 : 8 + 2 * cc + (q2 - 2);
        } else {
          kk = dd;
        }
        const int col = 16 * j + kk;
        uint8_t* at = qt + qtile_off(rr, col >> 3, D) + (col & 7) * 2;
        if constexpr (T::kBf16Mma) {
          *reinterpret_cast<__nv_bfloat16*>(at) = __float2bfloat16_rn(v[e]);
        } else {
          *reinterpret_cast<__half*>(at) = __float2half_rn(v[e] * up);
        }
      }
    }
  }
  __syncwarp();
  // ldmatrix.x4 of k-step j: lanes 0-7 rows 0-7 / chunk 2j, 8-15 rows 8-15 / 2j,
  // 16-23 rows 0-7 / 2j+1, 24-31 rows 8-15 / 2j+1 -> a0..a3 of the A fragment
  const int qr = (lane & 7) + ((lane >> 3) & 1) * 8;
  const uint32_t qbase = smem_addr(qt) + qr * D * 2;
  auto qfrag = [&](int j, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    const int chunk = 2 * j + (lane >> 4);
    ldsm_x4(qbase + ((chunk ^ (qr & 7)) << 4), a0, a1, a2, a3);
  };

  // causal limits (exclusive) of rows r and r + 8, in the sequence's token order
  int lim[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int row = wrow0 + r + 8 * hh;
    lim[hh] = row < TG ? p.seq_len - p.q_len + row / G + 1 : 0;
  }
  const float qk_scale[2] = {p.sm_scale_log2 * row_scale[0], p.sm_scale_log2 * row_scale[1]};

  [[maybe_unused]] uint32_t voff[4];
  if constexpr (FMT == KVQ_FMT_INT8) {
    const int mm = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4) voff[v4] = (8 * (mm & 1) + rr) * 128 + (((2 * v4 + (mm >> 1)) ^ rr) << 4);
  }

  float oacc[MT][2][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.f;
  // P' in hi + lo terms for fp32 output, one term for bf16 output (as in the decode kernel)
  const bool p_lo = !p.out_bf16;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  bool alive = true;

  for (int j = 0; j < n; ++j) {
    const int st = j % NST, rnd = j / NST;
    const bool got = mbar_wait(&full[st], rnd & 1, kWaitLimitNs);
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) atomicOr(p.status, KVQ_DEV_TIMEOUT);
      alive = false;
      break;
    }
    const uint32_t kblk = smem_addr(codes + st * Lo::kStageCode);
    const uint32_t vblk = kblk + Lo::kHeadCode;
    const uint8_t* ksc = scales + st * Lo::kStageScale;
    const uint8_t* vsc = ksc + Lo::kHeadScale;
    const int tok0 = (pg0 + j) * kPage;

    // ------------------------------------------------------------ S = Q K^T
    float sacc[2][2][4];  // [n-tile][accumulation chain]
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int u = 0; u < 2; ++u) sacc[i][u][0] = sacc[i][u][1] = sacc[i][u][2] = sacc[i][u][3] = 0.f;
    if constexpr (FMT == KVQ_FMT_INT8) {
#pragma unroll
      for (int cg = 0; cg < KS / 4; ++cg) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          uint32_t w[4];
          ldsm_x4(swz(kblk, 8 * i + (lane & 7), 4 * cg + (lane >> 3)), w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            uint32_t a0, a1, a2, a3;
            qfrag(4 * cg + m, a0, a1, a2, a3);
            const uint32_t x = w[m] ^ 0x80808080u;
            mma16816<false>(sacc[i][m & 1], a0, a1, a2, a3, i8pair_to_h2<0x4140>(x), i8pair_to_h2<0x4342>(x));
          }
        }
      }
    } else {
#pragma unroll
      for (int cg = 0; cg < KS / 2; ++cg) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          uint32_t w[4];
          ldsm_x4(swz(kblk, 8 * i + (lane & 7), 4 * cg + (lane >> 3)), w[0], w[1], w[2], w[3]);
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            uint32_t a0, a1, a2, a3;
            qfrag(2 * cg + m, a0, a1, a2, a3);
            mma16816<true>(sacc[i][m], a0, a1, a2, a3, w[2 * m], w[2 * m + 1]);
          }
        }
      }
    }

    // ------------------------------------------------------------ online softmax
    // lane: rows r (c0, c1) and r + 8 (c2, c3); tokens 2c, 2c+1 (n-tile 0), 8+2c, 9+2c (n-tile 1)
    const int tk[4] = {2 * c, 2 * c + 1, 8 + 2 * c, 9 + 2 * c};
    float ks4[4] = {1.f, 1.f, 1.f, 1.f};
    if constexpr (FMT == KVQ_FMT_INT8) {
      const float2 a = *reinterpret_cast<const float2*>(ksc + 8 * c);
      const float2 bb = *reinterpret_cast<const float2*>(ksc + 32 + 8 * c);
      ks4[0] = a.x; ks4[1] = a.y; ks4[2] = bb.x; ks4[3] = bb.y;
    }
    float pr[2][4];
    float alpha[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float z[4];
      z[0] = sacc[0][0][2 * hh] + sacc[0][1][2 * hh];
      z[1] = sacc[0][0][2 * hh + 1] + sacc[0][1][2 * hh + 1];
      z[2] = sacc[1][0][2 * hh] + sacc[1][1][2 * hh];
      z[3] = sacc[1][0][2 * hh + 1] + sacc[1][1][2 * hh + 1];
      float pmax = -INFINITY;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        z[u] = (tok0 + tk[u] < lim[hh]) ? z[u] * ks4[u] * qk_scale[hh] : -INFINITY;
        pmax = fmaxf(pmax, z[u]);
      }
      pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, 1));
      pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, 2));
      const float m_new = fmaxf(m_run[hh], pmax);
      // a row that has seen no visible key yet keeps m = -inf: scale 1, p = 0
      alpha[hh] = m_new == -INFINITY ? 1.f : exp2f(m_run[hh] - m_new);
      m_run[hh] = m_new;
      float psum = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        pr[hh][u] = m_new == -INFINITY ? 0.f : exp2f(z[u] - m_new);
        psum += pr[hh][u];
      }
      l_run[hh] = l_run[hh] * alpha[hh] + psum;
    }
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
      // O^T columns: n-tile 0 = rows 2c, 2c+1; n-tile 1 = rows 8+2c, 9+2c
      const float a00 = __shfl_sync(0xffffffffu, alpha[0], 8 * c), a01 = __shfl_sync(0xffffffffu, alpha[0], 8 * c + 4);
      const float a10 = __shfl_sync(0xffffffffu, alpha[1], 8 * c), a11 = __shfl_sync(0xffffffffu, alpha[1], 8 * c + 4);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        oacc[mt][0][0] *= a00;
        oacc[mt][0][1] *= a01;
        oacc[mt][0][2] *= a00;
        oacc[mt][0][3] *= a01;
        oacc[mt][1][0] *= a10;
        oacc[mt][1][1] *= a11;
        oacc[mt][1][2] *= a10;
        oacc[mt][1][3] *= a11;
      }
    }
    // P' (B operands of O^T = V^T P'^T, one per 8-row column tile): INT8 folds the
    // V scale of the token in; masked tokens (and NaN scales of unwritten slots
    // past the sequence) give exactly 0
    float vs4[4] = {1.f, 1.f, 1.f, 1.f};
    if constexpr (FMT == KVQ_FMT_INT8) {
      const float2 a = *reinterpret_cast<const float2*>(vsc + 8 * c);
      const float2 bb = *reinterpret_cast<const float2*>(vsc + 32 + 8 * c);
      vs4[0] = a.x; vs4[1] = a.y; vs4[2] = bb.x; vs4[3] = bb.y;
    }
    uint32_t phi[2][2], plo[2][2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float pv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) pv[u] = (tok0 + tk[u] < lim[hh]) ? pr[hh][u] * vs4[u] : 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if constexpr (T::kBf16Mma) {
          const __nv_bfloat162 hi = __floats2bfloat162_rn(pv[2 * u], pv[2 * u + 1]);
          const __nv_bfloat162 lo =
              __floats2bfloat162_rn(pv[2 * u] - __low2float(hi), pv[2 * u + 1] - __high2float(hi));
          phi[hh][u] = *reinterpret_cast<const uint32_t*>(&hi);
          plo[hh][u] = *reinterpret_cast<const uint32_t*>(&lo);
        } else {
          const __half2 hi = __floats2half2_rn(pv[2 * u], pv[2 * u + 1]);
          const __half2 lo = __floats2half2_rn(pv[2 * u] - __low2float(hi), pv[2 * u + 1] - __high2float(hi));
          phi[hh][u] = h2_as_u32(hi);
          plo[hh][u] = h2_as_u32(lo);
        }
      }
    }

    // ------------------------------------------------------------ O^T += V^T P'^T
    const int nvalid = min(kPage, p.seq_len - tok0);  // written slots of this page
    if constexpr (FMT == KVQ_FMT_INT8) {
      uint32_t vb[4];
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4) vb[v4] = vblk + voff[v4];
#pragma unroll
      for (int cp = 0; cp < MT / 2; ++cp) {
        uint32_t w[4];
        ldsm_x4_t(vb[cp & 3] + (cp >> 2) * (kPage * 128), w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t x0 = w[2 * u] ^ 0x80808080u;
          const uint32_t x1 = w[2 * u + 1] ^ 0x80808080u;
          const uint32_t a0 = i8pair_to_h2<0x4240>(x0), a1 = i8pair_to_h2<0x4341>(x0);
          const uint32_t a2 = i8pair_to_h2<0x4240>(x1), a3 = i8pair_to_h2<0x4341>(x1);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            mma16816<false>(oacc[2 * cp + u][nt], a0, a1, a2, a3, phi[nt][0], phi[nt][1]);
            if (p_lo) mma16816<false>(oacc[2 * cp + u][nt], a0, a1, a2, a3, plo[nt][0], plo[nt][1]);
          }
        }
      }
    } else {
      const uint32_t m0 = (2 * c < nvalid ? 0x0000FFFFu : 0u) | (2 * c + 1 < nvalid ? 0xFFFF0000u : 0u);
      const uint32_t m1 = (8 + 2 * c < nvalid ? 0x0000FFFFu : 0u) | (9 + 2 * c < nvalid ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int mm = lane >> 3;
        const int trow = 8 * (mm >> 1) + (lane & 7);
        uint32_t w[4];
        ldsm_x4_t(swz(vblk, trow, 2 * mt + (mm & 1)), w[0], w[1], w[2], w[3]);
        if (nvalid < kPage) {  // unwritten slots may hold NaN bit patterns: zero them
          w[0] &= m0; w[1] &= m0; w[2] &= m1; w[3] &= m1;
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          mma16816<true>(oacc[mt][nt], w[0], w[1], w[2], w[3], phi[nt][0], phi[nt][1]);
          if (p_lo) mma16816<true>(oacc[mt][nt], w[0], w[1], w[2], w[3], plo[nt][0], plo[nt][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ================================================================ epilogue
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
    if (!alive) {
      m_run[hh] = -INFINITY;
      l_run[hh] = 0.f;
    }
  }
  constexpr float kLn2 = 0.69314718055994530942f;
  float inv[2], lse[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const bool any = m_run[hh] != -INFINITY && l_run[hh] > 0.f;
    inv[hh] = any ? 1.f / l_run[hh] : 0.f;
    lse[hh] = any ? (m_run[hh] + log2f(l_run[hh])) * kLn2 : -INFINITY;
  }
  const bool direct = p.splits == 1;
  // output row of query row `row`: out[(i * Hq + h * G + g)] or the partial
  // row ((i * splits + s) * Hq + h * G + g)
  auto out_row = [&](int row) -> size_t {
    const int ti = row / G, g = row - ti * G;
    const size_t qh = (size_t)h * G + g;
    return direct ? (size_t)ti * p.num_q_heads + qh : ((size_t)ti * p.splits + s) * p.num_q_heads + qh;
  };
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const float w0 = __shfl_sync(0xffffffffu, inv[nt], 8 * c), w1 = __shfl_sync(0xffffffffu, inv[nt], 8 * c + 4);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int row = wrow0 + 8 * nt + 2 * c + e;
      if (row >= TG) continue;
      const size_t orow = out_row(row);
      const float wt = e ? w1 : w0;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        int da, db;
        if constexpr (FMT == KVQ_FMT_INT8) {
          da = 16 * mt + 2 * r;
          db = da + 1;
        } else {
          da = 16 * mt + r;
          db = da + 8;
        }
        const float va = oacc[mt][nt][e] * wt, vb = oacc[mt][nt][2 + e] * wt;
        if (direct && p.out_bf16) {
          __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.out) + orow * D;
          if (db == da + 1) {
            *reinterpret_cast<__nv_bfloat162*>(ob + da) = __floats2bfloat162_rn(va, vb);
          } else {
            ob[da] = __float2bfloat16_rn(va);
            ob[db] = __float2bfloat16_rn(vb);
          }
        } else {
          float* of = (direct ? reinterpret_cast<float*>(p.out) : p.o_part) + orow * D;
          if (db == da + 1) {
            *reinterpret_cast<float2*>(of + da) = make_float2(va, vb);
          } else {
            of[da] = va;
            of[db] = vb;
          }
        }
      }
    }
  }
  if (c == 0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = wrow0 + r + 8 * hh;
      if (row >= TG) continue;
      const size_t orow = out_row(row);
      if (direct) {
        if (p.lse_out) p.lse_out[orow] = lse[hh];
      } else {
        p.lse_part[orow] = lse[hh];
      }
    }
  }
}

template <int FMT, int D>
cudaError_t launch_pt(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p, int grid,
                      cudaStream_t stream) {
  using Lo = PrefillLayout<FMT, D>;
  prefill_kernel<FMT, D><<<grid, Lo::kThreads, Lo::kSmemBytes, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int FMT, int D>
PrefillInstance pinstance_of() {
  using Lo = PrefillLayout<FMT, D>;
  return PrefillInstance{reinterpret_cast<const void*>(&prefill_kernel<FMT, D>), Lo::kSmemBytes, Lo::kThreads,
                         Lo::kLaunchRegs, kPreRows};
}

}  // namespace

bool prefill_instance(int format, int head_dim, PrefillInstance* out) {
  if (format == KVQ_FMT_INT8 && head_dim == 256) *out = pinstance_of<KVQ_FMT_INT8, 256>();
  else if (format == KVQ_FMT_INT8 && head_dim == 128) *out = pinstance_of<KVQ_FMT_INT8, 128>();
  else if (format == KVQ_FMT_BF16 && head_dim == 256) *out = pinstance_of<KVQ_FMT_BF16, 256>();
  else if (format == KVQ_FMT_BF16 && head_dim == 128) *out = pinstance_of<KVQ_FMT_BF16, 128>();
  else return false;
  return true;
}

cudaError_t launch_prefill(int format, int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int grid, cudaStream_t stream) {
  if (format == KVQ_FMT_INT8 && head_dim == 256) return launch_pt<KVQ_FMT_INT8, 256>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_INT8 && head_dim == 128) return launch_pt<KVQ_FMT_INT8, 128>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_BF16 && head_dim == 256) return launch_pt<KVQ_FMT_BF16, 256>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_BF16 && head_dim == 128) return launch_pt<KVQ_FMT_BF16, 128>(tk, tv, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
