// prefill_tc.cu — causal attention of a prompt chunk over a paged INT8 / NVFP4 /
// BF16 cache on the fifth-generation tensor cores (tcgen05.mma, accumulators in TMEM)
// ("half-the-memory-int8-kv-cache", section "Read the prompt using a small
// temporary buffer": a chunk of prompt tokens does enough work per key that each
// key is converted once to fp16 and then used by many queries; the history is
// read in key ranges whose partial results are combined with their log-sum-exp
// weights, as for a generated token).
//
// The chunk's T tokens are the last T entries of one sequence's cache (L tokens
// in all); query token i sits at position L - T + i and sees tokens 0 .. L-T+i.
// A launch covers one chunk, or (a verify call) T tokens of each of a batch of
// sequences, each with its own block-table row and its length read on the device.
//
// Work item (one CTA): 128 query rows (token, query head) of one KV head of one
// sequence — the MMA's M — against one key range (a split; splits are merged by
// the merge kernel), in tiles of 64 keys (four pages).  Warp roles:
//   * warps 4..7 (converters): per tile, K codes -> fp16 (NVFP4: codes x group
//     scale, exact in fp16; INT8: the codes) in the canonical K-major
//     layout with the 128-byte swizzle (the B operand of S = Q K^T) and V codes
//     -> fp16 in the MN-major layout (the B operand of O = P V, no transpose); the
//     INT8 scales go to shared memory.  Keys past the range or the sequence, or
//     on a page whose id is out of the pool, are written as zeros, and a per-tile
//     mask of the keys read goes out with the scales: the softmax leaves the
//     others out, as the decode kernel does.
//   * warp 8, lane 0 (MMA): S(i) = Q K(i)^T into one of two TMEM buffers, then
//     O += P(i-1) V(i-1); each group of MMAs is committed to an mbarrier.
//   * warps 0..3 (softmax, one query row a thread): the q row (INT8: scaled by a
//     power of two so that it is exact in fp16) into Q in TMEM, the A operand of
//     S = Q K^T; per tile, S from TMEM (tcgen05.ld), the online softmax with the
//     row's causal limit, and P' (INT8: the V scale of each key folded in),
//     written over S(i) in TMEM as the fp16 / bf16 A operand of the P V product,
//     in hi + lo terms for fp32 output.  The running maximum is raised only when
//     a row's new maximum exceeds it by more than 2^8 (then the row of O in TMEM
//     is rescaled), so p <= 256.
// Every wait is bounded (%globaltimer); a timeout sets KVQ_DEV_TIMEOUT, the CTA
// waits for its issued MMAs, frees its TMEM and returns.
#include "decode.cuh"

namespace kvq {
namespace {

constexpr int kTcRows = 128;               // query rows of an item (the MMA's M)
constexpr int kTcKeys = 64;                // keys of a tile
constexpr int kTcPages = kTcKeys / kPage;  // pages of a tile
constexpr int kTcThreads = 9 * 32;
constexpr float kTcRescale = 8.0f;  // log2 of the largest p a stale maximum may give

template <int FMT, int D>
struct TcLayout {
  static constexpr int kAtoms = D / 64;                  // 128-byte swizzle atoms along D (fp16)
  static constexpr int kKBytes = kTcKeys * D * 2;        // [atom][64 keys][128 B]
  static constexpr int kVBytes = kTcKeys * D * 2;        // [8-key group][d atom][8 keys][128 B]
  static constexpr int kKAt = 0;                         // two K tiles
  static constexpr int kVAt = kKAt + 2 * kKBytes;        // two V tiles
  static constexpr int kScRing = 3;                      // scale buffers (tiles in flight)
  static constexpr int kScAt = kVAt + 2 * kVBytes;       // float k scales [3][64], v scales [3][64]
  // key-validity masks: uint16 [3][4 converter warps], bit k = key 16 w + k read
  static constexpr int kMaskAt = kScAt + 2 * kScRing * kTcKeys * 4;
  static constexpr int kBarAt = kMaskAt + 32;
  static constexpr int kNumBars = 14;
  static constexpr int kSlotAt = kBarAt + kNumBars * 8;
  static constexpr int kSmemBytes = 1024 + kSlotAt + 16;
  static_assert(kNumBars >= 14, "barriers");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  // TMEM columns: O (D), two S buffers of 64, and Q (D / 2: f16 / bf16 pairs).
  // P(i) is written over S(i) once the softmax has read S(i): the hi terms (32
  // columns of pairs) then the lo terms, the A operand of O += P V.  Q is the A
  // operand of S = Q K^T, so neither product reads an A operand from shared memory.
  static constexpr uint32_t kTmemO = 0;
  static constexpr uint32_t kTmemS = D;
  static constexpr uint32_t kTmemQ = D + 2 * kTcKeys;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kTmemQ + D / 2 <= kTmemCols, "TMEM columns");
  // MN-major V: byte offset between d atoms (leading) and between 8-key groups (strided)
  static constexpr uint32_t kVLbo = 1024, kVSbo = kAtoms * 1024;
};

// Per-buffer barriers alternate with the tile's parity (tile i uses buffer i & 1),
// so that no waiter can see a barrier two phases ahead of the one it waits for.
enum : int {
  kBarQ = 0,
  kBarP0,      // P(i) written into TMEM buffer 0 / 1 (softmax warps)
  kBarP1,
  kBarK0,      // K(i) converted, buffers 0 / 1 (converter warps)
  kBarK1,
  kBarV0,      // V(i) converted
  kBarV1,
  kBarS0,      // S(i) = Q K(i)^T done (commit)
  kBarS1,
  kBarKF0,     // S(i) done: K buffer i & 1 free (commit)
  kBarKF1,
  kBarO0,      // P(i) V(i) done (commit)
  kBarO1,
  kBarFinal,
  kBarCount
};

// byte offset of the 16-byte chunk holding elements d0 .. d0+7 (d0 % 8 == 0) of
// row r in a K-major tile of `rows` rows ([atom][rows][128 B], 128-byte swizzle)
__device__ __forceinline__ uint32_t kmajor_off(int r, int d0, int rows) {
  const int a = d0 >> 6, c = (d0 & 63) >> 3;
  return (uint32_t)(a * rows * 128 + r * 128 + ((c ^ (r & 7)) << 4));
}

// byte offset of elements d0 .. d0+7 of key n in the MN-major V tile
template <int D>
__device__ __forceinline__ uint32_t vtile_off(int n, int d0) {
  const int g = n >> 3, kr = n & 7, a = d0 >> 6, c = (d0 & 63) >> 3;
  return (uint32_t)(g * (D / 64) * 1024 + a * 1024 + kr * 128 + ((c ^ kr) << 4));
}

template <int FMT, int D, bool PLO>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const PrefillParams p) {
  using T = DecodeTraits<FMT, D>;
  using Lo = TcLayout<FMT, D>;
  constexpr bool kBf16 = T::kBf16Mma;
  constexpr int KS = D / 16;  // k-steps of S
  constexpr uint32_t kIdescS = umma_idesc_f16(kTcRows, kTcKeys, kBf16, false);
  constexpr uint32_t kIdescPV = umma_idesc_f16(kTcRows, D, kBf16, true);

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lo::kBarAt);
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + Lo::kSlotAt);  // [0] TMEM base, [1] abort flag
  float* ksc = reinterpret_cast<float*>(smem + Lo::kScAt);            // [3][64]
  float* vsc = ksc + Lo::kScRing * kTcKeys;                           // [3][64]
  uint16_t* kmask = reinterpret_cast<uint16_t*>(smem + Lo::kMaskAt);  // [3][4]
  const uint32_t sbase = smem_addr(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the merge of the key splits may be scheduled now (it waits for this grid)
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int b = 0; b < kBarCount; ++b) mbar_init(&bars[b], b <= kBarV1 ? 4 : 1);
    slot[1] = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(slot, Lo::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The launch is a programmatic dependent of the preceding kernel: the barriers
  // and the TMEM are set up while that kernel drains, and nothing it may write
  // (q, the block table, the sequence length, the pool) is read before it completes.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // work item: (sequence b, row block rb, KV head h, key split s), split fastest
  const int it = blockIdx.x;
  const int s = it % p.splits;
  const int rest = it / p.splits;
  const int h = rest % p.num_kv_heads;
  const int rest2 = rest / p.num_kv_heads;
  const int rb = p.row_blocks - 1 - rest2 % p.row_blocks;  // heaviest row blocks first
  const int b = rest2 / p.row_blocks;
  // the sequence length: from the launch, or (a verify call) from device memory,
  // clamped to the block table (an out-of-range value is flagged once a sequence)
  int seq_len = p.seq_len;
  if (p.seq_len_dev) {
    seq_len = p.seq_len_dev[b];
    if (seq_len < 0 || seq_len > p.max_pages * kPage) {
      if (threadIdx.x == 0 && s == 0 && h == 0 && rb == p.row_blocks - 1) atomicOr(p.status, KVQ_DEV_BAD_SEQLEN);
      seq_len = seq_len < 0 ? 0 : p.max_pages * kPage;
    }
  }
  const int32_t* btab = p.block_table + (size_t)b * p.max_pages;  // this sequence's block table
  const int G = p.num_q_heads / p.num_kv_heads;
  const int TG = p.q_len * G;
  const size_t tok_base = (size_t)b * p.q_len;  // the sequence's first query token in q, out and the partials
  const int row0 = rb * kTcRows;
  const int last_tok = min(p.q_len - 1, (row0 + kTcRows - 1) / G);
  const int kmax = seq_len - p.q_len + last_tok + 1;  // keys the block's last row sees
  const int np_all = kmax > 0 ? (kmax + kPage - 1) / kPage : 0;
  const int pg0 = (int)((int64_t)s * np_all / p.splits);
  const int npg = (int)((int64_t)(s + 1) * np_all / p.splits) - pg0;
  const int nt = (npg + kTcPages - 1) / kTcPages;
  const int key_end = min(seq_len, (pg0 + npg) * kPage);  // keys of this range (exclusive)
  const uint32_t tmem = slot[0];
  volatile uint32_t* abort_flag = slot + 1;
  auto wait = [&](int b, uint32_t parity) -> bool {  // one thread
    if (*abort_flag) return false;
    if (mbar_wait(&bars[b], parity, kWaitLimitNs)) return true;
    atomicOr(p.status, KVQ_DEV_TIMEOUT);
    *abort_flag = 1;
    return false;
  };
  auto wait_warp = [&](int b, uint32_t parity) -> bool {  // a whole warp, one answer for all its lanes
    return __all_sync(0xffffffffu, wait(b, parity));
  };

  if (warp == 8) {
    // ================================================================== MMA issue
    if (lane == 0 && nt > 0) {
      bool ok = wait(kBarQ, 0);
      tc_fence_after();
      // step i: S(i) (K(i) ready), then P(i-1) V(i-1); S runs one tile ahead
      for (int i = 0; ok && i <= nt; ++i) {
        if (i < nt) {
          if (!wait(kBarK0 + (i & 1), (i >> 1) & 1)) break;
          tc_fence_after();
          const uint32_t ds = tmem + Lo::kTmemS + (uint32_t)(i & 1) * kTcKeys;
          const uint32_t kb = sbase + Lo::kKAt + (uint32_t)(i & 1) * Lo::kKBytes;
#pragma unroll
          for (int k = 0; k < KS; ++k) {  // k-step of 16 elements: 8 columns of Q
            const int a = k >> 2, kk = k & 3;
            const uint64_t bd = umma_desc_sw128(kb + a * kTcKeys * 128 + 32 * kk, 16, 1024);
            umma_f16_ta(ds, tmem + Lo::kTmemQ + 8 * k, bd, kIdescS, k > 0 ? 1u : 0u);
          }
          umma_commit(&bars[kBarS0 + (i & 1)]);
          umma_commit(&bars[kBarKF0 + (i & 1)]);
        }
        if (i > 0) {
          const int j = i - 1;
          if (!wait(kBarP0 + (j & 1), (j >> 1) & 1) || !wait(kBarV0 + (j & 1), (j >> 1) & 1)) break;
          tc_fence_after();
          const uint32_t vb = sbase + Lo::kVAt + (uint32_t)(j & 1) * Lo::kVBytes;
          const uint32_t pa = tmem + Lo::kTmemS + (uint32_t)(j & 1) * kTcKeys;  // P(j) over S(j): hi, then lo
#pragma unroll
          for (int k = 0; k < kTcKeys / 16; ++k) {
            const uint64_t bd = umma_desc_sw128(vb + 2 * k * Lo::kVSbo, Lo::kVLbo, Lo::kVSbo);
            umma_f16_ta(tmem + Lo::kTmemO, pa + 8 * k, bd, kIdescPV, (j > 0 || k > 0) ? 1u : 0u);
          }
          if constexpr (PLO) {
#pragma unroll
            for (int k = 0; k < kTcKeys / 16; ++k) {
              const uint64_t bd = umma_desc_sw128(vb + 2 * k * Lo::kVSbo, Lo::kVLbo, Lo::kVSbo);
              umma_f16_ta(tmem + Lo::kTmemO, pa + kTcKeys / 2 + 8 * k, bd, kIdescPV, 1u);
            }
          }
          umma_commit(&bars[kBarO0 + (j & 1)]);
        }
      }
      // every MMA this thread issued has completed before the TMEM is freed
      umma_commit(&bars[kBarFinal]);
      if (!mbar_wait(&bars[kBarFinal], 0, kWaitLimitNs)) atomicOr(p.status, KVQ_DEV_TIMEOUT);
    }
  } else if (warp >= 4) {
    // ================================================================== converters
    const int ct = threadIdx.x - 128;
    const int n = ct >> 1, half = ct & 1;  // key of the tile, half of its row
    constexpr int kRowBytes = T::kRow;     // code bytes of a key row
    constexpr int kHalfBytes = kRowBytes / 2;
    constexpr int kChunks = kHalfBytes / 16;  // 16-byte source chunks of a half row
    uint8_t* ktiles = smem + Lo::kKAt;
    uint8_t* vtiles = smem + Lo::kVAt;
    // pool row of key n of tile i (-1: a key past the range or the sequence, or a
    // bad page id), in two steps so that the block-table read can run ahead:
    // page_of(i) reads the page id, row_from(i, id) validates it
    auto in_range = [&](int i) {  // key n of tile i lies in the range and the sequence
      const int jp = i * kTcPages + (n >> 4);  // page of the range
      return jp < npg && (pg0 + jp) * kPage + (n & 15) < key_end;
    };
    auto page_of = [&](int i) -> int { return in_range(i) ? btab[pg0 + i * kTcPages + (n >> 4)] : -1; };
    auto row_from = [&](int i, int pg) -> int64_t {
      if (!in_range(i)) return -1;
      if (pg < 0 || pg >= p.num_pages) {
        if (half == 0 && (n & 15) == 0) atomicOr(p.status, KVQ_DEV_BAD_PAGE);
        return -1;
      }
      return ((int64_t)pg * p.num_kv_heads + h) * kPage + (n & 15);
    };
    auto load = [&](const uint8_t* base, int64_t ro, uint4 (&raw)[kChunks]) {
      const uint4* src = reinterpret_cast<const uint4*>(base + (ro >= 0 ? ro : 0) * kRowBytes + half * kHalfBytes);
#pragma unroll
      for (int u = 0; u < kChunks; ++u) raw[u] = ro >= 0 ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
    };
    // write a half row (raw codes of key n) as fp16 / bf16 into K tile buffer b (which = 0) or V
    auto put = [&](int which, int b, const uint4 (&raw)[kChunks], uint2 gsc) {
      uint8_t* ktile = ktiles + b * Lo::kKBytes;
      uint8_t* vtile = vtiles + b * Lo::kVBytes;
      if constexpr (FMT == KVQ_FMT_NVFP4) {
        // 16 bytes = 32 values = two scale groups; E2M1 x E4M3 is exact in fp16
        // (at most 6 significant bits, magnitudes 2^-10 .. 2688)
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
          const uint32_t sb = u < 2 ? gsc.x : gsc.y;  // group scale bytes 2u, 2u+1 of the half row
          const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t bsel = 2 * (u & 1) + (j >> 1);  // byte of sb holding this word's group
            const __half2 sdh = u32_as_h2(e4m3x2_to_h2(prmt(sb, 0u, bsel | (bsel << 4))));
            uint32_t f[4];
            e2m1x8_to_h2x4(w[j], f);
            const uint4 o = make_uint4(h2_as_u32(__hmul2(u32_as_h2(f[0]), sdh)), h2_as_u32(__hmul2(u32_as_h2(f[1]), sdh)),
                                       h2_as_u32(__hmul2(u32_as_h2(f[2]), sdh)), h2_as_u32(__hmul2(u32_as_h2(f[3]), sdh)));
            const int d0 = half * (D / 2) + 32 * u + 8 * j;
            if (which == 0) *reinterpret_cast<uint4*>(ktile + kmajor_off(n, d0, kTcKeys)) = o;
            else *reinterpret_cast<uint4*>(vtile + vtile_off<D>(n, d0)) = o;
          }
        }
      } else if constexpr (FMT == KVQ_FMT_INT8) {
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
          const uint32_t w[4] = {raw[u].x ^ 0x80808080u, raw[u].y ^ 0x80808080u, raw[u].z ^ 0x80808080u,
                                 raw[u].w ^ 0x80808080u};
          const uint4 lo = make_uint4(i8pair_to_h2<0x4140>(w[0]), i8pair_to_h2<0x4342>(w[0]),
                                      i8pair_to_h2<0x4140>(w[1]), i8pair_to_h2<0x4342>(w[1]));
          const uint4 hi = make_uint4(i8pair_to_h2<0x4140>(w[2]), i8pair_to_h2<0x4342>(w[2]),
                                      i8pair_to_h2<0x4140>(w[3]), i8pair_to_h2<0x4342>(w[3]));
          const int d0 = half * (D / 2) + 16 * u;
          if (which == 0) {
            *reinterpret_cast<uint4*>(ktile + kmajor_off(n, d0, kTcKeys)) = lo;
            *reinterpret_cast<uint4*>(ktile + kmajor_off(n, d0 + 8, kTcKeys)) = hi;
          } else {
            *reinterpret_cast<uint4*>(vtile + vtile_off<D>(n, d0)) = lo;
            *reinterpret_cast<uint4*>(vtile + vtile_off<D>(n, d0 + 8)) = hi;
          }
        }
      } else {  // BF16: 8 elements a chunk, copied as they are
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
          const int d0 = half * (D / 2) + 8 * u;
          if (which == 0) *reinterpret_cast<uint4*>(ktile + kmajor_off(n, d0, kTcKeys)) = raw[u];
          else *reinterpret_cast<uint4*>(vtile + vtile_off<D>(n, d0)) = raw[u];
        }
      }
    };
    // Loads run a tile ahead of the conversions: at the start of tile i the
    // converters issue K(i + 1) and V(i + 1) (two register sets a tensor, used in
    // turn) and read the page ids of tile i + 2, so that no code load waits for
    // its block-table read and every load has a whole tile to land.  Where two
    // sets a tensor would not fit in the registers (8-bit rows of 256 values and
    // wider), V(i) is issued at the start of tile i and K(i + 1) once K(i) is
    // written.
    constexpr bool kAhead = kChunks <= 4;
    constexpr bool kVAhead = !kAhead && kChunks <= 8;  // V alone a tile ahead
    uint4 rk0[kChunks], rv0[kChunks], rk1[kAhead ? kChunks : 1], rv1[(kAhead || kVAhead) ? kChunks : 1];
    int64_t ro = nt > 0 ? row_from(0, page_of(0)) : -1;
    // every key-mask entry of this warp starts full (published with K(0))
    uint32_t partial_slots = 0;  // ring slots whose entry holds a partial mask
    if (lane == 0)
      for (int sl = 0; sl < Lo::kScRing; ++sl) kmask[sl * 4 + (warp - 4)] = 0xFFFFu;
    int pg_next = nt > 1 ? page_of(1) : -1;  // page id of tile i + 1
    if (nt > 0) {
      load(p.k_codes, ro, rk0);
      if constexpr (kAhead || kVAhead) load(p.v_codes, ro, rv0);
    }
    auto step = [&](int i, uint4 (&rk)[kChunks], uint4 (&rv)[kChunks], uint4 (&rk_next)[kChunks],
                    uint4 (&rv_next)[kChunks]) -> bool {
      const int64_t ro_next = i + 1 < nt ? row_from(i + 1, pg_next) : -1;
      pg_next = i + 2 < nt ? page_of(i + 2) : -1;
      float ksv = 0.f, vsv = 0.f;
      uint2 kgs = make_uint2(0, 0), vgs = make_uint2(0, 0);  // NVFP4: this half row's group scale bytes
      if constexpr (FMT == KVQ_FMT_NVFP4) {
        if (ro >= 0) {  // D/32 scale bytes a half row: 8 at D = 256, 4 at D = 128
          if constexpr (D == 256) {
            kgs = __ldg(reinterpret_cast<const uint2*>(p.k_scales + ro * 16 + half * 8));
            vgs = __ldg(reinterpret_cast<const uint2*>(p.v_scales + ro * 16 + half * 8));
          } else {
            kgs.x = __ldg(reinterpret_cast<const uint32_t*>(p.k_scales + ro * 8 + half * 4));
            vgs.x = __ldg(reinterpret_cast<const uint32_t*>(p.v_scales + ro * 8 + half * 4));
          }
        }
      }
      if constexpr (FMT == KVQ_FMT_INT8) {
        if (ro >= 0 && half == 0) {
          ksv = __ldg(reinterpret_cast<const float*>(p.k_scales) + ro);
          vsv = __ldg(reinterpret_cast<const float*>(p.v_scales) + ro);
        }
      }
      if constexpr (kAhead) {
        if (i + 1 < nt) {
          load(p.k_codes, ro_next, rk_next);
          load(p.v_codes, ro_next, rv_next);
        }
      } else if constexpr (kVAhead) {
        if (i + 1 < nt) load(p.v_codes, ro_next, rv_next);
      } else {
        load(p.v_codes, ro, rv);
      }
      // K buffer i & 1 is free once S(i-2) is done
      if (i > 1 && !wait_warp(kBarKF0 + (i & 1), ((i - 2) >> 1) & 1)) return false;
      {
        // keys on a page whose id is out of the pool (keys past the range are cut
        // by the rows' limits): the softmax leaves them out, as the decode does.
        // A warp rewrites its mask entry only for such a tile, and once after it.
        const bool bad = ro < 0 && in_range(i);
        const int slot = i % Lo::kScRing;
        if (__any_sync(0xffffffffu, bad)) {
          uint32_t m = __ballot_sync(0xffffffffu, !bad) & 0x55555555u;  // half 0 lanes: one bit a key
          m = (m | (m >> 1)) & 0x33333333u;
          m = (m | (m >> 2)) & 0x0F0F0F0Fu;
          m = (m | (m >> 4)) & 0x00FF00FFu;
          m = (m | (m >> 8)) & 0x0000FFFFu;
          if (lane == 0) kmask[slot * 4 + (warp - 4)] = static_cast<uint16_t>(m);
          partial_slots |= 1u << slot;
        } else if (partial_slots & (1u << slot)) {
          if (lane == 0) kmask[slot * 4 + (warp - 4)] = 0xFFFFu;
          partial_slots &= ~(1u << slot);
        }
      }
      if constexpr (FMT == KVQ_FMT_INT8) {
        // both scales of the tile go out with K: the softmax reads them once S is
        // done.  Ring of three: the last reader of this slot, the softmax of tile
        // i-3, finished before P(i-3) V(i-3), which V(i-1) above waited for.
        if (half == 0) {
          ksc[(i % Lo::kScRing) * kTcKeys + n] = ksv * p.sm_scale_log2;  // the softmax's log2 factor folded in
          vsc[(i % Lo::kScRing) * kTcKeys + n] = vsv;
        }
      }
      put(0, i & 1, rk, kgs);
      fence_proxy_async_smem();  // the tile's bytes become visible to the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarK0 + (i & 1)]);
      if (!kAhead && i + 1 < nt) load(p.k_codes, ro_next, rk_next);  // rk_next is rk: after it is written
      // V buffer i & 1 is free once P(i-2) V(i-2) is done
      if (i > 1 && !wait_warp(kBarO0 + (i & 1), ((i - 2) >> 1) & 1)) return false;
      put(1, i & 1, rv, vgs);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarV0 + (i & 1)]);
      ro = ro_next;
      return true;
    };
    if constexpr (kAhead) {
      for (int i = 0; i < nt; i += 2) {  // the two register sets take turns
        if (!step(i, rk0, rv0, rk1, rv1)) break;
        if (i + 1 < nt && !step(i + 1, rk1, rv1, rk0, rv0)) break;
      }
    } else if constexpr (kVAhead) {
      for (int i = 0; i < nt; i += 2) {  // the two V register sets take turns; K has one
        if (!step(i, rk0, rv0, rk0, rv1)) break;
        if (i + 1 < nt && !step(i + 1, rk0, rv1, rk0, rv0)) break;
      }
    } else {
      for (int i = 0; i < nt; ++i)
        if (!step(i, rk0, rv0, rk0, rv0)) break;
    }
  } else {
    // ================================================================== softmax
    const int rl = threadIdx.x;  // row of the item (warp w: TMEM lanes 32w .. 32w+31)
    const int row = row0 + rl;
    const bool live = row < TG;
    const int ti = live ? row / G : 0, g = live ? row - (row / G) * G : 0;
    const uint32_t tq = tmem + ((uint32_t)(32 * warp) << 16);  // this warp's TMEM lanes
    // ---- q row -> Q in TMEM, this thread's lane (INT8: scaled by 2^k so its
    // largest |q| is in [2^14, 2^15)); column c holds elements 2c (low half), 2c + 1
    float row_scale = 1.f;
    {
      const uint4* qrow =
          reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                         ((tok_base + ti) * p.num_q_heads + h * G + g) * D);
      float up = 1.f;
      if constexpr (!kBf16) {
        float amax = 0.f;
        for (int c8 = 0; c8 < D / 8; ++c8) {
          const uint4 v = live ? __ldg(qrow + c8) : make_uint4(0, 0, 0, 0);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xFFFF0000u))));
        }
        int k = 0;
        if (amax > 0.f) {
          int ex;
          frexpf(amax, &ex);
          k = min(126, max(-126, 15 - ex));
        }
        up = pow2f(k);
        row_scale = pow2f(-k);
      }
#pragma unroll 1
      for (int c16 = 0; c16 < D / 16; ++c16) {  // 16 elements: 8 columns
        uint32_t cols[8];
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          const uint4 v = live ? __ldg(qrow + 2 * c16 + h8) : make_uint4(0, 0, 0, 0);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            cols[4 * h8 + e] = kBf16 ? w[e]
                                     : h2_as_u32(__floats2half2_rn(__uint_as_float(w[e] << 16) * up,
                                                                   __uint_as_float(w[e] & 0xFFFF0000u) * up));
        }
        tmem_st8(tq + Lo::kTmemQ + 8 * c16, cols);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarQ]);
    }
    const int lim = live ? max(0, seq_len - p.q_len + ti + 1) : 0;  // keys this row sees (exclusive)
    const int kend = min(lim, key_end);
    // logit (log2 units) = S x kfac x rs with rs = the row's power of two (q was
    // scaled by 1/rs to be exact in fp16; 1 for BF16): INT8 kfac = the key's scale
    // x sm_scale x log2(e) (folded in by the converters), otherwise kfac =
    // sm_scale x log2(e) (NVFP4: x 1 / gs_K, the tiles hold values x gs).  kfac
    // carries the sign of sm_scale and rs > 0, so max(S x kfac) x rs is the
    // maximum logit.
    const float rs = row_scale;
    const float kconst = p.sm_scale_log2 * p.k_gs_inv;  // kfac of the non-INT8 formats
    float m_run = -INFINITY, l_run = 0.f;

    int done = 0;  // tiles completed
    for (int i = 0; i < nt; ++i) {
      if (!wait_warp((i & 1) ? kBarS1 : kBarS0, (i >> 1) & 1)) break;
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld32(tq + Lo::kTmemS + (uint32_t)(i & 1) * kTcKeys, sv[0]);
      tmem_ld32(tq + Lo::kTmemS + (uint32_t)(i & 1) * kTcKeys + 32, sv[1]);
      tmem_ld_wait();
      const int tok0 = (pg0 + i * kTcPages) * kPage;
      const float* ks = ksc + (i % Lo::kScRing) * kTcKeys;
      const float* vs = vsc + (i % Lo::kScRing) * kTcKeys;
      // pass 1: z = S x kfac (the logit before the row factor rs > 0) and the tile
      // maximum (four independent chains); only a tile that crosses the row's
      // limit, or holds keys that were not read (a bad page id), is masked
      const uint64_t km = *reinterpret_cast<const uint64_t*>(kmask + (i % Lo::kScRing) * 4);
      float z[kTcKeys];
#pragma unroll
      for (int t = 0; t < kTcKeys; ++t) z[t] = __uint_as_float(sv[t >> 5][t & 31]);
      float mxs[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      const int nvis = kend - tok0;  // visible keys of this tile for this row
#pragma unroll
      for (int c4 = 0; c4 < kTcKeys / 4; ++c4) {
        float kk[4] = {kconst, kconst, kconst, kconst};
        if constexpr (FMT == KVQ_FMT_INT8) {
          const float4 k4 = *reinterpret_cast<const float4*>(ks + 4 * c4);
          kk[0] = k4.x; kk[1] = k4.y; kk[2] = k4.z; kk[3] = k4.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 4 * c4 + e;
          float zz = z[t] * kk[e];
          if (nvis < kTcKeys) zz = t < nvis ? zz : -INFINITY;
          z[t] = zz;
          mxs[e] = fmaxf(mxs[e], zz);
        }
      }
      if (km != ~0ull) {  // keys that were not read (the same for the whole tile): out, and the maximum again
#pragma unroll
        for (int e = 0; e < 4; ++e) mxs[e] = -INFINITY;
#pragma unroll
        for (int t = 0; t < kTcKeys; ++t) {
          if (!((km >> t) & 1ull)) z[t] = -INFINITY;
          mxs[t & 3] = fmaxf(mxs[t & 3], z[t]);
        }
      }
      const float mx = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])) * rs;  // log2 units
      const bool resc = m_run != -INFINITY && mx > m_run + kTcRescale;
      if (__any_sync(0xffffffffu, resc)) {
        // O is rescaled once it holds P(i-1) V(i-1), before P(i) V(i) adds to it
        if (i > 0) {
          if (!wait_warp(kBarO0 + ((i - 1) & 1), ((i - 1) >> 1) & 1)) break;
          tc_fence_after();
        }
        const float alpha = resc ? exp2f(m_run - mx) : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tq + Lo::kTmemO + 32 * c, ov);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(tq + Lo::kTmemO + 32 * c, ov);
        }
        tmem_st_wait();
        if (resc) {
          l_run *= alpha;
          m_run = mx;
        }
      }
      if (m_run == -INFINITY) m_run = mx;  // first visible keys (still -inf if none)
      // P(i) goes over S(i), which this thread has read.  The last reader of those
      // columns before S(i), P(i-2) V(i-2), was issued before S(i), so the commit
      // that reported S(i) done covered it too.
      const uint32_t tp = tq + Lo::kTmemS + (uint32_t)(i & 1) * kTcKeys;  // this row's P(i): hi, lo 32 columns on
      // pass 2: p = 2^(z - m) <= 2^8 (ex2.approx.ftz: results below 2^-126 are 0,
      // a masked key's z = -inf gives exactly 0), P' = p v_scale, packed hi (+ lo)
      float psums[4] = {0.f, 0.f, 0.f, 0.f};
      const float msub = m_run == -INFINITY ? 0.f : m_run;  // a row with no visible key: every z is -inf
      uint32_t ph[8], pl[8];  // two groups of 8 keys: 8 words of key pairs, hi and lo
#pragma unroll
      for (int c8 = 0; c8 < kTcKeys / 8; ++c8) {
        uint32_t* hw = ph + 4 * (c8 & 1);
        [[maybe_unused]] uint32_t* lw = pl + 4 * (c8 & 1);
        float v8[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
        if constexpr (FMT == KVQ_FMT_INT8) {
          const float4 va = *reinterpret_cast<const float4*>(vs + 8 * c8);
          const float4 vb = *reinterpret_cast<const float4*>(vs + 8 * c8 + 4);
          v8[0] = va.x; v8[1] = va.y; v8[2] = va.z; v8[3] = va.w;
          v8[4] = vb.x; v8[5] = vb.y; v8[6] = vb.z; v8[7] = vb.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float pv[2];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const int t = 8 * c8 + 2 * e + q2;
            float pr;
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(pr) : "f"(fmaf(z[t], rs, -msub)));
            psums[q2 + 2 * (e & 1)] += pr;
            // the converters wrote v scale 0 for every key past the range or the
            // sequence, so every scale here is finite and a masked key gives 0
            pv[q2] = FMT == KVQ_FMT_INT8 ? pr * v8[2 * e + q2] : pr;
          }
          if constexpr (kBf16) {
            const __nv_bfloat162 hv = __floats2bfloat162_rn(pv[0], pv[1]);
            hw[e] = *reinterpret_cast<const uint32_t*>(&hv);
            if constexpr (PLO) {
              const __nv_bfloat162 lv = __floats2bfloat162_rn(pv[0] - __low2float(hv), pv[1] - __high2float(hv));
              lw[e] = *reinterpret_cast<const uint32_t*>(&lv);
            }
          } else {
            const __half2 hv = __floats2half2_rn(pv[0], pv[1]);
            hw[e] = h2_as_u32(hv);
            if constexpr (PLO) lw[e] = h2_as_u32(__floats2half2_rn(pv[0] - __low2float(hv), pv[1] - __high2float(hv)));
          }
        }
        if (c8 & 1) {  // keys 16 (c8 / 2) .. +15: columns 8 (c8 / 2) .. +7
          tmem_st8(tp + 8 * (c8 >> 1), ph);
          if constexpr (PLO) tmem_st8(tp + kTcKeys / 2 + 8 * (c8 >> 1), pl);
        }
      }
      l_run += (psums[0] + psums[1]) + (psums[2] + psums[3]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarP0 + (i & 1)]);
      done = i + 1;
    }
    // ================================================================ epilogue
    bool have_o = done == nt && nt > 0;
    if (have_o) {
      have_o = wait_warp(kBarO0 + ((nt - 1) & 1), ((nt - 1) >> 1) & 1);
      tc_fence_after();
    }
    if (done != nt) {  // aborted: this row's result is not valid
      m_run = -INFINITY;
      l_run = 0.f;
    }
    constexpr float kLn2 = 0.69314718055994530942f;
    const bool any = m_run != -INFINITY && l_run > 0.f;
    const float inv = any ? p.v_gs_inv / l_run : 0.f;
    const float lse = any ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
    const bool direct = p.splits == 1;
    const size_t qh = (size_t)h * G + g;
    const size_t orow =
        direct ? (tok_base + ti) * p.num_q_heads + qh : ((tok_base + ti) * p.splits + s) * p.num_q_heads + qh;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t ov[32];
      if (__any_sync(0xffffffffu, have_o)) {
        tmem_ld32(tq + Lo::kTmemO + 32 * c, ov);
        tmem_ld_wait();
      }
      if (!live) continue;
#pragma unroll
      for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(have_o ? __uint_as_float(ov[e]) * inv : 0.f);
      if (direct && p.out_bf16) {
        uint4* ob = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * D + 32 * c);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(ov[8 * v4 + 2 * e]),
                                                            __uint_as_float(ov[8 * v4 + 2 * e + 1]));
            w[e] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          ob[v4] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        uint4* of = reinterpret_cast<uint4*>((direct ? reinterpret_cast<float*>(p.out) : p.o_part) + orow * D + 32 * c);
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4) of[v4] = make_uint4(ov[4 * v4], ov[4 * v4 + 1], ov[4 * v4 + 2], ov[4 * v4 + 3]);
      }
    }
    if (live) {
      if (direct) {
        if (p.lse_out) p.lse_out[orow] = lse;
      } else {
        p.lse_part[orow] = lse;
      }
    }
  }
  // all TMEM reads and MMAs are complete: free the columns
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, Lo::kTmemCols);
  }
}

template <int FMT, int D>
cudaError_t launch_tc_t(const PrefillParams& p, int grid, cudaStream_t stream) {
  using Lo = TcLayout<FMT, D>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = Lo::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.out_bf16 ? cudaLaunchKernelEx(&cfg, prefill_tc_kernel<FMT, D, false>, p)
                    : cudaLaunchKernelEx(&cfg, prefill_tc_kernel<FMT, D, true>, p);
}

template <int FMT, int D>
PrefillInstance tc_instance_of() {
  using Lo = TcLayout<FMT, D>;
  return PrefillInstance{{reinterpret_cast<const void*>(&prefill_tc_kernel<FMT, D, true>),
                          reinterpret_cast<const void*>(&prefill_tc_kernel<FMT, D, false>)},
                         Lo::kSmemBytes,
                         kTcThreads,
                         0,
                         kTcRows};
}

}  // namespace

bool prefill_tc_instance(int format, int head_dim, PrefillInstance* out) {
  if (format == KVQ_FMT_NVFP4 && head_dim == 256) *out = tc_instance_of<KVQ_FMT_NVFP4, 256>();
  else if (format == KVQ_FMT_NVFP4 && head_dim == 128) *out = tc_instance_of<KVQ_FMT_NVFP4, 128>();
  else if (format == KVQ_FMT_INT8 && head_dim == 256) *out = tc_instance_of<KVQ_FMT_INT8, 256>();
  else if (format == KVQ_FMT_INT8 && head_dim == 128) *out = tc_instance_of<KVQ_FMT_INT8, 128>();
  else if (format == KVQ_FMT_BF16 && head_dim == 256) *out = tc_instance_of<KVQ_FMT_BF16, 256>();
  else if (format == KVQ_FMT_BF16 && head_dim == 128) *out = tc_instance_of<KVQ_FMT_BF16, 128>();
  else return false;
  return true;
}

cudaError_t launch_prefill_tc(int format, int head_dim, const PrefillParams& p, int grid, cudaStream_t stream) {
  if (format == KVQ_FMT_NVFP4 && head_dim == 256) return launch_tc_t<KVQ_FMT_NVFP4, 256>(p, grid, stream);
  if (format == KVQ_FMT_NVFP4 && head_dim == 128) return launch_tc_t<KVQ_FMT_NVFP4, 128>(p, grid, stream);
  if (format == KVQ_FMT_INT8 && head_dim == 256) return launch_tc_t<KVQ_FMT_INT8, 256>(p, grid, stream);
  if (format == KVQ_FMT_INT8 && head_dim == 128) return launch_tc_t<KVQ_FMT_INT8, 128>(p, grid, stream);
  if (format == KVQ_FMT_BF16 && head_dim == 256) return launch_tc_t<KVQ_FMT_BF16, 256>(p, grid, stream);
  if (format == KVQ_FMT_BF16 && head_dim == 128) return launch_tc_t<KVQ_FMT_BF16, 128>(p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
