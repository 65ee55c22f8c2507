// decode.cuh — split-KV GQA decode attention over a paged INT8 / NVFP4 / BF16 cache.
//
// What it computes: for every (sequence b, query head g) the softmax-weighted sum
// of the dequantized V rows, with logits sm_scale * q . k_hat over the sequence's
// tokens (split-KV / flash-decoding: "long-context-attention-and-lessons", section
// "Give more GPU workers a piece of the attention calculation").  Codes are
// dequantized in registers and never written back as a converted copy
// ("half-the-memory-int8-kv-cache", section "Read the compressed cache without
// copying it first").  One loaded page serves the whole GQA group ("Smaller KV
// cache, faster first token", section "Lever two": one KV block is loaded once
// for a whole group of query heads).
//
// Work item: one split (a range of whole pages) of one sequence for a group of
// HG consecutive KV heads, HG = gcd(Hkv, CW) (or a divisor of it that leaves the
// ring at least two stages), where CW is the number of consumer warps (8 at
// D = 256, 12 at D = 128).  CTAs are persistent, one per SM: the host planner
// packs the items onto the CTAs (longest first, each to the least-loaded CTA)
// and every CTA works through its list, so a batch of uneven sequences runs in
// one wave; each CTA's first item descriptor sits at a fixed place in the plan.
// The pool keeps the KV heads of a page next to each other, so the HG heads'
// code blocks of a page are one contiguous region and travel as ONE TMA box per
// tensor (16 KB at D = 256 INT8 with 4 heads); a 1-D bulk copy brings their
// scales.  Few large copies per page keep the producers ahead of the consumers.
// A launch sequence may also be one query token of a verify call (several
// query tokens a cache sequence, causal): see seq_len below.
//
//   * warps CW..CW+3 (2 or 4 of them produce): producer i walks every NP-th page
//     of the item through the block table (page ids staged in shared memory 32
//     at a time by its warp); its lane 0, per page, waits for the stage to be
//     free, then issues the K and V boxes (128-byte swizzle) and the two scale
//     copies, completing on the stage's mbarrier (expect-tx bytes).  Several
//     producers share the issuing because one thread issues only about one copy
//     per 300 ns.  The ring keeps at most kMaxInflight bytes in flight.
//   * warps 0..CW-1 (consumers): warp w owns KV head w % HG and, if CW / HG > 1,
//     every (CW/HG)-th page.  Per page (16 tokens) a warp computes S = q K^T for
//     its G <= 8 query heads with mma.m16n8k16 (heads are the M rows, tokens the N
//     columns, D the reduction), runs the online softmax on the accumulator
//     fragment, and accumulates O^T = V^T P'^T (D is the M dimension, heads the N
//     columns, tokens the reduction), so that S's accumulator layout is directly
//     P's operand layout.  Integer codes enter the tensor cores as exact f16
//     integers; the per-token INT8 scales are applied to the logits (K) and folded
//     into P (V); NVFP4 group scales multiply the operands (products of an E2M1
//     and an E4M3 value are exact in f16).  P' is split into hi + lo halves of two
//     MMAs, so P carries ~22 bits.
//   * registers: the producer warpgroup gives registers back (setmaxnreg) and
//     the consumer warpgroups take them (INT8 / BF16; NVFP4 keeps the launch
//     split).
//   * epilogue: the other warps of a head leave their (m, l, O) in the idle ring
//     and the head's first warp combines them; it stages the head's query rows
//     and writes them with one bulk copy — `out` directly for a sequence with one
//     split, otherwise the (o, lse) partials the merge kernel combines.
//   * start-up: the kernel is a programmatic dependent of the preceding kernel;
//     with KVQ_EARLY_START it reads the plan and page ids before waiting for it.
//
// All waits are bounded (%globaltimer); on timeout the kernel sets
// KVQ_DEV_TIMEOUT in the status word and stops instead of spinning.
#pragma once

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

constexpr int kPage = 16;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kMaxStages = 32;
constexpr int kMaxInflight = 160 * 1024;  // ring bytes a CTA keeps in flight
constexpr uint64_t kStartPaceNs = 500;    // start-up pacing between producers (first page of a CTA)

template <int FMT, int D>
struct DecodeTraits;

template <int D>
struct DecodeTraits<KVQ_FMT_INT8, D> {
  static constexpr bool kBf16Mma = false;
  static constexpr int kRow = D;        // code bytes per token row
  static constexpr int kScaleRow = 4;   // scale bytes per token row (one fp32)
};

template <int D>
struct DecodeTraits<KVQ_FMT_INT8_G32, D> {
  static constexpr bool kBf16Mma = false;
  static constexpr int kRow = D;
  static constexpr int kScaleRow = 4 * (D / 32);  // one fp32 per 32 elements (group-major in the block)
};

// INT8 codes (one scale per row or per 32 elements): the same code paths
template <int FMT>
__host__ __device__ constexpr bool int8_codes() { return FMT == KVQ_FMT_INT8 || FMT == KVQ_FMT_INT8_G32; }

template <int D>
struct DecodeTraits<KVQ_FMT_BF16, D> {
  static constexpr bool kBf16Mma = true;
  static constexpr int kRow = 2 * D;
  static constexpr int kScaleRow = 0;
};

template <int D>
struct DecodeTraits<KVQ_FMT_NVFP4, D> {
  static constexpr bool kBf16Mma = false;
  static constexpr int kRow = D / 2;        // two E2M1 codes a byte
  static constexpr int kScaleRow = D / 16;  // one E4M3 byte per 16 elements
};

// consumer warps per CTA: 8 at D = 256 (+1 producer = 9 warps: at most 3 per
// SM sub-partition, so <= 168 registers a thread) and 12 at D = 128 (13 warps:
// <= 128 registers, enough at D = 128).
template <int D>
constexpr int consumer_warps() { return D == 256 ? 8 : 12; }

template <int FMT, int D>
struct DecodeLayout {
  using T = DecodeTraits<FMT, D>;
  static constexpr int kCW = consumer_warps<D>();
  static constexpr int kMaxProducers = 4;  // producer warps (a thread issues one copy per ~300 ns)
  static constexpr int kThreads = (kCW + kMaxProducers) * 32;
  // Registers: the kernel launches with kLaunchRegs a thread (all of the SM's
  // 64K registers); the producer warpgroup then gives registers back
  // (setmaxnreg.dec to kProducerRegs) and the consumer warpgroups take them
  // (setmaxnreg.inc to kConsumerRegs).  The split never asks for more than the
  // launch allocation, and the host refuses to launch a build whose register
  // count differs from kLaunchRegs.
  // (NVFP4 keeps the launch allocation everywhere: its consumer code compiles
  // better without the split.)
  static constexpr bool kRegSplit = FMT != KVQ_FMT_NVFP4;
  static constexpr int kLaunchRegs = 65536 / kThreads / 8 * 8;
  static constexpr int kProducerRegs = kRegSplit ? (D == 256 ? 104 : 56) : kLaunchRegs;
  static constexpr int kConsumerRegs =
      ((kLaunchRegs * kThreads - kProducerRegs * kMaxProducers * 32) / (kCW * 32) / 8 * 8) > 256
          ? 256
          : ((kLaunchRegs * kThreads - kProducerRegs * kMaxProducers * 32) / (kCW * 32) / 8 * 8);
  static_assert(kCW % 4 == 0 && kMaxProducers == 4, "warpgroup-aligned roles");
  static_assert(kConsumerRegs * kCW * 32 + kProducerRegs * kMaxProducers * 32 <= kLaunchRegs * kThreads,
                "register split exceeds the launch allocation");
  static constexpr int kHeadCode = kPage * T::kRow;        // one head's K (or V) code block of a page
  static constexpr int kHeadScale = kPage * T::kScaleRow;  // one head's K (or V) scale block of a page
  static constexpr int kKSteps = D / 16;
  static constexpr int kMTiles = D / 16;
  // q fragments of one KV head (shared by that head's warps):
  // [k-step][dA / dB part][8 head rows][8 halves]
  static constexpr int kQBytes = kKSteps * 2 * 128;
  // Shared memory after the 1024-byte alignment slack: the stage ring and then
  // one q tile per head of the group (kAvail bytes together; the ring gets what
  // the group's hg tiles leave), then the barriers and the page-id buffer.
  static constexpr int kIdBytes = kMaxProducers * 2 * 32 * 4;
  static constexpr int kBadBytes = kMaxStages * 4;  // per stage: its page id was out of range
  static constexpr int kAvail = (227 * 1024 - 1024 - 2 * kMaxStages * 8 - kIdBytes - kBadBytes) / 1024 * 1024;
  static constexpr int kSmemBytes = 1024 + kAvail + 2 * kMaxStages * 8 + kIdBytes + kBadBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static __host__ __device__ constexpr int ring_bytes(int hg) { return (kAvail - hg * kQBytes) / 1024 * 1024; }
  // the smallest ring (a group of kCW heads): the epilogue's buffers fit in any
  static constexpr int kRingBytes = (kAvail - kCW * kQBytes) / 1024 * 1024;
  // epilogue exchange in the ring: each warp other than a head's first leaves its
  // accumulators (one float4 per lane and m-tile) and (m, l) of 8 head rows
  static constexpr int kPartOBytes = kMTiles * 32 * 16;
  static constexpr int kExchangeBytes = (kCW - 1) * (kPartOBytes + 8 * 8);
  // then one output staging block per head of the group: 8 rows of D fp32
  static constexpr int kStageAt = (kExchangeBytes + 127) / 128 * 128;
  static constexpr int kStageBytes = 8 * D * 4;
  static_assert(kStageAt + kCW * kStageBytes <= kRingBytes, "epilogue exchange and staging must fit in the ring");
};

// Producer warps and stage count for a head group of `hg` heads.  A single
// thread issues about one copy per 300 ns whatever its size, so several producer
// warps share the issuing: page i of an item is issued by producer i % NP and
// consumed by the head's warp i % WPH (WPH = warps per head).  The stage count is
// as large as the ring and kMaxInflight allow (at most kMaxStages) and a multiple
// of both, so
// within an item every stage has a fixed producer and a fixed set of consumer
// warps, each of which handled the stage's previous page itself before waiting on
// the next one: a parity wait can never be satisfied by a barrier that is still
// two phases behind.  (Between items the CTA synchronizes, so every stage is idle.)
template <int FMT, int D>
__host__ __device__ inline int decode_producers(int hg) {
  const int wph = DecodeLayout<FMT, D>::kCW / hg;
  return wph == 1 ? 2 : (wph == 2 ? 4 : (wph <= 4 ? wph : (wph % 4 == 0 ? 4 : 3)));
}

template <int FMT, int D>
__host__ __device__ inline int decode_stage_unit(int hg) {
  const int wph = DecodeLayout<FMT, D>::kCW / hg;
  const int np = decode_producers<FMT, D>(hg);
  return wph > np ? wph : np;  // wph and np divide each other
}

template <int FMT, int D>
__host__ __device__ inline int decode_stages(int hg) {
  using Lo = DecodeLayout<FMT, D>;
  const int unit = decode_stage_unit<FMT, D>(hg);
  const int stage = 2 * hg * (Lo::kHeadCode + Lo::kHeadScale);
  // at most kMaxInflight bytes a CTA: with every CTA asking for its whole ring at
  // the start, a deeper ring only delays each CTA's first page (measured: 6
  // stages of 33 KB took 1.6 us longer than 4 on the 32K batch-1 workload)
  int n = Lo::ring_bytes(hg) / stage;
  if (n > kMaxInflight / stage) n = kMaxInflight / stage;
  n = n < kMaxStages ? n : kMaxStages;
  return n / unit * unit;  // 0 if fewer than `unit` stages fit: such a group is not used
}

// Largest head group (a divisor of gcd(Hkv, CW)) whose ring holds at least two
// stages and one per producer / consumer group.  0 if none does.
template <int FMT, int D>
inline int decode_head_group(int hkv) {
  using Lo = DecodeLayout<FMT, D>;
  int g = hkv, b = Lo::kCW;
  while (b) {
    const int t = g % b;
    g = b;
    b = t;
  }
  for (int hg = g; hg >= 1; --hg) {
    if (g % hg) continue;
    const int nst = decode_stages<FMT, D>(hg);
    const int unit = decode_stage_unit<FMT, D>(hg);
    if (nst >= 2 && nst >= unit) return hg;
  }
  return 0;
}

// byte address (shared window) of 16-byte chunk `chunk` (0..kRow/16-1) of token
// row t in a swizzled head block starting at `block` (1024-byte aligned): the
// block is [row half][16 rows][128 bytes], chunk index XOR-ed with t % 8.
__device__ __forceinline__ uint32_t swz(uint32_t block, int t, int chunk) {
  return block + (chunk >> 3) * (kPage * 128) + t * 128 + (((chunk & 7) ^ (t & 7)) << 4);
}

// The same for a head block of any row size: rows of 128 bytes or more as above;
// 64-byte rows (NVFP4 at D = 128) travel as 8 rows of 128 bytes, each holding a
// token pair (token t is the low or high half of row t / 2), under the same
// 128-byte swizzle.
template <int ROW>
__device__ __forceinline__ uint32_t swz_row(uint32_t block, int t, int chunk) {
  if constexpr (ROW >= 128) return swz(block, t, chunk);
  else return swz(block, t >> 1, 4 * (t & 1) + chunk);
}

__device__ __forceinline__ float pow2f(int k) { return __int_as_float((127 + k) << 23); }  // k in [-126, 127]

// PLO: the P' operand carries a lo term (fp32 output); the launcher picks the
// instance from the output type, so the choice costs nothing inside the page loop.
template <int FMT, int D, bool PLO>
__global__ void __launch_bounds__(DecodeLayout<FMT, D>::kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeParams p) {
  using T = DecodeTraits<FMT, D>;
  using Lo = DecodeLayout<FMT, D>;
  constexpr int CW = Lo::kCW;
  constexpr int KS = Lo::kKSteps;

  // the merge kernel is launched as a programmatic dependent: let it be scheduled
  // (it waits for this grid's results before reading them)
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // This grid is itself launched as a programmatic dependent of the preceding
  // kernel.  Unless the caller promised that the plan and block tables are not
  // written by that kernel, wait for it before reading anything; otherwise the
  // producers wait just before their first copy and the consumers before they
  // read q and the sequence lengths.
  if (!p.early_start) asm volatile("griddepcontrol.wait;" ::: "memory");
  const int HG = p.heads_per_cta;
  const int WPH = CW / HG;
  const int NST = decode_stages<FMT, D>(HG);
  if (HG < 1 || CW % HG != 0 || NST < 2 || NST < decode_stage_unit<FMT, D>(HG)) {  // host picks valid groups
    if (threadIdx.x == 0) atomicOr(p.status, KVQ_DEV_BAD_PLAN);
    return;
  }
  const int stage_code = 2 * HG * Lo::kHeadCode;
  const int stage_scale = 2 * HG * Lo::kHeadScale;
  const int Hkv = p.num_kv_heads;
  const int NHG = Hkv / HG;
  const int G = p.num_q_heads / Hkv;

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (128-byte swizzle), derived from the shared array by
  // pointer arithmetic so that every access through it stays a shared-memory one
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* codes = smem;                                   // NST x [K heads][V heads]
  uint8_t* scales = smem + NST * stage_code;               // NST x [K heads][V heads]
  uint8_t* qfrag = smem + Lo::ring_bytes(HG);              // HG x kQBytes
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lo::kAvail);
  uint64_t* empty = full + kMaxStages;
  int* pid_s = reinterpret_cast<int*>(empty + kMaxStages);  // [producer][2][32] page ids
  // per stage, set by its producer before the stage's full barrier completes:
  // the page id was out of range, so the consumers mask every token of it
  int* bad_s = pid_s + Lo::kIdBytes / 4;

  // ---- plan: split offsets [batch + 1], C = gridDim.x, then (16-byte aligned) the
  // first item descriptor of every CTA, the CTAs' offsets into the list of their
  // further items, and that list.  A CTA reads its first descriptor at a fixed
  // place, so its producers can ask for page ids after one dependent load.
  const int C = static_cast<int>(gridDim.x);
  const int A = (p.batch + 2 + 3) & ~3;
  const int4* firsts = reinterpret_cast<const int4*>(p.plan + A);
  const int32_t* roff = p.plan + A + 4 * C;
  const int4* rest = reinterpret_cast<const int4*>(p.plan + ((A + 5 * C + 1 + 3) & ~3));
  const int n_items = p.total_splits * NHG;
  const int4 d0 = firsts[blockIdx.x];
  const int r0 = roff[blockIdx.x];
  const int r1 = roff[blockIdx.x + 1];
  if (p.plan[p.batch + 1] != C || r0 < 0 || r1 < r0 || r1 > n_items - C) {
    if (threadIdx.x == 0) atomicOr(p.status, KVQ_DEV_BAD_PLAN);
    return;
  }
  const int cnt = 1 + (r1 - r0);  // items of this CTA: d0, then rest[r0 .. r1)

  // Item = (sequence, split, head group, page range) of a descriptor
  // {b, split, first page, n | direct << 23 | group << 24}; identical in every thread.
  struct Item {
    int b, split, hg, L, page_begin, n;
    bool direct;  // the sequence has a single split: write `out` directly
  };
  auto unpack = [&](const int4 d, Item& w) -> bool {
    w.b = d.x;
    w.split = d.y;
    w.page_begin = d.z;
    w.n = d.w & 0x7FFFFF;
    w.direct = ((d.w >> 23) & 1) != 0;
    w.hg = static_cast<int>(static_cast<uint32_t>(d.w) >> 24);
    w.L = 0;
    return w.b >= 0 && w.b < p.batch && w.split >= 0 && w.split < p.total_splits && w.hg < NHG &&
           w.page_begin >= 0 && w.page_begin <= p.max_pages - w.n;
  };
  // Sequence b of the launch is query token i = b % q_len of cache sequence
  // b / q_len (one token a sequence when decoding).  Token i of T sits at position
  // L - T + i of its sequence and sees tokens 0 .. L - T + i: causal verification
  // of T proposed tokens whose K/V are the last T entries of the cache.
  auto seq_len = [&](int b) -> int {  // visible tokens of launch sequence b, clamped to its block table
    const int rb = b / p.q_len;
    int L = p.seq_lens[rb];
    if (L < 0 || L > p.max_pages * kPage) {
      if (threadIdx.x == 0) atomicOr(p.status, KVQ_DEV_BAD_SEQLEN);
      L = L < 0 ? 0 : p.max_pages * kPage;
    }
    L -= p.q_len - 1 - (b - rb * p.q_len);
    return L > 0 ? L : 0;
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  __shared__ int abort_flag;
  __shared__ int4 next_desc;
  __shared__ int4 cur_desc;

  // consumer identity (used only by consumer warps)
  const int hl = warp % HG;   // head within the group
  const int grp = warp / HG;  // page subset of this head's warps
  const int r = lane >> 2;    // head row of S / P, token group of V^T fragments
  const int c = lane & 3;
  const bool head_ok = r < G;

  // q of an item, as raw bf16 pairs in fragment column order (see below); issued
  // before the producer starts streaming so these loads are not queued behind it.
  uint32_t qraw[KS][2];
  auto load_q = [&](const Item& w) {
    const int hq = (w.hg * HG + hl) * G + r;
    const __nv_bfloat16* qrow =
        reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t)w.b * p.num_q_heads + hq) * D;
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      int dA, dB;
      if constexpr (int8_codes<FMT>()) {
        dA = 16 * j + 4 * c;
        dB = dA + 2;
      } else if constexpr (FMT == KVQ_FMT_BF16) {
        dA = 16 * j + 2 * c;
        dB = dA + 8;
      } else {
        dA = 32 * (j >> 1) + 8 * c + 4 * (j & 1);
        dB = dA + 2;
      }
      qraw[j][0] = head_ok ? *reinterpret_cast<const uint32_t*>(qrow + dA) : 0u;
      qraw[j][1] = head_ok ? *reinterpret_cast<const uint32_t*>(qrow + dB) : 0u;
    }
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], HG);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();  // before any load that depends on the descriptor: producers go on at once

  Item first;
  const bool first_ok = unpack(d0, first);
  if (warp < CW && p.early_start) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp < CW && first_ok) {
    first.L = seq_len(first.b);
    load_q(first);
  }

  const int NP = decode_producers<FMT, D>(HG);
  const int sync_threads = (CW + NP) * 32;  // consumers + active producers (item boundaries)
  if (warp >= CW) {
    // ================================================================ producers
    if constexpr (Lo::kRegSplit) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Lo::kProducerRegs));
    const int pi = warp - CW;
    if (pi >= NP) return;
    bool ok = true;
    int gidx = 0;                 // pages of this CTA before the current item
    int last_first = 0, last_n = 0;
    int* ids = pid_s + pi * 64;
    // this producer's pages of an item are idx = pi + NP*j; page_id(w, j) is the
    // validated page id of its page j (or -1)
    auto mine_of = [&](const Item& w) { return w.n > pi ? (w.n - pi + NP - 1) / NP : 0; };
    auto page_id = [&](const Item& w, int j) -> int {
      int v = -1;
      if (j < mine_of(w)) {
        v = p.block_tables[(size_t)(w.b / p.q_len) * p.max_pages + w.page_begin + pi + NP * j];
        if (v < 0 || v >= p.num_pages) {
          atomicOr(p.status, KVQ_DEV_BAD_PAGE);
          v = -1;
        }
      }
      return v;
    };
    Item w = first;
    bool valid = first_ok;
    int v0 = valid ? page_id(w, lane) : -1;  // ids of the item's first 32 pages of this producer
    if (p.early_start) asm volatile("griddepcontrol.wait;" ::: "memory");
    // Start-up pacing: producer i issues its first page i x 500 ns after producer
    // 0.  Every CTA asks for its whole ring at once otherwise, and the DRAM serves
    // that burst interleaved, so each CTA's first page (the one its consumers
    // wait for) lands last; paced, the first wave is one page a CTA.  Measured
    // on the 32K batch-1 workload: the call 0.5 us shorter.
    if (pi > 0 && lane == 0) {
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < (uint64_t)pi * kStartPaceNs) {
      }
    }
    __syncwarp();
    for (int k = 0; k < cnt; ++k) {
      if (valid) {
        const int n = w.n;
        const int mine = mine_of(w);
        last_first = gidx;  // drain bookkeeping, also right if this item is cut short
        last_n = n;
        ids[lane] = v0;
        __syncwarp();
        const size_t head0 = (size_t)w.hg * HG;
        int g = gidx + pi;  // global ring position of the next page
        int st = g % NST, rnd = g / NST;
        for (int base = 0, buf = 0; base < mine; base += 32, buf ^= 1) {
          const int nxt = page_id(w, base + 32 + lane);  // prefetch the next 32 ids
          if (lane == 0) {
            const int cnt32 = min(32, mine - base);
            for (int kk = 0; kk < cnt32; ++kk) {
              const int pg = ids[buf * 32 + kk];
              if (rnd > 0 && !mbar_wait(&empty[st], (rnd - 1) & 1, p.wait_limit_ns)) {
                atomicOr(p.status, KVQ_DEV_TIMEOUT);
                ok = false;
                break;
              }
              if (p.drop_copies) {
                // failure-path test: the stage is never filled, so its consumers' wait runs out
              } else if (pg >= 0) {
                bad_s[st] = 0;  // read by the consumers after this stage's full barrier completes
                uint8_t* kc = codes + st * stage_code;
                mbar_arrive_expect_tx(&full[st], stage_code + stage_scale);
                tma_load_5d(kc, &tm_k, 0, 0, 0, static_cast<int>(head0), pg, &full[st]);
                tma_load_5d(kc + HG * Lo::kHeadCode, &tm_v, 0, 0, 0, static_cast<int>(head0), pg, &full[st]);
                if constexpr (T::kScaleRow > 0) {
                  uint8_t* ks = scales + st * stage_scale;
                  const size_t off = ((size_t)pg * Hkv + head0) * Lo::kHeadScale;
                  bulk_load(ks, p.k_scales + off, HG * Lo::kHeadScale, &full[st]);
                  bulk_load(ks + HG * Lo::kHeadScale, p.v_scales + off, HG * Lo::kHeadScale, &full[st]);
                }
              } else {
                // an out-of-range page id (flagged in the status word): nothing is
                // loaded, and the consumers mask every token of the stage, so the
                // page contributes nothing whatever stale bytes the stage holds
                bad_s[st] = 1;
                mbar_arrive(&full[st]);
              }
              st += NP;
              if (st >= NST) {
                st -= NST;
                ++rnd;
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
          if (!ok) break;
          ids[(buf ^ 1) * 32 + lane] = nxt;
          __syncwarp();
        }
        gidx += n;
      }
      // the next item's descriptor and first page ids, fetched while the
      // consumers finish this one
      Item nw;
      bool nvalid = false;
      int nv0 = -1;
      if (ok && valid && k + 1 < cnt) {
        nvalid = unpack(rest[r0 + k], nw);
        if (nvalid) nv0 = page_id(nw, lane);
      }
      if (lane == 0 && !ok) abort_flag = 1;
      // the consumers' epilogue of this item is done: the ring is free
      asm volatile("bar.sync 2, %0;" ::"r"(sync_threads) : "memory");
      if (abort_flag || !valid) break;
      w = nw;
      valid = nvalid;
      v0 = nv0;
    }
    // Drain: before this warp (and so the CTA) can exit, every copy it issued has
    // landed.  Only the last item can have copies in flight: the consumers
    // finished the earlier ones before the item boundary.
    if (lane == 0) {
      for (int idx = pi; idx < last_n; idx += NP) {
        const int g = last_first + idx;
        if (g + NST < last_first + last_n) continue;  // a later page of this stage was issued
        if (!mbar_wait(&full[g % NST], (g / NST) & 1, p.wait_limit_ns)) {
          atomicOr(p.status, KVQ_DEV_TIMEOUT);
          break;
        }
      }
    }
    return;
  }

  // ================================================================== consumers
  if constexpr (Lo::kRegSplit) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Lo::kConsumerRegs));
  // Every warp of a head writes the head's q tile itself, with the same bytes as
  // the head's other warps, so its own writes already give it the whole tile;
  // tiles are rewritten only after the item boundary barrier.
  uint8_t* myq = qfrag + hl * Lo::kQBytes;
  const uint32_t qbase = smem_addr(myq) + ((lane >> 3) * 8 + (lane & 7)) * 16;
  // Per-lane byte offsets of the swizzled ldmatrix rows inside a head block,
  // one per value of (chunk & 7) of the iteration (the XOR with the row index
  // only touches the low three chunk bits; see swz()).  V (INT8, transposed):
  // matrix m = lane/8 is token block m%2, chunk 2 cp + m/2.
  [[maybe_unused]] uint32_t voff[4];
  if constexpr (int8_codes<FMT>()) {
    const int mm = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4) voff[v4] = (8 * (mm & 1) + rr) * 128 + (((2 * v4 + (mm >> 1)) ^ rr) << 4);
  }
  // epilogue exchange in the (then idle) ring: the WPH-1 other warps of each head
  // leave their accumulators in fragment order, [slot][m-tile][lane] float4, and
  // their (m, l) per head row, [slot][8] float2; slot = head * (WPH-1) + warp - 1.
  float4* part_o = reinterpret_cast<float4*>(codes);
  float2* part_ml = reinterpret_cast<float2*>(codes + (CW - 1) * Lo::kPartOBytes);
  constexpr float kLn2 = 0.69314718055994530942f;
  // P' is split into hi + lo f16 (bf16) terms for fp32 output; for bf16 output one
  // term is enough: its rounding (at most 2^-11 relative, 2^-8 for the BF16
  // cache's bf16 P) is not above the output's own rounding to bf16
  constexpr bool p_lo = PLO;

  int gidx = 0;  // pages of this CTA before the current item (global ring position)
  Item w = first, nw;
  bool ok_item = first_ok, next_ok = false;
  for (int k = 0; k < cnt; ++k) {
    if (!ok_item) {  // a bad plan entry: every thread of the CTA stops here
      if (threadIdx.x == 0) {
        atomicOr(p.status, KVQ_DEV_BAD_PLAN);
        abort_flag = 1;
      }
      asm volatile("bar.sync 2, %0;" ::"r"(sync_threads) : "memory");
      break;
    }
    // the next item's descriptor, fetched now and kept in shared memory (read in
    // the epilogue, after the barrier that ends this item's pages)
    // this item's descriptor is kept there too: the epilogue reads its sequence,
    // split and head group from shared memory, not from registers held through
    // the page loop
    if (threadIdx.x == 0) {
      cur_desc = k == 0 ? d0 : next_desc;
      next_desc = k + 1 < cnt ? rest[r0 + k] : make_int4(-1, -1, -1, -1);
    }
    // ---- q fragments (A operand rows = heads) for this item, converted from
    // the raw bf16 pairs loaded earlier.  Column (k) order per format, matching
    // the K fragments below: k-step j pairs (2c, 2c+1) with d dA(j, c) + {0, 1}
    // and (2c+8, 2c+9) with dB(j, c) + {0, 1}.
    float qk_scale = p.sm_scale_log2;
    {
      if constexpr (!T::kBf16Mma) {
        // bf16 -> f16 exactly: scale the head's row by a power of two so that its
        // largest |q| lands in [2^14, 2^15); every element within 2^28 of it is
        // then exactly representable in f16.  The power of two is undone on the
        // logits.
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < KS; ++j) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&qraw[j][u]);
            amax = fmaxf(amax, fmaxf(fabsf(__low2float(v)), fabsf(__high2float(v))));
          }
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int k = 0;
        if (amax > 0.f) {
          int e;
          frexpf(amax, &e);  // amax = m * 2^e, m in [0.5, 1)
          k = min(126, max(-126, 15 - e));
        }
        const float up = pow2f(k);
#pragma unroll
        for (int j = 0; j < KS; ++j) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&qraw[j][u]);
            qraw[j][u] = h2_as_u32(__floats2half2_rn(__low2float(v) * up, __high2float(v) * up));
          }
        }
        qk_scale *= pow2f(-k);
        if constexpr (FMT == KVQ_FMT_NVFP4) qk_scale *= p.k_gs_inv;
      }
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        uint32_t* m0 = reinterpret_cast<uint32_t*>(myq + (2 * j) * 128 + r * 16 + c * 4);
        m0[0] = qraw[j][0];
        m0[32] = qraw[j][1];  // next matrix (dB part), +128 bytes
      }
    }
    __syncwarp();

    // At D = 128 this item's q fragments (A operand, two k-steps per
    // ldmatrix.x4) fit in registers for all of its pages; at D = 256 they are
    // re-read from shared memory per page (the registers go to the accumulators).
    constexpr bool kQInRegs = D == 128;
    [[maybe_unused]] uint32_t qreg[kQInRegs ? KS : 1][2];
    if constexpr (kQInRegs) {
#pragma unroll
      for (int jj = 0; jj < KS / 2; ++jj)
        ldsm_x4(qbase + jj * 512, qreg[2 * jj][0], qreg[2 * jj][1], qreg[2 * jj + 1][0], qreg[2 * jj + 1][1]);
    }

    float oacc[Lo::kMTiles][4];
#pragma unroll
    for (int mt = 0; mt < Lo::kMTiles; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
    float m_run = -INFINITY;  // running max (log2 domain) of head r
    float l_run = 0.f;        // this lane's part of the running sum of head r
    const int n = w.n;
    const int L = w.L;
    const int page_begin = w.page_begin;

    bool alive = true;
    // this warp's pages: idx = grp, grp + WPH, ... ; global ring position gidx + idx
    int st = (gidx + grp) % NST, rnd = (gidx + grp) / NST;
    for (int idx = grp; idx < n; idx += WPH) {
      const bool got = mbar_wait(&full[st], rnd & 1, p.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) atomicOr(p.status, KVQ_DEV_TIMEOUT);
        alive = false;
        break;
      }
      const uint32_t kblk = smem_addr(codes + st * stage_code + hl * Lo::kHeadCode);
      const uint32_t vblk = kblk + HG * Lo::kHeadCode;
      const uint8_t* ksc = scales + st * stage_scale + hl * Lo::kHeadScale;
      const uint8_t* vsc = ksc + HG * Lo::kHeadScale;
      const int tok0 = (page_begin + idx) * kPage;
      const int nvalid = bad_s[st] ? 0 : min(kPage, L - tok0);  // a bad page id: no valid token

    // ---------------------------------------------------------- S = q K^T
    float sacc[2][2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int u = 0; u < 2; ++u) sacc[i][u][0] = sacc[i][u][1] = sacc[i][u][2] = sacc[i][u][3] = 0.f;

    // chunk groups of 4 x 16-byte chunks; q fragments of the group's k-steps are
    // fetched from shared memory (two k-steps per ldmatrix.x4).
    constexpr int QPG = int8_codes<FMT>() ? 4 : (FMT == KVQ_FMT_BF16 ? 2 : 8);  // k-steps per group
    constexpr int NCG = KS / QPG;
    // INT8 with one scale per 32 elements: each group's two k-steps go to a
    // fresh accumulator, which is scaled by the group's per-token K scale and
    // added to zg[n-tile][token] (the scales are [group][16 tokens] fp32)
    [[maybe_unused]] float zg[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    [[maybe_unused]] uint32_t ksw[2][4];
    if constexpr (FMT == KVQ_FMT_NVFP4) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if constexpr (D == 256) {
          const uint4 srow = *reinterpret_cast<const uint4*>(ksc + (8 * i + r) * 16);
          ksw[i][0] = srow.x; ksw[i][1] = srow.y; ksw[i][2] = srow.z; ksw[i][3] = srow.w;
        } else {  // D = 128: 8 group scales a token
          const uint2 srow = *reinterpret_cast<const uint2*>(ksc + (8 * i + r) * 8);
          ksw[i][0] = srow.x; ksw[i][1] = srow.y; ksw[i][2] = ksw[i][3] = 0u;
        }
      }
    }
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg) {
      uint32_t qa[QPG][2];
      if constexpr (kQInRegs) {
#pragma unroll
        for (int m = 0; m < QPG; ++m) {
          qa[m][0] = qreg[cg * QPG + m][0];
          qa[m][1] = qreg[cg * QPG + m][1];
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < QPG / 2; ++jj)
          ldsm_x4(qbase + (cg * (QPG / 2) + jj) * 512, qa[2 * jj][0], qa[2 * jj][1], qa[2 * jj + 1][0],
                  qa[2 * jj + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t w[4];
        ldsm_x4(swz_row<T::kRow>(kblk, 8 * i + (lane & 7), 4 * cg + (lane >> 3)), w[0], w[1], w[2], w[3]);
        if constexpr (FMT == KVQ_FMT_INT8) {
          // chunk = 16 d's = one k-step; lane gets bytes 4c..4c+3 of row 8i+r:
          // k (2c, 2c+1) <- d 16ch+4c+{0,1}, k (2c+8, 2c+9) <- d 16ch+4c+{2,3}.
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t x = w[m] ^ 0x80808080u;
            mma16816<false>(sacc[i][m & 1], qa[m][0], 0u, qa[m][1], 0u, i8pair_to_h2<0x4140>(x),
                            i8pair_to_h2<0x4342>(x));
          }
        } else if constexpr (FMT == KVQ_FMT_INT8_G32) {
          // chunks 4cg .. 4cg+3 are groups 2cg (m = 0, 1) and 2cg+1 (m = 2, 3)
#pragma unroll
          for (int gg = 0; gg < 2; ++gg) {
            float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
              const uint32_t x = w[2 * gg + mm] ^ 0x80808080u;
              mma16816<false>(t, qa[2 * gg + mm][0], 0u, qa[2 * gg + mm][1], 0u, i8pair_to_h2<0x4140>(x),
                              i8pair_to_h2<0x4342>(x));
            }
            const float2 sc = *reinterpret_cast<const float2*>(ksc + ((2 * cg + gg) * kPage + 8 * i + 2 * c) * 4);
            zg[i][0] = fmaf(t[0], sc.x, zg[i][0]);
            zg[i][1] = fmaf(t[1], sc.y, zg[i][1]);
          }
        } else if constexpr (FMT == KVQ_FMT_BF16) {
          // chunk = 8 d's; k-step uses chunks 2j (k 2c..) and 2j+1 (k 2c+8..).
          mma16816<true>(sacc[i][0], qa[0][0], 0u, qa[0][1], 0u, w[0], w[1]);
          mma16816<true>(sacc[i][1], qa[1][0], 0u, qa[1][1], 0u, w[2], w[3]);
        } else {
          // NVFP4: chunk = 32 d's; lane gets bytes 4c..4c+3 = d 32ch+8c..+7, split
          // into k-steps (ch, 0) and (ch, 1); the group scale of d is 2ch + c/2.
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int ch = 4 * cg + m;
            const uint32_t bsel = 2 * (ch & 1) + (c >> 1);
            const __half2 sdh = u32_as_h2(e4m3x2_to_h2(prmt(ksw[i][ch >> 1], 0u, bsel | (bsel << 4))));
            uint32_t f[4];
            e2m1x8_to_h2x4(w[m], f);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t b0 = h2_as_u32(__hmul2(u32_as_h2(f[2 * hh]), sdh));
              const uint32_t b1 = h2_as_u32(__hmul2(u32_as_h2(f[2 * hh + 1]), sdh));
              mma16816<false>(sacc[i][hh], qa[2 * m + hh][0], 0u, qa[2 * m + hh][1], 0u, b0, b1);
            }
          }
        }
      }
    }

    // ---------------------------------------------------------- online softmax
    // lane holds head r, tokens 2c, 2c+1 (n-tile 0) and 8+2c, 9+2c (n-tile 1).
    const int tk[4] = {2 * c, 2 * c + 1, 8 + 2 * c, 9 + 2 * c};
    float z[4];
    if constexpr (FMT == KVQ_FMT_INT8_G32) {  // K scales already applied per group
      z[0] = zg[0][0];
      z[1] = zg[0][1];
      z[2] = zg[1][0];
      z[3] = zg[1][1];
    } else {
      z[0] = sacc[0][0][0] + sacc[0][1][0];
      z[1] = sacc[0][0][1] + sacc[0][1][1];
      z[2] = sacc[1][0][0] + sacc[1][1][0];
      z[3] = sacc[1][0][1] + sacc[1][1][1];
    }
    float ks4[4] = {1.f, 1.f, 1.f, 1.f};
    if constexpr (FMT == KVQ_FMT_INT8) {
      const float2 a = *reinterpret_cast<const float2*>(ksc + 8 * c);
      const float2 bb = *reinterpret_cast<const float2*>(ksc + 32 + 8 * c);
      ks4[0] = a.x; ks4[1] = a.y; ks4[2] = bb.x; ks4[3] = bb.y;
    }
    float pmax = -INFINITY;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      z[u] = (tk[u] < nvalid) ? z[u] * ks4[u] * qk_scale : -INFINITY;
      pmax = fmaxf(pmax, z[u]);
    }
    pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, 1));
    pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, 2));
    const float m_new = fmaxf(m_run, pmax);
    // no valid token so far (only a page with a bad id): keep the state empty
    // instead of forming exp2(-inf - -inf)
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = exp2f(m_run - m_use);  // m_run = -inf -> 0
    m_run = m_new;
    float pr[4];
    float psum = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      pr[u] = exp2f(z[u] - m_use);  // masked tokens: exp2(-inf) = 0
      psum += pr[u];
    }
    l_run = l_run * alpha + psum;
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
      const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * c);      // head 2c
      const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * c + 4);  // head 2c+1
#pragma unroll
      for (int mt = 0; mt < Lo::kMTiles; ++mt) {
        oacc[mt][0] *= a0;
        oacc[mt][1] *= a1;
        oacc[mt][2] *= a0;
        oacc[mt][3] *= a1;
      }
    }
    // P' (B operand of O^T = V^T P'^T): INT8 folds the V scale of the token in.
    float pv[4];
    if constexpr (FMT == KVQ_FMT_INT8) {
      const float2 a = *reinterpret_cast<const float2*>(vsc + 8 * c);
      const float2 bb = *reinterpret_cast<const float2*>(vsc + 32 + 8 * c);
      const float vs4[4] = {a.x, a.y, bb.x, bb.y};
#pragma unroll
      for (int u = 0; u < 4; ++u) pv[u] = (tk[u] < nvalid) ? pr[u] * vs4[u] : 0.f;
    } else if constexpr (FMT == KVQ_FMT_INT8_G32) {  // the V scale depends on d: folded in per group below
#pragma unroll
      for (int u = 0; u < 4; ++u) pv[u] = (tk[u] < nvalid) ? pr[u] : 0.f;
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) pv[u] = pr[u];
    }
    uint32_t phi[2], plo[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if constexpr (T::kBf16Mma) {
        const __nv_bfloat162 hh = __floats2bfloat162_rn(pv[2 * u], pv[2 * u + 1]);
        const __nv_bfloat162 ll =
            __floats2bfloat162_rn(pv[2 * u] - __low2float(hh), pv[2 * u + 1] - __high2float(hh));
        phi[u] = *reinterpret_cast<const uint32_t*>(&hh);
        plo[u] = *reinterpret_cast<const uint32_t*>(&ll);
      } else {
        const __half2 hh = __floats2half2_rn(pv[2 * u], pv[2 * u + 1]);
        const __half2 ll = __floats2half2_rn(pv[2 * u] - __low2float(hh), pv[2 * u + 1] - __high2float(hh));
        phi[u] = h2_as_u32(hh);
        plo[u] = h2_as_u32(ll);
      }
    }

    // ---------------------------------------------------------- O^T += V^T P'^T
    const bool partial = nvalid < kPage;
    if constexpr (int8_codes<FMT>()) {
      // ldmatrix.trans of int8 pairs: lane gets [V[t][de], V[t][do], V[t+1][de], V[t+1][do]]
      // with t = 8tb+2c, de = 16ch+2r, do = de+1 -> m-tile ch rows r (de) and r+8 (do).
      uint32_t vb[4];
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4) vb[v4] = vblk + voff[v4];
#pragma unroll
      for (int cp = 0; cp < Lo::kMTiles / 2; ++cp) {
        uint32_t w[4];
        ldsm_x4_t(vb[cp & 3] + (cp >> 2) * (kPage * 128), w[0], w[1], w[2], w[3]);
        if constexpr (FMT == KVQ_FMT_INT8_G32) {
          // m-tiles 2cp, 2cp+1 are d 32cp .. 32cp+31: group cp.  P' = P x that
          // group's V scale of each token ([group][16 tokens] fp32).
          const float2 a = *reinterpret_cast<const float2*>(vsc + (cp * kPage + 2 * c) * 4);
          const float2 bb = *reinterpret_cast<const float2*>(vsc + (cp * kPage + 8 + 2 * c) * 4);
          const float g4[4] = {pv[0] * a.x, pv[1] * a.y, pv[2] * bb.x, pv[3] * bb.y};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            // a masked token (pv = 0) may meet a NaN scale in an unwritten slot
            const float e0 = pv[2 * u] != 0.f ? g4[2 * u] : 0.f;
            const float e1 = pv[2 * u + 1] != 0.f ? g4[2 * u + 1] : 0.f;
            const __half2 hh = __floats2half2_rn(e0, e1);
            phi[u] = h2_as_u32(hh);
            if constexpr (p_lo) plo[u] = h2_as_u32(__floats2half2_rn(e0 - __low2float(hh), e1 - __high2float(hh)));
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t x0 = w[2 * u] ^ 0x80808080u;
          const uint32_t x1 = w[2 * u + 1] ^ 0x80808080u;
          const uint32_t a0 = i8pair_to_h2<0x4240>(x0), a1 = i8pair_to_h2<0x4341>(x0);
          const uint32_t a2 = i8pair_to_h2<0x4240>(x1), a3 = i8pair_to_h2<0x4341>(x1);
          mma16816<false>(oacc[2 * cp + u], a0, a1, a2, a3, phi[0], phi[1]);
          if constexpr (p_lo) mma16816<false>(oacc[2 * cp + u], a0, a1, a2, a3, plo[0], plo[1]);
        }
      }
    } else if constexpr (FMT == KVQ_FMT_BF16) {
      // m-tile mt: rows r <- d 16mt+r (chunk 2mt), r+8 <- d 16mt+8+r (chunk 2mt+1)
      const uint32_t m0 = (2 * c < nvalid ? 0x0000FFFFu : 0u) | (2 * c + 1 < nvalid ? 0xFFFF0000u : 0u);
      const uint32_t m1 = (8 + 2 * c < nvalid ? 0x0000FFFFu : 0u) | (9 + 2 * c < nvalid ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int mt = 0; mt < Lo::kMTiles; ++mt) {
        const int mm = lane >> 3;
        const int trow = 8 * (mm >> 1) + (lane & 7);
        uint32_t w[4];
        ldsm_x4_t(swz(vblk, trow, 2 * mt + (mm & 1)), w[0], w[1], w[2], w[3]);
        if (partial) {  // unwritten slots may hold NaN bit patterns: zero them
          w[0] &= m0; w[1] &= m0; w[2] &= m1; w[3] &= m1;
        }
        mma16816<true>(oacc[mt], w[0], w[1], w[2], w[3], phi[0], phi[1]);
        if constexpr (p_lo) mma16816<true>(oacc[mt], w[0], w[1], w[2], w[3], plo[0], plo[1]);
      }
    } else if constexpr (D == 128) {
      // NVFP4 at D = 128 (64-byte rows): lane (r, c) reads the 8 bytes r (d
      // 16r..16r+15, scale group r) of token rows 2c, 2c+1 (MMA k 2c, 2c+1) and
      // 2c+8, 2c+9 (k 2c+8, 2c+9).  As at D = 256, the words of a token pair at
      // the same d merge into bytes that each hold one d for both tokens, first
      // token in the low nibble.  m-tile 4j+k takes d = 16r+8j+2k (row r) and d+1
      // (row r+8); every m-tile of the lane is in group r.
      uint2 vw[2][2];  // [token pair][first / second token]
#pragma unroll
      for (int tb = 0; tb < 2; ++tb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 8 * tb + 2 * c + e;
          asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                       : "=r"(vw[tb][e].x), "=r"(vw[tb][e].y)
                       : "r"(swz_row<T::kRow>(vblk, t, r >> 1) + 8 * (r & 1)));
        }
      uint32_t svp[2];  // [token pair]: f16x2 of group r over the pair's tokens
#pragma unroll
      for (int tb = 0; tb < 2; ++tb) {
        const int t = 8 * tb + 2 * c;
        const uint32_t sw = (uint32_t)vsc[t * 8 + r] | ((uint32_t)vsc[(t + 1) * 8 + r] << 8);
        const uint32_t vm = (t < nvalid ? 0x0000FFFFu : 0u) | (t + 1 < nvalid ? 0xFFFF0000u : 0u);
        svp[tb] = e4m3x2_to_h2(sw) & vm;  // unwritten slots may hold NaN scales
      }
      const __half2 sa = u32_as_h2(svp[0]), sb = u32_as_h2(svp[1]);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint32_t f[2][2][4];  // [token pair][even / odd d][byte k]
#pragma unroll
        for (int tb = 0; tb < 2; ++tb) {
          const uint32_t w0 = j == 0 ? vw[tb][0].x : vw[tb][0].y;
          const uint32_t w1 = j == 0 ? vw[tb][1].x : vw[tb][1].y;
          e2m1x8_to_h2x4(bitsel(w0, w1 << 4, 0x0F0F0F0Fu), f[tb][0]);
          e2m1x8_to_h2x4(bitsel(w0 >> 4, w1, 0x0F0F0F0Fu), f[tb][1]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t a0 = h2_as_u32(__hmul2(u32_as_h2(f[0][0][k]), sa));
          const uint32_t a1 = h2_as_u32(__hmul2(u32_as_h2(f[0][1][k]), sa));
          const uint32_t a2 = h2_as_u32(__hmul2(u32_as_h2(f[1][0][k]), sb));
          const uint32_t a3 = h2_as_u32(__hmul2(u32_as_h2(f[1][1][k]), sb));
          mma16816<false>(oacc[4 * j + k], a0, a1, a2, a3, phi[0], phi[1]);
          if constexpr (p_lo) mma16816<false>(oacc[4 * j + k], a0, a1, a2, a3, plo[0], plo[1]);
        }
      }
    } else {
      // NVFP4: lane (r, c) reads 16-byte chunk r (d 32r..32r+31) of token rows
      // 2c, 2c+1 (MMA k 2c, 2c+1) and 2c+8, 2c+9 (k 2c+8, 2c+9).  The words of a
      // token pair at the same d merge into bytes that each hold one d for both
      // tokens, first token in the low nibble (f[.][0]: even d, f[.][1]: odd d).
      // m-tile 4j+k takes d = 32r+8j+2k (row r) and d+1 (row r+8), both in
      // scale group 2r + j/2, so the group scale is one f16x2 per token pair.
      uint4 vw[2][2];  // [token pair][first / second token]
#pragma unroll
      for (int tb = 0; tb < 2; ++tb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 8 * tb + 2 * c + e;
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(vw[tb][e].x), "=r"(vw[tb][e].y), "=r"(vw[tb][e].z), "=r"(vw[tb][e].w)
                       : "r"(swz(vblk, t, r)));
        }
      uint32_t svp[2][2];  // [token pair][group 2r, 2r+1]: f16x2 over the pair's tokens
#pragma unroll
      for (int tb = 0; tb < 2; ++tb) {
        const int t = 8 * tb + 2 * c;
        const uint32_t s0 = *reinterpret_cast<const uint16_t*>(vsc + t * 16 + 2 * r);
        const uint32_t s1 = *reinterpret_cast<const uint16_t*>(vsc + (t + 1) * 16 + 2 * r);
        const uint32_t sw = s0 | (s1 << 16);  // bytes: (g0, t) (g1, t) (g0, t+1) (g1, t+1)
        const uint32_t vm = (t < nvalid ? 0x0000FFFFu : 0u) | (t + 1 < nvalid ? 0xFFFF0000u : 0u);
        svp[tb][0] = e4m3x2_to_h2(prmt(sw, 0u, 0x20u)) & vm;  // unwritten slots may hold NaN scales
        svp[tb][1] = e4m3x2_to_h2(prmt(sw, 0u, 0x31u)) & vm;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t f[2][2][4];  // [token pair][even / odd d][byte k]
#pragma unroll
        for (int tb = 0; tb < 2; ++tb) {
          const uint32_t w0 = j == 0 ? vw[tb][0].x : j == 1 ? vw[tb][0].y : j == 2 ? vw[tb][0].z : vw[tb][0].w;
          const uint32_t w1 = j == 0 ? vw[tb][1].x : j == 1 ? vw[tb][1].y : j == 2 ? vw[tb][1].z : vw[tb][1].w;
          e2m1x8_to_h2x4(bitsel(w0, w1 << 4, 0x0F0F0F0Fu), f[tb][0]);
          e2m1x8_to_h2x4(bitsel(w0 >> 4, w1, 0x0F0F0F0Fu), f[tb][1]);
        }
        const __half2 sa = u32_as_h2(svp[0][j >> 1]), sb = u32_as_h2(svp[1][j >> 1]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t a0 = h2_as_u32(__hmul2(u32_as_h2(f[0][0][k]), sa));
          const uint32_t a1 = h2_as_u32(__hmul2(u32_as_h2(f[0][1][k]), sa));
          const uint32_t a2 = h2_as_u32(__hmul2(u32_as_h2(f[1][0][k]), sb));
          const uint32_t a3 = h2_as_u32(__hmul2(u32_as_h2(f[1][1][k]), sb));
          mma16816<false>(oacc[4 * j + k], a0, a1, a2, a3, phi[0], phi[1]);
          if constexpr (p_lo) mma16816<false>(oacc[4 * j + k], a0, a1, a2, a3, plo[0], plo[1]);
        }
      }
    }
    (void)partial;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      st += WPH;
      if (st >= NST) {
        st -= NST;
        ++rnd;
      }
    }
    gidx += n;

    // ================================================================ epilogue
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (!alive) {
      m_run = -INFINITY;
      l_run = 0.f;
      if (lane == 0) abort_flag = 1;
    }
    // every consumer warp is past this item's last page: every stage has landed
    // and been read, and the producers wait for this item's end, so the ring can
    // hold the exchange.
    asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory");
    Item cw;
    unpack(cur_desc, cw);
    // the next item: q and length loads are issued once this warp's accumulators are written out
    auto next_item = [&]() {
      next_ok = k + 1 < cnt && unpack(next_desc, nw);
      if (next_ok) {
        load_q(nw);
        nw.L = seq_len(nw.b);
      }
    };
    const int others = WPH - 1;
    if (grp > 0) {
      const int slot = hl * others + grp - 1;
#pragma unroll
      for (int mt = 0; mt < Lo::kMTiles; ++mt)
        part_o[(slot * Lo::kMTiles + mt) * 32 + lane] = make_float4(oacc[mt][0], oacc[mt][1], oacc[mt][2], oacc[mt][3]);
      if (c == 0) part_ml[slot * 8 + r] = make_float2(m_run, l_run);
      next_item();  // the accumulators are in shared memory: registers are free
    }
    if (others > 0) asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory");
    if (grp == 0) {
      // combine the head's warps: weights per head row r (this lane's row of S)
      float M = m_run;
      for (int j = 0; j < others; ++j) M = fmaxf(M, part_ml[(hl * others + j) * 8 + r].x);
      const bool live = M != -INFINITY;
      float Lsum = live ? l_run * exp2f(m_run - M) : 0.f;
      for (int j = 0; j < others; ++j) {
        const float2 ml = part_ml[(hl * others + j) * 8 + r];
        if (live) Lsum += ml.y * exp2f(ml.x - M);
      }
      const bool any = live && Lsum > 0.f;
      float inv = any ? 1.f / Lsum : 0.f;
      const float lse = any ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
      if constexpr (FMT == KVQ_FMT_NVFP4) inv *= p.v_gs_inv;
      // accumulator columns are heads 2c and 2c+1: their weights live in lanes 8c and 8c+4
      {
        const float wr = any ? exp2f(m_run - M) * inv : 0.f;
        const float w0 = __shfl_sync(0xffffffffu, wr, 8 * c);
        const float w1 = __shfl_sync(0xffffffffu, wr, 8 * c + 4);
#pragma unroll
        for (int mt = 0; mt < Lo::kMTiles; ++mt) {
          oacc[mt][0] *= w0;
          oacc[mt][1] *= w1;
          oacc[mt][2] *= w0;
          oacc[mt][3] *= w1;
        }
      }
      for (int j = 0; j < others; ++j) {
        const int slot = hl * others + j;
        const float wr = any ? exp2f(part_ml[slot * 8 + r].x - M) * inv : 0.f;
        const float w0 = __shfl_sync(0xffffffffu, wr, 8 * c);
        const float w1 = __shfl_sync(0xffffffffu, wr, 8 * c + 4);
        const float4* src = part_o + slot * Lo::kMTiles * 32 + lane;
#pragma unroll
        for (int mt0 = 0; mt0 < Lo::kMTiles; mt0 += 4) {  // four m-tiles of loads in flight
          float4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) v[u] = src[(mt0 + u) * 32];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            oacc[mt0 + u][0] += v[u].x * w0;
            oacc[mt0 + u][1] += v[u].y * w1;
            oacc[mt0 + u][2] += v[u].z * w0;
            oacc[mt0 + u][3] += v[u].w * w1;
          }
        }
      }
      // Stage the head's G query rows (fp32, or bf16 for a direct bf16 output) in
      // shared memory, row-major, and copy them out with one bulk copy: the G
      // query heads of a KV head are consecutive rows of both `out` and the
      // partials.  The copy runs asynchronously; the ring is reused only after
      // its source reads are done.
      const bool direct = cw.direct;
      const bool to_bf16 = direct && p.out_bf16;
      uint8_t* stage = codes + Lo::kStageAt + hl * Lo::kStageBytes;
      const int row_bytes = to_bf16 ? 2 * D : 4 * D;
      auto put = [&](int hr, int d, float v0, float v1, bool pair) {  // elements d (and d+1 if pair) of row hr
        if (to_bf16) {
          const int byte = 2 * d;
          uint8_t* at = stage + hr * row_bytes + byte;
          if (pair) *reinterpret_cast<__nv_bfloat162*>(at) = __floats2bfloat162_rn(v0, v1);
          else *reinterpret_cast<__nv_bfloat16*>(at) = __float2bfloat16_rn(v0);
        } else {
          const int byte = 4 * d;
          uint8_t* at = stage + hr * row_bytes + byte;
          if (pair) *reinterpret_cast<float2*>(at) = make_float2(v0, v1);
          else *reinterpret_cast<float*>(at) = v0;
        }
      };
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hr = 2 * c + e;  // head row within the KV head's group
        if (hr >= G) continue;
#pragma unroll
        for (int mt = 0; mt < Lo::kMTiles; ++mt) {
          if constexpr (int8_codes<FMT>()) {
            put(hr, 16 * mt + 2 * r, oacc[mt][e], oacc[mt][2 + e], true);
          } else if constexpr (FMT == KVQ_FMT_BF16) {
            put(hr, 16 * mt + r, oacc[mt][e], 0.f, false);
            put(hr, 16 * mt + 8 + r, oacc[mt][2 + e], 0.f, false);
          } else {  // NVFP4: m-tile 4j+k of lane row r holds d = (D/8) r + 8j + 2k and d+1
            put(hr, (D / 8) * r + 8 * (mt >> 2) + 2 * (mt & 3), oacc[mt][e], oacc[mt][2 + e], true);
          }
        }
      }
      __syncwarp();
      const int qh0 = (cw.hg * HG + hl) * G;  // first query head of this KV head
      {
        const size_t row0 = direct ? (size_t)cw.b * p.num_q_heads + qh0 : (size_t)cw.split * p.num_q_heads + qh0;
        uint8_t* dst = direct ? reinterpret_cast<uint8_t*>(p.out) + row0 * row_bytes
                              : reinterpret_cast<uint8_t*>(p.o_part + row0 * D);
        if (direct && p.out_host) {  // host memory: plain 16-byte stores over the host link
          __syncwarp();
          for (int i = lane; i < G * row_bytes / 16; i += 32)
            *reinterpret_cast<uint4*>(dst + (size_t)i * 16) = *reinterpret_cast<const uint4*>(stage + i * 16);
        } else {
          fence_proxy_async_smem();  // the staged rows, written by this warp, become visible to the copy
          __syncwarp();
          if (lane == 0) bulk_store(dst, stage, G * row_bytes);
        }
      }
      if (c == 0 && r < G) {
        if (direct) {
          if (p.lse_out) p.lse_out[(size_t)cw.b * p.num_q_heads + qh0 + r] = lse;
        } else {
          p.lse_part[(size_t)cw.split * p.num_q_heads + qh0 + r] = lse;
        }
      }
      next_item();
    }
    // the ring (or, after the last item, the CTA's shared memory) may be reused
    // once the copy has read it; the copy's global writes complete on their own
    // and are visible to the next kernel once this grid has completed
    if (grp == 0 && lane == 0) bulk_wait_read();
    // with the producers: the ring may be refilled for the next item
    asm volatile("bar.sync 2, %0;" ::"r"(sync_threads) : "memory");
    if (abort_flag) break;
    w = nw;
    ok_item = next_ok;
  }
}

}  // namespace kvq
