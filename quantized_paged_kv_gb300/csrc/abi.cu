// abi.cu — the extern "C" entry points declared in include/kvq.h: argument
// validation, the host split planner, TMA tensor-map encoding and kernel dispatch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <functional>
#include <mutex>
#include <numeric>
#include <queue>
#include <string>
#include <utility>
#include <vector>

#include "kvq_internal.h"

namespace {

thread_local std::string g_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_error = buf;
  return code;
}

int succeed() {
  g_error.clear();
  return KVQ_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int64_t row_bytes(int format, int D) {
  switch (format) {
    case KVQ_FMT_BF16: return 2LL * D;
    case KVQ_FMT_INT8: return D;
    case KVQ_FMT_INT8_G32: return D;
    case KVQ_FMT_NVFP4: return D / 2;
    default: return -1;
  }
}

int64_t scale_row_bytes(int format, int D) {
  switch (format) {
    case KVQ_FMT_BF16: return 0;
    case KVQ_FMT_INT8: return 4;
    case KVQ_FMT_INT8_G32: return 4LL * (D / 32);
    case KVQ_FMT_NVFP4: return D / 16;
    default: return -1;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates the shape (and, if `pointers`, the device arrays) of a cache.
int check_cache(const kvq_cache* c, bool pointers) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "cache is NULL");
  if (c->format != KVQ_FMT_BF16 && c->format != KVQ_FMT_INT8 && c->format != KVQ_FMT_NVFP4 &&
      c->format != KVQ_FMT_INT8_G32)
    return fail(KVQ_ERR_INVALID_ARG, "unknown cache format %d", c->format);
  if (c->page_size != 16) return fail(KVQ_ERR_UNSUPPORTED, "page_size %d: only 16 is implemented", c->page_size);
  if (c->head_dim != 128 && c->head_dim != 256)
    return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d: only 128 and 256 are implemented", c->head_dim);
  if (c->num_kv_heads < 1) return fail(KVQ_ERR_INVALID_ARG, "num_kv_heads %d < 1", c->num_kv_heads);
  if (c->num_pages < 1) return fail(KVQ_ERR_INVALID_ARG, "num_pages %d < 1", c->num_pages);
  if ((int64_t)c->num_pages * c->num_kv_heads * c->page_size > 0x7FFFFFFFLL)
    return fail(KVQ_ERR_UNSUPPORTED, "num_pages * num_kv_heads * page_size exceeds 2^31 rows");
  if (c->format == KVQ_FMT_NVFP4) {
    if (!(std::isfinite(c->k_global_scale) && c->k_global_scale > 0.f && std::isfinite(c->v_global_scale) &&
          c->v_global_scale > 0.f))
      return fail(KVQ_ERR_INVALID_ARG, "NVFP4 global scales must be finite and > 0");
  }
  if (pointers) {
    if (!c->k_codes || !c->v_codes) return fail(KVQ_ERR_INVALID_ARG, "code arrays are NULL");
    if (!aligned16(c->k_codes) || !aligned16(c->v_codes))
      return fail(KVQ_ERR_INVALID_ARG, "code arrays must be 16-byte aligned");
    if (c->format != KVQ_FMT_BF16) {
      if (!c->k_scales || !c->v_scales) return fail(KVQ_ERR_INVALID_ARG, "scale arrays are NULL");
      if (!aligned16(c->k_scales) || !aligned16(c->v_scales))
        return fail(KVQ_ERR_INVALID_ARG, "scale arrays must be 16-byte aligned");
    }
  }
  return KVQ_OK;
}

// --------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 5-D map over a codes array [num_pages][Hkv][16 rows][row_bytes]: dimensions
// (innermost first) 128 bytes of a row half, 16 rows (stride row_bytes), row
// halves (stride 128), KV heads (stride 16 * row_bytes), pages.  One box = the
// `hg` consecutive heads of one page, landing in shared memory as
// [head][half][row][128 bytes] with the 128-byte swizzle the decode kernel's
// ldmatrix addressing expects.  Rows of 64 bytes (NVFP4 at head_dim 128): a head
// block of 16 rows is read as 8 rows of 128 bytes (token pairs), one half.
int make_code_map(CUtensorMap* map, void* base, int64_t num_pages, int64_t hkv, int64_t rbytes, int hg) {
  auto fn = encode_fn();
  if (!fn) return fail(KVQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (rbytes != 64 && rbytes % 128 != 0) return fail(KVQ_ERR_UNSUPPORTED, "code rows of %lld bytes", (long long)rbytes);
  const int64_t rows = rbytes >= 128 ? 16 : 16 * rbytes / 128;  // 128-byte rows of a head block
  const int64_t halves = rbytes >= 128 ? rbytes / 128 : 1;
  const int64_t row_stride = rbytes >= 128 ? rbytes : 128;
  const cuuint64_t dims[5] = {128, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(halves),
                              static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(row_stride), 128, static_cast<cuuint64_t>(16 * rbytes),
                                 static_cast<cuuint64_t>(16 * rbytes * hkv)};
  const cuuint32_t box[5] = {128, static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(halves),
                             static_cast<cuuint32_t>(hg), 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KVQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return KVQ_OK;
}

// KV heads per decode work item for a cache (0 if no kernel exists for it).
// Plan layout offsets (int32 entries): the first-item descriptors and the rest
// list start on 16-byte boundaries so the kernel can load a descriptor at once.
int64_t plan_first_at(int64_t batch) { return (batch + 2 + 3) / 4 * 4; }
int64_t plan_rest_at(int64_t batch, int64_t C) { return (plan_first_at(batch) + 5 * C + 1 + 3) / 4 * 4; }

// Where a caller buffer lives: device (or managed) memory, or pinned host memory
// the kernels reach over the host link (*host = 1).  Pageable host memory is
// refused.
int memory_kind(const void* ptr, const char* name, int32_t* host) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) return cuda_fail(e, name);
  if (a.type == cudaMemoryTypeUnregistered)
    return fail(KVQ_ERR_INVALID_ARG, "%s is pageable host memory: pass device or pinned host memory", name);
  if (host) *host = a.type == cudaMemoryTypeHost ? 1 : 0;
  return KVQ_OK;
}

int heads_per_cta(const kvq_cache* c) {
  kvq::DecodeInstance inst;
  if (!kvq::decode_instance(c->format, c->head_dim, &inst)) return 0;
  return inst.head_group(c->num_kv_heads);
}

// --------------------------------------------------------------- decode instances
int prepare_instance(int format, int D, kvq::DecodeInstance* inst) {
  if (!kvq::decode_instance(format, D, inst))
    return fail(KVQ_ERR_UNSUPPORTED, "no decode kernel for format %d head_dim %d", format, D);
  static std::mutex mu;
  static bool done[64][4][2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(KVQ_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  bool& d = done[dev][format][D == 256 ? 1 : 0];
  if (!d) {
    // the kernel's warp roles split its launch registers (setmaxnreg): the split
    // is only valid for the register count it was written for
    for (const void* kern : inst->kernels) {
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(decode kernel)");
      if (inst->launch_regs > 0 && fa.numRegs != inst->launch_regs)
        return fail(KVQ_ERR_UNSUPPORTED, "decode kernel built with %d registers a thread, its register split assumes %d",
                    fa.numRegs, inst->launch_regs);
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, inst->smem_bytes);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
    }
    d = true;
  }
  return KVQ_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Key splits of a prefill-kernel launch: the split count S in [1, 64] (at least
// one 64-key tile a split) that minimises a model of the call's time, fitted to
// measured prefill calls at 32K keys (2,048 / 512 / 6 tokens, S = 1 .. 64):
//   waves(S) x (10 us + 1.9 us x tiles a split) + [S > 1] (3.5 us + partials)
// with waves(S) = ceil(items x S / CTAs a wave), one CTA an SM, and the merge's
// partials written and read once at 6 TB/s.  Ties go to the smaller S.
int64_t pick_key_splits(int64_t items, int64_t pages, int64_t partial_bytes_per_split, int64_t ctas) {
  const int64_t cap = std::max<int64_t>(1, std::min<int64_t>(64, pages / 4));
  int64_t best = 1;
  double best_us = 0.0;
  for (int64_t S = 1; S <= cap; ++S) {
    const int64_t waves = (items * S + ctas - 1) / ctas;
    const int64_t tiles = (pages + 4 * S - 1) / (4 * S);
    double us = (double)waves * (10.0 + 1.9 * (double)tiles);
    if (S > 1) us += 3.5 + 2.0 * (double)partial_bytes_per_split * (double)S / 6.0e6;
    if (S == 1 || us < best_us) {
      best = S;
      best_us = us;
    }
  }
  return best;
}

// A verify call with enough query tokens a sequence goes to the prefill kernel,
// one launch for the whole batch: it reads every key once for all q_len query
// tokens, where the decode kernel reads the keys once a query token, but it has
// the larger fixed cost
// (measured at 32K keys: the decode kernel ~11 + 9.6 q_len us, the prefill kernel
// ~46 us for INT8, ~38 us for NVFP4, whatever q_len up to a 128-row tile; at 8K
// keys ~9 + 2.6 q_len against ~22 us).  The query-token threshold therefore
// falls with the context, known on the host only through the block table's
// width: for one sequence 4 tokens from 2,048 pages (32K tokens) up, 5 from
// 1,024, 6 from 512, 10 below, fewer for NVFP4 (cheaper to convert on the
// tensor-core path: 3, 3, 4, 8).  For a batch
// the crossover comes later (8 sequences of 4K-16K, INT8: 148 us at 4 tokens
// against 123 on the decode kernel, 153 against 175 at 6; 64 sequences of
// 0.5K-8K: 407 against 483 at 6): 6 tokens, 4 for NVFP4.  The key splits of
// that launch come from pick_key_splits with the block table's width as the
// context.
// 0: the call stays on the decode kernel.
constexpr int kVerifyLongPages = 1024;

int verify_route_min_tokens(int format, int32_t nseq, int64_t max_pages) {
  const bool nv = format == KVQ_FMT_NVFP4;
  if (nseq > 1) return nv ? 4 : 6;
  // one sequence (measured crossovers: 2K keys, the decode kernel still wins at 6
  // tokens; 8K from 6, NVFP4 4; 16K from 5, NVFP4 3; 32K from 4, NVFP4 3)
  if (max_pages >= 2 * kVerifyLongPages) return nv ? 3 : 4;
  if (max_pages >= kVerifyLongPages) return nv ? 3 : 5;
  if (max_pages >= kVerifyLongPages / 2) return nv ? 4 : 6;
  return nv ? 8 : 10;
}

// sms <= 0: the current device's SM count.
int verify_route_splits(const kvq_cache* cache, int32_t nseq, int32_t q_len, int32_t num_q_heads, int32_t max_pages,
                        int32_t sms) {
  if (nseq < 1 || num_q_heads % cache->num_kv_heads) return 0;
  if (q_len < verify_route_min_tokens(cache->format, nseq, max_pages)) return 0;
  const int64_t G = num_q_heads / cache->num_kv_heads;
  kvq::PrefillInstance inst;
  if (!kvq::prefill_tc_instance(cache->format, cache->head_dim, &inst)) return 0;
  int dev = 0;
  if (sms <= 0 && (cudaGetDevice(&dev) != cudaSuccess ||
                   cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess))
    return 0;
  const int64_t items = (int64_t)nseq * (((int64_t)q_len * G + inst.rows - 1) / inst.rows) * cache->num_kv_heads;
  return static_cast<int>(
      pick_key_splits(items, max_pages, (int64_t)nseq * q_len * num_q_heads * cache->head_dim * 4, sms));
}

}  // namespace

int kvq::record_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_error = buf;
  return code;
}

extern "C" {

int64_t kvq_bytes_per_token(int32_t format, int32_t num_kv_heads, int32_t head_dim) {
  if (num_kv_heads <= 0 || head_dim <= 0 || head_dim % 16 != 0) return -1;
  const int64_t rb = row_bytes(format, head_dim), sb = scale_row_bytes(format, head_dim);
  if (rb < 0 || sb < 0) return -1;
  return 2 * (rb + sb) * num_kv_heads;
}

int kvq_cache_array_bytes(int32_t format, int32_t num_pages, int32_t page_size, int32_t num_kv_heads,
                          int32_t head_dim, int64_t* codes_bytes, int64_t* scales_bytes) {
  if (num_pages < 0 || page_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 16 != 0)
    return fail(KVQ_ERR_INVALID_ARG, "bad pool shape");
  const int64_t rb = row_bytes(format, head_dim), sb = scale_row_bytes(format, head_dim);
  if (rb < 0) return fail(KVQ_ERR_INVALID_ARG, "unknown cache format %d", format);
  const int64_t rows = (int64_t)num_pages * num_kv_heads * page_size;
  if (codes_bytes) *codes_bytes = rows * rb;
  if (scales_bytes) *scales_bytes = rows * sb;
  return succeed();
}

int kvq_quant_append(const kvq_cache* cache, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                     int64_t n_tokens, int32_t* dev_status, uint32_t flags, void* stream) {
  int rc = check_cache(cache, true);
  if (rc) return rc;
  if (n_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "n_tokens %lld < 0", (long long)n_tokens);
  if (n_tokens == 0) return succeed();
  if (!k_new || !v_new || !slot_mapping) return fail(KVQ_ERR_INVALID_ARG, "k_new, v_new or slot_mapping is NULL");
  if (!aligned16(k_new) || !aligned16(v_new)) return fail(KVQ_ERR_INVALID_ARG, "k_new / v_new must be 16-byte aligned");
  if (n_tokens > ((int64_t)1 << 40) / cache->num_kv_heads)
    return fail(KVQ_ERR_UNSUPPORTED, "too many rows in one append");
  const bool checked = flags & KVQ_CHECKED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t capacity = (int64_t)cache->num_pages * cache->page_size;
  if (checked) {
    if (!dev_status) return fail(KVQ_ERR_INVALID_ARG, "KVQ_CHECKED append needs dev_status");
    std::vector<int64_t> slots(n_tokens);
    cudaError_t e = cudaMemcpyAsync(slots.data(), slot_mapping, n_tokens * sizeof(int64_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading slot_mapping");
    std::vector<int64_t> valid;
    valid.reserve(n_tokens);
    for (int64_t i = 0; i < n_tokens; ++i) {
      if (slots[i] >= capacity)
        return fail(KVQ_ERR_INVALID_ARG, "slot_mapping[%lld] = %lld >= capacity %lld", (long long)i,
                    (long long)slots[i], (long long)capacity);
      if (slots[i] >= 0) valid.push_back(slots[i]);
    }
    std::sort(valid.begin(), valid.end());
    const auto dup = std::adjacent_find(valid.begin(), valid.end());
    if (dup != valid.end()) return fail(KVQ_ERR_INVALID_ARG, "duplicate valid slot %lld in one append", (long long)*dup);
  }
  kvq::AppendParams p{};
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.slots = slot_mapping;
  p.k_codes = static_cast<uint8_t*>(cache->k_codes);
  p.v_codes = static_cast<uint8_t*>(cache->v_codes);
  p.k_scales = static_cast<uint8_t*>(cache->k_scales);
  p.v_scales = static_cast<uint8_t*>(cache->v_scales);
  p.status = dev_status;
  p.n_tokens = n_tokens;
  p.capacity = capacity;
  p.num_kv_heads = cache->num_kv_heads;
  p.check_finite = checked ? 1 : 0;
  p.rotate = (flags & KVQ_ROTATE) ? 1 : 0;
  p.k_gs = cache->k_global_scale;
  p.v_gs = cache->v_global_scale;
  cudaError_t e = kvq::launch_append(cache->format, cache->head_dim, p, st);
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  if (checked) {
    int32_t bits = 0;
    rc = kvq_read_status(dev_status, stream, &bits);
    if (rc) return rc;
  }
  return succeed();
}

int kvq_plan_splits(const kvq_cache* cache, const int32_t* seq_lens, int32_t batch, int32_t split_override,
                    int32_t target_ctas, int32_t* plan, int64_t plan_capacity, int32_t* total_splits,
                    int32_t* num_ctas) {
  int rc = check_cache(cache, false);
  if (rc) return rc;
  if (batch < 1) return fail(KVQ_ERR_INVALID_ARG, "batch %d < 1", batch);
  if (!seq_lens || !total_splits || !num_ctas) return fail(KVQ_ERR_INVALID_ARG, "NULL argument");
  if (split_override < 0 || target_ctas < 0) return fail(KVQ_ERR_INVALID_ARG, "negative split_override / target_ctas");
  const int hgs = heads_per_cta(cache);
  if (hgs <= 0) return fail(KVQ_ERR_UNSUPPORTED, "no decode kernel for this cache");
  const int nhg = cache->num_kv_heads / hgs;
  const int P = cache->page_size;
  std::vector<int64_t> npages(batch);
  int64_t total_pages = 0;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens[b] < 0) return fail(KVQ_ERR_INVALID_ARG, "seq_lens[%d] = %d < 0", b, seq_lens[b]);
    npages[b] = (seq_lens[b] + P - 1) / P;
    total_pages += npages[b];
  }
  int64_t target = target_ctas;
  if (target == 0) {
    kvq::DecodeInstance inst;
    rc = prepare_instance(cache->format, cache->head_dim, &inst);
    if (rc) return rc;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, inst.kernels[0], inst.threads, inst.smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "querying SM count / occupancy");
    target = (int64_t)sms * std::max(per_sm, 1);
  }
  target = std::max<int64_t>(target, 1);
  // Cost of a work item for the packing: its pages plus a fixed per-item cost
  // (prologue, epilogue and merge share), in page units.
  constexpr int64_t kItemCost = 8;
  // Longest-first packing of the items of a split choice onto C = min(target,
  // items) CTAs: returns the largest CTA load (the critical path).
  auto makespan = [&](const std::vector<int32_t>& sp) -> int64_t {
    std::vector<int64_t> sizes;
    for (int b = 0; b < batch; ++b)
      for (int s = 0; s < sp[b]; ++s) {
        const int64_t sz = (int64_t)(s + 1) * npages[b] / sp[b] - (int64_t)s * npages[b] / sp[b];
        for (int g = 0; g < nhg; ++g) sizes.push_back(sz + kItemCost);
      }
    std::sort(sizes.begin(), sizes.end(), std::greater<int64_t>());
    const int64_t C = std::min<int64_t>(target, (int64_t)sizes.size());
    std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> bins;
    for (int64_t i = 0; i < C; ++i) bins.push(0);
    int64_t worst = 0;
    for (int64_t sz : sizes) {
      const int64_t l = bins.top() + sz;
      bins.pop();
      bins.push(l);
      worst = std::max(worst, l);
    }
    return worst;
  };
  std::vector<int32_t> splits(batch, 1);
  if (split_override > 0) {
    for (int b = 0; b < batch; ++b)
      splits[b] = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(split_override, std::max<int64_t>(npages[b], 1))));
  } else {
    // Pages per split x = units / (target * m) for a few oversubscription factors
    // m (at least 4 pages): a sequence of n pages gets ceil(n / x) splits.  The
    // choice with the shortest critical path wins (ties: fewer items).
    const int64_t units = total_pages * nhg;  // (page, head group) units
    const double ms[] = {1.0, 1.25, 1.5, 2.0, 2.5, 3.0, 4.0, 6.0};
    int64_t best = -1, best_items = 0;
    for (double m : ms) {
      const double x = std::max(4.0, (double)units / ((double)target * m));
      std::vector<int32_t> sp(batch);
      int64_t items = 0;
      for (int b = 0; b < batch; ++b) {
        sp[b] = static_cast<int32_t>(std::max<int64_t>(1, (int64_t)std::ceil((double)npages[b] / x - 1e-9)));
        items += (int64_t)sp[b] * nhg;
      }
      const int64_t span = makespan(sp);
      if (best < 0 || span < best || (span == best && items < best_items)) {
        best = span;
        best_items = items;
        splits = sp;
      }
    }
    // Whole waves: for k = 1..4, the fewest pages per split whose items fit in
    // k x target (a batch of uneven sequences rarely lands just under a wave with
    // the factors above).  Taken only when strictly shorter.
    int64_t max_pages = 1;
    for (int b = 0; b < batch; ++b) max_pages = std::max(max_pages, npages[b]);
    auto items_at = [&](int64_t x) {
      int64_t n = 0;
      for (int b = 0; b < batch; ++b) n += std::max<int64_t>(1, (npages[b] + x - 1) / x) * nhg;
      return n;
    };
    for (int k = 1; k <= 4; ++k) {
      int64_t lo = 4, hi = std::max<int64_t>(4, max_pages);  // items_at is non-increasing in x
      if (items_at(hi) > k * target) continue;
      while (lo < hi) {
        const int64_t mid = (lo + hi) / 2;
        if (items_at(mid) <= k * target) hi = mid;
        else lo = mid + 1;
      }
      std::vector<int32_t> sp(batch);
      for (int b = 0; b < batch; ++b)
        sp[b] = static_cast<int32_t>(std::max<int64_t>(1, (npages[b] + lo - 1) / lo));
      const int64_t span = makespan(sp);
      if (span < best) {
        best = span;
        best_items = items_at(lo);
        splits = sp;
      }
    }
  }
  int64_t total = 0;
  for (int b = 0; b < batch; ++b) total += splits[b];
  if (total * nhg > 0x7FFFFFFF / 2) return fail(KVQ_ERR_UNSUPPORTED, "too many splits");
  const int64_t n_items = total * nhg;
  const int64_t C = std::min<int64_t>(target, n_items);  // persistent CTAs
  *total_splits = static_cast<int32_t>(total);
  *num_ctas = static_cast<int32_t>(C);
  if (nhg > 127) return fail(KVQ_ERR_UNSUPPORTED, "more than 127 KV-head groups");
  const int64_t A = plan_first_at(batch);
  const int64_t roff_at = A + 4 * C;
  const int64_t rest_at = plan_rest_at(batch, C);
  const int64_t need = rest_at + 4 * (n_items - C);
  if (!plan || plan_capacity < need)
    return fail(KVQ_ERR_WORKSPACE, "plan needs %lld int32 entries", (long long)need);
  for (int b = 0; b < batch; ++b)
    if (npages[b] >= (1 << 23)) return fail(KVQ_ERR_UNSUPPORTED, "sequence %d has too many pages", b);
  plan[0] = 0;
  for (int b = 0; b < batch; ++b) plan[b + 1] = plan[b] + splits[b];
  plan[batch + 1] = static_cast<int32_t>(C);
  for (int64_t i = batch + 2; i < A; ++i) plan[i] = 0;
  // Items with their descriptors and page counts; longest first, each onto the
  // CTA with the least work so far (a page costs 1, an item kItemCost more).
  struct Desc {
    int64_t cost;
    int32_t d[4];
  };
  std::vector<Desc> items;
  items.reserve(n_items);
  for (int b = 0; b < batch; ++b)
    for (int s = 0; s < splits[b]; ++s) {
      const int64_t pb = (int64_t)s * npages[b] / splits[b], pe = (int64_t)(s + 1) * npages[b] / splits[b];
      for (int g = 0; g < nhg; ++g) {
        Desc it;
        it.cost = pe - pb;
        it.d[0] = b;
        it.d[1] = plan[b] + s;
        it.d[2] = static_cast<int32_t>(pb);
        it.d[3] = static_cast<int32_t>((pe - pb) | ((splits[b] == 1 ? 1 : 0) << 23) | (g << 24));
        items.push_back(it);
      }
    }
  std::stable_sort(items.begin(), items.end(), [](const Desc& a, const Desc& b) { return a.cost > b.cost; });
  std::vector<std::vector<int64_t>> bins(C);
  std::vector<std::pair<int64_t, int32_t>> heap;  // (load, cta) min-heap
  heap.reserve(C);
  for (int32_t cta = 0; cta < C; ++cta) heap.emplace_back(0, cta);
  auto cmp = [](const auto& a, const auto& b) { return a.first > b.first || (a.first == b.first && a.second > b.second); };
  std::make_heap(heap.begin(), heap.end(), cmp);
  for (int64_t i = 0; i < n_items; ++i) {
    std::pop_heap(heap.begin(), heap.end(), cmp);
    auto& top = heap.back();
    bins[top.second].push_back(i);
    top.first += items[i].cost + kItemCost;
    std::push_heap(heap.begin(), heap.end(), cmp);
  }
  int32_t* roff = plan + roff_at;
  for (int64_t i = roff_at + C + 1; i < rest_at; ++i) plan[i] = 0;
  roff[0] = 0;
  for (int64_t cta = 0; cta < C; ++cta) {
    const auto& bin = bins[cta];  // never empty: the first C items go to distinct CTAs
    std::copy(items[bin[0]].d, items[bin[0]].d + 4, plan + A + 4 * cta);
    roff[cta + 1] = roff[cta] + static_cast<int32_t>(bin.size() - 1);
    for (size_t k = 1; k < bin.size(); ++k)
      std::copy(items[bin[k]].d, items[bin[k]].d + 4, plan + rest_at + 4 * (roff[cta] + k - 1));
  }
  return succeed();
}

int kvq_plan_verify_splits(const kvq_cache* cache, const int32_t* seq_lens, int32_t batch, int32_t q_len,
                           int32_t split_override, int32_t target_ctas, int32_t* plan, int64_t plan_capacity,
                           int32_t* total_splits, int32_t* num_ctas) {
  if (batch < 1) return fail(KVQ_ERR_INVALID_ARG, "batch %d < 1", batch);
  if (q_len < 1) return fail(KVQ_ERR_INVALID_ARG, "q_len %d < 1", q_len);
  if (!seq_lens) return fail(KVQ_ERR_INVALID_ARG, "seq_lens is NULL");
  if ((int64_t)batch * q_len > 0x7FFFFFFF / 4) return fail(KVQ_ERR_UNSUPPORTED, "batch x q_len too large");
  // query token i of sequence b sees the first L_b - q_len + 1 + i tokens (causal)
  std::vector<int32_t> lens((size_t)batch * q_len);
  for (int32_t b = 0; b < batch; ++b) {
    if (seq_lens[b] < 0) return fail(KVQ_ERR_INVALID_ARG, "seq_lens[%d] = %d < 0", b, seq_lens[b]);
    for (int32_t i = 0; i < q_len; ++i)
      lens[(size_t)b * q_len + i] = std::max(0, seq_lens[b] - q_len + 1 + i);
  }
  return kvq_plan_splits(cache, lens.data(), batch * q_len, split_override, target_ctas, plan, plan_capacity,
                         total_splits, num_ctas);
}

size_t kvq_decode_workspace_bytes(int32_t total_splits, int32_t num_q_heads, int32_t head_dim) {
  if (total_splits < 0 || num_q_heads < 0 || head_dim < 0) return 0;
  const size_t rows = (size_t)total_splits * num_q_heads;
  // status, lse partials, o partials, and room for a bf16 copy of q (total_splits >= rows of q)
  return 256 + align256(rows * sizeof(float)) + align256(rows * head_dim * sizeof(float)) + rows * head_dim * 2;
}

size_t kvq_verify_workspace_bytes(const kvq_cache* cache, int32_t batch, int32_t q_len, int32_t num_q_heads,
                                  int32_t total_splits, int32_t target_ctas) {
  if (batch < 1 || q_len < 1 || num_q_heads < 1 || total_splits < 0) {
    fail(KVQ_ERR_INVALID_ARG, "bad batch %d / q_len %d / num_q_heads %d / total_splits %d", batch, q_len, num_q_heads,
         total_splits);
    return 0;
  }
  if (check_cache(cache, false)) return 0;  // the reason is recorded
  if (target_ctas <= 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&target_ctas, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      cuda_fail(e, "querying the SM count");
      return 0;
    }
  }
  const size_t decode_need = kvq_decode_workspace_bytes(total_splits, num_q_heads, cache->head_dim);
  // a block table of 2^20 pages (16M tokens): the lowest token threshold, and as
  // many splits as any shorter table gets
  const int S = verify_route_splits(cache, batch, q_len, num_q_heads, 1 << 20, target_ctas);
  succeed();
  if (S <= 0) return decode_need;
  return std::max(decode_need, kvq_prefill_workspace_bytes(batch * q_len, num_q_heads, cache->head_dim, S));
}

int kvq_workspace_partials(void* workspace, int32_t total_splits, int32_t num_q_heads, int32_t head_dim,
                           float** o_part, float** lse_part) {
  if (!workspace || !o_part || !lse_part || total_splits < 0 || num_q_heads < 0 || head_dim < 0)
    return fail(KVQ_ERR_INVALID_ARG, "bad workspace arguments");
  const size_t rows = (size_t)total_splits * num_q_heads;
  char* base = static_cast<char*>(workspace);
  *lse_part = reinterpret_cast<float*>(base + 256);
  *o_part = reinterpret_cast<float*>(base + 256 + align256(rows * sizeof(float)));
  return succeed();
}

}  // extern "C"

namespace {

// The tensor-core prefill launch (and its merge) once every argument has been
// checked: q_len query tokens of each of `batch` sequences (block_table
// [batch][max_pages]), the length from the host (seq_len, batch 1) or, when
// seq_len_dev is not null, read by the kernel from device memory (a verify call).
int prefill_launch(const kvq_cache* cache, const void* q, int32_t batch, int32_t q_len, int32_t num_q_heads,
                   float sm_scale, const int32_t* block_table, int32_t max_pages, int32_t seq_len,
                   const int32_t* seq_len_dev, int32_t splits, void* workspace, void* out, int32_t out_dtype,
                   float* lse_out, uint32_t flags, void* stream) {
  const int D = cache->head_dim;
  const int G = num_q_heads / cache->num_kv_heads;
  kvq::PrefillInstance inst;
  if (!kvq::prefill_tc_instance(cache->format, D, &inst))
    return fail(KVQ_ERR_UNSUPPORTED, "no prefill kernel for format %d head_dim %d", cache->format, D);
  {
    static std::mutex mu;
    static bool done[64][4][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(KVQ_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    bool& d = done[dev][cache->format][D == 256 ? 1 : 0];
    if (!d) {
      for (const void* kern : inst.kernels) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(prefill kernel)");
        if (inst.launch_regs > 0 && fa.numRegs != inst.launch_regs)
          return fail(KVQ_ERR_UNSUPPORTED,
                      "prefill kernel built with %d registers a thread, its register split assumes %d", fa.numRegs,
                      inst.launch_regs);
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, inst.smem_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
      }
      d = true;
    }
  }
  kvq::PrefillParams p{};
  p.q = q;
  p.block_table = block_table;
  p.k_codes = static_cast<const uint8_t*>(cache->k_codes);
  p.v_codes = static_cast<const uint8_t*>(cache->v_codes);
  p.k_scales = static_cast<const uint8_t*>(cache->k_scales);
  p.v_scales = static_cast<const uint8_t*>(cache->v_scales);
  const size_t rows = splits > 1 ? (size_t)batch * q_len * splits * num_q_heads : 0;
  char* ws = static_cast<char*>(workspace);
  p.status = reinterpret_cast<int32_t*>(ws);
  p.lse_part = reinterpret_cast<float*>(ws + 256);
  p.o_part = reinterpret_cast<float*>(ws + 256 + align256(rows * sizeof(float)));
  p.out = out;
  p.lse_out = lse_out;
  p.batch = batch;
  p.q_len = q_len;
  p.seq_len = seq_len;
  p.seq_len_dev = seq_len_dev;
  p.max_pages = max_pages;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.num_pages = cache->num_pages;
  p.splits = splits;
  p.row_blocks = (q_len * G + inst.rows - 1) / inst.rows;
  p.out_bf16 = out_dtype == KVQ_OUT_BF16;
  p.sm_scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
  p.k_gs_inv = cache->format == KVQ_FMT_NVFP4 ? 1.0f / cache->k_global_scale : 1.0f;
  p.v_gs_inv = cache->format == KVQ_FMT_NVFP4 ? 1.0f / cache->v_global_scale : 1.0f;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t grid = (int64_t)batch * p.row_blocks * cache->num_kv_heads * splits;
  if (grid > 0x7FFFFFFF) return fail(KVQ_ERR_UNSUPPORTED, "grid too large");
  cudaError_t e = kvq::launch_prefill_tc(cache->format, D, p, static_cast<int>(grid), st);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  if (splits > 1) {
    e = kvq::launch_merge(p.o_part, p.lse_part, nullptr, splits, batch * q_len, num_q_heads, D, out, p.out_bf16,
                          lse_out, false, st);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  }
  if (flags & KVQ_CHECKED) {
    int32_t bits = 0;
    const int rc = kvq_read_status(workspace, stream, &bits);
    if (rc) return rc;
  }
  return succeed();
}

// Decode (q_len = 1) or causal verification of q_len tokens a sequence: the
// launch works on batch = nseq x q_len virtual sequences (query token i of cache
// sequence b is virtual sequence b * q_len + i, with b's block table and
// L_b - q_len + 1 + i visible tokens).
// clear_status: zero the workspace's status block on the stream once every
// argument has been checked, just before the first launch (a rejected call
// leaves the block as it was).
int decode_impl(const kvq_cache* cache, const void* q, int32_t nseq, int32_t q_len, int32_t num_q_heads,
                float sm_scale, const int32_t* block_tables, int32_t max_pages_per_seq, const int32_t* seq_lens,
                const int32_t* plan, int32_t total_splits, int32_t num_ctas, void* workspace, size_t workspace_bytes,
                void* out, int32_t out_dtype, float* lse_out, uint32_t flags, void* stream, bool clear_status = false) {
  int rc = check_cache(cache, true);
  if (rc) return rc;
  if (nseq < 1) return fail(KVQ_ERR_INVALID_ARG, "batch %d < 1", nseq);
  if (q_len < 1) return fail(KVQ_ERR_INVALID_ARG, "q_len %d < 1", q_len);
  if ((int64_t)nseq * q_len > 0x7FFFFFFF / 4) return fail(KVQ_ERR_UNSUPPORTED, "batch x q_len too large");
  const int32_t batch = nseq * q_len;  // virtual sequences of the launch
  if (!q || !block_tables || !seq_lens || !plan || !workspace || !out)
    return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer argument");
  if (num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                cache->num_kv_heads);
  const int G = num_q_heads / cache->num_kv_heads;
  if (G > 8) return fail(KVQ_ERR_UNSUPPORTED, "query heads per KV head %d > 8", G);
  if (max_pages_per_seq < 1) return fail(KVQ_ERR_INVALID_ARG, "max_pages_per_seq %d < 1", max_pages_per_seq);
  if (total_splits < batch) return fail(KVQ_ERR_INVALID_ARG, "total_splits %d < batch %d", total_splits, batch);
  if (num_ctas < 1) return fail(KVQ_ERR_INVALID_ARG, "num_ctas %d < 1", num_ctas);
  if ((int64_t)total_splits * cache->num_kv_heads > 0x7FFFFFFF) return fail(KVQ_ERR_UNSUPPORTED, "grid too large");
  if (out_dtype != KVQ_OUT_F32 && out_dtype != KVQ_OUT_BF16) return fail(KVQ_ERR_INVALID_ARG, "bad out_dtype");
  if (!(std::isfinite(sm_scale))) return fail(KVQ_ERR_INVALID_ARG, "sm_scale must be finite");
  if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(KVQ_ERR_INVALID_ARG, "q / out must be 16-byte aligned and workspace 256-byte aligned");
  const int D = cache->head_dim;
  const size_t need = kvq_decode_workspace_bytes(total_splits, num_q_heads, D);
  if (workspace_bytes < need)
    return fail(KVQ_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool checked = flags & KVQ_CHECKED;
  if (checked) {
    for (const auto& pr : {std::make_pair(q, "q"), std::make_pair(static_cast<const void*>(block_tables), "block_tables"),
                           std::make_pair(static_cast<const void*>(seq_lens), "seq_lens"),
                           std::make_pair(static_cast<const void*>(plan), "plan")}) {
      rc = memory_kind(pr.first, pr.second, nullptr);
      if (rc) return rc;
    }
    // host-side validation of the plan against seq_lens (the kernel also checks
    // every descriptor it uses)
    const int hgc = heads_per_cta(cache);
    if (hgc <= 0) return fail(KVQ_ERR_UNSUPPORTED, "no decode kernel for this cache");
    const int64_t nhg_checked = cache->num_kv_heads / hgc;
    const int64_t n_items = (int64_t)total_splits * nhg_checked;
    if (num_ctas > n_items) return fail(KVQ_ERR_INVALID_ARG, "num_ctas %d exceeds the number of work items", num_ctas);
    const int64_t A = plan_first_at(batch), roff_at = A + 4 * (int64_t)num_ctas;
    const int64_t rest_at = plan_rest_at(batch, num_ctas);
    std::vector<int32_t> h(rest_at + 4 * (n_items - num_ctas));
    std::vector<int32_t> real(nseq), lens(batch);
    cudaError_t e = cudaMemcpyAsync(h.data(), plan, h.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(real.data(), seq_lens, real.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading plan");
    for (int b = 0; b < nseq; ++b) {
      if (real[b] < 0) return fail(KVQ_ERR_INVALID_ARG, "seq_lens[%d] = %d < 0", b, real[b]);
      for (int i = 0; i < q_len; ++i) lens[b * q_len + i] = std::max(0, real[b] - (q_len - 1 - i));
    }
    if (h[0] != 0 || h[batch] != total_splits) return fail(KVQ_ERR_INVALID_ARG, "plan offsets do not span total_splits");
    for (int b = 0; b < batch; ++b)
      if (h[b + 1] <= h[b]) return fail(KVQ_ERR_INVALID_ARG, "plan gives sequence %d no split", b);
    if (h[batch + 1] != num_ctas)
      return fail(KVQ_ERR_INVALID_ARG, "plan CTA count %d != num_ctas %d", h[batch + 1], num_ctas);
    const int32_t* ro = h.data() + roff_at;
    if (ro[0] != 0 || ro[num_ctas] != n_items - num_ctas)
      return fail(KVQ_ERR_INVALID_ARG, "plan CTA offsets do not span the items");
    for (int64_t i = 0; i < num_ctas; ++i)
      if (ro[i + 1] < ro[i]) return fail(KVQ_ERR_INVALID_ARG, "plan CTA offsets decrease");
    std::vector<uint8_t> seen(n_items, 0);
    for (int64_t i = 0; i < n_items; ++i) {
      const int32_t* d = i < num_ctas ? h.data() + A + 4 * i : h.data() + rest_at + 4 * (i - num_ctas);
      const int b = d[0], split = d[1], pb = d[2];
      const int n = d[3] & 0x7FFFFF, direct = (d[3] >> 23) & 1, g = (uint32_t)d[3] >> 24;
      if (b < 0 || b >= batch || split < h[b] || split >= h[b + 1] || g >= nhg_checked)
        return fail(KVQ_ERR_INVALID_ARG, "plan item %lld names a bad sequence / split / head group", (long long)i);
      const int64_t S = h[b + 1] - h[b], sidx = split - h[b];
      const int64_t np = (lens[b] + cache->page_size - 1) / cache->page_size;
      if (pb != sidx * np / S || n != (sidx + 1) * np / S - pb || direct != (S == 1 ? 1 : 0))
        return fail(KVQ_ERR_INVALID_ARG, "plan item %lld does not match sequence %d's %d visible tokens", (long long)i,
                    b, lens[b]);
      if (pb + n > max_pages_per_seq)
        return fail(KVQ_ERR_INVALID_ARG, "plan item %lld runs past the block table", (long long)i);
      const int64_t key = (int64_t)split * nhg_checked + g;
      if (seen[key]) return fail(KVQ_ERR_INVALID_ARG, "plan item (split %d, group %d) appears twice", split, g);
      seen[key] = 1;
    }
  }
  int32_t q_host = 0, out_host = 0;
  rc = memory_kind(q, "q", &q_host);
  if (rc) return rc;
  rc = memory_kind(out, "out", &out_host);
  if (rc) return rc;
  // enough query tokens: the tensor-core prefill kernel (the plan was checked
  // above all the same, so a call is accepted or refused alike on both paths)
  if (!clear_status && !q_host && !out_host && !(flags & (KVQ_SKIP_MERGE | KVQ_TEST_STALL))) {
    const int S = verify_route_splits(cache, nseq, q_len, num_q_heads, max_pages_per_seq, 0);
    if (S > 0 && workspace_bytes >= kvq_prefill_workspace_bytes(nseq * q_len, num_q_heads, D, S))
      return prefill_launch(cache, q, nseq, q_len, num_q_heads, sm_scale, block_tables, max_pages_per_seq, 0,
                            seq_lens, S, workspace, out, out_dtype, lse_out, flags, stream);
  }
  kvq::DecodeInstance inst;
  rc = prepare_instance(cache->format, D, &inst);
  if (rc) return rc;
  const int hg = heads_per_cta(cache);
  if (hg <= 0 || cache->num_kv_heads % hg != 0) return fail(KVQ_ERR_UNSUPPORTED, "bad KV head grouping");
  CUtensorMap tk, tv;
  rc = make_code_map(&tk, cache->k_codes, cache->num_pages, cache->num_kv_heads, row_bytes(cache->format, D), hg);
  if (rc) return rc;
  rc = make_code_map(&tv, cache->v_codes, cache->num_pages, cache->num_kv_heads, row_bytes(cache->format, D), hg);
  if (rc) return rc;
  float *o_part = nullptr, *lse_part = nullptr;
  kvq_workspace_partials(workspace, total_splits, num_q_heads, D, &o_part, &lse_part);
  if (clear_status) {
    const cudaError_t ec = cudaMemsetAsync(workspace, 0, 256, st);
    if (ec != cudaSuccess) return cuda_fail(ec, "clearing the status block");
  }
  // q in pinned host memory: one copy into the workspace, read by the decode
  const void* q_dev = q;
  if (q_host) {
    const size_t rows = (size_t)total_splits * num_q_heads;
    void* q_stage = reinterpret_cast<char*>(o_part) + align256(rows * D * sizeof(float));
    const cudaError_t es = kvq::launch_q_stage(q, q_stage, (size_t)batch * num_q_heads * D * 2, st);
    if (es != cudaSuccess) return cuda_fail(es, "q staging launch");
    q_dev = q_stage;
  }
  kvq::DecodeParams p{};
  p.q = q_dev;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.plan = plan;
  p.k_scales = static_cast<const uint8_t*>(cache->k_scales);
  p.v_scales = static_cast<const uint8_t*>(cache->v_scales);
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.out = out;
  p.lse_out = lse_out;
  p.status = static_cast<int32_t*>(workspace);
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.max_pages = max_pages_per_seq;
  p.num_pages = cache->num_pages;
  p.total_splits = total_splits;
  p.heads_per_cta = hg;
  p.out_bf16 = out_dtype == KVQ_OUT_BF16;
  p.early_start = (flags & KVQ_EARLY_START) ? 1 : 0;
  p.drop_copies = (flags & KVQ_TEST_STALL) ? 1 : 0;
  p.wait_limit_ns = (flags & KVQ_TEST_STALL) ? 2000000ull : 2000000000ull;  // 2 ms / 2 s
  p.q_len = q_len;
  p.out_host = out_host;
  p.sm_scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
  p.k_gs_inv = cache->format == KVQ_FMT_NVFP4 ? 1.0f / cache->k_global_scale : 1.0f;
  p.v_gs_inv = cache->format == KVQ_FMT_NVFP4 ? 1.0f / cache->v_global_scale : 1.0f;
  // one persistent CTA per plan bin
  cudaError_t e = kvq::launch_decode(cache->format, D, tk, tv, p, num_ctas, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (!(flags & KVQ_SKIP_MERGE) && total_splits > batch) {
    // the split offsets come from the plan, which the decode kernel never writes
    e = kvq::launch_merge(o_part, lse_part, plan, 0, batch, num_q_heads, D, out, p.out_bf16, lse_out, true, st);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  }
  if (checked) {
    int32_t bits = 0;
    rc = kvq_read_status(workspace, stream, &bits);
    if (rc) return rc;
  }
  return succeed();
}

}  // namespace

int kvq::decode_clearing_status(const kvq_cache* cache, const void* q, int32_t batch, int32_t num_q_heads,
                                float sm_scale, const int32_t* block_tables, int32_t max_pages_per_seq,
                                const int32_t* seq_lens, const int32_t* plan, int32_t total_splits, int32_t num_ctas,
                                void* workspace, size_t workspace_bytes, void* out, int32_t out_dtype, float* lse_out,
                                uint32_t flags, void* stream) {
  return decode_impl(cache, q, batch, 1, num_q_heads, sm_scale, block_tables, max_pages_per_seq, seq_lens, plan,
                     total_splits, num_ctas, workspace, workspace_bytes, out, out_dtype, lse_out, flags, stream, true);
}

extern "C" {

int kvq_paged_decode_attention(const kvq_cache* cache, const void* q, int32_t batch, int32_t num_q_heads,
                               float sm_scale, const int32_t* block_tables, int32_t max_pages_per_seq,
                               const int32_t* seq_lens, const int32_t* plan, int32_t total_splits,
                               int32_t num_ctas, void* workspace, size_t workspace_bytes, void* out,
                               int32_t out_dtype, float* lse_out, uint32_t flags, void* stream) {
  return decode_impl(cache, q, batch, 1, num_q_heads, sm_scale, block_tables, max_pages_per_seq, seq_lens, plan,
                     total_splits, num_ctas, workspace, workspace_bytes, out, out_dtype, lse_out, flags, stream);
}

int kvq_paged_verify_attention(const kvq_cache* cache, const void* q, int32_t batch, int32_t q_len,
                               int32_t num_q_heads, float sm_scale, const int32_t* block_tables,
                               int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* plan,
                               int32_t total_splits, int32_t num_ctas, void* workspace, size_t workspace_bytes,
                               void* out, int32_t out_dtype, float* lse_out, uint32_t flags, void* stream) {
  return decode_impl(cache, q, batch, q_len, num_q_heads, sm_scale, block_tables, max_pages_per_seq, seq_lens, plan,
                     total_splits, num_ctas, workspace, workspace_bytes, out, out_dtype, lse_out, flags, stream);
}

int32_t kvq_prefill_splits(const kvq_cache* cache, int32_t q_len, int32_t num_q_heads, int32_t seq_len,
                           int32_t target_ctas) {
  int rc = check_cache(cache, false);
  if (rc) return -rc;
  if (q_len < 1 || seq_len < q_len || num_q_heads < 1 || num_q_heads % cache->num_kv_heads)
    return -fail(KVQ_ERR_INVALID_ARG, "bad q_len %d / seq_len %d / num_q_heads %d", q_len, seq_len, num_q_heads);
  kvq::PrefillInstance inst;
  if (!kvq::prefill_tc_instance(cache->format, cache->head_dim, &inst))
    return -fail(KVQ_ERR_UNSUPPORTED, "no prefill kernel for format %d head_dim %d", cache->format, cache->head_dim);
  int64_t target = target_ctas;
  if (target <= 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return -cuda_fail(e, "querying the SM count");
    target = sms;
  }
  const int64_t G = num_q_heads / cache->num_kv_heads;
  const int64_t items = (q_len * G + inst.rows - 1) / inst.rows * cache->num_kv_heads;
  const int64_t pages = (seq_len + cache->page_size - 1) / cache->page_size;
  const int64_t S = pick_key_splits(items, pages, (int64_t)q_len * num_q_heads * cache->head_dim * 4, target);
  succeed();
  return static_cast<int32_t>(S);
}

size_t kvq_prefill_workspace_bytes(int32_t q_len, int32_t num_q_heads, int32_t head_dim, int32_t splits) {
  if (q_len < 0 || num_q_heads < 0 || head_dim < 0 || splits < 1) return 0;
  const size_t rows = splits > 1 ? (size_t)q_len * splits * num_q_heads : 0;
  return 256 + align256(rows * sizeof(float)) + rows * head_dim * sizeof(float);
}

int kvq_paged_prefill_attention(const kvq_cache* cache, const void* q, int32_t q_len, int32_t num_q_heads,
                                float sm_scale, const int32_t* block_table, int32_t max_pages, int32_t seq_len,
                                int32_t splits, void* workspace, size_t workspace_bytes, void* out,
                                int32_t out_dtype, float* lse_out, uint32_t flags, void* stream) {
  int rc = check_cache(cache, true);
  if (rc) return rc;
  if (!q || !block_table || !workspace || !out) return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer argument");
  if (q_len < 1 || seq_len < q_len) return fail(KVQ_ERR_INVALID_ARG, "q_len %d must be in [1, seq_len %d]", q_len, seq_len);
  if (num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                cache->num_kv_heads);
  const int G = num_q_heads / cache->num_kv_heads;
  if (G > 8) return fail(KVQ_ERR_UNSUPPORTED, "query heads per KV head %d > 8", G);
  if ((int64_t)(seq_len + cache->page_size - 1) / cache->page_size > max_pages)
    return fail(KVQ_ERR_INVALID_ARG, "seq_len %d needs more than max_pages %d pages", seq_len, max_pages);
  if (splits < 1 || splits > 64) return fail(KVQ_ERR_INVALID_ARG, "splits %d not in [1, 64]", splits);
  if (out_dtype != KVQ_OUT_F32 && out_dtype != KVQ_OUT_BF16) return fail(KVQ_ERR_INVALID_ARG, "bad out_dtype");
  if (!std::isfinite(sm_scale)) return fail(KVQ_ERR_INVALID_ARG, "sm_scale must be finite");
  if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(KVQ_ERR_INVALID_ARG, "q / out must be 16-byte aligned and workspace 256-byte aligned");
  const int D = cache->head_dim;
  const size_t need = kvq_prefill_workspace_bytes(q_len, num_q_heads, D, splits);
  if (workspace_bytes < need) return fail(KVQ_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  rc = memory_kind(out, "out", nullptr);
  if (rc) return rc;
  return prefill_launch(cache, q, 1, q_len, num_q_heads, sm_scale, block_table, max_pages, seq_len, nullptr, splits,
                        workspace, out, out_dtype, lse_out, flags, stream);
}

int kvq_split_merge(const float* o_part, const float* lse_part, const int32_t* split_offsets, int32_t batch,
                    int32_t num_q_heads, int32_t head_dim, void* out, int32_t out_dtype, float* lse_out,
                    void* stream) {
  if (!o_part || !lse_part || !split_offsets || !out) return fail(KVQ_ERR_INVALID_ARG, "NULL device pointer argument");
  if (batch < 1 || num_q_heads < 1) return fail(KVQ_ERR_INVALID_ARG, "batch / num_q_heads < 1");
  if (head_dim != 128 && head_dim != 256) return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d", head_dim);
  if (out_dtype != KVQ_OUT_F32 && out_dtype != KVQ_OUT_BF16) return fail(KVQ_ERR_INVALID_ARG, "bad out_dtype");
  if (!aligned16(o_part) || !aligned16(out)) return fail(KVQ_ERR_INVALID_ARG, "o_part / out must be 16-byte aligned");
  cudaError_t e = kvq::launch_merge(o_part, lse_part, split_offsets, 0, batch, num_q_heads, head_dim, out,
                                    out_dtype == KVQ_OUT_BF16, lse_out, false, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return succeed();
}

int kvq_rotate_rows(const void* in, int32_t in_dtype, void* out, int32_t out_dtype, int64_t n_rows,
                    int32_t head_dim, int32_t inverse, void* stream) {
  if (n_rows < 0) return fail(KVQ_ERR_INVALID_ARG, "n_rows %lld < 0", (long long)n_rows);
  if (n_rows == 0) return succeed();
  if (!in || !out) return fail(KVQ_ERR_INVALID_ARG, "NULL pointer argument");
  if (head_dim != 128 && head_dim != 256) return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d (128 or 256)", head_dim);
  for (int32_t t : {in_dtype, out_dtype})
    if (t != KVQ_OUT_F32 && t != KVQ_OUT_BF16) return fail(KVQ_ERR_INVALID_ARG, "dtype %d is not f32 / bf16", t);
  if (in == out && in_dtype != out_dtype) return fail(KVQ_ERR_INVALID_ARG, "in place needs the same dtype");
  if (!aligned16(in) || !aligned16(out)) return fail(KVQ_ERR_INVALID_ARG, "in / out must be 16-byte aligned");
  int rc = memory_kind(in, "in", nullptr);
  if (rc) return rc;
  rc = memory_kind(out, "out", nullptr);
  if (rc) return rc;
  const cudaError_t e = kvq::launch_rotate(in, in_dtype == KVQ_OUT_BF16, out, out_dtype == KVQ_OUT_BF16, n_rows,
                                           head_dim, inverse != 0, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rotate launch");
  return succeed();
}

int kvq_read_status(void* dev_status, void* stream, int32_t* bits) {
  if (!dev_status) return fail(KVQ_ERR_INVALID_ARG, "dev_status is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev_status, 0, sizeof(v), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (bits) *bits = v;
  if (v & KVQ_DEV_TIMEOUT) return fail(KVQ_ERR_DEVICE_TIMEOUT, "a device pipeline wait timed out (status 0x%x)", v);
  if (v) return fail(KVQ_ERR_DEVICE_CHECK, "device status 0x%x (bad page/seq_len/plan/slot or non-finite input)", v);
  return succeed();
}

const char* kvq_last_error(void) { return g_error.c_str(); }

}  // extern "C"
