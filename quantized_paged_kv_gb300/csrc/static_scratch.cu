// static_scratch.cu — kvq_paged_decode_attention_static: the decode entry point
// with its scratch (status block, lse_part, o_part) in a fixed region of device
// memory that the library owns, so that the call allocates nothing.
//
// Who needs it: callers that hold no device allocator of their own — a plain C
// host loop that was handed only the cache and the query/output buffers — and
// callers whose device memory is committed in full to the page pool, where a
// per-call (or per-plan) workspace would have to come out of the pages.  Both
// can still size a plan on the host; neither can find room for a workspace.
//
// The region is one file-scope __device__ array.  Its address on a device is
// taken with that device current, by the first call made there
// (cudaGetSymbolAddress), and kept together with the ID of the CUDA context it
// was taken in; a later call in another context (after cudaDeviceReset, or once
// the primary context has been released and created again, which loads the
// module anew) looks the address up again.  The first call on a device should
// therefore come before any stream capture.  Every call on a device shares the
// region and finds the last call's contents in it: once its arguments have
// passed their checks, the call clears the status block (the only part that
// must start at zero; every partial row the merge reads is written by the
// decode first), and calls whose kernels overlap on the GPU race on it.
#include <cudaTypedefs.h>

#include <mutex>

#include "kvq_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
  unsigned long long ctx_id;  // CUDA context the address belongs to (0: none yet)
  void* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// ID of the calling thread's current CUDA context, 0 if there is none or the
// driver does not say (the address is then looked up again).
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Address of the region on the current device, in the current context.
int scratch_on_current_device(void** ptr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvq::record_error(KVQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return kvq::record_error(KVQ_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_context_id();
  if (id == 0 || g_scratch[dev].ctx_id != id || !g_scratch[dev].ptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);  // makes the device's primary context current if needed
    if (e != cudaSuccess || !p)
      return kvq::record_error(KVQ_ERR_CUDA, "cudaGetSymbolAddress(static decode scratch): %s",
                               cudaGetErrorString(e));
    g_scratch[dev].ptr = p;
    g_scratch[dev].ctx_id = current_context_id();
  }
  *ptr = g_scratch[dev].ptr;
  return KVQ_OK;
}

}  // namespace

extern "C" int kvq_paged_decode_attention_static(const kvq_cache* cache, const void* q, int32_t batch,
                                                 int32_t num_q_heads, float sm_scale,
                                                 const int32_t* block_tables, int32_t max_pages_per_seq,
                                                 const int32_t* seq_lens, const int32_t* plan,
                                                 int32_t total_splits, int32_t num_ctas, void* out,
                                                 int32_t out_dtype, float* lse_out, uint32_t flags,
                                                 void* stream) {
  if (!cache) return kvq::record_error(KVQ_ERR_INVALID_ARG, "cache is NULL");
  if (total_splits < 0 || num_q_heads < 0)
    return kvq::record_error(KVQ_ERR_INVALID_ARG, "negative total_splits / num_q_heads");
  const size_t need = kvq_decode_workspace_bytes(total_splits, num_q_heads, cache->head_dim);
  if (need > (size_t)KVQ_STATIC_SCRATCH_BYTES)
    return kvq::record_error(KVQ_ERR_WORKSPACE,
                             "decode needs %zu bytes of scratch (total_splits %d x num_q_heads %d x head_dim %d); "
                             "the static region holds %zu: use kvq_paged_decode_attention with a workspace",
                             need, total_splits, num_q_heads, cache->head_dim, (size_t)KVQ_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc) return rc;
  // the status block is cleared on `stream` only once the arguments have passed
  // the decode's checks, so a rejected call leaves an earlier call's bits in place
  return kvq::decode_clearing_status(cache, q, batch, num_q_heads, sm_scale, block_tables, max_pages_per_seq,
                                     seq_lens, plan, total_splits, num_ctas, scratch,
                                     (size_t)KVQ_STATIC_SCRATCH_BYTES, out, out_dtype, lse_out, flags, stream);
}
