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
// taken once, with that device current, by the first call made there
// (cudaGetSymbolAddress); that first call should therefore come before any
// stream capture.  Every call on a device shares the region and finds the last
// call's contents in it: the call clears the status block (the only part that
// must start at zero; every partial row the merge reads is written by the
// decode first), and calls whose kernels overlap on the GPU race on it.
#include <mutex>

#include "kvq_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Address of the region on the current device (set up on first use there).
int scratch_on_current_device(void** ptr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvq::record_error(KVQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return kvq::record_error(KVQ_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p)
      return kvq::record_error(KVQ_ERR_CUDA, "cudaGetSymbolAddress(static decode scratch): %s",
                               cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
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
  int rc = scratch_on_current_device(&scratch);
  if (rc) return rc;
  cudaError_t e = cudaMemsetAsync(scratch, 0, 256, reinterpret_cast<cudaStream_t>(stream));  // status block
  if (e != cudaSuccess) return kvq::record_error(KVQ_ERR_CUDA, "clearing the status block: %s", cudaGetErrorString(e));
  return kvq_paged_decode_attention(cache, q, batch, num_q_heads, sm_scale, block_tables, max_pages_per_seq, seq_lens,
                                    plan, total_splits, num_ctas, scratch, (size_t)KVQ_STATIC_SCRATCH_BYTES, out,
                                    out_dtype, lse_out, flags, stream);
}
