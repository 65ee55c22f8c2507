// kvq_internal.h — declarations shared by the library's translation units
// (kernel parameter blocks and the per-format launchers).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

struct DecodeParams {
  const void* q;               // bf16 [B][Hq][D]
  const int32_t* block_tables; // [B][max_pages]
  const int32_t* seq_lens;     // [B]
  const int32_t* plan;         // [B+1] split offsets, then [total] launch order
  const uint8_t* k_scales;     // pool scale arrays (INT8 / NVFP4)
  const uint8_t* v_scales;
  float* o_part;               // [total][Hq][D]
  float* lse_part;             // [total][Hq]
  void* out;                   // [B][Hq][D] f32 or bf16
  float* lse_out;              // [B][Hq] or null
  int32_t* status;             // device status word
  int32_t batch, num_q_heads, num_kv_heads, max_pages, num_pages, total_splits;
  int32_t q_len;               // query tokens a sequence: batch = sequences x q_len virtual sequences
  int32_t heads_per_cta;       // KV heads per work item (a divisor of num_kv_heads)
  int32_t out_bf16;
  int32_t early_start;         // read plan / block tables before waiting for the preceding kernel
  int32_t out_host;            // out is pinned host memory: direct rows are written with plain stores
  int32_t drop_copies;         // failure-path test: producers issue no page copies
  uint64_t wait_limit_ns;      // limit of every pipeline wait
  float sm_scale_log2;         // sm_scale * log2(e)
  float k_gs_inv, v_gs_inv;    // NVFP4: 1 / global scale
};

struct PrefillParams {
  const void* q;               // bf16 [batch][q_len][Hq][D]
  const int32_t* block_table;  // [batch][max_pages]
  const uint8_t* k_codes;      // pool code arrays [num_pages][Hkv][16][row bytes]
  const uint8_t* v_codes;
  const uint8_t* k_scales;     // pool scale arrays (INT8)
  const uint8_t* v_scales;
  float* o_part;               // [batch * q_len * splits][Hq][D] (splits > 1)
  float* lse_part;             // [batch * q_len * splits][Hq]
  void* out;                   // [batch][q_len][Hq][D] f32 or bf16 (splits == 1)
  float* lse_out;              // [batch][q_len][Hq] or null
  int32_t* status;             // device status word
  const int32_t* seq_len_dev;  // device [batch]: the sequence lengths, read by the kernel (null: seq_len, batch 1)
  int32_t batch, q_len, seq_len, num_q_heads, num_kv_heads, num_pages, max_pages;
  int32_t splits, row_blocks, out_bf16;
  float sm_scale_log2;
  float k_gs_inv, v_gs_inv;    // NVFP4: 1 / global scales (1 otherwise)
};

struct AppendParams {
  const uint16_t* k_new;       // bf16 [N][Hkv][D]
  const uint16_t* v_new;
  const int64_t* slots;        // [N]
  uint8_t* k_codes;
  uint8_t* v_codes;
  uint8_t* k_scales;
  uint8_t* v_scales;
  int32_t* status;             // nullable
  int64_t n_tokens;
  int64_t capacity;            // num_pages * page_size
  int32_t num_kv_heads;
  int32_t check_finite;
  int32_t rotate;              // rotate each row (bf16(R(x))) before quantizing it
  float k_gs, v_gs;            // NVFP4 global scales
};

// Per-(format, head_dim) decode instance description.
struct DecodeInstance {
  const void* kernels[2];      // __global__ functions: [0] fp32 output (P' hi + lo), [1] bf16 output (hi)
  int smem_bytes;
  int threads;
  int consumer_warps;          // consumer warps per CTA
  int row_bytes;               // code bytes per token row
  int (*head_group)(int hkv);  // KV heads per work item for num_kv_heads = hkv (0: none fits)
  int launch_regs;             // registers a thread the kernel's register split assumes at launch (0: no split)
};

bool decode_instance(int format, int head_dim, DecodeInstance* out);

struct PrefillInstance {
  const void* kernels[2];      // [0] fp32 output (P' hi + lo), [1] bf16 output (hi)
  int smem_bytes;
  int threads;
  int launch_regs;             // registers a thread the kernel's register split assumes (0: no split)
  int rows;                    // query rows of a work item
};
// rotation of rows (rotate.cu)
cudaError_t launch_rotate(const void* in, bool in_bf16, void* out, bool out_bf16, int64_t n_rows, int head_dim,
                          bool inverse, cudaStream_t stream);
// copy of the query block from host memory into the workspace (programmatic dependent)
cudaError_t launch_q_stage(const void* src, void* dst, size_t bytes, cudaStream_t stream);
// the prefill kernel (tcgen05 tensor cores, accumulators in TMEM)
bool prefill_tc_instance(int format, int head_dim, PrefillInstance* out);
cudaError_t launch_prefill_tc(int format, int head_dim, const PrefillParams& p, int grid, cudaStream_t stream);
cudaError_t launch_decode(int format, int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeParams& p, int grid, cudaStream_t stream);
cudaError_t launch_append(int format, int head_dim, const AppendParams& p, cudaStream_t stream);
// Record a printf-style message as the calling thread's last error; returns code.
int record_error(int code, const char* fmt, ...);
// kvq_paged_decode_attention that, once every argument has passed its checks,
// zeroes the workspace's 256-byte status block on the stream before launching
// (the static-scratch entry point's region keeps the previous call's bits).
int decode_clearing_status(const kvq_cache* cache, const void* q, int32_t batch, int32_t num_q_heads, float sm_scale,
                           const int32_t* block_tables, int32_t max_pages_per_seq, const int32_t* seq_lens,
                           const int32_t* plan, int32_t total_splits, int32_t num_ctas, void* workspace,
                           size_t workspace_bytes, void* out, int32_t out_dtype, float* lse_out, uint32_t flags,
                           void* stream);
// offsets: split offsets [batch + 1], or null when every sequence has
// uniform_splits splits (rows b * uniform_splits ...).  offsets_ready: the
// offsets are not written by the preceding kernel on the stream (read before
// waiting for it).
cudaError_t launch_merge(const float* o_part, const float* lse_part, const int32_t* offsets, int uniform_splits,
                         int batch, int num_q_heads, int head_dim, void* out, int out_bf16, float* lse_out,
                         bool offsets_ready, cudaStream_t stream);

}  // namespace kvq
