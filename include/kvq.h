/*
 * kvq.h — C ABI of libkvq: a quantized paged KV cache for GB300 (sm_103a).
 *
 * Three operations, each one kernel launch (or two) on the caller's stream:
 *
 *   kvq_quant_append            quantize new K/V rows and scatter them into pool slots
 *   kvq_paged_decode_attention  split-KV (flash-decoding) GQA decode attention that
 *                               reads the quantized pages directly
 *   kvq_paged_verify_attention  the same for several query tokens a sequence (causal)
 *   kvq_paged_prefill_attention causal attention of a prompt chunk over the cache
 *   kvq_rotate_rows         the rotation of rows before quantization (and its inverse)
 *   kvq_paged_decode_attention_static  the decode with library-owned scratch
 *   kvq_split_merge             log-sum-exp combine of the per-split partial results
 *
 * plus host helpers (byte accounting, split planning, workspace sizing, errors).
 *
 * Sources (the pages that define the operations):
 *   [int8-kv]   "half-the-memory-int8-kv-cache" (Making a ternary reasoning model
 *               fast in vLLM), sections "An 8-bit cache was already available" and
 *               "Read the compressed cache without copying it first".
 *   [long-ctx]  "long-context-attention-and-lessons", section "Give more GPU
 *               workers a piece of the attention calculation".
 *   [nvfp4]     "Building an NVFP4 KV cache for a hybrid Qwen model", sections
 *               "How 2,048 bytes became 576" and "Writing and reading the packed cache".
 *   [capstone]  "Smaller KV cache, faster first token", sections "Lever one:
 *               4-bit KV with TurboQuant" (K and V rotated before quantization)
 *               and "Lever two: block-sparse attention with BLASST" (one KV block
 *               is loaded once for a whole GQA group).
 *
 * Conventions for every call
 *   - Pointers named "device" are CUDA device pointers on the current device;
 *     "host" pointers are ordinary host memory.  The caller owns all memory
 *     (pools, workspace, outputs) and the stream; the library allocates nothing
 *     and, unless KVQ_CHECKED is given, never synchronizes, so raw calls can be
 *     captured into a CUDA graph.
 *   - q, block_tables, seq_lens, out and lse_out of a decode call may instead be
 *     pinned host memory (page-locked and known to CUDA, e.g. cudaHostAlloc): the
 *     kernels then read and write it directly over the host link (NVLink-C2C on
 *     Grace systems), with no separate copy.  Pageable host memory is refused.
 *     Pools, plans and workspaces are device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Every call returns a kvq_status; on failure kvq_last_error() returns a
 *     message (thread-local).  No exception or abort crosses the ABI.
 *   - Errors found on the device (an out-of-range page id or slot, a bounded
 *     wait that ran out) never fault or trap: the kernel skips the access, sets a
 *     bit in a device status word and finishes.  KVQ_CHECKED reads that word
 *     before returning; raw callers read it with kvq_read_status().  The tokens of
 *     a page with an out-of-range id are left out of the softmax by every
 *     attention kernel (decode, verify on either kernel, prefill).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,    /* a null pointer, bad size or inconsistent argument */
  KVQ_ERR_UNSUPPORTED = 2,    /* a shape the kernels do not implement (see below) */
  KVQ_ERR_WORKSPACE = 3,      /* workspace or plan buffer too small */
  KVQ_ERR_CUDA = 4,           /* a CUDA runtime call failed */
  KVQ_ERR_DEVICE_CHECK = 5,   /* the device status word reports invalid metadata */
  KVQ_ERR_DEVICE_TIMEOUT = 6  /* a bounded device wait ran out */
} kvq_status;

/* ---- cache formats ([int8-kv], [nvfp4]) --------------------------------- */
enum {
  KVQ_FMT_BF16 = 0,  /* bf16 values, no scales (comparison format) */
  KVQ_FMT_INT8 = 1,  /* int8 codes + one fp32 scale per (token, KV head), scale = absmax/127 */
  KVQ_FMT_NVFP4 = 2, /* E2M1 codes, 2 per byte (element 2j low nibble), one E4M3 scale per
                        16 elements, one fp32 global scale per tensor; x = fp4*scale/global */
  KVQ_FMT_INT8_G32 = 3 /* int8 codes + one fp32 scale per 32 consecutive elements of a row,
                        scale = absmax of the 32 / 127 ([int8-kv] "Is 8 bits enough?": one
                        scale per 32 values instead of one per 256); decode and verify only */
};

/* ---- output dtypes ------------------------------------------------------ */
enum { KVQ_OUT_F32 = 0, KVQ_OUT_BF16 = 1 };

/* ---- flags --------------------------------------------------------------- */
enum {
  KVQ_CHECKED = 1u,    /* validate metadata on the host, synchronize, read the device
                          status word; not graph-capturable ([nvfp4] "Testing the cache
                          without loading the model": the checked API syncs) */
  KVQ_SKIP_MERGE = 2u, /* decode only: leave the split partials in the workspace and
                          do not launch the merge (the caller calls kvq_split_merge) */
  KVQ_EARLY_START = 4u, /* decode only: the plan and the block tables of this call are
                          not written by the kernel just before it on the stream, so the
                          decode may read them (and find its first pages) while that
                          kernel is still running.  Every other input (q, the cache,
                          seq_lens) and every output is touched only after that kernel
                          has completed.  The decode kernel is always launched as a
                          programmatic dependent of the preceding kernel; without this
                          flag it waits for that kernel before reading anything. */
  KVQ_ROTATE = 8u,     /* append only: each new K and V row x is replaced by bf16(R(x)),
                          the rotation of kvq_rotate_rows, before it is quantized
                          ([capstone] "Lever one: 4-bit KV with TurboQuant": K and V
                          are rotated before they are quantized).  The stored codes
                          and scales are bit-identical to those of kvq_rotate_rows
                          (bf16 in and out) followed by a plain kvq_quant_append; the
                          rotated rows never go through memory.  The caller still
                          rotates q (and applies R^-1 to the decode's output). */
  KVQ_TEST_STALL = 1u << 30 /* decode only, for testing the failure path: the
                          producers issue no page copies and every pipeline wait
                          gives up after 2 ms, so the call ends with KVQ_DEV_TIMEOUT
                          in the status word (KVQ_ERR_DEVICE_TIMEOUT in checked mode)
                          and the context stays usable.  The outputs are undefined. */
};

/* device status word bits (kvq_read_status) */
enum {
  KVQ_DEV_BAD_PAGE = 1,      /* block-table entry outside [0, num_pages) */
  KVQ_DEV_BAD_SEQLEN = 2,    /* seq_len < 0 or > max_pages_per_seq * page_size */
  KVQ_DEV_BAD_PLAN = 4,      /* plan entry outside the batch / split range */
  KVQ_DEV_TIMEOUT = 8,       /* a pipeline wait gave up */
  KVQ_DEV_BAD_SLOT = 16,     /* append: slot >= num_pages * page_size */
  KVQ_DEV_NONFINITE = 32     /* append (checked): a non-finite input value */
};

/*
 * The paged pool ([capstone] "Why KV capacity drives TTFT under load": the cache
 * is managed in fixed-size blocks, like virtual-memory pages).
 *
 * Layout (all arrays dense, row-major, device memory, base 256-byte aligned):
 *   k_codes, v_codes   [num_pages][num_kv_heads][page_size][row_bytes]
 *                      row_bytes = 2*head_dim (BF16), head_dim (INT8, INT8_G32), head_dim/2 (NVFP4)
 *   k_scales, v_scales INT8:  [num_pages][num_kv_heads][page_size] float
 *                      INT8_G32: [num_pages][num_kv_heads][head_dim/32][page_size] float
 *                             (group-major inside each (page, KV head) block: the scale of
 *                             elements 32g .. 32g+31 of slot row i is at [.][.][g][i])
 *                      NVFP4: [num_pages][num_kv_heads][page_size][head_dim/16] E4M3 bytes
 *                      BF16:  unused (NULL)
 * Slot s is row (s % page_size) of page (s / page_size).  Each (page, KV head)
 * block is contiguous, so one page of one head streams as one 16-byte-aligned
 * block; the scales live in their own arrays so that code rows stay aligned
 * (the pages' vLLM layout put a 4-byte scale after each 256-byte row, which
 * blocked wide loads: [int8-kv] "Read the compressed cache without copying it first").
 *
 * Supported: page_size 16; head_dim 128 or 256 (every format); any num_kv_heads >= 1.
 * NVFP4 global scales must be finite and > 0 and must stay fixed while entries
 * are live ([nvfp4] "How 2,048 bytes became 576").
 */
typedef struct kvq_cache {
  void* k_codes;
  void* v_codes;
  void* k_scales;
  void* v_scales;
  int32_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t format;         /* KVQ_FMT_* */
  float k_global_scale;   /* NVFP4 only */
  float v_global_scale;   /* NVFP4 only */
} kvq_cache;

/* ---- host helpers: byte accounting ([int8-kv], [nvfp4]) ----------------- */

/* K+V bytes one token occupies in one layer (codes + scales, all KV heads):
 * BF16 4*D*Hkv, INT8 2*(D+4)*Hkv (520 per head at D=256), INT8_G32 2*(D+D/8)*Hkv
 * (576 per head at D=256), NVFP4 2*(D/2+D/16)*Hkv
 * (576 per token per layer at 2 heads, D=256).  Returns -1 for an unknown format
 * or a non-positive size.  Host only; no GPU needed. */
int64_t kvq_bytes_per_token(int32_t format, int32_t num_kv_heads, int32_t head_dim);

/* Sizes in bytes of one codes array and one scales array of a pool (each of K and
 * V has one of each).  Host only.  Returns KVQ_OK or KVQ_ERR_INVALID_ARG. */
int kvq_cache_array_bytes(int32_t format, int32_t num_pages, int32_t page_size,
                          int32_t num_kv_heads, int32_t head_dim,
                          int64_t* codes_bytes, int64_t* scales_bytes);

/* ---- kv_quant_append ([int8-kv] "An 8-bit cache was already available";
 *      [nvfp4] "Writing and reading the packed cache") ---------------------- */
/*
 * Quantize n_tokens new rows of K and V and write them into the pool.
 *   k_new, v_new   device, bf16 [n_tokens][num_kv_heads][head_dim]
 *   slot_mapping   device, int64 [n_tokens]; token i goes to slot slot_mapping[i];
 *                  a negative slot means "do not write" (padding).  Valid slots must
 *                  be unique within a call; KVQ_CHECKED rejects duplicates.
 *   dev_status     device int32 word (nullable).  Slots >= num_pages*page_size are
 *                  skipped and set KVQ_DEV_BAD_SLOT there; with KVQ_CHECKED a
 *                  non-finite input sets KVQ_DEV_NONFINITE.  KVQ_CHECKED needs it.
 * INT8: per (token, head) s = fp32(absmax/127), code = clamp(rne(fp32(x/s)),-127,127),
 *       s == 0 gives zero codes.
 * NVFP4: per group of 16: t = fp32(amax/6), scale byte = E4M3_rne_satfinite(fp32(t*gs)),
 *       code = E2M1_rne_satfinite(fp32(fp32(x*gs)/scale)) with the sign of x, zero
 *       codes when the scale is 0; element 2j in the low nibble.
 * BF16: the rows are copied.
 * flags: KVQ_CHECKED; KVQ_ROTATE (rotate each row before quantizing it, see above).
 * Overwriting a slot that holds older data is allowed.
 */
int kvq_quant_append(const kvq_cache* cache, const void* k_new, const void* v_new,
                     const int64_t* slot_mapping, int64_t n_tokens,
                     int32_t* dev_status, uint32_t flags, void* stream);

/* ---- split planning ([long-ctx]: split-KV; the split count trades merge
 *      overhead against parallelism) ----------------------------------------- */
/*
 * Choose, on the host, how many splits each sequence gets and how the work is
 * spread over persistent CTAs, and write the plan.  A work item is one split of
 * one sequence for a group of HG KV heads, HG = gcd(Hkv, consumer warps of the
 * kernel: 8 at D = 256, 12 at D = 128) (or a divisor of it when the shared-memory
 * ring needs smaller groups); NHG = Hkv / HG groups, total * NHG items.  Layout
 * (int32 entries; A = batch + 2 rounded up to a multiple of 4, R = A + 5C + 1
 * rounded up to a multiple of 4):
 *   plan[0..batch]          split_offsets: sequence b owns splits (and partial
 *                           slots) [plan[b], plan[b+1]); plan[0] = 0, plan[batch] = total
 *   plan[batch+1]           C = *num_ctas, the number of persistent CTAs
 *   plan[A .. A+4C)         the first item of each CTA, one 4-entry descriptor each
 *   plan[A+4C .. A+5C]      CTA c's further items are rest entries [o[c], o[c+1]),
 *                           o[0] = 0, o[C] = total * NHG - C
 *   plan[R ..]              the rest entries, one 4-entry descriptor each
 * A descriptor is {b, split, first page, n | direct << 23 | group << 24}: sequence
 * b's split `split` (a global split index) covers its pages [first page, first
 * page + n) for KV heads [group * HG, (group + 1) * HG); direct = the sequence has
 * a single split (the kernel writes `out` directly).  Split s of a sequence with
 * n pages and S splits covers pages [floor(s*n/S), floor((s+1)*n/S)) — whole
 * pages, sizes differing by at most one.  Items are packed onto the C CTAs longest
 * first, each onto the CTA with the least work so far, so an uneven batch runs in
 * one wave; a CTA's first item sits at a fixed place so that it can start loading
 * pages without first reading an offset.
 *   seq_lens        host int32 [batch], each >= 0
 *   split_override  > 0: S_b = clamp(split_override, 1, max(n_pages_b, 1));
 *                   0: automatic.  Candidate split sizes x (pages a split, at
 *                   least 4; S_b = ceil(n_pages_b / x)): x = NHG * total_pages /
 *                   (C * m) for m in {1, 1.25, 1.5, 2, 2.5, 3, 4, 6}, and for k =
 *                   1..4 the smallest x whose items fit in k * C (whole waves).
 *                   Each candidate's items are packed as below and its critical
 *                   path (the largest CTA load, a page costing 1 and an item 8
 *                   more) is computed; the shortest wins (ties: fewer items;
 *                   a whole-wave candidate only when strictly shorter).
 *   target_ctas     CTAs to plan for; 0 = measured on the current device (SM count
 *                   x resident decode CTAs per SM for this format/head_dim);
 *                   C = min(target_ctas, total * NHG)
 *   plan            host int32 buffer of plan_capacity entries (nullable for a size query)
 *   total_splits, num_ctas  out (always written when the inputs are valid)
 * Returns KVQ_ERR_WORKSPACE if plan is NULL or shorter than R + 4 * (total * NHG - C)
 * (at most batch + 9 + C + 4 * total * num_kv_heads).  The plan must be copied to
 * the device before kvq_paged_decode_attention, and plan, total_splits and
 * num_ctas passed there must come from the same call.
 */
int kvq_plan_splits(const kvq_cache* cache, const int32_t* seq_lens, int32_t batch,
                    int32_t split_override, int32_t target_ctas,
                    int32_t* plan, int64_t plan_capacity,
                    int32_t* total_splits, int32_t* num_ctas);

/* kvq_plan_splits for a verify call (kvq_paged_verify_attention) of q_len query
 * tokens a sequence: the plan covers the batch * q_len virtual sequences, in
 * order b * q_len + i, whose visible lengths max(0, seq_lens[b] - q_len + 1 + i)
 * this call computes (causal: query token i sits at position seq_lens[b] -
 * q_len + i).  seq_lens: host int32 [batch], the q_len new tokens included.
 * Every other argument, the plan layout and the return codes are those of
 * kvq_plan_splits (with batch * q_len in place of batch); KVQ_ERR_INVALID_ARG
 * for q_len < 1. */
int kvq_plan_verify_splits(const kvq_cache* cache, const int32_t* seq_lens, int32_t batch, int32_t q_len,
                           int32_t split_override, int32_t target_ctas, int32_t* plan, int64_t plan_capacity,
                           int32_t* total_splits, int32_t* num_ctas);

/* Workspace bytes for a decode call: a 256-byte status block, then
 * lse_part float[total_splits][num_q_heads] (padded to 256 bytes), then
 * o_part float[total_splits][num_q_heads][head_dim] (256-byte aligned), then room
 * for a bf16 copy of q (a query block in pinned host memory is copied there once
 * per call, so that the decode reads it from device memory).  The status block must be
 * zero before the first call (e.g. cudaMemset once); the library only ORs bits
 * into it and kvq_read_status clears it. */
size_t kvq_decode_workspace_bytes(int32_t total_splits, int32_t num_q_heads, int32_t head_dim);

/* Workspace bytes for kvq_paged_verify_attention: the larger of
 * kvq_decode_workspace_bytes(total_splits, num_q_heads, head_dim) and, for a
 * call the prefill kernel may take (q_len >= 4 for one sequence, >= 6 for a
 * batch; NVFP4 3 and 4),
 * kvq_prefill_workspace_bytes(q_len, num_q_heads, head_dim, S) for the largest
 * key split count S it may use (at most 64; see kvq_prefill_splits).
 * target_ctas: the SM count of the device the calls run on (0: the current
 * device's).  A smaller workspace keeps such a call on the decode kernel.
 * 0 for bad arguments (the reason in kvq_last_error). */
size_t kvq_verify_workspace_bytes(const kvq_cache* cache, int32_t batch, int32_t q_len, int32_t num_q_heads,
                                  int32_t total_splits, int32_t target_ctas);

/* Device pointers to the partials inside a workspace (host pointer arithmetic). */
int kvq_workspace_partials(void* workspace, int32_t total_splits, int32_t num_q_heads,
                           int32_t head_dim, float** o_part, float** lse_part);

/* ---- paged_decode_attention ([long-ctx] split-KV; [int8-kv] "Read the
 *      compressed cache without copying it first": dequantize in registers) --- */
/*
 * out[b][g] = softmax(sm_scale * q[b][g] . K_b^T) . V_b for every sequence b and
 * query head g, with K_b/V_b the dequantized cache rows of KV head g / (Hq/Hkv)
 * (consecutive query heads share a KV head), tokens 0..seq_lens[b]-1 in the order
 * of the block table.  Each of the num_ctas persistent CTAs works through its
 * list of (split, KV-head group) items and loads each page once for the whole
 * query-head group.
 *   q              device bf16 [batch][num_q_heads][head_dim]
 *   sm_scale       softmax scale, normally 1/sqrt(head_dim)
 *   block_tables   device int32 [batch][max_pages_per_seq]; page j of sequence b
 *   seq_lens       device int32 [batch]
 *   plan           device int32, the kvq_plan_splits output for these seq_lens;
 *                  total_splits and num_ctas are its two outputs
 *   workspace      device, >= kvq_decode_workspace_bytes(total_splits, Hq, D)
 *   out            device, [batch][num_q_heads][head_dim] float or bf16 (out_dtype)
 *   lse_out        device float [batch][num_q_heads] (nullable): natural-log
 *                  log-sum-exp of the scaled logits (-inf for an empty context)
 * An empty context gives out = 0.  Tokens past seq_len in the last page are never
 * read into the softmax, whatever their slots hold.  Sequences with a single
 * split are written directly; the others are combined by the merge kernel on the
 * same stream (unless KVQ_SKIP_MERGE).
 * Supported: num_q_heads % num_kv_heads == 0 and 1 <= num_q_heads/num_kv_heads <= 8.
 */
int kvq_paged_decode_attention(const kvq_cache* cache, const void* q, int32_t batch,
                               int32_t num_q_heads, float sm_scale,
                               const int32_t* block_tables, int32_t max_pages_per_seq,
                               const int32_t* seq_lens, const int32_t* plan,
                               int32_t total_splits, int32_t num_ctas,
                               void* workspace, size_t workspace_bytes,
                               void* out, int32_t out_dtype, float* lse_out,
                               uint32_t flags, void* stream);

/* ---- paged_verify_attention ([int8-kv] "Read the compressed cache without
 *      copying it first": one program both generates a token and checks several
 *      proposed ones; a verify step reads the whole context with 6 query tokens,
 *      36 query rows for 6 heads, and an MMA kernel of 8-row granularity avoids
 *      padding them) --------------------------------------------------------- */
/*
 * Causal attention for q_len query tokens a sequence whose K/V are already the
 * last q_len entries of its cache (seq_lens[b] tokens in all, appended by
 * kvq_quant_append): query token i of sequence b sits at position
 * seq_lens[b] - q_len + i and attends over tokens 0 .. seq_lens[b] - q_len + i
 * (none when that is negative: out = 0, lse = -inf).  The same kernels as
 * kvq_paged_decode_attention, run over batch * q_len virtual sequences — token i
 * of sequence b is virtual sequence b * q_len + i, with b's block table — so every
 * MMA tile holds the G query heads of one token (8-row granularity), and the
 * q_len tokens' items cover the same pages at about the same time, so a page
 * read for one token is mostly still in L2 for the others.
 * A call with enough query tokens a sequence goes instead, as one launch for
 * the batch, to the tensor-core kernel of kvq_paged_prefill_attention ([int8-kv]
 * "Read the prompt using a small temporary buffer": a block of query rows reads
 * each key once): for one sequence q_len >= 4 when its block table spans
 * 2,048 pages or more, >= 5 from 1,024, >= 6 from 512, >= 10 below (NVFP4: 3,
 * 3, 4, 8); for a batch q_len >= 6 (NVFP4: 4).  The kernel reads the sequence lengths on the device
 * and takes the key splits that kvq_prefill_splits picks with the block table's
 * width as the context.  This happens when q and out are device memory, neither
 * KVQ_SKIP_MERGE nor KVQ_TEST_STALL is set and the workspace holds
 * kvq_verify_workspace_bytes; the plan is still required (and checked under
 * KVQ_CHECKED), and the result is the same up to rounding order.  With q_len
 * the length of a prompt chunk, the call is a chunked prefill of the same number
 * of tokens for every sequence of a batch (kvq_paged_prefill_attention takes
 * one sequence).
 *   q              device bf16 [batch][q_len][num_q_heads][head_dim]
 *   seq_lens       device int32 [batch]: tokens in the cache, the q_len new ones included
 *   plan           kvq_plan_verify_splits(seq_lens, batch, q_len, ...): the plan
 *                  over the batch * q_len virtual lengths max(0, seq_lens[b] -
 *                  q_len + 1 + i), in order b * q_len + i
 *   workspace      >= kvq_decode_workspace_bytes(total_splits, num_q_heads, head_dim);
 *                  kvq_verify_workspace_bytes(...) also covers the routed call
 *   out            device [batch][q_len][num_q_heads][head_dim] float or bf16
 *   lse_out        device float [batch][q_len][num_q_heads] (nullable)
 * Everything else (flags included) as for kvq_paged_decode_attention; q_len = 1
 * is exactly kvq_paged_decode_attention.
 */
int kvq_paged_verify_attention(const kvq_cache* cache, const void* q, int32_t batch, int32_t q_len,
                               int32_t num_q_heads, float sm_scale,
                               const int32_t* block_tables, int32_t max_pages_per_seq,
                               const int32_t* seq_lens, const int32_t* plan,
                               int32_t total_splits, int32_t num_ctas,
                               void* workspace, size_t workspace_bytes,
                               void* out, int32_t out_dtype, float* lse_out,
                               uint32_t flags, void* stream);

/* ---- paged_prefill_attention ([int8-kv] "Read the prompt using a small temporary
 *      buffer": a chunk of prompt tokens reuses every key it reads many times, the
 *      cached history is read in sections whose partial results are combined with
 *      their attention weights, and each token sees only the tokens before it and
 *      itself) ---------------------------------------------------------------- */
/*
 * Causal attention of a prompt chunk: q holds the last q_len of one sequence's
 * seq_len tokens (their K/V already appended); chunk token i sits at position
 * seq_len - q_len + i and attends over tokens 0 .. seq_len - q_len + i of the
 * cache.  Each 64-key tile of the cache is converted once per work item into an
 * fp16 (BF16 cache: bf16) copy in shared memory (INT8: the exact integer codes;
 * NVFP4: E2M1 x E4M3 group scale, exact in fp16) and multiplied on the tensor
 * cores (tcgen05.mma, fp32 accumulators in tensor memory).  A work item is 128
 * query rows (token, query head) of one KV head against one of `splits` key
 * ranges; with splits > 1 the partials are combined by the merge kernel on the
 * same stream.  INT8, NVFP4 and BF16 caches at head_dim 128 or 256;
 * 1 <= num_q_heads / num_kv_heads <= 8.  INT8_G32 caches are refused with
 * KVQ_ERR_UNSUPPORTED (a per-32 scale cannot be folded into the logits or P,
 * and the scaled values are not exact in fp16).
 *   q              device bf16 [q_len][num_q_heads][head_dim]
 *   block_table    device int32 [max_pages]: the sequence's pages
 *   seq_len        host: tokens of the sequence, the q_len new ones included
 *   splits         1 .. 64 key ranges.  kvq_prefill_splits gives a default: the S
 *                  that minimises a model of the call fitted to measured calls,
 *                  waves(S) x (10 us + 1.9 us a 64-key tile of a split) plus, for
 *                  S > 1, the merge (3.5 us + the partials written and read at
 *                  6 TB/s), waves(S) = ceil(CTAs / target_ctas), at least one
 *                  tile a split
 *   workspace      device, >= kvq_prefill_workspace_bytes(q_len, num_q_heads, head_dim, splits),
 *                  256-byte aligned; its first word is the device status word
 *   out            device [q_len][num_q_heads][head_dim] float or bf16
 *   lse_out        device float [q_len][num_q_heads] (nullable)
 *   flags          KVQ_CHECKED: synchronize and read the status word
 */
int32_t kvq_prefill_splits(const kvq_cache* cache, int32_t q_len, int32_t num_q_heads, int32_t seq_len,
                           int32_t target_ctas);  /* >= 1, or minus a kvq_status */
size_t kvq_prefill_workspace_bytes(int32_t q_len, int32_t num_q_heads, int32_t head_dim, int32_t splits);
int kvq_paged_prefill_attention(const kvq_cache* cache, const void* q, int32_t q_len, int32_t num_q_heads,
                                float sm_scale, const int32_t* block_table, int32_t max_pages, int32_t seq_len,
                                int32_t splits, void* workspace, size_t workspace_bytes, void* out,
                                int32_t out_dtype, float* lse_out, uint32_t flags, void* stream);

/* ---- paged_decode_attention_static (no counterpart in the pages: an
 *      allocation-free variant of kvq_paged_decode_attention) ----------------- */
/* Bytes of the library's static decode scratch region on each device. */
#define KVQ_STATIC_SCRATCH_BYTES (16u << 20)
/*
 * The same computation, arguments and results as kvq_paged_decode_attention,
 * without the workspace: the status block and the partials live in a fixed
 * KVQ_STATIC_SCRATCH_BYTES region of device memory owned by the library, so the
 * call allocates nothing (for callers with no device allocator, or with device
 * memory committed in full to the page pool).
 *   - Returns KVQ_ERR_WORKSPACE, touching nothing, when
 *     kvq_decode_workspace_bytes(total_splits, num_q_heads, head_dim) exceeds
 *     KVQ_STATIC_SCRATCH_BYTES.
 *   - The first call on a device looks up the region's address there (with that
 *     device current); make that first call before any stream capture.
 *   - Each call clears the region's status block on `stream`, then runs the
 *     decode (and merge) there; with KVQ_CHECKED the status is read and cleared
 *     as in kvq_paged_decode_attention.
 *   - All calls on a device share the region, which keeps the last call's
 *     contents: calls whose kernels overlap on the GPU (other streams, other
 *     threads) race on it and give undefined results.  Serialize them.
 */
int kvq_paged_decode_attention_static(const kvq_cache* cache, const void* q, int32_t batch,
                                      int32_t num_q_heads, float sm_scale,
                                      const int32_t* block_tables, int32_t max_pages_per_seq,
                                      const int32_t* seq_lens, const int32_t* plan,
                                      int32_t total_splits, int32_t num_ctas,
                                      void* out, int32_t out_dtype, float* lse_out,
                                      uint32_t flags, void* stream);

/* ---- split_merge ([long-ctx]: merge with the normalisation terms; averaging
 *      the partial outputs would be wrong) ------------------------------------ */
/*
 * For every sequence with S_b = split_offsets[b+1]-split_offsets[b] >= 2 and query
 * head g: M = max_s lse[s], w_s = exp(lse[s] - M), out = sum_s w_s o[s] / sum_s w_s,
 * lse_out = M + log(sum_s w_s); empty splits (lse = -inf) have weight 0.  Rows are
 * o_part[(split_offsets[b]+s)*num_q_heads + g][head_dim], lse_part likewise.
 * Sequences with S_b = 1 are skipped (the decode kernel wrote them directly).
 *   o_part, lse_part, split_offsets  device; out, lse_out (nullable) device.
 */
int kvq_split_merge(const float* o_part, const float* lse_part, const int32_t* split_offsets,
                    int32_t batch, int32_t num_q_heads, int32_t head_dim,
                    void* out, int32_t out_dtype, float* lse_out, void* stream);

/* ---- rotate_rows ([capstone] "Lever one: 4-bit KV with TurboQuant": the K and V
 *      vectors are rotated before they are quantized, so that outliers spread
 *      over all dimensions) -------------------------------------------------- */
/*
 * out[r] = R(in[r]) (inverse != 0: R^-1) for n_rows rows of head_dim values, with
 * R(x) = head_dim^(-1/2) H (s * x): H the Sylvester Hadamard matrix, s_i = -1 iff
 * bit 31 of (i + 1) * 2654435761 mod 2^32 is set.  R is orthogonal: rotating q and
 * the cached K leaves the attention scores unchanged, and attention over rotated
 * V returns R(o), so a caller rotates new K/V rows before kvq_quant_append, rotates
 * q before the decode and applies the inverse to its output.  Arithmetic (it
 * fixes the bits): fp32 butterflies, stages h = 1, 2, ..., head_dim/2, pairs
 * (a, b) -> (a + b, a - b); one multiply by fp32(head_dim^-1/2); rounding to
 * the output type (bf16: nearest even).
 *   in, out    device or pinned host [n_rows][head_dim], KVQ_OUT_F32 (fp32) or
 *              KVQ_OUT_BF16 (bf16) each (in_dtype / out_dtype); out may equal in
 *              when the types match
 *   head_dim   128 or 256
 */
int kvq_rotate_rows(const void* in, int32_t in_dtype, void* out, int32_t out_dtype, int64_t n_rows,
                    int32_t head_dim, int32_t inverse, void* stream);

/* Synchronize `stream`, read and clear a device status word (the first int32 of a
 * decode workspace, or an append dev_status).  *bits receives the KVQ_DEV_* bits.
 * Returns KVQ_OK, KVQ_ERR_DEVICE_CHECK or KVQ_ERR_DEVICE_TIMEOUT. */
int kvq_read_status(void* dev_status, void* stream, int32_t* bits);

/* Last error message of the calling thread ("" if none). */
const char* kvq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
