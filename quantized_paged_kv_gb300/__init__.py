"""Quantized paged KV cache for GB300 (sm_103a): INT8 / NVFP4 / BF16 pools,
quantize-and-append, split-KV GQA decode attention and the log-sum-exp merge,
verification and chunked prefill over the cache, and the rotation of rows
before quantization.

The compute lives in libkvq.so (hand-written CUDA, C ABI in include/kvq.h);
this package is its ctypes binding (``_binding``, same names as the C entry
points), device-pool helpers (``cache``) and seeded input generators
(``workloads``).  Importing the package does not load the library; the first
call does, and raises if it has not been built.
"""
from . import _binding
from ._binding import (  # noqa: F401
    FORMATS, KVQ_CHECKED, KVQ_EARLY_START, KVQ_ROTATE, KVQ_SKIP_MERGE, KvqError, kvq_bytes_per_token, kvq_cache_array_bytes,
    kvq_decode_workspace_bytes, kvq_last_error, kvq_paged_decode_attention, kvq_plan_splits, kvq_plan_verify_splits,
    kvq_quant_append,
    kvq_paged_decode_attention_static, kvq_paged_prefill_attention, kvq_paged_verify_attention,
    kvq_prefill_splits, kvq_prefill_workspace_bytes, kvq_read_status, kvq_rotate_rows, kvq_split_merge,
    kvq_verify_workspace_bytes, kvq_workspace_partials, lib,
)
from .cache import DecodePlan, KVCache, decode, prefill, verify  # noqa: F401
