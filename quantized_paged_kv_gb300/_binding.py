"""ctypes binding of libkvq.so — argument marshalling only.

Every function here has the name of the C entry point it calls (include/kvq.h)
and does nothing but turn torch tensors into device pointers, torch streams into
cudaStream_t handles, and non-zero status codes into exceptions.  All of the work
runs in the library's sm_103a kernels; there is no fallback: if libkvq.so is
missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_int64, c_size_t, c_uint32, c_void_p

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libkvq.so")

KVQ_FMT_BF16, KVQ_FMT_INT8, KVQ_FMT_NVFP4, KVQ_FMT_INT8_G32 = 0, 1, 2, 3
KVQ_OUT_F32, KVQ_OUT_BF16 = 0, 1
KVQ_CHECKED, KVQ_SKIP_MERGE, KVQ_EARLY_START = 1, 2, 4
KVQ_ROTATE = 8  # append: rotate each new K/V row (bf16(R(x))) before quantizing it
KVQ_TEST_STALL = 1 << 30  # failure-path test: no page copies, every device wait gives up after 2 ms
KVQ_DEV_BAD_PAGE, KVQ_DEV_BAD_SEQLEN, KVQ_DEV_BAD_PLAN = 1, 2, 4
KVQ_DEV_TIMEOUT, KVQ_DEV_BAD_SLOT, KVQ_DEV_NONFINITE = 8, 16, 32
KVQ_STATIC_SCRATCH_BYTES = 16 << 20
FORMATS = {"bf16": KVQ_FMT_BF16, "int8": KVQ_FMT_INT8, "nvfp4": KVQ_FMT_NVFP4, "int8_g32": KVQ_FMT_INT8_G32}

# every symbol include/kvq.h declares
EXPORTS = (
    "kvq_bytes_per_token", "kvq_cache_array_bytes", "kvq_quant_append", "kvq_plan_splits", "kvq_plan_verify_splits",
    "kvq_decode_workspace_bytes", "kvq_verify_workspace_bytes", "kvq_workspace_partials", "kvq_paged_decode_attention",
    "kvq_paged_decode_attention_static", "kvq_paged_verify_attention", "kvq_prefill_splits",
    "kvq_prefill_workspace_bytes", "kvq_paged_prefill_attention", "kvq_split_merge", "kvq_read_status",
    "kvq_last_error", "kvq_rotate_rows",
)


class KvqCacheStruct(ctypes.Structure):
    _fields_ = [
        ("k_codes", c_void_p), ("v_codes", c_void_p), ("k_scales", c_void_p), ("v_scales", c_void_p),
        ("num_pages", c_int32), ("page_size", c_int32), ("num_kv_heads", c_int32), ("head_dim", c_int32),
        ("format", c_int32), ("k_global_scale", c_float), ("v_global_scale", c_float),
    ]


class KvqError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"[kvq status {code}] {msg}")
        self.code = code


_lib = None


def lib():
    """Load libkvq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "or python -m quantized_paged_kv_gb300.build")
    L = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    sig = {
        "kvq_bytes_per_token": (c_int64, [c_int32, c_int32, c_int32]),
        "kvq_cache_array_bytes": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32, POINTER(c_int64), POINTER(c_int64)]),
        "kvq_quant_append": (c_int32, [POINTER(KvqCacheStruct), P, P, P, c_int64, P, c_uint32, P]),
        "kvq_plan_splits": (c_int32, [POINTER(KvqCacheStruct), POINTER(c_int32), c_int32, c_int32, c_int32,
                                      POINTER(c_int32), c_int64, POINTER(c_int32), POINTER(c_int32)]),
        "kvq_plan_verify_splits": (c_int32, [POINTER(KvqCacheStruct), POINTER(c_int32), c_int32, c_int32, c_int32,
                                             c_int32, POINTER(c_int32), c_int64, POINTER(c_int32), POINTER(c_int32)]),
        "kvq_decode_workspace_bytes": (c_size_t, [c_int32, c_int32, c_int32]),
        "kvq_verify_workspace_bytes": (c_size_t, [POINTER(KvqCacheStruct), c_int32, c_int32, c_int32, c_int32,
                                                  c_int32]),
        "kvq_workspace_partials": (c_int32, [P, c_int32, c_int32, c_int32, POINTER(c_void_p), POINTER(c_void_p)]),
        "kvq_paged_decode_attention": (c_int32, [POINTER(KvqCacheStruct), P, c_int32, c_int32, c_float, P, c_int32,
                                                 P, P, c_int32, c_int32, P, c_size_t, P, c_int32, P, c_uint32, P]),
        "kvq_paged_decode_attention_static": (c_int32, [POINTER(KvqCacheStruct), P, c_int32, c_int32, c_float, P,
                                                        c_int32, P, P, c_int32, c_int32, P, c_int32, P, c_uint32, P]),
        "kvq_paged_verify_attention": (c_int32, [POINTER(KvqCacheStruct), P, c_int32, c_int32, c_int32, c_float, P,
                                                 c_int32, P, P, c_int32, c_int32, P, c_size_t, P, c_int32, P,
                                                 c_uint32, P]),
        "kvq_prefill_splits": (c_int32, [POINTER(KvqCacheStruct), c_int32, c_int32, c_int32, c_int32]),
        "kvq_prefill_workspace_bytes": (c_size_t, [c_int32, c_int32, c_int32, c_int32]),
        "kvq_paged_prefill_attention": (c_int32, [POINTER(KvqCacheStruct), P, c_int32, c_int32, c_float, P, c_int32,
                                                  c_int32, c_int32, P, c_size_t, P, c_int32, P, c_uint32, P]),
        "kvq_split_merge": (c_int32, [P, P, P, c_int32, c_int32, c_int32, P, c_int32, P, P]),
        "kvq_read_status": (c_int32, [P, P, POINTER(c_int32)]),
        "kvq_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    _lib = L
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc, name):
    if rc != 0:
        raise KvqError(rc, f"{name}: {lib().kvq_last_error().decode()}")


def _shapes(q, out, lse_out, block_tables, seq_lens, cache_struct):
    """The buffers a device call writes or indexes, against q's shape (q is [B, ..., Hq, D]):
    out holds q's element count, lse_out one value a query row, block_tables and
    seq_lens a row per sequence."""
    if out.numel() != q.numel():
        raise ValueError(f"out must hold {q.numel()} values (q's shape {tuple(q.shape)}), got {tuple(out.shape)}")
    if lse_out is not None and lse_out.numel() != q.numel() // q.shape[-1]:
        raise ValueError(f"lse_out must hold {q.numel() // q.shape[-1]} values, got {tuple(lse_out.shape)}")
    if q.shape[-1] != cache_struct.head_dim:
        raise ValueError(f"q's head_dim {q.shape[-1]} != the cache's {cache_struct.head_dim}")
    if block_tables is not None and (block_tables.dim() != 2 or block_tables.shape[0] < q.shape[0]):
        raise ValueError(f"block_tables must be [>= {q.shape[0]}, max_pages]")
    if seq_lens is not None and seq_lens.numel() < q.shape[0]:
        raise ValueError(f"seq_lens must hold {q.shape[0]} lengths")


def _need(t, dtype, name, device=True):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")


# ----------------------------------------------------------------- host helpers
def kvq_bytes_per_token(fmt, num_kv_heads, head_dim):
    return int(lib().kvq_bytes_per_token(FORMATS.get(fmt, fmt), num_kv_heads, head_dim))


def kvq_cache_array_bytes(fmt, num_pages, page_size, num_kv_heads, head_dim):
    cb, sb = c_int64(), c_int64()
    _check(lib().kvq_cache_array_bytes(FORMATS.get(fmt, fmt), num_pages, page_size, num_kv_heads, head_dim,
                                       ctypes.byref(cb), ctypes.byref(sb)), "kvq_cache_array_bytes")
    return cb.value, sb.value


def kvq_decode_workspace_bytes(total_splits, num_q_heads, head_dim):
    return int(lib().kvq_decode_workspace_bytes(total_splits, num_q_heads, head_dim))


def kvq_verify_workspace_bytes(cache_struct, batch, q_len, num_q_heads, total_splits, target_ctas=0):
    """Workspace bytes of a verify call, the tensor-core route of a one-sequence call included."""
    n = int(lib().kvq_verify_workspace_bytes(ctypes.byref(cache_struct), batch, q_len, num_q_heads, total_splits,
                                             target_ctas))
    if n == 0:
        raise KvqError(1, f"kvq_verify_workspace_bytes: {lib().kvq_last_error().decode()}")
    return n


def _plan(call, name, cache_struct, seq_lens, lead, split_override, target_ctas, virtual_batch):
    """A size query, then the plan itself; ``lead`` = the arguments between
    seq_lens and split_override (the batch, and q_len for a verify plan)."""
    sl = torch.as_tensor(list(seq_lens), dtype=torch.int32)
    total, nctas = c_int32(), c_int32()
    slp = sl.numpy().ctypes.data_as(POINTER(c_int32))
    rc = call(ctypes.byref(cache_struct), slp, *lead, split_override, target_ctas, None, 0, ctypes.byref(total),
              ctypes.byref(nctas))
    if rc not in (0, 3):  # 3 = KVQ_ERR_WORKSPACE (size query)
        _check(rc, name)
    # head groups per split <= num_kv_heads, so this bounds the plan length
    plan = torch.zeros(virtual_batch + 9 + nctas.value + 4 * total.value * cache_struct.num_kv_heads,
                       dtype=torch.int32)
    _check(call(ctypes.byref(cache_struct), slp, *lead, split_override, target_ctas,
                plan.numpy().ctypes.data_as(POINTER(c_int32)), plan.numel(), ctypes.byref(total),
                ctypes.byref(nctas)), name)
    return plan, total.value, nctas.value


def kvq_plan_splits(cache_struct, seq_lens, split_override=0, target_ctas=0):
    """seq_lens: host int sequence.  Returns (plan int32 CPU tensor, total_splits, num_ctas)."""
    B = len(seq_lens)
    return _plan(lib().kvq_plan_splits, "kvq_plan_splits", cache_struct, seq_lens, (B,), split_override,
                 target_ctas, B)


def kvq_plan_verify_splits(cache_struct, seq_lens, q_len, split_override=0, target_ctas=0):
    """The plan of a verify call over q_len query tokens a sequence (the causal
    visible lengths are computed by the library)."""
    B = len(seq_lens)
    return _plan(lib().kvq_plan_verify_splits, "kvq_plan_verify_splits", cache_struct, seq_lens, (B, q_len),
                 split_override, target_ctas, B * q_len)


def kvq_workspace_partials(workspace, total_splits, num_q_heads, head_dim):
    o, l = c_void_p(), c_void_p()
    _check(lib().kvq_workspace_partials(_ptr(workspace), total_splits, num_q_heads, head_dim, ctypes.byref(o),
                                        ctypes.byref(l)), "kvq_workspace_partials")
    return o.value, l.value


def kvq_read_status(dev_status, stream=None):
    """Returns (status code, bits) without raising."""
    bits = c_int32()
    rc = lib().kvq_read_status(_ptr(dev_status), _stream(stream), ctypes.byref(bits))
    return rc, bits.value


def kvq_last_error():
    return lib().kvq_last_error().decode()


# ----------------------------------------------------------------- device calls
def kvq_quant_append(cache_struct, k_new, v_new, slot_mapping, dev_status=None, flags=0, stream=None):
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    _need(slot_mapping, torch.int64, "slot_mapping")
    n = slot_mapping.numel()
    if k_new.shape != v_new.shape or k_new.shape[0] != n:
        raise ValueError("k_new / v_new must be [n_tokens, Hkv, D] and match slot_mapping")
    _check(lib().kvq_quant_append(ctypes.byref(cache_struct), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), n,
                                  _ptr(dev_status), flags, _stream(stream)), "kvq_quant_append")


def kvq_paged_decode_attention(cache_struct, q, sm_scale, block_tables, seq_lens, plan, total_splits, num_ctas,
                               workspace, out, lse_out=None, flags=0, stream=None):
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(plan, torch.int32, "plan")
    _need(workspace, torch.uint8, "workspace")
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    _need(out, out.dtype, "out")
    if lse_out is not None:
        _need(lse_out, torch.float32, "lse_out")
    _shapes(q, out, lse_out, block_tables, seq_lens, cache_struct)
    B, Hq, _ = q.shape
    od = KVQ_OUT_BF16 if out.dtype == torch.bfloat16 else KVQ_OUT_F32
    _check(lib().kvq_paged_decode_attention(
        ctypes.byref(cache_struct), _ptr(q), B, Hq, float(sm_scale), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), _ptr(plan), total_splits, num_ctas, _ptr(workspace), workspace.numel(), _ptr(out), od,
        _ptr(lse_out),
        flags, _stream(stream)), "kvq_paged_decode_attention")


def kvq_paged_decode_attention_static(cache_struct, q, sm_scale, block_tables, seq_lens, plan, total_splits,
                                      num_ctas, out, lse_out=None, flags=0, stream=None):
    """kvq_paged_decode_attention with the library's static scratch region in place of a workspace."""
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(plan, torch.int32, "plan")
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    _need(out, out.dtype, "out")
    if lse_out is not None:
        _need(lse_out, torch.float32, "lse_out")
    _shapes(q, out, lse_out, block_tables, seq_lens, cache_struct)
    B, Hq, _ = q.shape
    od = KVQ_OUT_BF16 if out.dtype == torch.bfloat16 else KVQ_OUT_F32
    _check(lib().kvq_paged_decode_attention_static(
        ctypes.byref(cache_struct), _ptr(q), B, Hq, float(sm_scale), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), _ptr(plan), total_splits, num_ctas, _ptr(out), od, _ptr(lse_out), flags, _stream(stream)),
        "kvq_paged_decode_attention_static")


def kvq_paged_verify_attention(cache_struct, q, sm_scale, block_tables, seq_lens, plan, total_splits, num_ctas,
                               workspace, out, lse_out=None, flags=0, stream=None):
    """q: bf16 [B, q_len, Hq, D]; out: [B, q_len, Hq, D]; lse_out: [B, q_len, Hq]."""
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(plan, torch.int32, "plan")
    _need(workspace, torch.uint8, "workspace")
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    _need(out, out.dtype, "out")
    if lse_out is not None:
        _need(lse_out, torch.float32, "lse_out")
    _shapes(q, out, lse_out, block_tables, seq_lens, cache_struct)
    B, T, Hq, _ = q.shape
    od = KVQ_OUT_BF16 if out.dtype == torch.bfloat16 else KVQ_OUT_F32
    _check(lib().kvq_paged_verify_attention(
        ctypes.byref(cache_struct), _ptr(q), B, T, Hq, float(sm_scale), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), _ptr(plan), total_splits, num_ctas, _ptr(workspace), workspace.numel(), _ptr(out), od,
        _ptr(lse_out), flags, _stream(stream)), "kvq_paged_verify_attention")


def kvq_prefill_splits(cache_struct, q_len, num_q_heads, seq_len, target_ctas=0):
    n = int(lib().kvq_prefill_splits(ctypes.byref(cache_struct), q_len, num_q_heads, seq_len, target_ctas))
    if n < 1:
        _check(-n, "kvq_prefill_splits")
    return n


def kvq_prefill_workspace_bytes(q_len, num_q_heads, head_dim, splits):
    return int(lib().kvq_prefill_workspace_bytes(q_len, num_q_heads, head_dim, splits))


def kvq_paged_prefill_attention(cache_struct, q, sm_scale, block_table, seq_len, splits, workspace, out,
                                lse_out=None, flags=0, stream=None):
    """q: bf16 [T, Hq, D] (the last T tokens of the sequence); block_table: int32 [max_pages]."""
    _need(q, torch.bfloat16, "q")
    _need(block_table, torch.int32, "block_table")
    _need(workspace, torch.uint8, "workspace")
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be float32 or bfloat16")
    _need(out, out.dtype, "out")
    if lse_out is not None:
        _need(lse_out, torch.float32, "lse_out")
    _shapes(q, out, lse_out, None, None, cache_struct)
    T, Hq, _ = q.shape
    od = KVQ_OUT_BF16 if out.dtype == torch.bfloat16 else KVQ_OUT_F32
    _check(lib().kvq_paged_prefill_attention(
        ctypes.byref(cache_struct), _ptr(q), T, Hq, float(sm_scale), _ptr(block_table), block_table.numel(),
        int(seq_len), splits, _ptr(workspace), workspace.numel(), _ptr(out), od, _ptr(lse_out), flags,
        _stream(stream)), "kvq_paged_prefill_attention")


def kvq_split_merge(o_part_ptr, lse_part_ptr, split_offsets, batch, num_q_heads, head_dim, out, lse_out=None,
                    stream=None):
    od = KVQ_OUT_BF16 if out.dtype == torch.bfloat16 else KVQ_OUT_F32
    _check(lib().kvq_split_merge(c_void_p(o_part_ptr), c_void_p(lse_part_ptr), _ptr(split_offsets), batch,
                                 num_q_heads, head_dim, _ptr(out), od, _ptr(lse_out), _stream(stream)),
           "kvq_split_merge")


def kvq_rotate_rows(x, out=None, inverse=False, stream=None):
    """out[..., :] = R(x[..., :]) (or R^-1) over the last axis (head_dim 128 / 256);
    x and out float32 or bfloat16, device or pinned host; out defaults to a new
    tensor of x's dtype on x's device (out may be x)."""
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be float32 or bfloat16")
    if out is None:
        out = torch.empty_like(x)
    if out.dtype not in (torch.float32, torch.bfloat16) or out.shape != x.shape:
        raise TypeError("out must be float32 or bfloat16 with x's shape")
    if not x.is_contiguous() or not out.is_contiguous():
        raise ValueError("x and out must be contiguous")
    D = x.shape[-1]
    dt = lambda t: KVQ_OUT_BF16 if t.dtype == torch.bfloat16 else KVQ_OUT_F32
    _check(lib().kvq_rotate_rows(_ptr(x), dt(x), _ptr(out), dt(out), ctypes.c_int64(x.numel() // max(D, 1)), D,
                                 1 if inverse else 0, _stream(stream)), "kvq_rotate_rows")
    return out

