"""paged_prefill_attention (causal attention of a prompt chunk over the paged
cache, read in place) on the GPU against the float64 oracle's paged_verify (the
same definition: T query tokens whose K/V are the last T cache entries).
Tolerance: max-abs 2e-3 (fp32 output) / 1e-2 (bf16 output)."""
import numpy as np
import pytest
import torch

from quantized_paged_kv_gb300 import workloads as W
from tests import harness as H
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    H.ensure_built()


def _check(wl, fmt, T, splits=0, out_dtype="f32", units=None, gs=(1.0, 1.0)):
    from quantized_paged_kv_gb300 import prefill

    assert wl.B == 1
    cache = H.gpu_cache(wl, fmt, gs=gs)
    q = wl.q_tokens(T)  # [1, T, Hq, D]
    qt = torch.from_numpy(q[0]).to(torch.bfloat16).cuda()
    od = {"f32": torch.float32, "bf16": torch.bfloat16}[out_dtype]
    out = torch.full((T, wl.Hq, wl.D), float("nan"), dtype=od, device="cuda")
    lse = torch.full((T, wl.Hq), float("nan"), device="cuda")
    bt = torch.from_numpy(wl.block_tables[0]).cuda()
    prefill(cache, qt, bt, int(wl.seq_lens[0]), out, wl.sm_scale, lse_out=lse, splits=splits, checked=True)
    torch.cuda.synchronize()
    pools = H.oracle_pools(wl, fmt, gs=gs)
    ref, ref_lse = oatt.paged_verify(fmt, pools, q, wl.block_tables, wl.seq_lens, wl.sm_scale, units=units)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    sel = ~np.isnan(ref_lse[0])
    err = np.abs(o - ref[0])[sel]
    assert np.all(np.isfinite(o[sel])), (fmt, T, splits)
    assert np.all(err <= H.bound(out_dtype, ref[0][sel])), (fmt, T, splits, err.max())
    assert np.abs(l[sel] - ref_lse[0][sel]).max() < 1e-3


@pytest.mark.parametrize("fmt", ["int8", "nvfp4", "bf16"])
@pytest.mark.parametrize("T", [1, 5, 37, 130])
def test_prefill_d256_gqa6(fmt, T):
    wl = W.make("tiny_int8", lens=("list", [700]), seed=41)
    for splits in (1, 3, 0):
        _check(wl, fmt, T, splits)


@pytest.mark.parametrize("fmt", ["int8", "nvfp4", "bf16"])
def test_prefill_d128_gqa4_bf16_out(fmt):
    wl = W.make("serving_int8", lens=("list", [1500]), seed=42)
    _check(wl, fmt, 200, 0, "bf16")
    _check(wl, fmt, 200, 2, "bf16")


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_prefill_nvfp4_tensor_global_scales(out_dtype):
    # the global scales of the NVFP4 page's standalone choice (448 * 6 / amax per tensor)
    wl = W.make("tiny_int8", lens=("list", [900]), seed=44)
    gs = H.global_scales(wl, "nvfp4")
    _check(wl, "nvfp4", 70, 0, out_dtype, gs=gs)
    _check(wl, "nvfp4", 70, 2, out_dtype, gs=gs)


def test_prefill_whole_sequence_and_tail_page():
    # T = seq_len (the first chunk of a prompt) and a seq_len that ends mid-page
    wl = W.make("tiny_int8", lens=("list", [333]), seed=43)
    _check(wl, "int8", 333, 0)
    _check(wl, "int8", 333, 4)


def test_prefill_long_context_sampled():
    """A 2,048-token chunk at the end of a 32K context (sampled query tokens)."""
    wl = W.make("long_int8")
    units = [(0, i, h) for i in (0, 1023, 2047) for h in (0, 3)]
    _check(wl, "int8", 2048, 0, units=units)
