"""paged_verify_attention (causal attention for several query tokens a
sequence) on the GPU against the float64 oracle's paged_verify, through the C ABI.
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


def _run(wl, fmt, T, split=0, out_dtype="f32", gs=(1.0, 1.0), checked=True):
    from quantized_paged_kv_gb300 import DecodePlan, verify

    cache = H.gpu_cache(wl, fmt, gs)
    plan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=split, q_len=T)
    q = wl.q_tokens(T)
    qt = torch.from_numpy(q).to(torch.bfloat16).cuda()
    od = {"f32": torch.float32, "bf16": torch.bfloat16}[out_dtype]
    out = torch.full((wl.B, T, wl.Hq, wl.D), float("nan"), dtype=od, device="cuda")
    lse = torch.full((wl.B, T, wl.Hq), float("nan"), device="cuda")
    bt = torch.from_numpy(wl.block_tables).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    verify(cache, plan, qt, bt, sl, out, wl.sm_scale, lse_out=lse, checked=checked)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), q, plan


def _compare(wl, fmt, T, split=0, out_dtype="f32", gs=(1.0, 1.0), units=None):
    out, lse, q, plan = _run(wl, fmt, T, split, out_dtype, gs)
    pools = H.oracle_pools(wl, fmt, gs, seqs=None if units is None else sorted({b for b, _, _ in units}))
    ref, ref_lse = oatt.paged_verify(fmt, pools, q, wl.block_tables, wl.seq_lens, wl.sm_scale, units=units)
    sel = ~np.isnan(ref_lse)
    rows = sel[..., None].repeat(wl.D, -1)
    assert np.all(np.isfinite(out[rows]))
    assert np.all(np.abs(out - ref)[rows] <= H.bound(out_dtype, ref[rows])), (fmt, T, split)
    fin = sel & np.isfinite(ref_lse)
    assert np.abs(lse[fin] - ref_lse[fin]).max() < 1e-3
    assert np.all(np.isneginf(lse[sel & ~np.isfinite(ref_lse)]))
    return plan


@pytest.mark.parametrize("fmt", ["int8", "int8_g32", "nvfp4", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 4, 6])
def test_verify_matches_the_oracle(fmt, T):
    # lengths include ones shorter than T: early query tokens then see nothing
    wl = W.make("tiny_int8", lens=("list", [700, 33, 4096, 5, 1]), seed=31)
    gs = H.global_scales(wl, fmt)
    for split in (1, 3, 0):
        _compare(wl, fmt, T, split, "f32", gs)


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
def test_verify_bf16_output_and_gqa_4(fmt):
    # D = 128, 4 query heads a KV head (the serving mix's shape)
    wl = W.make("serving_int8", lens=("list", [300, 1000, 2, 2500]), seed=32)
    _compare(wl, fmt, 3, 0, "bf16", H.global_scales(wl, fmt))


def test_single_token_verify_is_the_decode():
    from quantized_paged_kv_gb300 import DecodePlan, decode

    wl = W.make("tiny_int8", lens=("list", [700, 33, 4096]), seed=33)
    out_v, lse_v, q, plan = _run(wl, "int8", 1, 3)
    cache = H.gpu_cache(wl, "int8")
    dplan = DecodePlan(cache, wl.seq_lens, wl.Hq, split_override=3)
    o = torch.empty((wl.B, wl.Hq, wl.D), device="cuda")
    lse = torch.empty((wl.B, wl.Hq), device="cuda")
    decode(cache, dplan, torch.from_numpy(q[:, 0]).to(torch.bfloat16).cuda(), torch.from_numpy(wl.block_tables).cuda(),
           torch.from_numpy(wl.seq_lens).cuda(), o, wl.sm_scale, lse_out=lse, checked=True)
    torch.cuda.synchronize()
    assert np.array_equal(out_v[:, 0], o.cpu().numpy())
    assert np.array_equal(lse_v[:, 0], lse.cpu().numpy())


def test_verify_32k_six_tokens_sampled():
    """The pages' verify step shape: 6 query tokens x 6 query heads of a KV head,
    32K context, in the automatic plan the benchmark uses; sampled units."""
    wl = W.make("long_int8")
    units = [(0, i, h) for i in (0, 3, 5) for h in (0, 3)]
    _compare(wl, "int8", 6, 0, "f32", units=units)
