"""Verify calls with enough query tokens a sequence (one sequence: 10 on a block
table under 512 pages, 6 from 512, 5 from 1,024, 4 from 2,048, fewer for NVFP4;
a batch: 6, NVFP4 4) run on the tensor-core prefill kernel, one launch for the
whole batch, with the sequence lengths read on the device.  Checked against the float64 oracle's paged_verify (max-abs
2e-3 for fp32 output, 1e-2 or half a bf16 ulp for bf16 output), against the same
call kept on the decode kernel by a workspace too small for the route, through a
CUDA graph, and for the flag the kernel raises when the device length runs past
the block table."""
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


class _Call:
    """One verify call's tensors; run(workspace) calls it and returns (out, lse) as numpy."""

    def __init__(self, wl, fmt, T, gs=(1.0, 1.0), out_dtype="f32", split=0, seq_len=None):
        from quantized_paged_kv_gb300 import DecodePlan

        self.wl, self.T = wl, T
        self.cache = H.gpu_cache(wl, fmt, gs)
        self.plan = DecodePlan(self.cache, wl.seq_lens, wl.Hq, split_override=split, q_len=T)
        self.q = wl.q_tokens(T)
        self.qt = torch.from_numpy(self.q).to(torch.bfloat16).cuda()
        od = {"f32": torch.float32, "bf16": torch.bfloat16}[out_dtype]
        self.out = torch.full((wl.B, T, wl.Hq, wl.D), float("nan"), dtype=od, device="cuda")
        self.lse = torch.full((wl.B, T, wl.Hq), float("nan"), device="cuda")
        self.bt = torch.from_numpy(wl.block_tables).cuda()
        lens = wl.seq_lens if seq_len is None else np.array(np.atleast_1d(seq_len), np.int32)
        self.sl = torch.from_numpy(lens).cuda()

    def launch(self, workspace=None, checked=True):
        from quantized_paged_kv_gb300 import _binding as B

        ws = self.plan.workspace if workspace is None else workspace
        B.kvq_paged_verify_attention(self.cache.struct, self.qt, self.wl.sm_scale, self.bt, self.sl, self.plan.plan,
                                     self.plan.total_splits, self.plan.num_ctas, ws, self.out, self.lse,
                                     B.KVQ_CHECKED if checked else 0, None)

    def run(self, workspace=None, checked=True):
        self.out.fill_(float("nan"))
        self.lse.fill_(float("nan"))
        self.launch(workspace, checked)
        torch.cuda.synchronize()
        return self.out.float().cpu().numpy(), self.lse.cpu().numpy()

    def decode_only_workspace(self):
        """A workspace that holds the decode plan's partials only (too small for a routed call's)."""
        from quantized_paged_kv_gb300 import _binding as B

        n = B.kvq_decode_workspace_bytes(self.plan.total_splits, self.wl.Hq, self.wl.D)
        assert n <= self.plan.workspace.numel()
        return torch.zeros(n, dtype=torch.uint8, device="cuda")


def _compare(wl, fmt, T, out, lse, gs, out_dtype="f32", units=None):
    pools = H.oracle_pools(wl, fmt, gs)
    ref, ref_lse = oatt.paged_verify(fmt, pools, wl.q_tokens(T), wl.block_tables, wl.seq_lens, wl.sm_scale,
                                     units=units)
    sel = ~np.isnan(ref_lse)
    rows = sel[..., None].repeat(wl.D, -1)
    assert np.all(np.isfinite(out[rows]))
    err = np.abs(out - ref)[rows]
    assert np.all(err <= H.bound(out_dtype, ref[rows])), (fmt, T, err.max())
    fin = sel & np.isfinite(ref_lse)
    if fin.any():
        assert np.abs(lse[fin] - ref_lse[fin]).max() < 1e-3
    assert np.all(np.isneginf(lse[sel & ~np.isfinite(ref_lse)]))
    assert np.all(out[sel & ~np.isfinite(ref_lse)] == 0)


@pytest.mark.parametrize("fmt", ["int8", "nvfp4", "bf16"])
@pytest.mark.parametrize("T", [12, 22, 43])
@pytest.mark.parametrize("L", [3, 700, 5000])
def test_routed_verify_matches_the_oracle(fmt, T, L):
    """6 query heads a KV head: 72 to 258 rows (one to three 128-row blocks); L < T
    leaves the first tokens with no visible key; the key splits cover a ragged last page."""
    wl = W.make("tiny_int8", lens=("list", [L]), seed=51)
    gs = H.global_scales(wl, fmt)
    c = _Call(wl, fmt, T, gs)
    out, lse = c.run()
    _compare(wl, fmt, T, out, lse, gs)


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
def test_routed_verify_d128_gqa4_bf16_output(fmt):
    # 12 tokens x 4 query heads a KV head = 48 rows, D = 128
    wl = W.make("serving_int8", lens=("list", [2500]), seed=52)
    gs = H.global_scales(wl, fmt)
    c = _Call(wl, fmt, 12, gs, out_dtype="bf16")
    out, lse = c.run()
    _compare(wl, fmt, 12, out, lse, gs, out_dtype="bf16")


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
def test_route_and_decode_kernel_agree(fmt):
    """The same call on both kernels: each within the tolerance of the oracle, so
    within twice of each other; the two routes round differently, so the outputs
    are not bit-equal (the route was taken)."""
    wl = W.make("tiny_int8", lens=("list", [1500]), seed=53)
    gs = H.global_scales(wl, fmt)
    c = _Call(wl, fmt, 12, gs, split=1)
    routed = c.run()
    kept = c.run(c.decode_only_workspace())
    _compare(wl, fmt, 12, routed[0], routed[1], gs)
    _compare(wl, fmt, 12, kept[0], kept[1], gs)
    assert np.abs(routed[0] - kept[0]).max() <= 4e-3
    assert not np.array_equal(routed[0], kept[0])


@pytest.mark.parametrize("fmt,T", [("int8", 9), ("nvfp4", 7)])
def test_below_the_token_threshold_the_decode_kernel_runs(fmt, T):
    """A 94-page block table: fewer than 10 tokens (8 for NVFP4) stay on the
    decode kernel whatever the workspace (bit-equal)."""
    wl = W.make("tiny_int8", lens=("list", [1500]), seed=54)
    c = _Call(wl, fmt, T, H.global_scales(wl, fmt), split=1)
    a = c.run()
    big = torch.zeros(c.plan.workspace.numel() + (8 << 20), dtype=torch.uint8, device="cuda")
    b = c.run(big)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("fmt,T,routed", [("int8", 4, True), ("int8", 3, False), ("nvfp4", 3, True)])
def test_long_context_threshold(fmt, T, routed):
    """A 32K context (2,048-page block table): 4 tokens are routed (3 for NVFP4);
    sampled units against the oracle on either kernel, and the route decides
    whether the call's bits differ from the decode kernel's."""
    wl = W.make("long_int8")
    gs = H.global_scales(wl, fmt)
    c = _Call(wl, fmt, T, gs, split=1)
    auto = c.run()
    kept = c.run(c.decode_only_workspace())
    units = [(0, i, h) for i in (0, T - 1) for h in (1, 2)]
    _compare(wl, fmt, T, auto[0], auto[1], gs, units=units)
    assert np.array_equal(auto[0], kept[0]) != routed


def test_routed_verify_in_a_cuda_graph():
    """Captured once, replayed: the same bits as the eager call."""
    wl = W.make("tiny_int8", lens=("list", [3000]), seed=55)
    c = _Call(wl, "int8", 12)
    ref = c.run(checked=False)
    c.out.fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            c.launch(checked=False)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(c.out.cpu().numpy(), ref[0])
    assert np.array_equal(c.lse.cpu().numpy(), ref[1])


def test_device_length_past_the_block_table_is_flagged():
    """Unchecked call whose device seq_len runs past the block table: the kernel
    clamps it to the table's width (every read stays inside the table) and raises
    KVQ_DEV_BAD_SEQLEN in the status word."""
    from quantized_paged_kv_gb300 import _binding as B

    wl = W.make("tiny_int8", lens=("list", [700]), seed=56)
    width = wl.block_tables.shape[1]
    c = _Call(wl, "int8", 12, seq_len=width * 16 + 40)
    c.run(checked=False)
    rc, bits = B.kvq_read_status(c.plan.workspace, None)
    assert rc != 0 and bits & B.KVQ_DEV_BAD_SEQLEN


@pytest.mark.parametrize("fmt,T", [("int8", 6), ("nvfp4", 8)])
def test_routed_verify_32k_sampled(fmt, T):
    """The pages' verify shape (6 query tokens x 6 heads, 32K context) and 8 tokens
    in NVFP4, on sampled (token, KV head) units."""
    wl = W.make("long_int8")
    gs = H.global_scales(wl, fmt)
    c = _Call(wl, fmt, T, gs)
    out, lse = c.run()
    units = [(0, i, h) for i in (0, T // 2, T - 1) for h in (0, 3)]
    _compare(wl, fmt, T, out, lse, gs, units=units)


@pytest.mark.parametrize("fmt", ["int8", "nvfp4", "bf16"])
@pytest.mark.parametrize("T", [6, 22])
def test_batched_routed_verify_matches_the_oracle(fmt, T):
    """Four sequences in one launch: lengths 5 to 5,000 (one shorter than T, ragged
    last pages, a block table wider than most of them)."""
    wl = W.make("tiny_int8", lens=("list", [700, 5, 5000, 1300]), seed=57)
    gs = H.global_scales(wl, fmt)
    c = _Call(wl, fmt, T, gs)
    out, lse = c.run()
    _compare(wl, fmt, T, out, lse, gs)


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
def test_batched_route_and_decode_kernel_agree_d128_bf16_output(fmt):
    """Three sequences of the serving shape (4 query heads a KV head, D = 128), bf16
    output: both kernels within the oracle's tolerance, and the route was taken."""
    wl = W.make("serving_int8", lens=("list", [300, 2500, 1000]), seed=58)
    gs = H.global_scales(wl, fmt)
    c = _Call(wl, fmt, 8, gs, out_dtype="bf16", split=1)
    routed = c.run()
    kept = c.run(c.decode_only_workspace())
    _compare(wl, fmt, 8, routed[0], routed[1], gs, out_dtype="bf16")
    _compare(wl, fmt, 8, kept[0], kept[1], gs, out_dtype="bf16")
    assert not np.array_equal(routed[0], kept[0])


def test_batched_bad_device_length_is_flagged():
    """One of two sequences has a device length past the block table: flagged, and
    every read stays inside the table (clamped)."""
    from quantized_paged_kv_gb300 import _binding as B

    wl = W.make("tiny_int8", lens=("list", [700, 400]), seed=59)
    width = wl.block_tables.shape[1]
    c = _Call(wl, "int8", 6, seq_len=[700, width * 16 + 40])
    c.run(checked=False)
    rc, bits = B.kvq_read_status(c.plan.workspace, None)
    assert rc != 0 and bits & B.KVQ_DEV_BAD_SEQLEN


@pytest.mark.parametrize("fmt,T,routed", [("int8", 5, False), ("int8", 6, True), ("nvfp4", 3, False), ("nvfp4", 4, True)])
def test_batch_token_threshold(fmt, T, routed):
    """Two sequences: 6 query tokens a sequence take the tensor-core kernel (4 for
    NVFP4), fewer stay on the decode kernel; either way within the oracle's
    tolerance, and the route decides whether the bits differ from the decode
    kernel's."""
    wl = W.make("tiny_int8", lens=("list", [1500, 900]), seed=60)
    gs = H.global_scales(wl, fmt)
    c = _Call(wl, fmt, T, gs, split=1)
    auto = c.run()
    kept = c.run(c.decode_only_workspace())
    _compare(wl, fmt, T, auto[0], auto[1], gs)
    assert np.array_equal(auto[0], kept[0]) != routed


@pytest.mark.parametrize("fmt", ["int8", "nvfp4", "bf16"])
def test_routed_raw_mode_bad_page_ids_contribute_nothing(fmt):
    """Raw mode on the tensor-core route: block-table entries outside the pool are
    flagged and their pages' tokens are left out of the softmax, as on the decode
    kernel (the pool is sentinel-filled, so a page read anyway would show); each
    query token's result equals the oracle's attention over its visible tokens
    without those pages, and a token that sees only bad pages gives 0 and -inf."""
    from oracle import layout as olay
    from quantized_paged_kv_gb300 import _binding as B

    wl = W.make("tiny_int8", lens=("list", [700, 64, 300]), seed=61)
    gs = H.global_scales(wl, fmt)
    T = 6
    c = _Call(wl, fmt, T, gs)
    drop = {0: [0, 5, 43], 1: [0, 1, 2, 3], 2: [18]}  # sequence 1: every page; sequence 2: the last
    bad = wl.block_tables.copy()
    for b, js in drop.items():
        for j in js:
            bad[b, j] = wl.num_pages + 7 + j
    c.bt = torch.from_numpy(bad).cuda()
    out, lse = c.run(checked=False)
    rc, bits = B.kvq_read_status(c.plan.workspace, None)
    assert rc != 0 and bits == B.KVQ_DEV_BAD_PAGE
    pools = H.oracle_pools(wl, fmt, gs)
    q = wl.q_tokens(T)
    G = wl.Hq // wl.Hkv
    for b in range(wl.B):
        L = int(wl.seq_lens[b])
        for i in range(T):
            vis = max(0, L - T + 1 + i)
            keep = np.array([t for t in range(vis) if t // 16 not in drop[b]], dtype=np.int64)
            slots = olay.token_slots(wl.block_tables[b], vis, 16)[keep]
            for h in range(wl.Hkv):
                k = oatt.cache_rows(fmt, pools["k_codes"], pools.get("k_scales"), slots, h, gs[0])
                v = oatt.cache_rows(fmt, pools["v_codes"], pools.get("v_scales"), slots, h, gs[1])
                ro, rl = oatt.attend(q[b, i, h * G:(h + 1) * G], k, v, wl.sm_scale)
                rows = slice(h * G, (h + 1) * G)
                assert np.all(np.abs(out[b, i, rows] - ro) <= H.bound("f32", ro)), (fmt, b, i, h)
                if len(keep) == 0:
                    assert np.all(out[b, i, rows] == 0) and np.all(np.isneginf(lse[b, i, rows]))
                else:
                    assert np.abs(lse[b, i, rows] - rl).max() < 1e-3


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
def test_routed_verify_equals_the_prefill_call(fmt):
    """One sequence whose block table is exactly as wide as its pages: the routed
    verify call and kvq_paged_prefill_attention of the same tokens pick the same
    key splits and run the same kernel, so their outputs are the same bits."""
    from quantized_paged_kv_gb300 import _binding as B
    from quantized_paged_kv_gb300 import prefill

    wl = W.make("tiny_int8", lens=("list", [700]), seed=62)
    assert wl.block_tables.shape[1] == -(-700 // 16)
    gs = H.global_scales(wl, fmt)
    T = 12
    c = _Call(wl, fmt, T, gs)
    out_v, lse_v = c.run()
    S = B.kvq_prefill_splits(c.cache.struct, T, wl.Hq, 700)
    out_p = torch.full((T, wl.Hq, wl.D), float("nan"), device="cuda")
    lse_p = torch.full((T, wl.Hq), float("nan"), device="cuda")
    prefill(c.cache, c.qt[0].contiguous(), c.bt[0].contiguous(), 700, out_p, wl.sm_scale, lse_out=lse_p, splits=S,
            checked=True)
    torch.cuda.synchronize()
    assert np.array_equal(out_v[0], out_p.cpu().numpy())
    assert np.array_equal(lse_v[0], lse_p.cpu().numpy())


@pytest.mark.parametrize("fmt", ["int8", "nvfp4"])
def test_verify_entry_as_a_batched_chunked_prefill(fmt):
    """Two sequences, the last 200 tokens of each as query tokens (1,200 query
    rows a KV head, ten 128-row blocks): a chunked prefill of a batch through the
    verify entry, against the oracle on sampled (sequence, token, KV head) units."""
    wl = W.make("tiny_int8", lens=("list", [900, 1300]), seed=63)
    gs = H.global_scales(wl, fmt)
    T = 200
    c = _Call(wl, fmt, T, gs)
    out, lse = c.run()
    units = [(b, i, h) for b in (0, 1) for i in (0, 57, 128, 199) for h in (0, 3)]
    _compare(wl, fmt, T, out, lse, gs, units=units)
