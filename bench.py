"""Benchmark: split-KV decode attention over a paged INT8 KV cache on GB300.

Default workload (one decode-attention call = one step): B=1, 24 query / 4 KV
heads, D=256, 32,768-token context in 16-token pages scattered by a random block
table, INT8 cache with fp32 per-token-head scales, automatic split plan, fp32
output.  R independent layer pools (R x 68 MB > 4 x L2) are visited round-robin so
consecutive steps never hit a warm L2; R consecutive calls are captured in one
CUDA graph and replayed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--sweep]

Prints one JSON line (rank 0).  Under torchrun the job is one independent
problem of the workload per rank (own seed, own pools), the sequences sharded
across ranks with no exchange in the data path (weak scaling); the only
collectives are barriers and the max-over-ranks of the timings.  --impl reference times the float64 CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention µs/step and KV GB/s read (fraction of GB300 HBM peak)"
UNIT = "GB/s"
WORKLOAD = "long_int8"
HEADLINE_WORKLOAD = ("long-context batch-1 INT8 decode: B=1, Hq=24, Hkv=4, D=256, context 32768, page 16, "
                     "permuted pages, fp32 out")


# ----------------------------------------------------------------------------- helpers
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep", action="store_true", help="also measure the other workloads and the split sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="skip the nvidia-smi clock sampler")
    ap.add_argument("--min-seconds", type=float, default=MIN_TIMED_S,
                    help="shortest timed region of the headline (0: exactly the whole replays --steps asks for, "
                         "e.g. for a profiler's launch list)")
    ap.add_argument("--ncu-case", default=None, metavar="WORKLOAD",
                    help="profiling case: build the workload's pools (just over L2 in total), run --calls eager "
                         "decode calls over them and exit (no timing); for append_int8, --calls appends")
    ap.add_argument("--fmt", default="int8", choices=["int8", "nvfp4", "bf16"])
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--verify-tokens", type=int, default=0, help="profiling case: verify calls of this many tokens")
    ap.add_argument("--prefill-tokens", type=int, default=0, help="profiling case: prefill calls of this many tokens")
    return ap.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def kernel_sha():
    h = hashlib.sha256()
    for f in ("decode.cuh", "kvq_ptx.cuh", "decode_launch.cu"):
        with open(os.path.join(ROOT, "quantized_paged_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_record(workload):
    """DRAM bytes per decode launch from a committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        r = rec.get(workload)
        if r and r.get("kernel_sha") == kernel_sha():
            return r
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms in the background."""

    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "20", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- our arm
class LayerSet:
    """R layer pools of one workload + the per-call device arguments."""

    def __init__(self, wl, fmt, R, device, gs=(1.0, 1.0)):
        import torch

        import quantized_paged_kv_gb300 as kvq
        from quantized_paged_kv_gb300 import workloads as W

        self.wl, self.fmt, self.R = wl, fmt, R
        self.caches = []
        for r in range(R):
            c = kvq.KVCache(fmt, wl.num_pages, wl.Hkv, wl.D, device=device, k_global_scale=gs[0],
                            v_global_scale=gs[1], fill=0)
            for b in range(wl.B):
                if wl.seq_lens[b] == 0:
                    continue
                k, v = W.device_kv(wl, b, layer=r, device=device)
                c.append(k, v, torch.from_numpy(wl.slots(b)).to(device))
            self.caches.append(c)
        torch.cuda.synchronize()
        self.q = torch.from_numpy(wl.q()).to(torch.bfloat16).to(device)
        self.bt = torch.from_numpy(wl.block_tables).to(device)
        self.sl = torch.from_numpy(wl.seq_lens).to(device)
        od = torch.float32 if wl.out_dtype == "f32" else torch.bfloat16
        self.out = torch.empty((wl.B, wl.Hq, wl.D), dtype=od, device=device)
        self.device = device

    def plan(self, split=0):
        import quantized_paged_kv_gb300 as kvq

        return kvq.DecodePlan(self.caches[0], self.wl.seq_lens, self.wl.Hq, split_override=split, device=self.device)

    def call(self, r, plan, skip_merge=False):
        # the plan and block tables are written once, before any timed call: the
        # decode may read them while the previous call's kernels finish
        import quantized_paged_kv_gb300 as kvq

        kvq.decode(self.caches[r], plan, self.q, self.bt, self.sl, self.out, self.wl.sm_scale, skip_merge=skip_merge,
                   early_start=True)

    def kv_bytes(self):
        import quantized_paged_kv_gb300 as kvq

        return int(self.wl.seq_lens.sum()) * kvq.kvq_bytes_per_token(self.fmt, self.wl.Hkv, self.wl.D)


MIN_TIMED_S = 1.0  # the headline's timed region lasts at least this long, whatever --steps says


def time_graph(ls, plan, steps, warmup, skip_merge=False, barrier=None, sampler=None, min_seconds=0.0):
    """Capture R consecutive calls in a CUDA graph; replay to run `steps` calls
    (rounded up to whole replays, and to at least `min_seconds` of replays);
    returns (seconds per call, calls timed, clock record)."""
    import torch

    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for r in range(ls.R):  # eager warm-up of every layer (sets kernel attributes etc.)
            ls.call(r, plan, skip_merge)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for r in range(ls.R):
            ls.call(r, plan, skip_merge)
    reps = max(1, math.ceil(steps / ls.R))
    wreps = max(1, math.ceil(warmup / ls.R))
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        w0.record(stream)
        for _ in range(wreps):
            g.replay()
        w1.record(stream)
    stream.synchronize()
    if min_seconds > 0:  # enough replays to fill the minimum timed region (estimated from the warm-up)
        per_replay = max(w0.elapsed_time(w1) * 1e-3 / wreps, 1e-7)
        reps = max(reps, math.ceil(min_seconds / per_replay))
    if barrier:
        barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    if barrier:
        barrier()
    return e0.elapsed_time(e1) * 1e-3 / (reps * ls.R), reps * ls.R, clocks


def time_append(wl, fmt, dev, l2, steps, warmup=16, rotate=None):
    """kvq_quant_append of the workload's new tokens (the last `append_tail` tokens
    of every sequence), timed as a CUDA graph of R appends that cycle through R
    input sets and R pools, so that inputs and written pages are not L2-resident.
    rotate="fused": the append rotates each row itself (KVQ_ROTATE); "two_call":
    kvq_rotate_rows of K and V into scratch rows, then the plain append.  Bytes and
    GB/s count the append's own input and output either way."""
    import torch

    import quantized_paged_kv_gb300 as kvq
    from quantized_paged_kv_gb300 import workloads as W

    ks, vs, ss = [], [], []
    for b in range(wl.B):
        k, v = W.device_kv(wl, b, device=dev)
        ks.append(k[-wl.append_tail:])
        vs.append(v[-wl.append_tail:])
        ss.append(torch.from_numpy(wl.slots(b)[-wl.append_tail:]))
    k0, v0, s0 = torch.cat(ks), torch.cat(vs), torch.cat(ss).to(dev)
    n_tok = k0.shape[0]
    gs = (448.0 * 6.0 / float(k0.abs().max()), 448.0 * 6.0 / float(v0.abs().max())) if fmt == "nvfp4" else (1.0, 1.0)
    in_bytes = k0.numel() * 2 * 2
    out_bytes = n_tok * kvq.kvq_bytes_per_token(fmt, wl.Hkv, wl.D)
    R = max(2, math.ceil(2 * l2 / (in_bytes + out_bytes)))
    sets = []
    for r in range(R):  # distinct inputs (a permutation of the tokens' rows) and pools
        perm = torch.randperm(n_tok, device=dev, generator=torch.Generator(device=dev).manual_seed(r))
        cache = kvq.KVCache(fmt, wl.num_pages, wl.Hkv, wl.D, device=dev, k_global_scale=gs[0],
                            v_global_scale=gs[1], fill=0)
        sets.append((cache, k0[perm].contiguous(), v0[perm].contiguous(), s0))
    del k0, v0
    if rotate == "two_call":
        rk, rv = torch.empty_like(sets[0][1]), torch.empty_like(sets[0][2])

    def one(cache, k, v, s):
        if rotate == "two_call":
            kvq.kvq_rotate_rows(k.view(-1, wl.D), rk.view(-1, wl.D))
            kvq.kvq_rotate_rows(v.view(-1, wl.D), rv.view(-1, wl.D))
            cache.append(rk, rv, s)
        else:
            cache.append(k, v, s, rotate=rotate == "fused")

    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for cache, k, v, s in sets:
            one(cache, k, v, s)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for cache, k, v, s in sets:
            one(cache, k, v, s)
    reps = max(1, math.ceil(steps / R))
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(warmup / R))):
            g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / (reps * R)
    nbytes = in_bytes + out_bytes
    peak = measured_peaks()[0]["hbm_gbs"]
    del sets, g
    return {"us": round(t * 1e6, 3), "GBps": round(nbytes / t / 1e9, 1), "frac": round(nbytes / t / 1e9 / peak, 4),
            "bytes": nbytes, "inputs": R,
            "note": "CUDA graph of R appends over R input sets and R pools (inputs larger than L2)"}


def time_graph_fn(fn, R, reps=50):
    """CUDA graph of fn(0) .. fn(R-1); seconds per fn call over `reps` replays."""
    import torch

    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for r in range(R):
            fn(r)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for r in range(R):
            fn(r)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / (reps * R)


def time_rotation(dev, l2, peak):
    """kvq_rotate_rows over the append workload's new K/V rows (65,536 rows of 256
    bf16, in place over inputs larger than L2 in total), and the cost it adds
    around a 32K batch-1 decode call (q rotated before, the output rotated back)."""
    import torch

    import quantized_paged_kv_gb300 as kvq
    from quantized_paged_kv_gb300 import workloads as W

    res = {}
    rows, D = 8192 * 4 * 2, 256
    nbytes = rows * D * 2
    R = max(2, math.ceil(2 * l2 / (2 * nbytes)))
    bufs = [torch.randn(rows, D, device=dev).to(torch.bfloat16) for _ in range(R)]
    t = time_graph_fn(lambda r: kvq.kvq_rotate_rows(bufs[r], bufs[r]), R)
    res["rotate_rows/65536x256 bf16"] = {"us": round(t * 1e6, 3), "GBps": round(2 * nbytes / t / 1e9, 1),
                                         "frac": round(2 * nbytes / t / 1e9 / peak, 4), "inputs": R}
    del bufs
    wl = W.make("long_int8")
    ls = LayerSet(wl, "int8", 16, dev)
    plan = ls.plan(0)
    qr = torch.empty_like(ls.q)

    def rotated_call(r):
        kvq.kvq_rotate_rows(ls.q, qr)
        kvq.decode(ls.caches[r], plan, qr, ls.bt, ls.sl, ls.out, wl.sm_scale, early_start=True)
        kvq.kvq_rotate_rows(ls.out, ls.out, inverse=True)

    t_plain = time_graph_fn(lambda r: ls.call(r, plan), ls.R)
    t_rot = time_graph_fn(rotated_call, ls.R)
    res["rotated_decode/long_int8"] = {"us": round(t_rot * 1e6, 3), "plain_us": round(t_plain * 1e6, 3),
                                       "note": "q rotated before the call, the output rotated back after it"}
    del ls
    return res


def time_verify(ls, T, steps, warmup=16):
    """Verify calls (T query tokens a sequence, causal) over the R layer pools in
    one CUDA graph; KV GB/s counts each page once."""
    import torch

    import quantized_paged_kv_gb300 as kvq

    wl = ls.wl
    plan = kvq.DecodePlan(ls.caches[0], wl.seq_lens, wl.Hq, device=ls.device, q_len=T)
    q = torch.from_numpy(wl.q_tokens(T)).to(torch.bfloat16).to(ls.device)
    out = torch.empty((wl.B, T, wl.Hq, wl.D), dtype=ls.out.dtype, device=ls.device)
    stream = torch.cuda.Stream()

    def one(r):
        kvq.verify(ls.caches[r], plan, q, ls.bt, ls.sl, out, wl.sm_scale, early_start=True)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for r in range(ls.R):
            one(r)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for r in range(ls.R):
            one(r)
    reps = max(1, math.ceil(steps / ls.R))
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(warmup / ls.R))):
            g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / (reps * ls.R)
    nbytes = ls.kv_bytes()
    return {"us": round(t * 1e6, 3), "GBps": round(nbytes / t / 1e9, 1), "splits": plan.total_splits,
            "query_rows": T * wl.Hq, "note": "KV bytes counted once per call"}


def time_prefill(ls, T, peak_tf, reps=20):
    """Prefill of the last T tokens of layer pools' sequence (causal), CUDA graph of
    the R layers' calls; FLOPs = 4 * Hq * D * (visible keys summed over the T tokens)."""
    import torch

    import quantized_paged_kv_gb300 as kvq

    wl = ls.wl
    L = int(wl.seq_lens[0])
    q = torch.from_numpy(wl.q_tokens(T)[0]).to(torch.bfloat16).to(ls.device)
    out = torch.empty((T, wl.Hq, wl.D), dtype=ls.out.dtype, device=ls.device)
    bt = ls.bt[0].contiguous()
    splits = kvq.kvq_prefill_splits(ls.caches[0].struct, T, wl.Hq, L)
    ws = torch.zeros(kvq.kvq_prefill_workspace_bytes(T, wl.Hq, wl.D, splits), dtype=torch.uint8, device=ls.device)
    stream = torch.cuda.Stream()

    def one(r):
        kvq.prefill(ls.caches[r], q, bt, L, out, wl.sm_scale, splits=splits, workspace=ws)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for r in range(ls.R):
            one(r)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for r in range(ls.R):
            one(r)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / (reps * ls.R)
    visible = sum(L - T + i + 1 for i in range(T))
    flops = 4.0 * wl.Hq * wl.D * visible
    return {"us": round(t * 1e6, 2), "TFLOPs": round(flops / t / 1e12, 1), "frac_of_bf16_peak": round(flops / t / 1e12 / peak_tf, 4),
            "splits": splits, "context": L, "note": "tcgen05 kind::f16 (fp32 accumulate); peak = measured cuBLAS bf16 burst"}


def time_e2e(ls, plan, steps, warmup=3):
    """Through the public API with host buffers: every step hands the C ABI
    pinned host memory for q, the block table and seq_lens (inputs) and for the
    output; the kernels read and write it over the host link (NVLink-C2C), so the
    host->device and device->host transfers of the step happen inside the timed
    region, in the kernels' own loads and stores.  R consecutive steps are
    captured in one CUDA graph and replayed, as the device-side timing is.
    (Graph memcpy nodes between the kernels measured ~14 us a step here: more
    than the transfers themselves.)"""
    import torch

    import quantized_paged_kv_gb300 as kvq

    q_h = ls.q.cpu().pin_memory()
    bt_h = ls.bt.cpu().pin_memory()
    sl_h = ls.sl.cpu().pin_memory()
    out_h = torch.empty(ls.out.shape, dtype=ls.out.dtype).pin_memory()
    stream = torch.cuda.Stream()

    def one(r):
        # the block table is host memory written only by the host: early start stays valid
        kvq.decode(ls.caches[r], plan, q_h, bt_h, sl_h, out_h, ls.wl.sm_scale, early_start=True)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for r in range(ls.R):
            one(r)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for r in range(ls.R):
            one(r)
    reps = max(1, math.ceil(min(steps, 4000) / ls.R))
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(warmup / ls.R))):
            g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / (reps * ls.R)
    h2d = q_h.numel() * q_h.element_size() + bt_h.numel() * 4 + sl_h.numel() * 4
    d2h = out_h.numel() * out_h.element_size()
    return t, h2d, d2h


def time_e2e_eager(ls, plan, seconds=0.3):
    """The e2e step without a graph: the public API called from the host for
    every step (pinned host buffers as in time_e2e); seconds per step."""
    import torch

    import quantized_paged_kv_gb300 as kvq

    q_h = ls.q.cpu().pin_memory()
    bt_h = ls.bt.cpu().pin_memory()
    sl_h = ls.sl.cpu().pin_memory()
    out_h = torch.empty(ls.out.shape, dtype=ls.out.dtype).pin_memory()
    stream = torch.cuda.Stream()

    def run(n):
        with torch.cuda.stream(stream):
            for i in range(n):
                kvq.decode(ls.caches[i % ls.R], plan, q_h, bt_h, sl_h, out_h, ls.wl.sm_scale, early_start=True,
                           stream=stream)

    run(ls.R)  # warm-up
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(ls.R)
    e1.record(stream)
    stream.synchronize()
    n = max(ls.R, int(seconds / max(e0.elapsed_time(e1) * 1e-3 / ls.R, 1e-7)))
    e0.record(stream)
    run(n)
    e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / n


def layers_for(bytes_per_layer, l2_bytes, floor=8):
    return max(floor, math.ceil(4 * l2_bytes / max(bytes_per_layer, 1)))


# The oracle's timed sample: one (sequence, KV head) unit a worker process, its
# context truncated to at most this many tokens (the oracle's work per token is
# the same at any length), decoded over and over; for the append, the new
# tokens of one KV head quantized over and over.
ORACLE_CAP_TOKENS = 8192
ORACLE_CONFIGS = (("tiny_int8", "int8", "decode"), ("long_int8", "int8", "decode"),
                  ("serving_int8", "int8", "decode"), ("append_int8", "int8", "decode"),
                  ("append_int8", "int8", "append"), ("long_nvfp4", "nvfp4", "decode"))

_ORACLE_WORKER = """
import json, sys, time
sys.path.insert(0, ROOT)
import numpy as np
from oracle import attention as oatt, layout as olay
from quantized_paged_kv_gb300 import workloads as W
idx, cap = int(sys.argv[1]), int(sys.argv[2])

def sample(name, fmt, mode):
    base = W.make(name)
    b = idx % base.B
    h = (idx // base.B) % base.Hkv
    L = base.append_tail if mode == "append" else min(int(base.seq_lens[b]), cap)
    wl = W.make(name, lens=("list", [L]), seed=base.seed + 1000 * b)
    k, v = wl.kv(0)
    k, v = k[:, h, :], v[:, h, :]
    gs = 1.0
    if fmt == "nvfp4":
        gs = float(np.float32(2688.0) / np.float32(max(np.abs(k).max(), np.abs(v).max())))
    if mode == "append":
        def work():
            oatt.quantize_rows(fmt, k, gs)
            oatt.quantize_rows(fmt, v, gs)
        return L, work
    P = (L + 15) // 16
    row = {"int8": wl.D, "nvfp4": wl.D // 2}[fmt]
    sshape = (P, 1, 16) if fmt == "int8" else (P, 1, 16, wl.D // 16)
    sdt = np.float32 if fmt == "int8" else np.uint8
    pools = {"k_global_scale": gs, "v_global_scale": gs}
    for nm, x in (("k", k), ("v", v)):
        c = np.zeros((P, 1, 16, row), np.uint8)
        sc = np.zeros(sshape, sdt)
        cc, ss = oatt.quantize_rows(fmt, x, gs)
        olay.scatter_rows(c, np.arange(L), 0, cc)
        olay.scatter_rows(sc, np.arange(L), 0, ss)
        pools[nm + "_codes"], pools[nm + "_scales"] = c, sc
    q = wl.q()[:, h * wl.G:(h + 1) * wl.G]
    bt = np.arange(P, dtype=np.int32)[None]
    lens = np.array([L])
    def work():
        oatt.paged_decode(fmt, pools, q, bt, lens, wl.sm_scale)
    return L, work

for line in sys.stdin:  # commands: "<workload> <fmt> <mode> <seconds>", then "go"
    name, fmt, mode, seconds = line.split()
    L, work = sample(name, fmt, mode)
    work()
    sys.stdout.write("ready\\n"); sys.stdout.flush()
    sys.stdin.readline()
    t0 = time.perf_counter(); n = 0
    while time.perf_counter() - t0 < float(seconds):
        work(); n += 1
    dt = time.perf_counter() - t0
    sys.stdout.write(json.dumps({"token_heads_per_s": n * L / dt, "units": n, "tokens": L}) + "\\n")
    sys.stdout.flush()
"""


class _OracleWorkers:
    """Single-threaded oracle worker processes (one per core), reused for every
    workload; rates(n, ...) times a sample on the first n of them at once."""

    def __init__(self, count):
        code = _ORACLE_WORKER.replace("sys.path.insert(0, ROOT)", f"sys.path.insert(0, {ROOT!r})")
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                   CUDA_VISIBLE_DEVICES="")
        self.procs = [subprocess.Popen([sys.executable, "-c", code, str(i), str(ORACLE_CAP_TOKENS)],
                                       stdin=subprocess.PIPE, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                       text=True, env=env) for i in range(count)]

    def _line(self, pr):
        ln = pr.stdout.readline()
        if not ln:
            pr.wait(timeout=60)
            raise RuntimeError(pr.stderr.read()[-300:])
        return ln.strip()

    def rates(self, n, name, fmt, mode, seconds):
        sel = self.procs[:n]
        for pr in sel:
            pr.stdin.write(f"{name} {fmt} {mode} {seconds}\n")
            pr.stdin.flush()
        for pr in sel:  # every worker has built its sample: start them together
            if self._line(pr) != "ready":
                raise RuntimeError("oracle worker out of step")
        for pr in sel:
            pr.stdin.write("go\n")
            pr.stdin.flush()
        return [json.loads(self._line(pr)) for pr in sel]

    def close(self):
        for pr in self.procs:
            try:
                pr.stdin.close()
                pr.wait(timeout=30)
            except Exception:  # noqa: BLE001
                pr.kill()


def cpu_baseline(seconds=2.0):
    """The oracle timed on the host's cores, per workload: one single-threaded
    worker process per core at once (all cores), then one worker alone (one
    core).  Each worker times a bounded sample (ORACLE_CAP_TOKENS above) and
    reports token-heads per second; the call time of a workload is its
    token-heads over that rate (the sum of the workers' rates for all cores)."""
    import quantized_paged_kv_gb300 as kvq
    from quantized_paged_kv_gb300 import workloads as W

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    configs = {}
    workers = _OracleWorkers(cores)
    try:
        for name, fmt, mode in ORACLE_CONFIGS:
            wl = W.make(name)
            if mode == "append":
                token_heads = wl.append_tail * wl.B * wl.Hkv
                nbytes = token_heads * 4 * wl.D + wl.append_tail * wl.B * kvq.kvq_bytes_per_token(fmt, wl.Hkv, wl.D)
            else:
                token_heads = int(wl.seq_lens.sum()) * wl.Hkv
                nbytes = int(wl.seq_lens.sum()) * kvq.kvq_bytes_per_token(fmt, wl.Hkv, wl.D)
            r_all = sum(r["token_heads_per_s"] for r in workers.rates(cores, name, fmt, mode, seconds))
            r_one = workers.rates(1, name, fmt, mode, seconds)[0]["token_heads_per_s"]
            t_all, t_one = token_heads / r_all, token_heads / r_one
            configs[f"{name}/{fmt}/{mode}"] = {
                "us_per_call_all_cores": round(t_all * 1e6, 1), "us_per_call_1_core": round(t_one * 1e6, 1),
                "GBps_all_cores": round(nbytes / t_all / 1e9, 4), "GBps_1_core": round(nbytes / t_one / 1e9, 4),
                "token_heads_per_call": token_heads, "bytes_per_call": nbytes}
    except Exception as e:  # noqa: BLE001
        return {"value": None, "unit": UNIT, "cores": cores, "kind": "oracle", "error": str(e)[-300:],
                "configs": configs}
    finally:
        workers.close()
    head = configs[f"{WORKLOAD}/int8/decode"]
    return {"value": head["GBps_all_cores"], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"float64 numpy oracle, {cores} single-threaded worker processes at once (and one alone); "
                      f"each times one (sequence, KV head) unit of the workload, its context cut to at most "
                      f"{ORACLE_CAP_TOKENS} tokens, decoded over and over for {seconds:.0f} s (the append: that "
                      f"head's new tokens quantized); call time = the workload's token-heads / the measured rate",
            "per_core_value": head["GBps_1_core"], "us_per_step_equiv": head["us_per_call_all_cores"],
            "configs": configs}


def run_ours(args, rank, world, barrier, allmax):
    import torch

    import quantized_paged_kv_gb300 as kvq
    from quantized_paged_kv_gb300 import workloads as W

    kvq.lib()  # fails loudly if the CUDA library is missing
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)
    peaks, peak_kind = measured_peaks()

    # the job at N ranks is N independent problems of the workload, sharded by
    # sequence (one per rank here); problem 0 is the workload itself
    from quantized_paged_kv_gb300.dist import problem_seed, shard_sequences

    base = W.make(WORKLOAD)
    mine = shard_sequences([base.total_tokens] * world, world)[rank]
    wl = W.make(WORKLOAD, seed=problem_seed(base.seed, int(mine[0])))
    per_layer = int(wl.seq_lens.sum()) * kvq.kvq_bytes_per_token("int8", wl.Hkv, wl.D)
    R = layers_for(per_layer, l2, floor=16)
    ls = LayerSet(wl, "int8", R, dev)
    plan = ls.plan(0)
    sampler = ClockSampler(local) if rank == 0 and not args.no_clocks else None
    t_call, calls, clocks = time_graph(ls, plan, args.steps, args.warmup, barrier=barrier, sampler=sampler,
                                       min_seconds=args.min_seconds)
    t_call = allmax(t_call)
    if clocks is not None:
        clocks["window"] = f"sampled every 20 ms during the timed region ({calls * t_call:.2f} s)"
    t_dec, _, _ = time_graph(ls, plan, args.steps, args.warmup, skip_merge=True)
    t_dec = allmax(t_dec)
    e2e_t, h2d, d2h = time_e2e(ls, plan, args.steps, args.warmup)
    e2e_t = allmax(e2e_t)
    e2e_eager_t = allmax(time_e2e_eager(ls, plan, seconds=0.3 if args.min_seconds > 0 else 0.0))

    bytes_step = ls.kv_bytes()
    value = world * bytes_step / t_call / 1e9
    achieved = bytes_step / t_dec / 1e9
    peak = float(peaks["hbm_gbs"])
    tr = traffic_record(WORKLOAD)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": calls,
        "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": t_call * 1e3, "us_per_step": round(t_call * 1e6, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded N(0,1) K/V with 4 outlier channels x8, quantized by kvq_quant_append)",
        "config": {"workload": HEADLINE_WORKLOAD,
                   "split_plan": f"auto: {plan.total_splits} splits", "layers_rotated": R,
                   "l2": f"inputs larger than L2: {R} layer pools x {per_layer / 1e6:.1f} MB visited round-robin",
                   "timing": f"CUDA graph of R consecutive calls (decode + merge), replayed for at least "
                             f"{args.min_seconds:.1f} s (every call counted in steps), CUDA events",
                   "parallelism": f"dp{world}: one independent problem per rank, no data-path collective", "kv_bytes_per_step": bytes_step,
                   "us_per_16_layer_step": round(16 * t_call * 1e6, 2)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": "decode_kernel<INT8, 256, P' hi+lo>", "kernel_us": round(t_dec * 1e6, 3),
                     "frac_of_8TBs_nominal": round(achieved / 8000.0, 4),
                     "traffic": (tr["dram_bytes_per_launch"] if tr else None),
                     "traffic_algorithmic_ratio": (round(tr["dram_bytes_per_launch"] / bytes_step, 4) if tr else None)},
        "e2e": {"value": round(world * bytes_step / e2e_t / 1e9, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": round(e2e_t * 1e6, 3),
                "how": "public API per step with pinned host buffers for q, block table, seq_lens and out, read and "
                       "written by the kernels over NVLink-C2C (no separate copy); R steps in one CUDA graph, "
                       "CUDA events",
                "eager": {"value": round(world * bytes_step / e2e_eager_t / 1e9, 1), "unit": UNIT,
                          "us_per_step": round(e2e_eager_t * 1e6, 3),
                          "how": "the same public call made from the host every step, no graph: argument checks, "
                                 "two tensor-map encodes and the pointer queries run on the host each call"}},
        "gpu_launches": calls * (2 if plan.total_splits > wl.B else 1),
        "clocks": clocks,
    }
    if args.sweep and rank == 0:
        line["sweep"] = sweep(args, dev, l2, peak, float(peaks.get("bf16_tflops", 1900.0)))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    return line


def time_protocol(dev, l2, peak):
    """The timing protocol's controls on the 32K batch-1 workload: a read-only
    stream reference (torch's sum over 4 GiB, the read side of the copy peak),
    the distribution of single graph replays (median and min per call), an
    A-vs-A noise control (two identical graphs timed in alternation), INT8 and
    BF16 caches timed in alternating order, and eager (ungraphed) calls."""
    import statistics

    import torch

    import quantized_paged_kv_gb300 as kvq
    from quantized_paged_kv_gb300 import workloads as W

    res = {}
    buf = torch.ones(2**30, dtype=torch.float32, device=dev)  # 4 GiB, far above L2
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        buf.sum()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e-3)
    res["read_only_stream"] = {"GBps": round(buf.numel() * 4 / best / 1e9, 1), "how": "torch sum over 4 GiB fp32, best of 10"}
    del buf
    torch.cuda.empty_cache()

    wl = W.make("long_int8")
    per_layer = {f: int(wl.seq_lens.sum()) * kvq.kvq_bytes_per_token(f, wl.Hkv, wl.D) for f in ("int8", "bf16")}
    sets = {f: LayerSet(wl, f, layers_for(per_layer[f], l2, floor=2), dev) for f in ("int8", "bf16")}
    stream = torch.cuda.Stream()

    def graph_of(ls):
        plan = ls.plan(0)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for r in range(ls.R):
                ls.call(r, plan)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(ls.R):
                ls.call(r, plan)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        stream.synchronize()
        return g, plan

    def replay_us(g, R):  # one replay, microseconds per call
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) * 1e3 / R

    ls = sets["int8"]
    ga, plan = graph_of(ls)
    gb, _ = graph_of(ls)
    a, b = [], []
    for _ in range(30):  # A and A' alternate
        a.append(replay_us(ga, ls.R))
        b.append(replay_us(gb, ls.R))
    res["replays_long_int8"] = {"median_us": round(statistics.median(a), 3), "min_us": round(min(a), 3),
                                "max_us": round(max(a), 3), "replays": len(a), "calls_per_replay": ls.R}
    res["a_vs_a_long_int8"] = {"median_us_a": round(statistics.median(a), 3), "median_us_a2": round(statistics.median(b), 3),
                               "rel_diff": round(statistics.median(b) / statistics.median(a) - 1, 4)}
    gf = {"int8": ga, "bf16": graph_of(sets["bf16"])[0]}
    t = {"int8": [], "bf16": []}
    for i in range(20):  # alternating format order: int8, bf16, bf16, int8, ...
        order = ("int8", "bf16") if i % 2 == 0 else ("bf16", "int8")
        for f in order:
            t[f].append(replay_us(gf[f], sets[f].R))
    res["paired_formats_long"] = {f: {"median_us": round(statistics.median(v), 3),
                                      "GBps": round(per_layer[f] / (statistics.median(v) * 1e-6) / 1e9, 1)}
                                  for f, v in t.items()}
    torch.cuda.synchronize()  # eager calls: one launch sequence per call, no graph
    with torch.cuda.stream(stream):
        for r in range(ls.R):
            ls.call(r, plan)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = 0
        for _ in range(5):
            for r in range(ls.R):
                ls.call(r, plan)
                n += 1
        e1.record(stream)
    stream.synchronize()
    res["eager_long_int8"] = {"us": round(e0.elapsed_time(e1) * 1e3 / n, 3), "calls": n}
    del sets, ga, gb, gf
    return res


def sweep(args, dev, l2, peak, peak_tf=1937.0):
    """Split sweep and the other workloads (per-call µs and KV GB/s)."""
    import gc

    import torch

    import quantized_paged_kv_gb300 as kvq
    from quantized_paged_kv_gb300 import workloads as W

    res = {}
    steps = max(64, min(args.steps, 1000))

    def measure(wl, fmt, splits, gs=(1.0, 1.0), tag=None):
        per_layer = int(wl.seq_lens.sum()) * kvq.kvq_bytes_per_token(fmt, wl.Hkv, wl.D)
        R = layers_for(per_layer, l2, floor=2)
        ls = LayerSet(wl, fmt, R, dev, gs)
        for sp in splits:
            plan = ls.plan(sp)
            t, _, _ = time_graph(ls, plan, steps, 16)
            td, _, _ = time_graph(ls, plan, steps, 16, skip_merge=True)
            key = f"{tag or wl.name}/{fmt}/split={'auto' if sp == 0 else sp}"
            res[key] = {"us": round(t * 1e6, 3), "GBps": round(per_layer / t / 1e9, 1),
                        "frac": round(per_layer / t / 1e9 / peak, 4), "decode_kernel_us": round(td * 1e6, 3),
                        "splits": plan.total_splits, "layers": R}
        del ls
        gc.collect()
        torch.cuda.empty_cache()

    def tensor_gs(wl):  # the NVFP4 per-tensor global scales 448 * 6 / amax of K and of V
        ka, va = wl.tensor_amax()
        return (float(np.float32(2688.0) / np.float32(ka)), float(np.float32(2688.0) / np.float32(va)))

    wl = W.make("tiny_int8")
    measure(wl, "int8", (1, 4, 0))
    wl = W.make("long_int8")
    measure(wl, "int8", (1, 2, 4, 8, 16, 32, 38, 64, 0))
    measure(wl, "bf16", (16, 38, 64, 0))
    measure(wl, "int8_g32", (0,))  # INT8 with one scale per 32 values
    measure(wl, "nvfp4", (0,), tensor_gs(wl))  # the same workload in NVFP4
    wl = W.make("serving_int8")
    measure(wl, "int8", (0, 1))
    measure(wl, "int8_g32", (0,))
    measure(wl, "nvfp4", (0,), tensor_gs(wl))
    # the decode that follows the append workload's append: B = 8, contexts 4K..16K
    wl = W.make("append_int8")
    measure(wl, "int8", (0,))
    wl = W.make("long_nvfp4")
    measure(wl, "nvfp4", (0,), tensor_gs(wl))
    measure(wl, "nvfp4", (0,), (1.0, 1.0), tag="long_nvfp4(gs=1)")
    measure(wl, "int8", (0,))
    measure(wl, "bf16", (0,))
    # verify step: 6 query tokens a sequence over the 32K context (the pages' verify shape)
    wl = W.make("long_int8")
    per_layer = int(wl.seq_lens.sum()) * kvq.kvq_bytes_per_token("int8", wl.Hkv, wl.D)
    R = layers_for(per_layer, l2, floor=2)
    ls = LayerSet(wl, "int8", R, dev)
    for T in (2, 4, 6, 8):  # from 4 tokens a one-sequence call runs on the tensor-core kernel
        res[f"verify_long_int8/T={T}"] = time_verify(ls, T, steps)
    del ls
    gc.collect()
    torch.cuda.empty_cache()
    per_layer = int(wl.seq_lens.sum()) * kvq.kvq_bytes_per_token("nvfp4", wl.Hkv, wl.D)
    ls = LayerSet(wl, "nvfp4", layers_for(per_layer, l2, floor=2), dev, tensor_gs(wl))
    for T in (2, 3, 6):  # NVFP4 from 3 tokens
        res[f"verify_long_int8(nvfp4)/T={T}"] = time_verify(ls, T, steps)
    del ls
    gc.collect()
    torch.cuda.empty_cache()
    # a batch: the 8 sequences of 4K..16K of the append workload, 4 and 6 tokens a
    # sequence (the batch takes the tensor-core route from 6)
    wl = W.make("append_int8")
    per_layer = int(wl.seq_lens.sum()) * kvq.kvq_bytes_per_token("int8", wl.Hkv, wl.D)
    ls = LayerSet(wl, "int8", layers_for(per_layer, l2, floor=2), dev)
    for T in (4, 6, 8):
        res[f"verify_append_int8/T={T}"] = time_verify(ls, T, steps)
    del ls
    gc.collect()
    torch.cuda.empty_cache()
    # prefill: a 2,048-token chunk at the end of the 32K context (and the first chunk)
    wl = W.make("long_int8")
    for fmt, Ts in (("int8", (512, 2048)), ("nvfp4", (2048,))):
        ls = LayerSet(wl, fmt, 2, dev)
        for T in Ts:
            res[f"prefill_long_{fmt}/T={T}"] = time_prefill(ls, T, peak_tf=peak_tf)
        del ls
        gc.collect()
        torch.cuda.empty_cache()
    res.update(time_rotation(dev, l2, peak))
    gc.collect()
    torch.cuda.empty_cache()
    res.update(time_protocol(dev, l2, peak))
    gc.collect()
    torch.cuda.empty_cache()
    # quantize-and-append of 8192 tokens (the last 1024 of 8 sequences), INT8 (per row
    # and per 32 values) and NVFP4
    wl = W.make("append_int8")
    for fmt in ("int8", "int8_g32", "nvfp4"):
        res[f"append_{fmt}/8192 tokens"] = time_append(wl, fmt, dev, l2, steps)
        gc.collect()
        torch.cuda.empty_cache()
    # the same appends with the rows rotated first: in the append, or by a separate call
    for fmt in ("int8", "nvfp4"):
        for mode in ("fused", "two_call"):
            res[f"append_{fmt}_rotated_{mode}/8192 tokens"] = time_append(wl, fmt, dev, l2, steps, rotate=mode)
            gc.collect()
            torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The float64 CPU oracle timed on the host: each step decodes KV head (step % 4)
    of the 32,768-token sequence (one quarter of one step of our workload)."""
    import time as _t

    from oracle import attention as oatt
    from oracle import layout as olay
    from quantized_paged_kv_gb300 import workloads as W

    wl = W.make(WORKLOAD)
    k, v = wl.kv(0)
    slots = wl.slots(0)
    pools = {}
    for name, x in (("k", k), ("v", v)):
        c = np.zeros((wl.num_pages, wl.Hkv, 16, wl.D), np.uint8)
        s = np.zeros((wl.num_pages, wl.Hkv, 16), np.float32)
        for h in range(wl.Hkv):
            cc, ss = oatt.quantize_rows("int8", x[:, h, :])
            olay.scatter_rows(c, slots, h, cc)
            olay.scatter_rows(s, slots, h, ss)
        pools[name + "_codes"], pools[name + "_scales"] = c, s
    q = wl.q()
    steps = max(1, min(args.steps, 40))
    warm = max(1, min(args.warmup, 40))
    for i in range(warm):
        oatt.paged_decode("int8", pools, q, wl.block_tables, wl.seq_lens, wl.sm_scale, heads=[(0, i % 4)])
    t0 = _t.perf_counter()
    for i in range(steps):
        oatt.paged_decode("int8", pools, q, wl.block_tables, wl.seq_lens, wl.sm_scale, heads=[(0, i % 4)])
    dt = (_t.perf_counter() - t0) / steps
    nbytes = int(wl.seq_lens.sum()) * 2 * (wl.D + 4)  # one KV head
    value = nbytes / dt / 1e9
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded workload)",
        "config": {"workload": HEADLINE_WORKLOAD},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"float64 numpy oracle; each step decodes one KV head (6 query heads) of the "
                                   f"32,768-token sequence, a quarter of the workload's step, and GB/s counts that "
                                   f"head's bytes; BLAS may use up to {cores} threads"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_ncu_case(args):
    """A small, untimed case for ncu: pools of one workload just over the L2 size
    in total, then `calls` decode calls (decode + merge) visiting them in turn."""
    import torch

    import quantized_paged_kv_gb300 as kvq
    from quantized_paged_kv_gb300 import workloads as W

    kvq.lib()
    wl = W.make(args.ncu_case)
    if wl.append_tail:  # the workload's append: `calls` appends of its new tokens into one pool
        ks, vs, ss = [], [], []
        for b in range(wl.B):
            k, v = W.device_kv(wl, b, device="cuda")
            ks.append(k[-wl.append_tail:])
            vs.append(v[-wl.append_tail:])
            ss.append(torch.from_numpy(wl.slots(b)[-wl.append_tail:]))
        k, v, s = torch.cat(ks), torch.cat(vs), torch.cat(ss).cuda()
        cache = kvq.KVCache(args.fmt, wl.num_pages, wl.Hkv, wl.D, device="cuda", fill=0)
        for _ in range(args.calls):
            cache.append(k, v, s)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": args.ncu_case, "fmt": args.fmt, "calls": args.calls,
                          "tokens": int(k.shape[0])}), flush=True)
        return
    props = torch.cuda.get_device_properties(0)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)
    per_layer = int(wl.seq_lens.sum()) * kvq.kvq_bytes_per_token(args.fmt, wl.Hkv, wl.D)
    R = max(1, math.ceil(1.1 * l2 / max(per_layer, 1)))
    ls = LayerSet(wl, args.fmt, R, "cuda")  # NVFP4 global scale 1 (it does not change the work)
    plan = ls.plan(0)
    if args.prefill_tokens:
        T = args.prefill_tokens
        L = int(wl.seq_lens[0])
        q = torch.from_numpy(wl.q_tokens(T)[0]).to(torch.bfloat16).cuda()
        out = torch.empty((T, wl.Hq, wl.D), dtype=ls.out.dtype, device="cuda")
        ws = None
        for i in range(args.calls):
            ws = kvq.prefill(ls.caches[i % R], q, ls.bt[0].contiguous(), L, out, wl.sm_scale, workspace=ws)
    elif args.verify_tokens:
        T = args.verify_tokens
        plan = kvq.DecodePlan(ls.caches[0], wl.seq_lens, wl.Hq, q_len=T)
        q = torch.from_numpy(wl.q_tokens(T)).to(torch.bfloat16).cuda()
        out = torch.empty((wl.B, T, wl.Hq, wl.D), dtype=ls.out.dtype, device="cuda")
        for i in range(args.calls):
            kvq.verify(ls.caches[i % R], plan, q, ls.bt, ls.sl, out, wl.sm_scale)
    else:
        for i in range(args.calls):
            ls.call(i % R, plan)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": args.ncu_case, "fmt": args.fmt, "layers": R, "calls": args.calls,
                      "total_splits": plan.total_splits, "num_ctas": plan.num_ctas,
                      "kv_bytes_per_call": ls.kv_bytes()}), flush=True)


def main():
    args = parse()
    if args.ncu_case:
        run_ncu_case(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    from quantized_paged_kv_gb300.dist import RankGroup

    if world > 1:
        import torch

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    group = RankGroup.from_env("nccl")
    try:
        line = run_ours(args, rank, world, group.barrier, group.allmax)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        group.close()


if __name__ == "__main__":
    main()
