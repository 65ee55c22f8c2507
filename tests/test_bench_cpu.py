"""bench.py's host-side contract on a machine without a GPU: the reference arm
(the oracle timed on the host cores) prints one JSON line with the contract's
keys, the layer count keeps the timed pools above L2, and the committed DRAM
traffic record is used only while the decode kernel's sources are unchanged."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"] == {"workload": bench.HEADLINE_WORKLOAD}  # the same config string as our arm's
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_layers_keep_the_timed_pools_above_l2():
    l2 = 126 * 2**20
    for per_layer in (1 << 20, 68_157_440, 588_000_000, 2 * 10**9):
        R = bench.layers_for(per_layer, l2, floor=2)
        assert R >= 2 and (R * per_layer >= 4 * l2 or R == 2)
        assert bench.layers_for(per_layer, l2) >= 8  # default floor


def test_traffic_record_only_for_the_current_decode_source(tmp_path, monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        committed = json.load(f)["long_int8"]
    assert 0.99 < committed["dram_bytes_per_launch"] / committed["algorithmic_bytes_per_launch"] < 1.2
    rec = bench.traffic_record("long_int8")  # None while the record is older than the decode sources
    if rec is not None:
        assert rec["kernel_sha"] == bench.kernel_sha()
    # a record taken on other sources is ignored; the same record with the current hash is used
    fake = tmp_path / "profiles"
    fake.mkdir()
    stale = dict(committed, kernel_sha="0" * 16)
    (fake / "traffic.json").write_text(json.dumps({"long_int8": stale}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "quantized_paged_kv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("decode.cuh", "kvq_ptx.cuh", "decode_launch.cu"):
        (csrc / f).write_bytes(open(os.path.join(ROOT, "quantized_paged_kv_gb300", "csrc", f), "rb").read())
    assert bench.traffic_record("long_int8") is None
    (fake / "traffic.json").write_text(json.dumps({"long_int8": dict(committed, kernel_sha=bench.kernel_sha())}))
    assert bench.traffic_record("long_int8")["dram_bytes_per_launch"] == committed["dram_bytes_per_launch"]


def test_reference_arm_honours_the_warmup_count():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "5"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["steps"] == 2 and d["warmup"] == 5


def test_oracle_workers_time_every_kind_of_sample():
    """The per-workload oracle timing: decode samples of both formats and the
    append sample, on two workers at once and on one alone."""
    w = bench._OracleWorkers(2)
    try:
        for name, fmt, mode in (("tiny_int8", "int8", "decode"), ("append_int8", "int8", "append"),
                                ("serving_int8", "int8", "decode")):
            two = w.rates(2, name, fmt, mode, 0.2)
            one = w.rates(1, name, fmt, mode, 0.2)
            assert len(two) == 2 and len(one) == 1
            for r in two + one:
                assert r["token_heads_per_s"] > 0 and r["units"] >= 1
                assert r["tokens"] <= bench.ORACLE_CAP_TOKENS
            if mode == "append":
                assert one[0]["tokens"] == 1024
    finally:
        w.close()
