"""Host-side arithmetic of bench.py: the per-pass roofline entry, the
algorithmic work of a step, and the DRAM-traffic record lookup (which must
drop the figure once the kernel sources differ from those it was taken on)."""
import json
import os

import numpy as np

import bench
import medusa_synth as ms

PK = {"hbm": 6000.0, "bf16": 1800.0, "bf16_sustained": 1500.0, "src": "test"}


def test_roofline_entry_picks_the_binding_resource():
    # 1.2 GB and no flops in 0.5 ms: HBM-bound at 2.4 TB/s
    e = bench.roofline_entry({"bytes": 1.2e9, "flops": 0.0}, 0.5e-3, PK)
    assert e["bound"] == "hbm" and e["unit"] == "GB/s"
    assert abs(e["achieved"] - 2400.0) < 1e-6
    assert abs(e["frac"] - 0.4) < 1e-12
    assert abs(e["hbm_frac_nominal"] - 2400.0 / bench.NOMINAL_HBM_GBS) < 1e-12
    # 3 TFLOP over 10 MB in 4 ms: tensor-bound at 750 TFLOP/s
    e = bench.roofline_entry({"bytes": 1e7, "flops": 3e12}, 4e-3, PK)
    assert e["bound"] == "tensor" and e["unit"] == "TFLOP/s"
    assert abs(e["achieved"] - 750.0) < 1e-9
    assert abs(e["frac"] - 0.5) < 1e-12
    assert abs(e["tensor_frac_nominal"] - 750.0 / bench.NOMINAL_BF16_TFLOPS) < 1e-12


def test_pass_work_of_the_batch1_step():
    """The LM head, the head weights and the attention weights of the
    Vicuna-7B-shaped batch-1 workload, counted by hand."""
    w = ms.workload("vicuna7b-b1")
    N = 89
    P = np.array([2048], np.int64)
    work = bench.pass_work(w, N, P)
    lm = 32000 * 4096 * 2
    heads_w = 4 * 4096 * 4096 * 2
    assert work["lm_verify"]["bytes"] == lm + N * 4096 * 2 + N * 24
    assert work["lm_verify"]["flops"] == 2 * N * 4096 * 32000
    assert work["medusa_heads"]["bytes"] >= heads_w + lm
    qkv = (32 + 2 * 32) * 128 * 4096 * 2
    wo = 4096 * 32 * 128 * 2
    kv = 2048 * 32 * 128 * 2 * 2
    # plus the gathered embedding rows, the tree rows' K and V written to
    # the cache, and y
    rows = N * 4096 * 2 + N * 32 * 128 * 2 * 2 + N * 4096 * 2
    assert work["tree_attention"]["bytes"] == qkv + wo + kv + rows


def test_profiled_traffic_follows_the_sources(tmp_path, monkeypatch):
    rec = {"workload": "w", "call": "c", "sources": ["tree.cu"],
           "sources_sha256": bench.source_hash("tree.cu"), "dram_bytes_per_launch": 1234}
    p = tmp_path / "t.json"
    p.write_text(json.dumps({"records": [rec]}))
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(p))
    assert bench.profiled_traffic("w", "c") == 1234
    assert bench.profiled_traffic("w", "other") is None
    rec["sources_sha256"] = "0" * 64          # taken on other sources
    p.write_text(json.dumps({"records": [rec]}))
    assert bench.profiled_traffic("w", "c") is None
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(tmp_path / "missing.json"))
    assert bench.profiled_traffic("w", "c") is None


def test_committed_traffic_record():
    """The committed record names the dominant call of the headline workload
    and the kernel sources it was taken on; bench.py reports it exactly while
    those sources are unchanged, and nothing once they differ."""
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")) as f:
        recs = json.load(f)["records"]
    r = [x for x in recs if x["workload"] == bench.HEADLINE and x["call"] == "lm_verify"]
    assert len(r) == 1
    r = r[0]
    assert r["dram_bytes_per_launch"] > 0 and len(r["sources_sha256"]) == 64
    same = bench.source_hash(*r["sources"]) == r["sources_sha256"]
    want = r["dram_bytes_per_launch"] if same else None
    assert bench.profiled_traffic(bench.HEADLINE, "lm_verify") == want


def _reference_run(env_extra):
    import subprocess
    import sys
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl",
                           "reference", "--workload", "tiny-fp32", "--steps", "3", "--warmup", "3"],
                          capture_output=True, text=True, timeout=300, env=env, cwd=bench.ROOT)


def test_reference_arm_line():
    """The oracle arm prints one JSON line with the contract's keys: the same
    metric and unit as the GPU arm, its own timing counts, a cpu_baseline
    describing the run and an e2e entry with no host-device copies."""
    p = _reference_run({"RANK": "0"})
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC and j["unit"] == "steps/s"
    assert j["value"] > 0 and j["higher_is_better"] is True and j["n_gpus"] == 1
    assert 1 <= j["steps"] <= 3 and 0 <= j["warmup"] <= 3
    assert j["config"]["workload"] == "tiny-fp32"
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1
    assert "oracle step" in cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": "steps/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    p = _reference_run({"RANK": "1"})
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
