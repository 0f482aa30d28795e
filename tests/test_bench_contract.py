"""CPU checks of what the bench reports: the algorithmic byte counts that are
the numerator of its GB/s and roofline figures (worked by hand for the tiny
workload, and the canonical workload's figure that the committed profiles
quote), and the JSON line of the reference arm, which times the FP64 oracle
on the host (rank 0 only under a multi-rank launch)."""
import json
import math
import os
import subprocess
import sys

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_bytes_tiny_by_hand():
    # tiny: contexts 17 and 40, 4 query / 2 KV heads, head_dim 64
    kv = (17 + 40) * 2 * (2 * 64 + 4)          # codes of K and V + two FP16 scales
    tables = (math.ceil(17 / 16) + math.ceil(40 / 16)) * 4
    q_out = 2 * 4 * 64 * 2 * 2                  # q read and out written, 16-bit
    lens = 2 * 4
    w = W.make("tiny")
    assert w.decode_bytes_int8() == kv + tables + q_out + lens == 17124
    assert w.decode_bytes_kv16() == (17 + 40) * 2 * 4 * 64 + tables + q_out + lens


def test_canonical_decode_bytes_match_the_profiles():
    assert W.make("canonical").decode_bytes_int8() == 78463136


def _bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=600, env=e)
    return r


def test_reference_arm_line():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"].startswith("INT8-KV paged decode")
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] == 0
    assert line["config"]["workload"] == "mha"          # the headline workload
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_are_silent():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "0",
               env={"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_cpu_baseline_entry_runs_on_all_host_cores():
    import bench
    w = W.make("tiny")
    cb = bench.cpu_baseline(w, budget_s=0.5)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["cores"] == bench.host_cores()
    assert cb["single_thread_value"] > 0 and "host cores" in cb["sample"]
