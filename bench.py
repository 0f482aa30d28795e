#!/usr/bin/env python3
"""Benchmark of the INT8 paged KV-cache hot path on GB300.

One step = one layer's decode step of a workload: quantize-append of the
step's new tokens (if the workload appends), then the paged decode:

    kvq_quantize_append  ->  kvq_paged_decode

The headline line is taken on the largest workload that fits one GPU, the MHA
decode (64 sequences x 4096 tokens, 32 query = 32 KV heads, d 128, fp16,
2.18 GB of INT8 K/V per step); ``--workload`` picks another.  The same step is
timed on the native-16-bit twin (kvq_cache_append_kv16 ->
kvq_paged_decode_kv16) for the steps/s A/B, and through the C ABI with host
buffers (pinned H2D of the step's inputs and D2H of the output inside the
timed region) for the end-to-end figure.  ``configs`` repeats the INT8 and
twin timings on all five workloads (tiny, canonical, long, mha, serving).
L2 is flushed between timed steps (a 512 MB write, then a 512 MB read of
another buffer, so that the write's dirty lines are written back before the
step rather than inside it); each step is timed with CUDA events on the
launching stream.  A context sweep (2K/8K/32K, 16
sequences) compares the INT8 decode with the twin, and the chunked prefill
over the INT8 cache is timed on an 8K-token causal chunk (GQA 8).  The FP64
CPU oracle is timed on a bounded sample of the headline workload as the CPU
baseline.  K/V values are drawn on the GPU (``Workload.seq_kv_device``: the
workloads' recipe, torch's generator).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --prefill all|SHAPE [--steps K] [--warmup W]   # prefill lines only

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload (the path needs no exchange between GPUs).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "INT8-KV paged decode HBM GB/s (% of GB300 peak); decode steps/s vs BF16 KV"
UNIT = "GB/s"
FLUSH_BYTES = 512 << 20


def make_flush(torch, dev):
    """The L2 flush between timed steps: write a buffer four times the L2,
    then read another as large.  The write alone would leave the L2 full of
    dirty lines whose write-back then lands inside the next timed kernel;
    after the read the L2 holds clean lines of neither the workload nor the
    write."""
    wbuf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush():
        wbuf.zero_()
        rbuf.max()
    return flush
FALLBACK_HBM_GBS = 6800.0
# the kernels whose DRAM traffic the committed ncu summaries measured
DECODE_SOURCES = ("kvq_decode.cuh", "kvq_decode_int8.cu", "kvq_decode_int8_h2.cu",
                  "kvq_decode_int8_t2.cu", "kvq_ptx.cuh", "kvq_combine.cu", "kvq_api.cu")
HEADLINE = "mha"


def traffic_file(workload: str) -> str:
    return os.path.join(ROOT, "profiles", f"decode_int8_{workload}.traffic.txt")


# chunked-prefill shapes: (sequences, context L, chunk n = queries at the end
# of each sequence, query heads, KV heads); head_dim 128, bf16 activations
PREFILL_SHAPES = {
    "8k_full_gqa8": (1, 8192, 8192, 64, 8),
    "4k_chunk1k_gqa4": (4, 4096, 1024, 32, 8),
    "2k_chunk512_gqa4": (16, 2048, 512, 32, 8),
    "4k_full_mha": (2, 4096, 4096, 32, 32),
    "2k_full_gqa8": (1, 2048, 2048, 64, 8),
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=list(W.NAMES))
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload timings of all five workloads")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--settle", type=float, default=1.5,
                    help="seconds of untimed steps before the timed region (clock sampling)")
    ap.add_argument("--prefill", default=None, choices=["all"] + list(PREFILL_SHAPES),
                    help="chunked-prefill timing instead of the decode bench line: one JSON "
                         "line per shape (causal attention TFLOP/s against the tensor peak)")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--profile-g", type=int, default=0,
                    help="with --profile-arm: the group-size sweep's workload for G "
                         "(32 sequences x 4096 tokens, 8 KV heads, 8G query heads)")
    ap.add_argument("--no-g-sweep", action="store_true")
    ap.add_argument("--profile-seqs", type=int, default=0,
                    help="with --profile-arm: only the workload's first N sequences")
    ap.add_argument("--profile-arm", choices=["int8", "kv16", "int8cc", "append"], default=None,
                    help="profiling run: only this decode arm (one cache on the device), "
                         "or the step's INT8 quantize-append (append), warm-up + steps with "
                         "L2 flushes, a short timing line; no bench line")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(pg, device, xs):
    """Per-rank values -> their maximum over the ranks of `pg` (one
    all-reduce; unchanged without a process group).  The bench reports the
    slowest rank's time for every arm."""
    vals = [float(x) for x in xs]
    if pg is None:
        return vals
    import torch
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world: int, bytes_per_rank_step: float, step_ms: float) -> float:
    """Whole-job GB/s of `world` independent replicas, each moving
    `bytes_per_rank_step` per step, over the slowest rank's step time
    (weak scaling: the per-GPU work is fixed as the job grows)."""
    return world * bytes_per_rank_step / (step_ms * 1e-3) / 1e9


def decode_source_hash() -> str:
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, "int8_quantized_paged_tokenwise_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def read_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary ("key: value"
    lines), or None when it was taken on other sources or another workload."""
    try:
        kv = {}
        with open(traffic_file(workload)) as f:
            for line in f:
                line = line.strip()
                if line and not line.startswith("#") and ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_hash") == decode_source_hash() and kv.get("workload") == workload:
            return int(kv["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def config_of(w: W.Workload, extra=None):
    c = {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
         "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
         "kv_dtype": "int8+fp16-scale", "act_dtype": w.dtype,
         "context_tokens": int(w.context_lens.sum()), "max_context": w.max_context_len,
         "append_tokens_per_step": w.append_tokens(), "l2": "flushed between steps: 512 MB written, then 512 MB of another buffer read"}
    if extra:
        c.update(extra)
    return c


# ------------------------------------------------------------- CPU oracle ---
def oracle_inputs(w: W.Workload, seqs):
    """The oracle's inputs for whole sequences `seqs` (numpy draws of the
    workload recipe), generated before any timing starts."""
    return [(b, w.seq_q(b)) + tuple(w.seq_kv(b)) for b in seqs]


def oracle_seq_bytes(w: W.Workload, L: int) -> int:
    """Algorithmic bytes of one sequence's step: its decode (K/V payload and
    scales of L tokens, table entries, q and out) plus, when the workload
    appends, the quantize-append of its new token."""
    n = w.decode_bytes_int8_seq(L)
    if w.append:
        n += w.num_kv_heads * (2 * 2 * w.head_dim + 2 * (w.head_dim + 2)) + 8
    return n


def oracle_run(w: W.Workload, inputs):
    """The FP64 oracle as it stands, single thread, over prepared inputs: per
    sequence the quantize-append of its step token (if the workload appends;
    into a one-page cache) and the decode of all heads (which re-quantizes
    the context from the unpaged token arrays).  Returns (bytes, seconds)."""
    import oracle
    oracle.build()
    kc = np.zeros((1, w.num_kv_heads, 16, w.head_dim), np.int8)
    vc = np.zeros_like(kc)
    ks = np.zeros((1, w.num_kv_heads, 16), np.uint16)
    vs = np.zeros_like(ks)
    nbytes, t = 0, 0.0
    for b, q, k, v in inputs:
        L = len(k)
        slot = np.array([(L - 1) % 16], np.int64)
        t0 = time.perf_counter()
        if w.append and L:
            oracle.quantize_append(k[L - 1:], v[L - 1:], w.dtype, slot, kc, vc, ks, vs, 16)
        oracle.decode_sequence(q, k, v, w.dtype, w.sm_scale)
        t += time.perf_counter() - t0
        nbytes += oracle_seq_bytes(w, L)
    return nbytes, t


def time_oracle(w: W.Workload, budget_s: float, start_seq: int = 0, max_seqs: int | None = None,
                stride: int = 1):
    """Single thread: whole sequences start_seq, start_seq + stride, ... until
    the time budget is spent (each sequence's inputs drawn before its timed
    call).  Returns (GB/s, sequences, busy seconds)."""
    nbytes, t_total, n = 0, 0.0, 0
    b = start_seq
    while (max_seqs is None or n < max_seqs) and (t_total < budget_s or n == 0):
        x, t = oracle_run(w, oracle_inputs(w, [b % w.num_seqs]))
        nbytes += x
        t_total += t
        n += 1
        b += stride
    return nbytes / t_total / 1e9, n, t_total


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_job(job):
    """Pool worker: draw the inputs of its sequences, wait for every worker at
    the barrier, then run the oracle on them.  Returns (bytes, sequences,
    start, end) with wall-clock start/end times."""
    name, seqs, barrier = job
    w = W.make(name)
    inputs = oracle_inputs(w, seqs)
    import oracle
    oracle.build()
    barrier.wait(timeout=600)
    t0 = time.time()
    nbytes, _ = oracle_run(w, inputs)
    return nbytes, len(seqs), t0, time.time()


def time_oracle_parallel(w: W.Workload, seqs_per_worker: int, workers: int, rounds: int = 1,
                         warmup_rounds: int = 1):
    """The same oracle calls on `workers` spawned host processes, disjoint
    sequences, `rounds` times: each worker draws the inputs of its
    `seqs_per_worker` sequences, all workers start together at a barrier, and
    the round's time runs from the first start to the last finish.  Returns
    per round (GB/s, sequences, wall seconds)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = []
    with ctx.Manager() as mgr, ctx.Pool(workers) as pool:
        bar = mgr.Barrier(workers)

        def jobs(r, n):
            first = r * workers * n
            return [(w.name, [(first + i * n + j) % max(w.num_seqs, 1) for j in range(n)], bar)
                    for i in range(workers)]
        limit = 600.0 + 60.0 * seqs_per_worker          # seconds a round may take
        for r in range(warmup_rounds):                # imports and library load in each worker
            pool.map_async(_oracle_job, jobs(r, 1)).get(timeout=limit)
        for r in range(rounds):
            res = pool.map_async(_oracle_job, jobs(warmup_rounds + r, seqs_per_worker)).get(
                timeout=limit)
            wall = max(x[3] for x in res) - min(x[2] for x in res)
            out.append((sum(x[0] for x in res) / wall / 1e9, sum(x[1] for x in res), wall))
    return out


def cpu_baseline(w: W.Workload, budget_s: float = 6.0) -> dict:
    """The bench line's `cpu_baseline`: the oracle as it stands on a bounded
    sample of workload `w`, on every host core (spawned processes, disjoint
    sequences, about budget_s of oracle time each, input draws outside the
    timed region), with the single-thread figure beside it; the one-core
    figure, labelled, if the process pool cannot run."""
    gbs1, n1, t1 = time_oracle(w, budget_s=budget_s)
    single = f"{n1} whole-sequence steps, {t1:.1f} s on one core"
    cores = host_cores()
    per = max(1, int(round(budget_s / (t1 / n1))))
    what = ("quantize-append of the step token + decode of all heads" if w.append
            else "decode of all heads")
    try:
        gbs, n, t = time_oracle_parallel(w, per, cores)[0]
        return {"value": round(gbs, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": f"{n} whole-sequence steps ({per} per core) over {t:.1f} s of wall "
                          f"time on {cores} host cores (spawned processes started together, "
                          f"disjoint sequences, input draws before the start) of the "
                          f"{w.name} workload ({what}), FP64",
                "single_thread_value": round(gbs1, 6), "single_thread_sample": single}
    except Exception as e:  # the process pool is unavailable: the one-core figure
        return {"value": round(gbs1, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{single} of the {w.name} workload ({what}), FP64; process pool "
                          f"failed: {type(e).__name__}"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = W.make(args.workload)
    cores = host_cores()
    how = "one per host core in spawned processes started together"
    try:
        # each step: one whole sequence per host core, all cores at once
        res = time_oracle_parallel(w, 1, cores, rounds=args.steps,
                                   warmup_rounds=max(args.warmup, 1))
    except Exception as e:  # the process pool is unavailable: one core, labelled as such
        how = f"on one core (process pool failed: {type(e).__name__})"
        cores = 1
        for i in range(args.warmup):
            time_oracle(w, 0.0, start_seq=i, max_seqs=1)
        res = [time_oracle(w, 0.0, start_seq=args.warmup + i, max_seqs=1)
               for i in range(args.steps)]
    times = [t for _, _, t in res]
    total_bytes = sum(g * t for g, _, t in res)
    value = total_bytes / sum(times)
    what = ("quantize-append of the step token + decode, all heads" if w.append
            else "decode, all heads")
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, {"sample": f"{cores} sequences per step"}),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{cores} whole sequences of the {w.name} workload per step, "
                                   f"{how} ({what}; input draws outside the timed region)"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- clocks ---
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------------- GPU ---
class GpuWorkload:
    """A workload resident in HBM: INT8 cache, 16-bit twin cache, tables, q and
    the step's new tokens (K/V drawn on the GPU), plus host copies of the
    step's inputs for the end-to-end arm."""

    def __init__(self, w: W.Workload, dev, arms=("int8", "kv16")):
        import torch
        import int8_quantized_paged_tokenwise_gb300 as kvq
        self.torch, self.kvq, self.w, self.dev = torch, kvq, w, dev
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
        self.tdt = tdt

        def up(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(tdt)

        nb, bt, _ = w.tables()
        self.int8 = kvq.alloc_int8_cache(nb, w.num_kv_heads, w.head_dim, dev) if "int8" in arms else None
        self.kv16 = (kvq.alloc_kv16_cache(nb, w.num_kv_heads, w.head_dim, tdt, dev)
                     if "kv16" in arms else None)
        ks, vs, ss = [], [], []
        for b in range(w.num_seqs):
            L = int(w.context_lens[b])
            if L == 0:
                continue
            k, v = w.seq_kv_device(b, dev)
            n = int(w.prefix_lens[b])
            if n:
                s = torch.from_numpy(w.slots(b, 0, n)).to(dev)
                if self.int8 is not None:
                    kvq.kvq_quantize_append(k[:n], v[:n], s, *self.int8)
                if self.kv16 is not None:
                    kvq.kvq_cache_append_kv16(k[:n], v[:n], s, *self.kv16)
            if w.append:
                ks.append(k[L - 1:L]); vs.append(v[L - 1:L]); ss.append(w.slots(b, L - 1, L))
        if w.prefill_tokens:
            pk, pv = w.prefill_kv_device(dev)
            ks.append(pk); vs.append(pv); ss.append(w.prefill_slots())
        self.k_new = torch.cat(ks).contiguous() if ks else None
        self.v_new = torch.cat(vs).contiguous() if vs else None
        self.slots_h = np.concatenate(ss).astype(np.int64) if ss else None
        self.slots = torch.from_numpy(self.slots_h).to(dev) if ss else None
        self.k_new_h = self.k_new.view(torch.int16).cpu().numpy() if ks else None
        self.v_new_h = self.v_new.view(torch.int16).cpu().numpy() if vs else None
        self.q_h = w.q_all()
        self.q = up(self.q_h)
        self.bt_h = bt
        self.bt = torch.from_numpy(bt).to(dev)
        self.cl_h = w.context_lens.astype(np.int32)
        self.cl = torch.from_numpy(self.cl_h).to(dev)
        self.out = torch.empty_like(self.q)
        nbytes = kvq.kvq_decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                                w.head_dim, w.max_context_len)
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.split = nbytes > 0
        torch.cuda.synchronize()

    def append_int8(self):
        if self.k_new is not None:
            self.kvq.kvq_quantize_append(self.k_new, self.v_new, self.slots, *self.int8)

    def decode_int8(self):
        w = self.w
        self.kvq.kvq_paged_decode(self.q, *self.int8, self.bt, self.cl, w.max_context_len,
                                  w.sm_scale, out=self.out, workspace=self.ws)

    def append_kv16(self):
        if self.k_new is not None:
            self.kvq.kvq_cache_append_kv16(self.k_new, self.v_new, self.slots, *self.kv16)

    def decode_int8_cuda_cores(self):
        w = self.w
        self.kvq.kvq_paged_decode_cuda_cores(self.q, *self.int8, self.bt, self.cl,
                                             w.max_context_len, w.sm_scale, out=self.out,
                                             workspace=self.ws)

    def decode_kv16(self):
        w = self.w
        self.kvq.kvq_paged_decode_kv16(self.q, *self.kv16, self.bt, self.cl, w.max_context_len,
                                       w.sm_scale, out=self.out, workspace=self.ws)

    def launches_per_step(self):
        return (1 if self.k_new is not None else 0) + 1 + (1 if self.split else 0)


def arm_summary(w: W.Workload, step_ms, dec_ms, step16_ms, dec16_ms, peak, cc_ms=None) -> dict:
    """Per-workload figures of one INT8 arm and one 16-bit-twin arm (mean
    step and decode times in ms); cc_ms: the INT8 decode on the CUDA cores."""
    dec_gbs = w.decode_bytes_int8() / (dec_ms * 1e-3) / 1e9
    return {"group_size": w.group,
            "cuda_core_decode_us": None if cc_ms is None else round(1e3 * cc_ms, 3),
            "tensor_core_speedup": None if cc_ms is None else round(cc_ms / dec_ms, 3),"decode_us": round(1e3 * dec_ms, 3), "decode_gbs": round(dec_gbs, 1),
            "decode_pct_of_measured_peak": round(100 * dec_gbs / peak, 2),
            "decode_pct_of_nominal_8tbs": round(100 * dec_gbs / 8000.0, 2),
            "decode_bytes": w.decode_bytes_int8(),
            "bytes_per_decoded_token": round(w.decode_bytes_int8() / max(w.num_seqs, 1)),
            "append_tokens_per_step": w.append_tokens(),
            "step_us": round(1e3 * step_ms, 3),
            "step_gbs": round((w.append_bytes_int8() + w.decode_bytes_int8()) /
                              (step_ms * 1e-3) / 1e9, 1),
            "bf16_decode_us": round(1e3 * dec16_ms, 3),
            "bf16_decode_gbs": round(w.decode_bytes_kv16() / (dec16_ms * 1e-3) / 1e9, 1),
            "bf16_step_us": round(1e3 * step16_ms, 3),
            "int8_vs_bf16_decode_speed": round(dec16_ms / dec_ms, 3),
            "int8_vs_bf16_steps_per_s": round(step16_ms / step_ms, 3),
            "traffic": read_traffic(w.name)}


def measure_config(torch, w: W.Workload, dev, flush, steps, warmup, peak) -> dict:
    """The INT8 step and the twin's step of workload w (resident, L2 flushed
    between steps)."""
    g = GpuWorkload(w, dev)
    t_step, t_dec = time_arm(torch, flush, g.append_int8, g.decode_int8, steps, warmup)
    t_step16, t_dec16 = time_arm(torch, flush, g.append_kv16, g.decode_kv16, steps, warmup)
    _, t_cc = time_arm(torch, flush, lambda: None, g.decode_int8_cuda_cores, steps, warmup)
    del g
    torch.cuda.empty_cache()
    return arm_summary(w, *[statistics.mean(t) for t in (t_step, t_dec, t_step16, t_dec16)],
                       peak, statistics.mean(t_cc))


def time_arm(torch, flush, append, decode, steps, warmup, settle_s=0.0):
    """Per-step CUDA-event times (ms) of append+decode and of decode alone."""
    for _ in range(warmup):
        flush()
        append()
        decode()
    if settle_s > 0:
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < settle_s:
            for _ in range(50):
                append()
                decode()
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record()
        append()
        ev[i][1].record()
        decode()
        ev[i][2].record()
    torch.cuda.synchronize()
    step = [a.elapsed_time(c) for a, b, c in ev]
    dec = [b.elapsed_time(c) for a, b, c in ev]
    return step, dec


def time_e2e(torch, g: GpuWorkload, flush, steps, warmup):
    """Through the C ABI with host buffers, the way a serving engine drives
    it: the step's inputs (q, block tables, context lengths, and the new K/V
    rows with their slots when the workload appends) sit in one pinned host
    staging buffer and go to the GPU in one H2D copy; the calls take prepared
    arguments (pointers into the device copy of that buffer); the output comes
    back in one D2H copy.  All of it inside the timed region, every step."""
    import ctypes
    L = g.kvq.load()
    w = g.w
    parts = [("q", g.q_h.view(np.int16)), ("bt", np.ascontiguousarray(g.bt_h, dtype=np.int32)),
             ("cl", np.ascontiguousarray(g.cl_h, dtype=np.int32))]
    if g.k_new is not None:
        parts += [("k", g.k_new_h), ("v", g.v_new_h), ("s", g.slots_h.astype(np.int64))]
    offs, total = {}, 0
    for name, a in parts:
        offs[name] = total
        total += (a.nbytes + 255) // 256 * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    sh = stage_h.numpy()
    for name, a in parts:
        sh[offs[name]:offs[name] + a.nbytes] = np.ascontiguousarray(a).view(np.uint8).ravel()
    stage_d = torch.empty(total, dtype=torch.uint8, device=g.dev)
    h2d = sum(a.nbytes for _, a in parts)
    out_h = torch.empty(g.out.shape, dtype=torch.int16).pin_memory()
    d2h = out_h.numel() * 2
    base = stage_d.data_ptr()
    P = ctypes.c_void_p
    kc, vc, ksc, vsc = g.int8
    stream = P(torch.cuda.current_stream().cuda_stream)
    dt = 1 if w.dtype == "bf16" else 0
    dec_args = [P(base + offs["q"]), dt, w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                P(kc.data_ptr()), P(vc.data_ptr()), P(ksc.data_ptr()), P(vsc.data_ptr()),
                kc.shape[0], 16, P(base + offs["bt"]), g.bt.shape[1], P(base + offs["cl"]),
                w.max_context_len, w.sm_scale, P(g.out.data_ptr()), P(g.ws.data_ptr()),
                g.ws.numel(), stream]
    app_args = None
    if g.k_new is not None:
        T, Hkv, D = g.k_new.shape
        app_args = [P(base + offs["k"]), P(base + offs["v"]), Hkv * D, Hkv * D, T, Hkv, D, dt,
                    P(base + offs["s"]), P(kc.data_ptr()), P(vc.data_ptr()), P(ksc.data_ptr()),
                    P(vsc.data_ptr()), kc.shape[0], 16, stream]

    def step():
        stage_d.copy_(stage_h, non_blocking=True)
        if app_args is not None and L.kvq_quantize_append(*app_args) != 0:
            raise RuntimeError("kvq_quantize_append failed")
        if L.kvq_paged_decode(*dec_args) != 0:
            raise RuntimeError("kvq_paged_decode failed")
        out_h.copy_(g.out.view(torch.int16), non_blocking=True)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    # the staged call computes what the device-resident one (Python binding,
    # separate input tensors) does, bit for bit
    g.decode_int8()
    torch.cuda.synchronize()
    if not torch.equal(out_h, g.out.view(torch.int16).cpu()):
        raise RuntimeError("the end-to-end call's output differs from the device-resident call's")
    return [a.elapsed_time(b) for a, b in ev], h2d, d2h


def host_cost(torch, g: GpuWorkload, calls: int = 200) -> dict:
    """CPU time to submit one kvq_paged_decode (argument checks, launcher,
    tensor maps, launches), timed over back-to-back calls whose GPU work
    queues up behind each other: through the C ABI with prepared ctypes
    arguments, and through the Python binding."""
    import ctypes
    w, L = g.w, g.kvq.load()
    kc, vc, ks, vs = g.int8
    P = ctypes.c_void_p
    args = [P(g.q.data_ptr()), 1 if w.dtype == "bf16" else 0, w.num_seqs, w.num_q_heads,
            w.num_kv_heads, w.head_dim, P(kc.data_ptr()), P(vc.data_ptr()), P(ks.data_ptr()),
            P(vs.data_ptr()), kc.shape[0], 16, P(g.bt.data_ptr()), g.bt.shape[1],
            P(g.cl.data_ptr()), w.max_context_len, w.sm_scale, P(g.out.data_ptr()),
            P(g.ws.data_ptr()), g.ws.numel(), P(torch.cuda.current_stream().cuda_stream)]
    res = {}
    for name, fn in (("c_abi", lambda: L.kvq_paged_decode(*args)),
                     ("python_binding", g.decode_int8)):
        for _ in range(20):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(calls):
            fn()
        t = time.perf_counter() - t0
        torch.cuda.synchronize()
        res[name] = round(1e6 * t / calls, 2)
    res["calls"] = calls
    return res


def g_sweep_workload(G: int) -> W.Workload:
    """The tensor-core A/B's workload for query-group size G: 32 sequences of
    4096 tokens, 8 KV heads, 8 G query heads, d 128, bf16 (the same 272 MB of
    INT8 K/V for every G)."""
    return W.custom(32, 8 * G, 8, 128, "bf16", [4096] * 32, seed=300 + G, pool_factor=1)


def g_sweep(torch, dev, flush, steps):
    """The INT8 decode on the tensor cores (kvq_paged_decode) and on the CUDA
    cores (kvq_paged_decode_cuda_cores) for G = 1, 2, 4, 8 on the same pages."""
    res = {}
    for G in (1, 2, 4, 8):
        w = g_sweep_workload(G)
        g = GpuWorkload(w, dev, arms=("int8",))
        nop = lambda: None  # noqa: E731
        _, tt = time_arm(torch, flush, nop, g.decode_int8, steps, 3)
        _, tc = time_arm(torch, flush, nop, g.decode_int8_cuda_cores, steps, 3)
        mt, mc = statistics.mean(tt), statistics.mean(tc)
        res[str(G)] = {"tensor_core_us": round(1e3 * mt, 2), "cuda_core_us": round(1e3 * mc, 2),
                       "tensor_core_speedup": round(mc / mt, 3),
                       "tensor_core_gbs": round(w.decode_bytes_int8() / (mt * 1e-3) / 1e9, 1),
                       "cuda_core_gbs": round(w.decode_bytes_int8() / (mc * 1e-3) / 1e9, 1)}
        del g
        torch.cuda.empty_cache()
    return res


def sweep(torch, kvq, dev, flush, steps):
    """INT8 vs BF16-twin decode at 2K/8K/32K context (16 seqs, 32/8 heads,
    d 128, bf16), inputs drawn on the GPU from a seeded generator."""
    res = []
    gen = torch.Generator(device=dev)
    for ctx in (2048, 8192, 32768):
        gen.manual_seed(ctx)
        B, Hq, Hkv, D = 16, 32, 8, 128
        w = W.custom(B, Hq, Hkv, D, "bf16", [ctx] * B, seed=ctx, pool_factor=1)
        nb, bt, _ = w.tables()
        kc, vc, ksc, vsc = kvq.alloc_int8_cache(nb, Hkv, D, dev)
        k16, v16 = kvq.alloc_kv16_cache(nb, Hkv, D, torch.bfloat16, dev)
        for b in range(B):
            k = torch.randn((ctx, Hkv, D), generator=gen, device=dev, dtype=torch.bfloat16)
            v = torch.randn((ctx, Hkv, D), generator=gen, device=dev, dtype=torch.bfloat16)
            s = torch.from_numpy(w.slots(b, 0, ctx)).to(dev)
            kvq.kvq_quantize_append(k, v, s, kc, vc, ksc, vsc)
            kvq.kvq_cache_append_kv16(k, v, s, k16, v16)
        q = torch.randn((B, Hq, D), generator=gen, device=dev, dtype=torch.bfloat16)
        btd = torch.from_numpy(bt).to(dev)
        cl = torch.full((B,), ctx, dtype=torch.int32, device=dev)
        nbytes = kvq.kvq_decode_workspace_bytes(B, Hq, Hkv, D, ctx)
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        d8 = lambda: kvq.kvq_paged_decode(q, kc, vc, ksc, vsc, btd, cl, ctx, w.sm_scale,  # noqa
                                          out=out, workspace=ws)
        d16 = lambda: kvq.kvq_paged_decode_kv16(q, k16, v16, btd, cl, ctx, w.sm_scale,  # noqa
                                                out=out, workspace=ws)
        kw, vw = kvq.alloc_kv16_cache(nb, Hkv, D, torch.bfloat16, dev)

        def dwin():
            # the dequantize-window baseline: 16-bit window, then the 16-bit decode
            kvq.kvq_dequantize_window(kc, vc, ksc, vsc, btd, cl, ctx, torch.bfloat16, kw, vw)
            kvq.kvq_paged_decode_kv16(q, kw, vw, btd, cl, ctx, w.sm_scale, out=out, workspace=ws)
        # static per-tensor scales over the same codes (timing only: the codes
        # were written with per-token scales)
        dst = lambda: kvq.kvq_paged_decode_static(q, kc, vc, 0.05, 0.05, btd, cl, ctx,  # noqa
                                                  w.sm_scale, out=out, workspace=ws)
        nop = lambda: None  # noqa: E731
        _, t8 = time_arm(torch, flush, nop, d8, steps, 3)
        _, t16 = time_arm(torch, flush, nop, d16, steps, 3)
        _, tw = time_arm(torch, flush, nop, dwin, steps, 3)
        _, tst = time_arm(torch, flush, nop, dst, steps, 3)
        m8, m16, mw = statistics.mean(t8), statistics.mean(t16), statistics.mean(tw)
        mst = statistics.mean(tst)
        res.append({"context": ctx, "num_seqs": B, "int8_us": round(1e3 * m8, 2),
                    "bf16_us": round(1e3 * m16, 2),
                    "dequant_window_us": round(1e3 * mw, 2),
                    "dequant_window_speedup_vs_bf16": round(m16 / mw, 3),
                    "int8_static_us": round(1e3 * mst, 2),
                    "int8_gbs": round(w.decode_bytes_int8() / (m8 * 1e-3) / 1e9, 1),
                    "bf16_gbs": round(w.decode_bytes_kv16() / (m16 * 1e-3) / 1e9, 1),
                    "int8_speedup_vs_bf16": round(m16 / m8, 3)})
        del kc, vc, ksc, vsc, k16, v16, kw, vw
        torch.cuda.empty_cache()
    return res


def tensor_peak():
    """Dense 16-bit tensor-core peak (TFLOP/s): the measured bf16 GEMM burst
    figure (FP16 has the same nominal rate), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def prefill_measure(torch, kvq, dev, flush, names, steps, warmup):
    """Chunked prefill over the INT8 cache: per shape, the median CUDA-event
    time of one kvq_paged_prefill call (L2 flushed between calls) and the
    causal-attention FLOPs it performs, 4 Hq D per (query, visible key)."""
    peak, kind = tensor_peak()
    gen = torch.Generator(device=dev)
    res = []
    for name in names:
        B, L, n, Hq, Hkv = PREFILL_SHAPES[name]
        D = 128
        gen.manual_seed(L + n)
        w = W.custom(B, Hq, Hkv, D, "bf16", [L] * B, seed=L, pool_factor=1)
        nb, bt, _ = w.tables()
        kc, vc, ksc, vsc = kvq.alloc_int8_cache(nb, Hkv, D, dev)
        for b in range(B):
            k = torch.randn((L, Hkv, D), generator=gen, device=dev, dtype=torch.bfloat16)
            v = torch.randn((L, Hkv, D), generator=gen, device=dev, dtype=torch.bfloat16)
            kvq.kvq_quantize_append(k, v, torch.from_numpy(w.slots(b, 0, L)).to(dev),
                                    kc, vc, ksc, vsc)
        q = torch.randn((B * n, Hq, D), generator=gen, device=dev, dtype=torch.bfloat16)
        btd = torch.from_numpy(bt).to(dev)
        cl = torch.full((B,), L, dtype=torch.int32, device=dev)
        qs = torch.arange(0, B * n + 1, n, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        call = lambda: kvq.kvq_paged_prefill(q, kc, vc, ksc, vsc, btd, cl, qs, L, n,  # noqa
                                             w.sm_scale, out=out)
        _, t = time_arm(torch, flush, lambda: None, call, steps, warmup)
        ms = statistics.median(t)
        keys = B * sum(L - n + i + 1 for i in range(n))
        tflops = 4.0 * Hq * D * keys / (ms * 1e-3) / 1e12
        res.append({"shape": name, "num_seqs": B, "context": L, "chunk": n, "num_q_heads": Hq,
                    "num_kv_heads": Hkv, "head_dim": D, "ms": round(ms, 4),
                    "tflops": round(tflops, 1), "peak_tflops": peak, "peak_kind": kind,
                    "frac": round(tflops / peak, 4)})
        del kc, vc, ksc, vsc, q, out
        torch.cuda.empty_cache()
    return res


def profile_arm(torch, w, dev, args):
    """One decode arm alone (for ncu captures of a bounded device footprint)."""
    if args.profile_g:
        w = g_sweep_workload(args.profile_g)
    if args.profile_seqs:
        w = W.first_seqs(w, args.profile_seqs)
    kv16 = args.profile_arm == "kv16"
    g = GpuWorkload(w, dev, arms=("kv16",) if kv16 else ("int8",))
    flush = make_flush(torch, dev)
    nop = lambda: None  # noqa: E731
    dec = {"int8": g.decode_int8, "kv16": g.decode_kv16,
           "int8cc": g.decode_int8_cuda_cores, "append": g.append_int8}[args.profile_arm]
    _, t = time_arm(torch, flush, nop, dec, args.steps, args.warmup)
    ms = statistics.mean(t)
    if args.profile_arm == "append":
        nbytes = w.append_bytes_int8()
        print(json.dumps({"profile_arm": "append", "workload": w.name,
                          "append_tokens": w.append_tokens(), "append_us": round(1e3 * ms, 2),
                          "append_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}))
        return
    nbytes = w.decode_bytes_kv16() if kv16 else w.decode_bytes_int8()
    print(json.dumps({"profile_arm": args.profile_arm, "workload": w.name,
                      "decode_us": round(1e3 * ms, 2),
                      "decode_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}))


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    rank, local_rank, world = dist_env()
    import torch
    import int8_quantized_paged_tokenwise_gb300 as kvq
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    kvq.load(build_if_missing=False)

    if args.prefill:
        names = list(PREFILL_SHAPES) if args.prefill == "all" else [args.prefill]
        for r in prefill_measure(torch, kvq, dev, make_flush(torch, dev), names,
                                 args.steps, args.warmup):
            print(json.dumps({"prefill": r}), flush=True)
        return
    w = W.make(args.workload)
    if args.profile_arm:
        profile_arm(torch, w, dev, args)
        return
    g = GpuWorkload(w, dev)
    flush = make_flush(torch, dev)

    def barrier():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()

    clocks = ClockSampler(local_rank)
    barrier()
    t_step, t_dec = time_arm(torch, flush, g.append_int8, g.decode_int8, args.steps, args.warmup,
                             settle_s=args.settle)
    barrier()
    clk = clocks.stop()
    t_step16, t_dec16 = time_arm(torch, flush, g.append_kv16, g.decode_kv16, args.steps,
                                 args.warmup)
    t_e2e, h2d, d2h = time_e2e(torch, g, flush, args.steps, args.warmup)
    barrier()
    host_us = host_cost(torch, g)
    _, t_cc = time_arm(torch, flush, lambda: None, g.decode_int8_cuda_cores, args.steps,
                       args.warmup)

    step_ms, dec_ms, step16_ms, dec16_ms, e2e_ms = max_over_ranks(
        pg, dev, [statistics.mean(t) for t in (t_step, t_dec, t_step16, t_dec16, t_e2e)])
    step_bytes = w.append_bytes_int8() + w.decode_bytes_int8()
    value = job_throughput(world, step_bytes, step_ms)
    dec_gbs = w.decode_bytes_int8() / (dec_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    traffic = read_traffic(w.name)
    launches = args.steps * g.launches_per_step()
    del g
    torch.cuda.empty_cache()
    configs = None
    if not args.no_configs:
        configs = {}
        for name in W.NAMES:
            if name == w.name:
                configs[name] = arm_summary(w, step_ms, dec_ms, step16_ms, dec16_ms, peak,
                                            statistics.mean(t_cc))
            else:
                configs[name] = measure_config(torch, W.make(name), dev, flush, args.steps,
                                               args.warmup, peak)
    sw = None
    if not args.no_sweep:
        sw = sweep(torch, kvq, dev, flush, max(5, min(args.steps, 20)))
    gsw = None
    if not args.no_g_sweep:
        gsw = g_sweep(torch, dev, flush, max(5, min(args.steps, 20)))
    pf = None
    if not args.no_prefill:
        pf = prefill_measure(torch, kvq, dev, flush, ["8k_full_gqa8"], max(3, min(args.steps, 10)),
                             3)[0]
    cpu = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(w, budget_s=6.0)
    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 codes x fp16 (tensor cores), fp32 accumulate", "data": "synthetic",
        "config": config_of(w, {"parallelism": f"replicas x{world}"}),
        "decode_gbs": round(dec_gbs, 2),
        "decode_pct_of_measured_peak": round(100 * dec_gbs / peak, 2),
        "decode_pct_of_nominal_8tbs": round(100 * dec_gbs / 8000.0, 2),
        "decode_us": round(1e3 * dec_ms, 3),
        "bytes_per_decoded_token": round(w.decode_bytes_int8() / w.num_seqs),
        "steps_per_s": round(1e3 / step_ms, 1),
        "bf16_twin": {"steps_per_s": round(1e3 / step16_ms, 1), "decode_us": round(1e3 * dec16_ms, 3),
                      "decode_gbs": round(w.decode_bytes_kv16() / (dec16_ms * 1e-3) / 1e9, 2)},
        "int8_vs_bf16_steps_per_s": round(step16_ms / step_ms, 3),
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(dec_gbs / peak, 4), "traffic": traffic,
                     "peak_kind": peak_kind,
                     "kernel": "kvq_paged_decode (decode + split-K combine), algorithmic bytes "
                               f"{w.decode_bytes_int8()} per launch"},
        "e2e": {"value": round(job_throughput(world, step_bytes, e2e_ms), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5)},
        "host_us_per_call": host_us,
        "gpu_launches": launches,
        "clocks": clk,
        "cpu_baseline": cpu,
        "configs": configs,
        "context_sweep": sw,
        "tensor_core_ab": gsw,
        "chunked_prefill": pf,
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
