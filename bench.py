#!/usr/bin/env python3
"""Benchmark: one decode step of the paged-KV hot path on GB300.

A step is the whole hot path over one batch: the scatter of this step's new
K/V token of every sequence into its cache slot and the paged GQA decode.
By default a step is one forge_paged_append_gqa_decode launch per layer
(append fused into the decode kernel); --path separate times
forge_paged_kv_append followed by forge_paged_gqa_decode, --path qk the
fused call with RMSNorm + RoPE on q and the new k, and every run reports
the other paths too.  The default workload
is the Qwen3-4B-shaped attention layer: batch 32, context lengths uniform in
[512, 8192], 32 query / 8 KV heads, head_dim 128, 16-token blocks, 10 % free
blocks interleaved in the pool, bf16 storage.

Reported metric: decode KV-read bandwidth in GB/s (algorithmic bytes = q +
every cached token's K and V rows + out, per step) and microseconds per
layer-step.  Inputs are larger than L2 (the KV pool is ~0.63 GB against a
126 MB L2), so no flush is done between steps.  The dominant kernel is also
timed on its own over at least 50 graph replays of 20 launches (p10 / p50 /
p90 per launch), layer 0's output is checked against the oracle
(max_abs_err), and `per_config` repeats the kernel timing and the check for
every workload of the list (tiny, Qwen3-0.6B, skewed with fp32 and bf16
output, the 36-layer step); workloads whose pools are smaller than 4 x L2
rotate pool copies from launch to launch.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
Under torchrun each rank runs an independent replica of the workload on its
own GPU ("replicas only": the path has no exchange step).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-GQA decode: KV-read HBM GB/s (% of GB300 peak) and µs per layer-step"
PATH_NAMES = {
    "fused": "forge_paged_append_gqa_decode: append + decode in one launch per layer",
    "separate": "forge_paged_kv_append then forge_paged_gqa_decode, per layer",
    "qk": "forge_paged_qk_append_gqa_decode: RMSNorm + RoPE on q/k, append and decode in one launch per layer",
}
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 2**20  # GB300 L2


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 copy measurement)"


DECODE_KERNELS = {"online": "paged_gqa_decode_online_kernel", "two_pass": "paged_gqa_decode_split_kernel"}
PROFILE_FILES = {"online": "decode_online_qwen3_4b.md", "two_pass": "decode_split_qwen3_4b.md"}
# The single-pass kernel's ncu summary on the two latency-bound workloads, one traffic key each.
LATENCY_PROFILE = "decode_online_latency_workloads.md"
LATENCY_WORKLOADS = ("qwen3_0_6b", "skewed")


def _traffic_from_profile(src_hash: str, kernel: str, profile: str | None = None,
                          key: str = "dram_bytes_per_decode_call"):
    """DRAM bytes per launch of `kernel` (the Qwen3-4B decode launch, or with
    `profile` and `key` another kernel's) from its committed ncu summary, if
    that was taken on the current source; else None."""
    p = os.path.join(ROOT, "profiles", profile or PROFILE_FILES[kernel])
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != src_hash:
        return None
    try:
        return int(vals[key])
    except (KeyError, ValueError):
        return None


def _source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_gqa_06_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _decode_source_hash():
    return _source_hash(("decode.cu", "common.cuh", "abi.cu"))


def _decode_traffic(workload: str, kern: str):
    """DRAM bytes per decode launch on `workload` from the committed ncu
    summary that covers it, or None where none does."""
    if workload == "qwen3_4b":
        return _traffic_from_profile(_decode_source_hash(), kern)
    if workload in LATENCY_WORKLOADS and kern == "online":
        return _traffic_from_profile(_decode_source_hash(), kern, LATENCY_PROFILE,
                                     f"dram_bytes_per_decode_call_{workload}")
    return None


def _prefill_source_hash():
    return _source_hash(("prefill_tc.cu", "tcgen05.cuh", "common.cuh", "abi.cu"))


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i", gpu_id,
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for r in csv.reader(io.StringIO(out)):
            if len(r) < 8:
                continue
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + r[0].strip().split(".")[1]) if "." in r[0] else 0.0
                rows.append(dict(t=ts, sm=float(r[1]), max=float(r[2]), power=r[3].strip(),
                                 hw=r[4].strip(), hwt=r[5].strip(), swt=r[6].strip(), pcap=r[7].strip()))
            except (ValueError, IndexError):
                continue
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        inside = [r for r in rows if t0 - 0.15 <= r["t"] <= t1 + 0.15]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for r in use:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in use), "sm_max_mhz": max(r["max"] for r in use),
                "reasons": sorted(reasons), "samples": len(inside),
                "window": "timed region" if inside else "whole run (timed region shorter than one sample)"}


def _gpu_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else str(dev)


def max_over_ranks(values, device="cpu"):
    """Element-wise max of per-rank timings; every rank gets the result.
    The bench's job time is the slowest rank's (no exchange on the data path)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def aggregate_gbs(world, bytes_per_step, steps, max_ms):
    """Whole-job throughput: every rank processes its own batch each step."""
    return world * bytes_per_step * steps / (max_ms * 1e-3) / 1e9


def _seq_bytes(wl, b, out_bytes):
    return wl.Hq * wl.D * 2 + int(wl.context_lens[b]) * wl.Hkv * wl.D * 4 + wl.Hq * wl.D * out_bytes


def _timing_plan(wl, steps, graphs=True):
    """How the GPU arm times a workload, from its sizes and the run's
    arguments only (so both arms can state it): bytes of one step's KV pools,
    the number R of pool copies rotated step to step when those are smaller
    than 4 x L2, the steps per captured graph, and the copies a graph uses."""
    L = wl.layers
    step_pool_bytes = 2 * L * wl.NB * wl.Hkv * 16 * wl.D * 2
    R = min(64, max(1, -(-4 * L2_BYTES // step_pool_bytes)))
    chunk = max(c for c in range(1, max(1, 20 // L) + 1) if steps % c == 0) if graphs else 1
    copies_used = min(R, chunk) if graphs else R
    return step_pool_bytes, R, chunk, copies_used


def _l2_note(step_pool_bytes, R, copies_used):
    if R == 1:
        return f"no flush: inputs larger than L2 (KV pool {step_pool_bytes / 1e6:.0f} MB vs 126 MB L2)"
    return (f"{copies_used} copies of the KV pools rotated step to step "
            f"({copies_used * step_pool_bytes / 1e6:.0f} MB vs 126 MB L2)")


def _config_dict(wl, args=None, out_bytes=None):
    """The `config` object of the JSON line; the same for both arms."""
    s = wl.spec
    lens = wl.context_lens
    d = {"workload": f"{s.name}: {s.description}", "batch": s.B, "q_heads": s.Hq, "kv_heads": s.Hkv,
         "head_dim": s.D, "block_size": 16, "pool_blocks": wl.NB, "tokens": int(lens.sum()),
         "context_len_min": int(lens.min()), "context_len_max": int(lens.max()), "seed": wl.seed,
         "out_dtype": s.out_dtype, "parallelism": "replicas (one independent batch per GPU)"}
    if args is not None:
        graphs = getattr(args, "graphs", True)
        spb, R, chunk, used = _timing_plan(wl, args.steps, graphs)
        ob = out_bytes if out_bytes is not None else (4 if s.out_dtype == "f32" else 2)
        d.update({"launch": (f"CUDA graphs of {chunk} steps replayed" if graphs else "eager C-ABI calls"),
                  "l2": _l2_note(spb, R, used), "layers": wl.layers,
                  "bytes_per_step": wl.layers * wl.bytes_decode(ob),
                  "bytes_rule": "q + K/V rows of every cached token + out (token-exact)"})
    return d


# --------------------------------------------------------------------------- CPU oracle legs

def _oracle_prepare(wl):
    import oracle
    t = wl.layer(0)
    kc, vc = t["k_cache"].copy(), t["v_cache"].copy()
    oracle.paged_kv_append(t["k_new"], t["v_new"], wl.slot_mapping, kc, vc)
    return t, kc, vc


def _oracle_step(wl, t, kc, vc, seqs, threads):
    """Append + decode for a subset of sequences with the CPU oracle."""
    import oracle
    sel = np.asarray(seqs)
    oracle.paged_kv_append(t["k_new"][sel], t["v_new"][sel], wl.slot_mapping[sel], kc, vc)
    oracle.paged_gqa_decode(t["q"][sel], kc, vc, wl.block_tables[sel], wl.context_lens[sel], wl.scale,
                            nthreads=threads)


def cpu_baseline(wl, out_bytes, budget_s=12.0):
    """The oracle as it stands on this host's cores, over whole passes of the
    workload until about budget_s of work (at least one pass)."""
    import oracle
    threads = oracle.host_cores()
    t, kc, vc = _oracle_prepare(wl)
    all_seqs = list(range(wl.B))
    per_pass = sum(_seq_bytes(wl, b, out_bytes) for b in all_seqs)
    passes, elapsed = 0, 0.0
    t0 = time.perf_counter()
    while passes < 1 or (elapsed < budget_s and passes < 1000):
        _oracle_step(wl, t, kc, vc, all_seqs, threads)
        passes += 1
        elapsed = time.perf_counter() - t0
    gbs = per_pass * passes / elapsed / 1e9
    # the same passes on one thread, for about a sixth of the budget
    p1, e1 = 0, 0.0
    t1 = time.perf_counter()
    while p1 < 1 or (e1 < budget_s / 6 and p1 < 1000):
        _oracle_step(wl, t, kc, vc, all_seqs, 1)
        p1 += 1
        e1 = time.perf_counter() - t1
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{passes} full pass(es) of the workload (append + decode of all {wl.B} sequences"
                      f"{', layer 0 of ' + str(wl.layers) if wl.layers > 1 else ''}), "
                      f"{elapsed:.1f} s, fp64 C oracle with {threads} threads",
            "ms_per_step": round(1e3 * elapsed / passes, 3),
            "single_thread": {"value": round(per_pass * p1 / e1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{p1} full pass(es), {e1:.1f} s"}}


def run_reference(args, wl, out_bytes):
    """--impl reference: the CPU oracle as the reference arm."""
    import oracle
    ws, rank, _ = _dist()
    if rank != 0:
        return None
    threads = oracle.host_cores()
    t, kc, vc = _oracle_prepare(wl)
    # size each step's sample (a rotating subset of sequences) so that the
    # whole run takes about two minutes of CPU time
    probe0 = time.perf_counter()
    _oracle_step(wl, t, kc, vc, [0], threads)
    per_seq = max(1e-4, time.perf_counter() - probe0)
    budget = 120.0 / max(1, args.steps + args.warmup)
    nseq = int(max(1, min(wl.B, budget / per_seq)))
    order = list(range(wl.B))
    cursor = 0

    def next_sample():
        nonlocal cursor
        s = [order[(cursor + i) % wl.B] for i in range(nseq)]
        cursor = (cursor + nseq) % wl.B
        return s

    for _ in range(args.warmup):
        _oracle_step(wl, t, kc, vc, next_sample(), threads)
    total_bytes = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s = next_sample()
        _oracle_step(wl, t, kc, vc, s, threads)
        total_bytes += sum(_seq_bytes(wl, b, out_bytes) for b in s)
    el = time.perf_counter() - t0
    gbs = total_bytes / el / 1e9
    sample = (f"each step: append + decode of {nseq} of the {wl.B} sequences (rotating), "
              f"fp64 C oracle, {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config_dict(wl, args, out_bytes),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


# --------------------------------------------------------------------------- GPU leg

PER_CONFIG = ("tiny", "qwen3_0_6b", "qwen3_4b", "skewed", "skewed_bf16", "cb36")
TOL = {"f32": 2e-3, "bf16": 1.6e-2}   # max-abs error bound against the fp64 oracle


class Rig:
    """Device buffers of one workload for the timed loops.

    Layers share one block table and one pool [R*L, NB, Hkv, 16, D] (R
    identical copies, rotated step to step when one step's pools are
    smaller than 4 x L2); each layer has its own q, new K/V row and output.
    Layer 0 holds the seeded workload values (checked against the oracle);
    the other layers hold them too when ``host_layers`` is "all", else
    device-drawn N(0, 1) values with the same NaN poison (same shapes and
    structure, faster to make)."""

    def __init__(self, wl, dev, stream, steps, graphs, host_layers="all"):
        import torch
        self.torch, self.wl, self.dev, self.stream = torch, wl, dev, stream
        L = wl.layers
        self.step_pool_bytes, self.R, self.chunk, self.copies_used = _timing_plan(wl, steps, graphs)
        self.graphs = graphs
        self.t0 = wl.layer(0)
        self.host = {"q": torch.empty(L, wl.B, wl.Hq, wl.D, dtype=torch.bfloat16).pin_memory(),
                     "k_new": torch.empty(L, wl.B, wl.Hkv, wl.D, dtype=torch.bfloat16).pin_memory(),
                     "v_new": torch.empty(L, wl.B, wl.Hkv, wl.D, dtype=torch.bfloat16).pin_memory(),
                     "slots": torch.from_numpy(wl.slot_mapping).pin_memory(),
                     "tables": torch.from_numpy(wl.block_tables).pin_memory(),
                     "lens": torch.from_numpy(wl.context_lens).pin_memory()}
        R = self.R
        self.pool_k = torch.empty(R * L, wl.NB, wl.Hkv, 16, wl.D, dtype=torch.bfloat16, device=dev)
        self.pool_v = torch.empty_like(self.pool_k)
        gen = torch.Generator(device=dev)
        gen.manual_seed(wl.seed)
        pb, po = np.nonzero(wl.poison_mask())
        pb_d, po_d = torch.from_numpy(pb).to(dev), torch.from_numpy(po).to(dev)
        for layer in range(L):
            if layer == 0 or host_layers == "all":
                t = self.t0 if layer == 0 else wl.layer(layer)
                for k in ("q", "k_new", "v_new"):
                    self.host[k][layer].copy_(_bf(torch, t[k]))
                self.pool_k[layer].copy_(_bf(torch, t["k_cache"]))
                self.pool_v[layer].copy_(_bf(torch, t["v_cache"]))
            else:
                for k in ("q", "k_new", "v_new"):
                    self.host[k][layer].copy_(torch.randn(self.host[k].shape[1:], generator=gen, device=dev)
                                              .to(torch.bfloat16).cpu())
                for pool in (self.pool_k, self.pool_v):
                    pool[layer].normal_(generator=gen)
                    pool[layer][pb_d, :, po_d, :] = float("nan")
        for r in range(1, R):
            self.pool_k[r * L:(r + 1) * L].copy_(self.pool_k[:L])
            self.pool_v[r * L:(r + 1) * L].copy_(self.pool_v[:L])
        self.rot = 0
        self.d = {k: v.to(dev) for k, v in self.host.items()}
        self.out_dt = torch.bfloat16 if wl.spec.out_dtype == "bf16" else torch.float32
        self.d["out"] = torch.empty(L, wl.B, wl.Hq, wl.D, dtype=self.out_dt, device=dev)
        self.qw, self.kw = (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
                            for a in wl.qk_norm_weights(0))
        self.rope_table = None

    def next_copy(self):
        r = self.rot
        self.rot = (r + 1) % self.R
        return r * self.wl.layers

    # one step of each path over every layer (the step functions read their
    # buffers from self.d at call time: the end-to-end loop swaps them)
    def step_fused(self):
        from paged_kv_gqa_06_gb300 import binding as B
        d, wl, base = self.d, self.wl, self.next_copy()
        for layer in range(wl.layers):
            B.forge_paged_append_gqa_decode(d["q"][layer], d["k_new"][layer], d["v_new"][layer],
                                            self.pool_k[base + layer], self.pool_v[base + layer], d["tables"],
                                            d["lens"], wl.scale, d["out"][layer], stream=self.stream)

    def step_separate(self):
        from paged_kv_gqa_06_gb300 import binding as B
        d, wl, base = self.d, self.wl, self.next_copy()
        for layer in range(wl.layers):
            B.forge_paged_kv_append(d["k_new"][layer], d["v_new"][layer], d["slots"], self.pool_k[base + layer],
                                    self.pool_v[base + layer], stream=self.stream)
            B.forge_paged_gqa_decode(d["q"][layer], self.pool_k[base + layer], self.pool_v[base + layer],
                                     d["tables"], d["lens"], wl.scale, d["out"][layer], stream=self.stream)

    def step_decode_only(self):
        from paged_kv_gqa_06_gb300 import binding as B
        d, wl, base = self.d, self.wl, self.next_copy()
        for layer in range(wl.layers):
            B.forge_paged_gqa_decode(d["q"][layer], self.pool_k[base + layer], self.pool_v[base + layer],
                                     d["tables"], d["lens"], wl.scale, d["out"][layer], stream=self.stream)

    def step_qk(self):
        """The q/k path (per-head RMSNorm + RoPE on q and the new k) in the same launch."""
        from paged_kv_gqa_06_gb300 import binding as B
        if self.rope_table is None:
            self.rope_table = B.forge_rope_cos_sin_table(1e6, self.wl.D, self.wl.MB * 16).to(self.dev)
        d, wl, base = self.d, self.wl, self.next_copy()
        for layer in range(wl.layers):
            B.forge_paged_qk_append_gqa_decode(d["q"][layer], d["k_new"][layer], d["v_new"][layer],
                                               self.pool_k[base + layer], self.pool_v[base + layer], d["tables"],
                                               d["lens"], wl.scale, d["out"][layer], q_norm_weight=self.qw,
                                               k_norm_weight=self.kw, norm_eps=1e-6, rope_cos_sin=self.rope_table,
                                               stream=self.stream)

    def runner(self, fn, n):
        """A callable that runs `fn` n times: one CUDA graph replay (or eager calls)."""
        torch = self.torch
        if not self.graphs:
            def eager():
                for _ in range(n):
                    fn()
            return eager
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            with torch.cuda.graph(g, stream=self.stream):
                for _ in range(n):
                    fn()
        return g.replay

    def timed(self, run, n, per_call_events=False):
        """Device time (ms) of n runs on the stream: one total, or one per run."""
        torch = self.torch
        ev = [torch.cuda.Event(enable_timing=True) for _ in range((n if per_call_events else 1) + 1)]
        with torch.cuda.stream(self.stream):
            ev[0].record(self.stream)
            for r in range(n):
                run()
                if per_call_events:
                    ev[r + 1].record(self.stream)
            if not per_call_events:
                ev[1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(len(ev) - 1)]

    def sample_launches(self, fn, launches_per_call, min_samples=50, min_seconds=0.4, per_sample=20):
        """Per-launch device times (ms) of `fn` (one step: launches_per_call
        kernel launches): graph replays of ceil(per_sample / launches_per_call)
        steps each, timed one replay at a time with events on the stream, at
        least min_samples replays and min_seconds in all."""
        reps = max(1, -(-per_sample // launches_per_call))
        run = self.runner(fn, reps)
        self.timed(run, 3)                                  # warm
        est = self.timed(run, 5)[0] / 5
        n = max(min_samples, int(math.ceil(min_seconds * 1e3 / max(est, 1e-3))))
        per = self.timed(run, n, per_call_events=True)
        return [x / (reps * launches_per_call) for x in per], n * reps * launches_per_call

    def layer0_check(self):
        """What the CPU-baseline leg needs to check layer 0's output against
        the oracle: the workload, layer 0's inputs and the GPU output (host)."""
        return (self.wl, self.t0, self.d["out"][0].detach().double().cpu().numpy())


def _bf(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def _pcts(ms):
    return [round(float(np.percentile(ms, q)) * 1e3, 2) for q in (10, 50, 90)]


def measure_config(name, dev, stream):
    """One per_config entry: the fused step of workload `name` (one append +
    decode launch per layer) timed over at least 50 graph replays of at least
    20 launches, its bandwidth against the HBM peak, and layer 0's output
    against the oracle."""
    import torch

    from paged_kv_gqa_06_gb300 import binding
    from paged_kv_gqa_06_gb300 import workloads as W

    wl = W.make_workload(name)
    ob = 4 if wl.spec.out_dtype == "f32" else 2

    rig = Rig(wl, dev, stream, 20, True, host_layers="first")
    with torch.cuda.stream(stream):
        for _ in range(3):
            rig.step_fused()                         # sizes the split scratch before capture
    stream.synchronize()
    assert binding.forge_paged_get_device_error(stream) == 0
    check = rig.layer0_check()                       # the output of a fused step (append, then decode)
    w0 = time.time()
    per_launch, launches = rig.sample_launches(rig.step_fused, wl.layers)
    w1 = time.time()
    peak, _ = _peaks()
    bytes_layer = wl.bytes_decode(ob)
    mean_ms = statistics.fmean(per_launch)
    split, kern = binding.forge_paged_gqa_decode_plan(wl.B, wl.Hkv, wl.MB)
    entry = {"workload": f"{name}: {wl.spec.description}", "tokens": int(wl.context_lens.sum()),
             "layers": wl.layers, "kernel": DECODE_KERNELS[kern], "split_tokens": split,
             "us_per_layer_step": round(mean_ms * 1e3, 2), "us_p10_p50_p90": _pcts(per_launch),
             "gbs": round(bytes_layer / (mean_ms * 1e-3) / 1e9, 1),
             "frac": round(bytes_layer / (mean_ms * 1e-3) / 1e9 / peak, 4),
             "launches_timed": launches, "samples": len(per_launch),
             "l2": _l2_note(rig.step_pool_bytes, rig.R, min(rig.R, max(1, -(-20 // wl.layers)))),
             "max_abs_err": None, "tol": TOL[wl.spec.out_dtype], "out_dtype": wl.spec.out_dtype}
    del rig
    torch.cuda.empty_cache()
    return entry, (w0, w1), check


def run_native(args, wl, out_bytes):
    import torch
    import torch.distributed as dist

    from paged_kv_gqa_06_gb300 import binding

    ws, rank, local = _dist()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    binding.load_library()

    stream = torch.cuda.Stream(device=dev)
    rig = Rig(wl, dev, stream, args.steps, args.graphs, host_layers="all")
    L = wl.layers
    bytes_layer = wl.bytes_decode(out_bytes)
    bytes_step = L * bytes_layer
    paths = {"fused": rig.step_fused, "separate": rig.step_separate, "qk": rig.step_qk}
    step = paths[args.path]
    others = {k: v for k, v in paths.items() if k != args.path}
    kernel_only = rig.step_decode_only if args.path == "separate" else step
    launches_per_step = 2 * L if args.path == "separate" else L

    with torch.cuda.stream(stream):
        for _ in range(3):  # eager calls first: the decode sizes its workspace on this stream
            for fn in paths.values():
                fn()
    stream.synchronize()
    assert binding.forge_paged_get_device_error(stream) == 0

    # The timed loops replay CUDA graphs that each hold `chunk` whole steps,
    # the way a serving loop replays a captured decode step: no Python or
    # per-call launch overhead between kernels.  With --no-graphs the loops
    # make eager C-ABI calls instead.
    chunk = rig.chunk
    run_step = rig.runner(step, chunk)
    run_others = {k: rig.runner(v, chunk) for k, v in others.items()}
    reps = args.steps // chunk
    for run in (run_step, *run_others.values()):
        rig.timed(run, max(3, args.warmup) // chunk + 1)

    # ---------------- timed region (device-resident inputs)
    sampler = ClockSampler(_gpu_id(torch, dev.index or 0)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    w0 = time.time()
    ms_total = rig.timed(run_step, reps)[0]
    w1 = time.time()
    if ws > 1:
        dist.barrier()

    # ---------------- the dominant kernel alone: at least 50 samples of at
    # least 20 launches (graph replays, events on its stream), whatever --steps is
    decode_ms, dec_launches = rig.sample_launches(kernel_only, L, min_samples=args.kernel_samples,
                                                  min_seconds=0.4 if args.kernel_samples >= 50 else 0.0)
    w2 = time.time()
    # layer 0's output of the timed kernel, for the oracle check (the q/k path
    # computes another function: RMSNorm and RoPE first)
    checks = {wl.spec.name: rig.layer0_check()} if args.path != "qk" else {}

    # ---------------- the other ways of running the step, for comparison
    ms_others = {k: rig.timed(r, reps)[0] for k, r in run_others.items()}

    # ---------------- every configuration of the workload list, one after another
    per_config = {}
    if rank == 0 and ws == 1 and args.per_config:
        windows = {}
        for name in PER_CONFIG:
            if name == wl.spec.name:
                continue
            per_config[name], windows[name], checks[name] = measure_config(name, dev, stream)
    rows = sampler.stop() if sampler else []
    clocks = ClockSampler.summarize(rows, w0, w2) if sampler else None
    if clocks is not None:
        clocks["window"] = "timed region + dominant-kernel loop" if clocks["samples"] else clocks["window"]
    for name, (a, b) in (windows.items() if per_config else []):
        per_config[name]["sm_mhz"] = ClockSampler.summarize(rows, a, b)["sm_mhz"]

    # ---------------- end to end: host buffers, copies inside the timed region
    # Every step uploads its inputs from pinned host memory (one packed
    # buffer: q, k_new, v_new, slots, tables, lens) and reads its output back
    # to pinned host memory.  Uploads and read-backs run on their own streams
    # with NSETS device buffer sets, so later steps' uploads and earlier steps'
    # read-backs overlap step i's compute, as a serving loop would run them;
    # with four sets every event a step waits for has long completed.
    NSETS = 4
    host, d, out = rig.host, rig.d, rig.d["out"]
    out_dt = rig.out_dt
    fields = ("q", "k_new", "v_new", "slots", "tables", "lens")
    nbytes = {k: host[k].numel() * host[k].element_size() for k in fields}
    offs, total = {}, 0
    for k in fields:
        offs[k] = total
        total += (nbytes[k] + 255) // 256 * 256
    host_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
    for k in fields:
        host_pack[offs[k]:offs[k] + nbytes[k]].copy_(host[k].contiguous().view(-1).view(torch.uint8))
    dev_pack = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(NSETS)]
    out_e = [torch.empty_like(out) for _ in range(NSETS)]
    host_out_e = [torch.empty(out.shape, dtype=out_dt).pin_memory() for _ in range(NSETS)]
    views = []
    for sb in range(NSETS):
        v = {k: dev_pack[sb][offs[k]:offs[k] + nbytes[k]].view(host[k].dtype).view(host[k].shape) for k in fields}
        v["out"] = out_e[sb]
        views.append(v)
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_h2d = [torch.cuda.Event() for _ in range(NSETS)]
    ev_comp = [torch.cuda.Event() for _ in range(NSETS)]
    ev_d2h = [torch.cuda.Event() for _ in range(NSETS)]
    saved = dict(d)

    def e2e_run(n, t0=None, t1=None):
        if t0 is not None:
            t0.record(h2d_s)
        for sb in range(min(NSETS, n)):
            with torch.cuda.stream(h2d_s):
                dev_pack[sb].copy_(host_pack, non_blocking=True)
            ev_h2d[sb].record(h2d_s)
        for i in range(n):
            sb = i % NSETS
            stream.wait_event(ev_h2d[sb])
            if i >= NSETS:
                stream.wait_event(ev_d2h[sb])      # this buffer set's previous output is read back
            d.update(views[sb])
            with torch.cuda.stream(stream):
                step()
            ev_comp[sb].record(stream)
            d2h_s.wait_event(ev_comp[sb])
            with torch.cuda.stream(d2h_s):
                host_out_e[sb].copy_(out_e[sb], non_blocking=True)
            ev_d2h[sb].record(d2h_s)
            if i + NSETS < n:
                h2d_s.wait_event(ev_comp[sb])      # this buffer set's inputs are consumed
                with torch.cuda.stream(h2d_s):
                    dev_pack[sb].copy_(host_pack, non_blocking=True)
                ev_h2d[sb].record(h2d_s)
        if t1 is not None:
            t1.record(d2h_s)

    e2e_start, e2e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(3)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    e2e_run(args.steps, e2e_start, e2e_end)
    torch.cuda.synchronize(dev)
    e2e_ms = e2e_start.elapsed_time(e2e_end)
    d.update(saved)
    host_out = host_out_e[(args.steps - 1) % NSETS]
    assert binding.forge_paged_get_device_error(stream) == 0
    assert torch.isfinite(host_out.float()).all()

    names = sorted(ms_others)
    maxed = max_over_ranks([ms_total, e2e_ms] + [ms_others[k] for k in names], dev)
    ms_total, e2e_ms = maxed[0], maxed[1]
    ms_others = dict(zip(names, maxed[2:]))

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return None

    peak, peak_src = _peaks()
    ms_step = ms_total / args.steps
    value = aggregate_gbs(ws, bytes_step, args.steps, ms_total)
    dec_avg_ms = statistics.fmean(decode_ms)
    achieved = bytes_layer / (dec_avg_ms * 1e-3) / 1e9
    split_tokens, kern = binding.forge_paged_gqa_decode_plan(wl.B, wl.Hkv, wl.MB)
    traffic = _decode_traffic(wl.spec.name, kern)
    h2d = total  # the packed input buffer, as copied each step
    d2h = host_out.numel() * host_out.element_size()
    tol = TOL[wl.spec.out_dtype]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "us_per_layer_step": round(ms_step * 1e3 / L, 2),
        "pct_of_hbm_peak": round(100.0 * value / ws / peak, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "accumulate": "f32",
        "arithmetic": "bf16 operands on the tensor cores (softmax weights as bf16 high + low parts), fp32 "
                      "accumulation, softmax and split merge in fp32",
        "data": "synthetic",
        "config": _config_dict(wl, args, out_bytes),
        "roofline": {"bound": "hbm",
                     "kernel": (f"{DECODE_KERNELS[kern]} (one decode call; split merge inside)"
                                if args.path == "separate" else
                                f"{DECODE_KERNELS[kern]} with fused append (one launch per layer)"),
                     "split_tokens": split_tokens,
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "decode_us": round(dec_avg_ms * 1e3, 2),
                     "decode_us_p10_p50_p90": _pcts(decode_ms),
                     "launches_timed": dec_launches, "samples": len(decode_ms),
                     "peak_source": peak_src + ", of measured" if peak_src.startswith("measured") else peak_src},
        "max_abs_err": None, "tol": tol,
        "e2e": {"value": round(aggregate_gbs(ws, bytes_step, args.steps, e2e_ms), 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms / args.steps, 5),
                "how": "every step: its packed inputs copied from pinned host memory, the step through the "
                       "public binding (eager calls), its output copied back to pinned host memory; copies on "
                       f"their own streams, {NSETS} buffer sets, overlapping the neighbouring steps' compute"},
        "gpu_launches": launches_per_step * args.steps,
        "path": PATH_NAMES[args.path],
        "other_paths": {k: {"path": PATH_NAMES[k], "ms_per_step": round(v / args.steps, 5),
                            "us_per_layer_step": round(v / args.steps * 1e3 / L, 2),
                            "value": round(aggregate_gbs(ws, bytes_step, args.steps, v), 2)}
                        for k, v in ms_others.items()},
        "clocks": clocks,
    }
    if per_config:
        head = {"workload": line["config"]["workload"], "tokens": line["config"]["tokens"], "layers": L,
                "kernel": DECODE_KERNELS[kern], "split_tokens": split_tokens,
                "us_per_layer_step": round(dec_avg_ms * 1e3, 2), "us_p10_p50_p90": _pcts(decode_ms),
                "gbs": round(achieved, 1), "frac": round(achieved / peak, 4), "launches_timed": dec_launches,
                "samples": len(decode_ms), "l2": line["config"]["l2"], "max_abs_err": None, "tol": tol,
                "out_dtype": wl.spec.out_dtype, "sm_mhz": clocks["sm_mhz"] if clocks else None}
        per_config = {wl.spec.name: head, **per_config}
        line["per_config"] = {k: per_config[k] for k in PER_CONFIG if k in per_config}
    line["_checks"] = checks   # filled into max_abs_err by the CPU-baseline leg, then dropped
    if ws > 1:
        dist.destroy_process_group()
    return line


def check_outputs(line, checks):
    """CPU-baseline leg: layer 0's GPU output of every timed workload against
    the oracle on the same inputs (max-abs error, in the line and per_config)."""
    import oracle
    for name, (wl, t, got) in checks.items():
        kc, vc = t["k_cache"].copy(), t["v_cache"].copy()
        oracle.paged_kv_append(t["k_new"], t["v_new"], wl.slot_mapping, kc, vc)
        ref = oracle.paged_gqa_decode(t["q"], kc, vc, wl.block_tables, wl.context_lens, wl.scale)
        err = float(np.max(np.abs(got - ref))) if np.all(np.isfinite(got)) else float("inf")
        if name == line["config"]["workload"].split(":")[0]:
            line["max_abs_err"] = err
        if name in line.get("per_config", {}):
            line["per_config"][name]["max_abs_err"] = err


def run_serving(args, wl):
    """Continuous batching over the shared multi-layer pool.

    One step = one host driver step (forge_batch_step: retire, preempt,
    admit, grow every running row by one token), one forge_batch_apply
    (block tables, context lengths and slot mapping updated on the device)
    and the fused append + decode launch of every layer, replayed from one
    captured CUDA graph that reads those device tables.  Requests are kept
    outstanding in a closed loop (batch rows + 16): prompts lognormal like
    the workload's lengths, decode lengths uniform in [16, 256].  Prompt K/V
    is not written (prefill is not part of this path): the pool holds seeded
    random bf16 values.  Bytes per step follow the step's own context
    lengths, so the metric is the same as the static batch's.
    """
    import torch

    from paged_kv_gqa_06_gb300 import binding as B
    from paged_kv_gqa_06_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B.load_library()
    L, rows, bs = wl.layers, wl.B, 16
    mbps = wl.spec.hi // bs
    new_min, new_max, budget = 16, 256, 16384
    nb = int(wl.NB * 1.25)
    n_req = rows + 16 + 4 * (args.steps + args.warmup + 64)
    stream_req = W.request_stream(n_req, wl.spec.seed, prompt_median=wl.spec.median, prompt_sigma=wl.spec.sigma,
                                  prompt_max=mbps * bs - new_max, new_min=new_min, new_max=new_max)

    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.spec.seed)
    pool_k = torch.empty(L, nb, wl.Hkv, bs, wl.D, dtype=torch.bfloat16, device=dev)
    pool_v = torch.empty_like(pool_k)
    for t in (pool_k, pool_v):
        for layer in range(L):
            t[layer].normal_(generator=gen)
    q = torch.randn(L, rows, wl.Hq, wl.D, generator=gen, device=dev).to(torch.bfloat16)
    k_new = torch.randn(L, rows, wl.Hkv, wl.D, generator=gen, device=dev).to(torch.bfloat16)
    v_new = torch.randn(L, rows, wl.Hkv, wl.D, generator=gen, device=dev).to(torch.bfloat16)
    out = torch.empty(L, rows, wl.Hq, wl.D, dtype=torch.bfloat16, device=dev)
    tables = torch.full((rows, mbps), -1, dtype=torch.int32, device=dev)
    lens = torch.zeros(rows, dtype=torch.int32, device=dev)
    slots = torch.full((rows,), -1, dtype=torch.int64, device=dev)
    stream = torch.cuda.Stream(device=dev)

    pool = B.forge_kv_pool_create(nb, bs, mbps)
    batch = B.forge_batch_create(pool, rows, budget)
    state = {"next": 0, "outstanding": 0}

    def top_up():
        while state["outstanding"] < rows + 16 and state["next"] < n_req:
            i = state["next"]
            B.forge_batch_submit(batch, int(stream_req.seq_ids[i]), int(stream_req.prompts[i]),
                                 int(stream_req.max_new[i]))
            state["next"] += 1
            state["outstanding"] += 1

    def layers():
        for layer in range(L):
            B.forge_paged_append_gqa_decode(q[layer], k_new[layer], v_new[layer], pool_k[layer], pool_v[layer],
                                            tables, lens, wl.scale, out[layer], stream=stream)

    def driver_step(times=None):
        t0 = time.perf_counter()
        top_up()
        rep = B.forge_batch_step(batch)
        state["outstanding"] -= rep["retired"]
        t1 = time.perf_counter()
        B.forge_batch_apply(batch, tables, lens, slots, stream=stream)
        if times is not None:
            times[0] += t1 - t0
            times[1] += time.perf_counter() - t1
        return rep

    with torch.cuda.stream(stream):
        layers()                      # sizes the split workspace on this stream before capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layers()

    bytes_fixed = rows * wl.Hq * wl.D * 2 * 2      # q read + bf16 out written, per layer
    per_token = wl.Hkv * wl.D * 2 * 2               # K and V rows of one cached token, per layer
    warm = 0
    with torch.cuda.stream(stream):
        while True:                                 # fill the batch, then the requested warm-up
            rep = driver_step()
            graph.replay()
            warm += 1
            if (rep["running"] == rows and warm >= args.warmup) or warm >= args.warmup + 256:
                break
    stream.synchronize()

    sampler = ClockSampler(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0])
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total_bytes, host, stats = 0, [0.0, 0.0], {"admitted": 0, "retired": 0, "preempted": 0, "running": 0,
                                               "tokens": 0}
    w0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            rep = driver_step(host)
            graph.replay()
            total_bytes += L * (bytes_fixed + rep["tokens"] * per_token)
            for k in stats:
                stats[k] += rep[k]
        ev1.record(stream)
    stream.synchronize()
    w1 = time.time()
    clocks = ClockSampler.summarize(sampler.stop(), w0, w1)
    ms = ev0.elapsed_time(ev1)
    assert B.forge_paged_get_device_error(stream) == 0
    assert torch.isfinite(out.float()).all()
    B.forge_batch_destroy(batch)
    left = B.forge_kv_pool_used_blocks(pool)
    B.forge_kv_pool_destroy(pool)

    peak, peak_src = _peaks()
    gbs = total_bytes / (ms * 1e-3) / 1e9
    k = args.steps
    return {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": 1, "steps": k, "warmup": warm,
        "ms_per_step": round(ms / k, 5), "us_per_layer_step": round(ms / k * 1e3 / L, 2),
        "pct_of_hbm_peak": round(100 * gbs / peak, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
        "config": {"workload": f"{wl.spec.name} under continuous batching: {L} layers, {rows} rows, requests with "
                               f"lognormal prompts (median {wl.spec.median:g}, sigma {wl.spec.sigma:g}) and "
                               f"decode lengths U[{new_min},{new_max}], closed loop of rows + 16 outstanding",
                   "pool_blocks": nb, "max_blocks_per_seq": mbps, "token_budget": budget,
                   "launch": "per step: host driver step + forge_batch_apply (copy + 1 kernel), then one CUDA "
                             "graph of the fused append + decode launch of every layer",
                   "l2": f"no flush: KV pool {2 * pool_k.numel() * 2 / 1e9:.1f} GB vs 126 MB L2",
                   "bytes_rule": "per layer: q + K/V rows of every cached token after the step + out"},
        "driver": {"host_step_us": round(host[0] / k * 1e6, 1),
                   "apply_call_us": round(host[1] / k * 1e6, 1),
                   "apply_note": "host time of the forge_batch_apply call, including any wait for a staging "
                                 "buffer the device has not consumed yet (the host runs up to 4 steps ahead)",
                   "mean_running": round(stats["running"] / k, 2),
                   "mean_context_tokens": round(stats["tokens"] / max(1, stats["running"]), 1),
                   "admitted": stats["admitted"], "retired": stats["retired"], "preempted": stats["preempted"],
                   "blocks_left_after_destroy": left},
        "gpu_launches": k * (L + 1),
        "peak": peak, "peak_source": peak_src,
        "clocks": clocks,
    }


def run_prefill(args, name):
    """Paged prefill: the run's K/V appended (forge_paged_kv_append, one slot
    per token), then forge_paged_prefill over the batch.  A contraction, so
    the roofline is the tensor peak: algorithmic FLOPs are 4 * D per (query
    token, attended token, query head) -- QK^T and PV, causal pairs only."""
    import torch

    from paged_kv_gqa_06_gb300 import binding as B
    from paged_kv_gqa_06_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B.load_library()
    pw = W.make_prefill(name)
    t = pw.layer(0)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    copies = 4                                   # rotate cache copies so the K/V do not sit in L2
    kc = [bf(t["k_cache"]) for _ in range(copies)]
    vc = [bf(t["v_cache"]) for _ in range(copies)]
    q, k_new, v_new = bf(t["q"]), bf(t["k_new"]), bf(t["v_new"])
    slots = torch.from_numpy(pw.slot_mapping).to(dev)
    tables = torch.from_numpy(pw.block_tables).to(dev)
    lens = torch.from_numpy(pw.context_lens).to(dev)
    qs = torch.from_numpy(pw.query_start).to(dev)
    out_dt = torch.bfloat16 if pw.spec.out_dtype == "bf16" else torch.float32
    out = torch.empty(pw.T, pw.Hq, pw.D, dtype=out_dt, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(c, with_append=True):
        if with_append:
            B.forge_paged_kv_append(k_new, v_new, slots, kc[c], vc[c], stream=stream)
        B.forge_paged_prefill(q, kc[c], vc[c], tables, lens, qs, pw.scale, out, stream=stream)

    graphs = {}
    for key in (True, False):
        with torch.cuda.stream(stream):
            for c in range(copies):
                step(c, key)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in range(copies):
                step(c, key)
        graphs[key] = g
    reps = max(1, args.steps // copies)

    def timed(g, n):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(n):
                g.replay()
            ev1.record(stream)
        stream.synchronize()
        return ev0.elapsed_time(ev1) / (n * copies)

    for g in graphs.values():
        timed(g, max(1, args.warmup // copies + 1))
    sampler = ClockSampler(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0])
    time.sleep(0.3)
    w0 = time.time()
    ms_step = timed(graphs[True], reps)
    ms_kernel = timed(graphs[False], reps)
    w1 = time.time()
    clocks = ClockSampler.summarize(sampler.stop(), w0, w1)
    assert B.forge_paged_get_device_error(stream) == 0
    assert torch.isfinite(out.float()).all()

    pairs = pw.attended_pairs()
    flops = 4.0 * pw.D * pw.Hq * pairs
    kv_bytes = int(pw.context_lens.astype(np.int64).sum()) * pw.Hkv * pw.D * 2 * 2
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        with open(peaks_path) as f:
            peak, peak_src = float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, " \
                                                                 "cuBLAS bf16 GEMM burst), of measured"
    else:
        peak, peak_src = 1900.0, "fallback (1.9 PFLOP/s bf16 burst), of fallback"
    tflops_kernel = flops / (ms_kernel * 1e-3) / 1e12
    # DRAM bytes per launch from the committed ncu summary of the tcgen05 kernel
    # on this workload, if it was taken on the current sources
    traffic = (_traffic_from_profile(_prefill_source_hash(), "", "prefill_qwen3_4b.md",
                                     "dram_bytes_per_prefill_call")
               if name == "prefill_4b" and os.environ.get("FORGE_PREFILL_KERNEL") != "mma" else None)
    tflops_step = flops / (ms_step * 1e-3) / 1e12
    return {
        "metric": "paged prefill: attention TFLOP/s (causal pairs only) and us per call",
        "value": round(tflops_step, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": reps * copies,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
        "config": {"workload": f"{name}: {pw.spec.description}", "batch": pw.B, "query_tokens": pw.T,
                   "context_tokens": int(pw.context_lens.sum()), "attended_pairs": pairs,
                   "flops_rule": "4 * D * Hq per (query token, attended token)",
                   "step": "forge_paged_kv_append of the run's K/V + forge_paged_prefill, CUDA graph",
                   "l2": f"{copies} cache copies rotated ({copies * kv_bytes / 1e6:.0f} MB of K/V vs 126 MB L2)"},
        "roofline": {"bound": "tensor",
                     "kernel": ("paged_prefill_kernel (mma.sync m16n8k16, P as bf16 hi + lo)"
                                if os.environ.get("FORGE_PREFILL_KERNEL") == "mma" else
                                "paged_prefill_tc_kernel (tcgen05.mma, accumulators in TMEM, P from TMEM)"),
                     "achieved": round(tflops_kernel, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tflops_kernel / peak, 4), "traffic": traffic,
                     "prefill_us": round(ms_kernel * 1e3, 2), "peak_source": peak_src},
        "gpu_launches": 2 * reps * copies,
        "clocks": clocks,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="qwen3_4b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=["fused", "separate", "qk"], default="fused",
                    help="fused: forge_paged_append_gqa_decode; separate: append then decode; "
                         "qk: forge_paged_qk_append_gqa_decode with RMSNorm + RoPE")
    ap.add_argument("--no-graphs", dest="graphs", action="store_false",
                    help="time eager C-ABI calls instead of replaying captured steps")
    ap.add_argument("--prefill", action="store_true",
                    help="time the paged prefill on a prefill workload (default prefill_4b)")
    ap.add_argument("--kernel-samples", type=int, default=50,
                    help="graph replays (of 20 launches) timing the dominant kernel; below 50 (for profiler "
                         "runs) there is no minimum duration either")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip timing the other workloads of the list (per_config in the line)")
    ap.add_argument("--serving", action="store_true",
                    help="continuous batching through the block pool + batch driver (multi-layer workloads)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3

    from paged_kv_gqa_06_gb300 import workloads as W
    if args.prefill:
        import __graft_entry__
        __graft_entry__.build()
        name = args.workload if args.workload.startswith("prefill") else "prefill_4b"
        print(json.dumps(run_prefill(args, name)), flush=True)
        return 0
    wl = W.make_workload(args.workload)
    out_bytes = 4 if wl.spec.out_dtype == "f32" else 2

    if args.impl == "reference":
        line = run_reference(args, wl, out_bytes)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    ws, _, local = _dist()
    if local == 0:
        import __graft_entry__
        __graft_entry__.build()
    else:  # another rank on this node builds; wait for its library
        from paged_kv_gqa_06_gb300 import binding
        for _ in range(600):
            if os.path.exists(binding.LIB_PATH):
                break
            time.sleep(0.5)
    if args.serving:
        print(json.dumps(run_serving(args, wl)), flush=True)
        return 0
    line = run_native(args, wl, out_bytes)
    if line is None:
        return 0
    checks = line.pop("_checks")
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, out_bytes)
        check_outputs(line, checks)
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
