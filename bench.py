#!/usr/bin/env python
"""Benchmark of paged decode attention on one GPU (or N data-parallel replicas).

One step is one decode step of the whole attention stack of a workload, all through the C ABI
of libpkv.so, captured once in a CUDA graph and replayed:
  * paged GQA workloads (llama70b_b16, llama70b_mixed, edge_1p1b): per layer one fused launch
    that writes the step's new K/V rows to the slots the block table maps their positions to
    (slot mapping + KV append) and runs the paged decode attention;
  * prefix: the beam fork's copy-on-write block copies, then the fused append + decode;
  * ring: four draft tokens per sequence (sink + ring slot mapping, append, causal decode over
    every layer), a rollback of two, then one more token (mapping, append, decode).

The headline line is the largest single-GPU workload, llama70b_b16 (21.5 GB of K/V per step);
the other workloads are measured in the same run and reported under "per_workload", each with
its own roofline, end-to-end figure and clock record. Every timed region replays `--steps`
steps back to back, repeated until at least `--min-seconds` of GPU time has passed; the
median repeat is reported (ms_per_step x steps describes one repeat).

Printed (rank 0, one JSON line): the KV-read bandwidth (algorithmic fp16 K+V bytes the step
reads over the step time), decode tokens/s, the decode kernel's roofline against the
measured HBM copy peak, the end-to-end figure with host buffers (inputs copied in and the
attention output copied back every step), the fp64 CPU oracle's rate on a bounded sample of
the headline workload, the SM clocks seen during the timed regions and the kernel launch
count.

`--impl reference` times the CPU oracle alone (the reference arm): each step is a bounded
sample of the workload, sized so the whole run ends in a few minutes.
"""
from __future__ import annotations

import argparse
import copy as _copy
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_kv_cache_147_gb300 import replicas, workloads  # noqa: E402

METRIC = "paged decode attn: KV-read HBM GB/s (% of GB300 peak), decode tokens/s"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024
ALL_WORKLOADS = ["llama70b_b16", "edge_1p1b", "llama70b_mixed", "prefix", "ring", "prefill_70b",
                 "prefix_private", "spec_verify"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama70b_b16", choices=ALL_WORKLOADS,
                    help="the headline workload (default: the largest single-GPU one)")
    ap.add_argument("--also", default="edge_1p1b,llama70b_mixed,prefix,ring,prefill_70b,"
                                      "spec_verify",
                    help="comma-separated workloads measured after the headline and reported "
                         "under per_workload ('none': headline only)")
    ap.add_argument("--min-seconds", type=float, default=1.5,
                    help="each timed region repeats the --steps block until it has run this "
                         "long; the median repeat is reported")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the CPU-baseline sample")
    ap.add_argument("--kv", choices=["fp16", "fp8"], default="fp16",
                    help="fp8: an E4M3 cache with per-kv-head scales (paged GQA workloads): per "
                         "layer one launch appends the step's rows as E4M3 and decodes")
    ap.add_argument("--layers", type=int, default=None,
                    help="fewer layers than the workload's (small profiler captures; the "
                         "per-launch figures are unchanged, the step and the L2 note shrink)")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def load_tensor_peak():
    """Dense f16/bf16 tensor-core peak: the measured cuBLAS bf16 rates (f16 runs at the bf16
    rate on these tensor cores: nominal ratio 1), burst and sustained."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def prefill_flops(w) -> int:
    """Algorithmic flops of one chunked-prefill step over all layers: every visible (query,
    key) pair of every query head costs 2 x 128 for Q K^T and 2 x 128 for P V."""
    ctx = w.context_lens.astype(np.int64)
    first = ctx - w.q_len
    pairs = 0
    for b in range(w.num_seqs):
        i = np.arange(w.q_len, dtype=np.int64)
        pairs += int(np.maximum(0, np.minimum(ctx[b], first[b] + i + 1)).sum())
    return pairs * w.num_q_heads * w.head_dim * 4 * w.num_layers


def make_workload(name, layers=None):
    # the ring cache spans 24 layers of the 1.1B shape, so that a step exceeds L2
    if name == "ring":
        w = workloads.ring(num_layers=24)
    elif name == "prefix_private":
        w = workloads.prefix(private=True)
    else:
        w = workloads.WORKLOADS[name]()
    if layers is not None:
        w.num_layers = max(1, min(layers, w.num_layers))
    return w


def ring_phase_tokens(w) -> int:
    """K/V rows one ring decode launch reads per (sequence, kv head): the slots it holds."""
    hw = w.ring_len0.astype(np.int64) + w.q_len       # the drafts' high-water mark
    return int(np.minimum(hw, w.sink + w.window).sum())


def step_bytes(w, kv="fp16") -> int:
    """Algorithmic K+V bytes one step reads over all layers: every visible token of every
    (sequence, kv head) once. The ring step decodes twice per layer (the drafts, then the token
    after the rollback), each over the min(hw, sink + window) slots it holds. An E4M3 cache
    holds one byte per element instead of two."""
    if kv == "fp8":
        return w.kv_read_bytes() // 2
    if w.name == "ring":
        return 2 * ring_phase_tokens(w) * w.num_kv_heads * w.head_dim * 2 * 2 * w.num_layers
    return w.kv_read_bytes()


def unique_bytes(w) -> int:
    """K+V bytes of the distinct physical block rows a step reads (shared blocks once)."""
    used = {}
    for b in range(w.num_seqs):
        n = int(w.context_lens[b])
        for j in range((n + w.block_size - 1) // w.block_size):
            blk = int(w.block_tables[b, j])
            used[blk] = max(used.get(blk, 0), min(w.block_size, n - j * w.block_size))
    return sum(used.values()) * w.num_kv_heads * w.head_dim * 2 * 2 * w.num_layers


def describe(w, kv="fp16") -> dict:
    cl = w.context_lens.astype(np.int64)
    nbytes = step_bytes(w, kv)
    return {
        "workload": w.name,
        "layers": w.num_layers, "num_seqs": w.num_seqs, "q_len": w.q_len,
        "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
        "block_size": w.block_size, "pool_blocks_per_layer": w.num_blocks,
        "context_min_mean_max": [int(cl.min()), round(float(cl.mean()), 1), int(cl.max())],
        "kv_bytes_per_step": nbytes,
        "accumulate": "f32",
        "l2": (f"no flush: one step reads {nbytes / 1e9:.2f} GB of K/V, "
               f"more than the {L2_BYTES / 2**20:.0f} MiB L2") if nbytes > L2_BYTES else
              (f"no flush and a step of {nbytes / 1e6:.1f} MB of K/V, within the "
               f"{L2_BYTES / 2**20:.0f} MiB L2: not an HBM measurement"),
    }


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        self.gpu = ids[local_rank] if local_rank < len(ids) else str(local_rank)
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # nvidia-smi takes a moment to start: the timed region begins once it samples
        t_end = time.time() + 5.0
        while time.time() < t_end and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------ our arm
class Step:
    """Device-resident inputs of one decode step and the launches that make it.

    The per-step inputs and outputs are attributes named in `in_names` / `out_names` (the
    end-to-end measurement copies exactly those to and from the host)."""

    def __init__(self, w, dev, kv="fp16"):
        from paged_kv_cache_147_gb300 import pkv
        self.pkv = pkv
        self.w = w
        self.dev = dev
        # fused append + decode per layer (paged workloads), copy-on-write then fused (prefix),
        # drafts / rollback / one more token (ring), or the E4M3 form of the fused step
        self.kind = {"prefix": "prefix", "prefix_private": "prefix",
                     "ring": "ring"}.get(w.name, "fused")
        if kv == "fp8":
            if self.kind != "fused":
                raise SystemExit("--kv fp8 applies to the paged GQA workloads")
            self.kind = "fp8"
        Lr = w.num_layers
        self.k, self.v = w.pools(dev)
        if self.kind == "fp8":
            self._to_e4m3()
        if self.kind == "prefix":
            self._fork_tables()
        self.bt = torch.as_tensor(w.block_tables, device=dev)
        self.cl = torch.as_tensor(w.context_lens, device=dev)
        self.q = torch.stack([w.query(l, dev) for l in range(Lr)])
        kv_rows = [w.new_kv(l, dev) for l in range(Lr)]
        self.kn = torch.stack([a for a, _ in kv_rows])
        self.vn = torch.stack([b for _, b in kv_rows])
        self.out = torch.empty_like(self.q)
        seq, pos = w.new_token_positions()
        self.seq = torch.as_tensor(seq, device=dev)
        self.pos = torch.as_tensor(pos, device=dev)
        self.slots = torch.empty(seq.shape[0], dtype=torch.int64, device=dev)
        self.ws = pkv.make_workspace(w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads, dev)
        self.in_names = ["q", "kn", "vn", "bt", "cl"]
        self.out_names = ["out"]
        self.launches_per_step = Lr
        self.tokens_per_step = w.num_seqs * w.q_len
        if self.kind == "prefix":
            self.in_names += ["cow_src", "cow_dst"]
            self.launches_per_step = Lr + 1
        if self.kind == "ring":
            self._ring_setup()

    # -- workload-specific set-up -------------------------------------------------------------
    def _to_e4m3(self):
        """E4M3 pools from the same data, one scale per (layer, kv head): max |x| / 448."""
        w, dev = self.w, self.dev
        k8 = torch.empty(self.k.shape, dtype=torch.uint8, device=dev)
        v8 = torch.empty(self.v.shape, dtype=torch.uint8, device=dev)
        self.ks = torch.empty((w.num_layers, w.num_kv_heads), dtype=torch.float32, device=dev)
        self.vs = torch.empty_like(self.ks)
        for l in range(w.num_layers):
            for src, dst, sc in ((self.k, k8, self.ks), (self.v, v8, self.vs)):
                x = src[l].float()
                sc[l] = x.abs().amax(dim=(0, 2, 3)) / 448.0
                y = (x / sc[l][None, :, None, None]).clamp(-448.0, 448.0)
                dst[l] = y.to(torch.float8_e4m3fn).view(torch.uint8)
        self.k, self.v = k8, v8

    def _fork_tables(self):
        """The beam fork: children 60..63 share their parent's partly filled last block; the
        first three writers find it shared and copy it to a spare block (copy-on-write), the
        last writes in place. The step replays these copies and then the appends."""
        w = self.w
        tables = w.block_tables.copy()
        last = (int(w.context_lens[60]) - 1) // w.block_size
        shared = int(tables[60, last])
        spare = list(w.free_blocks)
        src, dst = [], []
        for child in (60, 61, 62):
            tables[child, last] = spare.pop(0)
            src.append(shared)
            dst.append(int(tables[child, last]))
        w.block_tables = tables
        self.cow_src = torch.tensor(src, dtype=torch.int32, device=self.dev)
        self.cow_dst = torch.tensor(dst, dtype=torch.int32, device=self.dev)
        self.cow_bytes = 2 * 2 * len(src) * w.num_kv_heads * w.block_size * w.head_dim * 2

    def _ring_setup(self):
        """Drafts at positions L0 .. L0+3 (hw = L = L0 + 4), then a rollback of two and one
        more token at L0 + 2 (L = L0 + 3, hw stays L0 + 4)."""
        w, dev, pkv = self.w, self.dev, self.pkv
        B, nd = w.num_seqs, w.q_len
        L0 = w.ring_len0.astype(np.int64)
        self.pos_b = torch.as_tensor(L0 + nd - 2, device=dev)
        self.seq_b = torch.arange(B, dtype=torch.int32, device=dev)
        self.L_a = torch.as_tensor(L0 + nd, device=dev)
        self.hw_a = self.L_a.clone()
        self.L_b = torch.as_tensor(L0 + nd - 1, device=dev)
        self.hw_b = self.hw_a.clone()
        self.slots_b = torch.empty(B, dtype=torch.int64, device=dev)
        self.q_b = torch.stack([w.draw((B, 1, w.num_q_heads, w.head_dim), l, 120, dev)
                                for l in range(w.num_layers)])
        self.kn_b = torch.stack([w.draw((B, w.num_kv_heads, w.head_dim), l, 121, dev)
                                 for l in range(w.num_layers)])
        self.vn_b = torch.stack([w.draw((B, w.num_kv_heads, w.head_dim), l, 122, dev)
                                 for l in range(w.num_layers)])
        self.out_b = torch.empty_like(self.q_b)
        self.rope = pkv.rope_table(w.sink + w.window).to(dev)
        self.in_names = ["q", "kn", "vn", "bt", "L_a", "hw_a", "q_b", "kn_b", "vn_b", "L_b",
                         "hw_b"]
        self.out_names = ["out", "out_b"]
        self.launches_per_step = 2 * w.num_layers
        self.tokens_per_step = B * (nd + 1)

    # -- the step ---------------------------------------------------------------------------------
    def run(self):
        p, w = self.pkv, self.w
        if self.kind == "ring":
            return self.run_ring_fused()
        if self.kind == "prefix":
            # the copies write the pools the fused call reads: it must not start early
            p.copy_blocks(self.k, self.v, self.cow_src, self.cow_dst)
            prev = p.set_early_start(False)
        for l in range(w.num_layers):
            if self.kind == "fp8":
                p.paged_attn_decode_append_fp8(self.out[l], self.q[l], self.kn[l], self.vn[l],
                                               self.k[l], self.v[l], self.ks[l], self.vs[l],
                                               self.bt, self.cl, w.scale, self.ws)
            else:
                p.paged_attn_decode_append(self.out[l], self.q[l], self.kn[l], self.vn[l],
                                           self.k[l], self.v[l], self.bt, self.cl, w.scale,
                                           self.ws)
        if self.kind == "prefix":
            p.set_early_start(prev)

    def run_ring_fused(self):
        """The streaming step, one launch per layer and phase: the drafts through every layer
        (their rows written to their ring slots and attended causally), the rollback (host
        state: the second phase's lengths), then one more token through every layer."""
        p, w = self.pkv, self.w
        for l in range(w.num_layers):
            p.ring_attn_decode_append(self.out[l], self.q[l], self.kn[l], self.vn[l], self.k[l],
                                      self.v[l], self.bt, self.L_a, self.hw_a, w.sink, w.window,
                                      self.rope, w.scale, self.ws)
        for l in range(w.num_layers):
            p.ring_attn_decode_append(self.out_b[l], self.q_b[l], self.kn_b[l], self.vn_b[l],
                                      self.k[l], self.v[l], self.bt, self.L_b, self.hw_b, w.sink,
                                      w.window, self.rope, w.scale, self.ws)

    def run_ring(self, decode=True, append=True):
        """The same step through separate calls (ring slot mapping, kv_append, ring decode),
        or the decode launches alone."""
        p, w = self.pkv, self.w
        if append:
            p.ring_slot_mapping(self.seq, self.pos, self.bt, w.sink, w.window, w.block_size,
                                out=self.slots)
        for l in range(w.num_layers):
            if append:
                p.kv_append(self.kn[l], self.vn[l], self.slots, self.k[l], self.v[l])
            if decode:
                p.ring_attn_decode(self.out[l], self.q[l], self.k[l], self.v[l], self.bt,
                                   self.L_a, self.hw_a, w.sink, w.window, self.rope, w.scale,
                                   self.ws)
        if append:
            p.ring_slot_mapping(self.seq_b, self.pos_b, self.bt, w.sink, w.window,
                                w.block_size, out=self.slots_b)
        for l in range(w.num_layers):
            if append:
                p.kv_append(self.kn_b[l], self.vn_b[l], self.slots_b, self.k[l], self.v[l])
            if decode:
                p.ring_attn_decode(self.out_b[l], self.q_b[l], self.k[l], self.v[l], self.bt,
                                   self.L_b, self.hw_b, w.sink, w.window, self.rope, w.scale,
                                   self.ws)

    def run_roofline(self):
        """The dominant kernel's launches alone: the fused (or ring) decode launches."""
        if self.kind == "ring":
            return self.run_ring(decode=True, append=False)
        if self.kind == "prefix":
            p, w = self.pkv, self.w
            for l in range(w.num_layers):
                p.paged_attn_decode_append(self.out[l], self.q[l], self.kn[l], self.vn[l],
                                           self.k[l], self.v[l], self.bt, self.cl, w.scale,
                                           self.ws)
            return
        return self.run()

    def roofline_launches(self) -> int:
        return 2 * self.w.num_layers if self.kind == "ring" else self.w.num_layers

    def run_append_only(self):
        """The standalone KV append of the step (slot mapping once, then one append per
        layer): what the fused call replaces, timed for comparison."""
        p, w = self.pkv, self.w
        p.slot_mapping(self.seq, self.pos, self.bt, w.block_size, out=self.slots)
        for l in range(w.num_layers):
            p.kv_append(self.kn[l], self.vn[l], self.slots, self.k[l], self.v[l])

    def run_decode_only(self):
        p, w = self.pkv, self.w
        for l in range(w.num_layers):
            if self.kind == "fp8":
                p.paged_attn_decode_fp8(self.out[l], self.q[l], self.k[l], self.v[l],
                                        self.ks[l], self.vs[l], self.bt, self.cl, w.scale,
                                        self.ws)
            else:
                p.paged_attn_decode(self.out[l], self.q[l], self.k[l], self.v[l], self.bt,
                                    self.cl, w.scale, self.ws)

    def graph_note(self) -> str:
        n = self.w.num_layers
        if self.kind == "ring":
            return (f"CUDA graph: {n} x ring_attn_decode_append ({self.w.q_len} causal drafts: "
                    "ring slot mapping + append + decode, one launch); rollback 2; "
                    f"{n} x ring_attn_decode_append (1 token)")
        if self.kind == "prefix":
            return (f"CUDA graph: copy_blocks (3 copy-on-write copies of the forked children's "
                    f"shared block), {n} x paged_attn_decode_append")
        if self.kind == "fp8":
            return (f"CUDA graph: {n} x paged_attn_decode_append_fp8 "
                    "(slot mapping + E4M3 append + decode, one launch)")
        return (f"CUDA graph: {n} x paged_attn_decode_append "
                "(slot mapping + KV append + decode, one launch)")

    def kernel_note(self) -> str:
        return {"fp8": "decode_kernel, E4M3 cache, fused append (paged_attn_decode_append_fp8)",
                "ring": "decode_kernel, sink + ring with RoPE on read, fused append "
                        "(ring_attn_decode_append)"}.get(
            self.kind, "decode_kernel, fused append (paged_attn_decode_append)")


def capture(fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                         # warm the host-side caches outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_repeats(run_block, warmup_block, min_s, clocks=None):
    """Runs warmup_block() once, then run_block() (one block of --steps steps) repeatedly,
    back to back, until at least min_s seconds of GPU time have passed (at least 3 repeats),
    timing each repeat with CUDA events on the current stream. Returns (median repeat
    seconds, repeats, total seconds, clocks)."""
    warmup_block()
    torch.cuda.synchronize()
    replicas.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    run_block()                      # sizes the repeat count (not reported)
    t1.record()
    t1.synchronize()
    once = max(t0.elapsed_time(t1) / 1e3, 1e-6)
    n = max(3, math.ceil(min_s / once))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    if clocks is not None:
        clocks.start()
    ev[0].record()
    for i in range(n):
        run_block()
        ev[i + 1].record()
    ev[-1].synchronize()
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks is not None else None
    replicas.barrier()
    per = [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(n)]
    return statistics.median(per), n, sum(per), clk


def time_graph(g, steps, warmup, min_s, clocks=None):
    def block(k=steps):
        for _ in range(k):
            g.replay()
    return time_repeats(block, lambda: block(warmup), min_s, clocks)


def traffic_record(w):
    """DRAM bytes per decode launch from a committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"paged_decode_{w.name}.traffic.json")
    src = os.path.join(ROOT, "paged_kv_cache_147_gb300", "csrc", "pkv_decode.cu")
    try:
        rec = json.load(open(path))
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if rec.get("source_sha256_16") == digest:
            return rec.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def measure_e2e(st, step_graph, args, bytes_step, dev, local_rank):
    """The step through the public API with its host traffic: every step copies its inputs from
    pinned host memory to the device and reads its attention output back. Measured twice:
    serially on one stream, and as a serving loop would run it, double-buffered (step i+1's
    inputs go up and step i's output comes down on copy streams while step i's kernels run).
    Both are timed over the same repeated blocks of --steps steps as the device figure; the
    pipelined figure is the reported value, the serial one is kept beside it."""
    ins = [getattr(st, n) for n in st.in_names]
    outs = [getattr(st, n) for n in st.out_names]
    host_in = [t.cpu().pin_memory() for t in ins]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])

    # serial: copy in, step, copy out, one stream
    def serial(n):
        for _ in range(n):
            for d, h in zip(ins, host_in):
                d.copy_(h, non_blocking=True)
            step_graph.replay()
            for h, d in zip(host_out[0], outs):
                h.copy_(d, non_blocking=True)

    s_med, s_rep, _, _ = time_repeats(lambda: serial(args.steps), lambda: serial(args.warmup),
                                      args.min_seconds)

    # double-buffered: a second set of input / output buffers (same pools and workspace) and
    # its own graph; the copy streams overlap the other set's kernels
    st2 = _copy.copy(st)
    for name in st.in_names + st.out_names:
        setattr(st2, name, getattr(st, name).clone())
    sets = [st, st2]
    graphs = [step_graph, capture(st2.run)]
    comp, cin, cout = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def upload(sidx):
        with torch.cuda.stream(cin):
            for n, h in zip(st.in_names, host_in):
                getattr(sets[sidx], n).copy_(h, non_blocking=True)
            ev_in[sidx].record(cin)

    def pipelined(n):
        main = torch.cuda.current_stream()
        for sm in (comp, cin, cout):
            sm.wait_stream(main)
        upload(0)
        for i in range(n):
            sidx = i & 1
            comp.wait_event(ev_in[sidx])      # this step's inputs are on the device
            comp.wait_event(ev_out[sidx])     # step i-2's output has left this set's buffer
            with torch.cuda.stream(comp):
                graphs[sidx].replay()
                ev_comp[sidx].record(comp)
            if i + 1 < n:
                cin.wait_event(ev_comp[1 - sidx])   # step i-1 no longer reads the other set
                upload(1 - sidx)
            cout.wait_event(ev_comp[sidx])
            with torch.cuda.stream(cout):
                for h, name in zip(host_out[sidx], st.out_names):
                    h.copy_(getattr(sets[sidx], name), non_blocking=True)
                ev_out[sidx].record(cout)
        for sm in (comp, cin, cout):
            main.wait_stream(sm)

    clocks = ClockSampler(local_rank)
    p_med, p_rep, _, clk = time_repeats(lambda: pipelined(args.steps),
                                        lambda: pipelined(args.warmup), args.min_seconds, clocks)
    p_el, p_bytes = replicas.aggregate(p_med, float(bytes_step) * args.steps, device=dev)
    s_el, s_bytes = replicas.aggregate(s_med, float(bytes_step) * args.steps, device=dev)
    return {"value": round(p_bytes / p_el / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(p_el / args.steps * 1e3, 4), "repeats": p_rep,
            "serial_value": round(s_bytes / s_el / 1e9, 2),
            "serial_ms_per_step": round(s_el / args.steps * 1e3, 4), "serial_repeats": s_rep,
            "clocks": clk,
            "path": "pinned host inputs -> device, C-ABI step (graph replay), attention output "
                    "-> pinned host; double-buffered: step i+1's inputs and step i's output "
                    "move on copy streams during step i (serial_value: one stream, no overlap)"}


def measure_workload(args, w, local_rank, world_size, kv="fp16"):
    """Every figure of one workload: the step, the dominant kernel's roofline, the standalone
    decode and append, and the end-to-end step."""
    dev = f"cuda:{local_rank}"
    from paged_kv_cache_147_gb300 import pkv
    st = Step(w, dev, kv=kv)
    step_graph = capture(st.run)
    steps, min_s = args.steps, args.min_seconds

    clocks = ClockSampler(local_rank)
    med, reps, _, clk = time_graph(step_graph, steps, args.warmup, min_s, clocks)
    bytes_step = step_bytes(w, kv)
    t_max, total_bytes = replicas.aggregate(med, float(bytes_step) * steps, device=dev)
    value = total_bytes / t_max / 1e9

    # dominant kernel: the decode launches. For the paged workloads they are the whole step
    # (the fused ones each overlapping the previous one's tail), so their average launch
    # duration is the step time over the launches. The prefix step also holds the copy-on-write
    # copies, the ring step its slot mappings and appends: there the decode launches are timed
    # alone. The prefix roofline counts the distinct block rows (the shared prefix once).
    nroof = st.roofline_launches()
    if st.kind in ("fused", "fp8", "ring"):
        per_launch = (t_max / steps) / nroof
    else:
        roof_graph = capture(st.run_roofline)
        r_med, _, _, _ = time_graph(roof_graph, steps, args.warmup, min_s / 2)
        per_launch = r_med / steps / nroof
    if w.name.startswith("prefix"):
        bytes_launch = unique_bytes(w) / w.num_layers
    else:
        bytes_launch = bytes_step / nroof
    peak, peak_kind = load_peaks()
    achieved = bytes_launch / per_launch / 1e9
    traffic = traffic_record(w) if kv == "fp16" else None

    extra = {}
    if st.kind in ("fused", "fp8", "prefix"):
        dg = capture(st.run_decode_only)
        d_med, _, _, _ = time_graph(dg, steps, args.warmup, min_s / 4)
        extra["unfused_decode_launch_us"] = round(d_med / steps / w.num_layers * 1e6, 3)
    if st.kind == "ring":
        ug = capture(st.run_ring)
        u_med, _, _, _ = time_graph(ug, steps, args.warmup, min_s / 4)
        extra["unfused_step_ms"] = round(u_med / steps * 1e3, 4)
        dg = capture(lambda: st.run_ring(decode=True, append=False))
        d_med, _, _, _ = time_graph(dg, steps, args.warmup, min_s / 4)
        extra["unfused_decode_launch_us"] = round(d_med / steps / nroof * 1e6, 3)
    if st.kind in ("fused", "prefix"):
        ag = capture(st.run_append_only)
        a_med, _, _, _ = time_graph(ag, steps, args.warmup, min_s / 4)
        extra["standalone_kv_append_launch_us"] = round(a_med / steps / w.num_layers * 1e6, 3)

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(st, step_graph, args, bytes_step, dev, local_rank)
    dev_err = pkv.device_error(clear=True)
    if dev_err:
        raise RuntimeError(f"device error word {dev_err:#x} after the {w.name} benchmark")

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world_size,
        "steps": steps, "warmup": args.warmup, "repeats": reps,
        "ms_per_step": round(t_max / steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 K/V, f16 q/out" if kv == "fp8" else "f16", "data": "synthetic",
        "config": describe(w, kv) | {"graph": st.graph_note(), "kv": kv,
                                     "parallelism": f"replicas x{world_size}",
                                     "timing": f"median of {reps} repeats of {steps} graph "
                                               f"replays (>= {min_s:g} s of GPU time)"},
        "decode_tokens_per_s": round(st.tokens_per_step * steps * world_size / t_max, 1),
        "pct_of_nominal_8tbs": round(100 * value / world_size / NOMINAL_HBM_GBS, 2),
        f"pct_of_{peak_kind}_hbm": round(100 * value / world_size / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": st.kernel_note(),
                     "launch_us": round(per_launch * 1e6, 3),
                     "algorithmic_bytes_per_launch": int(bytes_launch),
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)", **extra},
        "e2e": e2e,
        "gpu_launches": st.launches_per_step * steps * reps,
        "clocks": clk,
    }
    if w.name.startswith("prefix"):
        ub = unique_bytes(w)
        line["unique_kv_bytes_per_step"] = ub
        line["unique_gbs"] = round(ub * steps * world_size / t_max / 1e9, 2)
        line["cow_copy_bytes_per_step"] = st.cow_bytes
    del st, step_graph
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


class PrefillStep:
    """One chunked-prefill step: per layer the chunk's K/V rows are appended (slot mapping once,
    then kv_append) and the chunk attends causally over the paged cache (paged_prefill)."""

    def __init__(self, w, dev):
        from paged_kv_cache_147_gb300 import pkv
        self.pkv, self.w, self.dev = pkv, w, dev
        self.k, self.v = w.pools(dev)
        self.bt = torch.as_tensor(w.block_tables, device=dev)
        self.cl = torch.as_tensor(w.context_lens, device=dev)
        seq, pos = w.new_token_positions()
        self.seq = torch.as_tensor(seq, device=dev)
        self.pos = torch.as_tensor(pos, device=dev)
        self.slots = torch.empty(seq.shape[0], dtype=torch.int64, device=dev)
        self.q = torch.stack([w.query(l, dev) for l in range(w.num_layers)])
        kv_rows = [w.new_kv(l, dev) for l in range(w.num_layers)]
        self.kn = torch.stack([a for a, _ in kv_rows])
        self.vn = torch.stack([b for _, b in kv_rows])
        self.out = torch.empty_like(self.q)
        self.in_names = ["q", "kn", "vn", "bt", "cl", "seq", "pos"]
        self.out_names = ["out"]

    def run(self):
        p, w = self.pkv, self.w
        p.slot_mapping(self.seq, self.pos, self.bt, w.block_size, out=self.slots)
        for l in range(w.num_layers):
            p.kv_append(self.kn[l], self.vn[l], self.slots, self.k[l], self.v[l])
            p.paged_prefill(self.out[l], self.q[l], self.k[l], self.v[l], self.bt, self.cl,
                            w.scale)

    def run_roofline(self):
        p, w = self.pkv, self.w
        for l in range(w.num_layers):
            p.paged_prefill(self.out[l], self.q[l], self.k[l], self.v[l], self.bt, self.cl,
                            w.scale)


def measure_prefill(args, w, local_rank, world_size):
    """The chunked-prefill step (NEXT row of the hot path): TFLOP/s of the causal attention
    over the paged cache, with the prefill kernel's roofline against the tensor-core peak."""
    dev = f"cuda:{local_rank}"
    from paged_kv_cache_147_gb300 import pkv
    st = PrefillStep(w, dev)
    g = capture(st.run)
    steps, min_s = args.steps, args.min_seconds
    clocks = ClockSampler(local_rank)
    med, reps, _, clk = time_graph(g, steps, args.warmup, min_s, clocks)
    flops = prefill_flops(w)
    t_max, total = replicas.aggregate(med, float(flops) * steps, device=dev)
    value = total / t_max / 1e12
    rg = capture(st.run_roofline)
    r_med, _, _, _ = time_graph(rg, steps, args.warmup, min_s / 2)
    per_launch = r_med / steps / w.num_layers
    achieved = flops / w.num_layers / per_launch / 1e12
    burst, sustained, kind = load_tensor_peak()
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(st, g, args, flops, dev, local_rank)
        for key in ("value", "serial_value"):
            e2e[key] = round(e2e[key] * 1e9 / 1e12, 2)      # measured as flops / s / 1e9
        e2e["unit"] = "TFLOP/s"
    dev_err = pkv.device_error(clear=True)
    if dev_err:
        raise RuntimeError(f"device error word {dev_err:#x} after the prefill benchmark")
    line = {
        "metric": "chunked-prefill paged attention TFLOP/s (causal, f16 in, f32 accumulate)",
        "value": round(value, 2), "unit": "TFLOP/s", "steps": steps, "warmup": args.warmup,
        "repeats": reps, "ms_per_step": round(t_max / steps * 1e3, 4),
        "dtype": "f16", "config": {
            "workload": w.name, "layers": w.num_layers, "num_seqs": w.num_seqs,
            "chunk_q_len": w.q_len, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size,
            "context_after_chunk": [int(w.context_lens.min()), int(w.context_lens.max())],
            "flops_per_step": flops,
            "graph": f"CUDA graph: slot_mapping, {w.num_layers} x (kv_append + paged_prefill)",
            "timing": f"median of {reps} repeats of {steps} graph replays (>= {min_s:g} s)"},
        "chunk_tokens_per_s": round(w.num_seqs * w.q_len * steps * world_size / t_max, 1),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": sustained,
                     "unit": "TFLOP/s", "frac": round(achieved / sustained, 4),
                     "frac_of_burst_peak": round(achieved / burst, 4), "traffic": None,
                     "kernel": "prefill_kernel (paged_prefill, tcgen05.mma kind::f16)",
                     "launch_us": round(per_launch * 1e6, 3),
                     "algorithmic_flops_per_launch": flops // w.num_layers,
                     "peak_kind": f"{kind} bf16 dense, sustained (timed inside a seconds-long "
                                  "loop; f16 = bf16 rate); frac_of_burst_peak against "
                                  f"{burst:g}"},
        "e2e": e2e,
        "gpu_launches": (1 + 2 * w.num_layers) * steps * reps,
        "clocks": clk,
    }
    del st, g, rg
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def measure_spec_verify(args, local_rank, B=32, K=4, V=32000, seed=6):
    """Speculative-draft verification beside the ring decode: B sequences, K drafts each, a
    V-token vocabulary (fp32 logits of the target at K + 1 positions and of the draft at K);
    GB/s of logits read per call."""
    from paged_kv_cache_147_gb300 import pkv
    dev = f"cuda:{local_rank}"
    g0 = torch.Generator(device=dev)
    g0.manual_seed(seed)
    t = torch.randn((B, K + 1, V), generator=g0, device=dev) * 2
    d = (t[:, :K] + 0.3 * torch.randn((B, K, V), generator=g0, device=dev)).contiguous()
    x = torch.randint(0, V, (B, K), generator=g0, device=dev, dtype=torch.int32)
    ua = torch.rand((B, K), generator=g0, device=dev)
    us = torch.rand(B, generator=g0, device=dev)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    nt = torch.empty_like(n)
    g = capture(lambda: pkv.spec_verify(t, d, x, ua, us, n, nt))
    clocks = ClockSampler(local_rank)
    med, reps, _, clk = time_graph(g, args.steps, args.warmup, args.min_seconds, clocks)
    per = med / args.steps
    nbytes = (t.numel() + d.numel()) * 4
    peak, kind = load_peaks()
    dev_err = pkv.device_error(clear=True)
    if dev_err:
        raise RuntimeError(f"device error word {dev_err:#x} after the spec_verify benchmark")
    return {"metric": "speculative verify: logits GB/s", "value": round(nbytes / per / 1e9, 2),
            "unit": "GB/s", "steps": args.steps, "repeats": reps,
            "us_per_call": round(per * 1e6, 3), "dtype": "f32",
            "config": {"workload": "spec_verify", "num_seqs": B, "drafts": K, "vocab": V,
                       "logit_bytes_per_call": nbytes,
                       "l2": "no flush: the 37 MB of logits fit in L2; reported for the kernel's "
                             "own speed, not as an HBM measurement"},
            "roofline": {"bound": "hbm", "achieved": round(nbytes / per / 1e9, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(nbytes / per / 1e9 / peak, 4),
                         "kernel": "spec_verify_kernel (one cluster of CTAs per sequence)",
                         "peak_kind": f"{kind} (MEASURED_PEAKS.json hbm_gbs)"},
            "gpu_launches": args.steps * reps, "clocks": clk}


def run_ours(args, w, rank, local_rank, world_size):
    torch.cuda.set_device(local_rank)
    from paged_kv_cache_147_gb300 import pkv
    pkv.load()
    if w.name == "prefill_70b":
        line = measure_prefill(args, w, local_rank, world_size)
    else:
        line = measure_workload(args, w, local_rank, world_size, args.kv)
    also = [] if args.also in ("", "none") else [x for x in args.also.split(",") if x]
    per = []
    for name in also:
        if name == w.name or name not in ALL_WORKLOADS:
            continue
        if args.kv == "fp8" and name in ("prefix", "ring", "prefill_70b", "spec_verify"):
            continue
        gc.collect()
        torch.cuda.empty_cache()
        if name == "spec_verify":
            per.append(measure_spec_verify(args, local_rank))
            continue
        wx = make_workload(name, args.layers)
        if name == "prefill_70b":
            entry = measure_prefill(args, wx, local_rank, world_size)
            per.append(entry)
            continue
        entry = measure_workload(args, wx, local_rank, world_size, args.kv)
        for key in ("metric", "n_gpus", "higher_is_better", "scaling", "data", "vs_baseline"):
            entry.pop(key, None)
        per.append(entry)
    if per:
        line["per_workload"] = per
        line["gpu_launches_all_workloads"] = line["gpu_launches"] + sum(
            e["gpu_launches"] for e in per)
    return line


# ------------------------------------------------------------------------------ CPU oracle
_HOST_LAYERS = {}


def _host_layer(w, l):
    """Host copies of one layer's inputs, drawn once and reused (the oracle's append writes
    the same slots every step, so reuse does not change the work)."""
    if l not in _HOST_LAYERS:
        k, v = (t.numpy() for t in w.layer_pool(l))
        kn, vn = (t.numpy() for t in w.new_kv(l))
        _HOST_LAYERS[l] = (k, v, w.query(l).numpy(), kn, vn)
    return _HOST_LAYERS[l]


def oracle_sample(w, seqs, layers):
    """Runs the oracle's append + attention over `seqs` of each of `layers`; returns
    (seconds, kv bytes attended, threads used)."""
    import oracle
    secs, nbytes, threads = 0.0, 0, 1
    mask = np.zeros(w.num_seqs, dtype=np.uint8)
    mask[list(seqs)] = 1
    seq_ids, pos = w.new_token_positions()
    for l in layers:
        k, v, q, kn, vn = _host_layer(w, l)
        sel = np.isin(seq_ids, np.nonzero(mask)[0])
        t0 = time.perf_counter()
        slots = oracle.slot_mapping(seq_ids[sel], pos[sel], w.block_tables, w.block_size)
        oracle.kv_append(kn[sel], vn[sel], slots, k, v, w.block_size)
        _, threads = oracle.paged_attention(q, k, v, w.block_tables, w.context_lens,
                                            w.block_size, w.scale, seq_mask=mask,
                                            return_threads=True)
        secs += time.perf_counter() - t0
        nbytes += int(w.context_lens[mask.astype(bool)].astype(np.int64).sum()) * \
            w.num_kv_heads * w.head_dim * 4
    return secs, nbytes, threads


def cpu_baseline(w, budget_s, max_layers=4):
    """The oracle as it stands on all host cores: whole layers of the workload (all sequences,
    append + fp64 attention), cycling over its first max_layers layers (host copies of every
    layer of the 80-layer batches would not fit the host's memory) for about budget_s."""
    import oracle
    oracle.build()
    nl = min(w.num_layers, max_layers)
    secs, nbytes, threads = oracle_sample(w, range(w.num_seqs), [0])
    layers = 1   # layer evaluations
    while secs * (layers + 1) / layers < budget_s:
        s, b, threads = oracle_sample(w, range(w.num_seqs), [layers % nl])
        secs, nbytes, layers = secs + s, nbytes + b, layers + 1
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{layers} layer evaluations cycling over layers 0-{nl - 1} of "
                      f"{w.name}, all {w.num_seqs} sequences (append + fp64 attention), "
                      f"{secs:.1f} s"}


def run_reference(args, w, world_size):
    import oracle
    oracle.build()
    # calibrate: one sequence-sized unit of work, then size each step to fit the budget
    budget = 150.0 / max(1, args.steps + args.warmup)
    probe_s, _, _ = oracle_sample(w, range(min(4, w.num_seqs)), [0])
    per_seq = probe_s / min(4, w.num_seqs)
    n = int(max(1, min(w.num_seqs, budget / max(per_seq, 1e-6))))
    rng = np.random.default_rng(0)
    secs, nbytes, threads = 0.0, 0, 1
    for i in range(args.warmup + args.steps):
        seqs = rng.choice(w.num_seqs, size=n, replace=False)
        s, b, threads = oracle_sample(w, seqs, [0])
        if i >= args.warmup:
            secs, nbytes = secs + s, nbytes + b
    value = nbytes / secs / 1e9
    sample = (f"each step: {n} random of the {w.num_seqs} sequences of layer 0, "
              "append + fp64 attention")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world_size, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(describe(w), accumulate="f64"),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    rank, local_rank, world_size = replicas.world()
    w = make_workload(args.workload, args.layers)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w, world_size)), flush=True)
        return
    replicas.init()
    line = run_ours(args, w, rank, local_rank, world_size)
    if rank == 0:
        if not args.no_cpu_baseline and w.name != "ring" and args.kv == "fp16":
            line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    replicas.shutdown()


if __name__ == "__main__":
    main()
