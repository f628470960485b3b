#!/usr/bin/env python3
"""Benchmark of the MLA prefill hot path on one GB300 (or N replicas).

Metric: prefill query tokens per second per layer (one attention call over
all new tokens of the workload), with attention TFLOP/s and the fraction of
the measured tensor-core peak. Default workload: dense causal MLA prefill of
one 32,768-token prompt, 64 heads (the 16-chunk balanced pairing).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun each rank runs its own replica of the workload (no data-path
collective: the query rows of different prompts are independent); rank 0
prints one JSON line with the whole-job throughput.
"""
from __future__ import annotations

import argparse
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

METRIC = "MLA prefill query tok/s per layer at 32k ctx"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.remove(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
# Pieces the host-to-host dense call cuts the new tokens into (copies of one
# piece overlap the attention of the others).
E2E_PIECES = 32
SPARSE_E2E_PIECES = 8

def host_dense(w):
    from mla_prefill_attention_gb300 import inputs as I
    ps = w.seqs()
    q = I.gen_q_bf16(w.seed, ps.total_q, w.heads)
    kv, ks = I.gen_latent_cache(w.seed, ps)
    return ps, q, kv, ks


class DenseRun:
    """One step = one mla_prefill_dense call over every new token."""
    launches_per_step = 1

    def __init__(self, w, dev):
        import torch
        from mla_prefill_attention_gb300 import MLA_OP_DENSE, Seqs, mla_workspace_size
        from mla_prefill_attention_gb300 import flops as F
        self.w = w
        self.ps, q, kv, ks = host_dense(w)
        self.host = {"q": q, "kv": kv, "ks": ks}
        self.seqs = Seqs.from_paged(self.ps, device=dev)
        self.q = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(dev)
        self.kv = torch.from_numpy(kv).to(dev)
        self.ks = torch.from_numpy(ks).to(dev)
        T, H = self.ps.total_q, w.heads
        self.out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.ws = torch.empty(max(16, mla_workspace_size(MLA_OP_DENSE, self.seqs, H)), dtype=torch.uint8, device=dev)
        self.tokens = T
        self.flops = F.dense_flops(w.q_lens, w.prefix_lens, H)
        self.min_bytes = F.dense_min_bytes(T, H, sum(self.ps.seq_len(b) for b in range(self.ps.batch)))

    def step(self):
        from mla_prefill_attention_gb300 import mla_prefill_dense
        mla_prefill_dense(self.seqs, self.q, self.kv, self.ks, self.w.sm_scale, out=self.out, lse=self.lse,
                          workspace=self.ws)

    e2e_pieces = E2E_PIECES

    def e2e(self, steps, warmup):
        """The host-to-host call (mla_prefill_dense_host): inputs in pinned host
        memory, the cache and the queries (in E2E_PIECES pieces) copied in,
        attention, out and lse copied back, the copies overlapped with the
        attention of other pieces; all of it inside the timed region."""
        import torch
        from mla_prefill_attention_gb300 import MLA_OP_DENSE_HOST, mla_prefill_dense_host, mla_workspace_size
        hq = torch.from_numpy(self.host["q"].view(np.int16)).view(torch.bfloat16).pin_memory()
        hkv = torch.from_numpy(self.host["kv"]).pin_memory()
        hks = torch.from_numpy(self.host["ks"]).pin_memory()
        hout = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        hlse = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()
        ws = torch.empty(max(16, mla_workspace_size(MLA_OP_DENSE_HOST, self.seqs, self.w.heads)), dtype=torch.uint8,
                         device=self.q.device)

        def one():
            mla_prefill_dense_host(self.seqs, hq, hkv, hks, self.w.sm_scale, self.q, self.kv, self.ks, hout, self.out,
                                   lse_host=hlse, lse=self.lse, n_chunks=E2E_PIECES, workspace=ws)

        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            one()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        h2d = hq.numel() * 2 + hkv.numel() + hks.numel() * 4
        d2h = hout.numel() * 2 + hlse.numel() * 4
        return ms, h2d, d2h

    def oracle_rate(self, budget_s: float, seed: int = 0):
        """Oracle (fp64 CPU) on a bounded sample of query tokens, all heads:
        returns (sampled tokens, seconds, sampled algorithmic FLOPs)."""
        from oracle import oracle as O
        from mla_prefill_attention_gb300 import flops as F
        ps, h = self.ps, self.host
        T = ps.total_q
        rng = np.random.default_rng(seed)

        def flops_of(toks):
            tot = 0
            for t in toks:
                b = int(np.searchsorted(ps.cu_seqlens_q, t, side="right") - 1)
                pos = int(ps.prefix_lens[b]) + int(t) - int(ps.cu_seqlens_q[b])
                tot += (pos + 1) * self.w.heads * F.FLOPS_PER_PAIR_HEAD
            return tot

        probe = np.array([rng.integers(0, T)])
        t0 = time.perf_counter()
        O.mla_dense(ps, h["q"][probe], probe, h["kv"], h["ks"], self.w.sm_scale)
        dt = max(time.perf_counter() - t0, 1e-3)
        rate = flops_of(probe) / dt
        n = 1
        while n < T and flops_of(rng.integers(0, T, n * 2)) / rate < budget_s:
            n *= 2
        toks = np.sort(rng.integers(0, T, n))
        t0 = time.perf_counter()
        O.mla_dense(ps, h["q"][toks], toks, h["kv"], h["ks"], self.w.sm_scale)
        dt = time.perf_counter() - t0
        return len(toks), dt, flops_of(toks)


class SparseRun:
    """One step = mla_indexer_topk + mla_prefill_sparse over every new token."""
    launches_per_step = 2

    def __init__(self, w, dev):
        import torch
        from mla_prefill_attention_gb300 import MLA_OP_INDEXER, Seqs, inputs as I, mla_workspace_size
        from mla_prefill_attention_gb300 import flops as F
        self.w = w
        self.ps = w.seqs()
        q = I.gen_q_bf16(w.seed, self.ps.total_q, w.heads)
        kv, ks = I.gen_latent_cache(w.seed, self.ps)
        qi, wh, ki, kis = I.gen_indexer_inputs(w.seed, self.ps)
        self.host = dict(q=q, kv=kv, ks=ks, qi=qi, w=wh, ki=ki, kis=kis)
        self.seqs = Seqs.from_paged(self.ps, device=dev)
        self.d = {k: torch.from_numpy(v).to(dev) for k, v in self.host.items() if k != "q"}
        self.d["q"] = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(dev)
        T, H = self.ps.total_q, w.heads
        self.out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.idx = torch.empty((T, w.topk), dtype=torch.int32, device=dev)
        self.ws = torch.empty(mla_workspace_size(MLA_OP_INDEXER, self.seqs, 64, w.topk), dtype=torch.uint8,
                              device=dev)
        self.tokens = T
        self.indexer_flops = F.indexer_flops(w.q_lens, w.prefix_lens)
        self.sparse_flops = F.sparse_flops(w.q_lens, w.prefix_lens, H, w.topk)
        self.sparse_gathered_bytes = F.sparse_gathered_bytes(w.q_lens, w.prefix_lens, w.topk)
        self.flops = self.sparse_flops + self.indexer_flops
        self.min_bytes = None
        self.mid = []          # events between the two calls, one per step, when recording

    def step(self):
        import torch
        from mla_prefill_attention_gb300 import mla_indexer_topk, mla_prefill_sparse
        d = self.d
        mla_indexer_topk(self.seqs, d["qi"], d["w"], 0, d["ki"], d["kis"], self.w.topk, idx_out=self.idx,
                         workspace=self.ws)
        if self.mid is not None:
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            self.mid.append(e)
        mla_prefill_sparse(self.seqs, d["q"], d["kv"], d["ks"], self.w.sm_scale, self.idx, out=self.out, lse=self.lse)

    e2e_pieces = SPARSE_E2E_PIECES

    def e2e(self, steps, warmup):
        """The host-to-host sparse step (mla_prefill_sparse_host): every input in
        pinned host memory, the weights and caches copied in, then qi and q in
        SPARSE_E2E_PIECES pieces, each piece's indexer, top-k and sparse attention
        as its rows arrive, and its output, lse and selected indices copied back,
        the copies overlapped with the kernels of other pieces; all of it inside
        the timed region."""
        import torch
        from mla_prefill_attention_gb300 import mla_prefill_sparse_host
        h = {k: torch.from_numpy(v).pin_memory() for k, v in self.host.items() if k != "q"}
        h["q"] = torch.from_numpy(self.host["q"].view(np.int16)).view(torch.bfloat16).pin_memory()
        hout = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        hlse = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()
        hidx = torch.empty(self.idx.shape, dtype=torch.int32).pin_memory()
        d = self.d
        host_out = {"out": hout, "lse": hlse, "idx": hidx}
        dev_out = {"out": self.out, "lse": self.lse, "idx": self.idx}

        def one():
            mla_prefill_sparse_host(self.seqs, h, d, host_out, dev_out, self.w.sm_scale, w_token_stride=0,
                                    topk=self.w.topk, n_chunks=SPARSE_E2E_PIECES, workspace=self.ws)

        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            one()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        h2d = sum(t.numel() * t.element_size() for t in h.values())
        d2h = hout.numel() * 2 + hlse.numel() * 4 + hidx.numel() * 4
        return ms, h2d, d2h

    def oracle_rate(self, budget_s, seed=0):
        from oracle import oracle as O
        h, ps = self.host, self.ps
        rng = np.random.default_rng(seed)
        n = 1
        t_total, done, fl = 0.0, 0, 0
        while t_total < budget_s and done < ps.total_q:
            toks = np.sort(rng.integers(0, ps.total_q, n))
            t0 = time.perf_counter()
            idx = O.indexer_topk(ps, h["qi"][toks], h["w"], 0, toks, h["ki"], h["kis"], self.w.topk)
            O.mla_sparse(ps, h["q"][toks], toks, h["kv"], h["ks"], self.w.sm_scale, idx)
            t_total += time.perf_counter() - t0
            done += n
            n *= 2
        return done, t_total, done * (self.flops / ps.total_q)


class ChunkedRun:
    """One step = the whole chunked prefill of a long prompt through the
    library's chunk driver (chunked_prefill_sparse): for every chunk,
    mla_indexer_topk + mla_prefill_sparse after the cached prefix of the earlier
    chunks. Every chunk's queries are resident in HBM before timing. Also times
    the dense path on the final chunk (reported beside the step)."""

    def __init__(self, w, dev):
        import torch
        from mla_prefill_attention_gb300 import MLA_OP_DENSE, MLA_OP_INDEXER, chunk_bounds, chunk_seqs, inputs as I
        from mla_prefill_attention_gb300 import mla_workspace_size
        from mla_prefill_attention_gb300 import flops as F
        self.w, self.dev = w, dev
        self.ps = w.seqs()
        N = w.q_lens[0]
        kv, ks = I.gen_latent_cache(w.seed, self.ps)
        ki, kis = I.gen_indexer_keys(w.seed, self.ps)
        wh = I.gen_indexer_w(w.seed)
        self.host = dict(kv=kv, ks=ks, ki=ki, kis=kis, w=wh)
        self.d = {k: torch.from_numpy(v).to(dev) for k, v in self.host.items()}
        self.bounds = chunk_bounds(N, w.chunk)
        self.seqs = chunk_seqs(self.ps.block_table, self.ps.num_blocks, N, w.chunk, device=dev)
        self.q, self.qi = {}, {}
        for c, (s, e) in enumerate(self.bounds):
            q = I.gen_q_bf16(w.seed, N, w.heads, token_rows=np.arange(s, e))
            self.q[s] = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(dev)
            self.qi[s] = torch.from_numpy(I.gen_indexer_q(w.seed, N, token_rows=np.arange(s, e))).to(dev)
        max_c = max(e - s for s, e in self.bounds)
        ws = max(mla_workspace_size(MLA_OP_INDEXER, sq, 64, w.topk) for sq in self.seqs)
        ws = max(ws, mla_workspace_size(MLA_OP_DENSE, self.seqs[-1], w.heads), 16)
        H = w.heads
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.out = torch.empty((max_c, H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((max_c, H), dtype=torch.float32, device=dev)
        self.idx = torch.empty((max_c, w.topk), dtype=torch.int32, device=dev)
        self.tokens = N
        self.indexer_flops = F.indexer_flops(w.q_lens, w.prefix_lens)
        self.sparse_flops = F.sparse_flops(w.q_lens, w.prefix_lens, H, w.topk)
        self.sparse_gathered_bytes = F.sparse_gathered_bytes(w.q_lens, w.prefix_lens, w.topk)
        self.flops = self.sparse_flops + self.indexer_flops
        self.launches_per_step = 2 * len(self.bounds)
        self.chunk_ms = [0.0] * len(self.bounds)
        self.ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in self.bounds]
        self.min_bytes = None

    def step(self):
        from mla_prefill_attention_gb300 import chunked_prefill_sparse
        d = self.d
        nxt = {"c": None}

        def before(c):
            if c > 0:
                self.ev[c - 1][2].record()
            self.ev[c][0].record()

        chunked_prefill_sparse(self.ps.block_table, self.ps.num_blocks, self.tokens, self.w.chunk,
                               lambda s, e: self.q[s], d["kv"], d["ks"], lambda s, e: self.qi[s], d["w"], 0,
                               d["ki"], d["kis"], self.w.sm_scale, topk=self.w.topk, on_chunk=lambda *a: None,
                               out=self.out, lse=self.lse, idx=self.idx, workspace=self.ws, seqs_list=self.seqs,
                               before_chunk=before, after_indexer=lambda c: self.ev[c][1].record())
        self.ev[-1][2].record()

    def collect_chunk_ms(self):
        """Per-chunk times of the last step, and the two calls' totals over all chunks."""
        self.chunk_ms = [a.elapsed_time(c) for a, _, c in self.ev]
        self.split_total = (sum(a.elapsed_time(m) for a, m, _ in self.ev), sum(m.elapsed_time(c) for _, m, c in self.ev))

    def dense_last_chunk_ms(self, reps=3):
        """The dense path on the final chunk (same inputs), median of reps calls."""
        import torch
        from mla_prefill_attention_gb300 import mla_prefill_dense
        d = self.d
        s, e = self.bounds[-1]
        call = lambda: mla_prefill_dense(self.seqs[-1], self.q[s], d["kv"], d["ks"], self.w.sm_scale,
                                         out=self.out[:e - s], lse=self.lse[:e - s], workspace=self.ws)
        call()
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    def e2e(self, steps, warmup):
        return None

    def oracle_rate(self, budget_s, seed=0):
        """Oracle on random query tokens of random chunks (indexer + sparse),
        extrapolated by algorithmic FLOPs."""
        from oracle import oracle as O
        from mla_prefill_attention_gb300 import inputs as I, flops as F
        h, w = self.host, self.w
        rng = np.random.default_rng(seed)
        t_total, done, fl = 0.0, 0, 0
        while t_total < budget_s and done < 64:
            c = int(rng.integers(0, len(self.bounds)))
            s, e = self.bounds[c]
            t = int(rng.integers(0, e - s))
            sub = I.PagedSeqs(np.array([0, e - s], np.int32), np.array([s], np.int32), self.ps.block_table,
                              self.ps.num_blocks)
            q = I.gen_q_bf16(w.seed, w.q_lens[0], w.heads, token_rows=np.array([s + t]))
            qi = I.gen_indexer_q(w.seed, w.q_lens[0], token_rows=np.array([s + t]))
            t0 = time.perf_counter()
            idx = O.indexer_topk(sub, qi, h["w"], 0, np.array([t]), h["ki"], h["kis"], w.topk)
            O.mla_sparse(sub, q, np.array([t]), h["kv"], h["ks"], w.sm_scale, idx)
            t_total += time.perf_counter() - t0
            done += 1
            ctx = s + t + 1
            fl += min(ctx, w.topk) * w.heads * F.FLOPS_PER_PAIR_HEAD + ctx * F.H_IDX * F.D_IDX * 2
        return done, t_total, fl


RUNS = {"tiny512": DenseRun, "prefix12k": DenseRun, "dense32k": DenseRun, "ragged4": DenseRun,
        "sparse64k": SparseRun, "chunked200k": ChunkedRun}


# DRAM bytes (read + written) per launch of the timed kernels, from one ncu capture
# of dram__bytes_read.sum + dram__bytes_write.sum (one pass) on the bench's own
# command line for that workload. A kernel change invalidates its entry: set it to
# None until it is captured again.
TRAFFIC = {
    "dense32k": {"attention": 2455451904 + 2118966016},
    "sparse64k": {"indexer_topk": 75921408 + 25915904,        # the fast-path launch
                  "sparse_attention": 805456128 + 531233536},
}


def max_over_ranks(ms, device=None):
    """The slowest rank's time under torch.distributed (every rank calls it);
    unchanged in a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, tokens_per_rank, steps, total_ms):
    """Whole-job tokens per second: each of the world ranks runs its own replica
    of the workload, tokens_per_rank new tokens per step, in total_ms (the
    slowest rank's time)."""
    return world * tokens_per_rank * steps / (total_ms / 1000.0)


def time_steps(run, steps, warmup):
    import torch
    for _ in range(warmup):
        run.step()
    torch.cuda.synchronize()
    if hasattr(run, "mid"):
        run.mid = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per = []
    e0.record()
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run.step()
        b.record()
        per.append((a, b))
    e1.record()
    torch.cuda.synchronize()
    total_ms = e0.elapsed_time(e1)
    per_ms = [a.elapsed_time(b) for a, b in per]
    if getattr(run, "mid", None):
        run.split_ms = ([a.elapsed_time(m) for (a, _), m in zip(per, run.mid)],
                        [m.elapsed_time(b) for (_, b), m in zip(per, run.mid)])
    return total_ms, per_ms


KV_APPEND_BYTES_PER_TOKEN = 2 * 576 + 2 * 128 + 576 + 4 + 128 + 4   # bf16 rows in, e4m3 rows + fp32 scales out


def measure_kv_append(w, dev, reps=20):
    """The cache write of the workload's new tokens (latent row and indexer key),
    timed alone with CUDA events on the launching stream, L2 flushed before
    every launch. Rows are drawn for up to 8,192 tokens and repeated."""
    import torch
    from mla_prefill_attention_gb300 import Seqs, mla_kv_append
    from mla_prefill_attention_gb300 import inputs as I
    ps = w.seqs()
    T = ps.total_q
    g = min(T, 8192)
    lat = torch.from_numpy(I.gen_new_rows_bf16(w.seed, g, 576).view(np.int16)).to(dev).view(torch.bfloat16)
    kid = torch.from_numpy(I.gen_new_rows_bf16(w.seed, g, 128, I.T_NEWKIDX).view(np.int16)).to(dev)
    kid = kid.view(torch.bfloat16)
    reps_rows = -(-T // g)
    lat = lat.repeat(reps_rows, 1)[:T].contiguous()
    kid = kid.repeat(reps_rows, 1)[:T].contiguous()
    nb = ps.num_blocks
    kv = torch.zeros((nb, 256, 576), dtype=torch.uint8, device=dev)
    ks = torch.zeros((nb, 256), dtype=torch.float32, device=dev)
    ki = torch.zeros((nb, 256, 128), dtype=torch.uint8, device=dev)
    kis = torch.zeros((nb, 256), dtype=torch.float32, device=dev)
    seqs = Seqs.from_paged(ps, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        mla_kv_append(seqs, lat, kv, ks, kid, ki, kis)
    torch.cuda.synchronize()
    ev = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        mla_kv_append(seqs, lat, kv, ks, kid, ki, kis)
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    pk, src = peaks()
    gbs = T * KV_APPEND_BYTES_PER_TOKEN / (ms / 1000.0) / 1e9
    return {"tokens": T, "ms": ms, "tokens_per_s": T / (ms / 1000.0),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(pk["hbm_gbs"]), "unit": "GB/s",
                         "frac": gbs / float(pk["hbm_gbs"]), "traffic": None,
                         "bytes_per_token": KV_APPEND_BYTES_PER_TOKEN,
                         "peak_source": f"{src} hbm_gbs (copy, burst)",
                         "kernel": "kv_append_kernel: four tokens per warp, bf16 rows -> e4m3 + fp32 scale, "
                                   "L2 flushed before each launch"}}


MERGE_BYTES_PER_ROW_PART = 512 * 2 + 4    # one part's bf16 row and its lse


def measure_merge(w, dev, n_parts=2, reps=20):
    """The log-sum-exp merge of n_parts partial results of the workload's shape
    (all new tokens x heads rows of 512), timed alone with CUDA events, L2
    flushed before every launch."""
    import torch
    from mla_prefill_attention_gb300 import mla_merge_attn
    rows = w.seqs().total_q * w.heads
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    outs = [torch.randn((rows, 512), generator=g, device=dev).to(torch.bfloat16) for _ in range(n_parts)]
    lses = [torch.rand((rows,), generator=g, device=dev) * 20.0 for _ in range(n_parts)]
    out = torch.empty_like(outs[0])
    lse = torch.empty_like(lses[0])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        mla_merge_attn(outs, lses, out=out, lse=lse)
    torch.cuda.synchronize()
    ev = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        mla_merge_attn(outs, lses, out=out, lse=lse)
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    pk, src = peaks()
    nbytes = rows * MERGE_BYTES_PER_ROW_PART * (n_parts + 1)
    gbs = nbytes / (ms / 1000.0) / 1e9
    return {"rows": rows, "parts": n_parts, "ms": ms,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(pk["hbm_gbs"]), "unit": "GB/s",
                         "frac": gbs / float(pk["hbm_gbs"]), "traffic": None,
                         "bytes_per_row": MERGE_BYTES_PER_ROW_PART * (n_parts + 1),
                         "peak_source": f"{src} hbm_gbs (copy, burst)",
                         "kernel": "merge_kernel: one warp per 512-value row, fp32 weights, bf16 out; "
                                   "L2 flushed before each launch"}}


def config_of(w):
    c = {"workload": w.name, "batch": len(w.q_lens), "q_lens": w.q_lens, "prefix_lens": w.prefix_lens,
         "heads": w.heads, "d_qk": 576, "d_v": 512, "page": 256, "q_dtype": "bf16",
         "kv_dtype": "e4m3 + fp32 per-token scale", "sm_scale": "1/sqrt(192)", "parallelism": "replicas",
         "l2": "inputs larger than L2 (no flush needed)" if w.name in ("dense32k", "ragged4", "sparse64k",
                                                                       "prefix12k", "chunked200k") else "small inputs"}
    if w.sparse:
        c.update(topk=w.topk, indexer="64 heads x 128, e4m3")
    if w.chunk:
        c.update(chunk=w.chunk)
    return c


def e4m3_peak():
    """Dense e4m3 tensor peak: the measured sustained bf16 figure times the
    nominal e4m3:bf16 ratio of 2 (no e4m3 GEMM is measured)."""
    pk, src = peaks()
    bf16 = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
    return 2.0 * bf16, f"e4m3 dense = 2 x {src} bf16 sustained ({bf16:.1f} TFLOP/s; the nominal e4m3:bf16 ratio)"


def sparse_attention_roof(run, att_ms):
    """Sparse attention against both bounds: the e4m3 tensor roof (its MMAs
    are e4m3) and min(tensor, HBM x AI) with every selected row counted as read
    from HBM (the pessimistic gathered-bytes bound; unique cache rows fit L2)."""
    pk, src = peaks()
    peak, psrc = e4m3_peak()
    tf = run.sparse_flops / (att_ms / 1000.0) / 1e12
    hbm = float(pk["hbm_gbs"])
    ai = run.sparse_flops / run.sparse_gathered_bytes
    roof_ai = min(peak, hbm * ai / 1000.0)
    return {"ms": att_ms, "achieved": tf, "unit": "TFLOP/s", "tensor_peak": peak, "frac_tensor": tf / peak,
            "ai_flop_per_byte": ai, "hbm_gbs": hbm, "hbm_x_ai_roof": roof_ai, "frac_hbm_x_ai": tf / roof_ai,
            "gathered_bytes": run.sparse_gathered_bytes, "traffic": TRAFFIC.get(run.w.name, {}).get("sparse_attention"),
            "peak_source": f"{psrc}; {src} hbm_gbs (copy)",
            "kernel": "attn_f8_kernel<sparse>: tcgen05 e4m3, rows gathered by index"}


def roofline_of(run, per_ms):
    """(attention TFLOP/s, roofline object of the dominant kernel) of a timed run."""
    peak, psrc = e4m3_peak()
    kern_ms = statistics.mean(per_ms)
    tflops = run.flops / (kern_ms / 1000.0) / 1e12
    if isinstance(run, DenseRun):
        roof = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                "traffic": TRAFFIC.get(run.w.name, {}).get("attention"),
                "algorithmic_tflop": run.flops / 1e12, "peak_source": psrc,
                "note": "algorithmic FLOPs (2,176 per visible query-key-head triple) over the e4m3 roof; the kernel "
                        "issues two e4m3 MMAs per algorithmic product (two-term Q and P)",
                "kernel": "attn_f8_kernel: tcgen05 kind::f8f6f4, e4m3 cache tiles by TMA, two-term e4m3 Q and P, "
                          "64 rows x 128 keys"}
        return tflops, roof
    if isinstance(run, SparseRun):
        idx_ms, att_ms = statistics.mean(run.split_ms[0]), statistics.mean(run.split_ms[1])
        traffic = TRAFFIC.get(run.w.name, {}).get("indexer_topk")
        kernel = "indexer_topk_kernel: tcgen05 e4m3 scores, streaming exact top-k in shared memory"
    else:
        run.collect_chunk_ms()
        idx_ms, att_ms = run.split_total
        traffic = None
        kernel = "indexer_topk_kernel over all chunks: tcgen05 e4m3 scores, streaming exact top-k"
    idx_tf = run.indexer_flops / (idx_ms / 1000.0) / 1e12
    roof = {"bound": "tensor", "achieved": idx_tf, "peak": peak, "unit": "TFLOP/s", "frac": idx_tf / peak,
            "traffic": traffic, "peak_source": psrc, "kernel": kernel + ", the larger share of the step",
            "split_ms": {"indexer_topk": idx_ms, "sparse_attention": att_ms},
            "sparse_attention": sparse_attention_roof(run, att_ms)}
    return tflops, roof


def measure_workload(name, dev, steps, warmup, e2e=False):
    """One workload timed on its own (W warm-up steps, then K), for the extra
    objects of the default line: per-step time, throughput and rooflines; with
    e2e, also the same step host to host (the run's e2e method)."""
    import torch
    from mla_prefill_attention_gb300 import inputs as I
    w = I.WORKLOADS[name]
    run = RUNS[name](w, dev)
    total_ms, per_ms = time_steps(run, steps, warmup)
    tflops, roof = roofline_of(run, per_ms)
    obj = {"workload": name, "steps": steps, "warmup": warmup, "ms_per_step": total_ms / steps,
           "value": run.tokens * steps / (total_ms / 1000.0), "unit": "tok/s", "attention_tflops": tflops,
           "roofline": roof, "config": config_of(w)}
    if e2e:
        r = run.e2e(steps, warmup)
        if r is not None:
            ms, h2d, d2h = r
            obj["e2e"] = {"value": run.tokens / (ms / 1000.0), "unit": "tok/s", "ms_per_step": ms,
                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                          "pieces": getattr(run, "e2e_pieces", None)}
    if isinstance(run, ChunkedRun):
        obj["chunks"] = {"count": len(run.bounds), "chunk_tokens": w.chunk,
                         "ms_per_chunk_last_step": [round(x, 3) for x in run.chunk_ms],
                         "total_ms_last_step": round(sum(run.chunk_ms), 3),
                         "dense_last_chunk_ms": run.dense_last_chunk_ms(),
                         "sparse_last_chunk_ms": round(run.chunk_ms[-1], 3)}
    del run
    torch.cuda.empty_cache()
    return obj


def measure_ds_layout(name, dev, steps, warmup):
    """The workload on the 656-byte cache rows (mla_prefill_dense_ds /
    mla_prefill_sparse_ds, the sparse step's indices from mla_indexer_topk
    outside the timed calls): per-call time of the attention alone and its
    roofline against the bf16 tensor peak (these kernels run kind::f16)."""
    import torch
    from mla_prefill_attention_gb300 import (MLA_OP_DENSE_DS, Seqs, inputs as I, mla_indexer_topk, mla_prefill_dense_ds,
                                             mla_prefill_sparse_ds, mla_workspace_size)
    from mla_prefill_attention_gb300 import flops as F
    w = I.WORKLOADS[name]
    ps = w.seqs()
    seqs = Seqs.from_paged(ps, device=dev)
    q = torch.from_numpy(I.gen_q_bf16(w.seed, ps.total_q, w.heads).view(np.int16)).view(torch.bfloat16).to(dev)
    kv = torch.from_numpy(I.gen_latent_cache_ds(w.seed, ps)).to(dev)
    out = torch.empty((ps.total_q, w.heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((ps.total_q, w.heads), dtype=torch.float32, device=dev)
    if w.sparse:
        qi, wh, ki, kis = [torch.from_numpy(x).to(dev) for x in I.gen_indexer_inputs(w.seed, ps)]
        idx = mla_indexer_topk(seqs, qi, wh, 0, ki, kis, w.topk)
        flops = F.sparse_flops(w.q_lens, w.prefix_lens, w.heads, w.topk)
        call = lambda: mla_prefill_sparse_ds(seqs, q, kv, w.sm_scale, idx, out=out, lse=lse)
    else:
        ws = torch.empty(max(256, mla_workspace_size(MLA_OP_DENSE_DS, seqs, w.heads)), dtype=torch.uint8, device=dev)
        flops = F.dense_flops(w.q_lens, w.prefix_lens, w.heads)
        call = lambda: mla_prefill_dense_ds(seqs, q, kv, w.sm_scale, out=out, lse=lse, workspace=ws)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ev = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    pk, src = peaks()
    bf16 = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
    tf = flops / (ms / 1000.0) / 1e12
    obj = {"workload": name, "layout": "656-byte rows (512 e4m3 + 4 fp32 group scales + 64 bf16 RoPE)",
           "steps": steps, "warmup": warmup, "ms_per_call": ms, "value": ps.total_q / (ms / 1000.0),
           "unit": "tok/s", "attention_tflops": tf,
           "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16, "unit": "TFLOP/s", "frac": tf / bf16,
                        "peak_source": f"{src} bf16 sustained (kind::f16 MMAs)",
                        "kernel": "attn_ds kernel: dense rows converted once to f16 and loaded by TMA, sparse rows "
                                  "gathered and converted in shared memory; tcgen05 kind::f16, 64 rows x 80 keys"}}
    del q, kv, out, lse
    torch.cuda.empty_cache()
    return obj


def measure_mha(name, dev, steps, warmup):
    """The non-absorbed (MHA) path on a batch of short prompts (mla_prefill_mha:
    up-projection of every context row's keys and values, then causal attention
    per head), beside the absorbed dense path on the same prompts. FLOPs of the
    MHA path: 2 * 512 * 256 * heads per context row (up-projection) plus
    2 * (192 + 128) per visible (query, key, head) triple (attention)."""
    import torch
    from mla_prefill_attention_gb300 import (MLA_OP_DENSE, MLA_OP_MHA, Seqs, inputs as I, mla_prefill_dense,
                                             mla_prefill_mha, mla_workspace_size)
    from mla_prefill_attention_gb300 import flops as F
    w = I.WORKLOADS[name]
    ps = w.seqs()
    seqs = Seqs.from_paged(ps, device=dev)
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    q = bf(I.gen_q_mha(w.seed, ps.total_q, w.heads))
    wu = bf(I.gen_w_ukv(w.seed, w.heads))
    kv, ks = [torch.from_numpy(x).to(dev) for x in I.gen_latent_cache(w.seed, ps)]
    out = torch.empty((ps.total_q, w.heads, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((ps.total_q, w.heads), dtype=torch.float32, device=dev)
    ws = torch.empty(max(256, mla_workspace_size(MLA_OP_MHA, seqs, w.heads)), dtype=torch.uint8, device=dev)
    qa = bf(I.gen_q_bf16(w.seed, ps.total_q, w.heads))
    outa = torch.empty((ps.total_q, w.heads, 512), dtype=torch.bfloat16, device=dev)
    lsea = torch.empty((ps.total_q, w.heads), dtype=torch.float32, device=dev)
    wsa = torch.empty(max(16, mla_workspace_size(MLA_OP_DENSE, seqs, w.heads)), dtype=torch.uint8, device=dev)

    def timed(call):
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        ev = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call()
            b.record()
            ev.append((a, b))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    ms = timed(lambda: mla_prefill_mha(seqs, q, wu, kv, ks, w.sm_scale, out=out, lse=lse, workspace=ws))
    ms_abs = timed(lambda: mla_prefill_dense(seqs, qa, kv, ks, w.sm_scale, out=outa, lse=lsea, workspace=wsa))
    pairs = sum((p + n) * (p + n + 1) // 2 - p * (p + 1) // 2 for n, p in zip(w.q_lens, w.prefix_lens))
    ctx_rows = sum(n + p for n, p in zip(w.q_lens, w.prefix_lens))
    flops = 2.0 * 512 * 256 * w.heads * ctx_rows + 2.0 * (192 + 128) * w.heads * pairs
    pk, src = peaks()
    bf16 = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
    tf = flops / (ms / 1000.0) / 1e12
    abs_tf = F.dense_flops(w.q_lens, w.prefix_lens, w.heads) / (ms_abs / 1000.0) / 1e12
    obj = {"workload": name, "q_lens": w.q_lens, "heads": w.heads, "steps": steps, "warmup": warmup,
           "ms_per_call": ms, "value": ps.total_q / (ms / 1000.0), "unit": "tok/s", "tflops": tf,
           "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16, "unit": "TFLOP/s", "frac": tf / bf16,
                        "peak_source": f"{src} bf16 sustained (kind::f16 MMAs)",
                        "kernel": "mha up_kernel (M=128 rows x N=256, K=512) + attn_kernel (M=128 tokens, 64-key "
                                  "tiles, d_qk 192, d_v 128), bf16 tcgen05"},
           "absorbed_dense_same_prompts": {"ms_per_call": ms_abs, "value": ps.total_q / (ms_abs / 1000.0),
                                           "attention_tflops": abs_tf}}
    del q, wu, kv, ks, out, lse, ws, qa, outa, lsea, wsa
    torch.cuda.empty_cache()
    return obj


def cpu_info():
    """CPU model and the cores this process may run on (for the CPU baseline)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model", "hardware")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            model = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            model = next((l.split(":", 1)[1].strip() for l in model.splitlines() if l.startswith("Model name")), None)
        except (OSError, subprocess.SubprocessError):
            model = None
    try:
        affinity = len(os.sched_getaffinity(0))
    except AttributeError:
        affinity = os.cpu_count() or 1
    return {"cpu_model": model, "affinity_cores": affinity}


EXTRA_WORKLOADS = ("prefix12k", "ragged4", "sparse64k", "chunked200k")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="dense32k", choices=sorted(RUNS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kv-append", action="store_true", help="skip the separate cache-write measurement")
    ap.add_argument("--no-merge", action="store_true", help="skip the separate partial-result merge measurement")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads' objects")
    args = ap.parse_args()

    from mla_prefill_attention_gb300 import inputs as I
    w = I.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cinfo = cpu_info()
    cores = int(os.environ.get("OMP_NUM_THREADS", cinfo["affinity_cores"]))

    if args.impl == "reference":
        # the reference arm is the fp64 CPU oracle, on rank 0 only
        if rank != 0:
            return
        import __graft_entry__
        from oracle import oracle as O
        O.build()
        run = RUNS[args.workload].__new__(RUNS[args.workload])
        run.w = w
        if RUNS[args.workload] is DenseRun:
            run.ps, q, kv, ks = host_dense(w)
            run.host = {"q": q, "kv": kv, "ks": ks}
        else:
            raise SystemExit(json.dumps({"impl": "reference", "unavailable": "reference arm implemented for dense workloads"}))
        from mla_prefill_attention_gb300 import flops as F
        total_flops = F.dense_flops(w.q_lens, w.prefix_lens, w.heads)
        budget = max(2.0, 120.0 / max(1, args.steps + args.warmup))
        rates, sampled = [], 0
        for i in range(args.warmup + args.steps):
            n, dt, fl = run.oracle_rate(budget, seed=i)
            if i >= args.warmup:
                rates.append(run.ps.total_q / (dt * total_flops / fl))
                sampled += n
        val = statistics.median(rates)
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tok/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * run.ps.total_q / val,
                "extrapolated": True, "sampled_tokens_per_step": sampled // max(1, args.steps),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config_of(w),
                "cpu_baseline": {"value": val, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                 "extrapolated": True, "sampled_tokens_per_step": sampled // max(1, args.steps),
                                 **cinfo,
                                 "sample": f"random query tokens x {w.heads} heads per step (about "
                                           f"{sampled // max(1, args.steps)}), timed, extrapolated by algorithmic "
                                           f"FLOPs to all {run.ps.total_q} tokens"},
                "e2e": {"value": val, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    run = RUNS[args.workload](w, dev)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index if world == 1 else local)
    clocks.start()
    total_ms, per_ms = time_steps(run, args.steps, args.warmup)
    clk = clocks.stop()
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
        dist.barrier()

    ms_per_step = total_ms / args.steps
    value = job_throughput(world, run.tokens, args.steps, total_ms)
    tflops, roof = roofline_of(run, per_ms)
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": config_of(w),
            "attention_tflops": tflops,
            "roofline": roof,
            "gpu_launches": run.launches_per_step * args.steps}
    if clk:
        line["clocks"] = clk
    if isinstance(run, ChunkedRun):
        line["chunks"] = {"count": len(run.bounds), "chunk_tokens": run.w.chunk,
                          "ms_per_chunk_last_step": [round(x, 3) for x in run.chunk_ms],
                          "total_ms_last_step": round(sum(run.chunk_ms), 3),
                          "dense_last_chunk_ms": run.dense_last_chunk_ms(),
                          "sparse_last_chunk_ms": round(run.chunk_ms[-1], 3)}
    if rank == 0 and not args.no_e2e:
        r = run.e2e(args.steps, args.warmup)
        if r:
            ms, h2d, d2h = r
            line["e2e"] = {"value": world * run.tokens / (ms / 1000.0), "unit": "tok/s", "h2d_bytes_per_step": h2d,
                           "d2h_bytes_per_step": d2h}
            if getattr(run, "e2e_pieces", None):
                line["e2e"]["pieces"] = run.e2e_pieces
    if rank == 0 and not args.no_kv_append:
        line["kv_append"] = measure_kv_append(w, dev)
    if rank == 0 and not args.no_merge:
        line["lse_merge"] = measure_merge(w, dev)
    if rank == 0 and not args.no_cpu_baseline:
        n, dt, fl = run.oracle_rate(args.cpu_budget)
        val = run.tokens / (dt * run.flops / fl)
        line["cpu_baseline"] = {"value": val, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                "extrapolated": True, "sampled_tokens": n, **cinfo,
                                "sample": f"{n} random query tokens x all heads of the {w.name} workload "
                                          f"({dt:.1f} s), extrapolated by algorithmic FLOPs"}
    del run
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_extras:
        # the other workloads, each timed on its own outside the headline's timed region
        extras = {}
        for name in EXTRA_WORKLOADS:
            if name == w.name:
                continue
            k = 2 if name == "chunked200k" else min(args.steps, 5)
            extras[name] = measure_workload(name, dev, k, max(3, min(args.warmup, 3)),
                                            e2e=(name == "sparse64k" and not args.no_e2e))
        for name in ("dense32k", "sparse64k"):
            extras[name + "_656B"] = measure_ds_layout(name, dev, min(args.steps, 5), 3)
        extras["mha_short"] = measure_mha("mha_short", dev, min(args.steps, 10), 3)
        line["workloads"] = extras
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
