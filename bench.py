#!/usr/bin/env python
"""Benchmark of the sparse chunked-KV hot path.

One step runs the whole path over one synthetic job of the chosen workload:
chunked prefill of every sequence (chunk attention, window scores, top-B,
compaction into one shared pool), top-K chunk selection, then T static-KV
decode steps (split-KV attention + LSE merge), each one batched call over
every sequence.  The default workload is the batched serving mix: eight
sequences of a 32K prefix with chunk sizes C in {256, 1024, 4096}, the
largest single-GPU workload.  Inputs are resident in HBM before the timed
region; the prefill+selection and the T-step decode loop are each one CUDA
graph replay, bracketed by CUDA events on the launching stream.  L2 is
flushed (256 MiB write) between steps, outside the timed events.

value = decode-step attention throughput (algorithmic TFLOP/s, whole job);
extra keys give the decode step in microseconds and the chunked prefill in
GB/s and as a fraction of its roofline.  `per_config` times the 8K, 32K and
128K single-request workloads in the same run.  Multi-GPU (torchrun): every
rank runs its own job (independent problems, no collective on the data
path), value = work of all ranks / slowest rank's time.

--impl reference times the CPU oracle on the same workload (bounded sample).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 data-sheet figures (HBM3e 7.9 TB/s, dense bf16 2.25 PFLOP/s): a second
# denominator beside the measured one, for context only.
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}
WORKLOADS = ["tiny", "8k", "32k", "128k", "mix"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="pfd", choices=["pfd", "reference"])
    ap.add_argument("--config", default="mix", choices=WORKLOADS)
    ap.add_argument("--per-config", default="8k,32k,128k",
                    help="other workloads timed in the same run ('' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the timings of the scoring head, ranking readings, layers and "
                         "reselection")
    ap.add_argument("--seqs", default="",
                    help="comma list: run only these sequences of the workload (profiling)")
    ap.add_argument("--profile", default="", choices=["", "decode", "prefill"],
                    help="one small eager pass for a profiler, then exit: 'prefill' runs the "
                         "prefill twice; 'decode' runs the prefill, frees its tensors and runs "
                         "two decode calls")
    return ap.parse_args(argv)


def job_configs(name):
    """The sequences of a workload: the mix is eight, the others one."""
    from sparse_chunked_kv_gb300 import workloads as wl
    return wl.mix_configs() if name == "mix" else [wl.CONFIGS[name]]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------- cost model --
# Algorithmic work of the method (re-reads, padding and split partials are
# not counted).  Each takes one Config; the job totals sum over sequences.

def decode_flops(cfg):
    keys = cfg.n_select * (cfg.n_keep + 1) + cfg.n_live
    return 4.0 * cfg.n_q_heads * cfg.n_live * keys * cfg.head_dim


def decode_bytes(cfg):
    hq, hkv, d, lq = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_live
    kept = cfg.n_select * (cfg.n_keep + 1)
    return lq * hq * d * 2 * 2 + lq * 2 * hkv * d * 2 + kept * 2 * hkv * d * 2 + lq * hq * 4


def prefill_flops(cfg):
    r = cfg.chunk_size + 1
    return 4.0 * cfg.n_q_heads * cfg.n_chunks * r * r * cfg.head_dim + \
        2.0 * cfg.n_q_heads * cfg.n_chunks * cfg.n_win * r * cfg.head_dim


def prefill_bytes(cfg):
    n, c, b, w = cfg.n_chunks, cfg.chunk_size, cfg.n_keep, cfg.n_win
    hq, hkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    return (n * (c + 1) * (hq + 2 * hkv) * d * 2 + w * hq * d * 2 + n * (c + 1) * hq * d * 2
            + n * c * 4 + n * b * 4 + n * (b + 1) * 2 * hkv * d * 2 + 8 * n)


def total(fn, cfgs):
    return sum(fn(c) for c in cfgs)


def workload_name(name, cfgs):
    if len(cfgs) == 1:
        cfg = cfgs[0]
        return (f"{cfg.name}: one layer, N={cfg.n_chunks} chunks x C={cfg.chunk_size} (+BOS), "
                f"Hq={cfg.n_q_heads}/Hkv={cfg.n_kv_heads}, D={cfg.head_dim}, B={cfg.n_keep}, "
                f"K={cfg.n_select}, W={cfg.n_win}, L_d={cfg.n_resp}, T={cfg.n_steps}")
    c0 = cfgs[0]
    per = ", ".join(f"C={c.chunk_size}: N={c.n_chunks}, B={c.n_keep}, K={c.n_select}"
                    for c in cfgs[:3])
    return (f"{name}: batched serving mix of {len(cfgs)} sequences x "
            f"{c0.n_chunks * c0.chunk_size // 1024}K prefix, one layer, C cycling "
            f"256/1024/4096 ({per}), Hq={c0.n_q_heads}/Hkv={c0.n_kv_heads}, D={c0.head_dim}, "
            f"W={c0.n_win}, L_d={c0.n_resp}, T={c0.n_steps}; one shared permuted pool, batched "
            f"selection, one batched decode call per step")


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 20 ms; only
    the samples taken between mark_start() and mark_end() (the timed region)
    are reported."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, interval_ms=20):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.path = os.path.join("/tmp", f"pfd_clocks_{os.getpid()}.csv")
        self.marks = [0, None]

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def _lines(self):
        self.fh.flush()
        with open(self.path) as f:
            return f.read().count("\n")

    def mark_start(self):
        if self.proc is not None:
            self.marks[0] = self._lines()

    def mark_end(self):
        if self.proc is not None:
            self.marks[1] = self._lines()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            lines = f.read().splitlines()
        os.unlink(self.path)
        lo, hi = self.marks[0], self.marks[1] if self.marks[1] is not None else len(lines)
        window = "timed region"
        if hi - lo < 1:
            lo, hi, window = 0, len(lines), "whole run (no sample fell inside the timed region)"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines[lo:hi]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "interval_ms": self.interval_ms, "window": window,
                "reasons": sorted(reasons)}


# ------------------------------------------------------- traffic record --

def kernel_source_hash(csrc=None):
    """Hash of the decode kernels' source with comments and whitespace removed,
    so that a profile stays matched to its code across comment edits."""
    csrc = csrc or os.path.join(ROOT, "sparse_chunked_kv_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("attn_tc.cu", "sm103_ptx.cuh", "pfd_internal.cuh", "lse_merge.cu"):
        with open(os.path.join(csrc, name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(profile_name, key="traffic_bytes_per_launch"):
    """Per-launch DRAM bytes from a committed ncu summary, only if it was taken
    on the current kernel source (its source hash line matches)."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_val = re.search(key + r":\s*([0-9.eE+]+)", text)
    if not m_hash or not m_val or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_val.group(1))


# ------------------------------------------------------------ GPU path --

def prefill_shape(cfg):
    """Sequences of one prefill shape are prefilled in one call."""
    return (cfg.chunk_size, cfg.n_chunks, cfg.n_win, cfg.n_keep)


class Job:
    """Device-resident buffers of one job (one or more sequences sharing one
    chunk pool and chunk table) and the library calls of one step.

    The job orders its sequences by prefill shape (stably), so that the
    sequences of one shape are contiguous in the chunk table and are
    prefilled by one pfd_chunk_prefill_batch call; seq_ids[i] is sequence
    i's data seed (its index in the workload, plus seq0)."""

    def __init__(self, cfgs, seq0, device, max_steps=None):
        import torch

        from sparse_chunked_kv_gb300 import _abi
        from sparse_chunked_kv_gb300 import workloads as wl
        cfgs = list(cfgs)
        order = sorted(range(len(cfgs)), key=lambda i: prefill_shape(cfgs[i]))
        self.seq_ids = [seq0 + i for i in order]
        self.cfgs, self.abi, self.torch = [cfgs[i] for i in order], _abi, torch
        c0 = self.cfgs[0]
        hq, hkv, d = c0.n_q_heads, c0.n_kv_heads, c0.head_dim
        assert all((c.n_q_heads, c.n_kv_heads, c.head_dim, c.n_steps) == (hq, hkv, d, c0.n_steps)
                   for c in self.cfgs)
        self.hq, self.hkv, self.d, self.T = hq, hkv, d, c0.n_steps
        if max_steps is not None:
            self.T = min(self.T, max_steps)
        self.batch = len(self.cfgs)
        dev = device
        cu = lambda t: t.to(dev).contiguous()  # noqa: E731
        self.host, self.seqs = [], []
        pool_base, cu_n, cu_k, cu_lq = [0], [0], [0], [0]
        for c in self.cfgs:
            pool_base.append(pool_base[-1] + c.pool_rows)
            cu_n.append(cu_n[-1] + c.n_chunks)
            cu_k.append(cu_k[-1] + c.n_select)
            cu_lq.append(cu_lq[-1] + c.n_live)
        self.pool_rows, self.table_len = pool_base[-1], cu_n[-1]
        self.cu_n_host, self.cu_k_host, self.cu_lq_host = cu_n, cu_k, cu_lq
        self.pool_k = torch.zeros(self.pool_rows, hkv, d, dtype=torch.bfloat16, device=dev)
        self.pool_v = torch.zeros_like(self.pool_k)
        self.table = torch.zeros(self.table_len, 2, dtype=torch.int32, device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        # Runs of sequences of one prefill shape: (first sequence, count).
        self.groups = []
        for i, c in enumerate(self.cfgs):
            if self.groups and prefill_shape(self.cfgs[self.groups[-1]["i0"]]) == prefill_shape(c):
                self.groups[-1]["L"] += 1
            else:
                self.groups.append(dict(i0=i, L=1))
        ws = 0
        live = [[] for _ in range(self.T)]
        for grp in self.groups:
            # Each group's prefill inputs and outputs are stacked [L, ...];
            # every sequence's tensors are views of them.
            c, L = self.cfgs[grp["i0"]], grp["L"]
            rows = c.n_chunks * (c.chunk_size + 1)
            grp["q"] = torch.empty(L, rows, hq, d, dtype=torch.bfloat16, device=dev)
            grp["k"] = torch.empty(L, rows, hkv, d, dtype=torch.bfloat16, device=dev)
            grp["v"] = torch.empty_like(grp["k"])
            grp["q_win"] = torch.empty(L, c.n_win, hq, d, dtype=torch.bfloat16, device=dev)
            grp["slot_row"] = torch.empty(L, c.n_chunks, dtype=torch.int32, device=dev)
            grp["out"] = torch.empty_like(grp["q"])
            grp["scores"] = torch.empty(L, c.n_chunks, c.chunk_size + 1, dtype=torch.float32,
                                        device=dev)
            grp["kept"] = torch.empty(L, c.n_chunks, max(c.n_keep, 1), dtype=torch.int32,
                                      device=dev)
            grp["ws_bytes"] = (
                _abi.pfd_chunk_prefill_workspace(c.n_chunks, c.chunk_size, c.n_win, hq, hkv, d,
                                                 c.n_keep) if L == 1 else
                _abi.pfd_chunk_prefill_layers_workspace(L, c.n_chunks, c.chunk_size, c.n_win, hq,
                                                        hkv, d, c.n_keep))
            ws = max(ws, grp["ws_bytes"])
        for i, c in enumerate(self.cfgs):
            grp = next(g for g in self.groups if g["i0"] <= i < g["i0"] + g["L"])
            l = i - grp["i0"]
            req = wl.make_request(c, self.seq_ids[i])
            req["slot_row"] = (req["slot_row"] + pool_base[i]).to(torch.int32)
            self.host.append(req)
            sq = dict(cfg=c, n0=cu_n[i])
            for key in ("q", "k", "v", "q_win", "slot_row"):
                sq[key] = grp[key][l]
                sq[key].copy_(req[key])
            for key in ("out", "scores", "kept"):
                sq[key] = grp[key][l]
            self.seqs.append(sq)
            for t in range(self.T):
                live[t].append(wl.live_block(req, wl.make_step(c, self.seq_ids[i], t)))
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.s_i = cu(torch.cat([h["s_i"] for h in self.host]))
        self.s_p = cu(torch.cat([h["s_p"] for h in self.host]))
        self.s_out = torch.empty_like(self.s_i)
        self.sel = torch.empty(cu_k[-1], dtype=torch.int32, device=dev)
        self.cu_n = torch.tensor(cu_n, dtype=torch.int32, device=dev)
        self.cu_k = torch.tensor(cu_k, dtype=torch.int32, device=dev)
        self.cu_lq = torch.tensor(cu_lq, dtype=torch.int32, device=dev)
        self.max_n = max(c.n_chunks for c in self.cfgs)
        self.max_len = max(c.n_keep + 1 for c in self.cfgs)
        # live q, k, v of step t, sequences concatenated
        self.live = [tuple(cu(torch.cat([x[j] for x in live[t]])) for j in range(3))
                     for t in range(self.T)]
        self.n_splits = _abi.pfd_decode_plan_splits(self.batch, cu_lq, cu_k, hq, hkv, d,
                                                    self.max_len)
        self.dws_bytes = _abi.pfd_decode_workspace(self.batch, cu_lq, cu_k, hq, hkv, d,
                                                   self.max_len, self.n_splits)
        self.dws = torch.empty(max(self.dws_bytes, 256), dtype=torch.uint8, device=dev)
        self.dec_out = [torch.empty_like(ql) for ql, _, _ in self.live]
        self.dec_lse = [torch.empty(cu_lq[-1], hq, dtype=torch.float32, device=dev)
                        for _ in self.live]

    def release_prefill(self):
        """Drops the prefill's own inputs and outputs (the pool, table and
        selection stay), so that a decode profile holds little memory."""
        for sq in self.seqs + self.groups:
            for key in ("q", "k", "v", "out", "scores", "kept"):
                sq[key] = None
        self.ws = None

    def launches_per_step(self):
        prefill = sum(2 + (1 if self.cfgs[g["i0"]].n_win > 0 else 0) for g in self.groups)
        return prefill + 1 + self.T * (1 + (1 if self.n_splits > 1 else 0))

    def prefill_select(self):
        a, hq, hkv, d = self.abi, self.hq, self.hkv, self.d
        for grp in self.groups:
            sq = self.seqs[grp["i0"]]
            c, L = sq["cfg"], grp["L"]
            if L == 1:
                a.pfd_chunk_prefill(sq["q"], sq["k"], sq["v"], sq["q_win"] if c.n_win else None,
                                    c.n_chunks, c.chunk_size, c.n_win, hq, hkv, d, c.n_keep, 0.0,
                                    sq["out"], sq["scores"], sq["kept"], self.pool_k,
                                    self.pool_v, self.pool_rows, sq["slot_row"],
                                    self.table[sq["n0"]:], self.dev_err, self.ws,
                                    grp["ws_bytes"])
            else:
                a.pfd_chunk_prefill_batch(grp["q"], grp["k"], grp["v"],
                                          grp["q_win"] if c.n_win else None, L, c.n_chunks,
                                          c.chunk_size, c.n_win, hq, hkv, d, c.n_keep, 0.0,
                                          grp["out"], grp["scores"], grp["kept"], self.pool_k,
                                          self.pool_v, self.pool_rows, grp["slot_row"],
                                          self.table[sq["n0"]:], self.dev_err, self.ws,
                                          grp["ws_bytes"])
        if self.batch == 1:
            c = self.cfgs[0]
            a.pfd_select_chunks(self.s_i, self.s_p, c.n_chunks, c.n_select, self.sel, self.s_out)
        else:
            a.pfd_select_chunks_batched(self.s_i, self.s_p, self.cu_n, self.cu_k, self.batch,
                                        self.max_n, self.sel, self.s_out)

    def decode(self, t, q=None, k=None, v=None, out=None):
        ql, kl, vl = self.live[t]
        self.abi.pfd_decode_attention(
            q if q is not None else ql, k if k is not None else kl, v if v is not None else vl,
            self.cu_lq, self.cu_lq_host, self.pool_k, self.pool_v, self.pool_rows, self.table,
            self.table_len, self.sel, self.cu_k, self.cu_k_host, self.batch, self.hq, self.hkv,
            self.d, self.max_len, 0.0, self.n_splits,
            out if out is not None else self.dec_out[t], self.dec_lse[t], self.dev_err, self.dws,
            self.dws_bytes)


def capture(job, stream):
    """Warms the job once eagerly, then captures its prefill+selection and
    its T-step decode loop as two CUDA graphs."""
    import torch
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        job.prefill_select()
        for t in range(job.T):
            job.decode(t)
    torch.cuda.synchronize()
    if int(job.dev_err.item()) != 0:
        raise RuntimeError(f"device error word {int(job.dev_err.item())}")
    g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pre, stream=stream):
        job.prefill_select()
    with torch.cuda.graph(g_dec, stream=stream):
        for t in range(job.T):
            job.decode(t)
    torch.cuda.synchronize()
    return g_pre, g_dec


def replay_steps(g_pre, g_dec, stream, flush, n):
    """n steps (prefill graph, decode graph), L2 flushed between steps
    outside the events; returns the (prefill ms, decode ms) of each."""
    import torch
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    with torch.cuda.stream(stream):
        for ev in events:
            ev[0].record(stream)
            g_pre.replay()
            ev[1].record(stream)
            g_dec.replay()
            ev[2].record(stream)
            flush.zero_()
    torch.cuda.synchronize()
    return [(e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])) for e in events]


def run_gpu(args, cfgs, rank, world, device):
    import torch

    from sparse_chunked_kv_gb300 import _abi
    _abi.load()
    job = Job(cfgs, rank * len(cfgs), device)
    stream = torch.cuda.Stream(device)
    g_pre, g_dec = capture(job, stream)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    replay_steps(g_pre, g_dec, stream, flush, args.warmup)

    clocks = ClockSampler(device.index if device.index is not None else 0)
    clocks.start()
    time.sleep(0.5)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    t0 = time.perf_counter()
    times = replay_steps(g_pre, g_dec, stream, flush, args.steps)
    wall = time.perf_counter() - t0
    clocks.mark_end()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if int(job.dev_err.item()) != 0:
        raise RuntimeError(f"device error word {int(job.dev_err.item())}")
    pre_ms = [a for a, _ in times]
    dec_ms = [b for _, b in times]
    res = dict(pre_ms=statistics.mean(pre_ms), dec_ms=statistics.mean(dec_ms),
               step_ms=statistics.mean(a + b for a, b in times), wall=wall, clocks=clk,
               launches=job.launches_per_step() * args.steps, n_splits=job.n_splits)
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, job, stream)
    del g_pre, g_dec, job
    torch.cuda.empty_cache()
    return res


def time_workload(name, rank, device, reps=5):
    """Decode and prefill timings of another workload in the same run (its
    own job, graphs replayed reps times after 3 warm-ups, L2 flushed between
    replays)."""
    import torch
    cfgs = job_configs(name)
    job = Job(cfgs, rank * len(cfgs), device)
    stream = torch.cuda.Stream(device)
    g_pre, g_dec = capture(job, stream)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    replay_steps(g_pre, g_dec, stream, flush, 3)
    times = replay_steps(g_pre, g_dec, stream, flush, reps)
    if int(job.dev_err.item()) != 0:
        raise RuntimeError(f"{name}: device error word {int(job.dev_err.item())}")
    res = dict(cfgs=cfgs, pre_ms=statistics.median(a for a, _ in times),
               dec_ms=statistics.median(b for _, b in times), n_splits=job.n_splits, T=job.T)
    del g_pre, g_dec, job, flush
    torch.cuda.empty_cache()
    return res


def time_scoring_head(device, reps=10):
    """The chunk-score head on the 8K-prefix shape: 16 chunks x (64 window +
    256 pseudo-label rows) x the 152,064-entry vocabulary, logits drawn on
    the device from a seeded generator (N(0, 4), bf16).  One call reads
    1.56 GB (> L2), so no flush is needed; median of reps after 3 warm-ups."""
    import torch

    from sparse_chunked_kv_gb300 import _abi
    from sparse_chunked_kv_gb300 import workloads as wl
    n, r, v = 16, 64 + 256, wl.SCORING_VOCAB
    gen = torch.Generator(device=device).manual_seed(5)
    logits = (2.0 * torch.randn(n, r, v, generator=gen, device=device)).to(torch.bfloat16)
    labels = torch.randint(0, v, (r,), generator=gen, device=device, dtype=torch.int32)
    row_ll = torch.empty(n, r, dtype=torch.float32, device=device)
    score = torch.empty(n, dtype=torch.float32, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.Stream(device)
    ms = []
    with torch.cuda.stream(stream):
        for it in range(3 + reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            _abi.pfd_chunk_loglik(logits, labels, n, r, v, row_ll, score, err)
            e1.record(stream)
            e1.synchronize()
            if it >= 3:
                ms.append(e0.elapsed_time(e1))
    if int(err.item()) != 0:
        raise RuntimeError(f"scoring head: device error word {int(err.item())}")
    t = statistics.median(ms) * 1e-3
    nbytes = n * r * v * 2 + r * 4 + n * r * 4 + n * 4
    del logits
    torch.cuda.empty_cache()
    return {"workload": f"{n} chunks x {r} labelled rows x vocabulary {v}, bf16 logits",
            "us": t * 1e6, "gbs": nbytes / t / 1e9, "bytes": nbytes, "bound": "hbm",
            "timing": f"median of {reps} calls after 3 warm-ups (inputs larger than L2)"}


def _time_calls(fn, stream, reps, flush=None):
    """Median ms of fn() over reps calls after 3 warm-ups, CUDA events on
    `stream`, L2 flushed before each call when a flush buffer is given."""
    import torch
    ms = []
    with torch.cuda.stream(stream):
        for it in range(3 + reps):
            if flush is not None:
                flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if it >= 3:
                ms.append(e0.elapsed_time(e1))
    return statistics.median(ms)


def time_next_rows(device, reps=5):
    """The other rows of the path on the 8K-prefix workload (one request):
    the prefill under the other ranking readings, four layers' prefill in
    one call, and one reselection (chunk masses of all 16 chunks at decode
    step 0's normaliser, then the new top-K); the reselection also on the
    128K workload (all 512 chunks).  L2 flushed before every call."""
    import torch

    from sparse_chunked_kv_gb300 import _abi
    from sparse_chunked_kv_gb300 import workloads as wl
    out = {}
    stream = torch.cuda.Stream(device)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    cfg = wl.CTX_8K
    hq, hkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    req = wl.make_request(cfg, 0)
    cu = lambda t: t.to(device).contiguous()  # noqa: E731
    q, k, v, q_win, k_win = (cu(req[x]) for x in ("q", "k", "v", "q_win", "k_win"))
    slot = cu(req["slot_row"])
    n, c, b, w = cfg.n_chunks, cfg.chunk_size, cfg.n_keep, cfg.n_win
    pool_k = torch.zeros(cfg.pool_rows, hkv, d, dtype=torch.bfloat16, device=device)
    pool_v = torch.zeros_like(pool_k)
    o = torch.empty_like(q)
    scores = torch.empty(n * hkv, c + 1, dtype=torch.float32, device=device)
    kept = torch.empty(n * hkv, b, dtype=torch.int32, device=device)
    table = torch.empty(n, 2, dtype=torch.int32, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    ws_b = _abi.pfd_chunk_prefill_workspace(n, c, w, hq, hkv, d, b)
    ws = torch.empty(ws_b, dtype=torch.uint8, device=device)
    pflops, pbytes = prefill_flops(cfg), prefill_bytes(cfg)
    for key, per_head, kw in (("rank_per_kv_head", 1, None), ("rank_window_keys", 0, k_win),
                              ("rank_per_kv_head_window_keys", 1, k_win)):
        ms = _time_calls(lambda: _abi.pfd_chunk_prefill_ex(
            q, k, v, q_win, kw, n, c, w, hq, hkv, d, b, 0.0, per_head, o, scores, kept, pool_k,
            pool_v, cfg.pool_rows, slot, table, err, ws, ws_b), stream, reps, flush)
        out[key] = {"workload": "8k prefill (pfd_chunk_prefill_ex)", "us": ms * 1e3,
                    "tflops": pflops / (ms * 1e-3) / 1e12, "gbs": pbytes / (ms * 1e-3) / 1e9,
                    "bound": "tensor", "flops": pflops}
    # four layers in one call
    n_layers = 4
    lay = wl.make_layers(cfg, n_layers)
    lq, lk, lv, lqw = (cu(lay[x]) for x in ("q", "k", "v", "q_win"))
    lo = torch.empty_like(lq)
    lscores = torch.empty(n_layers, n, c + 1, dtype=torch.float32, device=device)
    lkept = torch.empty(n_layers, n, b, dtype=torch.int32, device=device)
    lpk = torch.zeros(n_layers, cfg.pool_rows, hkv, d, dtype=torch.bfloat16, device=device)
    lpv = torch.zeros_like(lpk)
    ltab = torch.empty(n_layers, n, 2, dtype=torch.int32, device=device)
    lws_b = _abi.pfd_chunk_prefill_layers_workspace(n_layers, n, c, w, hq, hkv, d, b)
    lws = torch.empty(lws_b, dtype=torch.uint8, device=device)
    ms = _time_calls(lambda: _abi.pfd_chunk_prefill_layers(
        lq, lk, lv, lqw, n_layers, n, c, w, hq, hkv, d, b, 0.0, lo, lscores, lkept, lpk, lpv,
        cfg.pool_rows, slot, ltab, err, lws, lws_b), stream, reps, flush)
    ms_single = _time_calls(lambda: [_abi.pfd_chunk_prefill(
        lq[l], lk[l], lv[l], lqw[l], n, c, w, hq, hkv, d, b, 0.0, lo[l], lscores[l], lkept[l],
        lpk[l], lpv[l], cfg.pool_rows, slot, ltab[l], err, lws, lws_b) for l in range(n_layers)],
        stream, reps, flush)
    out["multi_layer_prefill"] = {
        "workload": f"8k prefill x {n_layers} layers in one call (pfd_chunk_prefill_layers)",
        "us": ms * 1e3, "tflops": n_layers * pflops / (ms * 1e-3) / 1e12,
        "us_as_separate_calls": ms_single * 1e3, "bound": "tensor", "flops": n_layers * pflops}
    del lq, lk, lv, lo, lpk, lpv
    # reselection: masses of every chunk at step 0's normaliser + new top-K
    for name in ("8k", "128k"):
        cfg = wl.CONFIGS[name]
        job = Job([cfg], 0, device)
        job.prefill_select()
        job.decode(0)
        torch.cuda.synchronize()
        cu_n = [0, cfg.n_chunks]
        mws_b = _abi.pfd_chunk_mass_workspace(1, job.cu_lq_host, cu_n, job.hq, job.hkv)
        mws = torch.empty(max(mws_b, 256), dtype=torch.uint8, device=device)
        mass = torch.empty(cfg.n_chunks, dtype=torch.float32, device=device)
        cu_n_d = torch.tensor(cu_n, dtype=torch.int32, device=device)
        sel2 = torch.empty_like(job.sel)
        s2 = torch.empty_like(job.s_out)

        def resel():
            _abi.pfd_chunk_mass(job.live[0][0], job.cu_lq, job.cu_lq_host, job.pool_k,
                                job.pool_rows, job.table, job.table_len, cu_n, job.dec_lse[0], 1,
                                job.hq, job.hkv, job.d, 0.0, mass, job.dev_err, mws, mws_b)
            _abi.pfd_reselect_chunks(job.s_out, mass, 1.0, cu_n_d, job.cu_k, 1, cfg.n_chunks,
                                     sel2, s2)
        ms = _time_calls(resel, stream, reps, flush)
        if int(job.dev_err.item()) != 0:
            raise RuntimeError(f"reselection {name}: device error {int(job.dev_err.item())}")
        fl = 2.0 * job.hq * cfg.n_live * cfg.n_chunks * (cfg.n_keep + 1) * job.d
        out[f"reselection_{name}"] = {
            "workload": f"{name}: masses of all {cfg.n_chunks} chunks at decode step 0 + top-"
                        f"{cfg.n_select} (pfd_chunk_mass + pfd_reselect_chunks)",
            "us": ms * 1e3, "tflops": fl / (ms * 1e-3) / 1e12, "bound": "tensor", "flops": fl}
        del job
        torch.cuda.empty_cache()
    return out


def run_e2e(args, job, stream):
    """The same work through the C ABI from pinned host buffers.

    Decode: every decode step copies its live q, k, v host -> device (one
    pinned block per step into one of four rotating device blocks, on a copy
    stream that runs up to three steps ahead) and its output device -> host;
    the T calls and all their copies are one CUDA graph.  The decode value
    and the byte counts of the line cover exactly this work.  The prefill's
    own upload (every sequence's q, k, v, q_win, s_I, s_P, slot rows) is
    timed separately and reported beside it."""
    import torch
    pin = lambda t: t.pin_memory()  # noqa: E731
    pre_in = []
    for sq, h in zip(job.seqs, job.host):
        for key in ("q", "k", "v", "q_win", "slot_row"):
            pre_in.append((sq[key], pin(h[key].contiguous())))
    pre_in.append((job.s_i, pin(torch.cat([h["s_i"] for h in job.host]))))
    pre_in.append((job.s_p, pin(torch.cat([h["s_p"] for h in job.host]))))
    n_live = 4
    shapes = [x.shape for x in job.live[0]]
    sizes = [x.numel() for x in job.live[0]]

    def views(flat):
        out, off = [], 0
        for shp, n in zip(shapes, sizes):
            out.append(flat[off:off + n].view(shp))
            off += n
        return tuple(out)

    h_live = []
    for blk in job.live:
        flat = torch.empty(sum(sizes), dtype=torch.bfloat16).pin_memory()
        for dst, x in zip(views(flat), blk):
            dst.copy_(x.cpu())
        h_live.append(flat)
    h_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in job.dec_out]
    d_flat = [torch.empty(sum(sizes), dtype=torch.bfloat16, device=job.pool_k.device)
              for _ in range(n_live)]
    d_live = [views(f) for f in d_flat]
    pre_h2d = sum(h.numel() * h.element_size() for _, h in pre_in)
    dec_h2d = sum(x.numel() * x.element_size() for x in h_live)
    dec_d2h = sum(o.numel() * o.element_size() for o in h_out)

    copy_s = torch.cuda.Stream(stream.device)
    d2h_s = torch.cuda.Stream(stream.device)
    h2d_done = [torch.cuda.Event() for _ in range(n_live)]
    dec_done = [torch.cuda.Event() for _ in range(n_live)]

    def prefill_part():
        copy_s.wait_stream(stream)
        with torch.cuda.stream(copy_s):
            for d, h in pre_in:
                d.copy_(h, non_blocking=True)
        stream.wait_stream(copy_s)
        with torch.cuda.stream(stream):
            job.prefill_select()

    def decode_part():
        copy_s.wait_stream(stream)
        d2h_s.wait_stream(stream)
        for t in range(job.T):
            b = t % n_live
            dq, dk, dv = d_live[b]
            with torch.cuda.stream(copy_s):
                if t >= n_live:
                    copy_s.wait_event(dec_done[b])   # step t - n_live is done with block b
                d_flat[b].copy_(h_live[t], non_blocking=True)
                h2d_done[b].record(copy_s)
            with torch.cuda.stream(stream):
                stream.wait_event(h2d_done[b])
                job.decode(t, dq, dk, dv, job.dec_out[t])
                dec_done[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(dec_done[b])
                h_out[t].copy_(job.dec_out[t], non_blocking=True)
        stream.wait_stream(d2h_s)
        stream.wait_stream(copy_s)

    # Warm eagerly, then capture the calls and copies once, as a serving loop
    # would run them; every copy is a node of a graph replayed every step
    # inside the timed region.
    for _ in range(2):
        prefill_part()
        decode_part()
    torch.cuda.synchronize()
    g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pre, stream=stream):
        prefill_part()
    with torch.cuda.graph(g_dec, stream=stream):
        decode_part()
    torch.cuda.synchronize()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    pre_ms, dec_ms = [], []
    for it in range(max(1, args.warmup) + args.steps):
        with torch.cuda.stream(stream):
            marks[0].record(stream)
            g_pre.replay()
            marks[1].record(stream)
            g_dec.replay()
            marks[2].record(stream)
        torch.cuda.synchronize()
        if it >= max(1, args.warmup):
            pre_ms.append(marks[0].elapsed_time(marks[1]))
            dec_ms.append(marks[1].elapsed_time(marks[2]))
    return dict(pre_ms=statistics.mean(pre_ms), dec_ms=statistics.mean(dec_ms),
                pre_h2d=pre_h2d, dec_h2d=dec_h2d, dec_d2h=dec_d2h)


# ----------------------------------------------------------- CPU oracle --

def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def _oracle_decode_inputs(cfg, seq):
    """One sequence's oracle decode inputs: its pool (kept = the first B
    content rows; the decode cost does not depend on which), selection and
    the live block of step 0."""
    import numpy as np

    from oracle import pfd_oracle as orc
    from sparse_chunked_kv_gb300 import workloads as wl
    req = wl.make_request(cfg, seq)
    f = wl.to_f64
    kept = np.array([list(range(cfg.n_keep))] * cfg.n_chunks, dtype=np.int32)
    pk = np.zeros((cfg.pool_rows, cfg.n_kv_heads, cfg.head_dim))
    pv = np.zeros_like(pk)
    table = orc.compact(f(req["k"]), f(req["v"]), kept, req["slot_row"].numpy(), cfg.chunk_size,
                        pk, pv)
    sel, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    ql, kl, vl = wl.live_block(req, wl.make_step(cfg, seq, 0))
    return (f(ql), f(kl), f(vl), pk, pv, table, sel, cfg.sm_scale)


def oracle_decode_sample(cfgs, seconds):
    """Times full oracle decode steps of the job (fp64 CPU, every sequence)
    for about `seconds`; returns seconds per step."""
    from oracle import pfd_oracle as orc
    inputs = [_oracle_decode_inputs(c, i) for i, c in enumerate(cfgs)]
    n, t0 = 0, time.perf_counter()
    while True:
        for x in inputs:
            orc.decode_attention(*x)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 1000:
            break
    return el / n


def oracle_prefill_sample(cfgs, seconds):
    """Times the oracle's prefill (chunk attention + window scores) on one
    chunk of each distinct chunk size, scaled to the job's chunk counts."""
    from oracle import pfd_oracle as orc
    from sparse_chunked_kv_gb300 import workloads as wl
    distinct = {}
    for c in cfgs:
        distinct.setdefault(c.chunk_size, []).append(c)
    per = max(seconds / len(distinct), 1e-3)
    total_s = 0.0
    for group in distinct.values():
        cfg = group[0]
        req = wl.make_request(cfg, 0)
        rows = cfg.chunk_size + 1
        f = wl.to_f64
        q, k, v, qw = f(req["q"][:rows]), f(req["k"][:rows]), f(req["v"][:rows]), f(req["q_win"])
        n, t0 = 0, time.perf_counter()
        while True:
            orc.chunk_attention(q, k, v, 1, cfg.chunk_size, cfg.sm_scale)
            orc.window_scores(qw, k, 1, cfg.chunk_size, cfg.sm_scale)
            n += 1
            el = time.perf_counter() - t0
            if el >= per or n >= 1000:
                break
        total_s += (el / n) * sum(c.n_chunks for c in group)
    return total_s


def cpu_baseline(name, cfgs, seconds):
    dec_s = oracle_decode_sample(cfgs, seconds * 0.7)
    pre_s = oracle_prefill_sample(cfgs, seconds * 0.3)
    return {"value": total(decode_flops, cfgs) / dec_s / 1e12, "unit": "TFLOP/s",
            "cores": blas_threads(), "kind": "oracle",
            "sample": (f"fp64 numpy oracle: full decode steps of the {name} workload "
                       f"({len(cfgs)} sequence(s)) repeated for ~{0.7 * seconds:.0f} s "
                       f"({dec_s * 1e3:.1f} ms each); prefill rate from one chunk of each chunk "
                       f"size repeated for ~{0.3 * seconds:.0f} s, scaled to the job's chunks"),
            "decode_ms_per_step": dec_s * 1e3, "prefill_ms": pre_s * 1e3,
            "prefill_gbs": total(prefill_bytes, cfgs) / pre_s / 1e9}


def run_reference(args, cfgs, rank, name=None):
    if not isinstance(cfgs, (list, tuple)):
        cfgs = [cfgs]
    name = name or (cfgs[0].name if len(cfgs) == 1 else "mix")
    if rank != 0:
        return
    per_step = max(0.5, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_decode_sample(cfgs, 0.0)
    times = [oracle_decode_sample(cfgs, per_step) for _ in range(args.steps)]
    dec_s = statistics.mean(times)
    value = total(decode_flops, cfgs) / dec_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dec_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(name, cfgs),
                       "timed": "one oracle decode step of the whole job per step"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                             "kind": "oracle",
                             "sample": f"fp64 numpy oracle, full decode steps of {name} "
                                       f"({len(cfgs)} sequence(s)), ~{per_step:.1f} s per "
                                       f"timed step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


METRIC = "decode-step attention µs & TFLOP/s vs BF16 peak; chunk-prefill GB/s vs HBM peak"


def max_over_ranks(values, device):
    """Each timing's maximum over all ranks of the default process group
    (every rank receives the result): the job is as slow as its slowest rank."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tflops(world, flops_per_call, calls, ms):
    """Whole-job throughput: every rank ran `calls` calls of `flops_per_call`
    in at most `ms` milliseconds (weak scaling: fixed work per rank)."""
    return world * flops_per_call * calls / (ms * 1e-3) / 1e12


def roofline_fracs(cfgs, dec_ms_per_call, pre_ms, peaks):
    """Decode and prefill against the measured peaks: decode against the
    bf16 burst peak (a graph of back-to-back calls lasting milliseconds) and,
    as a second figure, the sustained one; prefill against
    max(bytes / HBM, flops / bf16 burst)."""
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    dflops = total(decode_flops, cfgs)
    dec_tflops = dflops / (dec_ms_per_call * 1e-3) / 1e12
    pflops, pbytes = total(prefill_flops, cfgs), total(prefill_bytes, cfgs)
    pre_s = pre_ms * 1e-3
    t_hbm, t_tc = pbytes / (hbm * 1e9), pflops / (burst * 1e12)
    t_nominal = max(pbytes / (NOMINAL_PEAKS["hbm_gbs"] * 1e9),
                    pflops / (NOMINAL_PEAKS["bf16_tflops"] * 1e12))
    return dict(decode_us=dec_ms_per_call * 1e3, decode_tflops=dec_tflops,
                decode_frac=dec_tflops / burst, decode_frac_sustained=dec_tflops / sustained,
                decode_frac_nominal=dec_tflops / NOMINAL_PEAKS["bf16_tflops"],
                prefill_us=pre_ms * 1e3, prefill_tflops=pflops / pre_s / 1e12,
                prefill_gbs=pbytes / pre_s / 1e9, prefill_bound="tensor" if t_tc >= t_hbm else "hbm",
                prefill_frac=max(t_hbm, t_tc) / pre_s, prefill_frac_nominal=t_nominal / pre_s)


def run_profile(args, cfgs, device):
    """One small eager pass for a profiler (see --profile)."""
    import torch
    job = Job(cfgs, 0, device, max_steps=2 if args.profile == "decode" else 1)
    job.prefill_select()
    if args.profile == "prefill":
        job.prefill_select()
    else:
        torch.cuda.synchronize()
        job.release_prefill()
        torch.cuda.empty_cache()
        job.decode(0)
        job.decode(1)
    torch.cuda.synchronize()
    if int(job.dev_err.item()) != 0:
        raise RuntimeError(f"device error word {int(job.dev_err.item())}")
    print(json.dumps({"profile": args.profile, "workload": workload_name(args.config, cfgs),
                      "decode_splits": job.n_splits}))


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cfgs = job_configs(args.config)
    if args.seqs:
        cfgs = [cfgs[int(i)] for i in args.seqs.split(",")]
    if args.profile:
        import torch
        run_profile(args, cfgs, torch.device("cuda", 0))
        return
    if args.impl == "reference":
        run_reference(args, cfgs, rank, args.config)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    res = run_gpu(args, cfgs, rank, world, device)
    if world > 1:
        res["dec_ms"], res["pre_ms"], res["step_ms"] = max_over_ranks(
            [res["dec_ms"], res["pre_ms"], res["step_ms"]], device)
    others, next_rows = {}, {}
    if rank == 0:
        for name in [x for x in args.per_config.split(",") if x and x != args.config]:
            others[name] = time_workload(name, 0, device)
        if not args.no_next_rows:
            next_rows["scoring_head"] = time_scoring_head(device)
            next_rows.update(time_next_rows(device))
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peaks, peak_kind = load_peaks()
    T = cfgs[0].n_steps
    dflops = total(decode_flops, cfgs)
    value = job_tflops(world, dflops, T, res["dec_ms"])
    fr = roofline_fracs(cfgs, res["dec_ms"] / T, res["pre_ms"], peaks)
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["step_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_name(args.config, cfgs), "global_batch": world * len(cfgs),
                   "seq_len": sum(c.n_chunks * c.chunk_size for c in cfgs) // len(cfgs),
                   "l2": "flushed between steps (256 MiB write), outside the timed events",
                   "decode_splits": res["n_splits"], "graphs": "prefill+select; T-step decode loop",
                   "parallelism": f"replicas x{world} (independent jobs)"},
        "decode_us_per_step": fr["decode_us"],
        "decode_tflops": fr["decode_tflops"],
        "prefill_us": fr["prefill_us"],
        "prefill_gbs": fr["prefill_gbs"],
        "prefill_tflops": fr["prefill_tflops"],
        "prefill_roofline_frac": fr["prefill_frac"],
        "roofline": {"kernel": "decode attention call (attention_kernel + lse_merge_kernel)",
                     "bound": "tensor", "achieved": fr["decode_tflops"], "peak": burst,
                     "peak_kind": f"{peak_kind} bf16 burst", "unit": "TFLOP/s",
                     "frac": fr["decode_frac"],
                     "frac_of_sustained": fr["decode_frac_sustained"],
                     "sustained_peak": sustained,
                     "frac_of_nominal": fr["decode_frac_nominal"],
                     "nominal_peak": NOMINAL_PEAKS["bf16_tflops"],
                     "traffic": recorded_traffic(f"decode_attention_{args.config}.md")},
        "prefill_roofline": {"bound": fr["prefill_bound"], "achieved_gbs": fr["prefill_gbs"],
                             "hbm_peak_gbs": hbm, "achieved_tflops": fr["prefill_tflops"],
                             "tensor_peak_tflops": burst, "frac": fr["prefill_frac"],
                             "peak_kind": f"{peak_kind} (HBM copy; bf16 burst)",
                             "frac_of_nominal": fr["prefill_frac_nominal"]},
        "clocks": res["clocks"],
        "gpu_launches": res["launches"],
        "wall_s_timed_region": res["wall"],
    }
    if others:
        line["per_config"] = {}
        for name, o in others.items():
            f2 = roofline_fracs(o["cfgs"], o["dec_ms"] / o["T"], o["pre_ms"], peaks)
            line["per_config"][name] = {
                "decode_us_per_step": f2["decode_us"], "decode_tflops": f2["decode_tflops"],
                "decode_frac": f2["decode_frac"], "decode_frac_sustained": f2["decode_frac_sustained"],
                "decode_frac_nominal": f2["decode_frac_nominal"],
                "decode_splits": o["n_splits"], "prefill_us": f2["prefill_us"],
                "prefill_tflops": f2["prefill_tflops"], "prefill_gbs": f2["prefill_gbs"],
                "prefill_bound": f2["prefill_bound"], "prefill_frac": f2["prefill_frac"],
                "prefill_frac_nominal": f2["prefill_frac_nominal"],
                "timing": "median of 5 graph replays after 3 warm-ups, L2 flushed between"}
    if next_rows:
        line["next_rows"] = {}
        for key, row in next_rows.items():
            row = dict(row)
            if row["bound"] == "hbm":
                row["frac"] = row["gbs"] / hbm
                row["peak"] = hbm
                row["peak_kind"] = f"{peak_kind} HBM copy"
            else:
                row["frac"] = row["tflops"] / burst
                row["peak"] = burst
                row["peak_kind"] = f"{peak_kind} bf16 burst"
            line["next_rows"][key] = row
    if "e2e" in res:
        e = res["e2e"]
        line["e2e"] = {"value": job_tflops(world, dflops, T, e["dec_ms"]), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": e["dec_h2d"], "d2h_bytes_per_step": e["dec_d2h"],
                       "decode_ms": e["dec_ms"],
                       "path": ("the T decode calls of a step through the C ABI, captured in a "
                                "CUDA graph with every call's live-block H2D copy from pinned "
                                "host memory and its output's D2H as graph nodes on copy streams "
                                "that overlap the kernels; value and byte counts cover exactly "
                                "these calls and copies"),
                       "prefill": {"ms": e["pre_ms"], "h2d_bytes": e["pre_h2d"],
                                   "path": "every sequence's prefill inputs uploaded from pinned "
                                           "memory, then the prefill and selection calls"}}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.config, cfgs, args.cpu_seconds)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
