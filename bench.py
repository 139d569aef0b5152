#!/usr/bin/env python
"""Benchmark of the sparse chunked-KV hot path (one request = one step).

One step runs the whole path over one synthetic request of the chosen
workload: chunked prefill (chunk attention, window scores, top-B, compaction
into the pool), top-K chunk selection, then T static-KV decode steps
(split-KV attention + LSE merge).  Inputs are resident in HBM before the timed
region; the prefill+selection and the T-step decode loop are each one CUDA
graph replay, bracketed by CUDA events on the launching stream.  L2 is
flushed (256 MiB write) between steps, outside the timed events.

value = decode-step attention throughput (algorithmic TFLOP/s, whole job);
extra keys give the decode step in microseconds and the chunked prefill in
GB/s and as a fraction of the HBM roofline.  Multi-GPU (torchrun): every rank
runs its own request (independent problems, no collective on the data path),
value = work of all ranks / slowest rank's time.

--impl reference times the CPU oracle on the same workload (bounded sample).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="pfd", choices=["pfd", "reference"])
    ap.add_argument("--config", default="8k", choices=["tiny", "8k", "32k", "128k"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------- cost model --

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


def workload_name(cfg):
    return (f"{cfg.name}: one layer, N={cfg.n_chunks} chunks x C={cfg.chunk_size} (+BOS), "
            f"Hq={cfg.n_q_heads}/Hkv={cfg.n_kv_heads}, D={cfg.head_dim}, B={cfg.n_keep}, "
            f"K={cfg.n_select}, W={cfg.n_win}, L_d={cfg.n_resp}, T={cfg.n_steps}")


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"pfd_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
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
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


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

class Request:
    """Device-resident buffers of one request and the calls of one step."""

    def __init__(self, cfg, seq, device):
        import torch

        from sparse_chunked_kv_gb300 import _abi
        from sparse_chunked_kv_gb300 import workloads as wl
        self.cfg, self.abi, self.torch = cfg, _abi, torch
        req = wl.make_request(cfg, seq)
        self.host = req
        dev = device
        cu = lambda t: t.to(dev).contiguous()  # noqa: E731
        self.q, self.k, self.v = cu(req["q"]), cu(req["k"]), cu(req["v"])
        self.q_win = cu(req["q_win"])
        self.s_i, self.s_p = cu(req["s_i"]), cu(req["s_p"])
        self.slot_row = cu(req["slot_row"])
        self.live = []
        for t in range(cfg.n_steps):
            ql, kl, vl = wl.live_block(req, wl.make_step(cfg, seq, t))
            self.live.append((cu(ql), cu(kl), cu(vl)))
        hq, hkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
        self.out = torch.empty_like(self.q)
        self.scores = torch.empty(cfg.n_chunks, cfg.chunk_size + 1, dtype=torch.float32, device=dev)
        self.kept = torch.empty(cfg.n_chunks, max(cfg.n_keep, 1), dtype=torch.int32, device=dev)
        self.pool_k = torch.zeros(cfg.pool_rows, hkv, d, dtype=torch.bfloat16, device=dev)
        self.pool_v = torch.zeros_like(self.pool_k)
        self.table = torch.empty(cfg.n_chunks, 2, dtype=torch.int32, device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws_bytes = _abi.pfd_chunk_prefill_workspace(cfg.n_chunks, cfg.chunk_size, cfg.n_win,
                                                         hq, hkv, d, cfg.n_keep)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.sel = torch.empty(cfg.n_select, dtype=torch.int32, device=dev)
        self.s_out = torch.empty(cfg.n_chunks, dtype=torch.float32, device=dev)
        lq = cfg.n_live
        self.cu_lq_host, self.cu_k_host = [0, lq], [0, cfg.n_select]
        self.cu_lq = torch.tensor(self.cu_lq_host, dtype=torch.int32, device=dev)
        self.cu_k = torch.tensor(self.cu_k_host, dtype=torch.int32, device=dev)
        self.max_len = cfg.n_keep + 1
        self.n_splits = _abi.pfd_decode_plan_splits(1, self.cu_lq_host, self.cu_k_host, hq, hkv, d,
                                                    self.max_len)
        self.dws_bytes = _abi.pfd_decode_workspace(1, self.cu_lq_host, self.cu_k_host, hq, hkv, d,
                                                   self.max_len, self.n_splits)
        self.dws = torch.empty(max(self.dws_bytes, 256), dtype=torch.uint8, device=dev)
        self.dec_out = [torch.empty_like(ql) for ql, _, _ in self.live]
        self.dec_lse = [torch.empty(lq, hq, dtype=torch.float32, device=dev) for _ in self.live]

    def launches_per_step(self):
        cfg = self.cfg
        prefill = 2 + (1 if cfg.n_win > 0 else 0)
        return prefill + 1 + cfg.n_steps * (1 + (1 if self.n_splits > 1 else 0))

    def prefill_select(self):
        cfg, a = self.cfg, self.abi
        a.pfd_chunk_prefill(self.q, self.k, self.v, self.q_win if cfg.n_win else None, cfg.n_chunks,
                            cfg.chunk_size, cfg.n_win, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                            cfg.n_keep, 0.0, self.out, self.scores, self.kept, self.pool_k,
                            self.pool_v, cfg.pool_rows, self.slot_row, self.table, self.dev_err,
                            self.ws, self.ws_bytes)
        a.pfd_select_chunks(self.s_i, self.s_p, cfg.n_chunks, cfg.n_select, self.sel, self.s_out)

    def decode(self, t, q=None, k=None, v=None, out=None):
        cfg = self.cfg
        ql, kl, vl = self.live[t]
        self.abi.pfd_decode_attention(
            q if q is not None else ql, k if k is not None else kl, v if v is not None else vl,
            self.cu_lq, self.cu_lq_host, self.pool_k, self.pool_v, cfg.pool_rows, self.table,
            cfg.n_chunks, self.sel, self.cu_k, self.cu_k_host, 1, cfg.n_q_heads, cfg.n_kv_heads,
            cfg.head_dim, self.max_len, 0.0, self.n_splits,
            out if out is not None else self.dec_out[t], self.dec_lse[t], self.dev_err, self.dws,
            self.dws_bytes)


def run_gpu(args, cfg, rank, world, device):
    import torch

    from sparse_chunked_kv_gb300 import _abi
    _abi.load()
    r = Request(cfg, rank, device)
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    # warm once eagerly (kernel attributes, module load), then capture graphs
    with torch.cuda.stream(stream):
        r.prefill_select()
        for t in range(cfg.n_steps):
            r.decode(t)
    torch.cuda.synchronize()
    if int(r.dev_err.item()) != 0:
        raise RuntimeError(f"device error word {int(r.dev_err.item())}")
    g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pre, stream=stream):
        r.prefill_select()
    with torch.cuda.graph(g_dec, stream=stream):
        for t in range(cfg.n_steps):
            r.decode(t)
    torch.cuda.synchronize()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def one_step(ev):
        ev[0].record(stream)
        g_pre.replay()
        ev[1].record(stream)
        g_dec.replay()
        ev[2].record(stream)

    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            one_step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
            flush.zero_()
    torch.cuda.synchronize()

    clocks = ClockSampler(device.index if device.index is not None else 0)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for s in range(args.steps):
            one_step(events[s])
            flush.zero_()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if int(r.dev_err.item()) != 0:
        raise RuntimeError(f"device error word {int(r.dev_err.item())}")
    pre_ms = [e[0].elapsed_time(e[1]) for e in events]
    dec_ms = [e[1].elapsed_time(e[2]) for e in events]
    step_ms = [a + b for a, b in zip(pre_ms, dec_ms)]
    res = dict(pre_ms=statistics.mean(pre_ms), dec_ms=statistics.mean(dec_ms),
               step_ms=statistics.mean(step_ms), wall=wall, clocks=clk,
               launches=r.launches_per_step() * args.steps, n_splits=r.n_splits)
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, r, stream)
    return res


def run_e2e(args, r, stream):
    """Same path through the C ABI from pinned host buffers: every step copies
    its inputs host->device and the decode outputs device->host."""
    import torch
    cfg = r.cfg
    pin = lambda t: t.pin_memory()  # noqa: E731
    h_q, h_k, h_v = pin(r.host["q"]), pin(r.host["k"]), pin(r.host["v"])
    h_qw, h_si, h_sp, h_slot = pin(r.host["q_win"]), pin(r.host["s_i"]), pin(r.host["s_p"]), \
        pin(r.host["slot_row"])
    # Each step's live q, k, v travel as one pinned block (one copy a step)
    # into one of N_LIVE device blocks, so the copies can run up to
    # N_LIVE - 1 steps ahead of the kernels.
    n_live = 4
    shapes = [x.shape for x in r.live[0]]
    sizes = [x.numel() for x in r.live[0]]

    def views(flat):
        out, off = [], 0
        for shp, n in zip(shapes, sizes):
            out.append(flat[off:off + n].view(shp))
            off += n
        return tuple(out)

    h_live = []
    for blk in r.live:
        flat = torch.empty(sum(sizes), dtype=torch.bfloat16).pin_memory()
        for dst, x in zip(views(flat), blk):
            dst.copy_(x.cpu())
        h_live.append(flat)
    h_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in r.dec_out]
    d_flat = [torch.empty(sum(sizes), dtype=torch.bfloat16, device=r.q.device) for _ in range(n_live)]
    d_live = [views(f) for f in d_flat]
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_qw, h_si, h_sp, h_slot))
    h2d += sum(x.numel() * x.element_size() for x in h_live)
    d2h = sum(o.numel() * o.element_size() for o in h_out)

    # Copies run on their own streams so that they overlap the kernels: the
    # inputs of the next decode steps go up while step t computes, and step
    # t's output comes down while step t+1 computes.  Every copy stays inside
    # the timed region.
    copy_s = torch.cuda.Stream(stream.device)
    d2h_s = torch.cuda.Stream(stream.device)
    h2d_done = [torch.cuda.Event() for _ in range(n_live)]
    dec_done = [torch.cuda.Event() for _ in range(n_live)]

    def step(ev):
        with torch.cuda.stream(stream):
            ev[0].record(stream)
        copy_s.wait_stream(stream)
        with torch.cuda.stream(copy_s):
            r.q.copy_(h_q, non_blocking=True)
            r.k.copy_(h_k, non_blocking=True)
            r.v.copy_(h_v, non_blocking=True)
            r.q_win.copy_(h_qw, non_blocking=True)
            r.s_i.copy_(h_si, non_blocking=True)
            r.s_p.copy_(h_sp, non_blocking=True)
            r.slot_row.copy_(h_slot, non_blocking=True)
        stream.wait_stream(copy_s)
        with torch.cuda.stream(stream):
            r.prefill_select()
            ev[1].record(stream)
        copy_s.wait_stream(stream)          # decode copies start after the prefill
        for t in range(cfg.n_steps):
            b = t % n_live
            dq, dk, dv = d_live[b]
            with torch.cuda.stream(copy_s):
                if t >= n_live:
                    copy_s.wait_event(dec_done[b])   # step t - n_live is done with block b
                d_flat[b].copy_(h_live[t], non_blocking=True)
                h2d_done[b].record(copy_s)
            with torch.cuda.stream(stream):
                stream.wait_event(h2d_done[b])
                r.decode(t, dq, dk, dv, r.dec_out[t])
                dec_done[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(dec_done[b])
                h_out[t].copy_(r.dec_out[t], non_blocking=True)
        stream.wait_stream(d2h_s)
        with torch.cuda.stream(stream):
            ev[2].record(stream)

    # Eager: one public-API call per decode step, issued from Python.
    for _ in range(max(1, args.warmup)):
        step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for s in range(args.steps):
        step(evs[s])
    torch.cuda.synchronize()
    eager_pre = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    eager_dec = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)

    # Graph: the same calls and copies captured once, as a serving loop would
    # run them; every H2D from pinned memory and every D2H is a node of the
    # graph, replayed every step inside the timed region.
    g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def prefill_part():
        copy_s.wait_stream(stream)
        with torch.cuda.stream(copy_s):
            r.q.copy_(h_q, non_blocking=True)
            r.k.copy_(h_k, non_blocking=True)
            r.v.copy_(h_v, non_blocking=True)
            r.q_win.copy_(h_qw, non_blocking=True)
            r.s_i.copy_(h_si, non_blocking=True)
            r.s_p.copy_(h_sp, non_blocking=True)
            r.slot_row.copy_(h_slot, non_blocking=True)
        stream.wait_stream(copy_s)
        with torch.cuda.stream(stream):
            r.prefill_select()

    def decode_part():
        copy_s.wait_stream(stream)
        d2h_s.wait_stream(stream)
        for t in range(cfg.n_steps):
            b = t % n_live
            dq, dk, dv = d_live[b]
            with torch.cuda.stream(copy_s):
                if t >= n_live:
                    copy_s.wait_event(dec_done[b])
                d_flat[b].copy_(h_live[t], non_blocking=True)
                h2d_done[b].record(copy_s)
            with torch.cuda.stream(stream):
                stream.wait_event(h2d_done[b])
                r.decode(t, dq, dk, dv, r.dec_out[t])
                dec_done[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(dec_done[b])
                h_out[t].copy_(r.dec_out[t], non_blocking=True)
        stream.wait_stream(d2h_s)
        stream.wait_stream(copy_s)

    with torch.cuda.graph(g_pre, stream=stream):
        prefill_part()
    with torch.cuda.graph(g_dec, stream=stream):
        decode_part()
    torch.cuda.synchronize()
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
    return dict(pre_ms=statistics.mean(pre_ms), dec_ms=statistics.mean(dec_ms), h2d=h2d, d2h=d2h,
                eager_pre_ms=eager_pre, eager_dec_ms=eager_dec)


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


def oracle_decode_sample(cfg, seconds):
    """Times full oracle decode steps of cfg (fp64 CPU) for about `seconds`."""
    from oracle import pfd_oracle as orc
    from sparse_chunked_kv_gb300 import workloads as wl
    req = wl.make_request(cfg, 0)
    f = wl.to_f64
    kept = [list(range(cfg.n_keep))] * cfg.n_chunks
    import numpy as np
    kept = np.array(kept, dtype=np.int32)
    pk = np.zeros((cfg.pool_rows, cfg.n_kv_heads, cfg.head_dim))
    pv = np.zeros_like(pk)
    table = orc.compact(f(req["k"]), f(req["v"]), kept, req["slot_row"].numpy(), cfg.chunk_size, pk, pv)
    sel, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    ql, kl, vl = wl.live_block(req, wl.make_step(cfg, 0, 0))
    ql, kl, vl = f(ql), f(kl), f(vl)
    n, t0 = 0, time.perf_counter()
    while True:
        orc.decode_attention(ql, kl, vl, pk, pv, table, sel, cfg.sm_scale)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 1000:
            break
    return el / n


def oracle_prefill_sample(cfg, seconds):
    """Times the oracle's prefill (chunk attention + window scores) on one chunk."""
    from oracle import pfd_oracle as orc
    from sparse_chunked_kv_gb300 import workloads as wl
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
        if el >= seconds or n >= 1000:
            break
    return (el / n) * cfg.n_chunks  # one chunk's time scaled to the workload's N chunks


def cpu_baseline(cfg, seconds):
    dec_s = oracle_decode_sample(cfg, seconds * 0.7)
    pre_s = oracle_prefill_sample(cfg, seconds * 0.3)
    return {"value": decode_flops(cfg) / dec_s / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": (f"fp64 numpy oracle: full decode steps of the {cfg.name} workload repeated "
                       f"for ~{0.7 * seconds:.0f} s ({dec_s * 1e3:.1f} ms each); prefill rate from "
                       f"one chunk repeated for ~{0.3 * seconds:.0f} s, scaled to N chunks"),
            "decode_ms_per_step": dec_s * 1e3, "prefill_ms": pre_s * 1e3,
            "prefill_gbs": prefill_bytes(cfg) / pre_s / 1e9}


def run_reference(args, cfg, rank):
    if rank != 0:
        return
    from sparse_chunked_kv_gb300 import workloads as wl  # noqa: F401
    per_step = max(0.5, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_decode_sample(cfg, 0.0)
    times = [oracle_decode_sample(cfg, per_step) for _ in range(args.steps)]
    dec_s = statistics.mean(times)
    value = decode_flops(cfg) / dec_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dec_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(cfg), "timed": "one oracle decode step per step"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                             "kind": "oracle",
                             "sample": f"fp64 numpy oracle, full decode steps of {cfg.name}, "
                                       f"~{per_step:.1f} s per timed step"},
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


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from sparse_chunked_kv_gb300 import workloads as wl
    cfg = wl.CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    res = run_gpu(args, cfg, rank, world, device)
    if world > 1:
        res["dec_ms"], res["pre_ms"], res["step_ms"] = max_over_ranks(
            [res["dec_ms"], res["pre_ms"], res["step_ms"]], device)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peaks, peak_kind = load_peaks()
    T = cfg.n_steps
    dec_us = res["dec_ms"] * 1e3 / T                       # one decode call (attention + merge)
    dflops = decode_flops(cfg)
    value = job_tflops(world, dflops, T, res["dec_ms"])
    per_launch_tflops = dflops / (dec_us * 1e-6) / 1e12
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    pre_gbs = prefill_bytes(cfg) / (res["pre_ms"] * 1e-3) / 1e9
    pre_tflops = prefill_flops(cfg) / (res["pre_ms"] * 1e-3) / 1e12
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    pre_roof_s = max(prefill_bytes(cfg) / (hbm * 1e9), prefill_flops(cfg) / (burst * 1e12))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["step_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_name(cfg), "global_batch": world,
                   "seq_len": cfg.n_chunks * cfg.chunk_size,
                   "l2": "flushed between steps (256 MiB write), outside the timed events",
                   "decode_splits": res["n_splits"], "graphs": "prefill+select; T-step decode loop",
                   "parallelism": f"replicas x{world} (independent requests)"},
        "decode_us_per_step": dec_us,
        "decode_tflops": per_launch_tflops,
        "prefill_us": res["pre_ms"] * 1e3,
        "prefill_gbs": pre_gbs,
        "prefill_tflops": pre_tflops,
        "prefill_roofline_frac": pre_roof_s / (res["pre_ms"] * 1e-3),
        "roofline": {"kernel": "decode attention call (attention_kernel + lse_merge_kernel)",
                     "bound": "tensor", "achieved": per_launch_tflops, "peak": sustained,
                     "peak_kind": f"{peak_kind} bf16 sustained", "unit": "TFLOP/s",
                     "frac": per_launch_tflops / sustained,
                     "traffic": recorded_traffic("decode_attention_8k.md")},
        "prefill_roofline": {"bound": "tensor" if prefill_flops(cfg) / (burst * 1e12) >=
                             prefill_bytes(cfg) / (hbm * 1e9) else "hbm",
                             "achieved_gbs": pre_gbs, "hbm_peak_gbs": hbm,
                             "achieved_tflops": pre_tflops, "tensor_peak_tflops": burst,
                             "frac": pre_roof_s / (res["pre_ms"] * 1e-3),
                             "peak_kind": peak_kind},
        "clocks": res["clocks"],
        "gpu_launches": res["launches"],
        "wall_s_timed_region": res["wall"],
    }
    if "e2e" in res:
        e = res["e2e"]
        line["e2e"] = {"value": job_tflops(world, dflops, T, e["dec_ms"]), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "prefill_ms": e["pre_ms"], "decode_ms": e["dec_ms"],
                       "path": ("C ABI calls (prefill + select, then one decode call per step) "
                                "captured in CUDA graphs with every step's H2D copies from pinned "
                                "host memory and D2H of its output as graph nodes on copy "
                                "streams that overlap the kernels"),
                       "eager_value": job_tflops(world, dflops, T, e["eager_dec_ms"]),
                       "eager_decode_ms": e["eager_dec_ms"],
                       "eager_path": "the same calls and copies issued from Python every step"}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
