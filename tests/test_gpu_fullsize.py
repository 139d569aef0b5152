"""Parity at the full workload sizes, in the launch configuration bench.py
times (its Job: per-sequence prefill into one shared pool, selection, one
batched decode call per step), with whole outputs compared to the oracle.

Per workload (8K, 32K, 128K, and all eight sequences of the batched mix):
  - chunk selection: all K of every sequence, bit-exact;
  - window scores of every chunk within the score tolerance, and every
    chunk's kept tokens bit-exact outside the 1e-5 tie band;
  - every pool slot (BOS + the kept rows) bit-exact, every table entry;
  - prefill output: every row of every chunk at 8K and 32K; at 128K and in
    the mix, every chunk's BOS, first and last rows plus 64 seeded rows;
  - decode output and lse: every live row, all heads, of the first and the
    last denoising step.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
from oracle import pfd_oracle as orc
from sparse_chunked_kv_gb300 import _abi
from sparse_chunked_kv_gb300 import workloads as wl
from tests import parity as P

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

f64 = wl.to_f64

# Workloads whose prefill output is compared at every row.
FULL_PREFILL_ROWS = {"8k", "32k"}
SEEDED_ROWS = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    _abi.load()


def _prefill_rows(cfg, gen):
    """Prefix rows checked at 128K and in the mix: each chunk's BOS, first
    and last content rows and SEEDED_ROWS seeded rows."""
    span = cfg.chunk_size + 1
    rows = []
    for j in range(cfg.n_chunks):
        pick = {0, 1, span - 1}
        pick.update(int(x) for x in torch.randint(0, span, (SEEDED_ROWS,), generator=gen))
        rows.extend(j * span + r for r in sorted(pick))
    return rows


def _check_prefill(name, cfg, req, scores, kept, out, gen, label):
    """Scores and kept tokens of every chunk; output rows as stated above."""
    q, k, v = f64(req["q"]), f64(req["k"]), f64(req["v"])
    s_ref = orc.window_scores(f64(req["q_win"]), k, cfg.n_chunks, cfg.chunk_size, cfg.sm_scale)
    s_gpu = scores.double().numpy()
    tol = P.score_tol(s_ref, cfg.n_win, cfg.n_q_heads)
    bad = np.argwhere(np.abs(s_gpu - s_ref) > tol)
    assert bad.size == 0, f"{label}: scores outside tolerance at {bad[:5].tolist()}"
    if cfg.n_keep > 0:
        P.check_kept(kept.numpy(), s_ref, cfg.n_keep)
    if name in FULL_PREFILL_ROWS:
        o_ref = orc.chunk_attention(q, k, v, cfg.n_chunks, cfg.chunk_size, cfg.sm_scale)
        P.assert_close_out(out.double().numpy(), o_ref, f"{label}: every prefill row")
    else:
        rows = _prefill_rows(cfg, gen)
        o_ref = orc.chunk_attention_rows(q, k, v, cfg.chunk_size, rows, cfg.sm_scale)
        P.assert_close_out(out[rows].double().numpy(), o_ref,
                           f"{label}: BOS/first/last + {SEEDED_ROWS} seeded rows of every chunk")


def _check_pool(cfg, req, kept, table, pool_k, pool_v, label, table_base):
    span = cfg.chunk_size + 1
    k, v = req["k"], req["v"]
    kept = kept.long()
    for j in range(cfg.n_chunks):
        base = int(req["slot_row"][j])
        assert table[table_base + j].tolist() == [base, cfg.n_keep + 1], f"{label} table {j}"
        src = torch.cat([torch.tensor([j * span]), j * span + 1 + kept[j, :cfg.n_keep]])
        n = cfg.n_keep + 1
        assert torch.equal(pool_k[base:base + n].view(torch.int16), k[src].view(torch.int16)), \
            f"{label} pool_k slot {j}"
        assert torch.equal(pool_v[base:base + n].view(torch.int16), v[src].view(torch.int16)), \
            f"{label} pool_v slot {j}"


@pytest.mark.parametrize("name", ["8k", "32k", "128k", "mix"])
def test_full_size_job(name):
    dev = torch.device("cuda", 0)
    job = bench.Job(bench.job_configs(name), 0, dev)
    cfgs = job.cfgs   # the job's order: sequences of one prefill shape together
    job.prefill_select()
    last = job.T - 1
    for t in (0, last):
        job.decode(t)
    torch.cuda.synchronize()
    assert int(job.dev_err.item()) == 0
    gen = torch.Generator().manual_seed(4242)
    table = job.table.cpu()
    pool_k, pool_v = job.pool_k.cpu(), job.pool_v.cpu()
    sel_host = job.sel.cpu().tolist()
    sel_ref_all = []
    for i, (c, req, sq) in enumerate(zip(cfgs, job.host, job.seqs)):
        label = c.name
        n0, k0, k1 = job.cu_n_host[i], job.cu_k_host[i], job.cu_k_host[i + 1]
        sel_ref, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), c.n_select)
        sel_ref = [n0 + int(x) for x in sel_ref]
        assert sel_host[k0:k1] == sel_ref, f"{label}: selection"
        sel_ref_all.extend(sel_ref)
        kept = sq["kept"][:, :c.n_keep].cpu()
        _check_prefill(name, c, req, sq["scores"].cpu(), kept, sq["out"].cpu(), gen, label)
        _check_pool(c, req, kept, table, pool_k, pool_v, label, n0)

    pk, pv, tab = f64(pool_k), f64(pool_v), table.numpy()
    sel_arr = np.array(sel_ref_all, dtype=np.int64)
    for t in (0, last):
        out, lse = job.dec_out[t].cpu(), job.dec_lse[t].cpu()
        for i, (c, req) in enumerate(zip(cfgs, job.host)):
            ql, kl, vl = wl.live_block(req, wl.make_step(c, job.seq_ids[i], t))
            o_ref, lse_ref = orc.decode_attention(
                f64(ql), f64(kl), f64(vl), pk, pv, tab,
                sel_arr[job.cu_k_host[i]:job.cu_k_host[i + 1]], c.sm_scale)
            lo, hi = job.cu_lq_host[i], job.cu_lq_host[i + 1]
            P.assert_close_out(out[lo:hi].double().numpy(), o_ref,
                               f"{c.name} decode step {t}, every live row")
            err = np.abs(lse[lo:hi].double().numpy() - lse_ref).max()
            assert err <= P.LSE_MAX_ABS, f"{c.name} decode lse step {t}: {err:.3e}"
