"""Parity at the full workload sizes, in the launch configuration bench.py
times: every call of the path runs at full size on the GPU, and sampled
outputs are checked against the oracle one by one.

Per workload:
  - chunk selection: all K, bit-exact;
  - scores and kept tokens of sampled chunks (first, last, a needle chunk, a
    seeded one), scores within rel 1e-4, kept bit-exact outside the tie band;
  - every pool slot: BOS + the kept rows, bit-exact; every table entry;
  - prefill output at sampled rows of the sampled chunks (BOS, first, middle,
    last and seeded rows), all heads;
  - decode output and lse at sampled live rows, all heads, for the first and
    the last denoising step.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
from oracle import pfd_oracle as orc
from sparse_chunked_kv_gb300 import _abi, api
from sparse_chunked_kv_gb300 import workloads as wl
from tests import parity as P

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

f64 = wl.to_f64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    _abi.load()


def _sample_chunks(cfg, req, gen):
    n = cfg.n_chunks
    picks = {0, n - 1, int(torch.randint(0, n, (1,), generator=gen))}
    if req["needle_chunks"]:
        picks.add(int(req["needle_chunks"][0]))
    return sorted(picks)


def _sample_rows(c, gen, extra=6):
    rows = {0, 1, c // 2, c}
    rows.update(int(x) for x in torch.randint(0, c + 1, (extra,), generator=gen))
    return sorted(rows)


def _sample_live(lq, gen, extra=10):
    rows = {0, lq // 2, lq - 1}
    rows.update(int(x) for x in torch.randint(0, lq, (extra,), generator=gen))
    return sorted(rows)


def _check_prefill_chunks(cfg, req, chunks, gen, scores, kept, out, label):
    """Scores, kept tokens and output rows of the sampled chunks."""
    span = cfg.chunk_size + 1
    q, k, v = req["q"], req["k"], req["v"]
    for j in chunks:
        lo = j * span
        k_j = f64(k[lo:lo + span])
        s_ref = orc.window_scores(f64(req["q_win"]), k_j, 1, cfg.chunk_size, cfg.sm_scale)
        s_gpu = scores[j:j + 1].double().numpy()
        tol = P.SCORE_RTOL * np.abs(s_ref) + 1e-6 * cfg.n_win * cfg.n_q_heads
        assert (np.abs(s_gpu - s_ref) <= tol).all(), f"{label} chunk {j}: scores"
        if cfg.n_keep > 0:
            P.check_kept(kept[j:j + 1].numpy(), s_ref, cfg.n_keep)
        local = _sample_rows(cfg.chunk_size, gen)
        o_ref = orc.chunk_attention_rows(f64(q[lo:lo + span]), k_j, f64(v[lo:lo + span]),
                                         cfg.chunk_size, local, cfg.sm_scale)
        got = out[[lo + r for r in local]].double().numpy()
        P.assert_close_out(got, o_ref, f"{label} chunk {j} output rows")


def _check_pool(cfg, req, kept, slot_row, table, pool_k, pool_v, label, table_base=0):
    span = cfg.chunk_size + 1
    k, v = req["k"], req["v"]
    kept = kept.long()
    for j in range(cfg.n_chunks):
        base = int(slot_row[j])
        assert table[table_base + j].tolist() == [base, cfg.n_keep + 1], f"{label} table {j}"
        src = torch.cat([torch.tensor([j * span]), j * span + 1 + kept[j, :cfg.n_keep]])
        n = cfg.n_keep + 1
        assert torch.equal(pool_k[base:base + n].view(torch.int16), k[src].view(torch.int16)), \
            f"{label} pool_k slot {j}"
        assert torch.equal(pool_v[base:base + n].view(torch.int16), v[src].view(torch.int16)), \
            f"{label} pool_v slot {j}"


@pytest.mark.parametrize("name", ["8k", "32k", "128k"])
def test_full_size_request(name):
    cfg = wl.CONFIGS[name]
    dev = torch.device("cuda", 0)
    r = bench.Request(cfg, 0, dev)
    r.prefill_select()
    for t in (0, cfg.n_steps - 1):
        r.decode(t)
    torch.cuda.synchronize()
    assert int(r.dev_err.item()) == 0
    req = r.host
    gen = torch.Generator().manual_seed(4242)

    sel_ref, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    assert r.sel.cpu().tolist() == [int(x) for x in sel_ref], f"{name}: selection"

    scores, kept, out = r.scores.cpu(), r.kept.cpu(), r.out.cpu()
    chunks = _sample_chunks(cfg, req, gen)
    _check_prefill_chunks(cfg, req, chunks, gen, scores, kept, out, name)
    table = r.table.cpu()
    pool_k, pool_v = r.pool_k.cpu(), r.pool_v.cpu()
    _check_pool(cfg, req, kept, req["slot_row"], table, pool_k, pool_v, name)

    pk, pv, tab = f64(pool_k), f64(pool_v), table.numpy()
    for t in (0, cfg.n_steps - 1):
        ql, kl, vl = wl.live_block(req, wl.make_step(cfg, 0, t))
        rows = _sample_live(cfg.n_live, gen)
        o_ref, lse_ref = orc.decode_attention(f64(ql)[rows], f64(kl), f64(vl), pk, pv, tab,
                                              sel_ref, cfg.sm_scale)
        got = r.dec_out[t].cpu()[rows].double().numpy()
        P.assert_close_out(got, o_ref, f"{name} decode step {t}")
        lse = r.dec_lse[t].cpu()[rows].double().numpy()
        assert np.abs(lse - lse_ref).max() <= P.LSE_MAX_ABS, f"{name} decode lse step {t}"


def test_full_size_batched_mix():
    """Eight 32K-prefix sequences with C in {256, 1024, 4096} sharing one
    permuted pool and one chunk table: per-sequence prefill into the shared
    pool, batched selection, and one batched decode call per step."""
    cfgs = wl.mix_configs()
    dev = torch.device("cuda", 0)
    hq, hkv, d = cfgs[0].n_q_heads, cfgs[0].n_kv_heads, cfgs[0].head_dim
    reqs = [wl.make_request(c, i) for i, c in enumerate(cfgs)]
    pool_base, cu_n, cu_k = [0], [0], [0]
    for c in cfgs:
        pool_base.append(pool_base[-1] + c.pool_rows)
        cu_n.append(cu_n[-1] + c.n_chunks)
        cu_k.append(cu_k[-1] + c.n_select)
    pool_rows, table_len = pool_base[-1], cu_n[-1]
    pool_k = torch.zeros(pool_rows, hkv, d, dtype=torch.bfloat16, device=dev)
    pool_v = torch.zeros_like(pool_k)
    table = torch.zeros(table_len, 2, dtype=torch.int32, device=dev)
    prefill = []
    for i, (c, req) in enumerate(zip(cfgs, reqs)):
        slot = (req["slot_row"] + pool_base[i]).to(torch.int32)
        res = api.chunk_prefill(P.cuda(req["q"]), P.cuda(req["k"]), P.cuda(req["v"]),
                                P.cuda(req["q_win"]), c.n_chunks, c.chunk_size, c.n_keep,
                                P.cuda(slot), pool_rows, pool_k=pool_k, pool_v=pool_v)
        table[cu_n[i]:cu_n[i + 1]] = res["table"]
        torch.cuda.synchronize()
        assert int(res["dev_err"][0]) == 0, f"mix{i}: prefill dev_err"
        prefill.append((slot, res["scores"].cpu(), res["kept_idx"].cpu(), res["out"].cpu()))
        del res
    s_i = torch.cat([req["s_i"] for req in reqs]).to(dev)
    s_p = torch.cat([req["s_p"] for req in reqs]).to(dev)
    cu_n_d = torch.tensor(cu_n, dtype=torch.int32, device=dev)
    cu_k_d = torch.tensor(cu_k, dtype=torch.int32, device=dev)
    sel, _ = api.select_chunks_batched(s_i, s_p, cu_n_d, cu_k_d, max(c.n_chunks for c in cfgs))
    torch.cuda.synchronize()
    sel_host = sel.cpu().tolist()

    gen = torch.Generator().manual_seed(777)
    table_h, pool_k_h, pool_v_h = table.cpu(), pool_k.cpu(), pool_v.cpu()
    sel_ref_all = []
    for i, (c, req) in enumerate(zip(cfgs, reqs)):
        sel_ref, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), c.n_select)
        sel_ref = [cu_n[i] + int(x) for x in sel_ref]
        assert sel_host[cu_k[i]:cu_k[i + 1]] == sel_ref, f"mix{i}: selection"
        sel_ref_all.extend(sel_ref)
        slot, scores, kept, out = prefill[i]
        chunks = _sample_chunks(c, req, gen)[:3]
        _check_prefill_chunks(c, req, chunks, gen, scores, kept, out, f"mix{i}")
        _check_pool(c, req, kept, slot, table_h, pool_k_h, pool_v_h, f"mix{i}",
                    table_base=cu_n[i])

    pk, pv, tab = f64(pool_k_h), f64(pool_v_h), table_h.numpy()
    sel_arr = np.array(sel_ref_all, dtype=np.int64)
    for t in (0, cfgs[0].n_steps - 1):
        lives = [wl.live_block(req, wl.make_step(c, i, t)) for i, (c, req) in
                 enumerate(zip(cfgs, reqs))]
        cu_lq = [0]
        for q, _, _ in lives:
            cu_lq.append(cu_lq[-1] + q.shape[0])
        out, lse = api.decode_attention(P.cuda(torch.cat([x[0] for x in lives])),
                                        P.cuda(torch.cat([x[1] for x in lives])),
                                        P.cuda(torch.cat([x[2] for x in lives])), pool_k, pool_v,
                                        table, sel, cu_lq=cu_lq, cu_k=cu_k,
                                        max_chunk_len=max(c.n_keep + 1 for c in cfgs))
        torch.cuda.synchronize()
        out, lse = out.cpu(), lse.cpu()
        for i, (c, (ql, kl, vl)) in enumerate(zip(cfgs, lives)):
            rows = _sample_live(ql.shape[0], gen, extra=4)
            o_ref, lse_ref = orc.decode_attention(f64(ql)[rows], f64(kl), f64(vl), pk, pv, tab,
                                                  sel_arr[cu_k[i]:cu_k[i + 1]], c.sm_scale)
            idx = [cu_lq[i] + r for r in rows]
            P.assert_close_out(out[idx].double().numpy(), o_ref, f"mix{i} decode step {t}")
            assert np.abs(lse[idx].double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS, \
                f"mix{i} decode lse step {t}"
