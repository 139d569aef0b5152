"""pfd_chunk_prefill_ex: the prefill under the other readings of the
intra-chunk ranking ("Two-Level Sparsity"), against the oracle:
  - per KV head: one ranking per (chunk, KV head), each head's slot column
    from its own kept set;
  - window keys in the denominator: the window rows' softmax over the
    chunk's keys and the W window keys.
Scores within the score tolerance, kept sets bit-exact outside the 1e-5 tie
band, pool bytes bit-exact per KV head, chunk-attention output unchanged,
and a decode step over the pool the call wrote.  The base mode (shared
ranking, chunk keys only) gives the bits of pfd_chunk_prefill."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import pfd_oracle as orc
from sparse_chunked_kv_gb300 import _abi, api
from sparse_chunked_kv_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

f64 = wl.to_f64

SHAPES = {
    "d64": wl.scaled(wl.TINY, n_chunks=4, chunk_size=96, n_keep=24, n_select=2, n_win=8,
                     n_resp=24),
    "gqa7": wl.scaled(wl.CTX_8K, n_chunks=3, chunk_size=200, n_keep=50, n_select=2, n_win=16,
                      n_resp=40),
    "8k": wl.CTX_8K,
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    _abi.load()


def _run(cfg, req, per_kv_head, window_keys):
    return api.chunk_prefill_ex(P.cuda(req["q"]), P.cuda(req["k"]), P.cuda(req["v"]),
                                P.cuda(req["q_win"]),
                                P.cuda(req["k_win"]) if window_keys else None, cfg.n_chunks,
                                cfg.chunk_size, cfg.n_keep, P.cuda(req["slot_row"]),
                                cfg.pool_rows, per_kv_head=per_kv_head)


@pytest.mark.parametrize("name", ["d64", "gqa7", "8k"])
@pytest.mark.parametrize("per_kv_head,window_keys", [(True, False), (False, True), (True, True)])
def test_rank_readings(name, per_kv_head, window_keys):
    cfg = SHAPES[name]
    req = wl.make_request(cfg, 0)
    res = _run(cfg, req, per_kv_head, window_keys)
    torch.cuda.synchronize()
    assert int(res["dev_err"].item()) == 0
    k, v = f64(req["k"]), f64(req["v"])
    s_ref = orc.window_scores_alt(f64(req["q_win"]), k, cfg.n_chunks, cfg.chunk_size, cfg.sm_scale,
                                  per_kv_head=per_kv_head,
                                  k_win=f64(req["k_win"]) if window_keys else None)
    s_gpu = res["scores"].cpu().double().numpy()
    assert s_gpu.shape == s_ref.shape
    tol = P.score_tol(s_ref, cfg.n_win, cfg.n_q_heads)
    assert (np.abs(s_gpu - s_ref) <= tol).all(), f"{name}: scores"
    rows = cfg.chunk_size + 1
    kept = res["kept_idx"].cpu().numpy()
    P.check_kept(kept.reshape(-1, cfg.n_keep), s_ref.reshape(-1, rows), cfg.n_keep)

    # pool: BOS + kept rows, per KV head when ranked per head
    pool_k, pool_v = res["pool_k"].cpu(), res["pool_v"].cpu()
    kh, vh = req["k"], req["v"]
    table = res["table"].cpu()
    for j in range(cfg.n_chunks):
        base = int(req["slot_row"][j])
        assert table[j].tolist() == [base, cfg.n_keep + 1]
        for g in range(cfg.n_kv_heads):
            kj = kept[j, g] if per_kv_head else kept[j]
            src = torch.tensor([j * rows] + [j * rows + 1 + int(t) for t in kj])
            n = cfg.n_keep + 1
            assert torch.equal(pool_k[base:base + n, g].view(torch.int16),
                               kh[src, g].view(torch.int16)), f"{name}: pool_k slot {j} head {g}"
            assert torch.equal(pool_v[base:base + n, g].view(torch.int16),
                               vh[src, g].view(torch.int16)), f"{name}: pool_v slot {j} head {g}"

    # chunk attention does not depend on the ranking
    some = [0, 1, rows - 1, rows + 3, cfg.n_chunks * rows - 1]
    o_ref = orc.chunk_attention_rows(f64(req["q"]), k, v, cfg.chunk_size, some, cfg.sm_scale)
    P.assert_close_out(res["out"].cpu()[some].double().numpy(), o_ref, f"{name}: prefill rows")

    # a decode step over the pool this call wrote
    sel_ref, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    ql, kl, vl = wl.live_block(req, wl.make_step(cfg, 0, 0))
    out, lse = api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), res["pool_k"],
                                    res["pool_v"], res["table"],
                                    P.cuda(torch.from_numpy(sel_ref)))
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), f64(pool_k), f64(pool_v),
                                          table.numpy(), sel_ref, cfg.sm_scale)
    P.assert_close_out(out.cpu().double().numpy(), o_ref, f"{name}: decode over the pool")
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS


def test_base_mode_is_pfd_chunk_prefill():
    cfg = SHAPES["gqa7"]
    req = wl.make_request(cfg, 1)
    a = _run(cfg, req, False, False)
    b = api.chunk_prefill(P.cuda(req["q"]), P.cuda(req["k"]), P.cuda(req["v"]),
                          P.cuda(req["q_win"]), cfg.n_chunks, cfg.chunk_size, cfg.n_keep,
                          P.cuda(req["slot_row"]), cfg.pool_rows)
    torch.cuda.synchronize()
    for key in ("out", "scores", "kept_idx", "pool_k", "pool_v", "table"):
        assert torch.equal(a[key], b[key]), key
