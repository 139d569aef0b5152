"""pfd_chunk_prefill_layers: L layers' prefill in one call, one pool per
layer.  Against L separate pfd_chunk_prefill calls (the same bits: the same
kernels run every layer's items), and against the oracle layer by layer:
scores, kept sets (tie band), every pool slot, the tables, and sampled
prefill rows of every chunk."""
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
    "small": (wl.scaled(wl.CTX_8K, n_chunks=3, chunk_size=200, n_keep=50, n_win=16), 3),
    "d64": (wl.scaled(wl.TINY, n_chunks=5, chunk_size=70, n_keep=20, n_win=12), 2),
    "8k_x4": (wl.CTX_8K, 4),
    "128k_like_x2": (wl.scaled(wl.CTX_128K, n_chunks=64), 2),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    _abi.load()


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_layers_match_single_calls_and_oracle(name):
    cfg, n_layers = SHAPES[name]
    lay = wl.make_layers(cfg, n_layers)
    slot = P.cuda(lay["slot_row"])
    res = api.chunk_prefill_layers(P.cuda(lay["q"]), P.cuda(lay["k"]), P.cuda(lay["v"]),
                                   P.cuda(lay["q_win"]), cfg.n_chunks, cfg.chunk_size,
                                   cfg.n_keep, slot, cfg.pool_rows)
    torch.cuda.synchronize()
    assert int(res["dev_err"].item()) == 0
    rows = cfg.chunk_size + 1
    gen = torch.Generator().manual_seed(9)
    for l in range(n_layers):
        single = api.chunk_prefill(P.cuda(lay["q"][l]), P.cuda(lay["k"][l]), P.cuda(lay["v"][l]),
                                   P.cuda(lay["q_win"][l]), cfg.n_chunks, cfg.chunk_size,
                                   cfg.n_keep, slot, cfg.pool_rows)
        torch.cuda.synchronize()
        for key in ("out", "scores", "kept_idx", "pool_k", "pool_v", "table"):
            assert torch.equal(res[key][l], single[key]), f"{name} layer {l}: {key} differs"
        req = lay["layers"][l]
        k, v = f64(req["k"]), f64(req["v"])
        s_ref = orc.window_scores(f64(req["q_win"]), k, cfg.n_chunks, cfg.chunk_size, cfg.sm_scale)
        s_gpu = res["scores"][l].cpu().double().numpy()
        assert (np.abs(s_gpu - s_ref) <= P.score_tol(s_ref, cfg.n_win, cfg.n_q_heads)).all()
        kept = res["kept_idx"][l].cpu()
        P.check_kept(kept.numpy(), s_ref, cfg.n_keep)
        table = res["table"][l].cpu()
        pk, pv = res["pool_k"][l].cpu(), res["pool_v"][l].cpu()
        for j in range(cfg.n_chunks):
            base = int(lay["slot_row"][j])
            assert table[j].tolist() == [base, cfg.n_keep + 1]
            src = torch.cat([torch.tensor([j * rows]), j * rows + 1 + kept[j].long()])
            assert torch.equal(pk[base:base + cfg.n_keep + 1].view(torch.int16),
                               req["k"][src].view(torch.int16))
            assert torch.equal(pv[base:base + cfg.n_keep + 1].view(torch.int16),
                               req["v"][src].view(torch.int16))
        pick = []
        for j in range(cfg.n_chunks):
            pick += [j * rows, j * rows + 1, j * rows + rows - 1,
                     j * rows + int(torch.randint(0, rows, (1,), generator=gen))]
        o_ref = orc.chunk_attention_rows(f64(req["q"]), k, v, cfg.chunk_size, pick, cfg.sm_scale)
        P.assert_close_out(res["out"][l].cpu()[pick].double().numpy(), o_ref,
                           f"{name} layer {l}: prefill rows")


BATCH_SHAPES = {
    "small_x3": (wl.scaled(wl.CTX_8K, n_chunks=3, chunk_size=200, n_keep=50, n_win=16), 3),
    "d64_x2": (wl.scaled(wl.TINY, n_chunks=5, chunk_size=70, n_keep=20, n_win=12), 2),
    "mix_c256_x3": (wl.scaled(wl.mix_configs()[0], n_chunks=16), 3),
}


@pytest.mark.parametrize("name", sorted(BATCH_SHAPES))
def test_batch_matches_single_calls_into_one_pool(name):
    """pfd_chunk_prefill_batch: L same-shaped requests, each with its own
    permuted slots in one shared pool (request l's slots offset by l pools
    and reversed for odd l), against L pfd_chunk_prefill calls into the same
    pool: every output, the whole pool and the table, bit for bit, and the
    scores and kept sets against the oracle."""
    cfg, n_req = BATCH_SHAPES[name]
    reqs = [wl.make_request(cfg, seq) for seq in range(n_req)]
    slots = []
    for l, r in enumerate(reqs):
        s = r["slot_row"].clone() if l % 2 == 0 else r["slot_row"].flip(0).clone()
        slots.append(s + l * cfg.pool_rows)
    pool_rows = n_req * cfg.pool_rows
    stack = lambda key: P.cuda(torch.stack([r[key] for r in reqs]))  # noqa: E731
    slot_b = P.cuda(torch.stack(slots).to(torch.int32))
    hkv, d = cfg.n_kv_heads, cfg.head_dim
    pk_b = torch.zeros(pool_rows, hkv, d, dtype=torch.bfloat16, device="cuda")
    pv_b = torch.zeros_like(pk_b)
    tab_b = torch.zeros(n_req, cfg.n_chunks, 2, dtype=torch.int32, device="cuda")
    res = api.chunk_prefill_batch(stack("q"), stack("k"), stack("v"), stack("q_win"),
                                  cfg.n_chunks, cfg.chunk_size, cfg.n_keep, slot_b, pk_b, pv_b,
                                  tab_b)
    torch.cuda.synchronize()
    assert int(res["dev_err"].item()) == 0
    pk_s, pv_s = torch.zeros_like(pk_b), torch.zeros_like(pv_b)
    for l, r in enumerate(reqs):
        single = api.chunk_prefill(P.cuda(r["q"]), P.cuda(r["k"]), P.cuda(r["v"]),
                                   P.cuda(r["q_win"]), cfg.n_chunks, cfg.chunk_size, cfg.n_keep,
                                   P.cuda(slots[l].to(torch.int32)), pool_rows)
        torch.cuda.synchronize()
        assert int(single["dev_err"].item()) == 0
        for key in ("out", "scores", "kept_idx"):
            assert torch.equal(res[key][l], single[key]), f"{name} request {l}: {key} differs"
        assert torch.equal(tab_b[l], single["table"]), f"{name} request {l}: table differs"
        for j in range(cfg.n_chunks):
            base = int(slots[l][j])
            n = cfg.n_keep + 1
            pk_s[base:base + n] = single["pool_k"][base:base + n]
            pv_s[base:base + n] = single["pool_v"][base:base + n]
        s_ref = orc.window_scores(f64(r["q_win"]), f64(r["k"]), cfg.n_chunks, cfg.chunk_size,
                                  cfg.sm_scale)
        s_gpu = res["scores"][l].cpu().double().numpy()
        assert (np.abs(s_gpu - s_ref) <= P.score_tol(s_ref, cfg.n_win, cfg.n_q_heads)).all()
        P.check_kept(res["kept_idx"][l].cpu().numpy(), s_ref, cfg.n_keep)
    assert torch.equal(pk_b.view(torch.int16), pk_s.view(torch.int16)), f"{name}: pool_k"
    assert torch.equal(pv_b.view(torch.int16), pv_s.view(torch.int16)), f"{name}: pool_v"
