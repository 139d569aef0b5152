"""The host-side check behind __graft_entry__.smoke(): it accepts results
that equal the oracle's and rejects each kind of wrong result a kernel could
return (no GPU needed: the "GPU" results here are built from the oracle)."""
import copy

import numpy as np
import pytest
import torch

import __graft_entry__ as entry
from oracle import pfd_oracle as orc
from sparse_chunked_kv_gb300 import workloads as wl


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


@pytest.fixture(scope="module")
def case():
    cfg = entry.smoke_config()
    req = wl.make_request(cfg, 0)
    live = wl.live_block(req, wl.make_step(cfg, 0, 0))
    f = wl.to_f64
    n, c, b = cfg.n_chunks, cfg.chunk_size, cfg.n_keep
    rows = c + 1
    scores = orc.window_scores(f(req["q_win"]), f(req["k"]), n, c, cfg.sm_scale)
    kept = orc.top_b(scores, b)
    pool_k = torch.zeros(cfg.pool_rows, cfg.n_kv_heads, cfg.head_dim, dtype=torch.bfloat16)
    pool_v = pool_k.clone()
    table = torch.empty(n, 2, dtype=torch.int32)
    for j in range(n):
        base = int(req["slot_row"][j])
        src = torch.tensor([j * rows] + [j * rows + 1 + int(t) for t in kept[j]])
        pool_k[base:base + b + 1] = req["k"][src]
        pool_v[base:base + b + 1] = req["v"][src]
        table[j] = torch.tensor([base, b + 1])
    sel, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    out = orc.chunk_attention(f(req["q"]), f(req["k"]), f(req["v"]), n, c, cfg.sm_scale)
    dec, lse = orc.decode_attention(*(f(x) for x in live), pool_k.double().numpy(),
                                    pool_v.double().numpy(), table.numpy(), sel, cfg.sm_scale)
    kept_buf = torch.zeros(n, b + 3, dtype=torch.int32)        # a strided view, as the API returns
    kept_buf[:, :b] = torch.from_numpy(kept)
    res = dict(out=_bf16(out), scores=torch.from_numpy(scores.astype(np.float32)),
               kept_idx=kept_buf[:, :b], table=table, pool_k=pool_k, pool_v=pool_v)
    got = entry.smoke_results(res, torch.from_numpy(sel.astype(np.int32)), _bf16(dec),
                              torch.from_numpy(lse.astype(np.float32)))
    return cfg, req, live, got


def test_oracle_results_pass(case):
    entry.smoke_check(*case)


def _planted(got, what):
    bad = copy.deepcopy(got)
    if what == "kept_token":
        j = 1
        row = [int(t) for t in bad["kept"][j]]
        spare = next(t for t in range(100) if t not in row)
        row[-1] = spare
        bad["kept"][j] = sorted(row)
    elif what == "kept_order":
        bad["kept"][0] = bad["kept"][0][::-1]
    elif what == "pool_row":
        base = int(bad["table"][2][0])
        bad["pool_k_bits"][base + 3] = bad["pool_k_bits"][base + 4]
    elif what == "pool_bos":
        base = int(bad["table"][0][0])
        bad["pool_v_bits"][base] = 0
    elif what == "table_len":
        bad["table"][3][1] += 1
    elif what == "sel_order":
        bad["sel"] = bad["sel"][::-1]
    elif what == "scores_shift":
        bad["scores"] = np.roll(bad["scores"], 1, axis=1)
    elif what == "prefill_out":
        bad["out"] = bad["out"] * 1.05
    elif what == "decode_out":
        bad["dec_out"] = bad["dec_out"][:, ::-1]
    elif what == "lse":
        bad["lse"] = bad["lse"] + 2e-3
    elif what == "nan":
        bad["dec_out"][0, 0, 0] = np.nan
    return bad


@pytest.mark.parametrize("what", ["kept_token", "kept_order", "pool_row", "pool_bos",
                                  "table_len", "sel_order", "scores_shift", "prefill_out",
                                  "decode_out", "lse", "nan"])
def test_each_wrong_result_fails(case, what):
    cfg, req, live, got = case
    with pytest.raises(AssertionError):
        entry.smoke_check(cfg, req, live, _planted(got, what))
