"""pfd_decode_attention_static_scratch: the decode call whose split partials
live in the library's static device scratch.  Called through the C ABI and
compared with pfd_decode_attention (caller workspace) on two calls in a row,
and with the oracle."""
from __future__ import annotations

import os
import re

import numpy as np
import pytest
import torch

from tests import parity as P
from oracle import pfd_oracle as orc
from sparse_chunked_kv_gb300 import _abi, api
from sparse_chunked_kv_gb300 import workloads as wl

f64 = wl.to_f64


def test_scratch_size_matches_header():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "pfd.h")).read()
    m = re.search(r"#define PFD_DECODE_STATIC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m is not None
    assert int(m.group(1)) << int(m.group(2)) == _abi.DECODE_STATIC_SCRATCH_BYTES


def _step_inputs(cfg, step):
    req = wl.make_request(cfg, 0)
    scores = orc.window_scores(f64(req["q_win"]), f64(req["k"]), cfg.n_chunks, cfg.chunk_size,
                               cfg.sm_scale)
    kept = orc.top_b(scores, cfg.n_keep)
    pk, pv, table = P.oracle_pool(cfg, req, kept, req["slot_row"], cfg.pool_rows)
    sel, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    ql, kl, vl = wl.live_block(req, wl.make_step(cfg, 0, step))
    return pk, pv, table, sel, ql, kl, vl


def _static_call(q, k, v, pk, pv, table, sel, n_splits, max_chunk_len):
    total_lq, hq, d = q.shape
    hkv = k.shape[1]
    cu_lq_host, cu_k_host = [0, total_lq], [0, sel.shape[0]]
    cu_lq = torch.tensor(cu_lq_host, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(cu_k_host, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(total_lq, hq, dtype=torch.float32, device="cuda")
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _abi.pfd_decode_attention_static_scratch(q, k, v, cu_lq, cu_lq_host, pk, pv, pk.shape[0],
                                             table, table.shape[0], sel, cu_k, cu_k_host, 1, hq,
                                             hkv, d, max_chunk_len, 0.0, n_splits, out, lse,
                                             dev_err)
    return out, lse, dev_err


@pytest.mark.gpu
@pytest.mark.parametrize("n_splits", [3, 0])
def test_static_scratch_matches_workspace_call(n_splits):
    cfg = wl.scaled(wl.CTX_8K, n_chunks=6, n_select=3, n_resp=100)
    for step in (0, 1):   # two calls in a row reuse the same scratch
        pk, pv, table, sel, ql, kl, vl = _step_inputs(cfg, step)
        dq, dk, dv = P.cuda(ql), P.cuda(kl), P.cuda(vl)
        dpk, dpv = P.cuda(P.bf16_of(pk)), P.cuda(P.bf16_of(pv))
        dtab, dsel = P.cuda(torch.from_numpy(table)), P.cuda(torch.from_numpy(sel))
        max_len = int(table[:, 1].max())
        out_s, lse_s, err_s = _static_call(dq, dk, dv, dpk, dpv, dtab, dsel, n_splits, max_len)
        out_w, lse_w = api.decode_attention(dq, dk, dv, dpk, dpv, dtab, dsel, n_splits=n_splits)
        torch.cuda.synchronize()
        assert int(err_s.item()) == 0
        got, want = out_s.cpu().double().numpy(), out_w.cpu().double().numpy()
        P.assert_close_out(got, want, f"static scratch vs workspace (step {step})")
        assert np.abs(lse_s.cpu().double().numpy() - lse_w.cpu().double().numpy()).max() \
            <= P.LSE_MAX_ABS
        o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel,
                                              cfg.sm_scale)
        P.assert_close_out(got, o_ref, f"static scratch vs oracle (step {step})")
        assert np.abs(lse_s.cpu().double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS


@pytest.mark.gpu
def test_static_scratch_rejects_oversized_work():
    """Sizes whose split partials exceed the static scratch are refused on the
    host with PFD_ERR_UNSUPPORTED; nothing is launched.  The tensors are sized
    for the call all the same."""
    total_lq, hq, hkv, d, n_splits = 2048, 28, 4, 128, 64
    need = _abi.pfd_decode_workspace(1, [0, total_lq], [0, 1], hq, hkv, d, 64, n_splits)
    assert need > _abi.DECODE_STATIC_SCRATCH_BYTES
    q = torch.zeros(total_lq, hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(total_lq, hkv, d, dtype=torch.bfloat16, device="cuda")
    pk = torch.zeros(64, hkv, d, dtype=torch.bfloat16, device="cuda")
    table = torch.tensor([[0, 64]], dtype=torch.int32, device="cuda")
    sel = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(_abi.PfdError, match="PFD_ERR_UNSUPPORTED"):
        _static_call(q, k, k, pk, pk, table, sel, n_splits, 64)
