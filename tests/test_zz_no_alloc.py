"""pfd_decode_attention_static_scratch: the decode call whose split partials
live in the library's static device scratch, for callers that cannot
allocate device memory where they call (a host program linking only libpfd,
a hook inside a runtime that owns every device byte).  Called through the C
ABI and compared with pfd_decode_attention (caller workspace) at the same
split count, bit for bit, on two calls in a row, and with the oracle; checked
to change neither the device's free memory nor torch's allocated bytes."""
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


def _static_splits(cu_lq_host, cu_k_host, hq, hkv, d, max_chunk_len):
    """The split count pfd_decode_attention_static_scratch uses with
    n_splits == 0: the plan, lowered until its partials fit the scratch."""
    batch = len(cu_lq_host) - 1
    s = _abi.pfd_decode_plan_splits(batch, cu_lq_host, cu_k_host, hq, hkv, d, max_chunk_len)
    while s > 1 and _abi.pfd_decode_workspace(batch, cu_lq_host, cu_k_host, hq, hkv, d,
                                              max_chunk_len, s) > _abi.DECODE_STATIC_SCRATCH_BYTES:
        s -= 1
    return s


class _Call:
    """Device arguments of one decode step, allocated up front so that the
    static-scratch call itself can be checked to allocate nothing."""

    def __init__(self, q, k, v, pk, pv, table, sel, cu_lq_host, cu_k_host, max_chunk_len):
        self.q, self.k, self.v, self.pk, self.pv, self.table, self.sel = q, k, v, pk, pv, table, sel
        self.cu_lq_host, self.cu_k_host = list(cu_lq_host), list(cu_k_host)
        self.cu_lq = torch.tensor(self.cu_lq_host, dtype=torch.int32, device="cuda")
        self.cu_k = torch.tensor(self.cu_k_host, dtype=torch.int32, device="cuda")
        self.hq, self.d = q.shape[1], q.shape[2]
        self.hkv = k.shape[1]
        self.max_len = max_chunk_len
        self.out = torch.empty_like(q)
        self.lse = torch.empty(q.shape[0], self.hq, dtype=torch.float32, device="cuda")
        self.dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def static(self, n_splits):
        _abi.pfd_decode_attention_static_scratch(
            self.q, self.k, self.v, self.cu_lq, self.cu_lq_host, self.pk, self.pv,
            self.pk.shape[0], self.table, self.table.shape[0], self.sel, self.cu_k,
            self.cu_k_host, len(self.cu_lq_host) - 1, self.hq, self.hkv, self.d, self.max_len,
            0.0, n_splits, self.out, self.lse, self.dev_err)
        return self.out, self.lse

    def workspace(self, n_splits):
        return api.decode_attention(self.q, self.k, self.v, self.pk, self.pv, self.table,
                                    self.sel, cu_lq=self.cu_lq_host, cu_k=self.cu_k_host,
                                    n_splits=n_splits, max_chunk_len=self.max_len)

    def splits(self, n_splits):
        return n_splits or _static_splits(self.cu_lq_host, self.cu_k_host, self.hq, self.hkv,
                                          self.d, self.max_len)


def _check_allocates_nothing(call, n_splits):
    """After a warm-up call, a static-scratch call changes neither the
    device's free memory nor torch's allocated bytes."""
    call.static(n_splits)
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    call.static(n_splits)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "the static-scratch call changed free memory"
    assert torch.cuda.memory_allocated() == alloc0


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
        call = _Call(dq, dk, dv, dpk, dpv, dtab, dsel, [0, ql.shape[0]], [0, sel.shape[0]],
                     max_len)
        if step == 0:
            _check_allocates_nothing(call, n_splits)
        out_s, lse_s = call.static(n_splits)
        out_w, lse_w = call.workspace(call.splits(n_splits))
        torch.cuda.synchronize()
        assert int(call.dev_err.item()) == 0
        # Same kernels, same split count: the same bits.
        assert torch.equal(out_s, out_w), f"static scratch vs workspace out (step {step})"
        assert torch.equal(lse_s, lse_w), f"static scratch vs workspace lse (step {step})"
        got = out_s.cpu().double().numpy()
        o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel,
                                              cfg.sm_scale)
        P.assert_close_out(got, o_ref, f"static scratch vs oracle (step {step})")
        assert np.abs(lse_s.cpu().double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS


def _random_batch(seed, lqs, chunk_lens, hq=28, hkv=4, d=128):
    """A batched step over a random pool: sequence b has lqs[b] live rows and
    selects the chunks of lengths chunk_lens[b] (slots in a permuted pool)."""
    gen = torch.Generator().manual_seed(seed)
    lens = [n for seq in chunk_lens for n in seq]
    order = torch.randperm(len(lens), generator=gen).tolist()
    rows, table = 0, [None] * len(lens)
    for i in order:
        table[i] = [rows, lens[i]]
        rows += lens[i]
    pool_k = torch.randn(rows, hkv, d, generator=gen).to(torch.bfloat16)
    pool_v = torch.randn(rows, hkv, d, generator=gen).to(torch.bfloat16)
    total = sum(lqs)
    q = torch.randn(total, hq, d, generator=gen).to(torch.bfloat16)
    k = torch.randn(total, hkv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(total, hkv, d, generator=gen).to(torch.bfloat16)
    cu_lq, cu_k = [0], [0]
    for lq, seq in zip(lqs, chunk_lens):
        cu_lq.append(cu_lq[-1] + lq)
        cu_k.append(cu_k[-1] + len(seq))
    sel = torch.arange(len(lens), dtype=torch.int32)
    return _Call(P.cuda(q), P.cuda(k), P.cuda(v), P.cuda(pool_k), P.cuda(pool_v),
                 P.cuda(torch.tensor(table, dtype=torch.int32)), P.cuda(sel), cu_lq, cu_k,
                 max(lens))


@pytest.mark.gpu
@pytest.mark.parametrize("shape", ["mix256", "long1024"])
def test_static_scratch_lowers_splits_to_fit(shape):
    """n_splits == 0 on sizes whose planned split count needs more than the
    static scratch: the call lowers the count until the partials fit, runs,
    allocates nothing, and gives the bits of the workspace call at that
    count, on two calls in a row."""
    if shape == "mix256":
        # eight sequences, C in {256, 1024, 4096} with B = C/4 and K*C = 8K
        per = [[65] * 32, [257] * 8, [1025] * 2]
        call = _random_batch(11, [256] * 8, [per[i % 3] for i in range(8)])
    else:
        call = _random_batch(12, [1024], [[129] * 128])
    b = len(call.cu_lq_host) - 1
    plan = _abi.pfd_decode_plan_splits(b, call.cu_lq_host, call.cu_k_host, call.hq, call.hkv,
                                       call.d, call.max_len)
    need = _abi.pfd_decode_workspace(b, call.cu_lq_host, call.cu_k_host, call.hq, call.hkv,
                                     call.d, call.max_len, plan)
    assert need > _abi.DECODE_STATIC_SCRATCH_BYTES, "case must exceed the scratch at its plan"
    s = call.splits(0)
    assert 1 < s < plan
    _check_allocates_nothing(call, 0)
    for _ in range(2):
        out_s, lse_s = (x.clone() for x in call.static(0))
        out_w, lse_w = call.workspace(s)
        torch.cuda.synchronize()
        assert int(call.dev_err.item()) == 0
        assert torch.equal(out_s, out_w) and torch.equal(lse_s, lse_w)


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
    call = _Call(q, k, k, pk, pk, table, sel, [0, total_lq], [0, 1], 64)
    with pytest.raises(_abi.PfdError, match="PFD_ERR_UNSUPPORTED"):
        call.static(n_splits)
