"""The decode step split across devices, on one GPU through the C ABI:
partials (pfd_decode_partial) over disjoint parts of the selection, the
live block's keys in one part only, merged by pfd_lse_merge, equal one
pfd_decode_attention call and the oracle.  The parts follow the chunk-range
ownership of sparse_chunked_kv_gb300.multigpu, as the ranks of a multi-GPU
job would compute them."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import pfd_oracle as orc
from sparse_chunked_kv_gb300 import _abi, api
from sparse_chunked_kv_gb300 import multigpu as mg
from sparse_chunked_kv_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

f64 = wl.to_f64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    _abi.load()


def _batch(seed, lqs, n_chunks, n_sel, slot_len, hq=28, hkv=4, d=128):
    """Sequences b with lqs[b] live rows, n_chunks[b] chunks of slot_len[b]
    pool rows each (permuted slots, one shared table) and n_sel[b] selected
    chunks (a seeded choice, in rank order)."""
    gen = torch.Generator().manual_seed(seed)
    cu_n, cu_k, cu_lq, lens, sel = [0], [0], [0], [], []
    for lq, n, k, ln in zip(lqs, n_chunks, n_sel, slot_len):
        sel.extend(cu_n[-1] + int(x) for x in torch.randperm(n, generator=gen)[:k])
        cu_n.append(cu_n[-1] + n)
        cu_k.append(cu_k[-1] + k)
        cu_lq.append(cu_lq[-1] + lq)
        lens.extend([ln] * n)
    order = torch.randperm(len(lens), generator=gen).tolist()
    row, table = 0, [None] * len(lens)
    for i in order:
        table[i] = [row, lens[i]]
        row += lens[i]
    bf = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)  # noqa: E731
    return dict(pk=bf(row, hkv, d), pv=bf(row, hkv, d), q=bf(cu_lq[-1], hq, d),
                k=bf(cu_lq[-1], hkv, d), v=bf(cu_lq[-1], hkv, d),
                table=torch.tensor(table, dtype=torch.int32), sel=sel, cu_n=cu_n, cu_k=cu_k,
                cu_lq=cu_lq, scale=1.0 / np.sqrt(d))


def _dev(pr):
    return {k: P.cuda(pr[k]) for k in ("pk", "pv", "q", "k", "v", "table")}


@pytest.mark.parametrize("world,shape", [(2, "8k"), (3, "mix"), (4, "128k")])
def test_partials_merge_to_one_call(world, shape):
    if shape == "8k":
        pr = _batch(1, [320], [16], [4], [257])
    elif shape == "mix":
        pr = _batch(2, [320, 320, 320], [128, 32, 8], [32, 8, 2], [65, 257, 1025])
    else:
        pr = _batch(3, [576], [512], [64], [129])
    d = _dev(pr)
    parts_o, parts_lse = [], []
    for rank in range(world):
        sel_r, cu_r = mg.local_selection(pr["sel"], pr["cu_k"], pr["cu_n"], rank, world)
        o, lse = api.decode_partial(d["q"], d["k"], d["v"], d["pk"], d["pv"], d["table"],
                                    P.cuda(torch.tensor(sel_r, dtype=torch.int32)), pr["cu_lq"],
                                    cu_r, mg.self_keys_on(rank))
        parts_o.append(o)
        parts_lse.append(lse)
    out, lse = api.lse_merge(torch.stack(parts_o), torch.stack(parts_lse))
    sel_d = P.cuda(torch.tensor(pr["sel"], dtype=torch.int32))
    ref_out, ref_lse = api.decode_attention(d["q"], d["k"], d["v"], d["pk"], d["pv"], d["table"],
                                            sel_d, cu_lq=pr["cu_lq"], cu_k=pr["cu_k"])
    torch.cuda.synchronize()
    P.assert_close_out(out.cpu().double().numpy(), ref_out.cpu().double().numpy(),
                       f"{shape}: merged partials vs one call")
    assert (lse - ref_lse).abs().max().item() <= P.LSE_MAX_ABS
    pk, pv, tab = f64(pr["pk"]), f64(pr["pv"]), pr["table"].numpy()
    out_h, lse_h = out.cpu().double().numpy(), lse.cpu().double().numpy()
    for b in range(len(pr["cu_lq"]) - 1):
        lo, hi = pr["cu_lq"][b], pr["cu_lq"][b + 1]
        rows = list(range(lo, hi)) if hi - lo <= 320 else list(range(lo, hi, 3))
        o_ref, lse_ref = orc.decode_attention(
            f64(pr["q"][rows]), f64(pr["k"][lo:hi]), f64(pr["v"][lo:hi]), pk, pv, tab,
            pr["sel"][pr["cu_k"][b]:pr["cu_k"][b + 1]], pr["scale"])
        P.assert_close_out(out_h[rows], o_ref, f"{shape} seq {b}: merged partials vs oracle")
        assert np.abs(lse_h[rows] - lse_ref).max() <= P.LSE_MAX_ABS


@pytest.mark.parametrize("self_keys", [0, 1])
def test_partial_alone_matches_oracle_state(self_keys):
    """A partial over a subset (self block in or out) is that subset's own
    softmax output and log-sum-exp."""
    pr = _batch(4, [200], [12], [5], [97])
    d = _dev(pr)
    sub = pr["sel"][1:4]
    o, lse = api.decode_partial(d["q"], d["k"], d["v"], d["pk"], d["pv"], d["table"],
                                P.cuda(torch.tensor(sub, dtype=torch.int32)), pr["cu_lq"],
                                [0, len(sub)], self_keys, n_splits=2)
    torch.cuda.synchronize()
    pk, pv, tab = f64(pr["pk"]), f64(pr["pv"]), pr["table"].numpy()
    kk = [orc.gather_selected(pk, tab, sub)]
    vv = [orc.gather_selected(pv, tab, sub)]
    if self_keys:
        kk.append(f64(pr["k"]))
        vv.append(f64(pr["v"]))
    m, l, acc = orc.split_partials(f64(pr["q"]), np.concatenate(kk), np.concatenate(vv), 7,
                                   pr["scale"])
    P.assert_close_out(o.cpu().double().numpy(), acc / l[..., None], "partial output")
    assert np.abs(lse.cpu().double().numpy() - (m + np.log(l))).max() <= P.LSE_MAX_ABS


def test_empty_partial_and_its_merge():
    """No selected chunk and no live-block keys: o = 0, lse = -inf; merged
    with a real partial, it has weight 0 (the result is that partial)."""
    pr = _batch(5, [100, 60], [6, 4], [2, 1], [33, 17])
    d = _dev(pr)
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    o0, l0 = api.decode_partial(d["q"], d["k"], d["v"], d["pk"], d["pv"], d["table"], empty,
                                pr["cu_lq"], [0, 0, 0], 0)
    sel_d = P.cuda(torch.tensor(pr["sel"], dtype=torch.int32))
    o1, l1 = api.decode_partial(d["q"], d["k"], d["v"], d["pk"], d["pv"], d["table"], sel_d,
                                pr["cu_lq"], pr["cu_k"], 1)
    out, lse = api.lse_merge(torch.stack([o0, o1]), torch.stack([l0, l1]))
    torch.cuda.synchronize()
    assert torch.all(o0 == 0) and torch.all(torch.isneginf(l0))
    # (lse * log2 e) * ln 2: the same value up to fp32 rounding
    assert torch.allclose(lse, l1, rtol=1e-6, atol=1e-6)
    P.assert_close_out(out.cpu().double().numpy(), o1.cpu().double().numpy(), "merge with empty")
    out2, lse2 = api.lse_merge(torch.stack([o0, o0]), torch.stack([l0, l0]))
    torch.cuda.synchronize()
    assert torch.all(out2 == 0) and torch.all(torch.isneginf(lse2))
