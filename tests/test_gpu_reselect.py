"""Dynamic chunk reselection on the GPU against the oracle: the attention
mass of every chunk (selected or not) at a decode step's normaliser
(pfd_chunk_mass, fed with that step's lse from pfd_decode_attention), and
the new selection top-K of fl32(s + fl32(lambda * mass))
(pfd_reselect_chunks).

Tolerance of a mass: logits are fp32 sums of exact bf16 products (about
1e-6 relative), exp2 is the approximate unit (2^-22 relative) and the lse
comes from the decode call (about 1e-6 absolute against the oracle's); a
mass is a sum of up to ~10^6 such terms in fp32, so rel 1e-3 + abs 1e-6 is
far from both.  The selection is compared exactly except where the
oracle's s' values of two chunks lie within the mass tolerance times lambda
of each other (a tie the tolerance cannot decide); lambda = 0 must give the
static selection exactly."""
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
MASS_RTOL, MASS_ATOL = 1e-3, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    _abi.load()


def _step(cfgs):
    """Prefill every sequence into one shared pool, select, and run decode
    step 0 (batched); returns the device state and host copies."""
    dev = torch.device("cuda")
    c0 = cfgs[0]
    reqs = [wl.make_request(c, i) for i, c in enumerate(cfgs)]
    pool_base, cu_n, cu_k = [0], [0], [0]
    for c in cfgs:
        pool_base.append(pool_base[-1] + c.pool_rows)
        cu_n.append(cu_n[-1] + c.n_chunks)
        cu_k.append(cu_k[-1] + c.n_select)
    pool_k = torch.zeros(pool_base[-1], c0.n_kv_heads, c0.head_dim, dtype=torch.bfloat16,
                         device=dev)
    pool_v = torch.zeros_like(pool_k)
    table = torch.zeros(cu_n[-1], 2, dtype=torch.int32, device=dev)
    for i, (c, req) in enumerate(zip(cfgs, reqs)):
        slot = (req["slot_row"] + pool_base[i]).to(torch.int32)
        res = api.chunk_prefill(P.cuda(req["q"]), P.cuda(req["k"]), P.cuda(req["v"]),
                                P.cuda(req["q_win"]), c.n_chunks, c.chunk_size, c.n_keep,
                                P.cuda(slot), pool_base[-1], pool_k=pool_k, pool_v=pool_v)
        table[cu_n[i]:cu_n[i + 1]] = res["table"]
    s_i = torch.cat([r["s_i"] for r in reqs]).to(dev)
    s_p = torch.cat([r["s_p"] for r in reqs]).to(dev)
    cu_n_d = torch.tensor(cu_n, dtype=torch.int32, device=dev)
    cu_k_d = torch.tensor(cu_k, dtype=torch.int32, device=dev)
    max_n = max(c.n_chunks for c in cfgs)
    sel, s_static = api.select_chunks_batched(s_i, s_p, cu_n_d, cu_k_d, max_n)
    lives = [wl.live_block(r, wl.make_step(c, i, 0)) for i, (c, r) in enumerate(zip(cfgs, reqs))]
    cu_lq = [0]
    for q, _, _ in lives:
        cu_lq.append(cu_lq[-1] + q.shape[0])
    q = P.cuda(torch.cat([x[0] for x in lives]))
    out, lse = api.decode_attention(q, P.cuda(torch.cat([x[1] for x in lives])),
                                    P.cuda(torch.cat([x[2] for x in lives])), pool_k, pool_v,
                                    table, sel, cu_lq=cu_lq, cu_k=cu_k,
                                    max_chunk_len=max(c.n_keep + 1 for c in cfgs))
    torch.cuda.synchronize()
    return dict(cfgs=cfgs, reqs=reqs, lives=lives, q=q, lse=lse, pool_k=pool_k, pool_v=pool_v,
                table=table, cu_n=cu_n, cu_k=cu_k, cu_lq=cu_lq, cu_n_d=cu_n_d, cu_k_d=cu_k_d,
                max_n=max_n, sel=sel, s_static=s_static)


def _oracle_mass(st):
    """The oracle's masses of every chunk, with the oracle's own decode lse."""
    pk, pv, tab = f64(st["pool_k"].cpu()), f64(st["pool_v"].cpu()), st["table"].cpu().numpy()
    sel = st["sel"].cpu().numpy()
    out = np.zeros(tab.shape[0])
    for i, (c, (ql, kl, vl)) in enumerate(zip(st["cfgs"], st["lives"])):
        k0, k1 = st["cu_k"][i], st["cu_k"][i + 1]
        _, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, tab, sel[k0:k1],
                                          c.sm_scale)
        chunks = list(range(st["cu_n"][i], st["cu_n"][i + 1]))
        out[chunks] = orc.chunk_mass(f64(ql), pk, tab, chunks, lse_ref, c.sm_scale)
    return out


CASES = {
    "8k": [wl.CTX_8K],
    "small_d64": [wl.scaled(wl.TINY, n_chunks=6, chunk_size=100, n_keep=30, n_select=3,
                            n_win=8, n_resp=20)],
    "128k": [wl.CTX_128K],
    # many small chunks: several chunks per mass item (four, the last group
    # partial) on the D = 64 kernel, with ragged slots of 7 rows
    "d64_many": [wl.scaled(wl.TINY, n_chunks=1102, chunk_size=24, n_keep=6, n_select=4,
                           n_win=8, n_resp=20)],
    "mix3": [wl.scaled(c, n_chunks=32768 // c.chunk_size // 4, n_select=max(1, c.n_select // 2))
             for c in wl.mix_configs()[:3]],
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_chunk_mass_and_reselection(name):
    st = _step(CASES[name])
    batch = len(st["cfgs"])
    mass, err = api.chunk_mass(st["q"], st["pool_k"], st["table"], st["lse"], st["cu_lq"],
                               st["cu_n"])
    mass2, _ = api.chunk_mass(st["q"], st["pool_k"], st["table"], st["lse"], st["cu_lq"],
                              st["cu_n"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(mass, mass2), "repeated calls must give the same bits"
    want = _oracle_mass(st)
    got = mass.cpu().double().numpy()
    bad = np.abs(got - want) > MASS_RTOL * np.abs(want) + MASS_ATOL
    assert not bad.any(), f"{name}: mass of chunks {np.nonzero(bad)[0][:5]}"
    # selected chunks and the live block share the step's attention: the
    # selected chunks' masses sum below one, per sequence
    sel = st["sel"].cpu().numpy()
    for i in range(batch):
        k0, k1 = st["cu_k"][i], st["cu_k"][i + 1]
        assert got[sel[k0:k1]].sum() < 1.0 + 1e-4

    s_static = st["s_static"].cpu().numpy()
    for lam in (0.0, 1.0, 50.0):
        new_sel, s2 = api.reselect_chunks(st["s_static"], mass, lam, st["cu_n_d"], st["cu_k_d"],
                                          st["max_n"])
        torch.cuda.synchronize()
        new_sel = new_sel.cpu().tolist()
        if lam == 0.0:
            assert new_sel == st["sel"].cpu().tolist()
        band = 2 * lam * (MASS_RTOL * np.abs(want) + MASS_ATOL).max()
        for i in range(batch):
            n0, n1, k0, k1 = st["cu_n"][i], st["cu_n"][i + 1], st["cu_k"][i], st["cu_k"][i + 1]
            ref, s2_ref = orc.reselect_chunks(s_static[n0:n1], want[n0:n1], lam, k1 - k0)
            ref = [n0 + int(x) for x in ref]
            g = new_sel[k0:k1]
            if g != ref:
                for a, b in zip(g, ref):
                    assert abs(float(s2_ref[a - n0]) - float(s2_ref[b - n0])) <= band, \
                        f"{name} lambda {lam}: {g} vs {ref}"
