"""The multi-GPU split of a decode step, host side, as two gloo ranks on CPU.

Each rank prefills a contiguous chunk range (no exchange), computes the
partial state of the selected chunks that live in its range -- the live
block's keys on the owner only -- and the partials are all-gathered in the
layout pfd_lse_merge takes.  The partials here come from the oracle (the
ranks have no GPU); the test checks the partition and the gather: the
owner's log-sum-exp merge of the gathered partials equals the oracle's
one-softmax decode over all selected chunks and the live block.
"""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

from sparse_chunked_kv_gb300 import multigpu as mg

WORLD = 2


def test_chunk_ranges_partition_every_sequence():
    for n in (1, 2, 5, 16, 511):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                lo, hi = mg.chunk_range(n, r, world)
                seen.extend(range(lo, hi))
                assert all(mg.owner_of(c, n, world) == r for c in range(lo, hi))
            assert seen == list(range(n))


def test_local_selection_splits_sel_exactly_once():
    cu_n, cu_k = [0, 16, 24, 536], [0, 4, 6, 70]
    sel = [3, 15, 0, 8, 16 + 7, 16 + 1] + [24 + x for x in range(0, 512, 8)]
    for world in (1, 2, 4):
        parts = [mg.local_selection(sel, cu_k, cu_n, r, world) for r in range(world)]
        for b in range(3):
            got = sorted(c for s, cu in parts for c in s[cu[b]:cu[b + 1]])
            assert got == sorted(sel[cu_k[b]:cu_k[b + 1]])
            for r, (s, cu) in enumerate(parts):
                chunk_ids = [c - cu_n[b] for c in s[cu[b]:cu[b + 1]]]
                n_b = cu_n[b + 1] - cu_n[b]
                assert all(mg.owner_of(c, n_b, world) == r for c in chunk_ids)
                # selection order is kept within a rank
                order = [sel.index(c) for c in s[cu[b]:cu[b + 1]]]
                assert order == sorted(order)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    """Two sequences sharing one table; pool slots of random length."""
    rng = np.random.default_rng(5)
    hq, hkv, d = 4, 2, 8
    cu_n, lens = [0, 6, 10], [5, 9, 3, 7, 4, 6, 8, 2, 5, 3]
    table, row = [], 0
    for n in lens:
        table.append((row, n))
        row += n
    pool_k, pool_v = rng.standard_normal((row, hkv, d)), rng.standard_normal((row, hkv, d))
    cu_k = [0, 3, 5]
    sel = [4, 0, 5, 8, 6]                      # table indices, per sequence in rank order
    cu_lq = [0, 5, 9]
    q = rng.standard_normal((9, hq, d))
    ks, vs = rng.standard_normal((9, hkv, d)), rng.standard_normal((9, hkv, d))
    return dict(hq=hq, hkv=hkv, d=d, cu_n=cu_n, table=np.array(table), pool_k=pool_k,
                pool_v=pool_v, cu_k=cu_k, sel=sel, cu_lq=cu_lq, q=q, ks=ks, vs=vs, scale=0.4)


def _partial(orc, pr, b, sel_b, self_keys):
    """(o, lse) of sequence b's live rows over its local keys (oracle)."""
    lo, hi = pr["cu_lq"][b], pr["cu_lq"][b + 1]
    q = pr["q"][lo:hi]
    parts = [(pr["pool_k"][r:r + n], pr["pool_v"][r:r + n]) for r, n in pr["table"][sel_b]]
    if self_keys:
        parts.append((pr["ks"][lo:hi], pr["vs"][lo:hi]))
    if not parts:
        return np.zeros(q.shape), np.full(q.shape[:2], -np.inf)
    kk = np.concatenate([k for k, _ in parts])
    vv = np.concatenate([v for _, v in parts])
    m, l, acc = orc.split_partials(q, kk, vv, pr["hq"] // pr["hkv"], pr["scale"])
    return acc / l[..., None], m + np.log(l)


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    from oracle import pfd_oracle as orc
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        pr = _problem()
        sel_l, cu_l = mg.local_selection(pr["sel"], pr["cu_k"], pr["cu_n"], rank, WORLD)
        o_parts, l_parts = [], []
        for b in range(len(pr["cu_lq"]) - 1):
            o, lse = _partial(orc, pr, b, sel_l[cu_l[b]:cu_l[b + 1]], mg.self_keys_on(rank))
            o_parts.append(o)
            l_parts.append(lse)
        part_o = torch.from_numpy(np.concatenate(o_parts))
        part_lse = torch.from_numpy(np.concatenate(l_parts))
        o_all, l_all = mg.gather_partials(part_o, part_lse, WORLD)
        result = None
        if rank == mg.OWNER:
            # log-sum-exp merge of the gathered (o, lse) states: the oracle's
            # merge of states (m, l, acc) = (lse, 1, o)
            states = [(l_all[r].numpy(), np.where(np.isinf(l_all[r].numpy()), 0.0, 1.0),
                       o_all[r].numpy()) for r in range(WORLD)]
            result = orc.lse_merge(states)
        out.put((rank, len(sel_l), result, None))
    except Exception as e:   # report instead of leaving the parent waiting
        out.put((rank, -1, None, repr(e)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_merge_equals_one_softmax():
    from oracle import pfd_oracle as orc
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(WORLD):
        rank, n_local, merged, err = out.get(timeout=240)
        assert err is None, f"rank {rank}: {err}"
        res[rank] = (n_local, merged)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    pr = _problem()
    assert sum(n for n, _ in res.values()) == len(pr["sel"])
    assert all(n > 0 for n, _ in res.values()), "both ranks hold selected chunks"
    got_o, got_lse = res[mg.OWNER][1]
    for b in range(2):
        lo, hi = pr["cu_lq"][b], pr["cu_lq"][b + 1]
        want_o, want_lse = orc.decode_attention(
            pr["q"][lo:hi], pr["ks"][lo:hi], pr["vs"][lo:hi], pr["pool_k"], pr["pool_v"],
            pr["table"], pr["sel"][pr["cu_k"][b]:pr["cu_k"][b + 1]], pr["scale"])
        assert np.max(np.abs(got_o[lo:hi] - want_o)) < 1e-12
        assert np.max(np.abs(got_lse[lo:hi] - want_lse)) < 1e-12
