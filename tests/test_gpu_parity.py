"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle on
seeded inputs small enough for the oracle to check every output."""
import numpy as np
import pytest
import torch

from oracle import pfd_oracle as orc
from sparse_chunked_kv_gb300 import _abi, api
from sparse_chunked_kv_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

f64 = wl.to_f64

# Small cases spanning several tiles and ragged tails: (name, config).
PREFILL_CASES = [
    ("tiny", wl.TINY),
    ("gqa7_c512", wl.scaled(wl.CTX_8K, n_chunks=3, n_select=2)),
    ("gqa7_c100_ragged", wl.scaled(wl.CTX_8K, n_chunks=2, chunk_size=100, n_keep=37, n_select=1,
                                   n_win=7, n_resp=9)),
    ("d64_c1000", wl.scaled(wl.TINY, n_chunks=2, chunk_size=1000, n_keep=333, n_win=5)),
    ("keep_all", wl.scaled(wl.TINY, n_chunks=3, chunk_size=48, n_keep=48, n_select=3)),
    ("keep_none", wl.scaled(wl.TINY, n_chunks=3, chunk_size=48, n_keep=0, n_select=2)),
    ("no_window", wl.scaled(wl.TINY, n_chunks=2, chunk_size=64, n_keep=10, n_win=0, n_resp=17)),
    ("one_token_chunks", wl.scaled(wl.TINY, n_chunks=5, chunk_size=1, n_keep=1, n_win=3)),
    ("d64_c1500", wl.scaled(wl.TINY, n_chunks=2, chunk_size=1500, n_keep=400, n_win=5)),
    ("c1024_keep_all_but_one", wl.scaled(wl.TINY, n_chunks=2, chunk_size=1024, n_keep=1023, n_win=4)),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    _abi.load()


@pytest.mark.parametrize("name,cfg", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_prefill_parity(name, cfg):
    req = wl.make_request(cfg, 0)
    res = P.run_prefill(cfg, req)
    assert int(res["dev_err"][0]) == 0
    o_ref = orc.chunk_attention(f64(req["q"]), f64(req["k"]), f64(req["v"]), cfg.n_chunks,
                                cfg.chunk_size, cfg.sm_scale)
    P.assert_close_out(res["out"].double().numpy(), o_ref, "prefill out")
    s_ref = orc.window_scores(f64(req["q_win"]), f64(req["k"]), cfg.n_chunks, cfg.chunk_size,
                              cfg.sm_scale)
    s_gpu = res["scores"].double().numpy()
    tol = P.score_tol(s_ref, cfg.n_win, cfg.n_q_heads)
    assert (np.abs(s_gpu - s_ref) <= tol).all(), f"scores: max diff {np.abs(s_gpu - s_ref).max()}"
    if cfg.n_keep > 0:
        P.check_kept(res["kept_idx"].numpy(), s_ref, cfg.n_keep)
    P.check_pool(cfg, req, res)


# The largest sizes the prefill accepts: C = 8192 content tokens per chunk,
# and W * G = 512 window rows per KV group (W = 128 at G = 4, W = 256 at G = 2).
MAX_CASES = [
    ("c8192_wg512", wl.scaled(wl.TINY, n_chunks=2, chunk_size=8192, n_keep=2049, n_win=128)),
    ("w256_g2", wl.scaled(wl.TINY, n_q_heads=4, n_kv_heads=2, n_chunks=2, chunk_size=300,
                          n_keep=101, n_win=256)),
]


@pytest.mark.parametrize("name,cfg", MAX_CASES, ids=[c[0] for c in MAX_CASES])
def test_prefill_maximum_sizes(name, cfg):
    """Every score, kept set and pool slot; the output at each chunk's BOS,
    first and last rows and 64 seeded rows (the oracle's full output at
    C = 8192 would take it minutes)."""
    req = wl.make_request(cfg, 0)
    res = P.run_prefill(cfg, req)
    assert int(res["dev_err"][0]) == 0
    span = cfg.chunk_size + 1
    gen = np.random.default_rng(7)
    rows = sorted({int(r) for j in range(cfg.n_chunks)
                   for r in [j * span, j * span + 1, (j + 1) * span - 1,
                             *(j * span + gen.integers(0, span, 64))]})
    o_ref = orc.chunk_attention_rows(f64(req["q"]), f64(req["k"]), f64(req["v"]), cfg.chunk_size,
                                     rows, cfg.sm_scale)
    P.assert_close_out(res["out"][rows].double().numpy(), o_ref, "prefill out, sampled rows")
    s_ref = orc.window_scores(f64(req["q_win"]), f64(req["k"]), cfg.n_chunks, cfg.chunk_size,
                              cfg.sm_scale)
    s_gpu = res["scores"].double().numpy()
    tol = P.score_tol(s_ref, cfg.n_win, cfg.n_q_heads)
    assert (np.abs(s_gpu - s_ref) <= tol).all(), f"scores: max diff {np.abs(s_gpu - s_ref).max()}"
    P.check_kept(res["kept_idx"].numpy(), s_ref, cfg.n_keep)
    P.check_pool(cfg, req, res)


def test_prefill_by_chunk_ranges_matches_one_call():
    """Chunks are independent up to selection: calling the prefill once per
    range of chunks (as a caller overlapping input copies would) gives the
    same bits as one call, into one shared pool."""
    cfg = wl.scaled(wl.CTX_8K, n_chunks=5, chunk_size=100, n_keep=37, n_win=7)
    req = wl.make_request(cfg, 2)
    rows = cfg.chunk_size + 1
    slot = req["slot_row"].to(torch.int32)
    q, k, v, qw = (P.cuda(req[x]) for x in ("q", "k", "v", "q_win"))
    whole = api.chunk_prefill(q, k, v, qw, cfg.n_chunks, cfg.chunk_size, cfg.n_keep, P.cuda(slot),
                              cfg.pool_rows)
    pk = torch.zeros_like(whole["pool_k"])
    pv = torch.zeros_like(whole["pool_v"])
    parts = []
    for j0, j1 in ((0, 2), (2, 3), (3, 5)):
        r0, r1 = j0 * rows, j1 * rows
        parts.append(api.chunk_prefill(q[r0:r1], k[r0:r1], v[r0:r1], qw, j1 - j0, cfg.chunk_size,
                                       cfg.n_keep, P.cuda(slot[j0:j1]), cfg.pool_rows,
                                       pool_k=pk, pool_v=pv))
    torch.cuda.synchronize()
    bits = {torch.bfloat16: torch.int16, torch.float32: torch.int32, torch.int32: torch.int32}
    for key in ("out", "scores", "kept_idx", "table"):
        got = torch.cat([part[key] for part in parts])
        assert torch.equal(got.view(bits[got.dtype]), whole[key].view(bits[got.dtype])), key
    assert torch.equal(pk.view(torch.int16), whole["pool_k"].view(torch.int16))
    assert torch.equal(pv.view(torch.int16), whole["pool_v"].view(torch.int16))


def test_prefill_pool_padding_untouched():
    cfg = wl.scaled(wl.TINY, n_chunks=4, chunk_size=80, n_keep=20)
    req = wl.make_request(cfg, 3)
    res = P.run_prefill(cfg, req, pool_pad=5, pool_fill=float("nan"))
    stride = cfg.n_keep + 1 + 5
    for j in range(cfg.n_chunks):
        base = int(res["slot_row"][j])
        pad = res["pool_k"][base + cfg.n_keep + 1:base + stride]
        assert torch.isnan(pad.float()).all()
    P.check_pool(cfg, req, res)


def _select_cases():
    g = torch.Generator().manual_seed(5)
    cases = []
    for n, k in ((8, 2), (16, 4), (32, 8), (512, 64), (128, 32), (1, 1), (300, 300)):
        cases.append((torch.randn(n, generator=g), torch.randn(n, generator=g), k))
    ties = torch.round(torch.randn(200, generator=g) * 2) / 2
    cases.append((ties, torch.zeros(200), 50))
    cases.append((torch.tensor([0.0, -0.0, 1.0, -0.0, 0.0]), torch.tensor([-0.0, 0.0, -1.0, 0.0, -0.0]), 3))
    cases.append((torch.tensor([1.0, 0.5, 1.0, 0.75]), torch.tensor([0.0, 0.0, 2.0 ** -25, 0.0]), 4))
    cases.append((torch.full((64,), 0.5), torch.full((64,), 0.25), 10))
    return cases


@pytest.mark.parametrize("case", range(len(_select_cases())))
def test_select_bit_exact(case):
    s_i, s_p, k = _select_cases()[case]
    sel, s = api.select_chunks(P.cuda(s_i.float()), P.cuda(s_p.float()), k)
    sel_ref, s_ref = orc.select_chunks(s_i.float().numpy(), s_p.float().numpy(), k)
    assert sel.cpu().tolist() == sel_ref.tolist()
    assert np.array_equal(s.cpu().numpy().view(np.uint32) & 0x7FFFFFFF,
                          s_ref.view(np.uint32) & 0x7FFFFFFF)


def test_select_batched_bit_exact():
    g = torch.Generator().manual_seed(9)
    ns, ks = [128, 32, 8, 128, 5], [32, 8, 2, 1, 5]
    s_i, s_p = torch.randn(sum(ns), generator=g), torch.randn(sum(ns), generator=g)
    cu_n = torch.tensor([0] + list(np.cumsum(ns)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(np.cumsum(ks)), dtype=torch.int32)
    sel, _ = api.select_chunks_batched(P.cuda(s_i), P.cuda(s_p), P.cuda(cu_n), P.cuda(cu_k), max(ns))
    want = []
    for b in range(len(ns)):
        lo = int(cu_n[b])
        r, _ = orc.select_chunks(s_i[lo:lo + ns[b]].numpy(), s_p[lo:lo + ns[b]].numpy(), ks[b])
        want += [lo + int(x) for x in r]
    assert sel.cpu().tolist() == want


def _decode_inputs(cfg, seq=0, step=0, pad=0, fill=0.0):
    """Oracle-built pool for cfg (the GPU decode is checked on the oracle's pool)."""
    req = wl.make_request(cfg, seq)
    scores = orc.window_scores(f64(req["q_win"]), f64(req["k"]), cfg.n_chunks, cfg.chunk_size,
                               cfg.sm_scale)
    kept = orc.top_b(scores, cfg.n_keep)
    stride = cfg.n_keep + 1 + pad
    slot = (req["slot_row"] // cfg.slot_stride) * stride
    pool_rows = cfg.n_chunks * stride
    pk, pv, table = P.oracle_pool(cfg, req, kept, slot, pool_rows, fill)
    sel, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    ql, kl, vl = wl.live_block(req, wl.make_step(cfg, seq, step))
    return req, pk, pv, table, sel, ql, kl, vl


# 12 splits cut the tiny case's ~190 keys into splits of one or two 16-row
# key groups, far below one 128-key tile each.
@pytest.mark.parametrize("n_splits", [0, 1, 2, 3, 4, 5, 7, 8, 12])
@pytest.mark.parametrize("cfg_name", ["tiny", "gqa7"])
def test_decode_parity(cfg_name, n_splits):
    cfg = wl.TINY if cfg_name == "tiny" else wl.scaled(wl.CTX_8K, n_chunks=6, n_select=3, n_resp=100)
    _, pk, pv, table, sel, ql, kl, vl = _decode_inputs(cfg)
    o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel, cfg.sm_scale)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), P.cuda(P.bf16_of(pk)),
                                    P.cuda(P.bf16_of(pv)), P.cuda(torch.from_numpy(table)),
                                    P.cuda(torch.from_numpy(sel)), n_splits=n_splits, dev_err=dev_err)
    torch.cuda.synchronize()
    assert int(dev_err.item()) == 0
    P.assert_close_out(out.cpu().double().numpy(), o_ref, "decode out")
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS


@pytest.mark.parametrize("n_splits", [2, 3, 4, 5])
def test_decode_odd_pair_count(n_splits):
    """3 query heads on 1 KV head over 37 live rows: 111 (row, head) pairs, so the
    merge's last warp holds a single pair when it takes two per warp."""
    cfg = wl.scaled(wl.TINY, n_q_heads=3, n_kv_heads=1, n_win=16, n_resp=21)
    _, pk, pv, table, sel, ql, kl, vl = _decode_inputs(cfg)
    assert ql.shape[0] * ql.shape[1] % 2 == 1
    o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel, cfg.sm_scale)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), P.cuda(P.bf16_of(pk)),
                                    P.cuda(P.bf16_of(pv)), P.cuda(torch.from_numpy(table)),
                                    P.cuda(torch.from_numpy(sel)), n_splits=n_splits, dev_err=dev_err)
    torch.cuda.synchronize()
    assert int(dev_err.item()) == 0
    P.assert_close_out(out.cpu().double().numpy(), o_ref, "decode out (odd pairs)")
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS


def test_decode_nan_padding_is_masked():
    cfg = wl.scaled(wl.TINY, n_keep=57, n_select=3)     # 58-row slots: ragged 16-row groups
    _, pk, pv, table, sel, ql, kl, vl = _decode_inputs(cfg, pad=7, fill=float("nan"))
    o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel, cfg.sm_scale)
    for n_splits in (1, 4):
        out, lse = api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), P.cuda(P.bf16_of(pk)),
                                        P.cuda(P.bf16_of(pv)), P.cuda(torch.from_numpy(table)),
                                        P.cuda(torch.from_numpy(sel)), n_splits=n_splits)
        P.assert_close_out(out.cpu().double().numpy(), o_ref, "decode out (NaN padding)")
        assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS


def test_running_max_jumps_between_tiles():
    """Logits that grow by far more than 2^8 from tile to tile force the
    rescale of O (and the redo of a tile's probabilities) on every tile."""
    cfg = wl.scaled(wl.TINY, n_chunks=2, chunk_size=700, n_keep=200, n_select=2, n_win=16,
                    n_resp=48)
    req = wl.make_request(cfg, 0)
    rows = cfg.chunk_size + 1
    ramp = torch.linspace(0.2, 6.0, rows).repeat(cfg.n_chunks)[:, None, None]
    req["k"] = (req["k"].float() * ramp).to(torch.bfloat16)
    res = P.run_prefill(cfg, req)
    assert int(res["dev_err"][0]) == 0
    o_ref = orc.chunk_attention(f64(req["q"]), f64(req["k"]), f64(req["v"]), cfg.n_chunks,
                                cfg.chunk_size, cfg.sm_scale)
    P.assert_close_out(res["out"].double().numpy(), o_ref, "prefill out (ramped keys)")
    s_ref = orc.window_scores(f64(req["q_win"]), f64(req["k"]), cfg.n_chunks, cfg.chunk_size,
                              cfg.sm_scale)
    P.check_kept(res["kept_idx"].numpy(), s_ref, cfg.n_keep)
    # decode: live keys much larger than the pool's so the last split tile jumps
    pk, pv, table = P.oracle_pool(cfg, req, orc.top_b(s_ref, cfg.n_keep), res["slot_row"],
                                  res["pool_rows"])
    sel = np.array([1, 0], dtype=np.int32)
    ql, kl, vl = wl.live_block(req, wl.make_step(cfg, 0, 0))
    kl = (kl.float() * 8.0).to(torch.bfloat16)
    o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel, cfg.sm_scale)
    for n_splits in (1, 2):
        out, lse = api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), P.cuda(P.bf16_of(pk)),
                                        P.cuda(P.bf16_of(pv)), P.cuda(torch.from_numpy(table)),
                                        P.cuda(torch.from_numpy(sel)), n_splits=n_splits)
        P.assert_close_out(out.cpu().double().numpy(), o_ref, "decode out (jumping max)")
        assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS


# Chunks of one and of two keys per selecting thread.
@pytest.mark.parametrize("chunk_size,n_keep", [(300, 77), (1200, 301)])
def test_prefill_exact_ties_keep_lowest_indices(chunk_size, n_keep):
    """Exact score ties at the B-th place are broken towards the lower token
    index.  Chunk 0: all C content keys identical, so every content score
    ties and the kept tokens are 0..B-1.  Chunk 1: the key ranked B-th is
    copied onto the key ranked B+1-th, two exactly equal scores; when they
    straddle the B-th place, the lower index is kept."""
    cfg = wl.scaled(wl.TINY, n_chunks=2, chunk_size=chunk_size, n_keep=n_keep, n_win=8)
    req = wl.make_request(cfg, 0)
    rows = cfg.chunk_size + 1
    k = req["k"].clone()
    k[1:rows] = k[1]
    s_ref = orc.window_scores(f64(req["q_win"]), f64(k), cfg.n_chunks, cfg.chunk_size,
                              cfg.sm_scale)
    order = np.argsort(-s_ref[1, 1:], kind="stable")
    b_th, nxt = int(order[cfg.n_keep - 1]), int(order[cfg.n_keep])
    k[rows + 1 + nxt] = k[rows + 1 + b_th]
    res = P.run_prefill(cfg, {**req, "k": k})
    assert int(res["dev_err"][0]) == 0
    assert res["kept_idx"][0].tolist() == list(range(cfg.n_keep))
    s2 = orc.window_scores(f64(req["q_win"]), f64(k), cfg.n_chunks, cfg.chunk_size,
                           cfg.sm_scale)
    assert s2[1, 1 + b_th] == s2[1, 1 + nxt]
    P.check_kept(res["kept_idx"].numpy(), s2, cfg.n_keep)
    lo, hi = min(b_th, nxt), max(b_th, nxt)
    ref = set(orc.top_b(s2, cfg.n_keep)[1].tolist())
    kept = set(res["kept_idx"][1].tolist())
    if (lo in ref) != (hi in ref):                 # the tie straddles the B-th place
        assert lo in kept and hi not in kept


def _spike(k, rows, u, size):
    k = k.float().clone()
    for r in rows:
        k[r] = size * u
    return k.to(torch.bfloat16)


@pytest.mark.parametrize("size", [40.0, 100.0])
def test_logit_spike_in_later_tile(size):
    """A key far above every earlier logit of its row (about 2^72 above the
    running max for size 100, 2^29 for size 40) in the first and in the
    second 64-key half of later tiles, for some rows of a warp and not for
    others: the O rescale and the per-row reference stay exact."""
    cfg = wl.scaled(wl.TINY, n_chunks=2, chunk_size=700, n_keep=200, n_select=2, n_win=16,
                    n_resp=48)
    req = wl.make_request(cfg, 0)
    gen = torch.Generator().manual_seed(11)
    d = cfg.head_dim
    u = torch.randn(d, generator=gen)
    u = u / u.norm()
    rows = cfg.chunk_size + 1
    # content row r is key r - 1 of the tensor-core pipeline: tile (r-1)//128,
    # column (r-1)%128 -> half 0 of tile 2 (row 1+256+10), half 1 of tile 4
    # (row 1+512+100), and half 1 of chunk 1's tile 1 (row 1+128+70)
    spikes = [1 + 256 + 10, 1 + 512 + 100, rows + 1 + 128 + 70]
    req["k"] = torch.stack([_spike(req["k"][:, h], spikes, u, size)
                            for h in range(cfg.n_kv_heads)], dim=1)
    qf = req["q"].float() + 4.0 * u
    req["q"] = qf.to(torch.bfloat16)
    res = P.run_prefill(cfg, req)
    assert int(res["dev_err"][0]) == 0
    o_ref = orc.chunk_attention(f64(req["q"]), f64(req["k"]), f64(req["v"]), cfg.n_chunks,
                                cfg.chunk_size, cfg.sm_scale)
    P.assert_close_out(res["out"].double().numpy(), o_ref, f"prefill out (spike {size})")
    s_ref = orc.window_scores(f64(req["q_win"]), f64(req["k"]), cfg.n_chunks, cfg.chunk_size,
                              cfg.sm_scale)
    s_gpu = res["scores"].double().numpy()
    tol = P.score_tol(s_ref, cfg.n_win, cfg.n_q_heads)
    assert (np.abs(s_gpu - s_ref) <= tol).all(), f"scores: max diff {np.abs(s_gpu - s_ref).max()}"
    # decode: spikes in the live keys (the last tiles of the single split)
    pk, pv, table = P.oracle_pool(cfg, req, orc.top_b(s_ref, cfg.n_keep), res["slot_row"],
                                  res["pool_rows"])
    sel = np.array([1, 0], dtype=np.int32)
    ql, kl, vl = wl.live_block(req, wl.make_step(cfg, 0, 0))
    ql = (ql.float() + 4.0 * u).to(torch.bfloat16)
    kl = torch.stack([_spike(kl[:, h], [5, 40], u, size) for h in range(cfg.n_kv_heads)], dim=1)
    o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel, cfg.sm_scale)
    for n_splits in (1, 2):
        out, lse = api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), P.cuda(P.bf16_of(pk)),
                                        P.cuda(P.bf16_of(pv)), P.cuda(torch.from_numpy(table)),
                                        P.cuda(torch.from_numpy(sel)), n_splits=n_splits)
        P.assert_close_out(out.cpu().double().numpy(), o_ref, f"decode out (spike {size})")
        assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS


def test_decode_batched_shared_pool():
    """Three sequences with different chunk sizes and live lengths in one pool."""
    cfgs = [wl.scaled(wl.TINY, chunk_size=c, n_keep=b, n_select=k, n_resp=r, n_chunks=n)
            for c, b, k, r, n in ((64, 16, 3, 40, 6), (256, 64, 2, 17, 4), (32, 8, 4, 100, 8))]
    pool_k, pool_v, tables, sels, qs, ks, vs, refs = [], [], [], [], [], [], [], []
    row_base, table_base = 0, 0
    for i, cfg in enumerate(cfgs):
        _, pk, pv, table, sel, ql, kl, vl = _decode_inputs(cfg, seq=i)
        o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel,
                                              cfg.sm_scale)
        refs.append((o_ref, lse_ref))
        pool_k.append(pk)
        pool_v.append(pv)
        t = table.copy()
        t[:, 0] += row_base
        tables.append(t)
        sels.append(sel + table_base)
        row_base += pk.shape[0]
        table_base += table.shape[0]
        qs.append(ql)
        ks.append(kl)
        vs.append(vl)
    cu_lq = [0] + list(np.cumsum([q.shape[0] for q in qs]))
    cu_k = [0] + list(np.cumsum([len(s) for s in sels]))
    for n_splits in (0, 1, 3):
        out, lse = api.decode_attention(
            P.cuda(torch.cat(qs)), P.cuda(torch.cat(ks)), P.cuda(torch.cat(vs)),
            P.cuda(P.bf16_of(np.concatenate(pool_k))), P.cuda(P.bf16_of(np.concatenate(pool_v))),
            P.cuda(torch.from_numpy(np.concatenate(tables))),
            P.cuda(torch.from_numpy(np.concatenate(sels).astype(np.int32))), cu_lq=cu_lq, cu_k=cu_k,
            n_splits=n_splits)
        out, lse = out.cpu().double().numpy(), lse.cpu().double().numpy()
        for b, (o_ref, lse_ref) in enumerate(refs):
            P.assert_close_out(out[cu_lq[b]:cu_lq[b + 1]], o_ref, f"batched decode seq {b}")
            assert np.abs(lse[cu_lq[b]:cu_lq[b + 1]] - lse_ref).max() <= P.LSE_MAX_ABS


def test_decode_bad_entries_raise_device_error():
    cfg = wl.TINY
    _, pk, pv, table, sel, ql, kl, vl = _decode_inputs(cfg)
    bad_table = table.copy()
    bad_table[sel[0], 0] = pk.shape[0] + 100          # slot beyond the pool
    bad_sel = sel.copy()
    bad_sel[-1] = 1000                                 # index beyond the table
    for tab, s, bit in ((bad_table, sel, _abi.DEVERR_TABLE), (table, bad_sel, _abi.DEVERR_SEL)):
        dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, _ = api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), P.cuda(P.bf16_of(pk)),
                                      P.cuda(P.bf16_of(pv)), P.cuda(torch.from_numpy(tab)),
                                      P.cuda(torch.from_numpy(s)), dev_err=dev_err)
        torch.cuda.synchronize()
        assert int(dev_err.item()) & bit
        assert torch.isfinite(out.float()).all()


def test_prefill_bad_slot_raises_device_error():
    cfg = wl.scaled(wl.TINY, n_chunks=3, chunk_size=32, n_keep=8)
    req = wl.make_request(cfg, 0)
    slot = torch.tensor([0, 9, 1000], dtype=torch.int32)
    res = api.chunk_prefill(P.cuda(req["q"]), P.cuda(req["k"]), P.cuda(req["v"]),
                            P.cuda(req["q_win"]), cfg.n_chunks, cfg.chunk_size, cfg.n_keep,
                            P.cuda(slot), 27)
    torch.cuda.synchronize()
    assert int(res["dev_err"].item()) & _abi.DEVERR_SLOT
    assert res["table"][2].tolist() == [0, 0]
    assert res["table"][1].tolist() == [9, 9]


def test_static_pool_unchanged_by_decode_steps():
    cfg = wl.TINY
    req = wl.make_request(cfg, 0)
    res = P.run_prefill(cfg, req)
    pk0, pv0 = res["pool_k_dev"].clone(), res["pool_v_dev"].clone()
    sel, _ = api.select_chunks(P.cuda(req["s_i"]), P.cuda(req["s_p"]), cfg.n_select)
    for t in range(cfg.n_steps):
        ql, kl, vl = wl.live_block(req, wl.make_step(cfg, 0, t))
        api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), res["pool_k_dev"],
                             res["pool_v_dev"], res["table_dev"], sel, n_splits=2)
    torch.cuda.synchronize()
    assert torch.equal(pk0.view(torch.int16), res["pool_k_dev"].view(torch.int16))
    assert torch.equal(pv0.view(torch.int16), res["pool_v_dev"].view(torch.int16))


def test_end_to_end_tiny_every_step():
    """Prefill -> select -> T decode steps on the GPU pool, each step vs the
    oracle on the oracle's own pool (the kept sets must agree first)."""
    cfg = wl.TINY
    req = wl.make_request(cfg, 0)
    res = P.run_prefill(cfg, req)
    s_ref = orc.window_scores(f64(req["q_win"]), f64(req["k"]), cfg.n_chunks, cfg.chunk_size,
                              cfg.sm_scale)
    ref_kept, n_diff = P.check_kept(res["kept_idx"].numpy(), s_ref, cfg.n_keep)
    assert n_diff == 0, "tie-band swaps on the tiny workload"
    pk, pv, table = P.oracle_pool(cfg, req, ref_kept, res["slot_row"], res["pool_rows"])
    sel, _ = api.select_chunks(P.cuda(req["s_i"]), P.cuda(req["s_p"]), cfg.n_select)
    sel_ref, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    assert sel.cpu().tolist() == sel_ref.tolist()
    for t in range(cfg.n_steps):
        ql, kl, vl = wl.live_block(req, wl.make_step(cfg, 0, t))
        out, lse = api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), res["pool_k_dev"],
                                        res["pool_v_dev"], res["table_dev"], sel)
        o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel_ref,
                                              cfg.sm_scale)
        P.assert_close_out(out.cpu().double().numpy(), o_ref, f"decode step {t}")
        assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= P.LSE_MAX_ABS


def test_outputs_aligned_to_16_but_not_32_bytes():
    """Output buffers that start 16 bytes past a 32-byte boundary take the
    16-byte store path; results are the same as the oracle's."""
    cfg = wl.scaled(wl.CTX_8K, n_chunks=2, chunk_size=100, n_keep=20, n_select=2, n_resp=30)
    req = wl.make_request(cfg, 0)
    rows, hq, d = req["q"].shape
    base = torch.empty(rows * hq * d + 64, dtype=torch.bfloat16, device="cuda")
    off = (32 - base.data_ptr() % 32) // 2 + 8      # element offset: 16 bytes past a 32-byte boundary
    out = base[off:off + rows * hq * d].view(rows, hq, d)
    assert out.data_ptr() % 32 == 16
    slot = req["slot_row"].to(torch.int32)
    res = api.chunk_prefill(P.cuda(req["q"]), P.cuda(req["k"]), P.cuda(req["v"]), P.cuda(req["q_win"]),
                            cfg.n_chunks, cfg.chunk_size, cfg.n_keep, P.cuda(slot), cfg.pool_rows,
                            out=out)
    torch.cuda.synchronize()
    assert int(res["dev_err"][0]) == 0
    o_ref = orc.chunk_attention(f64(req["q"]), f64(req["k"]), f64(req["v"]), cfg.n_chunks,
                                cfg.chunk_size, cfg.sm_scale)
    P.assert_close_out(out.cpu().double().numpy(), o_ref, "prefill out (16-byte aligned)")
    _, pk, pv, table, sel, ql, kl, vl = _decode_inputs(cfg)
    o_ref, _ = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel, cfg.sm_scale)
    lq = ql.shape[0]
    base = torch.empty(lq * hq * d + 64, dtype=torch.bfloat16, device="cuda")
    off = (32 - base.data_ptr() % 32) // 2 + 8
    dout = base[off:off + lq * hq * d].view(lq, hq, d)
    for n_splits in (1, 3):
        api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), P.cuda(P.bf16_of(pk)),
                             P.cuda(P.bf16_of(pv)), P.cuda(torch.from_numpy(table)),
                             P.cuda(torch.from_numpy(sel)), n_splits=n_splits, out=dout)
        torch.cuda.synchronize()
        P.assert_close_out(dout.cpu().double().numpy(), o_ref, "decode out (16-byte aligned)")


def test_decode_bf16_partials_error_margin(capsys):
    """The split partials are stored as bf16 O / l with fp32 (m, l): the
    extra rounding against one split, measured on the 8K workload's step 0
    (every live row and head), for S = 1, 4 and 7.  Prints the figures and
    checks each against the oracle at the parity tolerance."""
    cfg = wl.CTX_8K
    req = wl.make_request(cfg, 0)
    scores = orc.window_scores(f64(req["q_win"]), f64(req["k"]), cfg.n_chunks, cfg.chunk_size,
                               cfg.sm_scale)
    kept = orc.top_b(scores, cfg.n_keep)
    pk, pv, table = P.oracle_pool(cfg, req, kept, req["slot_row"], cfg.pool_rows)
    sel, _ = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    ql, kl, vl = wl.live_block(req, wl.make_step(cfg, 0, 0))
    o_ref, lse_ref = orc.decode_attention(f64(ql), f64(kl), f64(vl), pk, pv, table, sel,
                                          cfg.sm_scale)
    dpk, dpv = P.cuda(P.bf16_of(pk)), P.cuda(P.bf16_of(pv))
    dtab, dsel = P.cuda(torch.from_numpy(table)), P.cuda(torch.from_numpy(sel))
    outs = {}
    for s in (1, 4, 7):
        out, lse = api.decode_attention(P.cuda(ql), P.cuda(kl), P.cuda(vl), dpk, dpv, dtab, dsel,
                                        n_splits=s)
        torch.cuda.synchronize()
        outs[s] = (out.cpu().double().numpy(), lse.cpu().double().numpy())
    lines = []
    for s, (o, l) in outs.items():
        mx, mean = P.assert_close_out(o, o_ref, f"S={s} vs oracle")
        lerr = np.abs(l - lse_ref).max()
        assert lerr <= P.LSE_MAX_ABS
        lines.append(f"S={s} vs oracle: out max {mx:.3e} mean {mean:.3e}; lse max {lerr:.3e}")
    for s in (4, 7):
        d = np.abs(outs[s][0] - outs[1][0])
        lines.append(f"S={s} vs S=1: out max {d.max():.3e} mean {d.mean():.3e}")
    with capsys.disabled():
        print("\n" + "\n".join(lines))
