"""Pins of the CPU oracle against things other than itself.

Each ``check_*`` takes the oracle module (or a deliberately broken copy of it)
and raises AssertionError when the oracle disagrees with the pin.  The pins are
library routines computing the same quantity another way (torch's fp64
scaled-dot-product attention with an explicit mask), counting formulations of
the rank rules, brute force with scalar loops, closed forms and invariants.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch


def rand(gen, *shape):
    return torch.randn(*shape, generator=gen, dtype=torch.float64).numpy()


def sdpa(q, k, v, mask=None, scale=None):
    """torch fp64 SDPA on [L, D] x [S, D] -> [L, D]; mask True = attend."""
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(x))[None, None] for x in (q, k, v))
    mt = None if mask is None else torch.from_numpy(mask)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mt, scale=scale)
    return o[0, 0].numpy()


# ----------------------------------------------------------- chunk attention --

def check_chunk_attention(orc, seed=1, n=3, c=6, hq=4, hkv=2, d=8):
    """Chunked prefill == dense attention over the whole prefix with a
    block-diagonal mask (torch SDPA), head by head."""
    gen = torch.Generator().manual_seed(seed)
    rows = n * (c + 1)
    q, k, v = rand(gen, rows, hq, d), rand(gen, rows, hkv, d), rand(gen, rows, hkv, d)
    scale = 0.37
    got = orc.chunk_attention(q, k, v, n, c, scale)
    blk = np.arange(rows) // (c + 1)
    mask = blk[:, None] == blk[None, :]
    for h in range(hq):
        g = h // (hq // hkv)
        want = sdpa(q[:, h], k[:, g], v[:, g], mask, scale)
        assert np.max(np.abs(got[:, h] - want)) < 1e-12, "chunk attention != masked dense SDPA"
        some = [0, c, c + 1, rows - 1, rows // 2]
        at_rows = orc.chunk_attention_rows(q, k, v, c, some, scale)
        assert np.max(np.abs(at_rows[:, h] - want[some])) < 1e-12, \
            "chunk attention at sampled rows != masked dense SDPA"


# ------------------------------------------------------------ window scores --

def check_scores_vs_sdpa(orc, seed=2, n=3, c=5, w=4, hq=6, hkv=2, d=8):
    """Attention with V = identity returns the probability matrix itself;
    its column sums over window rows and heads are the scores."""
    gen = torch.Generator().manual_seed(seed)
    rows = n * (c + 1)
    k = rand(gen, rows, hkv, d)
    q_win = rand(gen, w, hq, d)
    scale = 0.41
    got = orc.window_scores(q_win, k, n, c, scale)
    assert got.shape == (n, c + 1)
    eye = np.eye(c + 1)
    for j in range(n):
        want = np.zeros(c + 1)
        for h in range(hq):
            g = h // (hq // hkv)
            p = sdpa(q_win[:, h], k[j * (c + 1):(j + 1) * (c + 1), g], eye, None, scale)
            want += p.sum(axis=0)
        assert np.max(np.abs(got[j] - want)) < 1e-12, "scores != column sums of SDPA probabilities"


def check_scores_brute_force(orc, seed=3):
    """Scalar loops with math.exp on a tiny case."""
    gen = torch.Generator().manual_seed(seed)
    n, c, w, hq, hkv, d = 2, 3, 2, 2, 1, 3
    rows = n * (c + 1)
    k = rand(gen, rows, hkv, d)
    q_win = rand(gen, w, hq, d)
    scale = 0.9
    got = orc.window_scores(q_win, k, n, c, scale)
    for j in range(n):
        for t in range(c + 1):
            total = 0.0
            for ww in range(w):
                for h in range(hq):
                    x = [scale * sum(q_win[ww, h, e] * k[j * (c + 1) + u, 0, e] for e in range(d))
                         for u in range(c + 1)]
                    total += math.exp(x[t]) / sum(math.exp(xu) for xu in x)
            assert abs(got[j, t] - total) < 1e-12, "scores != scalar brute force"


def check_scores_invariants(orc, seed=4):
    """Each window row's probabilities sum to one, so every chunk's scores sum
    to W * Hq; equal keys share the mass uniformly; one dominant key takes it."""
    gen = torch.Generator().manual_seed(seed)
    n, c, w, hq, hkv, d = 4, 9, 3, 4, 2, 8
    rows = n * (c + 1)
    k = rand(gen, rows, hkv, d)
    q_win = rand(gen, w, hq, d)
    got = orc.window_scores(q_win, k, n, c, 0.3)
    assert np.max(np.abs(got.sum(axis=1) - w * hq)) < 1e-10, "scores do not sum to W*Hq"
    k_eq = np.repeat(k[:1], rows, axis=0)
    got = orc.window_scores(q_win, k_eq, n, c, 0.3)
    assert np.max(np.abs(got - w * hq / (c + 1))) < 1e-12, "equal keys must split the mass evenly"
    q1 = np.ones((1, 1, 4))
    k1 = np.zeros((c + 1, 1, 4))
    k1[5] = 100.0
    got = orc.window_scores(q1, k1, 1, c, 1.0)
    assert abs(got[0, 5] - 1.0) < 1e-12 and got[0, :5].max() < 1e-100, "dominant key must take all mass"


def check_scores_single_row(orc, seed=5):
    """W = 1, Hq = 1: the score row is one softmax row (torch.softmax)."""
    gen = torch.Generator().manual_seed(seed)
    c, d = 11, 16
    k = rand(gen, c + 1, 1, d)
    q_win = rand(gen, 1, 1, d)
    got = orc.window_scores(q_win, k, 1, c, 0.25)
    logits = torch.from_numpy(0.25 * (q_win[0, 0] @ k[:, 0].T))
    want = torch.softmax(logits, dim=0).numpy()
    assert np.max(np.abs(got[0] - want)) < 1e-14, "single-row scores != softmax"


# ----------------------------------------------------------------- ranking --

def beats(a_val, a_idx, b_val, b_idx):
    """True when (a_val, a_idx) ranks strictly before (b_val, b_idx):
    larger value first, -0 == +0, NaN last, ties to the lower index."""
    a_nan, b_nan = math.isnan(a_val), math.isnan(b_val)
    if a_nan != b_nan:
        return b_nan
    if not a_nan and a_val != b_val:
        return a_val > b_val
    return a_idx < b_idx


def kept_by_counting(values, n_keep):
    """Index t is kept iff fewer than n_keep indices beat it (O(n^2))."""
    vals = [float(x) for x in values]
    kept = []
    for t, vt in enumerate(vals):
        n_beat = sum(1 for u, vu in enumerate(vals) if u != t and beats(vu, u, vt, t))
        if n_beat < n_keep:
            kept.append(t)
    return kept


def ranked_by_counting(values, n_take):
    """The first n_take indices in rank order, by counting who beats whom."""
    vals = [float(x) for x in values]
    rank = {}
    for t, vt in enumerate(vals):
        rank[t] = sum(1 for u, vu in enumerate(vals) if u != t and beats(vu, u, vt, t))
    return [t for t, _ in sorted(rank.items(), key=lambda kv: kv[1])][:n_take]


def top_b_cases():
    gen = np.random.default_rng(7)
    cases = []
    cases.append(gen.standard_normal((5, 17)))
    cases.append(np.round(gen.standard_normal((4, 21)) * 2) / 2)           # many exact ties
    z = np.zeros((2, 9))
    z[0, 3], z[1, 2] = -0.0, -0.0
    z[0, 5] = 1.0
    cases.append(z)                                                        # +/-0 ties
    cases.append(np.full((3, 12), 0.25))                                   # all equal
    base = np.ones((1, 7))
    base[0, 4] = 1.0 + 1e-12                                              # equal after fp32 rounding
    cases.append(base)
    return cases


def check_top_b(orc):
    for scores in top_b_cases():
        n, rows = scores.shape
        for n_keep in sorted({0, 1, 3, rows - 2, rows - 1}):
            if n_keep > rows - 1:
                continue
            got = orc.top_b(scores, n_keep)
            assert got.shape == (n, n_keep)
            for j in range(n):
                want = kept_by_counting(scores[j, 1:].astype(np.float32), n_keep)
                assert list(got[j]) == want, f"top_b mismatch on row {j}, B={n_keep}"


def check_select(orc):
    gen = np.random.default_rng(11)
    cases = [
        (gen.standard_normal(13).astype(np.float32), gen.standard_normal(13).astype(np.float32)),
        (np.round(gen.standard_normal(16)).astype(np.float32), np.zeros(16, np.float32)),
        (np.array([0.0, -0.0, 1.0, 0.0], np.float32), np.array([-0.0, 0.0, -1.0, -0.0], np.float32)),
        # 1 + 2^-25 rounds to 1 in fp32: chunk 2 ties chunk 0 and loses on index
        (np.array([1.0, 0.5, 1.0, 0.75], np.float32),
         np.array([0.0, 0.0, 2.0 ** -25, 0.0], np.float32)),
        (np.full(9, 0.5, np.float32), np.full(9, 0.25, np.float32)),
    ]
    for s_i, s_p in cases:
        n = s_i.shape[0]
        s_want = [float(np.float32(np.float32(a) + np.float32(b))) for a, b in zip(s_i, s_p)]
        for k_sel in sorted({1, 2, n // 2, n}):
            sel, s = orc.select_chunks(s_i, s_p, k_sel)
            assert [float(x) for x in s] == s_want, "s must be the fp32 sum"
            assert list(sel) == ranked_by_counting(s_want, k_sel), "select order mismatch"


# ------------------------------------------------------------------ decode --

def check_split_equals_concat(orc, seed=8):
    """Split per chunk + LSE merge == one softmax over the concatenation."""
    gen = torch.Generator().manual_seed(seed)
    hq, hkv, d, lq = 6, 2, 16, 9
    pool_rows = 40
    pool_k, pool_v = rand(gen, pool_rows, hkv, d), rand(gen, pool_rows, hkv, d)
    table = np.array([[0, 5], [7, 9], [20, 1], [25, 15]], dtype=np.int32)
    sel = np.array([3, 0, 2], dtype=np.int32)
    q, ks, vs = rand(gen, lq, hq, d), rand(gen, lq, hkv, d), rand(gen, lq, hkv, d)
    out1, lse1 = orc.decode_attention(q, ks, vs, pool_k, pool_v, table, sel, 0.3)
    out2, lse2 = orc.decode_attention_split(q, ks, vs, pool_k, pool_v, table, sel, 0.3)
    assert np.max(np.abs(out1 - out2)) < 1e-12 and np.max(np.abs(lse1 - lse2)) < 1e-12


def check_split_at_arbitrary_points(orc, seed=14):
    """Split + LSE merge at arbitrary cut points of the concatenated keys
    (inside chunk slots and across their edges, not only at chunk
    boundaries) == one softmax over the concatenation (torch SDPA and
    torch.logsumexp), for several random cut sets."""
    gen = torch.Generator().manual_seed(seed)
    hq, hkv, d, lq = 6, 2, 16, 7
    pool_k, pool_v = rand(gen, 48, hkv, d), rand(gen, 48, hkv, d)
    table = np.array([[0, 11], [13, 9], [30, 17]], dtype=np.int32)
    sel = np.array([2, 0, 1], dtype=np.int32)
    q, ks, vs = rand(gen, lq, hq, d), rand(gen, lq, hkv, d), rand(gen, lq, hkv, d)
    kk = np.concatenate([orc.gather_selected(pool_k, table, sel), ks], axis=0)
    vv = np.concatenate([orc.gather_selected(pool_v, table, sel), vs], axis=0)
    n_keys = kk.shape[0]
    for trial in range(6):
        n_cuts = 1 + trial
        cuts = sorted(torch.randperm(n_keys - 1, generator=gen)[:n_cuts].add(1).tolist())
        edges = [0] + cuts + [n_keys]
        parts = [orc.split_partials(q, kk[a:b], vv[a:b], hq // hkv, 0.4)
                 for a, b in zip(edges[:-1], edges[1:])]
        out, lse = orc.lse_merge(parts)
        for h in range(hq):
            g = h // (hq // hkv)
            want = sdpa(q[:, h], kk[:, g], vv[:, g], None, 0.4)
            assert np.max(np.abs(out[:, h] - want)) < 1e-12, f"split at {cuts} != one softmax"
            lg = torch.from_numpy(0.4 * q[:, h] @ kk[:, g].T)
            assert np.max(np.abs(lse[:, h] - torch.logsumexp(lg, dim=1).numpy())) < 1e-12


def check_decode_vs_sdpa(orc, seed=9):
    """Decode == SDPA over [selected rows ; live rows]; lse == logsumexp."""
    gen = torch.Generator().manual_seed(seed)
    hq, hkv, d, lq = 4, 2, 8, 5
    pool_k, pool_v = rand(gen, 30, hkv, d), rand(gen, 30, hkv, d)
    table = np.array([[2, 6], [10, 4], [16, 11]], dtype=np.int32)
    sel = np.array([2, 1], dtype=np.int32)
    q, ks, vs = rand(gen, lq, hq, d), rand(gen, lq, hkv, d), rand(gen, lq, hkv, d)
    out, lse = orc.decode_attention(q, ks, vs, pool_k, pool_v, table, sel, 0.5)
    rows = list(range(16, 27)) + list(range(10, 14))
    kk = np.concatenate([pool_k[rows], ks], axis=0)
    vv = np.concatenate([pool_v[rows], vs], axis=0)
    for h in range(hq):
        g = h // 2
        want = sdpa(q[:, h], kk[:, g], vv[:, g], None, 0.5)
        assert np.max(np.abs(out[:, h] - want)) < 1e-12, "decode != SDPA"
        lg = torch.from_numpy(0.5 * q[:, h] @ kk[:, g].T)
        assert np.max(np.abs(lse[:, h] - torch.logsumexp(lg, dim=1).numpy())) < 1e-12


def check_dense_equivalence(orc, seed=10):
    """K = N and B = C: the whole sparse path (scores, top-B, compaction,
    selection, decode) equals dense attention of the live rows over every
    prefix row (BOS rows included) and the live rows (torch SDPA)."""
    gen = torch.Generator().manual_seed(seed)
    n, c, w, hq, hkv, d, lq = 3, 6, 2, 4, 2, 8, 5
    rows = n * (c + 1)
    k, v = rand(gen, rows, hkv, d), rand(gen, rows, hkv, d)
    q_win = rand(gen, w, hq, d)
    scale = 0.35
    scores = orc.window_scores(q_win, k, n, c, scale)
    kept = orc.top_b(scores, c)
    slot = np.array([2 * (c + 1), 0, c + 1], dtype=np.int32)       # permuted slots
    pool_k, pool_v = np.zeros((rows, hkv, d)), np.zeros((rows, hkv, d))
    table = orc.compact(k, v, kept, slot, c, pool_k, pool_v)
    sel, _ = orc.select_chunks(rand(gen, n).astype(np.float32), np.zeros(n, np.float32), n)
    q, ks, vs = rand(gen, lq, hq, d), rand(gen, lq, hkv, d), rand(gen, lq, hkv, d)
    out, _ = orc.decode_attention(q, ks, vs, pool_k, pool_v, table, sel, scale)
    kk = np.concatenate([k, ks], axis=0)
    vv = np.concatenate([v, vs], axis=0)
    for h in range(hq):
        g = h // 2
        want = sdpa(q[:, h], kk[:, g], vv[:, g], None, scale)
        assert np.max(np.abs(out[:, h] - want)) < 1e-12, "K=N, B=C path != dense attention"


def check_compact(orc, seed=12):
    gen = torch.Generator().manual_seed(seed)
    n, c, hkv, d, b = 3, 5, 2, 4, 2
    rows = n * (c + 1)
    k, v = rand(gen, rows, hkv, d), rand(gen, rows, hkv, d)
    kept = np.array([[0, 4], [1, 2], [3, 4]], dtype=np.int32)
    slot = np.array([6, 0, 3], dtype=np.int32)
    pk, pv = np.full((9, hkv, d), np.nan), np.full((9, hkv, d), np.nan)
    table = orc.compact(k, v, kept, slot, c, pk, pv)
    assert table.tolist() == [[6, 3], [0, 3], [3, 3]]
    for j in range(n):
        src = [j * (c + 1)] + [j * (c + 1) + 1 + t for t in kept[j]]
        assert np.array_equal(pk[slot[j]:slot[j] + b + 1], k[src])
        assert np.array_equal(pv[slot[j]:slot[j] + b + 1], v[src])


# -------------------------------------------------------------- cost model --

def check_cost_model(orc):
    """The oracle's MAC counts equal the closed forms, and they scale as the
    per-step complexity O(N C^2 + (L_d^2 + K C) T) says: prefill linear in N
    and quadratic in C; decode independent of N at fixed K, B, Lq."""
    gen = torch.Generator().manual_seed(13)
    hq, hkv, d = 4, 2, 8
    for n, c, w in itertools.product((2, 3), (4, 7), (0, 3)):
        rows = n * (c + 1)
        q, k, v = rand(gen, rows, hq, d), rand(gen, rows, hkv, d), rand(gen, rows, hkv, d)
        cnt = orc.MacCounter()
        orc.chunk_attention(q, k, v, n, c, 0.3, counter=cnt)
        orc.window_scores(rand(gen, w, hq, d), k, n, c, 0.3, counter=cnt)
        assert cnt.macs == orc.prefill_macs(n, c, w, hq, d)
        assert cnt.macs == 2 * hq * n * (c + 1) ** 2 * d + hq * n * w * (c + 1) * d
    macs = []
    for n in (4, 8):
        pool_k, pool_v = rand(gen, n * 3, hkv, d), rand(gen, n * 3, hkv, d)
        table = np.array([[3 * j, 3] for j in range(n)], dtype=np.int32)
        sel = np.array([1, 3], dtype=np.int32)
        lq = 5
        q, ks, vs = rand(gen, lq, hq, d), rand(gen, lq, hkv, d), rand(gen, lq, hkv, d)
        cnt = orc.MacCounter()
        orc.decode_attention(q, ks, vs, pool_k, pool_v, table, sel, 0.3, counter=cnt)
        assert cnt.macs == orc.decode_step_macs(lq, 6, hq, d) == 2 * hq * lq * (6 + lq) * d
        macs.append(cnt.macs)
    assert macs[0] == macs[1], "decode cost must not depend on N"


# ------------------------------------------------- alternative rankings --

def check_scores_alt_readings(orc, seed=16):
    """Per-KV-head scores: column sums of SDPA-with-identity probabilities
    over each KV head's query heads; summed over KV heads they are the
    shared scores.  Window keys in the denominator: the chunk columns of the
    probability matrix over [chunk keys ; window keys] (SDPA with V =
    identity over the concatenation); the scores then sum to less than
    W * Hq by exactly the mass on the window keys."""
    gen = torch.Generator().manual_seed(seed)
    n, c, w, hq, hkv, d = 3, 5, 4, 6, 2, 8
    rows = n * (c + 1)
    k = rand(gen, rows, hkv, d)
    q_win = rand(gen, w, hq, d)
    k_win = rand(gen, w, hkv, d)
    scale = 0.4
    per = orc.window_scores_alt(q_win, k, n, c, scale, per_kv_head=True)
    shared = orc.window_scores(q_win, k, n, c, scale)
    assert np.max(np.abs(per.sum(axis=1) - shared)) < 1e-12
    with_w = orc.window_scores_alt(q_win, k, n, c, scale, k_win=k_win)
    with_w_per = orc.window_scores_alt(q_win, k, n, c, scale, per_kv_head=True, k_win=k_win)
    assert np.max(np.abs(with_w_per.sum(axis=1) - with_w)) < 1e-12
    for j in range(n):
        lo = j * (c + 1)
        window_mass = 0.0
        for h in range(hq):
            g = h // (hq // hkv)
            keys = np.concatenate([k[lo:lo + c + 1, g], k_win[:, g]], axis=0)
            eye = np.eye(keys.shape[0])
            pm = sdpa(q_win[:, h], keys, eye, None, scale)       # [W, C+1+W] probabilities
            window_mass += pm[:, c + 1:].sum()
            want_g = np.zeros(c + 1)
            for h2 in range(g * (hq // hkv), (g + 1) * (hq // hkv)):
                want_g += sdpa(q_win[:, h2], keys, eye, None, scale)[:, :c + 1].sum(axis=0)
            assert np.max(np.abs(with_w_per[j, g] - want_g)) < 1e-12
        assert abs(with_w[j].sum() - (w * hq - window_mass)) < 1e-10


def check_per_head_topb_and_compact(orc, seed=17):
    """Per-KV-head top-B equals top_b on each head's row; each head's
    column of a slot holds BOS and that head's kept rows only."""
    gen = torch.Generator().manual_seed(seed)
    n, c, hkv, d, b = 3, 9, 2, 4, 3
    scores = rand(gen, n, hkv, c + 1)
    kept = orc.top_b_per_head(scores, b)
    for j in range(n):
        for g in range(hkv):
            assert kept[j, g].tolist() == sorted(ranked_by_counting(
                [float(np.float32(x)) for x in scores[j, g, 1:]], b))
    rows = n * (c + 1)
    k, v = rand(gen, rows, hkv, d), rand(gen, rows, hkv, d)
    slot = np.array([8, 0, 4], dtype=np.int32)
    pk, pv = np.full((12, hkv, d), np.nan), np.full((12, hkv, d), np.nan)
    table = orc.compact_per_head(k, v, kept, slot, c, pk, pv)
    assert table.tolist() == [[8, 4], [0, 4], [4, 4]]
    for j in range(n):
        for g in range(hkv):
            src = [j * (c + 1)] + [j * (c + 1) + 1 + int(t) for t in kept[j, g]]
            assert np.array_equal(pk[slot[j]:slot[j] + b + 1, g], k[src, g])
            assert np.array_equal(pv[slot[j]:slot[j] + b + 1, g], v[src, g])


def check_layers_are_independent(orc, seed=18):
    """Multi-layer prefill: each layer equals the single-layer prefill of its
    own tensors (chunk attention against SDPA with a block mask), and
    reversing the layer order reverses the results."""
    gen = torch.Generator().manual_seed(seed)
    n_layers, n, c, w, hq, hkv, d, b = 3, 2, 5, 3, 4, 2, 8, 2
    rows = n * (c + 1)
    q, k, v = rand(gen, n_layers, rows, hq, d), rand(gen, n_layers, rows, hkv, d), \
        rand(gen, n_layers, rows, hkv, d)
    q_win = rand(gen, n_layers, w, hq, d)
    slot = np.array([3, 0], dtype=np.int32)
    res = orc.chunk_prefill_layers(q, k, v, q_win, n, c, b, slot, 6, 0.3)
    rev = orc.chunk_prefill_layers(q[::-1], k[::-1], v[::-1], q_win[::-1], n, c, b, slot, 6, 0.3)
    blk = np.arange(rows) // (c + 1)
    mask = blk[:, None] == blk[None, :]
    for l in range(n_layers):
        for h in range(hq):
            want = sdpa(q[l, :, h], k[l, :, h // 2], v[l, :, h // 2], mask, 0.3)
            assert np.max(np.abs(res[l]["out"][:, h] - want)) < 1e-12
        s1 = orc.window_scores(q_win[l], k[l], n, c, 0.3)
        assert np.max(np.abs(res[l]["scores"] - s1)) < 1e-12
        assert np.array_equal(res[l]["kept"], orc.top_b(s1, b))
        for j in range(n):                      # layer l's pool holds layer l's own rows
            src = [j * (c + 1)] + [j * (c + 1) + 1 + int(t) for t in res[l]["kept"][j]]
            assert np.array_equal(res[l]["pool_k"][slot[j]:slot[j] + b + 1], k[l, src])
            assert np.array_equal(res[l]["pool_v"][slot[j]:slot[j] + b + 1], v[l, src])
        for key in ("out", "scores", "kept", "pool_k", "pool_v", "table"):
            assert np.array_equal(res[l][key], rev[n_layers - 1 - l][key])


# ------------------------------------------------------------ reselection --

def check_chunk_mass(orc, seed=19):
    """The masses of the selected chunks plus the live block's mass sum to
    one at the step's own lse (the decode softmax, pinned to SDPA, sums to
    one); a selected chunk's mass is e^(m - lse) l of its split partial
    (the "free" decode mass); an unselected chunk's mass equals a brute-force
    scalar loop."""
    gen = torch.Generator().manual_seed(seed)
    hq, hkv, d, lq = 4, 2, 8, 5
    pool_k, pool_v = rand(gen, 40, hkv, d), rand(gen, 40, hkv, d)
    table = np.array([[0, 7], [9, 5], [20, 11], [33, 4]], dtype=np.int32)
    sel = np.array([2, 0], dtype=np.int32)
    q, ks, vs = rand(gen, lq, hq, d), rand(gen, lq, hkv, d), rand(gen, lq, hkv, d)
    scale = 0.45
    _, lse = orc.decode_attention(q, ks, vs, pool_k, pool_v, table, sel, scale)
    m_sel = orc.chunk_mass(q, pool_k, table, sel, lse, scale)
    self_mass = 0.0
    for h in range(hq):
        logits = scale * (q[:, h] @ ks[:, h // 2].T)
        self_mass += np.exp(logits - lse[:, h:h + 1]).sum()
    assert abs(m_sel.sum() + self_mass / (lq * hq) - 1.0) < 1e-12
    for i, c in enumerate(sel):
        lo, n = table[c]
        m, l, _ = orc.split_partials(q, pool_k[lo:lo + n], pool_v[lo:lo + n], 2, scale)
        assert abs((np.exp(m - lse) * l).sum() / (lq * hq) - m_sel[i]) < 1e-12
    got = orc.chunk_mass(q, pool_k, table, [3], lse, scale)[0]
    want = 0.0
    for r in range(lq):
        for h in range(hq):
            for t in range(33, 37):
                x = scale * sum(q[r, h, e] * pool_k[t, h // 2, e] for e in range(d))
                want += math.exp(x - lse[r, h])
    assert abs(got - want / (lq * hq)) < 1e-12


def check_reselect(orc):
    """lambda = 0 gives the static selection; the ranking follows the
    counting rule on fl32(s + fl32(lambda * mass)); a large enough mass lifts
    an unselected chunk into the selection."""
    rng = np.random.default_rng(3)
    s = rng.standard_normal(12).astype(np.float32)
    mass = rng.random(12).astype(np.float32)
    sel0, _ = orc.reselect_chunks(s, mass, 0.0, 4)
    static, _ = orc.select_chunks(s, np.zeros(12, np.float32), 4)
    assert list(sel0) == list(static)
    for lam in (0.5, 3.0, 100.0):
        sel, s2 = orc.reselect_chunks(s, mass, lam, 5)
        want = [float(np.float32(np.float32(x) + np.float32(np.float32(lam) * np.float32(m))))
                for x, m in zip(s, mass)]
        assert [float(x) for x in s2] == want
        assert list(sel) == ranked_by_counting(want, 5)
    low = int(np.argmin(s))
    boost = np.zeros(12, np.float32)
    boost[low] = 1.0
    sel, _ = orc.reselect_chunks(s, boost, float(s.max() - s.min()) + 1.0, 1)
    assert list(sel) == [low]


# ----------------------------------------------------------- chunk scores --

def check_loglik_vs_cross_entropy(orc, seed=15):
    """Summed label log-likelihood == -(torch cross-entropy, summed), the
    library's own log-softmax + NLL, chunk by chunk, and the row values."""
    gen = torch.Generator().manual_seed(seed)
    n, r, v = 3, 5, 37
    z = torch.randn(n, r, v, generator=gen, dtype=torch.float64) * 3.0
    y = torch.randint(0, v, (r,), generator=gen)
    score, rows = orc.chunk_loglik(z.numpy(), y.numpy())
    for j in range(n):
        ce = torch.nn.functional.cross_entropy(z[j], y, reduction="none").numpy()
        assert np.max(np.abs(rows[j] + ce)) < 1e-12, "row log-likelihood != -cross-entropy"
        assert abs(score[j] + ce.sum()) < 1e-11, "chunk score != -summed cross-entropy"


def check_loglik_closed_forms(orc):
    """Uniform logits give -R log V; one class gives 0; two classes give the
    log-sigmoid of the logit margin; adding a constant to a row changes
    nothing (log-softmax is shift invariant)."""
    z = np.full((2, 4, 9), 0.7)
    score, _ = orc.chunk_loglik(z, np.array([0, 3, 8, 5]))
    assert np.allclose(score, -4 * math.log(9.0), rtol=0, atol=1e-12)
    score, _ = orc.chunk_loglik(np.random.default_rng(0).standard_normal((3, 6, 1)), np.zeros(6, int))
    assert np.all(score == 0.0)
    a = np.array([[[1.5, -0.25], [0.0, 2.0], [-3.0, 1.0]]])
    score, rows = orc.chunk_loglik(a, np.array([0, 1, 0]))
    want = [-math.log1p(math.exp(-(1.5 + 0.25))), -math.log1p(math.exp(-2.0)),
            -math.log1p(math.exp(4.0))]
    assert np.max(np.abs(rows[0] - want)) < 1e-12
    shifted = a + np.array([[[10.0], [-7.0], [3.5]]])
    assert np.max(np.abs(orc.chunk_loglik(shifted, np.array([0, 1, 0]))[1] - rows)) < 1e-12


def check_hand_worked_pipeline(orc):
    """A two-chunk example worked out by hand, end to end: prefill, ranking,
    compaction, selection, one decode step, chunk masses and reselection,
    with keys whose logits are logs of small integers so every probability
    is an exact fraction.

    One query head, one KV head, D = 2, scale 1; every query is (1, 0), so a
    key's logit is its first coordinate.
      chunk 0 rows (BOS, t1, t2, t3): logits ln 6, 0, ln 2, ln 3 -> p = (6, 1, 2, 3) / 12
      chunk 1 rows: all logits 0 -> p = 1/4 each
    """
    ln = math.log
    rows = 4
    k = np.zeros((2 * rows, 1, 2))
    k[0:4, 0, 0] = [ln(6), 0.0, ln(2), ln(3)]
    k[:, 0, 1] = [5.0, -3.0, 7.0, 1.0, 2.0, 9.0, -4.0, 6.0]        # never reaches a logit
    v = np.zeros((2 * rows, 1, 2))
    v[0:4, 0] = [[12, 0], [24, -12], [0, 12], [12, 12]]
    v[4:8, 0] = [[4, 0], [0, 4], [4, 4], [0, 0]]
    q = np.zeros((2 * rows, 1, 2))
    q[:, 0, 0] = 1.0
    q_win = np.zeros((2, 1, 2))
    q_win[:, 0, 0] = 1.0

    # chunk attention: each chunk's rows see only that chunk's four keys
    out = orc.chunk_attention(q, k, v, 2, 3, 1.0)
    assert np.allclose(out[0:4, 0], [11.0, 4.0], rtol=0, atol=1e-12), "chunk 0 output != (11, 4)"
    assert np.allclose(out[4:8, 0], [2.0, 2.0], rtol=0, atol=1e-12), "chunk 1 output != (2, 2)"

    # window scores: two identical window rows, so twice each probability
    scores = orc.window_scores(q_win, k, 2, 3, 1.0)
    assert np.allclose(scores, [[1.0, 1 / 6, 1 / 3, 1 / 2], [0.5, 0.5, 0.5, 0.5]],
                       rtol=0, atol=1e-12), "window scores"

    # with the window's own keys (logits 0 and ln 2, e^x summing to 3) in the
    # denominator: chunk 0's row sums 12 + 3 = 15, chunk 1's 4 + 3 = 7
    k_win = np.zeros((2, 1, 2))
    k_win[:, 0, 0] = [0.0, ln(2)]
    alt = orc.window_scores_alt(q_win, k, 2, 3, 1.0, k_win=k_win)
    assert np.allclose(alt, [[12 / 15, 2 / 15, 4 / 15, 6 / 15], [2 / 7] * 4], rtol=0, atol=1e-12), (
        "scores with the window keys in the denominator")

    # top-2 of the content tokens: BOS (the largest score of chunk 0) is not
    # ranked; chunk 1's four-way tie keeps the lowest indices
    kept = orc.top_b(scores, 2)
    assert kept.tolist() == [[1, 2], [0, 1]], f"kept {kept.tolist()}"

    # slots at rows 5 and 0 of a 9-row pool: BOS then the kept rows
    pool_k = np.full((9, 1, 2), np.nan)
    pool_v = np.full((9, 1, 2), np.nan)
    table = orc.compact(k, v, kept, np.array([5, 0]), 3, pool_k, pool_v)
    assert table.tolist() == [[5, 3], [0, 3]]
    assert np.array_equal(pool_v[5:8, 0], [[12, 0], [0, 12], [12, 12]])
    assert np.array_equal(pool_v[0:3, 0], [[4, 0], [0, 4], [4, 4]])
    assert np.isnan(pool_v[3:5]).all() and np.isnan(pool_v[8]).all(), "rows outside the slots"

    # s = s_I + s_P = (0.5, -1.5): chunk 0 first
    sel, s = orc.select_chunks(np.array([-1.0, -2.0]), np.array([1.5, 0.5]), 2)
    assert sel.tolist() == [0, 1] and s.tolist() == [0.5, -1.5]

    # decode, one live row with key logit 0 and value (0, 24): weights
    # (6, 2, 3 | 1, 1, 1 | 1) / 15 over chunk 0's slot, chunk 1's slot, itself
    k_self = np.array([[[0.0, 8.0]]])
    v_self = np.array([[[0.0, 24.0]]])
    dec, lse = orc.decode_attention(q[:1], k_self, v_self, pool_k, pool_v, table, sel, 1.0)
    assert np.allclose(dec[0, 0], [116 / 15, 92 / 15], rtol=0, atol=1e-12), f"decode {dec[0, 0]}"
    assert abs(lse[0, 0] - ln(15)) < 1e-12, "decode lse != ln 15"
    # chunk 1 alone: weights (1, 1, 1 | 1) / 4
    dec1, lse1 = orc.decode_attention(q[:1], k_self, v_self, pool_k, pool_v, table, sel[1:], 1.0)
    assert np.allclose(dec1[0, 0], [2.0, 8.0], rtol=0, atol=1e-12) and abs(lse1[0, 0] - ln(4)) < 1e-12

    # attention mass at the step's lse: 11/15 on chunk 0, 3/15 on chunk 1
    # (the live row keeps the last 1/15)
    mass = orc.chunk_mass(q[:1], pool_k, table, [0, 1], lse, 1.0)
    assert np.allclose(mass, [11 / 15, 3 / 15], rtol=0, atol=1e-12), f"mass {mass}"
    # reselecting one chunk from s = (-1.5, 0.5): chunk 0 overtakes chunk 1
    # once lam * (11/15 - 3/15) > 2, that is lam > 3.75
    for lam, want in ((0.0, 1), (3.5, 1), (4.0, 0)):
        sel2, s2 = orc.reselect_chunks(np.array([-1.5, 0.5]), mass, lam, 1)
        assert sel2.tolist() == [want], (lam, sel2.tolist())
        assert np.allclose(s2, [-1.5 + lam * 11 / 15, 0.5 + lam / 5], rtol=0, atol=1e-6)


ALL_CHECKS = [
    check_chunk_attention, check_scores_vs_sdpa, check_scores_brute_force, check_scores_invariants,
    check_scores_single_row, check_top_b, check_select, check_split_equals_concat,
    check_split_at_arbitrary_points, check_loglik_vs_cross_entropy, check_loglik_closed_forms,
    check_scores_alt_readings, check_per_head_topb_and_compact, check_layers_are_independent,
    check_chunk_mass, check_reselect,
    check_decode_vs_sdpa, check_dense_equivalence, check_compact, check_cost_model,
    check_hand_worked_pipeline,
]
