"""Plain fp64 CPU oracle for the sparse chunked-KV prefill and decode path.

TEST INFRASTRUCTURE ONLY.  This module is the independent definition that the
CUDA path is checked against.  Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it; the library itself never
does, and shares no code, table or helper with it.

Every function here follows the method as stated in the technical summary of
"Prefilling-dLLM: Predictive Prefilling for Long-Context Inference in
Diffusion Language Models" (gist.science pages, es/nl/ko/ja).  Citation keys
used below:

  [M1]  Methodology, 1. Chunked Prefill and KV Caching -- the prefix is split
        into N non-overlapping chunks of fixed size C, a BOS token is put in
        front of every chunk, each chunk is processed on its own with
        bidirectional attention inside the chunk; chunks are scored with
        s_I and s_P and the K best by s = s_I + s_P are kept.
  [M2]  Methodology, 2. Two-Level Sparsity -- only the top-K chunks take part
        in decode attention (inter-chunk); inside a chunk, tokens are ranked
        by the cumulative bidirectional attention weight they receive from
        the query tokens and only the top-B are kept in the KV cache
        (intra-chunk).
  [M3]  Methodology, 3. Decoding with Static KV Reuse -- the cached KV of the
        selected chunks is static across all T denoising steps; only the
        query and response tokens are recomputed; per-step cost drops from
        O((L_p+L_d)^2 T) to O(N C^2 + (L_d^2 + K C) T).
  [AK]  Attention Kernel Optimization -- the split-S kernel partitions the KV
        dimension, processes the non-contiguous chunks independently and
        merges the partial results by a log-sum-exp reduction.

Readings where the pages leave a step open (each is stated where it is used):
  R1  BOS is row 0 of every chunk (C+1 rows per chunk) and is always kept in
      the cache; top-B ranks only the C content tokens.
  R2  "cumulative attention weight with the query tokens" is the column sum,
      over all query-window rows and all query heads, of the window rows'
      softmax probabilities over the chunk's own C+1 keys.  One token
      selection is shared by every head.
  R3  Ranking decisions are taken on fp32 values (the precision the kernels
      rank in): scores are rounded to fp32 before top-B, s = fl32(s_I + s_P)
      is an fp32 add.  Ties go to the lower index; -0.0 equals +0.0; NaN
      ranks below every number.  s_I and s_P are both "higher = more
      relevant" (a caller holding a raw NLL negates it).
  R4  The decode live block (query window + response, Lq rows) attends to
      itself and to the kept rows of the selected chunks, with no mask.
  R5  The softmax scale is 1/sqrt(D) unless given.
  R7  Dynamic reselection (the pages list static selection as a limitation):
      at a reselection step the live rows score every chunk j of the
      sequence by the attention mass its cached rows would receive at that
      step's normaliser, mass_j = mean over (row, head) of
      sum over the slot's rows t of exp(sm_scale q . k_t - lse), lse the
      step's decode log-sum-exp; for a selected chunk this is its share of
      the step's attention.  The new selection is the top-K of
      s'_j = fl32(s_j + fl32(lambda * mass_j)), s_j = fl32(s_I + s_P), with
      the ranking rules of R3; lambda = 0 keeps the static selection.
  R6  The chunk scores come from the model's logits: s_I is the
      log-likelihood of the query-window tokens and s_P that of the
      pseudo-labels, each conditioned on the chunk -- the sum over the
      labelled rows of log softmax(logits)[label].  s_I is the negated NLL
      of the pages, so that both are "higher = more relevant" (R3).

Inputs are float64 arrays (bf16 tensors widened exactly) and int arrays.
All arithmetic is fp64 with numpy's matmul/exp/log; nothing is blocked,
fused or reordered beyond the definitions.
"""
from __future__ import annotations

import math

import numpy as np


class MacCounter:
    """Counts multiply-accumulates of the attention matmuls the oracle runs."""

    def __init__(self) -> None:
        self.macs = 0

    def add(self, m: int, n: int, k: int) -> None:
        self.macs += int(m) * int(n) * int(k)


def _count(counter, m, n, k):
    if counter is not None:
        counter.add(m, n, k)


def softmax_rows(x: np.ndarray) -> np.ndarray:
    """Row-wise softmax of fp64 logits (max-subtracted for range only)."""
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


# --------------------------------------------------------------- prefill --

def chunk_attention(q, k, v, n_chunks, chunk_size, sm_scale, counter=None):
    """[M1] Bidirectional attention inside each BOS-prefixed chunk.

    q: [N*(C+1), Hq, D]; k, v: [N*(C+1), Hkv, D]; query head h reads KV head
    h // (Hq/Hkv).  Chunk j owns rows j*(C+1) .. j*(C+1)+C (row 0 = BOS, R1)
    and sees no key outside itself.  Returns O: [N*(C+1), Hq, D] fp64.
    """
    rows = chunk_size + 1
    n_q_heads, head_dim = q.shape[1], q.shape[2]
    group = n_q_heads // k.shape[1]
    out = np.empty(q.shape, dtype=np.float64)
    for j in range(n_chunks):
        lo, hi = j * rows, (j + 1) * rows
        for h in range(n_q_heads):
            g = h // group
            logits = sm_scale * (q[lo:hi, h, :] @ k[lo:hi, g, :].T)
            p = softmax_rows(logits)
            out[lo:hi, h, :] = p @ v[lo:hi, g, :]
            _count(counter, rows, rows, head_dim)
            _count(counter, rows, rows, head_dim)
    return out


def chunk_attention_rows(q, k, v, chunk_size, rows, sm_scale):
    """[M1] The chunk-attention output at the listed prefix rows only.

    rows: global row indices into q.  Row r belongs to chunk r // (C+1) and
    attends to that chunk's C+1 rows, exactly as in chunk_attention; this
    evaluates the same definition at fewer rows, so that sampled rows of a
    large prefix can be checked.  Returns [len(rows), Hq, D] fp64.
    """
    span = chunk_size + 1
    n_q_heads, head_dim = q.shape[1], q.shape[2]
    group = n_q_heads // k.shape[1]
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    out = np.empty((len(rows), n_q_heads, head_dim), dtype=np.float64)
    chunk_of = rows // span
    for j in np.unique(chunk_of):
        at = np.nonzero(chunk_of == j)[0]      # positions in `rows` of chunk j's rows
        lo = int(j) * span
        for h in range(n_q_heads):
            g = h // group
            logits = sm_scale * (q[rows[at], h, :] @ k[lo:lo + span, g, :].T)
            out[at, h, :] = softmax_rows(logits) @ v[lo:lo + span, g, :]
    return out


def window_scores(q_win, k, n_chunks, chunk_size, sm_scale, counter=None):
    """[M2] + R2: cumulative attention weight each chunk row receives.

    For window row w and query head h the probabilities are the softmax of
    sm_scale * q_win[w, h] . k[t, g] over the chunk's own C+1 rows t; the
    score of row t is their sum over all W window rows and all Hq heads.
    q_win: [W, Hq, D].  Returns [N, C+1] fp64 (column 0 is BOS).
    """
    rows = chunk_size + 1
    n_win, n_q_heads, head_dim = q_win.shape
    group = n_q_heads // k.shape[1]
    scores = np.zeros((n_chunks, rows), dtype=np.float64)
    if n_win == 0:
        return scores
    for j in range(n_chunks):
        lo, hi = j * rows, (j + 1) * rows
        for h in range(n_q_heads):
            g = h // group
            logits = sm_scale * (q_win[:, h, :] @ k[lo:hi, g, :].T)  # [W, C+1]
            scores[j] += softmax_rows(logits).sum(axis=0)
            _count(counter, n_win, rows, head_dim)
    return scores


def window_scores_alt(q_win, k, n_chunks, chunk_size, sm_scale, per_kv_head=False, k_win=None):
    """[M2] under the two other readings of the ranking.

    per_kv_head: the column sums run over the query heads of each KV head
      separately (one token ranking per KV head); returns [N, Hkv, C+1].
    k_win ([W, Hkv, D] or None): when given, each window row's softmax runs
      over the chunk's C+1 keys and the W window keys together; the scores
      are still the probabilities of the chunk's keys.
    Otherwise as window_scores (whose result is the sum over KV heads of the
    per-KV-head scores).
    """
    rows = chunk_size + 1
    n_win, n_q_heads, head_dim = q_win.shape
    n_kv = k.shape[1]
    group = n_q_heads // n_kv
    scores = np.zeros((n_chunks, n_kv, rows), dtype=np.float64)
    if n_win == 0:
        return scores if per_kv_head else scores.sum(axis=1)
    for j in range(n_chunks):
        lo, hi = j * rows, (j + 1) * rows
        for h in range(n_q_heads):
            g = h // group
            keys = k[lo:hi, g, :]
            if k_win is not None:
                keys = np.concatenate([keys, k_win[:, g, :]], axis=0)
            p = softmax_rows(sm_scale * (q_win[:, h, :] @ keys.T))
            scores[j, g] += p[:, :rows].sum(axis=0)
    return scores if per_kv_head else scores.sum(axis=1)


def _rank_key(value, index):
    """R3: descending value, NaN last, ties to the lower index, -0 == +0."""
    value = float(value)
    if math.isnan(value):
        return (1, 0.0, index)
    return (0, -value, index)


def top_b(scores, n_keep):
    """[M2] + R1 + R3: the n_keep best content tokens of every chunk.

    scores: [N, C+1] (column 0 = BOS, never ranked).  Ranking uses the fp32
    rounding of each score.  Returns kept: [N, n_keep] int32, each row in
    ascending order of the in-chunk content index 0..C-1 (content index t
    is chunk row t+1).
    """
    n_chunks, rows = scores.shape
    content = scores[:, 1:].astype(np.float32)
    kept = np.empty((n_chunks, n_keep), dtype=np.int32)
    for j in range(n_chunks):
        order = sorted(range(rows - 1), key=lambda t: _rank_key(content[j, t], t))
        kept[j] = sorted(order[:n_keep])
    return kept


def compact(k, v, kept, slot_row, chunk_size, pool_k, pool_v):
    """[M1]/[M2] + R1: copy BOS and the kept rows of every chunk to its slot.

    Chunk j's slot starts at pool row slot_row[j] and holds, in order, the BOS
    row and the kept rows in ascending order (all heads of a row together).
    pool_k / pool_v ([pool_rows, Hkv, D]) are written in place.  Returns the
    chunk table [N, 2] int32 of (first pool row, length = n_keep + 1).
    """
    rows = chunk_size + 1
    n_chunks, n_keep = kept.shape
    table = np.empty((n_chunks, 2), dtype=np.int32)
    for j in range(n_chunks):
        src = [j * rows] + [j * rows + 1 + int(t) for t in kept[j]]
        base = int(slot_row[j])
        pool_k[base:base + n_keep + 1] = k[src]
        pool_v[base:base + n_keep + 1] = v[src]
        table[j] = (base, n_keep + 1)
    return table


def top_b_per_head(scores, n_keep):
    """[M2] per-KV-head reading: top_b applied to every (chunk, KV head)
    score row of scores [N, Hkv, C+1]; returns kept [N, Hkv, n_keep]."""
    n_chunks, n_kv, rows = scores.shape
    return top_b(scores.reshape(n_chunks * n_kv, rows), n_keep).reshape(n_chunks, n_kv, n_keep)


def compact_per_head(k, v, kept, slot_row, chunk_size, pool_k, pool_v):
    """[M1]/[M2] per-KV-head reading: KV head g of chunk j's slot holds, in
    order, head g of the BOS row and of head g's kept rows (ascending).
    kept: [N, Hkv, B].  Returns the chunk table as compact does."""
    rows = chunk_size + 1
    n_chunks, n_kv, n_keep = kept.shape
    table = np.empty((n_chunks, 2), dtype=np.int32)
    for j in range(n_chunks):
        base = int(slot_row[j])
        for g in range(n_kv):
            src = [j * rows] + [j * rows + 1 + int(t) for t in kept[j, g]]
            pool_k[base:base + n_keep + 1, g] = k[src, g]
            pool_v[base:base + n_keep + 1, g] = v[src, g]
        table[j] = (base, n_keep + 1)
    return table


def chunk_prefill_layers(q, k, v, q_win, n_chunks, chunk_size, n_keep, slot_row, pool_rows,
                         sm_scale):
    """[M1] over L layers: every layer caches the KV of its own chunks, so
    layer l is the single-layer prefill (chunk_attention, window_scores,
    top_b, compact) of its own tensors into its own pool.

    q, k, v: [L, N*(C+1), H, D]; q_win [L, W, Hq, D]; slot_row [N] (the same
    slots in every layer's pool of pool_rows rows).  Returns a list, one dict
    per layer, with out, scores, kept, pool_k, pool_v and table.
    """
    layers = []
    for l in range(q.shape[0]):
        out = chunk_attention(q[l], k[l], v[l], n_chunks, chunk_size, sm_scale)
        scores = window_scores(q_win[l], k[l], n_chunks, chunk_size, sm_scale)
        kept = top_b(scores, n_keep)
        pool_k = np.zeros((pool_rows,) + k.shape[2:])
        pool_v = np.zeros((pool_rows,) + v.shape[2:])
        table = compact(k[l], v[l], kept, slot_row, chunk_size, pool_k, pool_v)
        layers.append(dict(out=out, scores=scores, kept=kept, pool_k=pool_k, pool_v=pool_v,
                           table=table))
    return layers


def select_chunks(s_i, s_p, n_select):
    """[M1] + R3: the n_select chunks with the largest s = fl32(s_I + s_P).

    The add is one fp32 operation (round to nearest even).  Returns
    (sel [n_select] int32 in rank order, s [N] float32).
    """
    s = np.asarray(s_i, dtype=np.float32) + np.asarray(s_p, dtype=np.float32)
    order = sorted(range(s.shape[0]), key=lambda j: _rank_key(s[j], j))
    return np.array(order[:n_select], dtype=np.int32), s


# ---------------------------------------------------------------- decode --

def gather_selected(pool, table, sel):
    """Rows of the selected chunks' slots, concatenated in `sel` order."""
    parts = [pool[int(table[c, 0]):int(table[c, 0]) + int(table[c, 1])] for c in sel]
    if not parts:
        return pool[0:0]
    return np.concatenate(parts, axis=0)


def decode_attention(q, k_self, v_self, pool_k, pool_v, table, sel, sm_scale, counter=None):
    """[M2] + [M3] + R4: one softmax over selected-chunk rows and the live block.

    q: [Lq, Hq, D]; k_self, v_self: [Lq, Hkv, D].  The keys of every live
    row are the kept rows of the selected chunks followed by all Lq live rows.
    Returns (out [Lq, Hq, D], lse [Lq, Hq]) with lse in natural log.
    """
    keys_k = np.concatenate([gather_selected(pool_k, table, sel), k_self], axis=0)
    keys_v = np.concatenate([gather_selected(pool_v, table, sel), v_self], axis=0)
    n_live, n_q_heads, head_dim = q.shape
    group = n_q_heads // k_self.shape[1]
    out = np.empty(q.shape, dtype=np.float64)
    lse = np.empty((n_live, n_q_heads), dtype=np.float64)
    for h in range(n_q_heads):
        g = h // group
        logits = sm_scale * (q[:, h, :] @ keys_k[:, g, :].T)
        m = logits.max(axis=1, keepdims=True)
        e = np.exp(logits - m)
        denom = e.sum(axis=1, keepdims=True)
        out[:, h, :] = (e @ keys_v[:, g, :]) / denom
        lse[:, h] = m[:, 0] + np.log(denom[:, 0])
        _count(counter, n_live, keys_k.shape[0], head_dim)
        _count(counter, n_live, keys_k.shape[0], head_dim)
    return out, lse


def split_partials(q, keys_k, keys_v, group, sm_scale):
    """[AK] One split's partial softmax state: (m, l, acc) per row and head.

    m = max logit, l = sum exp(x - m), acc = sum exp(x - m) v over the
    split's keys only.  Shapes: m, l [Lq, Hq]; acc [Lq, Hq, D].
    """
    n_live, n_q_heads, head_dim = q.shape
    m = np.empty((n_live, n_q_heads))
    l = np.empty((n_live, n_q_heads))
    acc = np.empty((n_live, n_q_heads, head_dim))
    for h in range(n_q_heads):
        g = h // group
        logits = sm_scale * (q[:, h, :] @ keys_k[:, g, :].T)
        m[:, h] = logits.max(axis=1)
        e = np.exp(logits - m[:, h:h + 1])
        l[:, h] = e.sum(axis=1)
        acc[:, h, :] = e @ keys_v[:, g, :]
    return m, l, acc


def lse_merge(parts):
    """[AK] Log-sum-exp merge of split partials into (out, lse)."""
    m_all = np.stack([p[0] for p in parts])            # [S, Lq, Hq]
    big_m = m_all.max(axis=0)
    w = [np.exp(p[0] - big_m) for p in parts]
    big_l = sum(wi * p[1] for wi, p in zip(w, parts))
    acc = sum(wi[..., None] * p[2] for wi, p in zip(w, parts))
    return acc / big_l[..., None], big_m + np.log(big_l)


def decode_attention_split(q, k_self, v_self, pool_k, pool_v, table, sel, sm_scale):
    """[AK] Split per selected chunk plus one self-block split, LSE-merged."""
    group = q.shape[1] // k_self.shape[1]
    parts = []
    for c in sel:
        lo, n = int(table[c, 0]), int(table[c, 1])
        parts.append(split_partials(q, pool_k[lo:lo + n], pool_v[lo:lo + n], group, sm_scale))
    parts.append(split_partials(q, k_self, v_self, group, sm_scale))
    return lse_merge(parts)


# ---------------------------------------------------- reselection (R7) --

def chunk_mass(q, pool_k, table, chunks, lse, sm_scale):
    """R7: mean attention mass of each listed chunk at the normaliser lse.

    q: [Lq, Hq, D] live rows; pool_k [pool_rows, Hkv, D]; table [.., 2];
    chunks: table indices; lse [Lq, Hq] (natural log).  Returns [len(chunks)]
    fp64: sum over rows, heads and the chunk's slot rows of
    exp(sm_scale q . k - lse), divided by Lq * Hq.
    """
    n_live, n_q_heads, _ = q.shape
    group = n_q_heads // pool_k.shape[1]
    out = np.zeros(len(chunks))
    for i, c in enumerate(chunks):
        lo, n = int(table[c, 0]), int(table[c, 1])
        total = 0.0
        for h in range(n_q_heads):
            logits = sm_scale * (q[:, h, :] @ pool_k[lo:lo + n, h // group, :].T)   # [Lq, n]
            total += np.exp(logits - lse[:, h:h + 1]).sum()
        out[i] = total / (n_live * n_q_heads)
    return out


def reselect_chunks(s, mass, lam, n_select):
    """R7 + R3: the n_select chunks with the largest
    s' = fl32(fl32(s) + fl32(fl32(lam) * fl32(mass))) (two fp32 roundings,
    round to nearest even); returns (sel [n_select] in rank order, s' [N])."""
    s32 = np.asarray(s, dtype=np.float32)
    bonus = np.float32(lam) * np.asarray(mass, dtype=np.float32)
    s2 = (s32 + bonus.astype(np.float32)).astype(np.float32)
    order = sorted(range(s2.shape[0]), key=lambda j: _rank_key(s2[j], j))
    return np.array(order[:n_select], dtype=np.int32), s2


# ------------------------------------------------------- chunk scores --

def chunk_loglik(logits, labels):
    """[M1] + R6: summed label log-likelihood of every chunk.

    logits: [N, R, V] (the model's outputs at R labelled positions when
    conditioned on chunk j); labels: [R] ints in [0, V) (the query-window
    tokens for s_I, the pseudo-labels for s_P).  Row r's log-probability of
    its label is logits[j, r, y_r] - log(sum_v exp(logits[j, r, v])).
    Returns (score [N], rows [N, R]) in fp64.
    """
    z = np.asarray(logits, dtype=np.float64)
    y = np.asarray(labels, dtype=np.int64)
    m = z.max(axis=-1, keepdims=True)
    lse = m[..., 0] + np.log(np.exp(z - m).sum(axis=-1))
    picked = np.take_along_axis(z, y[None, :, None].repeat(z.shape[0], axis=0), axis=-1)[..., 0]
    rows = picked - lse
    return rows.sum(axis=1), rows


# ------------------------------------------------------ cost model [M3] --

def prefill_macs(n_chunks, chunk_size, n_win, n_q_heads, head_dim):
    """Closed form of the prefill attention MACs: QK^T and PV per chunk and
    head over C+1 rows, plus the window rows' QK^T for the scores."""
    rows = chunk_size + 1
    return 2 * n_q_heads * n_chunks * rows * rows * head_dim + n_q_heads * n_chunks * n_win * rows * head_dim


def decode_step_macs(n_live, kept_rows_total, n_q_heads, head_dim):
    """Closed form of one decode step's MACs: Lq rows against the selected
    chunks' kept rows plus the Lq live rows, QK^T and PV."""
    return 2 * n_q_heads * n_live * (kept_rows_total + n_live) * head_dim
