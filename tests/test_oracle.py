"""CPU tests: the oracle against its pins, and planted mistakes against the pins."""
import numpy as np
import pytest

from oracle import pfd_oracle as orc
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(orc)


class Mutant:
    """The oracle with some functions replaced by broken versions."""

    def __init__(self, **overrides):
        self.__dict__.update(overrides)

    def __getattr__(self, name):
        return getattr(orc, name)


def _chunk_attention_global(q, k, v, n, c, scale, counter=None):
    # mistake: attends across chunk boundaries (no block-diagonal mask)
    out = np.empty(q.shape)
    g = q.shape[1] // k.shape[1]
    for h in range(q.shape[1]):
        p = orc.softmax_rows(scale * q[:, h] @ k[:, h // g].T)
        out[:, h] = p @ v[:, h // g]
    return out


def _chunk_attention_bad_gqa(q, k, v, n, c, scale, counter=None):
    # mistake: query head h reads KV head h % Hkv instead of h // G
    hkv = k.shape[1]
    out = np.empty(q.shape)
    rows = c + 1
    for j in range(n):
        sl = slice(j * rows, (j + 1) * rows)
        for h in range(q.shape[1]):
            p = orc.softmax_rows(scale * q[sl, h] @ k[sl, h % hkv].T)
            out[sl, h] = p @ v[sl, h % hkv]
    return out


def _scores_wrong_axis(q_win, k, n, c, scale, counter=None):
    # mistake: normalises over the window rows instead of over the keys
    rows = c + 1
    g = q_win.shape[1] // k.shape[1]
    out = np.zeros((n, rows))
    for j in range(n):
        for h in range(q_win.shape[1]):
            x = scale * q_win[:, h] @ k[j * rows:(j + 1) * rows, h // g].T
            out[j] += orc.softmax_rows(x.T).T.sum(axis=0)
    return out


def _scores_no_scale(q_win, k, n, c, scale, counter=None):
    return orc.window_scores(q_win, k, n, c, 1.0)


def _scores_drops_last_head(q_win, k, n, c, scale, counter=None):
    # mistake: the sum over query heads stops one head short
    rows = c + 1
    g = q_win.shape[1] // k.shape[1]
    out = np.zeros((n, rows))
    for j in range(n):
        for h in range(q_win.shape[1] - 1):
            x = scale * q_win[:, h] @ k[j * rows:(j + 1) * rows, h // g].T
            out[j] += orc.softmax_rows(x).sum(axis=0)
    return out


def _top_b_high_index_ties(scores, n_keep):
    content = scores[:, 1:].astype(np.float32)
    kept = np.empty((scores.shape[0], n_keep), np.int32)
    for j in range(scores.shape[0]):
        order = sorted(range(content.shape[1]), key=lambda t: (-float(content[j, t]), -t))
        kept[j] = sorted(order[:n_keep])
    return kept


def _top_b_with_bos(scores, n_keep):
    kept = np.empty((scores.shape[0], n_keep), np.int32)
    for j in range(scores.shape[0]):
        order = sorted(range(scores.shape[1]), key=lambda t: (-float(np.float32(scores[j, t])), t))
        kept[j] = sorted(order[:n_keep])
    return kept


def _select_fp64(s_i, s_p, n_select):
    s = s_i.astype(np.float64) + s_p.astype(np.float64)
    order = sorted(range(s.shape[0]), key=lambda j: (-s[j], j))
    return np.array(order[:n_select], np.int32), s.astype(np.float32)


def _decode_no_self(q, ks, vs, pk, pv, table, sel, scale, counter=None):
    return orc.decode_attention(q, ks[:0], vs[:0], pk, pv, table, sel, scale)


def _decode_split_no_rescale(q, ks, vs, pk, pv, table, sel, scale):
    group = q.shape[1] // ks.shape[1]
    parts = [orc.split_partials(q, pk[t[0]:t[0] + t[1]], pv[t[0]:t[0] + t[1]], group, scale)
             for t in (table[c] for c in sel)]
    parts.append(orc.split_partials(q, ks, vs, group, scale))
    l = sum(p[1] for p in parts)
    acc = sum(p[2] for p in parts)
    return acc / l[..., None], np.log(l)


def _lse_merge_drops_max(parts):
    # mistake: weighs each split by its denominator alone, ignoring its max
    big_l = sum(p[1] for p in parts)
    acc = sum(p[1][..., None] * (p[2] / p[1][..., None]) for p in parts)
    m_all = np.stack([p[0] for p in parts]).max(axis=0)
    return acc / big_l[..., None], m_all + np.log(big_l)


def _loglik_no_max_shift(logits, labels):
    # mistake: picks the label logit but normalises with the max only
    z = np.asarray(logits, dtype=np.float64)
    y = np.asarray(labels)
    rows = np.take_along_axis(z, y[None, :, None].repeat(z.shape[0], 0), -1)[..., 0] - z.max(-1)
    return rows.sum(1), rows


def _loglik_wrong_label_axis(logits, labels):
    # mistake: gathers the label along the row axis instead of the vocabulary
    z = np.asarray(logits, dtype=np.float64)
    lse = np.log(np.exp(z).sum(-1))
    idx = np.minimum(np.asarray(labels), z.shape[1] - 1)
    rows = z[:, idx, 0] - lse
    return rows.sum(1), rows


def _scores_alt_window_keys_ignored(q_win, k, n, c, scale, per_kv_head=False, k_win=None):
    # mistake: drops the window keys from the denominator
    return orc.window_scores_alt(q_win, k, n, c, scale, per_kv_head=per_kv_head, k_win=None)


def _compact_per_head_shared_rows(k, v, kept, slot_row, c, pk, pv):
    # mistake: copies every head's rows from KV head 0's kept set
    return orc.compact_per_head(k, v, np.repeat(kept[:, :1], kept.shape[1], axis=1), slot_row, c,
                                pk, pv)


def _mass_without_normaliser(q, pool_k, table, chunks, lse, scale):
    # mistake: forgets to subtract the step's log-sum-exp
    return orc.chunk_mass(q, pool_k, table, chunks, np.zeros_like(lse), scale)


def _reselect_single_rounding(s, mass, lam, n_select):
    # mistake: s + lambda * mass in fp64 (one rounding at the end)
    s2 = (np.asarray(s, np.float64) + lam * np.asarray(mass, np.float64)).astype(np.float32)
    order = sorted(range(len(s2)), key=lambda j: orc._rank_key(s2[j], j))
    return np.array(order[:n_select], np.int32), s2


def _compact_without_bos(k, v, kept, slot_row, c, pool_k, pool_v):
    rows = c + 1
    n_chunks, n_keep = kept.shape
    table = np.empty((n_chunks, 2), dtype=np.int32)
    for j in range(n_chunks):
        src = [j * rows + 1 + int(t) for t in kept[j]]
        base = int(slot_row[j])
        pool_k[base:base + n_keep] = k[src]
        pool_v[base:base + n_keep] = v[src]
        table[j] = (base, n_keep)
    return table


def _scores_without_bos_key(q_win, k, n, c, scale, counter=None):
    rows = c + 1
    keep = np.ones(k.shape[0], dtype=bool)
    keep[::rows] = False
    s = np.zeros((n, rows))
    s[:, 1:] = orc.window_scores(q_win, k[keep], n, c - 1, scale)
    return s


def _layers_share_window_rows(q, k, v, q_win, n, c, b, slot, pool_rows, scale):
    return orc.chunk_prefill_layers(q, k, v, np.repeat(q_win[:1], q_win.shape[0], axis=0), n, c, b,
                                    slot, pool_rows, scale)


def _layers_share_one_pool(q, k, v, q_win, n, c, b, slot, pool_rows, scale):
    layers = orc.chunk_prefill_layers(q, k, v, q_win, n, c, b, slot, pool_rows, scale)
    for lay in layers:                      # every layer compacted into layer 0's pool
        lay["pool_k"], lay["pool_v"] = layers[0]["pool_k"], layers[0]["pool_v"]
    return layers


def _select_tie_high_index(s_i, s_p, n_select):
    s = np.asarray(s_i, np.float32) + np.asarray(s_p, np.float32)
    order = sorted(range(len(s)), key=lambda j: (-float(s[j]), -j))
    return np.array(order[:n_select], np.int32), s


def _mass_rows_only(q, pool_k, table, chunks, lse, scale):
    # averaged over the live rows but summed over the heads
    return orc.chunk_mass(q, pool_k, table, chunks, lse, scale) * q.shape[1]


def _scores_alt_wrong_group(q_win, k, n, c, scale, per_kv_head=False, k_win=None):
    # query head h read against KV head h % Hkv instead of h // G
    hq, hkv = q_win.shape[1], k.shape[1]
    perm = [h2 for g in range(hkv) for h2 in range(g, hq, hkv)]
    return orc.window_scores_alt(q_win[:, perm], k, n, c, scale, per_kv_head=per_kv_head,
                                 k_win=k_win)


MUTANTS = {
    "cross_chunk_attention": (Mutant(chunk_attention=_chunk_attention_global), pins.check_chunk_attention),
    "gqa_mapping": (Mutant(chunk_attention=_chunk_attention_bad_gqa), pins.check_chunk_attention),
    "scores_softmax_axis": (Mutant(window_scores=_scores_wrong_axis), pins.check_scores_vs_sdpa),
    "scores_scale_dropped": (Mutant(window_scores=_scores_no_scale), pins.check_scores_brute_force),
    "scores_one_head": (Mutant(window_scores=_scores_drops_last_head), pins.check_scores_vs_sdpa),
    "topb_tie_high_index": (Mutant(top_b=_top_b_high_index_ties), pins.check_top_b),
    "topb_ranks_bos": (Mutant(top_b=_top_b_with_bos), pins.check_top_b),
    "select_in_fp64": (Mutant(select_chunks=_select_fp64), pins.check_select),
    "decode_drops_self_block": (Mutant(decode_attention=_decode_no_self), pins.check_decode_vs_sdpa),
    "merge_without_rescale": (Mutant(decode_attention_split=_decode_split_no_rescale),
                              pins.check_split_equals_concat),
    "merge_drops_split_max": (Mutant(lse_merge=_lse_merge_drops_max),
                              pins.check_split_at_arbitrary_points),
    "loglik_normaliser_dropped": (Mutant(chunk_loglik=_loglik_no_max_shift),
                                  pins.check_loglik_vs_cross_entropy),
    "loglik_label_axis": (Mutant(chunk_loglik=_loglik_wrong_label_axis),
                          pins.check_loglik_closed_forms),
    "scores_window_keys_dropped": (Mutant(window_scores_alt=_scores_alt_window_keys_ignored),
                                   pins.check_scores_alt_readings),
    "per_head_compact_shared_rows": (Mutant(compact_per_head=_compact_per_head_shared_rows),
                                     pins.check_per_head_topb_and_compact),
    "mass_without_normaliser": (Mutant(chunk_mass=_mass_without_normaliser), pins.check_chunk_mass),
    "reselect_single_rounding": (Mutant(reselect_chunks=_reselect_single_rounding),
                                 pins.check_reselect),
    "compact_without_bos": (Mutant(compact=_compact_without_bos), pins.check_hand_worked_pipeline),
    "select_tie_high_index": (Mutant(select_chunks=_select_tie_high_index), pins.check_select),
    "mass_summed_over_heads": (Mutant(chunk_mass=_mass_rows_only), pins.check_chunk_mass),
    "alt_scores_wrong_kv_group": (Mutant(window_scores_alt=_scores_alt_wrong_group),
                                  pins.check_scores_alt_readings),
    "layers_share_window_rows": (Mutant(chunk_prefill_layers=_layers_share_window_rows),
                                 pins.check_layers_are_independent),
    "layers_share_one_pool": (Mutant(chunk_prefill_layers=_layers_share_one_pool),
                              pins.check_layers_are_independent),
    "scores_without_bos_key": (Mutant(window_scores=_scores_without_bos_key),
                               pins.check_hand_worked_pipeline),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    mutant, check = MUTANTS[name]
    with pytest.raises(AssertionError):
        check(mutant)
