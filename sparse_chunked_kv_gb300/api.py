"""Tensor-level helpers over the C ABI: shape checks, output and workspace
allocation through torch, then one call into libpfd.  No arithmetic of the
method happens here.
"""
from __future__ import annotations

import torch

from . import _abi


def _need_cuda(*tensors):
    for t in tensors:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("expected contiguous CUDA tensors")


def chunk_prefill(q, k, v, q_win, n_chunks, chunk_size, n_keep, slot_row, pool_rows,
                  sm_scale=0.0, pool_k=None, pool_v=None, out=None, stream=None):
    """Chunked prefill of one request (pfd_chunk_prefill).  Returns a dict with
    out, scores, kept_idx, pool_k, pool_v, table ([N, 2] int32) and dev_err."""
    _need_cuda(q, k, v, q_win, slot_row)
    rows, hq, d = q.shape
    hkv = k.shape[1]
    w = 0 if q_win is None else q_win.shape[0]
    dev = q.device
    if out is None:
        out = torch.empty_like(q)
    if pool_k is None:
        pool_k = torch.zeros(pool_rows, hkv, d, dtype=torch.bfloat16, device=dev)
    if pool_v is None:
        pool_v = torch.zeros(pool_rows, hkv, d, dtype=torch.bfloat16, device=dev)
    scores = torch.empty(n_chunks, chunk_size + 1, dtype=torch.float32, device=dev)
    kept = torch.empty(n_chunks, max(n_keep, 1), dtype=torch.int32, device=dev)
    table = torch.empty(n_chunks, 2, dtype=torch.int32, device=dev)
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = _abi.pfd_chunk_prefill_workspace(n_chunks, chunk_size, w, hq, hkv, d, n_keep)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _abi.pfd_chunk_prefill(q, k, v, q_win if w > 0 else None, n_chunks, chunk_size, w, hq, hkv, d,
                           n_keep, sm_scale, out, scores, kept, pool_k, pool_v, pool_rows,
                           slot_row, table, dev_err, ws, ws_bytes, stream)
    return dict(out=out, scores=scores, kept_idx=kept[:, :n_keep], pool_k=pool_k, pool_v=pool_v,
                table=table, dev_err=dev_err, workspace=ws)


def chunk_prefill_ex(q, k, v, q_win, k_win, n_chunks, chunk_size, n_keep, slot_row, pool_rows,
                     per_kv_head=False, sm_scale=0.0, pool_k=None, pool_v=None, stream=None):
    """pfd_chunk_prefill_ex: the prefill under the other ranking readings
    (per_kv_head; window keys k_win in the denominator).  Returns the dict of
    chunk_prefill, with scores [N, Hkv, C+1] and kept_idx [N, Hkv, B] per
    KV head."""
    _need_cuda(q, k, v, q_win, k_win, slot_row)
    rows, hq, d = q.shape
    hkv = k.shape[1]
    w = q_win.shape[0]
    dev = q.device
    out = torch.empty_like(q)
    if pool_k is None:
        pool_k = torch.zeros(pool_rows, hkv, d, dtype=torch.bfloat16, device=dev)
    if pool_v is None:
        pool_v = torch.zeros(pool_rows, hkv, d, dtype=torch.bfloat16, device=dev)
    per = hkv if per_kv_head else 1
    scores = torch.empty(n_chunks * per, chunk_size + 1, dtype=torch.float32, device=dev)
    kept = torch.empty(n_chunks * per, max(n_keep, 1), dtype=torch.int32, device=dev)
    table = torch.empty(n_chunks, 2, dtype=torch.int32, device=dev)
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = _abi.pfd_chunk_prefill_workspace(n_chunks, chunk_size, w, hq, hkv, d, n_keep)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _abi.pfd_chunk_prefill_ex(q, k, v, q_win, k_win, n_chunks, chunk_size, w, hq, hkv, d, n_keep,
                              sm_scale, int(per_kv_head), out, scores, kept, pool_k, pool_v,
                              pool_rows, slot_row, table, dev_err, ws, ws_bytes, stream)
    if per_kv_head:
        scores = scores.view(n_chunks, hkv, chunk_size + 1)
        kept = kept.view(n_chunks, hkv, -1)
    return dict(out=out, scores=scores, kept_idx=kept[..., :n_keep], pool_k=pool_k,
                pool_v=pool_v, table=table, dev_err=dev_err, workspace=ws)


def chunk_prefill_layers(q, k, v, q_win, n_chunks, chunk_size, n_keep, slot_row, pool_rows,
                         sm_scale=0.0, stream=None):
    """pfd_chunk_prefill_layers: L layers' prefill in one call.  q, k, v:
    [L, N*(C+1), H, D]; q_win [L, W, Hq, D].  Returns a dict with out,
    scores [L, N, C+1], kept_idx [L, N, B], pool_k / pool_v
    [L, pool_rows, Hkv, D], table [L, N, 2] and dev_err."""
    _need_cuda(q, k, v, q_win, slot_row)
    n_layers, rows, hq, d = q.shape
    hkv = k.shape[2]
    w = q_win.shape[1]
    dev = q.device
    out = torch.empty_like(q)
    pool_k = torch.zeros(n_layers, pool_rows, hkv, d, dtype=torch.bfloat16, device=dev)
    pool_v = torch.zeros_like(pool_k)
    scores = torch.empty(n_layers, n_chunks, chunk_size + 1, dtype=torch.float32, device=dev)
    kept = torch.empty(n_layers, n_chunks, max(n_keep, 1), dtype=torch.int32, device=dev)
    table = torch.empty(n_layers, n_chunks, 2, dtype=torch.int32, device=dev)
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = _abi.pfd_chunk_prefill_layers_workspace(n_layers, n_chunks, chunk_size, w, hq, hkv,
                                                       d, n_keep)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _abi.pfd_chunk_prefill_layers(q, k, v, q_win if w > 0 else None, n_layers, n_chunks,
                                  chunk_size, w, hq, hkv, d, n_keep, sm_scale, out, scores, kept,
                                  pool_k, pool_v, pool_rows, slot_row, table, dev_err, ws,
                                  ws_bytes, stream)
    return dict(out=out, scores=scores, kept_idx=kept[..., :n_keep], pool_k=pool_k,
                pool_v=pool_v, table=table, dev_err=dev_err, workspace=ws)


def chunk_prefill_batch(q, k, v, q_win, n_chunks, chunk_size, n_keep, slot_row, pool_k, pool_v,
                        table, sm_scale=0.0, stream=None):
    """pfd_chunk_prefill_batch: L same-shaped requests' prefill in one call,
    their slots in one shared pool.  q, k, v: [L, N*(C+1), H, D]; q_win
    [L, W, Hq, D]; slot_row [L, N] absolute pool rows; pool_k / pool_v
    [pool_rows, Hkv, D] and table [L, N, 2] are written in place.  Returns a
    dict with out, scores [L, N, C+1], kept_idx [L, N, B] and dev_err."""
    _need_cuda(q, k, v, q_win, slot_row, pool_k, pool_v, table)
    n_req, rows, hq, d = q.shape
    hkv = k.shape[2]
    w = q_win.shape[1]
    dev = q.device
    out = torch.empty_like(q)
    scores = torch.empty(n_req, n_chunks, chunk_size + 1, dtype=torch.float32, device=dev)
    kept = torch.empty(n_req, n_chunks, max(n_keep, 1), dtype=torch.int32, device=dev)
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = _abi.pfd_chunk_prefill_layers_workspace(n_req, n_chunks, chunk_size, w, hq, hkv, d,
                                                       n_keep)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _abi.pfd_chunk_prefill_batch(q, k, v, q_win if w > 0 else None, n_req, n_chunks, chunk_size,
                                 w, hq, hkv, d, n_keep, sm_scale, out, scores, kept, pool_k,
                                 pool_v, pool_k.shape[0], slot_row, table, dev_err, ws, ws_bytes,
                                 stream)
    return dict(out=out, scores=scores, kept_idx=kept[..., :n_keep], dev_err=dev_err, workspace=ws)


def select_chunks(s_i, s_p, n_select, stream=None):
    """Top-K chunk selection (pfd_select_chunks).  Returns (sel, s)."""
    _need_cuda(s_i, s_p)
    n = s_i.shape[0]
    sel = torch.empty(n_select, dtype=torch.int32, device=s_i.device)
    s = torch.empty(n, dtype=torch.float32, device=s_i.device)
    _abi.pfd_select_chunks(s_i, s_p, n, n_select, sel, s, stream)
    return sel, s


def select_chunks_batched(s_i, s_p, cu_n, cu_k, max_n, stream=None):
    """Batched selection (pfd_select_chunks_batched); sel holds table indices."""
    _need_cuda(s_i, s_p, cu_n, cu_k)
    batch = cu_n.shape[0] - 1
    total_k = int(cu_k[-1].item())
    sel = torch.empty(max(total_k, 1), dtype=torch.int32, device=s_i.device)
    s = torch.empty_like(s_i)
    _abi.pfd_select_chunks_batched(s_i, s_p, cu_n, cu_k, batch, max_n, sel, s, stream)
    return sel[:total_k], s


def decode_attention(q, k_self, v_self, pool_k, pool_v, table, sel, cu_lq=None, cu_k=None,
                     sm_scale=0.0, n_splits=0, max_chunk_len=None, out=None, lse=None,
                     dev_err=None, workspace=None, stream=None):
    """Static-KV decode attention of one step (pfd_decode_attention).

    Single sequence when cu_lq / cu_k are None.  cu_lq, cu_k may be CPU
    int32 tensors (copied to the device) or pairs (device, host list).
    Returns (out, lse)."""
    _need_cuda(q, k_self, v_self, pool_k, pool_v, table, sel)
    dev = q.device
    total_lq, hq, d = q.shape
    hkv = k_self.shape[1]
    if cu_lq is None:
        cu_lq_host, cu_k_host = [0, total_lq], [0, sel.shape[0]]
    else:
        cu_lq_host, cu_k_host = [int(x) for x in cu_lq], [int(x) for x in cu_k]
    batch = len(cu_lq_host) - 1
    cu_lq_dev = torch.tensor(cu_lq_host, dtype=torch.int32).to(dev, non_blocking=True)
    cu_k_dev = torch.tensor(cu_k_host, dtype=torch.int32).to(dev, non_blocking=True)
    if max_chunk_len is None:
        max_chunk_len = int(table[:, 1].max().item()) if table.shape[0] > 0 else 0
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(total_lq, hq, dtype=torch.float32, device=dev)
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = _abi.pfd_decode_workspace(batch, cu_lq_host, cu_k_host, hq, hkv, d, max_chunk_len,
                                         n_splits)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _abi.pfd_decode_attention(q, k_self, v_self, cu_lq_dev, cu_lq_host, pool_k, pool_v,
                              pool_k.shape[0], table, table.shape[0], sel, cu_k_dev, cu_k_host,
                              batch, hq, hkv, d, max_chunk_len, sm_scale, n_splits, out, lse,
                              dev_err, workspace, ws_bytes, stream)
    return out, lse


def decode_partial(q, k_self, v_self, pool_k, pool_v, table, sel, cu_lq, cu_k, self_keys,
                   sm_scale=0.0, n_splits=0, max_chunk_len=None, part_o=None, part_lse=None,
                   dev_err=None, stream=None):
    """One device's share of a decode step (pfd_decode_partial): the partial
    state over the given selected chunks, plus the live block's keys when
    self_keys.  cu_lq, cu_k: host lists.  Returns (part_o, part_lse)."""
    _need_cuda(q, k_self, v_self, pool_k, pool_v, table)
    dev = q.device
    total_lq, hq, d = q.shape
    hkv = k_self.shape[1]
    cu_lq_host, cu_k_host = [int(x) for x in cu_lq], [int(x) for x in cu_k]
    batch = len(cu_lq_host) - 1
    cu_lq_dev = torch.tensor(cu_lq_host, dtype=torch.int32).to(dev)
    cu_k_dev = torch.tensor(cu_k_host, dtype=torch.int32).to(dev)
    if sel is None or sel.numel() == 0:
        sel = torch.zeros(1, dtype=torch.int32, device=dev)
    if max_chunk_len is None:
        max_chunk_len = int(table[:, 1].max().item()) if table.shape[0] > 0 else 0
    if part_o is None:
        part_o = torch.empty_like(q)
    if part_lse is None:
        part_lse = torch.empty(total_lq, hq, dtype=torch.float32, device=dev)
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = _abi.pfd_decode_partial_workspace(batch, cu_lq_host, cu_k_host, hq, hkv, d,
                                                 max_chunk_len, self_keys, n_splits)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _abi.pfd_decode_partial(q, k_self, v_self, cu_lq_dev, cu_lq_host, pool_k, pool_v,
                            pool_k.shape[0], table, table.shape[0], sel, cu_k_dev, cu_k_host,
                            batch, hq, hkv, d, max_chunk_len, sm_scale, self_keys, n_splits,
                            part_o, part_lse, dev_err, ws, ws_bytes, stream)
    return part_o, part_lse


def lse_merge(part_o, part_lse, out=None, lse=None, stream=None):
    """Log-sum-exp merge of stacked partials (pfd_lse_merge):
    part_o [S, rows, Hq, D], part_lse [S, rows, Hq].  Returns (out, lse)."""
    _need_cuda(part_o, part_lse)
    s, rows, hq, d = part_o.shape
    if out is None:
        out = torch.empty(rows, hq, d, dtype=part_o.dtype, device=part_o.device)
    if lse is None:
        lse = torch.empty(rows, hq, dtype=torch.float32, device=part_o.device)
    _abi.pfd_lse_merge(part_o, part_lse, s, rows, hq, d, out, lse, stream)
    return out, lse


def chunk_loglik(logits, labels, row_ll=None, score=None, dev_err=None, stream=None):
    """Summed label log-likelihood per chunk (pfd_chunk_loglik): logits
    [N, R, V] bf16, labels [R] int32.  Returns (score [N], row_ll [N, R],
    dev_err)."""
    _need_cuda(logits, labels)
    n, r, v = logits.shape
    dev = logits.device
    if row_ll is None:
        row_ll = torch.empty(n, r, dtype=torch.float32, device=dev)
    if score is None:
        score = torch.empty(n, dtype=torch.float32, device=dev)
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    _abi.pfd_chunk_loglik(logits, labels, n, r, v, row_ll, score, dev_err, stream)
    return score, row_ll, dev_err


def chunk_mass(q, pool_k, table, lse, cu_lq, cu_n, sm_scale=0.0, mass=None, dev_err=None,
               stream=None):
    """Attention mass of every chunk at the step's normaliser (pfd_chunk_mass).
    cu_lq, cu_n: host lists.  Returns (mass [table_len], dev_err)."""
    _need_cuda(q, pool_k, table, lse)
    dev = q.device
    total_lq, hq, d = q.shape
    hkv = pool_k.shape[1]
    cu_lq_host, cu_n_host = [int(x) for x in cu_lq], [int(x) for x in cu_n]
    batch = len(cu_lq_host) - 1
    cu_lq_dev = torch.tensor(cu_lq_host, dtype=torch.int32).to(dev)
    if mass is None:
        mass = torch.zeros(table.shape[0], dtype=torch.float32, device=dev)
    if dev_err is None:
        dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_bytes = _abi.pfd_chunk_mass_workspace(batch, cu_lq_host, cu_n_host, hq, hkv)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    _abi.pfd_chunk_mass(q, cu_lq_dev, cu_lq_host, pool_k, pool_k.shape[0], table, table.shape[0],
                        cu_n_host, lse, batch, hq, hkv, d, sm_scale, mass, dev_err, ws, ws_bytes,
                        stream)
    return mass, dev_err


def reselect_chunks(s, mass, lam, cu_n, cu_k, max_n, stream=None):
    """New selection from s + lambda * mass (pfd_reselect_chunks).  cu_n, cu_k:
    device int32.  Returns (sel, s')."""
    _need_cuda(s, mass, cu_n, cu_k)
    batch = cu_n.shape[0] - 1
    total_k = int(cu_k[-1].item())
    sel = torch.empty(max(total_k, 1), dtype=torch.int32, device=s.device)
    s2 = torch.empty_like(s)
    _abi.pfd_reselect_chunks(s, mass, lam, cu_n, cu_k, batch, max_n, sel, s2, stream)
    return sel[:total_k], s2
