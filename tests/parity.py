"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the CPU oracle on the same seeded inputs, and compare with the stated
tolerances:
  - chunk selection and pool bytes: bit-exact;
  - kept token indices: bit-exact except for tokens whose oracle score lies
    within 1e-5 (relative) of the chunk's B-th largest score;
  - attention outputs (bf16 in, fp32 accumulate): max-abs 2e-2, mean-abs 2e-3;
  - decode lse: max-abs 1e-3;
  - window scores: |gpu - oracle| <= 1e-4 * |oracle| + 1e-6 * W * Hq per
    element (score_tol).  A score is an fp32 sum of W*Hq probabilities, each
    carrying about 1e-6 of relative error from the fp32 exponent and
    normaliser, so the absolute term grows with the number of terms: at
    W = 64, Hq = 28 it is 1.8e-3, against scores of order 1..100.  The kept
    indices stay bit-exact outside the 1e-5 tie band whatever this
    tolerance is.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import pfd_oracle as orc
from sparse_chunked_kv_gb300 import api
from sparse_chunked_kv_gb300 import workloads as wl

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3
TIE_REL = 1e-5
SCORE_RTOL = 1e-4
SCORE_ATOL_PER_TERM = 1e-6


def score_tol(ref, n_win, n_q_heads):
    """Per-element tolerance of the fp32 window scores against the oracle."""
    return SCORE_RTOL * np.abs(ref) + SCORE_ATOL_PER_TERM * max(1, n_win * n_q_heads)

f64 = wl.to_f64


def cuda(t):
    return t.to("cuda", non_blocking=False).contiguous()


def assert_close_out(got, want, what):
    err = np.abs(np.asarray(got, dtype=np.float64) - want)
    assert np.isfinite(err).all(), f"{what}: non-finite values"
    assert err.max() <= OUT_MAX_ABS, f"{what}: max-abs {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def check_kept(gpu_kept, ref_scores, n_keep):
    """gpu_kept [N, B] vs the oracle's top-B, allowing swaps inside the tie band."""
    ref_kept = orc.top_b(ref_scores, n_keep)
    content = ref_scores[:, 1:]
    c32 = content.astype(np.float32)
    n_diff = 0
    for j in range(gpu_kept.shape[0]):
        g = [int(x) for x in gpu_kept[j]]
        assert g == sorted(g) and len(set(g)) == n_keep, f"chunk {j}: kept list not ascending/unique"
        assert all(0 <= x < content.shape[1] for x in g)
        diff = set(g) ^ set(int(x) for x in ref_kept[j])
        if diff:
            bth = float(np.sort(c32[j])[::-1][n_keep - 1])
            for t in diff:
                assert abs(content[j, t] - bth) <= TIE_REL * abs(bth), (
                    f"chunk {j}: token {t} score {content[j, t]!r} outside the tie band of {bth!r}")
            n_diff += 1
    return ref_kept, n_diff


def run_prefill(cfg, req, pool_pad=0, pool_fill=0.0, chunks=None):
    """GPU prefill; returns dict of CPU results.  pool_pad extra rows per slot
    are filled with pool_fill (e.g. NaN) and must stay untouched."""
    stride = cfg.n_keep + 1 + pool_pad
    slot = (req["slot_row"] // cfg.slot_stride) * stride
    pool_rows = cfg.n_chunks * stride
    pk = torch.full((pool_rows, cfg.n_kv_heads, cfg.head_dim), pool_fill, dtype=torch.bfloat16,
                    device="cuda")
    pv = pk.clone()
    res = api.chunk_prefill(cuda(req["q"]), cuda(req["k"]), cuda(req["v"]),
                            cuda(req["q_win"]) if cfg.n_win > 0 else None, cfg.n_chunks,
                            cfg.chunk_size, cfg.n_keep, cuda(slot.to(torch.int32)), pool_rows,
                            pool_k=pk, pool_v=pv)
    torch.cuda.synchronize()
    out = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in res.items() if k != "workspace"}
    out["slot_row"] = slot.to(torch.int32)
    out["pool_rows"] = pool_rows
    out["pool_k_dev"] = res["pool_k"]
    out["pool_v_dev"] = res["pool_v"]
    out["table_dev"] = res["table"]
    return out


def check_pool(cfg, req, res):
    """Pool slots hold BOS + the GPU's kept rows, bit for bit; table matches."""
    rows = cfg.chunk_size + 1
    kept = res["kept_idx"].long()
    table = res["table"]
    k, v = req["k"], req["v"]
    for j in range(cfg.n_chunks):
        base = int(res["slot_row"][j])
        assert table[j].tolist() == [base, cfg.n_keep + 1]
        src = torch.cat([torch.tensor([j * rows]), j * rows + 1 + kept[j]])
        assert torch.equal(res["pool_k"][base:base + cfg.n_keep + 1].view(torch.int16),
                           k[src].view(torch.int16)), f"pool_k slot of chunk {j}"
        assert torch.equal(res["pool_v"][base:base + cfg.n_keep + 1].view(torch.int16),
                           v[src].view(torch.int16)), f"pool_v slot of chunk {j}"


def oracle_pool(cfg, req, kept, slot_row, pool_rows, fill=0.0):
    pk = np.full((pool_rows, cfg.n_kv_heads, cfg.head_dim), fill)
    pv = np.full((pool_rows, cfg.n_kv_heads, cfg.head_dim), fill)
    table = orc.compact(f64(req["k"]), f64(req["v"]), kept, slot_row.numpy(), cfg.chunk_size, pk, pv)
    return pk, pv, table


def bf16_of(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)
