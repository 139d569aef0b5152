"""Seeded synthetic workloads for the chunked prefill + static-KV decode path.

This module only draws inputs.  It holds none of the method's arithmetic and
is shared by the tests, the benchmark and the smoke check; both the CUDA path
and the CPU oracle are fed from what it returns.

Recipe (every tensor is drawn on the CPU from ``torch.Generator`` seeded
``1000 * config_id + seq``, in this fixed order):

  q, k, v        [N*(C+1), H, D]  fp32 N(0,1) -> bf16 (round to nearest even);
                 row j*(C+1) of chunk j is its BOS row, drawn like the rest.
  q_win          [W, Hq, D]       query-window rows (the "query tokens").
  k_win, v_win   [W, Hkv, D]      the window rows' keys/values in the live block.
  needle chunks  int              which chunks hold needles ("random": seeded
                                  choice; "uniform": chunk of a uniformly drawn
                                  prefix position; "spread": evenly spaced).
  needle rows    8 content rows per needle chunk, seeded positions; the key of
                 a needle row for KV head g is
                 0.5 * mean over (w, h in group g) of q_win[w, h] + N(0, 0.5^2).
  s_I, s_P       [N] fp32 N(0,1); s_I += 3 on needle chunks.
  slot order     identity, or a seeded permutation of the N pool slots.

The live block of decode step t is [q_win ; q_resp_t] (and the same for k, v):
the window rows are drawn once, the L_d response rows are redrawn every step
from a generator seeded ``1000 * config_id + seq + 7919 * (t + 1)``.
"""
from __future__ import annotations

import dataclasses
import math

import torch

NEEDLES_PER_CHUNK = 8


@dataclasses.dataclass(frozen=True)
class Config:
    """One attention layer of one request: N chunks of C tokens (+BOS)."""
    name: str
    config_id: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_chunks: int
    chunk_size: int
    n_keep: int          # B, kept content tokens per chunk
    n_select: int        # K, selected chunks
    n_win: int           # W, query-window rows
    n_resp: int          # L_d, response rows
    n_steps: int         # T, denoising steps
    pool_order: str = "identity"   # or "permuted"
    n_needle_chunks: int = 1
    needle_mode: str = "random"    # "random" | "uniform" | "spread"

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def rows(self) -> int:
        return self.n_chunks * (self.chunk_size + 1)

    @property
    def n_live(self) -> int:
        return self.n_win + self.n_resp

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def slot_stride(self) -> int:
        return self.n_keep + 1

    @property
    def pool_rows(self) -> int:
        return self.n_chunks * self.slot_stride


def _cfg(name, cid, hq, hkv, d, n, c, b, k, w, ld, t, **kw):
    return Config(name, cid, hq, hkv, d, n, c, b, k, w, ld, t, **kw)


# The five workloads: a tiny parity case and 8K / 32K / 128K prefixes with
# Dream-7B-like heads (28 query heads, 4 KV heads, D = 128).
TINY = _cfg("tiny", 0, 8, 2, 64, 8, 256, 64, 2, 32, 32, 4, n_needle_chunks=1, needle_mode="random")
CTX_8K = _cfg("8k", 1, 28, 4, 128, 16, 512, 256, 4, 64, 256, 64, n_needle_chunks=2, needle_mode="random")
CTX_32K = _cfg("32k", 2, 28, 4, 128, 32, 1024, 512, 8, 64, 256, 128, pool_order="permuted",
               n_needle_chunks=4, needle_mode="uniform")
CTX_128K = _cfg("128k", 3, 28, 4, 128, 512, 256, 128, 64, 64, 512, 64, n_needle_chunks=16,
                needle_mode="spread")


def mix_configs():
    """Batched serving mix: 8 sequences of a 32K prefix, C in {256, 1024, 4096}
    by sequence index mod 3, B = C/4, K = 8192 / C, W = 64, L_d = 256, T = 64."""
    out = []
    for i in range(8):
        c = (256, 1024, 4096)[i % 3]
        out.append(_cfg(f"mix{i}", 4, 28, 4, 128, 32768 // c, c, c // 4, 8192 // c, 64, 256, 64,
                        pool_order="permuted", n_needle_chunks=4, needle_mode="uniform"))
    return out


CONFIGS = {c.name: c for c in (TINY, CTX_8K, CTX_32K, CTX_128K)}


def scaled(cfg: Config, **changes) -> Config:
    """A copy of cfg with some sizes changed (for small parity cases)."""
    return dataclasses.replace(cfg, **changes)


def _bf16(gen, *shape):
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make_request(cfg: Config, seq: int = 0) -> dict:
    """Draws the prefix, the query window and the chunk scores of one request."""
    gen = torch.Generator().manual_seed(1000 * cfg.config_id + seq)
    hq, hkv, d, n, c = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_chunks, cfg.chunk_size
    rows = cfg.rows
    q = _bf16(gen, rows, hq, d)
    k = _bf16(gen, rows, hkv, d)
    v = _bf16(gen, rows, hkv, d)
    q_win = _bf16(gen, cfg.n_win, hq, d)
    k_win = _bf16(gen, cfg.n_win, hkv, d)
    v_win = _bf16(gen, cfg.n_win, hkv, d)

    n_needle = min(cfg.n_needle_chunks, n)
    if cfg.needle_mode == "spread":
        needle_chunks = sorted({int((i + 0.5) * n / n_needle) for i in range(n_needle)})
    elif cfg.needle_mode == "uniform":
        chosen = []
        while len(chosen) < n_needle:
            pos = int(torch.randint(0, n * c, (1,), generator=gen))
            if pos // c not in chosen:
                chosen.append(pos // c)
        needle_chunks = sorted(chosen)
    else:
        needle_chunks = sorted(torch.randperm(n, generator=gen)[:n_needle].tolist())
    needle_rows = []
    if cfg.n_win > 0:
        qw = q_win.float().reshape(cfg.n_win, hkv, cfg.group, d)
        target = 0.5 * qw.mean(dim=(0, 2))                       # [Hkv, D]
    else:
        target = torch.zeros(hkv, d)
    k = k.clone()
    for j in needle_chunks:
        pos = torch.randperm(c, generator=gen)[:min(NEEDLES_PER_CHUNK, c)]
        for t in sorted(pos.tolist()):
            row = j * (c + 1) + 1 + t
            noise = 0.5 * torch.randn(hkv, d, generator=gen, dtype=torch.float32)
            k[row] = (target + noise).to(torch.bfloat16)
            needle_rows.append((j, t))

    s_i = torch.randn(n, generator=gen, dtype=torch.float32)
    s_p = torch.randn(n, generator=gen, dtype=torch.float32)
    for j in needle_chunks:
        s_i[j] += 3.0
    if cfg.pool_order == "permuted":
        order = torch.randperm(n, generator=gen)
    else:
        order = torch.arange(n)
    slot_row = (order * cfg.slot_stride).to(torch.int32)
    return dict(q=q, k=k, v=v, q_win=q_win, k_win=k_win, v_win=v_win, s_i=s_i, s_p=s_p,
                slot_row=slot_row, needle_chunks=needle_chunks, needle_rows=needle_rows)


def make_layers(cfg: Config, n_layers: int, seq: int = 0) -> dict:
    """L layers of one request: layer l is make_request(cfg, seq + 101 * l);
    q, k, v [L, N*(C+1), H, D] and q_win [L, W, Hq, D] stacked; the slots
    (slot_row) are layer 0's, shared by every layer's pool."""
    reqs = [make_request(cfg, seq + 101 * l) for l in range(n_layers)]
    out = {key: torch.stack([r[key] for r in reqs]) for key in ("q", "k", "v", "q_win")}
    out["slot_row"] = reqs[0]["slot_row"]
    out["layers"] = reqs
    return out


def make_step(cfg: Config, seq: int, step: int) -> dict:
    """Draws the response rows of denoising step `step`."""
    gen = torch.Generator().manual_seed(1000 * cfg.config_id + seq + 7919 * (step + 1))
    q = _bf16(gen, cfg.n_resp, cfg.n_q_heads, cfg.head_dim)
    k = _bf16(gen, cfg.n_resp, cfg.n_kv_heads, cfg.head_dim)
    v = _bf16(gen, cfg.n_resp, cfg.n_kv_heads, cfg.head_dim)
    return dict(q=q, k=k, v=v)


def live_block(req: dict, step_inputs: dict) -> tuple:
    """The live rows of one step: the window rows followed by the response rows."""
    q = torch.cat([req["q_win"], step_inputs["q"]], dim=0)
    k = torch.cat([req["k_win"], step_inputs["k"]], dim=0)
    v = torch.cat([req["v_win"], step_inputs["v"]], dim=0)
    return q, k, v


# Vocabulary of the scoring-head workload: a 7B-scale language model's
# vocabulary size (152,064 entries).
SCORING_VOCAB = 152064


def make_logits(n_chunks: int, n_rows: int, vocab: int, seed: int, scale: float = 2.0) -> tuple:
    """Synthetic logits [N, R, V] bf16 ~ N(0, scale^2) and labels [R] int32
    uniform in [0, V), drawn in that order from a generator seeded `seed`."""
    gen = torch.Generator().manual_seed(seed)
    logits = (scale * torch.randn(n_chunks, n_rows, vocab, generator=gen)).to(torch.bfloat16)
    labels = torch.randint(0, vocab, (n_rows,), generator=gen, dtype=torch.int64).to(torch.int32)
    return logits, labels


def to_f64(t: torch.Tensor):
    """Exact widening of a bf16/fp32 CPU tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()
