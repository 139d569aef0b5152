"""CPU tests of the seeded input recipe and of the stored oracle regression values."""
import json
import os

import numpy as np
import torch

from sparse_chunked_kv_gb300 import workloads as wl
from tests.golden import make_golden

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.json")


def test_request_is_deterministic():
    a, b = wl.make_request(wl.TINY, 0), wl.make_request(wl.TINY, 0)
    for name in ("q", "k", "v", "q_win", "s_i", "s_p", "slot_row"):
        assert torch.equal(a[name], b[name])
    c = wl.make_request(wl.TINY, 1)
    assert not torch.equal(a["q"], c["q"])


def test_request_shapes_and_needles():
    cfg = wl.TINY
    req = wl.make_request(cfg, 0)
    assert req["q"].shape == (cfg.rows, cfg.n_q_heads, cfg.head_dim)
    assert req["k"].dtype == torch.bfloat16
    assert req["q_win"].shape == (cfg.n_win, cfg.n_q_heads, cfg.head_dim)
    assert len(req["needle_chunks"]) == cfg.n_needle_chunks
    assert len(req["needle_rows"]) == wl.NEEDLES_PER_CHUNK * cfg.n_needle_chunks
    for j, t in req["needle_rows"]:
        assert j in req["needle_chunks"] and 0 <= t < cfg.chunk_size


def test_permuted_slots_are_a_permutation():
    req = wl.make_request(wl.CTX_32K, 0)
    cfg = wl.CTX_32K
    rows = sorted(req["slot_row"].tolist())
    assert rows == [j * cfg.slot_stride for j in range(cfg.n_chunks)]
    assert req["slot_row"].tolist() != rows


def test_step_inputs_redrawn():
    a, b = wl.make_step(wl.TINY, 0, 0), wl.make_step(wl.TINY, 0, 1)
    assert not torch.equal(a["q"], b["q"])
    assert torch.equal(a["q"], wl.make_step(wl.TINY, 0, 0)["q"])


def test_mix_configs():
    mix = wl.mix_configs()
    assert len(mix) == 8
    assert sum(c.n_chunks for c in mix) == 496
    for c in mix:
        assert c.n_chunks * c.chunk_size == 32768
        assert c.n_select * c.chunk_size == 8192
        assert c.n_keep * 4 == c.chunk_size


def test_golden_oracle_regression():
    with open(GOLDEN) as f:
        want = json.load(f)
    got = make_golden.compute()
    assert got["input_sha256"] == want["input_sha256"], "seeded inputs drifted"
    assert got["sel"] == want["sel"]
    assert got["kept_sha256"] == want["kept_sha256"]
    np.testing.assert_allclose(got["score_chunk_sums"], want["score_chunk_sums"], rtol=0, atol=1e-9)
    np.testing.assert_allclose(got["score_first_row"], want["score_first_row"], rtol=1e-12)
