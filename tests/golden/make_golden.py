"""Writes tests/golden/tiny_oracle.json from the CPU oracle alone.

The pages print no worked example with numbers, so the stored values here are
regression values of the oracle on the seeded tiny workload (8 chunks of 256
tokens + BOS, 8 query / 2 KV heads, D = 64, W = 32, B = 64, K = 2).  They pin
the seeded input recipe and the oracle against silent drift (for example a
change of torch's CPU generator between versions); they are not evidence of
correctness, which the pins in oracle_pins.py provide.

Run from the repository root:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from oracle import pfd_oracle as orc  # noqa: E402
from sparse_chunked_kv_gb300 import workloads as wl  # noqa: E402


def input_digest(req):
    h = hashlib.sha256()
    for name in ("q", "k", "v", "q_win", "k_win", "v_win", "s_i", "s_p", "slot_row"):
        h.update(req[name].contiguous().view(-1).view(dtype=__import__("torch").uint8).numpy().tobytes())
    return h.hexdigest()


def compute():
    cfg = wl.TINY
    req = wl.make_request(cfg, 0)
    scores = orc.window_scores(wl.to_f64(req["q_win"]), wl.to_f64(req["k"]), cfg.n_chunks,
                               cfg.chunk_size, cfg.sm_scale)
    kept = orc.top_b(scores, cfg.n_keep)
    sel, s = orc.select_chunks(req["s_i"].numpy(), req["s_p"].numpy(), cfg.n_select)
    return dict(
        config=cfg.name,
        input_sha256=input_digest(req),
        needle_chunks=req["needle_chunks"],
        sel=[int(x) for x in sel],
        s=[float(x) for x in s],
        kept_first_chunk=[int(x) for x in kept[0]],
        kept_sha256=hashlib.sha256(np.ascontiguousarray(kept).tobytes()).hexdigest(),
        score_chunk_sums=[float(x) for x in scores.sum(axis=1)],
        score_first_row=[float(x) for x in scores[0, :8]],
    )


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(out, "w") as f:
        json.dump(compute(), f, indent=1)
    print("wrote", out)
