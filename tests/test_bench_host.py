"""Host logic of bench.py that needs no GPU: matching committed ncu
summaries to the kernels they were taken on."""
import os


def test_profile_hash_ignores_comments_not_code(tmp_path):
    """A committed ncu summary stays matched to its kernels across comment
    edits, and stops matching once the code changes."""
    import shutil

    import bench
    src = os.path.join(bench.ROOT, "sparse_chunked_kv_gb300", "csrc")
    dst = tmp_path / "csrc"
    shutil.copytree(src, dst)
    base = bench.kernel_source_hash(str(dst))
    assert base == bench.kernel_source_hash()
    attn = dst / "attn_tc.cu"
    text = attn.read_text()
    attn.write_text("// a new comment line\n" + text.replace("{", "{  /* spaced */ ", 1))
    assert bench.kernel_source_hash(str(dst)) == base
    attn.write_text(text.replace("kRescaleThreshold = 8.0f", "kRescaleThreshold = 7.0f", 1))
    assert "kRescaleThreshold = 7.0f" in attn.read_text()
    assert bench.kernel_source_hash(str(dst)) != base


def test_job_groups_same_shaped_sequences():
    """The bench job orders a mixed batch by prefill shape, so each group's
    chunks and table entries are contiguous for one batched prefill call;
    every sequence keeps its own data seed, its tensors are views of its
    group's stacked buffers, and its slots lie in its own region of the one
    pool."""
    import torch

    import bench
    from sparse_chunked_kv_gb300 import workloads as wl
    cfgs = [wl.scaled(c, n_chunks=4) for c in wl.mix_configs()]
    job = bench.Job(cfgs, 0, torch.device("cpu"), max_steps=1)
    assert job.seq_ids == [0, 3, 6, 1, 4, 7, 2, 5]
    assert [c.chunk_size for c in job.cfgs] == [256] * 3 + [1024] * 3 + [4096] * 2
    assert [(g["i0"], g["L"]) for g in job.groups] == [(0, 3), (3, 3), (6, 2)]
    assert job.launches_per_step() == 3 * 3 + 1 + job.T
    for g in job.groups:
        for l in range(g["L"]):
            sq = job.seqs[g["i0"] + l]
            assert sq["q"].data_ptr() == g["q"][l].data_ptr()
            assert sq["n0"] == job.cu_n_host[g["i0"] + l]
    # each sequence's data is its own seed's request
    for i, c in enumerate(job.cfgs):
        ref = wl.make_request(c, job.seq_ids[i])
        assert torch.equal(job.seqs[i]["q"], ref["q"])
    # slots: absolute rows inside the sequence's pool region, never overlapping
    used = torch.zeros(job.pool_rows, dtype=torch.int32)
    base = 0
    for i, c in enumerate(job.cfgs):
        rows = job.seqs[i]["slot_row"].long()
        assert int(rows.min()) >= base and int(rows.max()) + c.n_keep + 1 <= base + c.pool_rows
        for r in rows.tolist():
            used[r:r + c.n_keep + 1] += 1
        base += c.pool_rows
    assert int(used.max()) == 1


# Algorithmic sizes of each workload, worked out by hand from its shapes
# before the bench existed: prefill GFLOP, prefill MB, decode GFLOP per
# step, decode MB per step, to 2-4 significant digits.
WORKLOAD_SIZES = {
    "tiny": (1.15, 5.6, 0.025, 0.23),
    "8k": (64.1, 143, 6.18, 7.4),
    "32k": (497, 572, 20.3, 13.7),
    "128k": (545, 2292, 72.9, 26.4),
    "mix": (5780, 4443, 87.5, 76),
}


def test_cost_model_matches_oracle_counts_and_table():
    """The work the bench divides by is the method's: its flop counts equal
    twice the oracle's counted multiply-adds for the same shapes, and every
    figure agrees with the hand-worked sizes to their printed precision."""
    import math

    import bench
    from oracle import pfd_oracle as orc
    for name, (pg, pmb, dg, dmb) in WORKLOAD_SIZES.items():
        cfgs = bench.job_configs(name)
        for c in cfgs:
            assert bench.prefill_flops(c) == 2 * orc.prefill_macs(
                c.n_chunks, c.chunk_size, c.n_win, c.n_q_heads, c.head_dim)
            kept = c.n_select * (c.n_keep + 1)
            assert bench.decode_flops(c) == 2 * orc.decode_step_macs(
                c.n_live, kept, c.n_q_heads, c.head_dim)
        got = (bench.total(bench.prefill_flops, cfgs) / 1e9,
               bench.total(bench.prefill_bytes, cfgs) / 1e6,
               bench.total(bench.decode_flops, cfgs) / 1e9,
               bench.total(bench.decode_bytes, cfgs) / 1e6)
        for g, want in zip(got, (pg, pmb, dg, dmb)):
            # printed to 2-3 significant digits
            digits = max(2, len(str(want).replace(".", "").lstrip("0")))
            assert math.isclose(g, want, rel_tol=0.6 * 10.0 ** (1 - digits)), (name, g, want)


def test_roofline_fractions():
    """Decode against the bf16 burst, sustained and nominal peaks; prefill
    against the slower of its HBM and tensor times, measured and nominal."""
    import math

    import bench
    cfgs = bench.job_configs("mix")
    peaks = {"hbm_gbs": 6691.8, "bf16_tflops": 1910.6, "bf16_tflops_sustained": 1723.9}
    fr = bench.roofline_fracs(cfgs, 0.090, 5.08, peaks)
    tflops = bench.total(bench.decode_flops, cfgs) / 90e-6 / 1e12
    assert math.isclose(fr["decode_tflops"], tflops)
    assert math.isclose(fr["decode_frac"], tflops / 1910.6)
    assert math.isclose(fr["decode_frac_sustained"], tflops / 1723.9)
    assert math.isclose(fr["decode_frac_nominal"], tflops / 2250.0)
    assert fr["prefill_bound"] == "tensor"
    t_tc = bench.total(bench.prefill_flops, cfgs) / 1910.6e12
    assert math.isclose(fr["prefill_frac"], t_tc / 5.08e-3)
    assert math.isclose(fr["prefill_frac_nominal"],
                        bench.total(bench.prefill_flops, cfgs) / 2250e12 / 5.08e-3)
    # the 128K prefill moves more bytes than its flops take at the peak
    fr = bench.roofline_fracs(bench.job_configs("128k"), 0.0839, 1.104, peaks)
    assert fr["prefill_bound"] == "hbm"
    t_hbm = bench.total(bench.prefill_bytes, bench.job_configs("128k")) / 6691.8e9
    assert math.isclose(fr["prefill_frac"], t_hbm / 1.104e-3)


def test_bench_line_carries_the_contract_keys(monkeypatch, capsys):
    """bench.main's one JSON line, with the GPU timings faked: every key the
    benchmark contract names is present and follows from the timings."""
    import json
    import math
    import sys

    import bench
    peaks = {"hbm_gbs": 6691.8, "bf16_tflops": 1910.6, "bf16_tflops_sustained": 1723.9}
    clocks = {"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": [], "samples": 11}
    fake = dict(pre_ms=5.08, dec_ms=64 * 0.090, step_ms=5.08 + 64 * 0.090, wall=0.3,
                clocks=clocks, launches=74 * 20, n_splits=1,
                e2e=dict(dec_ms=64 * 0.144, dec_h2d=64 * 23_592_960, dec_d2h=64 * 18_350_080,
                         pre_ms=60.0, pre_h2d=1_000_000))

    def workload(name, rank, device, reps=5):
        cfgs = bench.job_configs(name)
        return dict(cfgs=cfgs, pre_ms=1.0, dec_ms=cfgs[0].n_steps * 0.05, n_splits=4,
                    T=cfgs[0].n_steps)

    monkeypatch.setattr(bench, "run_gpu", lambda args, cfgs, rank, world, device: dict(fake))
    monkeypatch.setattr(bench, "time_workload", workload)
    monkeypatch.setattr(bench, "time_scoring_head",
                        lambda device: {"us": 238.1, "gbs": 6539.0, "bound": "hbm"})
    monkeypatch.setattr(bench, "time_next_rows",
                        lambda device: {"layers": {"us": 360.0, "tflops": 712.0, "bound": "tensor"}})
    monkeypatch.setattr(bench, "load_peaks", lambda: (dict(peaks), "measured"))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--no-cpu-baseline"])
    for var in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    bench.main()
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "clocks", "gpu_launches", "e2e"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["higher_is_better"] is True
    assert line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["config"]["workload"].startswith("mix")
    cfgs = bench.job_configs("mix")
    tflops = bench.total(bench.decode_flops, cfgs) / 90e-6 / 1e12
    assert math.isclose(line["value"], tflops)
    roof = line["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(roof)
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["peak"] == 1910.6
    assert math.isclose(roof["frac"], roof["achieved"] / roof["peak"])
    assert math.isclose(roof["frac_of_nominal"], tflops / 2250.0)
    e2e = line["e2e"]
    assert {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"} <= set(e2e)
    assert math.isclose(e2e["value"], bench.total(bench.decode_flops, cfgs) / 144e-6 / 1e12)
    assert line["gpu_launches"] == 74 * 20 and line["clocks"] == clocks
    assert set(line["per_config"]) == {"8k", "32k", "128k"}
    assert math.isclose(line["next_rows"]["scoring_head"]["frac"], 6539.0 / 6691.8)
    assert math.isclose(line["next_rows"]["layers"]["frac"], 712.0 / 1910.6)
