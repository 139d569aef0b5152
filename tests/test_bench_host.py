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
