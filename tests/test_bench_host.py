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
