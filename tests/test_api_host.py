"""The Python layer has no CPU path: every public call refuses host tensors
before it touches the library, and a missing library is an error, not a
fallback."""
import pytest
import torch

from sparse_chunked_kv_gb300 import _abi, api


def _bf(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def _i32(*shape):
    return torch.zeros(*shape, dtype=torch.int32)


def _f32(*shape):
    return torch.zeros(*shape, dtype=torch.float32)


CALLS = {
    "chunk_prefill": lambda: api.chunk_prefill(_bf(10, 4, 64), _bf(10, 2, 64), _bf(10, 2, 64),
                                               _bf(2, 4, 64), 2, 4, 2, _i32(2), 6),
    "chunk_prefill_ex": lambda: api.chunk_prefill_ex(_bf(10, 4, 64), _bf(10, 2, 64), _bf(10, 2, 64),
                                                     _bf(2, 4, 64), _bf(2, 2, 64), 2, 4, 2, _i32(2),
                                                     6),
    "chunk_prefill_layers": lambda: api.chunk_prefill_layers(
        _bf(2, 10, 4, 64), _bf(2, 10, 2, 64), _bf(2, 10, 2, 64), _bf(2, 2, 4, 64), 2, 4, 2, _i32(2),
        6),
    "chunk_prefill_batch": lambda: api.chunk_prefill_batch(
        _bf(2, 10, 4, 64), _bf(2, 10, 2, 64), _bf(2, 10, 2, 64), _bf(2, 2, 4, 64), 2, 4, 2,
        _i32(2, 2), _bf(12, 2, 64), _bf(12, 2, 64), _i32(2, 2, 2)),
    "select_chunks": lambda: api.select_chunks(_f32(4), _f32(4), 2),
    "select_chunks_batched": lambda: api.select_chunks_batched(_f32(4), _f32(4), _i32(2), _i32(2),
                                                               4),
    "decode_attention": lambda: api.decode_attention(_bf(8, 4, 64), _bf(8, 2, 64), _bf(8, 2, 64),
                                                     _bf(6, 2, 64), _bf(6, 2, 64), _i32(2, 2),
                                                     _i32(1)),
    "decode_partial": lambda: api.decode_partial(_bf(8, 4, 64), _bf(8, 2, 64), _bf(8, 2, 64),
                                                 _bf(6, 2, 64), _bf(6, 2, 64), _i32(2, 2), _i32(1),
                                                 [0, 8], [0, 1], 1),
    "lse_merge": lambda: api.lse_merge(_bf(2, 8, 4, 64), _f32(2, 8, 4)),
    "chunk_loglik": lambda: api.chunk_loglik(_bf(2, 3, 50), _i32(3)),
    "chunk_mass": lambda: api.chunk_mass(_bf(8, 4, 64), _bf(6, 2, 64), _i32(2, 2), _f32(8, 4),
                                         [0, 8], [0, 2]),
    "reselect_chunks": lambda: api.reselect_chunks(_f32(4), _f32(4), 1.0, _i32(2), _i32(2), 4),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_public_calls_refuse_host_tensors(name, monkeypatch):
    def no_library():
        raise AssertionError("the library was reached with host tensors")
    monkeypatch.setattr(_abi, "load", no_library)
    with pytest.raises(ValueError, match="CUDA"):
        CALLS[name]()


def test_every_public_call_is_covered():
    public = {n for n in dir(api) if not n.startswith("_") and callable(getattr(api, n))
              and getattr(getattr(api, n), "__module__", "") == api.__name__}
    assert public == set(CALLS)


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "LIB_PATH", str(tmp_path / "libpfd.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _abi.load()
