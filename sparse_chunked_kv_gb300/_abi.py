"""ctypes binding of libpfd's C ABI: one Python function per exported symbol,
with the same name and argument order.  Arguments are marshalled only:
tensors become device pointers, streams become cudaStream_t handles, and a
status other than PFD_OK raises PfdError.  Every computation runs in the CUDA
kernels of libpfd; there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpfd.so")

PFD_OK = 0
STATUS_NAMES = {0: "PFD_OK", 1: "PFD_ERR_INVALID_ARG", 2: "PFD_ERR_UNSUPPORTED", 3: "PFD_ERR_CUDA"}

# PFD_DECODE_STATIC_SCRATCH_BYTES of include/pfd.h
DECODE_STATIC_SCRATCH_BYTES = 32 << 20

DEVERR_TABLE, DEVERR_SEL, DEVERR_SLOT, DEVERR_TIMEOUT, DEVERR_SHAPE, DEVERR_LABEL = 1, 2, 4, 8, 16, 32

# (restype, argtypes) of every exported symbol, in the order of include/pfd.h.
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_I64 = ctypes.c_int64
_F = ctypes.c_float
SIGNATURES = {
    "pfd_chunk_prefill_workspace": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "pfd_chunk_prefill": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P,
                               _I64, _P, _P, _P, _P, _SZ, _P]),
    "pfd_chunk_prefill_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P,
                                  _P, _P, _P, _I64, _P, _P, _P, _P, _SZ, _P]),
    "pfd_chunk_prefill_layers_workspace": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "pfd_chunk_prefill_layers": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                                      _P, _P, _P, _I64, _P, _P, _P, _P, _SZ, _P]),
    "pfd_chunk_prefill_batch": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                                     _P, _P, _P, _I64, _P, _P, _P, _P, _SZ, _P]),
    "pfd_chunk_loglik": (_I, [_P, _P, _I, _I, _I64, _P, _P, _P, _P]),
    "pfd_select_chunks": (_I, [_P, _P, _I, _I, _P, _P, _P]),
    "pfd_select_chunks_batched": (_I, [_P, _P, _P, _P, _I, _I, _P, _P, _P]),
    "pfd_decode_plan_splits": (_I, [_I, _P, _P, _I, _I, _I, _I]),
    "pfd_decode_workspace": (_SZ, [_I, _P, _P, _I, _I, _I, _I, _I]),
    "pfd_decode_attention": (_I, [_P, _P, _P, _P, _P, _P, _P, _I64, _P, ctypes.c_int32, _P, _P, _P,
                                  _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P, _SZ, _P]),
    "pfd_decode_attention_static_scratch": (_I, [_P, _P, _P, _P, _P, _P, _P, _I64, _P,
                                                 ctypes.c_int32, _P, _P, _P, _I, _I, _I, _I, _I,
                                                 _F, _I, _P, _P, _P, _P]),
    "pfd_decode_partial_workspace": (_SZ, [_I, _P, _P, _I, _I, _I, _I, _I, _I]),
    "pfd_decode_partial": (_I, [_P, _P, _P, _P, _P, _P, _P, _I64, _P, ctypes.c_int32, _P, _P, _P,
                                _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "pfd_lse_merge": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "pfd_chunk_mass_workspace": (_SZ, [_I, _P, _P, _I, _I]),
    "pfd_chunk_mass": (_I, [_P, _P, _P, _P, _I64, _P, ctypes.c_int32, _P, _P, _I, _I, _I, _I, _F,
                            _P, _P, _P, _SZ, _P]),
    "pfd_reselect_chunks": (_I, [_P, _P, _F, _P, _P, _I, _I, _P, _P, _P]),
    "pfd_status_string": (ctypes.c_char_p, [_I]),
    "pfd_abi_version": (_I, []),
}


class PfdError(RuntimeError):
    """A libpfd call returned a status other than PFD_OK."""


_lib = None


def load():
    """Loads libpfd.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpfd.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x):
    """Device/host pointer of a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _host_i32(arr):
    """A host int32 buffer (ctypes array) from a list / CPU tensor."""
    vals = arr.tolist() if hasattr(arr, "tolist") else list(arr)
    return (ctypes.c_int32 * len(vals))(*[int(v) for v in vals])


def _check(status):
    if status != PFD_OK:
        raise PfdError(load().pfd_status_string(status).decode())


def pfd_abi_version():
    return load().pfd_abi_version()


def pfd_status_string(status):
    return load().pfd_status_string(int(status)).decode()


def pfd_chunk_prefill_workspace(N, C, W, Hq, Hkv, D, B):
    return load().pfd_chunk_prefill_workspace(N, C, W, Hq, Hkv, D, B)


def pfd_chunk_prefill(q, k, v, q_win, N, C, W, Hq, Hkv, D, B, sm_scale, out, scores, kept_idx,
                      pool_k, pool_v, pool_rows, slot_row, table, dev_err, workspace,
                      workspace_bytes, stream=None):
    _check(load().pfd_chunk_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(q_win), N, C, W, Hq, Hkv, D, B, float(sm_scale), _ptr(out),
        _ptr(scores), _ptr(kept_idx), _ptr(pool_k), _ptr(pool_v), int(pool_rows), _ptr(slot_row),
        _ptr(table), _ptr(dev_err), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def pfd_select_chunks(s_I, s_P, N, K, sel, s_out, stream=None):
    _check(load().pfd_select_chunks(_ptr(s_I), _ptr(s_P), N, K, _ptr(sel), _ptr(s_out),
                                    _stream(stream)))


def pfd_select_chunks_batched(s_I, s_P, cu_n, cu_k, batch, max_n, sel, s_out, stream=None):
    _check(load().pfd_select_chunks_batched(_ptr(s_I), _ptr(s_P), _ptr(cu_n), _ptr(cu_k), batch,
                                            max_n, _ptr(sel), _ptr(s_out), _stream(stream)))


def pfd_decode_plan_splits(batch, cu_lq_host, cu_k_host, Hq, Hkv, D, max_chunk_len):
    a, b = _host_i32(cu_lq_host), _host_i32(cu_k_host)
    return load().pfd_decode_plan_splits(batch, ctypes.cast(a, _P), ctypes.cast(b, _P), Hq, Hkv, D,
                                         max_chunk_len)


def pfd_decode_workspace(batch, cu_lq_host, cu_k_host, Hq, Hkv, D, max_chunk_len, n_splits):
    a, b = _host_i32(cu_lq_host), _host_i32(cu_k_host)
    return load().pfd_decode_workspace(batch, ctypes.cast(a, _P), ctypes.cast(b, _P), Hq, Hkv, D,
                                       max_chunk_len, n_splits)


def pfd_decode_attention(q, k_self, v_self, cu_lq, cu_lq_host, pool_k, pool_v, pool_rows, table,
                         table_len, sel, cu_k, cu_k_host, batch, Hq, Hkv, D, max_chunk_len,
                         sm_scale, n_splits, out, lse, dev_err, workspace, workspace_bytes,
                         stream=None):
    a, b = _host_i32(cu_lq_host), _host_i32(cu_k_host)
    _check(load().pfd_decode_attention(
        _ptr(q), _ptr(k_self), _ptr(v_self), _ptr(cu_lq), ctypes.cast(a, _P), _ptr(pool_k),
        _ptr(pool_v), int(pool_rows), _ptr(table), int(table_len), _ptr(sel), _ptr(cu_k),
        ctypes.cast(b, _P), batch, Hq, Hkv, D, max_chunk_len, float(sm_scale), n_splits, _ptr(out),
        _ptr(lse), _ptr(dev_err), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def pfd_decode_attention_static_scratch(q, k_self, v_self, cu_lq, cu_lq_host, pool_k, pool_v,
                                        pool_rows, table, table_len, sel, cu_k, cu_k_host, batch,
                                        Hq, Hkv, D, max_chunk_len, sm_scale, n_splits, out, lse,
                                        dev_err, stream=None):
    """pfd_decode_attention with its split partials in the library's static
    device scratch (no workspace argument, nothing allocated)."""
    a, b = _host_i32(cu_lq_host), _host_i32(cu_k_host)
    status = load().pfd_decode_attention_static_scratch(
        _ptr(q), _ptr(k_self), _ptr(v_self), _ptr(cu_lq), ctypes.cast(a, _P), _ptr(pool_k),
        _ptr(pool_v), int(pool_rows), _ptr(table), int(table_len), _ptr(sel), _ptr(cu_k),
        ctypes.cast(b, _P), batch, Hq, Hkv, D, max_chunk_len, float(sm_scale), n_splits, _ptr(out),
        _ptr(lse), _ptr(dev_err), _stream(stream))
    if status == 2:
        need = pfd_decode_workspace(batch, cu_lq_host, cu_k_host, Hq, Hkv, D, max_chunk_len,
                                    n_splits)
        if need > DECODE_STATIC_SCRATCH_BYTES:
            raise PfdError(f"PFD_ERR_UNSUPPORTED: these sizes need {need} bytes of decode scratch, "
                           f"more than the static {DECODE_STATIC_SCRATCH_BYTES} bytes")
    _check(status)


def pfd_decode_partial_workspace(batch, cu_lq_host, cu_k_host, Hq, Hkv, D, max_chunk_len,
                                 self_keys, n_splits):
    a, b = _host_i32(cu_lq_host), _host_i32(cu_k_host)
    return load().pfd_decode_partial_workspace(batch, ctypes.cast(a, _P), ctypes.cast(b, _P), Hq,
                                               Hkv, D, max_chunk_len, int(self_keys), n_splits)


def pfd_decode_partial(q, k_self, v_self, cu_lq, cu_lq_host, pool_k, pool_v, pool_rows, table,
                       table_len, sel, cu_k, cu_k_host, batch, Hq, Hkv, D, max_chunk_len,
                       sm_scale, self_keys, n_splits, part_o, part_lse, dev_err, workspace,
                       workspace_bytes, stream=None):
    a, b = _host_i32(cu_lq_host), _host_i32(cu_k_host)
    _check(load().pfd_decode_partial(
        _ptr(q), _ptr(k_self), _ptr(v_self), _ptr(cu_lq), ctypes.cast(a, _P), _ptr(pool_k),
        _ptr(pool_v), int(pool_rows), _ptr(table), int(table_len), _ptr(sel), _ptr(cu_k),
        ctypes.cast(b, _P), batch, Hq, Hkv, D, max_chunk_len, float(sm_scale), int(self_keys),
        n_splits, _ptr(part_o), _ptr(part_lse), _ptr(dev_err), _ptr(workspace),
        int(workspace_bytes), _stream(stream)))


def pfd_lse_merge(part_o, part_lse, n_parts, rows, Hq, D, out, lse, stream=None):
    _check(load().pfd_lse_merge(_ptr(part_o), _ptr(part_lse), n_parts, rows, Hq, D, _ptr(out),
                                _ptr(lse), _stream(stream)))


def pfd_chunk_loglik(logits, labels, N, R, V, row_ll, score, dev_err, stream=None):
    _check(load().pfd_chunk_loglik(_ptr(logits), _ptr(labels), N, R, int(V), _ptr(row_ll),
                                   _ptr(score), _ptr(dev_err), _stream(stream)))


def pfd_chunk_prefill_ex(q, k, v, q_win, k_win, N, C, W, Hq, Hkv, D, B, sm_scale, per_kv_head, out,
                         scores, kept_idx, pool_k, pool_v, pool_rows, slot_row, table, dev_err,
                         workspace, workspace_bytes, stream=None):
    _check(load().pfd_chunk_prefill_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(q_win), _ptr(k_win), N, C, W, Hq, Hkv, D, B,
        float(sm_scale), int(per_kv_head), _ptr(out), _ptr(scores), _ptr(kept_idx), _ptr(pool_k),
        _ptr(pool_v), int(pool_rows), _ptr(slot_row), _ptr(table), _ptr(dev_err), _ptr(workspace),
        int(workspace_bytes), _stream(stream)))


def pfd_chunk_prefill_layers_workspace(L, N, C, W, Hq, Hkv, D, B):
    return load().pfd_chunk_prefill_layers_workspace(L, N, C, W, Hq, Hkv, D, B)


def pfd_chunk_prefill_layers(q, k, v, q_win, L, N, C, W, Hq, Hkv, D, B, sm_scale, out, scores,
                             kept_idx, pool_k, pool_v, pool_rows, slot_row, table, dev_err,
                             workspace, workspace_bytes, stream=None):
    _check(load().pfd_chunk_prefill_layers(
        _ptr(q), _ptr(k), _ptr(v), _ptr(q_win), L, N, C, W, Hq, Hkv, D, B, float(sm_scale),
        _ptr(out), _ptr(scores), _ptr(kept_idx), _ptr(pool_k), _ptr(pool_v), int(pool_rows),
        _ptr(slot_row), _ptr(table), _ptr(dev_err), _ptr(workspace), int(workspace_bytes),
        _stream(stream)))


def pfd_chunk_prefill_batch(q, k, v, q_win, L, N, C, W, Hq, Hkv, D, B, sm_scale, out, scores,
                            kept_idx, pool_k, pool_v, pool_rows, slot_row, table, dev_err,
                            workspace, workspace_bytes, stream=None):
    _check(load().pfd_chunk_prefill_batch(
        _ptr(q), _ptr(k), _ptr(v), _ptr(q_win), L, N, C, W, Hq, Hkv, D, B, float(sm_scale),
        _ptr(out), _ptr(scores), _ptr(kept_idx), _ptr(pool_k), _ptr(pool_v), int(pool_rows),
        _ptr(slot_row), _ptr(table), _ptr(dev_err), _ptr(workspace), int(workspace_bytes),
        _stream(stream)))


def pfd_chunk_mass_workspace(batch, cu_lq_host, cu_n_host, Hq, Hkv):
    a, b = _host_i32(cu_lq_host), _host_i32(cu_n_host)
    return load().pfd_chunk_mass_workspace(batch, ctypes.cast(a, _P), ctypes.cast(b, _P), Hq, Hkv)


def pfd_chunk_mass(q, cu_lq, cu_lq_host, pool_k, pool_rows, table, table_len, cu_n_host, lse,
                   batch, Hq, Hkv, D, sm_scale, mass, dev_err, workspace, workspace_bytes,
                   stream=None):
    a, b = _host_i32(cu_lq_host), _host_i32(cu_n_host)
    _check(load().pfd_chunk_mass(
        _ptr(q), _ptr(cu_lq), ctypes.cast(a, _P), _ptr(pool_k), int(pool_rows), _ptr(table),
        int(table_len), ctypes.cast(b, _P), _ptr(lse), batch, Hq, Hkv, D, float(sm_scale),
        _ptr(mass), _ptr(dev_err), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def pfd_reselect_chunks(s, mass, lam, cu_n, cu_k, batch, max_n, sel, s_out, stream=None):
    _check(load().pfd_reselect_chunks(_ptr(s), _ptr(mass), float(lam), _ptr(cu_n), _ptr(cu_k),
                                      batch, max_n, _ptr(sel), _ptr(s_out), _stream(stream)))
