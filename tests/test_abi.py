"""CPU tests of the C ABI: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host with a status code
(no kernel runs; these calls return before touching a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch  # noqa: F401  (loads the CUDA runtime libraries first)

import __graft_entry__ as entry
from sparse_chunked_kv_gb300 import _abi

HEADER = os.path.join(entry.ROOT, "include", "pfd.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_abi.LIB_PATH):
        entry.build()
    return _abi.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pfd_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for want in ("pfd_chunk_prefill", "pfd_select_chunks", "pfd_decode_attention"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], stdout=subprocess.PIPE,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pfd_\w+)", out))
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, missing
    assert set(_abi.SIGNATURES) == set(declared_symbols())


def declared_prototypes():
    """{name: (return type, [parameter types])} of every prototype in the
    header, with comments removed and parameter names dropped."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    protos = {}
    for ret, name, params in re.findall(
            r"([A-Za-z_][\w ]*?\**)\s*\b(pfd_[a-z_]+)\s*\(([^;{]*?)\)\s*;", text):
        kinds = []
        for prm in params.split(","):
            prm = " ".join(prm.split())
            if not prm or prm == "void":
                continue
            kinds.append(re.sub(r"\s*\b\w+$", "", prm) if not prm.endswith("*") else prm)
        protos[name] = (" ".join(ret.split()), kinds)
    return protos


def _ctype_of(c_type):
    """The ctypes type a C parameter or return type must be marshalled as."""
    if "*" in c_type:
        return ctypes.c_char_p if c_type.replace(" ", "") == "constchar*" else ctypes.c_void_p
    base = c_type.replace("const ", "").strip()
    return {"pfd_stream_t": ctypes.c_void_p, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t,
            "float": ctypes.c_float, "int32_t": ctypes.c_int32, "int": ctypes.c_int,
            "pfd_status": ctypes.c_int}[base]


def test_binding_signatures_match_the_header():
    """Every ctypes signature has the header's parameter count and, position
    by position, a type of the same width and kind, so no argument is
    marshalled into the wrong register or truncated."""
    protos = declared_prototypes()
    assert set(protos) == set(_abi.SIGNATURES)
    for name, (ret, params) in protos.items():
        res, args = _abi.SIGNATURES[name]
        assert len(args) == len(params), (name, len(args), len(params))
        assert ctypes.sizeof(res) == ctypes.sizeof(_ctype_of(ret)), (name, ret)
        for i, (got, c_type) in enumerate(zip(args, params)):
            want = _ctype_of(c_type)
            assert ctypes.sizeof(got) == ctypes.sizeof(want), (name, i, c_type)
            assert (got is ctypes.c_float) == (want is ctypes.c_float), (name, i, c_type)
            assert (got in (ctypes.c_void_p, ctypes.c_char_p)) == (
                want in (ctypes.c_void_p, ctypes.c_char_p)), (name, i, c_type)


def test_version_and_status_strings(lib):
    assert _abi.pfd_abi_version() == 2
    assert _abi.pfd_status_string(0) == "PFD_OK"
    assert _abi.pfd_status_string(1) == "PFD_ERR_INVALID_ARG"
    assert _abi.pfd_status_string(2) == "PFD_ERR_UNSUPPORTED"


def _prefill_status(lib, **over):
    a = dict(q=256, k=256, v=256, q_win=256, N=2, C=16, W=4, Hq=4, Hkv=2, D=64, B=4, scale=0.0,
             out=256, scores=256, kept=256, pk=256, pv=256, pool_rows=10, slot=256, table=256,
             err=0, ws=256,
             ws_bytes=1 << 20, stream=0)
    a.update(over)
    return lib.pfd_chunk_prefill(a["q"], a["k"], a["v"], a["q_win"], a["N"], a["C"], a["W"], a["Hq"],
                                 a["Hkv"], a["D"], a["B"], a["scale"], a["out"], a["scores"],
                                 a["kept"], a["pk"], a["pv"], a["pool_rows"], a["slot"], a["table"],
                                 a["err"] or None, a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("over,status", [
    (dict(N=0), 1), (dict(C=0), 1), (dict(B=17), 1), (dict(B=-1), 1), (dict(Hq=5), 1),
    (dict(D=96), 2), (dict(C=9000), 2), (dict(W=200, Hq=8, Hkv=2), 2), (dict(q=0), 1),
    (dict(q_win=0), 1), (dict(pool_rows=4), 1), (dict(ws_bytes=0), 1), (dict(q=12), 1),
    (dict(ws=300), 1),
])
def test_prefill_host_checks(lib, over, status):
    assert _prefill_status(lib, **over) == status


def _prefill_batch_status(lib, L=2, **over):
    a = dict(q=256, k=256, v=256, q_win=256, N=2, C=16, W=4, Hq=4, Hkv=2, D=64, B=4, scale=0.0,
             out=256, scores=256, kept=256, pk=256, pv=256, pool_rows=20, slot=256, table=256,
             err=0, ws=256, ws_bytes=1 << 20, stream=0)
    a.update(over)
    return lib.pfd_chunk_prefill_batch(a["q"], a["k"], a["v"], a["q_win"], L, a["N"], a["C"],
                                       a["W"], a["Hq"], a["Hkv"], a["D"], a["B"], a["scale"],
                                       a["out"], a["scores"], a["kept"], a["pk"], a["pv"],
                                       a["pool_rows"], a["slot"], a["table"], a["err"] or None,
                                       a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("L,over,status", [
    (0, {}, 1), (2, dict(N=0), 1), (2, dict(B=17), 1), (2, dict(D=96), 2), (2, dict(slot=0), 1),
    (2, dict(table=0), 1), (2, dict(q_win=0), 1), (2, dict(ws_bytes=0), 1), (2, dict(q=12), 1),
])
def test_prefill_batch_host_checks(lib, L, over, status):
    """The batched prefill refuses bad arguments on the host, before any
    launch, with the same codes as the single-request call."""
    assert _prefill_batch_status(lib, L, **over) == status


def test_prefill_workspace_sizes(lib):
    small = lib.pfd_chunk_prefill_workspace(2, 16, 4, 4, 2, 64, 4)
    none = lib.pfd_chunk_prefill_workspace(2, 16, 0, 4, 2, 64, 4)
    assert small > 0 and small % 256 == 0 and none == 0
    assert lib.pfd_chunk_prefill_workspace(0, 16, 4, 4, 2, 64, 4) == 0


def test_select_host_checks(lib):
    assert lib.pfd_select_chunks(8, 8, 4, 5, 8, None, None) == 1
    assert lib.pfd_select_chunks(8, 8, 0, 0, 8, None, None) == 1
    assert lib.pfd_select_chunks(None, 8, 4, 2, 8, None, None) == 1
    assert lib.pfd_select_chunks(8, 8, 20000, 2, 8, None, None) == 2
    assert lib.pfd_select_chunks_batched(8, 8, 8, 8, 0, 4, 8, None, None) == 1


def test_decode_host_checks_and_plan(lib):
    cu_lq = (ctypes.c_int32 * 2)(0, 320)
    cu_k = (ctypes.c_int32 * 2)(0, 4)
    bad_lq = (ctypes.c_int32 * 2)(0, 0)
    args = [256, 256, 256, 256, cu_lq, 256, 256, 100, 256, 16, 256, 256, cu_k, 1, 28, 4, 128, 257,
            0.0, 1, 256, None, None, None, 0, None]
    a = list(args)
    a[0] = 8                      # misaligned q
    assert lib.pfd_decode_attention(*a) == 1
    a = list(args)
    a[19] = 2                     # two splits need a workspace
    assert lib.pfd_decode_attention(*a) == 1
    a = list(args)
    a[4] = bad_lq
    assert lib.pfd_decode_attention(*a) == 1
    a = list(args)
    a[16] = 80
    assert lib.pfd_decode_attention(*a) == 2
    a = list(args)
    a[14] = 27
    assert lib.pfd_decode_attention(*a) == 1
    a = list(args)
    a[19] = 65
    assert lib.pfd_decode_attention(*a) == 1
    s = _abi.pfd_decode_plan_splits(1, [0, 320], [0, 4], 28, 4, 128, 257)
    assert 1 <= s <= 64
    assert _abi.pfd_decode_workspace(1, [0, 320], [0, 4], 28, 4, 128, 257, 1) == 0
    ws2 = _abi.pfd_decode_workspace(1, [0, 320], [0, 4], 28, 4, 128, 257, 2)
    assert ws2 >= 2 * 320 * 28 * (2 * 4 + 128 * 2)   # fp32 (m, l) and bf16 O per row and split


def test_chunk_mass_items_per_call(lib):
    """pfd_chunk_mass groups up to 8 consecutive chunks per item, the most
    that still leaves 512 items: its workspace holds 8 partials per (item,
    chunk of the item), so the size shows the choice."""
    def ws(n_chunks, lq, hq=28, hkv=4):
        return lib.pfd_chunk_mass_workspace(1, (ctypes.c_int32 * 2)(0, lq),
                                            (ctypes.c_int32 * 2)(0, n_chunks), hq, hkv)
    align = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # 128K-like: 512 chunks, 576 live rows (16 pairs of 18-token tiles)
    assert ws(512, 576) == align(512 // 8 * 4 * 16 * 8 * 8 * 4)
    # 8K-like: 16 chunks, 320 rows (9 pairs): 2 chunks per item would give
    # 8 * 4 * 9 = 288 items (< 512), so one chunk per item (576 items)
    assert ws(16, 320) == align(16 * 4 * 9 * 1 * 8 * 4)
    # 130 chunks, 9 pairs: 2 per item gives 65 * 36 = 2340 items; 4 per item
    # 33 * 36 = 1188; 8 per item 17 * 36 = 612 >= 512
    assert ws(130, 320) == align(17 * 36 * 8 * 8 * 4)
    assert ws(0, 320) == 0


def test_partial_and_merge_host_checks(lib):
    """pfd_decode_partial needs part_lse and self_keys in {0, 1};
    pfd_lse_merge checks its counts, head dim and alignment on the host."""
    cu_lq = (ctypes.c_int32 * 2)(0, 320)
    cu_k = (ctypes.c_int32 * 2)(0, 4)
    args = [256, 256, 256, 256, cu_lq, 256, 256, 100, 256, 16, 256, 256, cu_k, 1, 28, 4, 128, 257,
            0.0, 1, 1, 256, 256, None, None, 0, None]
    a = list(args)
    a[22] = None                  # part_lse is required
    assert lib.pfd_decode_partial(*a) == 1
    a = list(args)
    a[19] = 2                     # self_keys must be 0 or 1
    assert lib.pfd_decode_partial(*a) == 1
    a = list(args)
    a[0] = 8                      # misaligned q
    assert lib.pfd_decode_partial(*a) == 1
    assert lib.pfd_lse_merge(256, 256, 0, 4, 4, 128, 256, None, None) == 1
    assert lib.pfd_lse_merge(256, 256, 2, 4, 4, 96, 256, None, None) == 2
    assert lib.pfd_lse_merge(256, 256, 65, 4, 4, 128, 256, None, None) == 2
    assert lib.pfd_lse_merge(258, 256, 2, 4, 4, 128, 256, None, None) == 1
    assert lib.pfd_lse_merge(None, 256, 2, 4, 4, 128, 256, None, None) == 1
    # without the live block the planner sees fewer keys, never more splits
    with_self = _abi.pfd_decode_partial_workspace(1, [0, 320], [0, 4], 28, 4, 128, 257, 1, 0)
    assert with_self == _abi.pfd_decode_workspace(1, [0, 320], [0, 4], 28, 4, 128, 257, 0)
    assert _abi.pfd_decode_partial_workspace(1, [0, 320], [0, 4], 28, 4, 128, 257, 0, 1) == 0


def test_decode_split_plan_of_the_bench_workloads(lib):
    """The automatic split counts of the benchmark's decode calls on a
    152-SM GB300 (the count the planner assumes with no device): the batched
    mix has enough (sequence, KV head, query-tile pair) items to fill the GPU
    unsplit; the single requests split their keys 4 or 7 ways."""
    import torch

    import bench
    if torch.cuda.is_available():
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        if sms != 152:
            pytest.skip(f"plan stated for 152 SMs, device has {sms}")
    want = {"tiny": 1, "8k": 4, "32k": 4, "128k": 7, "mix": 1}
    for name, splits in want.items():
        cfgs = bench.job_configs(name)
        cu_lq, cu_k = [0], [0]
        for c in cfgs:
            cu_lq.append(cu_lq[-1] + c.n_live)
            cu_k.append(cu_k[-1] + c.n_select)
        c0 = cfgs[0]
        got = _abi.pfd_decode_plan_splits(len(cfgs), cu_lq, cu_k, c0.n_q_heads, c0.n_kv_heads,
                                          c0.head_dim, max(c.n_keep + 1 for c in cfgs))
        assert got == splits, (name, got)


def test_scoring_head_mass_and_reselect_host_checks(lib):
    """Every call here is refused on the host (no call reaches a kernel)."""
    i32 = ctypes.c_int32
    # pfd_chunk_loglik(logits, labels, N, R, V, row_ll, score, dev_err, stream)
    assert lib.pfd_chunk_loglik(None, 256, 2, 3, 50, 256, 256, None, None) == 1
    assert lib.pfd_chunk_loglik(256, 256, 0, 3, 50, 256, 256, None, None) == 1
    assert lib.pfd_chunk_loglik(256, 256, 2, 0, 50, 256, 256, None, None) == 1
    assert lib.pfd_chunk_loglik(256, 256, 2, 3, 0, 256, 256, None, None) == 1
    assert lib.pfd_chunk_loglik(256, 256, 65536, 32768, 50, 256, 256, None, None) == 2
    assert lib.pfd_chunk_loglik(256, 256, 2, 3, 1 << 31, 256, 256, None, None) == 2

    # pfd_chunk_mass(q, cu_lq, cu_lq_host, pool_k, pool_rows, table, table_len, cu_n_host,
    #                lse, batch, Hq, Hkv, D, sm_scale, mass, dev_err, ws, ws_bytes, stream)
    def mass(**over):
        a = dict(q=256, cu_lq=256, lq_host=(i32 * 2)(0, 320), pk=256, pool_rows=100, table=256,
                 table_len=16, n_host=(i32 * 2)(0, 16), lse=256, batch=1, Hq=28, Hkv=4, D=128,
                 mass=256, ws=256, ws_bytes=1 << 20)
        a.update(over)
        return lib.pfd_chunk_mass(a["q"], a["cu_lq"], a["lq_host"], a["pk"], a["pool_rows"],
                                  a["table"], a["table_len"], a["n_host"], a["lse"], a["batch"],
                                  a["Hq"], a["Hkv"], a["D"], 0.0, a["mass"], None, a["ws"],
                                  a["ws_bytes"], None)
    assert mass(q=None) == 1
    assert mass(lse=None) == 1
    assert mass(D=96) == 2
    assert mass(batch=65, lq_host=(i32 * 66)(*range(0, 66)), n_host=(i32 * 66)(*range(66))) == 2
    assert mass(batch=0) == 1
    assert mass(Hq=27) == 1
    assert mass(n_host=(i32 * 2)(0, 17)) == 1          # more chunks than table entries
    assert mass(lq_host=(i32 * 2)(1, 320)) == 1        # offsets must start at 0
    assert mass(q=264) == 1                             # 8-byte aligned only
    assert mass(ws_bytes=0) == 1
    assert mass(ws=272) == 1                            # workspace must be 256-byte aligned
    assert mass(pool_rows=1 << 31) == 2

    # pfd_reselect_chunks(s, mass, lambda, cu_n, cu_k, batch, max_n, sel, s_out, stream)
    assert lib.pfd_reselect_chunks(None, 256, 1.0, 256, 256, 1, 8, 256, None, None) == 1
    assert lib.pfd_reselect_chunks(256, 256, 1.0, 256, 256, 0, 8, 256, None, None) == 1
    assert lib.pfd_reselect_chunks(256, 256, 1.0, 256, 256, 1, 0, 256, None, None) == 1
    assert lib.pfd_reselect_chunks(256, 256, -0.5, 256, 256, 1, 8, 256, None, None) == 1
    assert lib.pfd_reselect_chunks(256, 256, float("nan"), 256, 256, 1, 8, 256, None, None) == 1
    assert lib.pfd_reselect_chunks(256, 256, 1.0, 256, 256, 1, 16385, 256, None, None) == 2
    assert lib.pfd_select_chunks_batched(8, 8, 8, 8, 1, 16385, 8, None, None) == 2


def test_prefill_variant_host_checks(lib):
    """pfd_chunk_prefill_ex and pfd_chunk_prefill_layers refuse bad
    arguments on the host."""
    def ex(per_kv_head=0, C=16, k_win=256, N=2):
        return lib.pfd_chunk_prefill_ex(256, 256, 256, 256, k_win, N, C, 4, 4, 2, 64, 4, 0.0,
                                        per_kv_head, 256, 256, 256, 256, 256, 10, 256, 256, None,
                                        256, 1 << 20, None)
    assert ex(per_kv_head=2) == 1
    assert ex(per_kv_head=-1) == 1
    assert ex(C=9000) == 2
    assert ex(N=0) == 1

    def layers(L=2, N=2, C=16, B=4, D=64):
        return lib.pfd_chunk_prefill_layers(256, 256, 256, 256, L, N, C, 4, 4, 2, D, B, 0.0, 256,
                                            256, 256, 256, 256, 10, 256, 256, None, 256, 1 << 20,
                                            None)
    assert layers(L=0) == 1
    assert layers(B=17) == 1
    assert layers(D=96) == 2
    assert layers(L=1 << 15, N=1 << 10) == 2             # more than 2^24 chunks in one call
    assert lib.pfd_chunk_prefill_layers_workspace(0, 2, 16, 4, 4, 2, 64, 4) == 0
    one = lib.pfd_chunk_prefill_workspace(6, 16, 4, 4, 2, 64, 4)
    assert lib.pfd_chunk_prefill_layers_workspace(3, 2, 16, 4, 4, 2, 64, 4) == one


def test_static_scratch_host_checks(lib):
    """The static-scratch decode refuses, before it looks up its buffer, a
    missing batch, a negative split count and an explicit split count whose
    partials exceed the buffer."""
    i32 = ctypes.c_int32

    def call(batch=1, n_splits=0, lq=320, k=4):
        return lib.pfd_decode_attention_static_scratch(
            256, 256, 256, 256, (i32 * 2)(0, lq), 256, 256, 100, 256, 16, 256, 256,
            (i32 * 2)(0, k), batch, 28, 4, 128, 257, 0.0, n_splits, 256, None, None, None)
    assert call(batch=0) == 1
    assert call(n_splits=-1) == 1
    # 64 splits of 8192 live rows x 28 heads: far above the 32 MiB buffer
    assert call(n_splits=64, lq=8192, k=64) == 2


C_CONSUMER = r"""
#include <stdio.h>
#include <string.h>
#include "pfd.h"

int main(void) {
  if (pfd_abi_version() != 2) return 1;
  if (strcmp(pfd_status_string(PFD_ERR_UNSUPPORTED), "PFD_ERR_UNSUPPORTED") != 0) return 2;
  /* host-side checks only: null inputs are refused before any launch */
  if (pfd_select_chunks(NULL, NULL, 4, 2, NULL, NULL, NULL) != PFD_ERR_INVALID_ARG) return 3;
  if (pfd_chunk_prefill_workspace(16, 512, 64, 28, 4, 128, 256) == 0) return 4;
  printf("ok\n");
  return 0;
}
"""


def test_header_serves_a_plain_c_program(lib, tmp_path):
    """include/pfd.h compiles as strict C11 and C++17, and a C program links
    against libpfd.so and calls it with no torch or CUDA headers involved."""
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    inc = os.path.join(entry.ROOT, "include")
    libdir = os.path.dirname(_abi.LIB_PATH)
    flags = ["-Wall", "-Wextra", "-Werror", "-pedantic", "-I" + inc]
    subprocess.run(["g++", "-std=c++17", *flags, "-x", "c++", "-fsyntax-only", str(src)],
                   check=True)
    exe = tmp_path / "consumer"
    subprocess.run(["gcc", "-std=c11", *flags, str(src), "-L" + libdir, "-lpfd",
                    "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], stdout=subprocess.PIPE, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout)
