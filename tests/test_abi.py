"""The C-ABI library builds, loads and exports every entry point that
include/csa.h declares; host-side argument checks reject bad calls before any
launch.  CPU only: no call here reaches a kernel."""
import ctypes as C
import os
import re
import subprocess

import pytest

import fp4_sparse_attention_csa_gb300 as csa
from fp4_sparse_attention_csa_gb300 import build as csa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    csa_build.build()
    return csa.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "csa.h")).read()
    return sorted(set(re.findall(r"CSA_API\s+[\w\s\*]+?\b(csa_\w+)\s*\(", text)))


def test_header_declares_the_five_entry_points():
    names = declared_functions()
    for n in ("csa_append", "csa_index_score", "csa_topk", "csa_sparse_attn", "csa_decode", "csa_step"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert C.cast(getattr(lib, name), C.c_void_p).value


def test_status_strings(lib):
    for s, name in csa.STATUS_NAMES.items():
        assert csa.csa_status_string(s)
    assert csa.csa_status_string(0) == "ok"


def test_null_arguments_are_rejected_before_launch(lib):
    assert lib.csa_append(None, None, None, None, 0, None, None, None, None, 0, None) == 1
    assert lib.csa_index_score(None, None, 16, None, None, None, 0, None, 0, None) == 1
    assert lib.csa_topk(1, None, 512, None, 512, 256, None, None, 0, None) == 2      # k != 512
    assert lib.csa_topk(1, None, 512, None, 512, 512, None, None, 0, None) == 1
    assert lib.csa_sparse_attn(None, None, None, None, 64, None, 1.0, None, None, None, 0, None) == 1
    assert lib.csa_decode(None, None, None, 64, None, None, 64, None, 1.0, None, None, None, None, 0, None) == 1


def test_step_checks_both_halves_before_any_launch(lib):
    """csa_step validates the append's and the decode's arguments before its
    first launch: a bad decode half is rejected (1 = invalid argument, 3 =
    workspace too small) although the append half is valid and has tokens.
    Without a GPU a launch would return 4 (CUDA error) instead."""
    assert lib.csa_step(None, None, None, None, 0, None, None, None, None, None, 64, None, None, 64, None, 1.0,
                        None, None, None, None, 0, None) == 1
    buf = (C.c_uint8 * 4096)()
    base = (C.addressof(buf) + 255) & ~255
    pt = (C.c_int32 * 4)()
    ints = (C.c_int32 * 8)()
    cache = csa.CsaCache(base, base, C.addressof(pt), 1, 1, 1, 2)
    rows = csa.CsaRows(1, C.addressof(ints), C.addressof(ints), 16, 1)
    args = [C.byref(cache), None, C.addressof(ints), C.addressof(ints), 1, base, base, base, None, C.byref(rows),
            64, None, base, 64, base, 1.0, base, None, None, base, 4096, None]
    assert lib.csa_step(*args) == 1                       # q_idx missing
    args[11] = base
    args[20] = 0
    assert lib.csa_step(*args) == 3                       # decode workspace too small
    args[20] = 4096
    args[13] = 0
    assert lib.csa_step(*args) == 2                       # n_heads out of range


def test_unsupported_head_counts_are_rejected_before_launch(lib):
    """The attention kernel is built for 16, 32 and 64 heads and the index
    score for 1..128 indexer heads: any other count returns 2 (unsupported)
    from csa_decode, csa_step and csa_sparse_attn before a launch (without a
    GPU a launch would return 4)."""
    buf = (C.c_uint8 * 65536)()
    base = (C.addressof(buf) + 255) & ~255
    pt = (C.c_int32 * 4)()
    ints = (C.c_int32 * 8)()
    cache = csa.CsaCache(base, base, C.addressof(pt), 1, 1, 1, 2)
    rows = csa.CsaRows(1, C.addressof(ints), C.addressof(ints), 16, 1)
    ws_n = csa.csa_workspace_size(csa.OP_DECODE, 1, 16, 64)
    assert ws_n <= 65536 - 256
    for H, Hi in [(48, 64), (8, 64), (128, 64), (63, 64), (64, 0), (64, 129)]:
        assert lib.csa_decode(C.byref(cache), None, C.byref(rows), Hi, base, base, H, base, 1.0, base, None, None,
                              base, ws_n, None) == 2, (H, Hi)
        assert lib.csa_step(C.byref(cache), None, C.addressof(ints), C.addressof(ints), 1, base, base, base, None,
                            C.byref(rows), Hi, base, base, H, base, 1.0, base, None, None, base, ws_n, None) == 2
    for H in (48, 8, 128):
        assert lib.csa_sparse_attn(C.byref(cache), None, C.byref(rows), base, H, base, 1.0, base, None, base, 256,
                                   None) == 2, H
    for Hi in (0, 129):
        assert lib.csa_index_score(C.byref(cache), C.byref(rows), Hi, base, base, base, 64, base, ws_n, None) == 2


def test_wait_budget_setter(lib):
    assert lib.csa_set_wait_budget(1000) == 0
    assert lib.csa_set_wait_budget(0) == 0            # back to the default


def test_bad_cache_descriptors(lib):
    buf = (C.c_uint8 * 256)()
    base = C.addressof(buf)
    aligned = (base + 127) & ~127
    pt = (C.c_int32 * 4)()
    cache = csa.CsaCache(aligned, aligned, C.addressof(pt), 1, 1, 1, 3)   # pool ratio 3
    assert lib.csa_append(C.byref(cache), None, C.addressof(pt), C.addressof(pt), 0, None, None, None,
                          None, 0, None) == 1
    cache = csa.CsaCache(aligned + 8, aligned, C.addressof(pt), 1, 1, 1, 2)  # misaligned pool
    assert lib.csa_append(C.byref(cache), None, C.addressof(pt), C.addressof(pt), 0, None, None, None,
                          None, 0, None) == 1


def test_workspace_sizes_without_device(lib):
    assert csa.csa_workspace_size(csa.OP_APPEND, 0, 0, 0) == 256
    assert csa.csa_workspace_size(csa.OP_TOPK, 10, 1000, 0) == 256
    assert csa.csa_workspace_size(csa.OP_INDEX_SCORE, 192, 3000, 64) >= 192 * 128 * 68
    assert csa.csa_workspace_size(99, 1, 1, 1) == 0
    # attention: the status word, plus the tail split's partials only when the
    # rows exceed the device's SM count (none is known without a device)
    for rows, heads in [(1, 64), (4, 64), (30, 16), (128, 64), (200, 64)]:
        assert csa.csa_workspace_size(csa.OP_SPARSE_ATTN, rows, 262144, heads) == 256
    # decode = the score step's workspace + the scores [R, ld] + the top-k [R, 512]
    R, n = 128, 65536
    assert csa.csa_workspace_size(csa.OP_DECODE, R, n, 64) >= (
        csa.csa_workspace_size(csa.OP_INDEX_SCORE, R, n, 64) + 4 * R * n + 4 * R * 512)


def test_empty_calls_return_ok_without_a_launch(lib):
    """Zero rows (and zero tokens) is a valid call that launches nothing: on a
    machine without a GPU any launch would fail with 4 (CUDA error)."""
    buf = (C.c_uint8 * 4096)()
    base = (C.addressof(buf) + 255) & ~255
    pt = (C.c_int32 * 4)()
    ints = (C.c_int32 * 8)()
    cache = csa.CsaCache(base, base, C.addressof(pt), 1, 1, 1, 2)
    rows = csa.CsaRows(0, None, None, 0, 1)
    assert lib.csa_decode(C.byref(cache), None, C.byref(rows), 64, None, None, 64, None, 1.0, None, None, None,
                          None, 0, None) == 0
    assert lib.csa_index_score(C.byref(cache), C.byref(rows), 64, None, None, None, 1, None, 0, None) == 0
    assert lib.csa_sparse_attn(C.byref(cache), None, C.byref(rows), None, 64, None, 1.0, None, None, None, 0,
                               None) == 0
    assert lib.csa_topk(0, None, 512, None, 0, 512, None, None, 0, None) == 0
    assert lib.csa_append(C.byref(cache), None, C.addressof(ints), C.addressof(ints), 0, None, None, base, None, 0,
                          None) == 0
    assert lib.csa_step(C.byref(cache), None, C.addressof(ints), C.addressof(ints), 0, None, None, base, None,
                        C.byref(rows), 64, None, None, 64, None, 1.0, None, None, None, None, 0, None) == 0


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++11")])
def test_header_compiles_as_plain_c_and_cpp(tmp_path, lang, std):
    """include/csa.h is a plain C header (C99, and C++ through extern "C"):
    a host program needs only it and the CUDA runtime's declarations."""
    import shutil
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("no CUDA headers")
    src = tmp_path / ("use." + ("c" if lang == "c" else "cpp"))
    src.write_text('#include "csa.h"\n'
                   'int main(void) { csa_status_t (*f)(const csa_cache_t*, const csa_window_t*, const int32_t*,'
                   ' const int32_t*, int32_t, const void*, const void*, void*, void*, size_t, cudaStream_t)'
                   ' = csa_append; (void)f; return (int)csa_workspace_size(CSA_OP_DECODE, 0, 0, 0) * 0; }\n')
    p = subprocess.run([cc, "-std=" + std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src)],
                       capture_output=True, text=True)
    assert p.returncode == 0, p.stderr


def test_two_level_filter_bounds_before_launch(lib):
    assert lib.csa_topk_two_level(1, None, 512, None, 512, 0, None, None, 0, None) == 2       # blocks < 1
    assert lib.csa_topk_two_level(1, None, 512, None, 512, 129, None, None, 0, None) == 2     # blocks > 128
    assert lib.csa_topk_two_level(1, None, 300000, None, 262145, 8, None, None, 0, None) == 2  # row too long
    assert lib.csa_topk_two_level(1, None, 512, None, 512, 8, None, None, 0, None) == 1       # NULL scores
    assert lib.csa_topk_two_level(0, None, 512, None, 512, 8, None, None, 0, None) == 0       # nothing to do
