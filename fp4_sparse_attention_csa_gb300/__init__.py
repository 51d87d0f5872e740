"""Python binding of libcsa.so, the GB300 CSA decode hot path (include/csa.h).

This module only marshals arguments: torch tensors are passed to the C ABI by
device pointer, on the current CUDA stream.  Every step of the path runs in
the library's CUDA kernels; there is no CPU or PyTorch fallback, and a missing
library raises CsaError.  The function names mirror the C entry points.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import build as _build

_LIB_PATH = _build.LIB
_lock = threading.Lock()
_lib = None

CSA_OK = 0
STATUS_NAMES = {0: "CSA_OK", 1: "CSA_ERR_INVALID_ARGUMENT", 2: "CSA_ERR_UNSUPPORTED",
                3: "CSA_ERR_WORKSPACE_TOO_SMALL", 4: "CSA_ERR_CUDA", 5: "CSA_ERR_DEVICE_FAULT",
                6: "CSA_ERR_TIMEOUT"}
FLAG_PAGE_OOB, FLAG_ROW_INVALID, FLAG_TOPK_OOB, FLAG_TIMEOUT, FLAG_APPEND = 0x1, 0x2, 0x4, 0x8, 0x10
OP_APPEND, OP_INDEX_SCORE, OP_TOPK, OP_SPARSE_ATTN, OP_DECODE = range(5)
D, DI, TOPK, WINDOW, PAGE = 512, 128, 512, 128, 64
KV_PAGE_BYTES, IDX_PAGE_BYTES = 18432, 4352


class CsaError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class CsaCache(C.Structure):
    _fields_ = [("kv_pool", C.c_void_p), ("idx_pool", C.c_void_p), ("page_table", C.c_void_p),
                ("num_pages", C.c_int32), ("num_requests", C.c_int32),
                ("max_pages_per_req", C.c_int32), ("pool_ratio", C.c_int32)]


class CsaWindow(C.Structure):
    _fields_ = [("e4m3", C.c_void_p), ("scale", C.c_void_p), ("capacity", C.c_int32)]


class CsaCompress(C.Structure):
    _fields_ = [("kv_gamma", C.c_void_p), ("idx_gamma", C.c_void_p), ("eps", C.c_float),
                ("rope_cos", C.c_void_p), ("rope_sin", C.c_void_p), ("rope_rows", C.c_int32)]


class CsaOpts(C.Structure):
    _fields_ = [("plan_in", C.c_void_p), ("plan_out", C.c_void_p), ("rope_cos", C.c_void_p),
                ("rope_sin", C.c_void_p), ("rope_rows", C.c_int32), ("candidate_blocks", C.c_int32)]


class CsaRows(C.Structure):
    _fields_ = [("num_rows", C.c_int32), ("row_req", C.c_void_p), ("row_pos", C.c_void_p),
                ("max_entries", C.c_int32), ("max_rows_per_req", C.c_int32)]


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load the in-tree libcsa.so (raises CsaError when it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise CsaError(-1, f"libcsa.so not built at {_LIB_PATH}; run __graft_entry__.build()")
            L = C.CDLL(_LIB_PATH)
            vp, i32, f32, sz = C.c_void_p, C.c_int32, C.c_float, C.c_size_t
            L.csa_workspace_size.argtypes = [i32, i32, i32, i32]
            L.csa_workspace_size.restype = sz
            L.csa_append.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, vp]
            L.csa_append_compress.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp]
            L.csa_index_score.argtypes = [vp, vp, i32, vp, vp, vp, i32, vp, sz, vp]
            L.csa_topk.argtypes = [i32, vp, i32, vp, i32, i32, vp, vp, sz, vp]
            L.csa_sparse_attn.argtypes = [vp, vp, vp, vp, i32, vp, f32, vp, vp, vp, sz, vp]
            L.csa_decode.argtypes = [vp, vp, vp, i32, vp, vp, i32, vp, f32, vp, vp, vp, vp, sz, vp]
            L.csa_index_score_noalloc.argtypes = [vp, vp, i32, vp, vp, vp, i32, vp]
            L.csa_step.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, i32, vp, vp, i32, vp, f32, vp, vp,
                                   vp, vp, sz, vp]
            L.csa_step_ex.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, i32, vp, vp, i32, vp, f32, vp, vp,
                                      vp, vp, vp, sz, vp]
            L.csa_topk_two_level.argtypes = [i32, vp, i32, vp, i32, i32, vp, vp, sz, vp]
            L.csa_sparse_attn_ex.argtypes = [vp, vp, vp, vp, i32, vp, f32, vp, vp, vp, vp, sz, vp]
            L.csa_decode_ex.argtypes = [vp, vp, vp, i32, vp, vp, i32, vp, f32, vp, vp, vp, vp, vp, sz, vp]
            L.csa_check_device_status.argtypes = [vp, vp, C.POINTER(C.c_uint32)]
            L.csa_set_wait_budget.argtypes = [C.c_int64]
            L.csa_status_string.argtypes = [i32]
            L.csa_status_string.restype = C.c_char_p
            for fn in ("csa_append", "csa_append_compress", "csa_index_score", "csa_topk", "csa_sparse_attn",
                       "csa_decode", "csa_step", "csa_index_score_noalloc", "csa_check_device_status",
                       "csa_set_wait_budget", "csa_sparse_attn_ex", "csa_decode_ex", "csa_step_ex",
                       "csa_topk_two_level"):
                getattr(L, fn).restype = C.c_int
            _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(rc, where):
    if rc != CSA_OK:
        raise CsaError(rc, where)


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


# ---- descriptors ------------------------------------------------------------------
def make_cache(kv_pool, idx_pool, page_table, num_pages, pool_ratio):
    return CsaCache(_ptr(kv_pool), _ptr(idx_pool), _ptr(page_table), int(num_pages),
                    int(page_table.shape[0]), int(page_table.shape[1]), int(pool_ratio))


def make_window(e4m3, scale, capacity):
    return CsaWindow(_ptr(e4m3), _ptr(scale), int(capacity))


def make_rows(row_req, row_pos, max_entries, max_rows_per_req):
    return CsaRows(int(row_req.numel()), _ptr(row_req), _ptr(row_pos), int(max_entries), int(max_rows_per_req))


# ---- entry points (same names as the C ABI) ----------------------------------------
def csa_workspace_size(op, num_rows, max_entries, n_heads):
    return int(lib().csa_workspace_size(op, num_rows, max_entries, n_heads))


def make_compress(kv_gamma=None, idx_gamma=None, eps=1e-6, rope_cos=None, rope_sin=None):
    """Compressor-step arguments of csa_append_compress (fp32 device tensors;
    rope tables [rows, 32])."""
    rows = 0 if rope_cos is None else int(rope_cos.shape[0])
    return CsaCompress(_ptr(kv_gamma), _ptr(idx_gamma), float(eps), _ptr(rope_cos), _ptr(rope_sin), rows)


def csa_append_compress(cache, window, pos0, tok_off, total_tokens, kv_in, idx_in, pending, compress, ws=None,
                        stream=None):
    rc = lib().csa_append_compress(C.byref(cache), C.byref(window) if window is not None else None, _ptr(pos0),
                                   _ptr(tok_off), int(total_tokens), _ptr(kv_in), _ptr(idx_in), _ptr(pending),
                                   C.byref(compress), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_append_compress")


def csa_append(cache, window, pos0, tok_off, total_tokens, kv_in, idx_in, pending, ws=None, stream=None):
    rc = lib().csa_append(C.byref(cache), C.byref(window) if window is not None else None, _ptr(pos0),
                          _ptr(tok_off), int(total_tokens), _ptr(kv_in), _ptr(idx_in), _ptr(pending),
                          _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_append")


def csa_index_score(cache, rows, n_idx_heads, q_idx, w, scores, ld, ws, stream=None):
    rc = lib().csa_index_score(C.byref(cache), C.byref(rows), int(n_idx_heads), _ptr(q_idx), _ptr(w),
                               _ptr(scores), int(ld), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_index_score")


def csa_index_score_noalloc(cache, rows, n_idx_heads, q_idx, w, scores, ld, stream=None):
    """csa_index_score with the library's fixed scratch array (no workspace)."""
    rc = lib().csa_index_score_noalloc(C.byref(cache), C.byref(rows), int(n_idx_heads), _ptr(q_idx), _ptr(w),
                                       _ptr(scores), int(ld), _stream(stream))
    _check(rc, "csa_index_score_noalloc")


def csa_topk(num_rows, scores, ld, n_valid, max_n, k, out_idx, ws=None, stream=None):
    rc = lib().csa_topk(int(num_rows), _ptr(scores), int(ld), _ptr(n_valid), int(max_n), int(k),
                        _ptr(out_idx), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_topk")


def csa_topk_two_level(num_rows, scores, ld, n_valid, max_n, blocks, out_idx, ws=None, stream=None):
    rc = lib().csa_topk_two_level(int(num_rows), _ptr(scores), int(ld), _ptr(n_valid), int(max_n), int(blocks),
                                  _ptr(out_idx), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_topk_two_level")


def csa_sparse_attn(cache, window, rows, topk_idx, n_heads, q, softmax_scale, out, lse, ws, stream=None):
    rc = lib().csa_sparse_attn(C.byref(cache), C.byref(window) if window is not None else None,
                               C.byref(rows), _ptr(topk_idx), int(n_heads), _ptr(q), float(softmax_scale),
                               _ptr(out), _ptr(lse), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_sparse_attn")


def make_opts(plan_in=None, plan_out=None, rope_cos=None, rope_sin=None, candidate_blocks=0):
    """Options of the selection and attention steps: plans [R, 512] int32,
    rotary tables [rows, 32] fp32, two-level candidate blocks (0: flat)."""
    rows = 0 if rope_cos is None else int(rope_cos.shape[0])
    return CsaOpts(_ptr(plan_in), _ptr(plan_out), _ptr(rope_cos), _ptr(rope_sin), rows, int(candidate_blocks))


def _opt(o):
    return C.byref(o) if o is not None else None


def csa_sparse_attn_ex(cache, window, rows, topk_idx, n_heads, q, softmax_scale, out, lse, opts, ws, stream=None):
    rc = lib().csa_sparse_attn_ex(C.byref(cache), C.byref(window) if window is not None else None,
                                  C.byref(rows), _ptr(topk_idx), int(n_heads), _ptr(q), float(softmax_scale),
                                  _ptr(out), _ptr(lse), _opt(opts), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_sparse_attn_ex")


def csa_decode_ex(cache, window, rows, n_idx_heads, q_idx, w, n_heads, q, softmax_scale, out, lse, topk_out, opts,
                  ws, stream=None):
    rc = lib().csa_decode_ex(C.byref(cache), C.byref(window) if window is not None else None, C.byref(rows),
                             int(n_idx_heads), _ptr(q_idx), _ptr(w), int(n_heads), _ptr(q), float(softmax_scale),
                             _ptr(out), _ptr(lse), _ptr(topk_out), _opt(opts), _ptr(ws), _nbytes(ws),
                             _stream(stream))
    _check(rc, "csa_decode_ex")


def csa_step_ex(cache, window, pos0, tok_off, total_tokens, kv_in, idx_in, pending, compress, rows, n_idx_heads,
                q_idx, w, n_heads, q, softmax_scale, out, lse, topk_out, opts, ws, stream=None):
    rc = lib().csa_step_ex(C.byref(cache), C.byref(window) if window is not None else None, _ptr(pos0),
                           _ptr(tok_off), int(total_tokens), _ptr(kv_in), _ptr(idx_in), _ptr(pending),
                           C.byref(compress) if compress is not None else None, C.byref(rows), int(n_idx_heads),
                           _ptr(q_idx), _ptr(w), int(n_heads), _ptr(q), float(softmax_scale), _ptr(out), _ptr(lse),
                           _ptr(topk_out), _opt(opts), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_step_ex")


def csa_decode(cache, window, rows, n_idx_heads, q_idx, w, n_heads, q, softmax_scale, out, lse, topk_out, ws,
               stream=None):
    rc = lib().csa_decode(C.byref(cache), C.byref(window) if window is not None else None, C.byref(rows),
                          int(n_idx_heads), _ptr(q_idx), _ptr(w), int(n_heads), _ptr(q), float(softmax_scale),
                          _ptr(out), _ptr(lse), _ptr(topk_out), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_decode")


def csa_step(cache, window, pos0, tok_off, total_tokens, kv_in, idx_in, pending, compress, rows, n_idx_heads,
             q_idx, w, n_heads, q, softmax_scale, out, lse, topk_out, ws, stream=None):
    """csa_append(_compress) then csa_decode in one call (compress may be None)."""
    rc = lib().csa_step(C.byref(cache), C.byref(window) if window is not None else None, _ptr(pos0),
                        _ptr(tok_off), int(total_tokens), _ptr(kv_in), _ptr(idx_in), _ptr(pending),
                        C.byref(compress) if compress is not None else None, C.byref(rows), int(n_idx_heads),
                        _ptr(q_idx), _ptr(w), int(n_heads), _ptr(q), float(softmax_scale), _ptr(out), _ptr(lse),
                        _ptr(topk_out), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "csa_step")


def csa_check_device_status(ws, stream=None):
    """Synchronises the stream; returns (status, flags) and clears the flags.
    ws=None reads the status word of csa_index_score_noalloc's fixed array."""
    flags = C.c_uint32(0)
    rc = lib().csa_check_device_status(_ptr(ws), _stream(stream), C.byref(flags))
    return int(rc), int(flags.value)


def csa_set_wait_budget(sm_clocks):
    """Bound (in SM clocks) on each wait of the index score's pipeline; <= 0
    restores the default.  Process-wide."""
    _check(lib().csa_set_wait_budget(int(sm_clocks)), "csa_set_wait_budget")


def csa_status_string(status):
    return lib().csa_status_string(int(status)).decode()
