"""ctypes front end of the CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its Python binding)
never loads it.  The oracle itself is plain C (csa_oracle.c), built here with
gcc at -O2 -ffp-contract=off, no fast-math.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csa_oracle.c")
HDR = os.path.join(HERE, "csa_oracle.h")
LIB = os.path.join(HERE, "liboracle.so")

KV_PAGE, IDX_PAGE, D, DI, TOPK, WINDOW = 18432, 4352, 512, 128, 512, 128

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, fp32 strict) if missing or stale."""
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(LIB)
            u8, f32, i32, i64 = C.c_uint8, C.c_float, C.c_int32, C.c_int64
            vp = C.c_void_p
            L.or_e2m1_decode.argtypes, L.or_e2m1_decode.restype = [u8], f32
            L.or_e2m1_encode.argtypes, L.or_e2m1_encode.restype = [f32], u8
            L.or_e4m3_decode.argtypes, L.or_e4m3_decode.restype = [u8], f32
            L.or_e4m3_encode.argtypes, L.or_e4m3_encode.restype = [f32], u8
            L.or_e8m0_decode.argtypes, L.or_e8m0_decode.restype = [u8], f32
            L.or_e8m0_block_code.argtypes, L.or_e8m0_block_code.restype = [f32], u8
            for fn in ("or_nvfp4_block", "or_mxfp4_block"):
                getattr(L, fn).argtypes = [vp, vp, vp]
                getattr(L, fn).restype = None
            for fn in ("or_quant_main_entry", "or_quant_idx_entry", "or_quant_window_token"):
                getattr(L, fn).argtypes = [vp, vp, vp]
                getattr(L, fn).restype = None
            L.or_append.argtypes = [vp, vp, vp, vp, vp, vp, vp]
            L.or_append_compress.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
            L.or_append_compress.restype = C.c_int
            L.or_compress_vec.argtypes = [vp, C.c_int, vp, f32, vp, vp]
            L.or_compress_vec.restype = None
            L.or_append.restype = C.c_int
            L.or_index_score.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, i64]
            L.or_index_score.restype = None
            L.or_topk_row.argtypes = [vp, i32, vp]
            L.or_topk_row.restype = None
            L.or_attention_row.argtypes = [vp, i32, i32, vp, i32, vp, f32, vp, vp]
            L.or_attention_row.restype = None
            L.or_topk_two_level.argtypes = [vp, i32, i32, vp]
            L.or_topk_two_level.restype = None
            L.or_attention_row_rope.argtypes = [vp, i32, i32, vp, i32, vp, f32, vp, vp, i32, vp, vp]
            L.or_attention_row_rope.restype = C.c_int
            L.or_decode.argtypes = [vp, i32, vp, vp, i32, vp, vp, i32, vp, f32, vp, vp, vp, vp, i64, i32]
            L.or_decode.restype = None
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---- scalar codes ------------------------------------------------------------
def e2m1_decode(c): return lib().or_e2m1_decode(int(c))
def e2m1_encode(v): return lib().or_e2m1_encode(float(v))
def e4m3_decode(c): return lib().or_e4m3_decode(int(c))
def e4m3_encode(v): return lib().or_e4m3_encode(float(v))
def e8m0_decode(c): return lib().or_e8m0_decode(int(c))
def e8m0_block_code(a): return lib().or_e8m0_block_code(float(a))


def nvfp4_block(x16):
    x = _c(x16, np.float32)
    assert x.size == 16
    codes, sc = np.zeros(16, np.uint8), np.zeros(1, np.uint8)
    lib().or_nvfp4_block(_p(x), _p(codes), _p(sc))
    return codes, int(sc[0])


def mxfp4_block(x32):
    x = _c(x32, np.float32)
    assert x.size == 32
    codes, sc = np.zeros(32, np.uint8), np.zeros(1, np.uint8)
    lib().or_mxfp4_block(_p(x), _p(codes), _p(sc))
    return codes, int(sc[0])


def quant_main_entry(x512):
    x = _c(x512, np.float32)
    data, sc = np.zeros(256, np.uint8), np.zeros(32, np.uint8)
    lib().or_quant_main_entry(_p(x), _p(data), _p(sc))
    return data, sc


def quant_idx_entry(y128):
    y = _c(y128, np.float32)
    data, sc = np.zeros(64, np.uint8), np.zeros(4, np.uint8)
    lib().or_quant_idx_entry(_p(y), _p(data), _p(sc))
    return data, sc


def quant_window_token(x512):
    x = _c(x512, np.float32)
    codes, sc = np.zeros(512, np.uint8), np.zeros(1, np.float32)
    lib().or_quant_window_token(_p(x), _p(codes), _p(sc))
    return codes, float(sc[0])


# ---- cache -------------------------------------------------------------------
class _CacheStruct(C.Structure):
    _fields_ = [("kv_pool", C.c_void_p), ("idx_pool", C.c_void_p), ("page_table", C.c_void_p),
                ("num_pages", C.c_int32), ("num_requests", C.c_int32),
                ("max_pages_per_req", C.c_int32), ("pool_ratio", C.c_int32),
                ("win_codes", C.c_void_p), ("win_scale", C.c_void_p), ("win_cap", C.c_int32)]


class _CompressStruct(C.Structure):
    _fields_ = [("kv_gamma", C.c_void_p), ("idx_gamma", C.c_void_p), ("eps", C.c_float),
                ("rope_cos", C.c_void_p), ("rope_sin", C.c_void_p), ("rope_rows", C.c_int32)]


def compress_vec(v, gamma=None, eps=1e-6, cos32=None, sin32=None):
    """RMSNorm + rotate-half RoPE of one pooled vector (512 or 128 values),
    as the compressor applies it before quantisation; returns a new array."""
    v = np.array(v, dtype=np.float32, copy=True)
    g = None if gamma is None else _c(gamma, np.float32)
    cs = None if cos32 is None else _c(cos32, np.float32)
    sn = None if sin32 is None else _c(sin32, np.float32)
    lib().or_compress_vec(_p(v), int(v.size), _p(g), float(eps), _p(cs), _p(sn))
    return v


class Cache:
    """The oracle's own copy of the paged FP4 cache, FP8 window and pending tokens."""

    def __init__(self, num_pages, page_table, pool_ratio, win_cap=256, window=True):
        self.page_table = _c(page_table, np.int32)
        self.B, self.max_pages = self.page_table.shape
        self.num_pages = int(num_pages)
        self.P = int(pool_ratio)
        self.win_cap = int(win_cap)
        self.kv_pool = np.zeros(self.num_pages * KV_PAGE, np.uint8)
        self.idx_pool = np.zeros(self.num_pages * IDX_PAGE, np.uint8)
        self.win_codes = np.zeros(self.B * self.win_cap * D, np.uint8) if window else None
        self.win_scale = np.zeros(self.B * self.win_cap, np.float32) if window else None
        self.pending = np.zeros((self.B, D + DI), np.uint16)

    def struct(self, window=True):
        w = window and self.win_codes is not None
        return _CacheStruct(self.kv_pool.ctypes.data, self.idx_pool.ctypes.data,
                            self.page_table.ctypes.data, self.num_pages, self.B, self.max_pages,
                            self.P, self.win_codes.ctypes.data if w else None,
                            self.win_scale.ctypes.data if w else None, self.win_cap)

    def append(self, pos0, tok_off, kv_in, idx_in, window=True, compress=None):
        """Append tokens (bf16 bits) for all requests; pending is updated in place.
        compress: None, or a dict with any of kv_gamma [512], idx_gamma [128],
        eps, rope_cos / rope_sin [rows, 32] (fp32) for the compressor steps."""
        pos0, tok_off = _c(pos0, np.int32), _c(tok_off, np.int32)
        kv_in, idx_in = _c(kv_in, np.uint16), _c(idx_in, np.uint16)
        s = self.struct(window)
        if compress is None:
            return lib().or_append(C.byref(s), _p(pos0), _p(tok_off), _p(kv_in), _p(idx_in),
                                   _p(self.pending), _p(self.pending))
        keep = {k: (None if compress.get(k) is None else _c(compress[k], np.float32))
                for k in ("kv_gamma", "idx_gamma", "rope_cos", "rope_sin")}
        rows = 0 if keep["rope_cos"] is None else int(keep["rope_cos"].shape[0])
        cs = _CompressStruct(_p(keep["kv_gamma"]), _p(keep["idx_gamma"]), float(compress.get("eps", 1e-6)),
                             _p(keep["rope_cos"]), _p(keep["rope_sin"]), rows)
        return lib().or_append_compress(C.byref(s), _p(pos0), _p(tok_off), _p(kv_in), _p(idx_in),
                                        _p(self.pending), _p(self.pending), C.byref(cs))

    def main_entry(self, b, e):
        page = int(self.page_table[b, e // 64])
        base = page * KV_PAGE
        return (self.kv_pool[base + (e % 64) * 256: base + (e % 64) * 256 + 256],
                self.kv_pool[base + 16384 + (e % 64) * 32: base + 16384 + (e % 64) * 32 + 32])

    def idx_entry(self, b, e):
        """(data[64], scales[4]) of indexer entry e: 8-entry groups of 544 B,
        data byte k of slot 8g+r at 544g + 128(k//16) + 16r + k%16, scale byte
        j at 544g + 512 + 4r + j."""
        page = int(self.page_table[b, e // 64])
        base = page * IDX_PAGE + 544 * ((e % 64) // 8)
        r = (e % 64) % 8
        k = np.arange(64)
        data = self.idx_pool[base + 128 * (k // 16) + 16 * r + k % 16]
        sc = self.idx_pool[base + 512 + 4 * r + np.arange(4)]
        return data, sc

    def window_slot(self, b, p):
        s = b * self.win_cap + p % self.win_cap
        return self.win_codes[s * D:(s + 1) * D], float(self.win_scale[s])


def index_score(cache, row_req, row_pos, q_idx, w, ld=None):
    row_req, row_pos = _c(row_req, np.int32), _c(row_pos, np.int32)
    q_idx, w = _c(q_idx, np.uint16), _c(w, np.float32)
    R, Hi = w.shape
    n = (row_pos.astype(np.int64) + 1) // cache.P
    ld = int(ld or max(int(n.max()) if R else 1, 1))
    scores = np.full((R, ld), np.nan, np.float32)
    s = cache.struct()
    lib().or_index_score(C.byref(s), R, _p(row_req), _p(row_pos), Hi, _p(q_idx), _p(w),
                         _p(scores), ld)
    return scores


def topk_row(scores, n):
    sc = _c(scores[:n], np.float32)
    out = np.zeros(TOPK, np.int32)
    lib().or_topk_row(_p(sc), int(n), _p(out))
    return out


def topk_two_level(scores, n, blocks):
    """Two-level candidate filter: top `blocks` pages of 64 by their largest
    score, then the exact top-512 among their entries."""
    sc = _c(scores[:n], np.float32)
    out = np.zeros(TOPK, np.int32)
    lib().or_topk_two_level(_p(sc), int(n), int(blocks), _p(out))
    return out


def attention_row(cache, req, pos, topk, q_row, softmax_scale):
    topk, q_row = _c(topk, np.int32), _c(q_row, np.uint16)
    H = q_row.size // D
    out, lse = np.zeros((H, D), np.float32), np.zeros(H, np.float32)
    s = cache.struct()
    lib().or_attention_row(C.byref(s), int(req), int(pos), _p(topk), H, _p(q_row),
                           float(softmax_scale), _p(out), _p(lse))
    return out, lse


def attention_row_rope(cache, req, pos, topk, q_row, softmax_scale, rope_cos, rope_sin):
    """attention_row with the query (row position) and the window tokens (their
    positions) rotated by the tables; returns (out, lse, rc)."""
    topk, q_row = _c(topk, np.int32), _c(q_row, np.uint16)
    cs, sn = _c(rope_cos, np.float32), _c(rope_sin, np.float32)
    H = q_row.size // D
    out, lse = np.zeros((H, D), np.float32), np.zeros(H, np.float32)
    s = cache.struct()
    rc = lib().or_attention_row_rope(C.byref(s), int(req), int(pos), _p(topk), H, _p(q_row),
                                     float(softmax_scale), _p(cs), _p(sn), int(cs.shape[0]), _p(out), _p(lse))
    return out, lse, int(rc)


def decode(cache, row_req, row_pos, q_idx, w, q, softmax_scale, threads=1):
    """score -> top-512 -> attention for every row; returns (out, lse, topk, scores)."""
    row_req, row_pos = _c(row_req, np.int32), _c(row_pos, np.int32)
    q_idx, w, q = _c(q_idx, np.uint16), _c(w, np.float32), _c(q, np.uint16)
    R, Hi = w.shape
    H = q.shape[1]
    n = (row_pos.astype(np.int64) + 1) // cache.P
    ld = max(int(n.max()) if R else 1, 1)
    scores = np.full((R, ld), np.nan, np.float32)
    out = np.zeros((R, H, D), np.float32)
    lse = np.zeros((R, H), np.float32)
    topk = np.zeros((R, TOPK), np.int32)
    s = cache.struct()
    lib().or_decode(C.byref(s), R, _p(row_req), _p(row_pos), Hi, _p(q_idx), _p(w), H, _p(q),
                    float(softmax_scale), _p(out), _p(lse), _p(topk), _p(scores), ld, int(threads))
    return out, lse, topk, scores


def build_cache(wl, requests=None, upto="ctx", window=True, threads=1):
    """Build the oracle cache of workload `wl` from its seeded tokens.

    upto="ctx": all tokens (history + the step's new ones);
    upto="hist": history only (the step's append is then done separately).
    Only `requests` (default: all) are filled.  Tokens older than the window
    are appended without the window write, which leaves the same state (the
    ring keeps only the last win_cap positions) at a fraction of the cost.
    Requests own disjoint pages, so they are built in parallel when
    threads > 1.
    """
    reqs = list(range(wl.B)) if requests is None else list(requests)
    cache = Cache(wl.num_pages, wl.page_table, wl.P, wl.win_cap, window=window)

    def one(b):
        stop = int(wl.ctx_len[b] if upto == "ctx" else wl.hist_len[b])
        cut = max(0, stop - wl.win_cap) if window else stop
        for lo, hi, win in ((0, cut, False), (cut, stop, window)):
            for c0 in range(lo, hi, 8192):
                c1 = min(hi, c0 + 8192)
                x, y = wl.tokens(b, c0, c1)
                pos0 = np.zeros(wl.B, np.int32)
                pos0[b] = c0
                tok_off = np.zeros(wl.B + 1, np.int32)
                tok_off[b + 1:] = c1 - c0
                rc = cache.append(pos0, tok_off, x, y, window=win)
                assert rc == 0, rc

    if threads > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, reqs))
    else:
        for b in reqs:
            one(b)
    return cache
