"""Parity judgement rules shared by the GPU tests (comparisons only).

J-1  cache bytes: equal, byte for byte.
J-2  top-512 sets: with s* the oracle's 512th-largest score,
       A   = {i : s_i > s* (1 + 1e-4)}           (must all be selected)
       Bnd = {i : |s_i - s*| <= 1e-4 |s*|}        (may be selected)
     required  A <= GPU <= A u Bnd  and |GPU| = min(512, n); the output is in
     ascending index order and padded with -1.  When s* == 0 the lowest
     indices win, which pins the result.
J-3  attention: per (row, head) vector,
       |o_gpu - o_ref| <= 2e-3 * max|o_ref| + half an ulp of bf16 at o_ref
     (the second term is the unavoidable rounding of a bf16 output), and
     |lse_gpu - lse_ref| <= 1e-4.
"""
import numpy as np

REL_BAND = 1e-4
ATTN_TOL = 2e-3
LSE_TOL = 1e-4


def check_topk_row(gpu_row, scores, n, k=512):
    gpu_row = np.asarray(gpu_row)
    m = min(k, n)
    sel = gpu_row[:m]
    assert (gpu_row[m:] == -1).all(), "padding must be -1"
    assert (sel >= 0).all() and (sel < n).all(), "index outside the visible range"
    assert (np.diff(sel) > 0).all(), "indices must be strictly ascending"
    if n <= k:
        assert np.array_equal(sel, np.arange(n))
        return 0
    s = scores[:n].astype(np.float64)
    order = np.lexsort((np.arange(n), -s))
    s_star = s[order[k - 1]]
    band = REL_BAND * abs(s_star)
    A = set(np.nonzero(s > s_star + band)[0].tolist())
    Bnd = set(np.nonzero(np.abs(s - s_star) <= band)[0].tolist())
    G = set(sel.tolist())
    assert A <= G, f"{len(A - G)} entries above the band missing"
    assert G <= (A | Bnd), f"{len(G - A - Bnd)} entries below the band selected"
    if s_star == 0.0:
        assert np.array_equal(sel, np.sort(order[:k]))
    return len(G - set(order[:k].tolist()))      # picks that differ inside the band


def bf16_half_ulp(x):
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 0.5 * np.exp2(e - 7), 0.0)


def check_attention(out_gpu, out_ref, lse_gpu=None, lse_ref=None):
    """out_* [..., 512]; returns (max normalised error, relative L2)."""
    g = np.asarray(out_gpu, np.float64)
    r = np.asarray(out_ref, np.float64)
    scale = np.abs(r).max(axis=-1, keepdims=True)
    bound = ATTN_TOL * scale + bf16_half_ulp(r)
    err = np.abs(g - r)
    bad = ~(err <= bound)                    # a NaN output counts as beyond tolerance
    assert not bad.any(), f"{int(bad.sum())} elements beyond tolerance; worst excess {float(np.nanmax(err - bound)):.3e}"
    if lse_gpu is not None:
        le = np.abs(np.asarray(lse_gpu, np.float64) - np.asarray(lse_ref, np.float64))
        assert float(le.max()) <= LSE_TOL, f"lse error {float(le.max()):.3e}"
    norm = float((err / np.maximum(scale, 1e-30)).max())
    rel_l2 = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    return norm, rel_l2
