"""Independent brute-force restatements used to pin the oracle.

Nothing here is imported from the oracle or the CUDA library.  Code tables are
derived from the bit-level definitions of the formats ([OCP] MX v1.0 for E2M1
and E8M0, OCP FP8 for E4M3), rounding is a nearest-value search in exact
rational arithmetic, and the block scale rules are re-derived from their
definitions.  Everything is pure Python (plus numpy/torch fp64 for the dense
checks), slow, and meant for tiny inputs only.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


# ---- code tables from the bit layouts ----------------------------------------
def e2m1_value(code: int) -> Fraction:
    """E2M1: sign | 2 exponent bits (bias 1) | 1 mantissa bit; no inf/NaN."""
    code = int(code)
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return -v if s else v


def e4m3_value(code: int):
    """E4M3 "fn": sign | 4 exponent bits (bias 7) | 3 mantissa bits; S.1111.111 = NaN."""
    code = int(code)
    s, e, m = (code >> 7) & 1, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return None
    v = Fraction(m, 8) * Fraction(2) ** (-6) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def e8m0_value(code: int):
    code = int(code)
    return None if code == 255 else Fraction(2) ** (code - 127)


# ---- nearest-value rounding with ties to the even code -----------------------
def nearest_code(x: Fraction, codes_values):
    """Codes are (code, value) with value >= 0, sorted by value; returns the
    code of the nearest value, ties to the even code, saturating at the top."""
    best = None
    for c, v in codes_values:
        d = abs(x - v)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


E2M1_POS = [(c, e2m1_value(c)) for c in range(8)]
E4M3_POS = [(c, e4m3_value(c)) for c in range(127)]   # finite, non-negative


def e2m1_encode(x: float) -> int:
    f = Fraction(x)
    mag = nearest_code(abs(f), E2M1_POS)
    return mag | (8 if math.copysign(1.0, x) < 0 else 0)


def e4m3_encode(x: float) -> int:
    f = Fraction(x)
    mag = 126 if abs(f) >= 448 else nearest_code(abs(f), E4M3_POS)
    return mag | (0x80 if math.copysign(1.0, x) < 0 else 0)


def f32(x) -> float:
    return float(np.float32(x))


# ---- block quantisers, re-derived ----------------------------------------------
def nvfp4_block(x16):
    """Scale = E4M3(fp32(amax / 6)); codes = e2m1(fp32(x / s)); s == 0 -> all 0."""
    xs = [f32(v) for v in x16]
    amax = max(abs(v) for v in xs)
    sf = float(np.float32(amax) / np.float32(6.0))
    S = e4m3_encode(sf)
    s = float(e4m3_value(S))
    if s == 0:
        return [0] * 16, S
    return [e2m1_encode(float(np.float32(v) / np.float32(s))) for v in xs], S


def mxfp4_block(x32):
    """MX rule: X = 2^(floor(log2 amax) - emax(E2M1)=2); codes = e2m1(x / X)."""
    xs = [Fraction(f32(v)) for v in x32]
    amax = max(abs(v) for v in xs)
    if amax == 0:
        return [0] * 32, 0
    e = 0                                   # exact floor(log2 amax) by search
    while Fraction(2) ** (e + 1) <= amax:
        e += 1
    while Fraction(2) ** e > amax:
        e -= 1
    E = max(-127, min(127, e - 2))
    X = Fraction(2) ** E
    codes = []
    for v, raw in zip(xs, x32):
        q = v / X
        mag = nearest_code(abs(q), E2M1_POS)
        codes.append(mag | (8 if math.copysign(1.0, f32(raw)) < 0 else 0))
    return codes, E + 127


# ---- score, top-k and attention on tiny inputs ----------------------------------
def dequant_fp4(codes, scales, block):
    return np.array([float(e2m1_value(c)) * float(scales[i // block]) for i, c in enumerate(codes)],
                    dtype=np.float64)


def score_fp64(qhat, khat, w):
    """score_i = sum_h w_h relu(q_h . k_i), all in fp64."""
    dots = qhat @ khat.T                         # [Hi, n]
    return (w[:, None] * np.maximum(dots, 0.0)).sum(axis=0)


def topk_sorted(scores, k=512):
    order = sorted(range(len(scores)), key=lambda i: (-scores[i], i))
    sel = sorted(order[:k])
    return sel + [-1] * (k - len(sel))


def dense_attention_fp64(q, keys, scale):
    """q [H, D], keys [n, D] (K = V); softmax attention in fp64 via torch."""
    import torch
    qt = torch.tensor(q, dtype=torch.float64)
    kt = torch.tensor(keys, dtype=torch.float64)
    logits = scale * qt @ kt.T
    p = torch.softmax(logits, dim=-1)
    out = p @ kt
    lse = torch.logsumexp(logits, dim=-1)
    return out.numpy(), lse.numpy(), p.numpy()
