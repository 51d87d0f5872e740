"""Seeded synthetic workloads for the CSA decode path.

This module only draws random numbers and lays out shapes: token latents,
indexer keys, queries, head weights, context lengths, page tables and the row
metadata of one decode step.  It holds none of the method's arithmetic (no
pooling, quantisation, scoring or attention), so both the CUDA path and the
CPU oracle can take their inputs from it.

Shapes follow the workloads the pages describe:
  * [SGL] "DeepSeek-V4.1 Flash on SGLang: from 35 to 873 tokens/s":
    "DSpark adaptation and optimization" (verify handles up to 6 rows per
    request: anchor + block of 5) and "How to reproduce" (random 4k/1k);
    "Architecture changes and KV cache compression" (2:1 pooled caches and one
    unpooled cache, top 512 global positions).
  * [VLLM] "DeepSeek-V4.1-Flash runs 5.3x faster on vLLM...": "SWA bounded
    replay" (128-position FP8 window).

Every random stream is keyed by a numpy SeedSequence built from the workload
seed and a purpose tag, so any request's tokens can be regenerated on their
own (the oracle only rebuilds the requests it checks).

bf16 values are carried as uint16 bit patterns (numpy has no bf16 dtype);
fp32 draws are rounded to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

D = 512          # main latent width
DI = 128         # indexer key width
PAGE = 64        # entries per page
CHUNK = 4096     # tokens per independently seeded generation chunk

# purpose tags for the seed streams
_TAG_LEN, _TAG_TOK, _TAG_STEP, _TAG_SAL, _TAG_PERM, _TAG_TIE = range(6)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    """One decode step of one CSA layer over a batch of requests.

    Request b holds ctx_len[b] tokens at positions 0..ctx_len[b]-1.  The step
    appends its last new_tok[b] tokens and decodes one query row at each of
    those positions, so rows of a request are contiguous and ordered by
    position (row_req is non-decreasing).
    """
    name: str
    seed: int
    B: int
    H: int
    Hi: int
    P: int
    ctx_len: np.ndarray          # int64 [B]
    new_tok: np.ndarray          # int32 [B]
    page_table: np.ndarray       # int32 [B, max_pages]; unused slots = -1
    num_pages: int
    win_cap: int = 256
    softmax_scale: float = 1.0 / math.sqrt(D)
    salient_scale: float = 4.0
    salient_frac: float = 0.0    # fraction of entries whose tokens are scaled
    tie: dict = field(default_factory=dict)   # config with constructed ties

    # ---- derived shapes ---------------------------------------------------
    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def hist_len(self) -> np.ndarray:
        return (self.ctx_len - self.new_tok).astype(np.int64)

    @property
    def R(self) -> int:
        return int(self.new_tok.sum())

    @property
    def row_req(self) -> np.ndarray:
        return np.repeat(np.arange(self.B, dtype=np.int32), self.new_tok)

    @property
    def row_pos(self) -> np.ndarray:
        out = [np.arange(h, h + t, dtype=np.int32) for h, t in zip(self.hist_len, self.new_tok)]
        return np.concatenate(out) if out else np.zeros(0, np.int32)

    @property
    def step_tok_off(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.new_tok)]).astype(np.int32)

    @property
    def step_pos0(self) -> np.ndarray:
        return self.hist_len.astype(np.int32)

    def entries(self, b: int) -> int:
        """Entries of request b once the step's tokens are appended."""
        return int(self.ctx_len[b]) // self.P

    def row_entries(self) -> np.ndarray:
        return ((self.row_pos.astype(np.int64) + 1) // self.P).astype(np.int32)

    @property
    def max_entries(self) -> int:
        return int(self.row_entries().max()) if self.R else 0

    # ---- random tensors -----------------------------------------------------
    def _salient_entries(self, b: int) -> np.ndarray:
        n = self.entries(b)
        k = int(round(self.salient_frac * n))
        if k == 0:
            return np.zeros(0, np.int64)
        return np.sort(_rng(self.seed, _TAG_SAL, b).choice(n, size=k, replace=False))

    def _tie_sets(self, b: int):
        n = self.entries(b)
        g, s = self.tie["group"], self.tie["salient"]
        pick = _rng(self.seed, _TAG_TIE, b).choice(n, size=g + s, replace=False)
        src = _rng(self.seed, _TAG_TIE, b, 1).standard_normal(DI, dtype=np.float32)
        return np.sort(pick[:g]), np.sort(pick[g:]), src

    def tokens(self, b: int, start: int, stop: int):
        """bf16 bits of tokens [start, stop) of request b: (x [n,512], y [n,128])."""
        xs, ys = [], []
        if stop <= start:
            return np.zeros((0, D), np.uint16), np.zeros((0, DI), np.uint16)
        sal = self._salient_entries(b) if self.salient_frac > 0 else None
        ties = self._tie_sets(b) if self.tie else None
        for c in range(start // CHUNK, (stop - 1) // CHUNK + 1):
            lo, hi = c * CHUNK, (c + 1) * CHUNK
            g = _rng(self.seed, _TAG_TOK, b, c)
            x = g.standard_normal((CHUNK, D), dtype=np.float32)
            y = g.standard_normal((CHUNK, DI), dtype=np.float32)
            tok = np.arange(lo, hi, dtype=np.int64)
            if sal is not None and sal.size:
                m = np.isin(tok // self.P, sal)
                x[m] *= np.float32(self.salient_scale)
                y[m] *= np.float32(self.salient_scale)
            if ties is not None:
                grp, hot, src = ties
                y[np.isin(tok // self.P, hot)] *= np.float32(self.tie["salient_scale"])
                y[np.isin(tok // self.P, grp)] = src * np.float32(self.tie["group_scale"])
            a, z = max(start, lo) - lo, min(stop, hi) - lo
            xs.append(x[a:z])
            ys.append(y[a:z])
        return f32_to_bf16_bits(np.concatenate(xs)), f32_to_bf16_bits(np.concatenate(ys))

    def step_queries(self):
        """q_idx bf16 [R,Hi,128], w fp32 [R,Hi] ~ U(0,1), q bf16 [R,H,512]."""
        g = _rng(self.seed, _TAG_STEP)
        R = self.R
        q_idx = f32_to_bf16_bits(g.standard_normal((R, self.Hi, DI), dtype=np.float32))
        w = g.random((R, self.Hi), dtype=np.float32)
        q = f32_to_bf16_bits(g.standard_normal((R, self.H, D), dtype=np.float32))
        return q_idx, w, q

    def step_tokens(self):
        """The step's new tokens, concatenated by request: (x [T,512], y [T,128])."""
        xs, ys = [], []
        for b in range(self.B):
            x, y = self.tokens(b, int(self.hist_len[b]), int(self.ctx_len[b]))
            xs.append(x)
            ys.append(y)
        return np.concatenate(xs), np.concatenate(ys)


def _pages(ctx_len: np.ndarray, P: int, shuffle_seed: int | None):
    ent = ctx_len // P
    npg = (ent + PAGE - 1) // PAGE
    max_pages = max(int(npg.max()), 1)
    num_pages = int(npg.sum())
    ids = np.arange(num_pages, dtype=np.int32)
    if shuffle_seed is not None:
        ids = _rng(shuffle_seed, _TAG_PERM).permutation(num_pages).astype(np.int32)
    pt = np.full((len(ctx_len), max_pages), -1, np.int32)
    o = 0
    for b, k in enumerate(npg):
        pt[b, :k] = ids[o:o + k]
        o += int(k)
    return pt, max(num_pages, 1)


def custom(name: str, seed: int, ctx_len, new_tok, H: int, Hi: int, P: int = 2,
           shuffle: bool = False, win_cap: int = 256, salient_frac: float = 0.0,
           tie: dict | None = None) -> Workload:
    ctx = np.asarray(ctx_len, np.int64)
    new = np.asarray(new_tok, np.int32)
    assert ctx.shape == new.shape and (new <= ctx).all() and (new >= 0).all()
    pt, num_pages = _pages(ctx, P, seed if shuffle else None)
    return Workload(name=name, seed=seed, B=len(ctx), H=H, Hi=Hi, P=P, ctx_len=ctx,
                    new_tok=new, page_table=pt, num_pages=num_pages, win_cap=win_cap,
                    salient_frac=salient_frac, tie=tie or {})


def compress_inputs(seed: int, rows: int) -> dict:
    """Seeded inputs of the compressor steps: RMSNorm weights U(0.5, 1.5) for
    the latent (512) and the indexer key (128), eps, and rotary tables
    cos/sin [rows, 32] of seeded uniform angles (fp32).  No method arithmetic:
    these are the weights and tables a caller supplies."""
    g = _rng(seed, 0x434D50)
    th = g.uniform(0.0, 2.0 * math.pi, (rows, 32))
    return {"kv_gamma": g.uniform(0.5, 1.5, 512).astype(np.float32),
            "idx_gamma": g.uniform(0.5, 1.5, 128).astype(np.float32), "eps": 1e-6,
            "rope_cos": np.cos(th).astype(np.float32), "rope_sin": np.sin(th).astype(np.float32)}


CONFIG_NAMES = {
    1: "tiny decode: 1 row, 16 heads, 4096 tokens -> 2048 entries",
    2: "single-request long decode: 1 row, 64 heads, 32768 tokens -> 16384 entries, 5% salient x4",
    3: "speculative verify: 32 requests x 6 rows, 64 heads, 3072-5120 (+0-1024) tokens, append of 6",
    4: "serving batch: 128 requests x 1 row, 64 heads, 4k-128k log-uniform tokens, shuffled pages",
    5: "unpooled long context: 4 requests x 1 row, 64 heads, 262144 entries, ties at rank 512",
    6: "chunked prefill / extend: 4 requests x 128 rows, 64 heads, 8192-16384 history + 128-token chunk",
}


def config(cfg: int) -> Workload:
    """The five decode step shapes and the chunked-prefill / extend shape (6),
    seeded with cfg - 1."""
    seed = cfg - 1
    if cfg == 1:
        return custom("cfg1", seed, [4096], [1], H=16, Hi=16)
    if cfg == 2:
        return custom("cfg2", seed, [32768], [1], H=64, Hi=64, salient_frac=0.05)
    if cfg == 3:
        g = _rng(seed, _TAG_LEN)
        hist = g.integers(3072, 5121, size=32) + g.integers(0, 1025, size=32)
        return custom("cfg3", seed, hist + 6, [6] * 32, H=64, Hi=64)
    if cfg == 4:
        g = _rng(seed, _TAG_LEN)
        ctx = np.round(np.exp(g.uniform(math.log(4096), math.log(131072), size=128))).astype(np.int64)
        return custom("cfg4", seed, ctx, [1] * 128, H=64, Hi=64, shuffle=True)
    if cfg == 5:
        tie = {"group": 1024, "group_scale": 8.0, "salient": 300, "salient_scale": 16.0}
        return custom("cfg5", seed, [262144] * 4, [1] * 4, H=64, Hi=64, P=1, tie=tie)
    if cfg == 6:
        # an extend step: each request appends a 128-token chunk and every chunk
        # position is a query row; the 256-slot window ring holds the 127
        # positions before the chunk and the chunk itself, so every row sees its
        # full 128-position window
        g = _rng(seed, _TAG_LEN)
        hist = g.integers(8192, 16385, size=4)
        return custom("cfg6", seed, hist + 128, [128] * 4, H=64, Hi=64, shuffle=True, win_cap=256)
    raise ValueError(f"unknown config {cfg}")
