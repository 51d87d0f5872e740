"""Pins for the CPU oracle: everything here checks the oracle against something
other than itself -- numbers the pages print, format definitions restated from
their bit layouts, a library decoder (torch float8_e4m3fn), exhaustive or
brute-force searches, closed forms and invariants.  CPU only."""
import math

import numpy as np
import pytest
import torch

import bruteforce as BF
import oracle
from fp4_sparse_attention_csa_gb300 import workloads as W
from util import read_golden


# ---- P-1: entry sizes, a closed form against the pages' printed numbers -------
def test_entry_sizes_match_pages():
    g = {k: int(v) for k, v in read_golden("page_constants.txt")}
    main = 512 // 2 + 512 // 16          # 512 e2m1 nibbles + one E4M3 per 16
    idx = 128 // 2 + 128 // 32           # 128 e2m1 nibbles + one E8M0 per 32
    assert main == g["main_kv_entry_bytes"] and idx == g["indexer_k_entry_bytes"]
    pooled, unpooled = g["pair_pooled_caches"], g["global_kv_caches"] - g["pair_pooled_caches"]
    assert (main + idx) * (pooled * 0.5 + unpooled) == g["logical_bytes_per_token"]
    # the oracle's quantisers write exactly those byte counts
    data, sc = oracle.quant_main_entry(np.ones(512, np.float32))
    assert data.size + sc.size == g["main_kv_entry_bytes"]
    data, sc = oracle.quant_idx_entry(np.ones(128, np.float32))
    assert data.size + sc.size == g["indexer_k_entry_bytes"]


# ---- P-2: code tables ---------------------------------------------------------
def test_e2m1_table_from_bit_layout():
    for c in range(16):
        assert oracle.e2m1_decode(c) == float(BF.e2m1_value(c)), c
    assert [oracle.e2m1_decode(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_table_all_256_codes():
    lib_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        o = oracle.e4m3_decode(c)
        ref = BF.e4m3_value(c)
        if ref is None:
            assert math.isnan(o) and math.isnan(lib_vals[c]), c
        else:
            assert o == float(ref) == lib_vals[c], c
            assert math.copysign(1, o) == math.copysign(1, lib_vals[c])


def test_e4m3_printed_points():
    for code, val in read_golden("e4m3_points.txt"):
        o = oracle.e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(o)
        else:
            assert o == float(val) and math.copysign(1, o) == math.copysign(1, float(val))


def test_e8m0_table():
    for c in range(255):
        assert oracle.e8m0_decode(c) == math.ldexp(1.0, c - 127)
    assert math.isnan(oracle.e8m0_decode(255))


# ---- P-3: rounding -------------------------------------------------------------
def test_e2m1_rne_points():
    for v, code in read_golden("e2m1_rne_points.txt"):
        assert oracle.e2m1_encode(np.float32(v)) == int(code), v


def test_e2m1_random_against_bruteforce():
    g = np.random.default_rng(11)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    mids = (grid[1:] + grid[:-1]) / 2
    vals = np.concatenate([g.normal(0, 3, 3000).astype(np.float32),
                           mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 10),
                           g.uniform(-8, 8, 1000).astype(np.float32)])
    for v in vals:
        assert oracle.e2m1_encode(v) == BF.e2m1_encode(float(v)), v


def test_e4m3_encode_against_bruteforce_and_library():
    g = np.random.default_rng(12)
    vals = np.concatenate([
        (g.standard_normal(3000) * np.exp2(g.uniform(-12, 9, 3000))).astype(np.float32),
        np.array([0.0, -0.0, 448, 449, 464, 465, 1e6, -1e6, 2**-10, 2**-9 * 1.5, 2**-7 * 1.0625],
                 np.float32)])
    lib = torch.tensor(np.clip(vals, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, l in zip(vals, lib):
        o = oracle.e4m3_encode(v)
        assert o == BF.e4m3_encode(float(v)), v
        assert o == l, (v, o, l)


# ---- P-4: block quantisers against brute force ---------------------------------
def _blocks(n, size, seed):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        x = g.standard_normal(size).astype(np.float32) * np.float32(2.0 ** g.integers(-20, 12))
        if i % 17 == 0:
            x[:] = 0
        if i % 13 == 0:
            x[g.integers(0, size)] = -0.0
        if i % 7 == 0:
            x[: size // 2] = 0
        out.append(x)
    return out


def test_nvfp4_block_bruteforce():
    for x in _blocks(300, 16, 1):
        codes, sc = oracle.nvfp4_block(x)
        bc, bs = BF.nvfp4_block(x)
        assert sc == bs and list(codes) == bc, x


def test_mxfp4_block_bruteforce():
    for x in _blocks(300, 32, 2):
        codes, sc = oracle.mxfp4_block(x)
        bc, bs = BF.mxfp4_block(x)
        assert sc == bs and list(codes) == bc, x


def test_entry_packing_nibble_order():
    x = np.zeros(512, np.float32)
    x[0], x[1] = 6.0, -0.5            # block 0: amax 6 -> scale E4M3(1.0)
    data, sc = oracle.quant_main_entry(x)
    assert sc[0] == 0x38 and data[0] == (0x7 | (0x9 << 4))
    y = np.zeros(128, np.float32)
    y[2], y[3] = 1.0, -1.5            # amax 1.5: E = 0 - 2 -> code 125, 1.0/0.25 = 4
    data, sc = oracle.quant_idx_entry(y)
    assert sc[0] == 125 and data[1] == (0x6 | (0xF << 4))


# ---- P-5: idempotence and the amax code ------------------------------------------
def _deq(codes, scale, dec):
    return np.array([oracle.e2m1_decode(c) * dec(scale) for c in codes], np.float32)


def test_requantisation_is_idempotent():
    # NVFP4: holds when the E4M3 scale is a normal number (code >= 8): then
    # amax / s lies within 6 * (1 +- 2^-4) and rounds back to 6.  With a
    # subnormal scale the scale's own rounding is too coarse for that.
    for x in _blocks(150, 16, 3):
        c1, s1 = oracle.nvfp4_block(x)
        c2, s2 = oracle.nvfp4_block(_deq(c1, s1, oracle.e4m3_decode))
        if s1 >= 8:
            assert (c1[np.argmax(np.abs(x))] & 7) == 7
            assert s1 == s2 and np.array_equal(c1 & 7, c2 & 7)
    for x in _blocks(150, 32, 4):
        c1, s1 = oracle.mxfp4_block(x)
        c2, s2 = oracle.mxfp4_block(_deq(c1, s1, oracle.e8m0_decode))
        if np.any(c1 & 7):
            assert s1 == s2 and np.array_equal(c1 & 7, c2 & 7)


def test_mxfp4_amax_lands_on_4_or_6():
    for x in _blocks(100, 32, 5):
        if not np.any(x):
            continue
        codes, _ = oracle.mxfp4_block(x)
        assert (codes[np.argmax(np.abs(x))] & 7) in (6, 7)


# ---- cache fixtures ----------------------------------------------------------------
def _tiny_cache(ctx, Hi=2, H=2, seed=0, P=2):
    wl = W.custom("tiny", seed, [ctx], [1], H=H, Hi=Hi, P=P)
    return wl, oracle.build_cache(wl)


def _bf_idx_entry(cache, b, e):
    data, sc = cache.idx_entry(b, e)
    codes = [(data[k // 2] >> (4 * (k % 2))) & 15 for k in range(128)]
    return BF.dequant_fp4(codes, [BF.e8m0_value(s) for s in sc], 32)


def _bf_main_entry(cache, b, e):
    data, sc = cache.main_entry(b, e)
    codes = [(data[k // 2] >> (4 * (k % 2))) & 15 for k in range(512)]
    return BF.dequant_fp4(codes, [BF.e4m3_value(s) for s in sc], 16)


def _bf_qhat(q128_bits):
    qf = W.bf16_bits_to_f32(q128_bits)
    out = []
    for b in range(4):
        codes, sc = BF.mxfp4_block(qf[32 * b:32 * b + 32])
        out.extend(float(BF.e2m1_value(c)) * float(BF.e8m0_value(sc)) for c in codes)
    return np.array(out)


# ---- P-6: score ---------------------------------------------------------------------
def test_score_bruteforce_exact_with_power_of_two_weights():
    wl, cache = _tiny_cache(32, Hi=2)                # n = 16 entries
    q_idx, _, _ = wl.step_queries()
    w = np.array([[0.5, 2.0]], np.float32)           # exact products
    sc = oracle.index_score(cache, wl.row_req, wl.row_pos, q_idx, w)
    qhat = np.stack([_bf_qhat(q_idx[0, h]) for h in range(2)])
    khat = np.stack([_bf_idx_entry(cache, 0, e) for e in range(16)])
    ref = BF.score_fp64(qhat, khat, w[0].astype(np.float64))
    assert np.array_equal(sc[0, :16].astype(np.float64), ref)


def test_score_bruteforce_uniform_weights():
    wl, cache = _tiny_cache(30, Hi=3, seed=3)        # n = 15 entries
    q_idx, w, _ = wl.step_queries()
    sc = oracle.index_score(cache, wl.row_req, wl.row_pos, q_idx, w)
    qhat = np.stack([_bf_qhat(q_idx[0, h]) for h in range(3)])
    khat = np.stack([_bf_idx_entry(cache, 0, e) for e in range(15)])
    ref = BF.score_fp64(qhat, khat, w[0].astype(np.float64))
    np.testing.assert_allclose(sc[0, :15], ref, rtol=2e-6, atol=0)


def test_score_closed_form_self_product():
    """One head, w = 1, the cached key equals the query: score = |q_hat|^2."""
    wl = W.custom("self", 5, [2], [1], H=1, Hi=1, P=1)   # row at pos 1 sees 2 entries
    q_idx, _, _ = wl.step_queries()
    cache = oracle.Cache(wl.num_pages, wl.page_table, 1, window=False)
    x = np.zeros((2, 512), np.uint16)
    y = np.stack([q_idx[0, 0], q_idx[0, 0]])
    assert cache.append([0], [0, 2], x, y, window=False) == 0
    sc = oracle.index_score(cache, wl.row_req, wl.row_pos, q_idx, np.ones((1, 1), np.float32))
    qh = _bf_qhat(q_idx[0, 0])
    assert sc[0, 0] == sc[0, 1] == np.float32(np.dot(qh, qh))


# ---- P-7 / P-8: top-k -----------------------------------------------------------------
@pytest.mark.parametrize("n", [0, 1, 5, 511, 512, 513, 600])
def test_topk_bruteforce(n):
    g = np.random.default_rng(n)
    s = g.integers(0, 40, n).astype(np.float32) / 4       # many exact ties
    out = oracle.topk_row(s, n)
    assert list(out) == BF.topk_sorted(list(s), 512)


def test_topk_all_zero_scores_pick_lowest_indices():
    out = oracle.topk_row(np.zeros(3000, np.float32), 3000)
    assert list(out) == list(range(512))


def test_zero_weights_give_lowest_indices():
    wl, cache = _tiny_cache(2400, Hi=2, seed=7)           # n = 1200 entries
    q_idx, _, q = wl.step_queries()
    w = np.zeros((1, 2), np.float32)
    _, _, topk, scores = oracle.decode(cache, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale)
    assert not np.any(scores[0, :1200]) and list(topk[0]) == list(range(512))


def test_topk_duplicates_resolve_to_lowest_index():
    s = np.zeros(1000, np.float32)
    s[100:700] = 3.0          # 600 equal winners
    s[900] = 5.0
    out = oracle.topk_row(s, 1000)
    assert list(out) == list(range(100, 611)) + [900]


# ---- P-9: attention -----------------------------------------------------------------
def _keys_bruteforce(cache, b, pos, topk, P=2):
    n = (pos + 1) // P
    keys = [_bf_main_entry(cache, b, e) for e in topk if 0 <= e < n]
    for p in range(max(0, pos - 127), pos + 1):
        codes, s = cache.window_slot(b, p)
        keys.append(np.array([float(BF.e4m3_value(c)) * s for c in codes]))
    return np.stack(keys)


def test_attention_equals_dense_when_topk_covers_everything():
    wl, cache = _tiny_cache(700, Hi=2, H=3, seed=9)      # n = 350 <= 512
    q_idx, w, q = wl.step_queries()
    out, lse, topk, _ = oracle.decode(cache, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale)
    assert list(topk[0, :350]) == list(range(350)) and (topk[0, 350:] == -1).all()
    keys = _keys_bruteforce(cache, 0, int(wl.row_pos[0]), topk[0])
    qf = W.bf16_bits_to_f32(q[0]).astype(np.float64)
    ref, ref_lse, p = BF.dense_attention_fp64(qf, keys, wl.softmax_scale)
    np.testing.assert_allclose(out[0], ref, rtol=0, atol=2e-6 * np.abs(ref).max())
    np.testing.assert_allclose(lse[0], ref_lse, rtol=0, atol=2e-6)
    # softmax weights recovered from the oracle's lse sum to one
    logits = wl.softmax_scale * qf @ keys.T
    np.testing.assert_allclose(np.exp(logits - lse[0][:, None].astype(np.float64)).sum(-1), 1.0,
                               rtol=0, atol=1e-6)


def test_attention_single_key_returns_that_value():
    wl, cache = _tiny_cache(1, Hi=1, H=2, seed=4)         # pos 0: no entry, one window key
    q_idx, w, q = wl.step_queries()
    out, lse, topk, _ = oracle.decode(cache, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale)
    assert (topk == -1).all()
    codes, s = cache.window_slot(0, 0)
    v = np.array([oracle.e4m3_decode(c) for c in codes], np.float32) * np.float32(s)
    assert np.array_equal(out[0, 0], v) and np.array_equal(out[0, 1], v)


def test_attention_identical_keys_return_the_key():
    wl = W.custom("same", 2, [40], [1], H=2, Hi=1, P=2)
    cache = oracle.Cache(wl.num_pages, wl.page_table, 2, window=True)
    x = np.tile(W.f32_to_bf16_bits(np.linspace(-2, 2, 512, dtype=np.float32)), (40, 1))
    y = np.tile(W.f32_to_bf16_bits(np.ones(128, np.float32)), (40, 1))
    cache.append([0], [0, 40], x, y)
    _, _, q = wl.step_queries()
    assert len({cache.window_slot(0, p)[0].tobytes() for p in range(40)}) == 1
    # window keys only (no global entry selected): every key is the same v
    out, _ = oracle.attention_row(cache, 0, 39, np.full(512, -1, np.int32), q[0], wl.softmax_scale)
    codes, s = cache.window_slot(0, 39)
    v = np.array([oracle.e4m3_decode(c) for c in codes], np.float32) * np.float32(s)
    np.testing.assert_allclose(out, np.stack([v, v]), rtol=0, atol=1e-6 * np.abs(v).max())
    # plus 20 identical pooled entries: still dense softmax attention over those keys
    topk = np.array(list(range(20)) + [-1] * 492, np.int32)
    out, _ = oracle.attention_row(cache, 0, 39, topk, q[0], wl.softmax_scale)
    keys = _keys_bruteforce(cache, 0, 39, topk)
    ref, _, _ = BF.dense_attention_fp64(W.bf16_bits_to_f32(q[0]).astype(np.float64), keys, wl.softmax_scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=2e-6 * np.abs(ref).max())


# ---- P-10: append bookkeeping ---------------------------------------------------------
@pytest.mark.parametrize("P", [1, 2])
def test_append_in_one_call_equals_token_by_token(P):
    wl = W.custom("app", 6, [301, 290, 7], [1, 1, 1], H=1, Hi=1, P=P)
    whole = oracle.Cache(wl.num_pages, wl.page_table, P, win_cap=160)
    xs, ys = zip(*[wl.tokens(b, 0, int(wl.ctx_len[b])) for b in range(wl.B)])
    off = np.concatenate([[0], np.cumsum([len(x) for x in xs])])
    assert whole.append(np.zeros(3, np.int32), off, np.concatenate(xs), np.concatenate(ys)) == 0
    step = oracle.Cache(wl.num_pages, wl.page_table, P, win_cap=160)
    g = np.random.default_rng(0)
    pos = np.zeros(3, np.int64)
    while (pos < wl.ctx_len).any():          # random chunk sizes, odd and even starts
        t = np.minimum(g.integers(0, 4, 3), wl.ctx_len - pos)
        xx = np.concatenate([xs[b][pos[b]:pos[b] + t[b]] for b in range(3)])
        yy = np.concatenate([ys[b][pos[b]:pos[b] + t[b]] for b in range(3)])
        assert step.append(pos.astype(np.int32), np.concatenate([[0], np.cumsum(t)]), xx, yy) == 0
        pos += t
    assert np.array_equal(whole.kv_pool, step.kv_pool)
    assert np.array_equal(whole.idx_pool, step.idx_pool)
    assert np.array_equal(whole.win_codes, step.win_codes)
    assert np.array_equal(whole.win_scale, step.win_scale)
    for b in range(3):
        if P == 2 and wl.ctx_len[b] % 2 == 1:
            assert np.array_equal(whole.pending[b], step.pending[b])


def test_append_entry_is_pooled_pair():
    wl = W.custom("pool", 8, [11], [1], H=1, Hi=1)
    cache = oracle.build_cache(wl)
    x, y = wl.tokens(0, 0, 11)
    xf, yf = W.bf16_bits_to_f32(x), W.bf16_bits_to_f32(y)
    for e in range(5):
        px = (xf[2 * e] + xf[2 * e + 1]) * np.float32(0.5)
        py = (yf[2 * e] + yf[2 * e + 1]) * np.float32(0.5)
        d, s = oracle.quant_main_entry(px)
        assert np.array_equal(np.concatenate(cache.main_entry(0, e)), np.concatenate([d, s]))
        d, s = oracle.quant_idx_entry(py)
        assert np.array_equal(np.concatenate(cache.idx_entry(0, e)), np.concatenate([d, s]))
    # pending holds token 10 (unpaired); the window holds every token
    assert np.array_equal(cache.pending[0], np.concatenate([x[10], y[10]]))
    for p in range(11):
        codes, s = cache.window_slot(0, p)
        c2, s2 = oracle.quant_window_token(xf[p])
        assert np.array_equal(codes, c2) and s == s2


def test_window_quantiser_against_library_e4m3():
    g = np.random.default_rng(3)
    x = g.standard_normal(512).astype(np.float32)
    codes, s = oracle.quant_window_token(x)
    assert s == np.float32(np.abs(x).max()) / np.float32(448)
    ref = torch.tensor(x / np.float32(s)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(codes, ref.numpy())


def test_indexer_page_byte_layout():
    """An indexer entry's bytes sit where the format description puts them:
    8-entry groups of 544 B, data byte k of slot 8g+r at 544g + 128(k//16) +
    16r + k%16, scale byte j at 544g + 512 + 4r + j."""
    wl = W.custom("layout", 9, [2 * 29 + 2], [1], H=1, Hi=1, P=2)   # entries 0..29
    cache = oracle.build_cache(wl)
    x, y = wl.tokens(0, 0, 60)
    yf = W.bf16_bits_to_f32(y)
    e = 29                                                          # group 3, r = 5
    data, sc = oracle.quant_idx_entry((yf[2 * e] + yf[2 * e + 1]) * np.float32(0.5))
    page = int(wl.page_table[0, 0]) * 4352
    for k in range(64):
        assert cache.idx_pool[page + 544 * 3 + 128 * (k // 16) + 16 * 5 + k % 16] == data[k]
    for j in range(4):
        assert cache.idx_pool[page + 544 * 3 + 512 + 4 * 5 + j] == sc[j]


# ---------------------------------------------------------------- compressor
# The fused compressor ([SGL] "DSpark adaptation and optimization": pooling,
# RMSNorm, RoPE and quantisation in one step) on a pooled vector: RMSNorm with
# a gamma input, then rotate-half RoPE on the last 64 dims.

def _ulp32(x):
    return np.spacing(np.abs(np.float32(x))).astype(np.float64)


@pytest.mark.parametrize("dim", [512, 128])
def test_rmsnorm_closed_form(dim):
    """Against the fp64 definition x * gamma / sqrt(mean(x^2) + eps): a few
    fp32 roundings apart, for random vectors and gammas."""
    g = np.random.default_rng(dim)
    for _ in range(20):
        x = (g.standard_normal(dim) * np.exp(g.uniform(-3, 3))).astype(np.float32)
        gam = g.uniform(0.5, 1.5, dim).astype(np.float32)
        got = oracle.compress_vec(x, gamma=gam, eps=1e-6).astype(np.float64)
        x64 = x.astype(np.float64)
        ref = x64 * gam / np.sqrt(np.mean(x64 * x64) + 1e-6)
        assert (np.abs(got - ref) <= 8 * _ulp32(ref) + 1e-30).all()


def test_rmsnorm_constant_vector_and_unit_rms():
    """A constant vector c maps to c / sqrt(c^2 + eps) in every element (the
    sum of squares is exact for c a power of two); with gamma = 1 and eps
    small the output has unit RMS."""
    for c in (0.25, 2.0, 64.0):
        x = np.full(512, c, np.float32)
        got = oracle.compress_vec(x, gamma=np.ones(512, np.float32), eps=1e-6)
        ref = c / np.sqrt(c * c + 1e-6)
        assert np.abs(got.astype(np.float64) - ref).max() <= 2 * _ulp32(ref)
    x = np.random.default_rng(7).standard_normal(128).astype(np.float32)
    got = oracle.compress_vec(x, gamma=np.ones(128, np.float32), eps=1e-12).astype(np.float64)
    assert abs(np.sqrt(np.mean(got * got)) - 1.0) < 1e-6


def test_rope_special_angles():
    """cos = 1, sin = 0 leaves the vector unchanged; cos = 0, sin = 1 maps each
    pair (a, b) of the last 64 dims to (-b, a) exactly; the first dims never
    move."""
    x = np.random.default_rng(3).standard_normal(512).astype(np.float32)
    one, zero = np.ones(32, np.float32), np.zeros(32, np.float32)
    assert np.array_equal(oracle.compress_vec(x, cos32=one, sin32=zero), x)
    got = oracle.compress_vec(x, cos32=zero, sin32=one)
    assert np.array_equal(got[:448], x[:448])
    assert np.array_equal(got[448:480], -x[480:512])
    assert np.array_equal(got[480:512], x[448:480])


def test_rope_is_a_rotation():
    """Each pair keeps its length, and rotating by theta then by -theta
    returns the input, up to fp32 rounding."""
    g = np.random.default_rng(11)
    x = g.standard_normal(128).astype(np.float32)
    th = g.uniform(0, 2 * np.pi, 32)
    c, s = np.cos(th).astype(np.float32), np.sin(th).astype(np.float32)
    y = oracle.compress_vec(x, cos32=c, sin32=s)
    n0 = np.hypot(x[64:96].astype(np.float64), x[96:128].astype(np.float64))
    n1 = np.hypot(y[64:96].astype(np.float64), y[96:128].astype(np.float64))
    assert np.allclose(n0, n1, rtol=1e-6, atol=1e-7)
    z = oracle.compress_vec(y, cos32=c, sin32=-s)
    assert np.allclose(z, x, rtol=0, atol=1e-6)
    assert np.array_equal(y[:64], x[:64])


@pytest.mark.parametrize("P", [2, 1])
def test_compressed_append_token_by_token_equals_one_call(P):
    """With the compressor on, appending a request's tokens one at a time
    writes the same bytes as appending them in one call (pooling partners,
    pending token and rotary positions line up)."""
    g = np.random.default_rng(40 + P)
    B, L = 2, 150
    pages_per_req = (L // P + 63) // 64 + 1
    pt = np.arange(B * pages_per_req, dtype=np.int32).reshape(B, pages_per_req)
    kv = (g.standard_normal((B, L, 512)) * 2).astype(np.float32)
    ix = g.standard_normal((B, L, 128)).astype(np.float32)
    to_bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    kvb, ixb = to_bits(kv), to_bits(ix)
    th = g.uniform(0, 2 * np.pi, (L, 32))
    cmp = {"kv_gamma": g.uniform(0.5, 1.5, 512), "idx_gamma": g.uniform(0.5, 1.5, 128), "eps": 1e-6,
           "rope_cos": np.cos(th), "rope_sin": np.sin(th)}
    one = oracle.Cache(B * pages_per_req, pt, P)
    assert one.append(np.zeros(B, np.int32), np.array([0, L, 2 * L], np.int32),
                      kvb.reshape(-1, 512), ixb.reshape(-1, 128), compress=cmp) == 0
    step = oracle.Cache(B * pages_per_req, pt, P)
    for p in range(L):
        assert step.append(np.full(B, p, np.int32), np.array([0, 1, 2], np.int32),
                           kvb[:, p].reshape(-1, 512), ixb[:, p].reshape(-1, 128), compress=cmp) == 0
    assert np.array_equal(one.kv_pool, step.kv_pool) and np.array_equal(one.idx_pool, step.idx_pool)
    plain = oracle.Cache(B * pages_per_req, pt, P)
    plain.append(np.zeros(B, np.int32), np.array([0, L, 2 * L], np.int32), kvb.reshape(-1, 512), ixb.reshape(-1, 128))
    assert not np.array_equal(plain.kv_pool, one.kv_pool)     # the steps did change the entries


# ---- P-12: rotary attention (query and window tokens; NEXT f-3) ------------------
# A quarter turn (cos 0, sin 1) maps each pair (a, b) of the last 64 dims to
# (-b, a): an exact permutation with a sign flip, both for E4M3 window codes and
# for bf16 query bits.  So the rotary oracle with quarter-turn table rows must
# equal the plain oracle (itself pinned by P-9) run on inputs permuted by hand.
def _tables(rows, turned):
    cs = np.ones((rows, 32), np.float32)
    sn = np.zeros((rows, 32), np.float32)
    for r in turned:
        cs[r], sn[r] = 0.0, 1.0
    return cs, sn


def _turn_e4m3(codes):
    c = codes.copy()
    a, b = codes[448:480].copy(), codes[480:512].copy()
    c[448:480] = b ^ np.uint8(0x80)                        # -b: the E4M3 sign bit
    c[480:512] = a
    return c


def _turn_bf16(q_row):
    q = q_row.copy()
    a, b = q_row[..., 448:480].copy(), q_row[..., 480:512].copy()
    q[..., 448:480] = b ^ np.uint16(0x8000)               # -b: the bf16 sign bit
    q[..., 480:512] = a
    return q


def _rope_case():
    wl, cache = _tiny_cache(700, Hi=2, H=3, seed=12)      # row at 699: 350 entries, window 572..699
    q_idx, w, q = wl.step_queries()
    _, _, topk, _ = oracle.decode(cache, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale)
    return wl, cache, q, topk


def test_rope_identity_tables_change_nothing():
    wl, cache, q, topk = _rope_case()
    cs, sn = _tables(700, [])
    o, l, rc = oracle.attention_row_rope(cache, 0, 699, topk[0], q[0], wl.softmax_scale, cs, sn)
    o0, l0 = oracle.attention_row(cache, 0, 699, topk[0], q[0], wl.softmax_scale)
    assert rc == 0 and np.array_equal(o, o0) and np.array_equal(l, l0)


def test_rope_window_token_turned_with_its_own_position():
    """Only table row 600 turns: exactly the window token at position 600 is
    rotated, as key and as value; the query (row 699) and the rest are not."""
    wl, cache, q, topk = _rope_case()
    cs, sn = _tables(700, [600])
    o, l, rc = oracle.attention_row_rope(cache, 0, 699, topk[0], q[0], wl.softmax_scale, cs, sn)
    codes, _ = cache.window_slot(0, 600)
    codes[:] = _turn_e4m3(codes.copy())
    o0, l0 = oracle.attention_row(cache, 0, 699, topk[0], q[0], wl.softmax_scale)
    assert rc == 0 and np.array_equal(o, o0) and np.array_equal(l, l0)


def test_rope_query_turned_with_the_row_position():
    wl, cache, q, topk = _rope_case()
    cs, sn = _tables(700, [699])
    o, l, rc = oracle.attention_row_rope(cache, 0, 699, topk[0], q[0], wl.softmax_scale, cs, sn)
    # row 699 also turns the window token at 699 (the row's own token)
    codes, _ = cache.window_slot(0, 699)
    codes[:] = _turn_e4m3(codes.copy())
    o0, l0 = oracle.attention_row(cache, 0, 699, topk[0], _turn_bf16(q[0]), wl.softmax_scale)
    assert rc == 0 and np.array_equal(o, o0) and np.array_equal(l, l0)


def test_rope_leaves_global_entries_as_stored():
    """Every table row turns: the query and all 128 window tokens are turned,
    the 350 global entries (rotated when appended) are used as stored."""
    wl, cache, q, topk = _rope_case()
    cs, sn = _tables(700, range(700))
    o, l, rc = oracle.attention_row_rope(cache, 0, 699, topk[0], q[0], wl.softmax_scale, cs, sn)
    kv_before = cache.kv_pool.copy()
    for p in range(572, 700):
        codes, _ = cache.window_slot(0, p)
        codes[:] = _turn_e4m3(codes.copy())
    o0, l0 = oracle.attention_row(cache, 0, 699, topk[0], _turn_bf16(q[0]), wl.softmax_scale)
    assert np.array_equal(cache.kv_pool, kv_before)
    assert rc == 0 and np.array_equal(o, o0) and np.array_equal(l, l0)
    # and the rotation is not a no-op here
    o1, _ = oracle.attention_row(cache, 0, 699, topk[0], q[0], wl.softmax_scale)
    assert not np.array_equal(o, o1)


def test_rope_row_beyond_the_tables_is_rejected():
    wl, cache, q, topk = _rope_case()
    cs, sn = _tables(699, [])                              # rows 0..698 only
    o, l, rc = oracle.attention_row_rope(cache, 0, 699, topk[0], q[0], wl.softmax_scale, cs, sn)
    assert rc == -1 and not o.any() and np.isneginf(l).all()


# ---- P-13: two-level candidate filter (NEXT f-2) ---------------------------------
@pytest.mark.parametrize("n", [1, 63, 64, 65, 700, 5000, 40000])
def test_two_level_keeping_every_block_is_the_flat_selection(n):
    g = np.random.default_rng(n)
    sc = (g.integers(0, 300, n) / 7).astype(np.float32)    # many ties
    nb = (n + 63) // 64
    assert np.array_equal(oracle.topk_two_level(sc, n, nb), oracle.topk_row(sc, n))
    assert np.array_equal(oracle.topk_two_level(sc, n, nb + 9), oracle.topk_row(sc, n))


@pytest.mark.parametrize("seed,ties", [(1, False), (2, True), (3, True)])
def test_two_level_with_512_blocks_is_the_flat_selection(seed, ties):
    """Every entry of the flat top 512 lies in a block whose largest score is at
    least the 512th score, and (ties broken toward lower indices at both levels)
    those blocks are among the first 512 blocks: 512 kept blocks lose nothing."""
    g = np.random.default_rng(seed)
    n = 64 * 1500 + 17
    sc = g.standard_normal(n).astype(np.float32)
    if ties:
        sc = np.round(sc * 4) / 4                         # heavy ties, also at rank 512
        sc[::97] = sc.max()
    assert np.array_equal(oracle.topk_two_level(sc, n, 512), oracle.topk_row(sc, n))


def test_two_level_keeps_only_the_chosen_blocks():
    sc = np.zeros(128, np.float32)
    sc[5] = 9.0                                           # block 0: one high entry
    sc[64:] = 5.0                                         # block 1: all medium
    out = oracle.topk_two_level(sc, 128, 1)
    assert list(out[:64]) == list(range(64)) and (out[64:] == -1).all()
    out = oracle.topk_two_level(sc, 128, 2)
    assert list(out[:128]) == list(range(128))


def test_two_level_equal_block_scores_go_to_the_lower_block():
    sc = np.full(64 * 3, -1.0, np.float32)
    sc[70] = 2.0                                          # block 1
    sc[130] = 2.0                                         # block 2, same block score
    sc[10] = 1.0                                          # block 0, lower score
    out = oracle.topk_two_level(sc, 64 * 3, 1)
    assert list(out[:64]) == list(range(64, 128))
    out = oracle.topk_two_level(sc, 64 * 3, 2)
    assert list(out[:128]) == list(range(64, 192))
