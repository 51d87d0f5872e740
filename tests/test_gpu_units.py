"""GPU parity of each C-ABI entry point against the CPU oracle, at sizes the
oracle finishes in seconds but that span several tiles, pages and ragged
tails, plus the edge cases of the method (n = 0, n < 512, n = 512, odd and
even positions, the pending token, rows sharing a request)."""
import numpy as np
import pytest
import torch

import parity
import oracle
import fp4_sparse_attention_csa_gb300 as csa
from fp4_sparse_attention_csa_gb300 import workloads as W
from fp4_sparse_attention_csa_gb300.session import DeviceState

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    csa.build.build()
    oracle.build()
    torch.cuda.set_device(0)


def _pools_equal(st, ref):
    assert np.array_equal(st.kv_pool.cpu().numpy(), ref.kv_pool), "main-KV pool bytes differ"
    assert np.array_equal(st.idx_pool.cpu().numpy(), ref.idx_pool), "indexer pool bytes differ"
    if ref.win_codes is not None:
        assert np.array_equal(st.win_codes.cpu().numpy(), ref.win_codes), "window codes differ"
        assert np.array_equal(st.win_scale.cpu().numpy(), ref.win_scale), "window scales differ"


# ---------------------------------------------------------------- append (J-1)
@pytest.mark.parametrize("P", [2, 1])
def test_append_bit_exact_history_and_step(P):
    ctx = [1, 2, 3, 63, 64, 65, 129, 300, 1025, 2048]
    new = [1, 2, 1, 6, 3, 1, 6, 2, 5, 1]
    wl = W.custom("app", 11, ctx, new, H=16, Hi=16, P=P, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    rc, flags = csa.csa_check_device_status(st.ws_append)
    assert rc == 0 and flags == 0
    ref = oracle.build_cache(wl, upto="hist")
    x, y = wl.step_tokens()
    assert ref.append(wl.step_pos0, wl.step_tok_off, x, y) == 0
    _pools_equal(st, ref)
    if P == 2:
        pend = st.pending.view(torch.uint16).cpu().numpy()
        odd = (wl.ctx_len % 2) == 1                  # an unpaired last token exists
        assert np.array_equal(pend[odd], ref.pending[odd])


def test_append_token_by_token_equals_bulk():
    wl = W.custom("tbt", 12, [37, 40, 9], [1, 1, 1], H=16, Hi=16)
    bulk = DeviceState(wl)
    bulk.build_history()
    one = DeviceState(wl)
    for p in range(int(wl.hist_len.max())):
        active = [b for b in range(wl.B) if p < wl.hist_len[b]]
        pos0 = np.zeros(wl.B, np.int32)
        cnt = np.zeros(wl.B, np.int64)
        xs, ys = [], []
        for b in active:
            x, y = wl.tokens(b, p, p + 1)
            pos0[b], cnt[b] = p, 1
            xs.append(x)
            ys.append(y)
        one.append(pos0, np.concatenate([[0], np.cumsum(cnt)]), np.concatenate(xs), np.concatenate(ys))
    torch.cuda.synchronize()
    assert torch.equal(bulk.kv_pool, one.kv_pool) and torch.equal(bulk.idx_pool, one.idx_pool)
    assert torch.equal(bulk.win_codes, one.win_codes) and torch.equal(bulk.win_scale, one.win_scale)


def test_append_flags_bad_page_without_writing():
    wl = W.custom("bad", 13, [200], [1], H=16, Hi=16)
    st = DeviceState(wl)
    st.page_table[0, 1] = wl.num_pages + 5            # entries 64..127 point outside the pool
    st.build_history()
    rc, flags = csa.csa_check_device_status(st.ws_append)
    assert rc == 5 and (flags & csa.FLAG_PAGE_OOB)
    # entries 64..127 were not written anywhere; the other pages hold data
    kv = st.kv_pool.view(wl.num_pages, -1)
    assert int(kv[int(wl.page_table[0, 0])].count_nonzero()) > 0


# ------------------------------------------------------------ index score
def _check_scores(wl, got, ld, Hi):
    """Every visible score within the fp32 summation bound of the oracle's,
    scores past a row's visible range untouched (NaN)."""
    ref = oracle.build_cache(wl)
    q_idx, w, _ = wl.step_queries()
    ref_sc = oracle.index_score(ref, wl.row_req, wl.row_pos, q_idx, w, ld)
    # sum_h |w_h| relu(q_h . k): the scale of the fp32 rounding in either sum
    mag = oracle.index_score(ref, wl.row_req, wl.row_pos, q_idx, np.abs(w), ld)
    # The score is sum_h w_h * relu(q_h . k) (the pages fix no summation order
    # or fusing); the oracle adds products in head order, the kernel uses fused
    # multiply-adds on even/odd head pairs.  Each fp32 sum of Hi terms is within
    # gamma_(Hi+1) * mag of the exact value, so the two are within twice that.
    u = 2.0 ** -24
    tol_f = 2.0 * (Hi + 1) * u / (1.0 - (Hi + 1) * u)
    n = wl.row_entries()
    for r in range(wl.R):
        g, o, m = got[r, :n[r]], ref_sc[r, :n[r]], mag[r, :n[r]]
        fin = np.isfinite(o)
        assert np.array_equal(np.isfinite(g), fin) and np.array_equal(g[~fin], o[~fin]), r
        err = np.abs(g[fin].astype(np.float64) - o[fin].astype(np.float64))
        assert (err <= tol_f * m[fin].astype(np.float64)).all(), (r, float((err / np.maximum(m[fin], 1e-30)).max()))
        assert np.isnan(got[r, n[r]:]).all(), "scores past the visible range must be untouched"


def _score(st, s, wl, Hi):
    ld = ((max(wl.max_entries, 1) + 63) // 64) * 64
    scores = torch.full((wl.R, ld), float("nan"), device="cuda")
    ws = torch.zeros(csa.csa_workspace_size(csa.OP_INDEX_SCORE, wl.R, wl.max_entries, 16), dtype=torch.uint8,
                     device="cuda")
    csa.csa_index_score(st.cache, s["rows"], Hi, s["q_idx"], s["w"], scores, ld, ws)
    rc, flags = csa.csa_check_device_status(ws)
    return scores, ld, rc, flags


# Hi up to the declared 128; rows of one request share the MMA's N up to 128
# columns (64 heads: 2 rows; 8 heads: 16 rows), so these cover one and two
# accumulators per consumer group and multi-row segments.
@pytest.mark.parametrize("Hi,rows", [(16, 1), (64, 1), (64, 6), (16, 24), (32, 3), (96, 1), (128, 1), (128, 3),
                                     (40, 5), (8, 20)])
def test_index_score_matches_oracle(Hi, rows):
    ctx = [2, 127, 128, 129, 257, 1024 + 7, 1030, 4096 + 77]
    wl = W.custom("score", 21 + Hi + rows, [c + rows for c in ctx], [rows] * len(ctx), H=16, Hi=Hi, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    scores, ld, rc, flags = _score(st, s, wl, Hi)
    assert rc == 0 and flags == 0, flags
    _check_scores(wl, scores.cpu().numpy(), ld, Hi)


@pytest.mark.parametrize("rows_per_req", [1, 2])
def test_index_score_many_short_segments(rows_per_req):
    """Hundreds of one- and two-tile requests: a CTA's few items span several
    segments, whose q images go through the two buffers faster than the
    segments' tiles are scored (the loads must go out in segment order)."""
    cyc = [1, 2, 3, 100, 260, 700, 1025, 1600, 3000]
    ctx = [cyc[i % len(cyc)] + rows_per_req for i in range(200)]
    wl = W.custom("score_short", 61 + rows_per_req, ctx, [rows_per_req] * len(ctx), H=16, Hi=32)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    scores, ld, rc, flags = _score(st, s, wl, 32)
    assert rc == 0 and flags == 0, flags
    _check_scores(wl, scores.cpu().numpy(), ld, 32)


def test_index_score_rows_without_entries():
    """Rows at position 0 of a pair-pooled cache see no entry: they get no
    segment, write nothing, and the rows around them score as usual (a row
    group made of such rows once left a gap in the segment numbering)."""
    ctx = [1, 300, 1, 1, 5000, 1, 129, 1]
    wl = W.custom("score0", 29, ctx, [1] * len(ctx), H=16, Hi=64, shuffle=True)
    assert (wl.row_entries() == 0).sum() == 5
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    scores, ld, rc, flags = _score(st, s, wl, 64)
    assert rc == 0 and flags == 0, flags
    _check_scores(wl, scores.cpu().numpy(), ld, 64)


def test_identical_entries_score_identically():
    """Bitwise-identical indexer entries get bitwise-identical scores wherever
    they sit in a tile or page."""
    wl = W.custom("ident", 31, [3000], [1], H=16, Hi=64, P=1)
    st = DeviceState(wl)
    x, y = wl.tokens(0, 0, 3000)
    y[:] = y[17]
    st.append(np.zeros(1, np.int32), np.array([0, 3000], np.int32), x, y)
    s = st.step_inputs()
    ld = 3008
    scores = torch.zeros((1, ld), device="cuda")
    ws = torch.zeros(csa.csa_workspace_size(csa.OP_INDEX_SCORE, 1, 3000, 16), dtype=torch.uint8, device="cuda")
    csa.csa_index_score(st.cache, s["rows"], 64, s["q_idx"], s["w"], scores, ld, ws)
    g = scores[0, :3000].cpu().numpy()
    assert len(set(g.tolist())) == 1


# ------------------------------------------------------------------- top-k
@pytest.mark.parametrize("n", [0, 1, 300, 511, 512, 513, 1000, 5000, 70000, 262144, 300000])
def test_topk_exact_with_ties(n):
    g = np.random.default_rng(n)
    R = 3
    ld = max(64, ((n + 63) // 64) * 64)
    sc = (g.integers(0, 200, (R, ld)) / 8).astype(np.float32)    # many exact ties
    sc[1] = -sc[1]                                                  # negative scores
    sc[2, : n // 2] = 0.0
    sc[2, n // 3: n // 2] = -0.0                                    # -0 equals +0
    nv = np.array([n, n, n], np.int32)
    out = torch.empty((R, 512), dtype=torch.int32, device="cuda")
    csa.csa_topk(R, torch.from_numpy(sc).cuda(), ld, torch.from_numpy(nv).cuda(), n, 512, out)
    got = out.cpu().numpy()
    for r in range(R):
        assert np.array_equal(got[r], oracle.topk_row(sc[r], n)), r


@pytest.mark.parametrize("n", [20000, 65536])
def test_topk_candidate_overflow(n):
    """More than 4096 entries tie at the 512th value: the per-row kernel's
    candidate list overflows and the whole-row radix path decides."""
    g = np.random.default_rng(n + 1)
    R, ld = 2, n
    sc = g.standard_normal((R, ld)).astype(np.float32)
    sc[0, ::3] = 1.5                                 # a third of the row ties
    sc[0, 7] = 9.0
    sc[1, :] = np.float32(2.0) ** -140               # subnormal spread
    sc[1, ::5] = np.float32(3.0) * np.float32(2.0) ** -140
    nv = np.array([n, n], np.int32)
    out = torch.empty((R, 512), dtype=torch.int32, device="cuda")
    csa.csa_topk(R, torch.from_numpy(sc).cuda(), ld, torch.from_numpy(nv).cuda(), n, 512, out)
    got = out.cpu().numpy()
    for r in range(R):
        assert np.array_equal(got[r], oracle.topk_row(sc[r], n)), r


def test_topk_rows_of_different_lengths():
    g = np.random.default_rng(5)
    R, ld = 9, 40000
    sc = g.standard_normal((R, ld)).astype(np.float32)
    nv = np.array([0, 5, 512, 513, 1000, 17000, 39999, 40000, 600], np.int32)
    out = torch.empty((R, 512), dtype=torch.int32, device="cuda")
    csa.csa_topk(R, torch.from_numpy(sc).cuda(), ld, torch.from_numpy(nv).cuda(), ld, 512, out)
    got = out.cpu().numpy()
    for r in range(R):
        assert np.array_equal(got[r], oracle.topk_row(sc[r], int(nv[r]))), r


def test_topk_long_and_short_rows_in_one_call():
    """Rows longer than 16384 entries take a whole cluster, shorter ones a CTA
    each, in one launch: the boundary lengths, a short row whose cut ties
    overflow the candidate list, and rows of at most 512 entries."""
    g = np.random.default_rng(11)
    R, ld = 8, 50000
    sc = g.standard_normal((R, ld)).astype(np.float32)
    sc[3, :9000:3] = 2.5                             # a third of a short row ties
    sc[3, 5] = 7.0
    sc[5] = np.round(sc[5] * 4) / 4                  # coarse values: many ties at the cut
    nv = np.array([50000, 16384, 16385, 9000, 700, 30000, 513, 0], np.int32)
    out = torch.empty((R, 512), dtype=torch.int32, device="cuda")
    csa.csa_topk(R, torch.from_numpy(sc).cuda(), ld, torch.from_numpy(nv).cuda(), ld, 512, out)
    got = out.cpu().numpy()
    for r in range(R):
        assert np.array_equal(got[r], oracle.topk_row(sc[r], int(nv[r]))), r


# --------------------------------------------------------------- attention
@pytest.mark.parametrize("H,ctx,rows", [(16, [1, 2, 100, 700, 1025, 3000], 1), (64, [300, 2100], 1),
                                        (32, [1500, 2000], 6)])
def test_sparse_attention_matches_oracle(H, ctx, rows):
    wl = W.custom("attn", 41 + H, ctx, [min(rows, c) for c in ctx], H=H, Hi=16, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    ref = oracle.build_cache(wl)
    q_idx, w, q = wl.step_queries()
    _, _, topk, _ = oracle.decode(ref, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale)
    tk = torch.from_numpy(topk).cuda()
    out = torch.empty((wl.R, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.R, H), device="cuda")
    ws = torch.zeros(csa.csa_workspace_size(csa.OP_SPARSE_ATTN, wl.R, wl.max_entries, H), dtype=torch.uint8,
                     device="cuda")
    csa.csa_sparse_attn(st.cache, st.window, s["rows"], tk, H, s["q"], wl.softmax_scale, out, lse, ws)
    rc, flags = csa.csa_check_device_status(ws)
    assert rc == 0 and flags == 0, flags
    o_ref = np.zeros((wl.R, H, 512), np.float32)
    l_ref = np.zeros((wl.R, H), np.float32)
    for r in range(wl.R):
        o_ref[r], l_ref[r] = oracle.attention_row(ref, wl.row_req[r], wl.row_pos[r], topk[r], q[r],
                                                  wl.softmax_scale)
    norm, l2 = parity.check_attention(out.float().cpu().numpy(), o_ref, lse.cpu().numpy(), l_ref)
    print(f"attention H={H}: max normalised err {norm:.2e}, rel L2 {l2:.2e}")


@pytest.mark.parametrize("cfg,compress", [(3, False), (4, False), (3, True)])
def test_step_call_equals_append_then_decode(cfg, compress):
    """csa_step (the append and the decode in one call, the score prep running
    beside the append) leaves every cache byte and every output bit equal to
    csa_append followed by csa_decode."""
    wl = W.config(cfg)
    states = []
    for fused in (False, True):
        st = DeviceState(wl)
        st.build_history()
        if compress:
            st.set_compress(W.compress_inputs(cfg, int(wl.ctx_len.max())))
        s = st.step_inputs()
        if fused:
            st.step(s)
        else:
            st.step_append(s)
            st.step_decode(s)
        rc, flags = csa.csa_check_device_status(s["ws"])
        assert rc == 0 and flags == 0, (fused, flags)
        states.append((st, s))
    (a, sa), (b, sb) = states
    same = lambda x, y: torch.equal(x.contiguous().view(torch.uint8), y.contiguous().view(torch.uint8))
    for name in ("kv_pool", "idx_pool", "win_codes", "win_scale", "pending"):
        x, y = getattr(a, name), getattr(b, name)
        assert (x is None and y is None) or same(x, y), name
    for key in ("topk", "out", "lse"):
        assert same(sa[key], sb[key]), key


@pytest.mark.parametrize("R", [30, 40, 60])
def test_attention_cluster_split_counts(R):
    """Row counts that give 5, 3 and 2 splits per row: the row's CTAs run as one
    cluster and merge their partials in shared memory (5-CTA clusters may be cut
    to fewer splits where they would not all be resident at once)."""
    ctx = list(np.random.default_rng(R).integers(2100, 4000, R))
    wl = W.custom("attn_cl", 90 + R, ctx, [1] * R, H=64, Hi=16, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    st.step_decode(s)
    rc, flags = csa.csa_check_device_status(s["ws"])
    assert rc == 0 and flags == 0, flags
    ref = oracle.build_cache(wl)
    q_idx, w, q = wl.step_queries()
    out, lse, topk, scores = oracle.decode(ref, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale, threads=8)
    gt = s["topk"].cpu().numpy()
    n = wl.row_entries()
    for r in range(wl.R):
        parity.check_topk_row(gt[r], scores[r], int(n[r]))
        if not np.array_equal(gt[r], topk[r]):
            out[r], lse[r] = oracle.attention_row(ref, wl.row_req[r], wl.row_pos[r], gt[r], q[r], wl.softmax_scale)
    norm, l2 = parity.check_attention(s["out"].float().cpu().numpy(), out, s["lse"].cpu().numpy(), lse)
    print(f"attention R={R}: max normalised err {norm:.2e}, rel L2 {l2:.2e}")


def test_attention_many_rows_single_split():
    """Enough rows that each row runs in one CTA (no split merge)."""
    ctx = list(np.random.default_rng(7).integers(600, 1400, 160))
    wl = W.custom("attn1", 47, ctx, [1] * 160, H=16, Hi=16)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    st.step_decode(s)
    rc, flags = csa.csa_check_device_status(s["ws"])
    assert rc == 0 and flags == 0
    ref = oracle.build_cache(wl)
    q_idx, w, q = wl.step_queries()
    out, lse, topk, scores = oracle.decode(ref, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale, threads=8)
    gt = s["topk"].cpu().numpy()
    n = wl.row_entries()
    for r in range(wl.R):
        parity.check_topk_row(gt[r], scores[r], int(n[r]))
    parity.check_attention(s["out"].float().cpu().numpy(), out, s["lse"].cpu().numpy(), lse)


def test_decode_more_rows_than_sms_mixed_lengths():
    """More rows than SMs (the attention runs in two waves) of very different
    lengths: rows with no entry, with one to four tiles, with partial windows;
    the index score's CTAs then hold many short segments."""
    base = [1, 2, 3, 100, 260, 700, 1025, 1600, 3000]
    ctx = [base[i % len(base)] for i in range(200)]
    wl = W.custom("attn_sk", 53, ctx, [1] * 200, H=32, Hi=32)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    st.step_decode(s)
    rc, flags = csa.csa_check_device_status(s["ws"])
    assert rc == 0 and flags == 0
    ref = oracle.build_cache(wl)
    q_idx, w, q = wl.step_queries()
    out, lse, topk, scores = oracle.decode(ref, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale, threads=8)
    gt = s["topk"].cpu().numpy()
    n = wl.row_entries()
    for r in range(wl.R):
        parity.check_topk_row(gt[r], scores[r], int(n[r]))
    parity.check_attention(s["out"].float().cpu().numpy(), out, s["lse"].cpu().numpy(), lse)


@pytest.mark.parametrize("H", [64, 16])
def test_attention_tail_split(H):
    """Rows just past one wave of one CTA per SM: the last wave's rows are
    split over several CTAs whose partials merge through the workspace.  The
    output matches the oracle with and without the split (a workspace too
    small for the partials runs every row whole), the rows before the tail are
    bit-equal either way, and a second call on the same workspace (arrival
    counters back at zero) gives the same bits."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    R = sms + 7
    base = [600, 1500, 2600, 4100]
    ctx = [base[i % len(base)] + i for i in range(R)]
    wl = W.custom("tail", 71, ctx, [1] * R, H=H, Hi=16, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    ref = oracle.build_cache(wl)
    q_idx, w, q = wl.step_queries()
    _, _, topk, _ = oracle.decode(ref, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale, threads=8)
    tk = torch.from_numpy(topk).cuda()
    full = csa.csa_workspace_size(csa.OP_SPARSE_ATTN, R, wl.max_entries, H)
    assert full > 256                                    # partials for 7 rows x 5 splits
    assert csa.csa_workspace_size(csa.OP_SPARSE_ATTN, sms, wl.max_entries, H) == 256
    o_ref = np.zeros((R, H, 512), np.float32)
    l_ref = np.zeros((R, H), np.float32)
    for r in range(R):
        o_ref[r], l_ref[r] = oracle.attention_row(ref, wl.row_req[r], wl.row_pos[r], topk[r], q[r],
                                                  wl.softmax_scale)
    outs = []
    ws_full = torch.zeros(full, dtype=torch.uint8, device="cuda")
    for ws in (ws_full, torch.zeros(256, dtype=torch.uint8, device="cuda"), ws_full):
        out = torch.full((R, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((R, H), float("nan"), device="cuda")
        csa.csa_sparse_attn(st.cache, st.window, s["rows"], tk, H, s["q"], wl.softmax_scale, out, lse, ws)
        rc, flags = csa.csa_check_device_status(ws)
        assert rc == 0 and flags == 0, flags
        parity.check_attention(out.float().cpu().numpy(), o_ref, lse.cpu().numpy(), l_ref)
        outs.append((out.view(torch.int16).cpu().numpy(), lse.cpu().numpy()))
    assert np.array_equal(outs[0][0][:sms], outs[1][0][:sms])
    assert np.array_equal(outs[0][1][:sms], outs[1][1][:sms])
    assert np.array_equal(outs[0][0], outs[2][0]) and np.array_equal(outs[0][1], outs[2][1])


def test_decode_tail_split_with_a_workspace_reused_across_shapes():
    """One workspace serves decodes of different row counts: the tail split's
    arrival counters sit after the scores and the top-k, so their place moves
    with the shapes and lands on bytes an earlier call wrote; each call zeroes
    them first.  All rows, then a prefix of them, then all rows again: every
    output matches the oracle and the repeated call is bit-equal."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    R, Rp = sms + 40, sms + 7
    ctx = [600 + 23 * i for i in range(R)]
    wl = W.custom("tailws", 81, ctx, [1] * R, H=16, Hi=16, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    ws = torch.zeros(max(csa.csa_workspace_size(csa.OP_DECODE, n, wl.max_entries, wl.H) for n in (R, Rp)),
                     dtype=torch.uint8, device="cuda")
    ref = oracle.build_cache(wl)
    q_idx, w, q = wl.step_queries()
    _, _, _, scores = oracle.decode(ref, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale, threads=8)
    n = wl.row_entries()

    def run(k):
        rows = csa.make_rows(s["row_req"][:k], s["row_pos"][:k], wl.max_entries, 1)
        out = torch.full((k, wl.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((k, wl.H), float("nan"), device="cuda")
        topk = torch.empty((k, 512), dtype=torch.int32, device="cuda")
        csa.csa_decode(st.cache, st.window, rows, wl.Hi, s["q_idx"][:k], s["w"][:k], wl.H, s["q"][:k],
                       wl.softmax_scale, out, lse, topk, ws)
        rc, flags = csa.csa_check_device_status(ws)
        assert rc == 0 and flags == 0, flags
        gt = topk.cpu().numpy()
        o_ref = np.zeros((k, wl.H, 512), np.float32)
        l_ref = np.zeros((k, wl.H), np.float32)
        for r in range(k):
            parity.check_topk_row(gt[r], scores[r], int(n[r]))
            o_ref[r], l_ref[r] = oracle.attention_row(ref, wl.row_req[r], wl.row_pos[r], gt[r], q[r],
                                                      wl.softmax_scale)
        parity.check_attention(out.float().cpu().numpy(), o_ref, lse.cpu().numpy(), l_ref)
        return out, lse

    out0, lse0 = run(R)
    run(Rp)
    out2, lse2 = run(R)
    assert torch.equal(out2.view(torch.int16), out0.view(torch.int16)) and torch.equal(lse2, lse0)


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("H,Hi,rows", [(16, 16, 1), (64, 64, 6), (32, 32, 2), (64, 128, 2), (16, 96, 1)])
def test_decode_end_to_end(H, Hi, rows):
    ctx = [1, 3, 513 * 2, 1024 + 1, 2500, 5000 + 3]
    wl = W.custom("dec", 51 + rows, ctx, [min(rows, c) for c in ctx], H=H, Hi=Hi, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    st.step_decode(s)
    rc, flags = csa.csa_check_device_status(s["ws"])
    assert rc == 0 and flags == 0, flags
    ref = oracle.build_cache(wl)
    q_idx, w, q = wl.step_queries()
    _, _, _, scores = oracle.decode(ref, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale)
    gt = s["topk"].cpu().numpy()
    n = wl.row_entries()
    o_ref = np.zeros((wl.R, H, 512), np.float32)
    l_ref = np.zeros((wl.R, H), np.float32)
    for r in range(wl.R):
        parity.check_topk_row(gt[r], scores[r], int(n[r]))
        o_ref[r], l_ref[r] = oracle.attention_row(ref, wl.row_req[r], wl.row_pos[r], gt[r], q[r], wl.softmax_scale)
    parity.check_attention(s["out"].float().cpu().numpy(), o_ref, s["lse"].cpu().numpy(), l_ref)


def test_plan_reused_across_layers():
    """Cross-layer reuse: layers that read the same cache share one top-512
    plan (csa_decode's topk_out); each further layer runs only the sparse
    attention with its own q, and matches a full csa_decode for that layer
    bit for bit."""
    ctx = [700, 2500, 5003, 9000]
    wl = W.custom("plan", 61, ctx, [1] * len(ctx), H=64, Hi=64, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    st.step_decode(s)                                    # layer 0: score + top-512 + attention
    plan = s["topk"].clone()
    g = np.random.default_rng(7)
    ws_a = torch.zeros(csa.csa_workspace_size(csa.OP_SPARSE_ATTN, wl.R, wl.max_entries, wl.H), dtype=torch.uint8,
                       device="cuda")
    for layer in (1, 2):
        q_l = torch.from_numpy(W.f32_to_bf16_bits(g.standard_normal((wl.R, wl.H, 512)).astype(np.float32))
                               .view(np.int16)).cuda().view(torch.bfloat16)
        out_p = torch.empty_like(s["out"])
        lse_p = torch.empty_like(s["lse"])
        csa.csa_sparse_attn(st.cache, st.window, s["rows"], plan, wl.H, q_l, wl.softmax_scale, out_p, lse_p, ws_a)
        s_full = dict(s)
        s_full["q"] = q_l
        s_full["out"], s_full["lse"] = torch.empty_like(s["out"]), torch.empty_like(s["lse"])
        s_full["topk"] = torch.empty_like(s["topk"])
        st.step_decode(s_full)
        torch.cuda.synchronize()
        assert torch.equal(s_full["topk"], plan)           # the same cache and indexer query: the same plan
        assert torch.equal(out_p, s_full["out"]) and torch.equal(lse_p, s_full["lse"])


def test_decode_is_deterministic():
    wl = W.custom("det", 61, [3000, 5000], [2, 1], H=64, Hi=64)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    st.step_decode(s)
    o1, t1 = s["out"].clone(), s["topk"].clone()
    st.step_decode(s)
    assert torch.equal(o1, s["out"]) and torch.equal(t1, s["topk"])


# ------------------------------------------------ compressed append (NEXT f-3)
def _compress_dev(c):
    return {k: (torch.from_numpy(c[k]).cuda() if isinstance(c[k], np.ndarray) else c[k]) for k in c}


@pytest.mark.parametrize("P", [2, 1])
def test_append_compress_bit_exact(P):
    """csa_append_compress (RMSNorm with gamma, rotate-half RoPE, then the
    quantisers) writes the same bytes as the oracle, over two calls per
    request (whole history, then a few tokens with odd and even starts, so
    pooling crosses the pending token)."""
    ctx = [1, 2, 3, 63, 64, 65, 129, 300, 1025]
    new = [1, 2, 1, 6, 3, 1, 6, 2, 5]
    wl = W.custom("cmp", 14 + P, ctx, new, H=16, Hi=16, P=P, shuffle=True)
    cmp = W.compress_inputs(14 + P, int(wl.ctx_len.max()))
    dcmp = _compress_dev(cmp)
    st = DeviceState(wl)
    ref = oracle.Cache(wl.num_pages, wl.page_table, wl.P, wl.win_cap)
    comp = csa.make_compress(dcmp["kv_gamma"], dcmp["idx_gamma"], dcmp["eps"], dcmp["rope_cos"], dcmp["rope_sin"])
    for lo_of, hi_of in ((lambda b: 0, lambda b: int(wl.hist_len[b])),
                         (lambda b: int(wl.hist_len[b]), lambda b: int(wl.ctx_len[b]))):
        xs, ys, cnt = [], [], []
        pos0 = np.zeros(wl.B, np.int32)
        for b in range(wl.B):
            lo, hi = lo_of(b), hi_of(b)
            x, y = wl.tokens(b, lo, hi)
            xs.append(x)
            ys.append(y)
            pos0[b] = lo
            cnt.append(hi - lo)
        tok_off = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        X, Y = np.concatenate(xs), np.concatenate(ys)
        csa.csa_append_compress(st.cache, st.window, torch.from_numpy(pos0).cuda(), torch.from_numpy(tok_off).cuda(),
                                int(tok_off[-1]), torch.from_numpy(X.view(np.int16)).cuda(),
                                torch.from_numpy(Y.view(np.int16)).cuda(), st.pending, comp, st.ws_append)
        assert ref.append(pos0, tok_off, X, Y, compress=cmp) == 0
    rc, flags = csa.csa_check_device_status(st.ws_append)
    assert rc == 0 and flags == 0, flags
    _pools_equal(st, ref)
    plain = oracle.build_cache(wl)                       # the steps changed the entries
    assert not np.array_equal(plain.kv_pool, ref.kv_pool)


def test_append_compress_flags_positions_beyond_the_tables():
    wl = W.custom("cmpf", 16, [200], [1], H=16, Hi=16)
    cmp = W.compress_inputs(16, 100)                      # rows for positions 0..99 only
    dcmp = _compress_dev(cmp)
    st = DeviceState(wl)
    comp = csa.make_compress(dcmp["kv_gamma"], dcmp["idx_gamma"], dcmp["eps"], dcmp["rope_cos"], dcmp["rope_sin"])
    x, y = wl.tokens(0, 0, 200)
    csa.csa_append_compress(st.cache, st.window, torch.zeros(1, dtype=torch.int32).cuda(),
                            torch.tensor([0, 200], dtype=torch.int32).cuda(), 200,
                            torch.from_numpy(x.view(np.int16)).cuda(), torch.from_numpy(y.view(np.int16)).cuda(),
                            st.pending, comp, st.ws_append)
    rc, flags = csa.csa_check_device_status(st.ws_append)
    assert rc == 5 and (flags & csa.FLAG_APPEND)
    ref = oracle.Cache(wl.num_pages, wl.page_table, wl.P, wl.win_cap)
    assert ref.append(np.zeros(1, np.int32), np.array([0, 200], np.int32), x, y, compress=cmp) == -3
    _pools_equal(st, ref)                                 # entries 0..49 written, the rest untouched


# ------------------------------------------ decode plan (NEXT f-4) and rotary q (f-3)
def _host_plan(wl, topk):
    """Each selected index through the page table: page * 64 + slot, -1 kept."""
    plan = np.full_like(topk, -1)
    for r in range(wl.R):
        b = int(wl.row_req[r])
        for j, e in enumerate(topk[r]):
            if e >= 0:
                plan[r, j] = int(wl.page_table[b, e // 64]) * 64 + int(e) % 64
    return plan


def test_decode_plan_is_the_resolved_selection_and_later_layers_reuse_it():
    """csa_decode_ex writes the plan (every selected index resolved through the
    page table); a further layer's csa_sparse_attn_ex reading that plan instead
    of the indices gives the same bits as reading the indices."""
    ctx = [700, 2500, 5003, 9000, 130, 3]
    wl = W.custom("plan2", 62, ctx, [1] * len(ctx), H=64, Hi=64, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    plan = torch.full((wl.R, 512), -7, dtype=torch.int32, device="cuda")
    csa.csa_decode_ex(st.cache, st.window, s["rows"], wl.Hi, s["q_idx"], s["w"], wl.H, s["q"], wl.softmax_scale,
                      s["out"], s["lse"], s["topk"], csa.make_opts(plan_out=plan), s["ws"])
    rc, flags = csa.csa_check_device_status(s["ws"])
    assert rc == 0 and flags == 0, flags
    topk = s["topk"].cpu().numpy()
    assert np.array_equal(plan.cpu().numpy(), _host_plan(wl, topk))
    ws_a = torch.zeros(256, dtype=torch.uint8, device="cuda")
    g = np.random.default_rng(8)
    for layer in (1, 2):
        q_l = torch.from_numpy(W.f32_to_bf16_bits(g.standard_normal((wl.R, wl.H, 512)).astype(np.float32))
                               .view(np.int16)).cuda().view(torch.bfloat16)
        o_i, l_i = torch.empty_like(s["out"]), torch.empty_like(s["lse"])
        o_p, l_p = torch.empty_like(s["out"]), torch.empty_like(s["lse"])
        csa.csa_sparse_attn(st.cache, st.window, s["rows"], s["topk"], wl.H, q_l, wl.softmax_scale, o_i, l_i, ws_a)
        csa.csa_sparse_attn_ex(st.cache, st.window, s["rows"], None, wl.H, q_l, wl.softmax_scale, o_p, l_p,
                               csa.make_opts(plan_in=plan), ws_a)
        rc, flags = csa.csa_check_device_status(ws_a)
        assert rc == 0 and flags == 0, flags
        assert torch.equal(o_i, o_p) and torch.equal(l_i, l_p)


_E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6], np.float64)


def _rope_key_norm(ref, b, pos, sel):
    """Largest norm of the last 64 dims over a row's keys (selected entries and
    window tokens); rotations keep it."""
    best = 0.0
    for e in sel[sel >= 0]:
        data, sc = ref.main_entry(b, int(e))
        codes = np.stack([data & 15, data >> 4], axis=1).reshape(-1)
        v = _E2M1[codes] * np.repeat([oracle.e4m3_decode(c) for c in sc], 16)
        best = max(best, float(np.linalg.norm(v[448:])))
    for p in range(max(0, pos - 127), pos + 1):
        codes, s = ref.window_slot(b, p)
        v = np.array([oracle.e4m3_decode(c) for c in codes[448:]]) * s
        best = max(best, float(np.linalg.norm(v)))
    return best


def _check_rope_attention(wl, ref, topk, q, out, lse, o_ref, l_ref):
    """J-3 on the outputs.  For lse: the rotated query and window tokens are
    rounded once to fp16 for the tensor cores (unrotated, both are exact there),
    so each logit may move by scale * 2 * 2^-11 * |q_rope| * |k_rope| on top of
    the fp32 rounding the 1e-4 rule covers (Cauchy-Schwarz over the 64 rotated
    dims); the lse moves by at most the largest such change."""
    norm, l2 = parity.check_attention(out, o_ref)
    u = 2.0 ** -11
    for r in range(wl.R):
        qn = np.linalg.norm(W.bf16_bits_to_f32(q[r]).astype(np.float64)[:, 448:], axis=1)
        kn = _rope_key_norm(ref, int(wl.row_req[r]), int(wl.row_pos[r]), topk[r])
        tol = parity.LSE_TOL + wl.softmax_scale * 2 * u * qn * kn
        assert (np.abs(lse[r].astype(np.float64) - l_ref[r]) <= tol).all(), r
    return norm, l2


def _rope_tables(seed, rows):
    c = W.compress_inputs(seed, rows)
    return torch.from_numpy(c["rope_cos"]).cuda(), torch.from_numpy(c["rope_sin"]).cuda(), c


@pytest.mark.parametrize("H,ctx,rows", [(64, [1, 60, 700, 2100, 5000], 1), (16, [400, 3000], 6)])
def test_rotary_attention_matches_oracle(H, ctx, rows):
    """The query and the window tokens rotated inside the attention step, the
    global entries as stored, against the oracle's rotary attention (J-3)."""
    wl = W.custom("rope", 63 + H, ctx, [min(rows, c) for c in ctx], H=H, Hi=16, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    ref = oracle.build_cache(wl)
    q_idx, w, q = wl.step_queries()
    _, _, topk, _ = oracle.decode(ref, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale)
    cs, sn, c = _rope_tables(63, int(wl.ctx_len.max()))
    out = torch.empty((wl.R, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.R, H), device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    csa.csa_sparse_attn_ex(st.cache, st.window, s["rows"], torch.from_numpy(topk).cuda(), H, s["q"],
                           wl.softmax_scale, out, lse, csa.make_opts(rope_cos=cs, rope_sin=sn), ws)
    rc, flags = csa.csa_check_device_status(ws)
    assert rc == 0 and flags == 0, flags
    o_ref = np.zeros((wl.R, H, 512), np.float32)
    l_ref = np.zeros((wl.R, H), np.float32)
    for r in range(wl.R):
        o_ref[r], l_ref[r], rc_o = oracle.attention_row_rope(ref, wl.row_req[r], wl.row_pos[r], topk[r], q[r],
                                                             wl.softmax_scale, c["rope_cos"], c["rope_sin"])
        assert rc_o == 0
    norm, l2 = _check_rope_attention(wl, ref, topk, q, out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref)
    print(f"rotary attention H={H}: max normalised err {norm:.2e}, rel L2 {l2:.2e}")
    # a row past the tables is flagged and left empty
    short_c, short_s = cs[: int(wl.row_pos.max())].contiguous(), sn[: int(wl.row_pos.max())].contiguous()
    csa.csa_sparse_attn_ex(st.cache, st.window, s["rows"], torch.from_numpy(topk).cuda(), H, s["q"],
                           wl.softmax_scale, out, lse, csa.make_opts(rope_cos=short_c, rope_sin=short_s), ws)
    rc, flags = csa.csa_check_device_status(ws)
    assert rc == 5 and (flags & csa.FLAG_ROW_INVALID)
    last = int(np.argmax(wl.row_pos))
    assert not out[last].float().any() and torch.isneginf(lse[last]).all()


def test_step_ex_rotates_keys_query_and_window_with_one_table():
    """csa_step_ex with the compressor's rotary tables in both places equals
    csa_append_compress + csa_decode_ex bit for bit, and matches the oracle
    (compressed cache, rotary attention on the GPU's selection)."""
    ctx = [3000, 4100, 777, 5003]
    wl = W.custom("steprope", 64, ctx, [6, 6, 6, 6], H=64, Hi=64, shuffle=True)
    cs, sn, c = _rope_tables(64, int(wl.ctx_len.max()))
    dev = {k: (torch.from_numpy(v).cuda() if isinstance(v, np.ndarray) else v) for k, v in c.items()}
    comp = csa.make_compress(dev["kv_gamma"], dev["idx_gamma"], dev["eps"], dev["rope_cos"], dev["rope_sin"])
    opts = csa.make_opts(rope_cos=cs, rope_sin=sn)
    states = []
    for fused in (False, True):
        st = DeviceState(wl)
        st.set_compress(c)
        # history through the compressed append too
        pos0 = np.zeros(wl.B, np.int32)
        cnt = wl.hist_len.astype(np.int64)
        xs, ys = zip(*[wl.tokens(b, 0, int(wl.hist_len[b])) for b in range(wl.B)])
        csa.csa_append_compress(st.cache, st.window, torch.from_numpy(pos0).cuda(),
                                torch.from_numpy(np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)).cuda(),
                                int(cnt.sum()), torch.from_numpy(np.concatenate(xs).view(np.int16)).cuda(),
                                torch.from_numpy(np.concatenate(ys).view(np.int16)).cuda(), st.pending, comp,
                                st.ws_append)
        s = st.step_inputs()
        if fused:
            csa.csa_step_ex(st.cache, st.window, s["pos0"], s["tok_off"], wl.R, s["kv_new"], s["idx_new"],
                            st.pending, comp, s["rows"], wl.Hi, s["q_idx"], s["w"], wl.H, s["q"], wl.softmax_scale,
                            s["out"], s["lse"], s["topk"], opts, s["ws"])
        else:
            csa.csa_append_compress(st.cache, st.window, s["pos0"], s["tok_off"], wl.R, s["kv_new"], s["idx_new"],
                                    st.pending, comp, st.ws_append)
            csa.csa_decode_ex(st.cache, st.window, s["rows"], wl.Hi, s["q_idx"], s["w"], wl.H, s["q"],
                              wl.softmax_scale, s["out"], s["lse"], s["topk"], opts, s["ws"])
        rc, flags = csa.csa_check_device_status(s["ws"])
        assert rc == 0 and flags == 0, (fused, flags)
        states.append((st, s))
    (a, sa), (b, sb) = states
    for key in ("topk", "out", "lse"):
        assert torch.equal(sa[key], sb[key]), key
    assert torch.equal(a.kv_pool, b.kv_pool) and torch.equal(a.idx_pool, b.idx_pool)
    ref = oracle.Cache(wl.num_pages, wl.page_table, wl.P, wl.win_cap)
    xs, ys = zip(*[wl.tokens(bq, 0, int(wl.ctx_len[bq])) for bq in range(wl.B)])
    tok = np.concatenate([[0], np.cumsum(wl.ctx_len)]).astype(np.int32)
    assert ref.append(np.zeros(wl.B, np.int32), tok, np.concatenate(xs), np.concatenate(ys), compress=c) == 0
    assert np.array_equal(b.kv_pool.cpu().numpy(), ref.kv_pool)
    q_idx, w, q = wl.step_queries()
    _, _, _, scores = oracle.decode(ref, wl.row_req, wl.row_pos, q_idx, w, q, wl.softmax_scale)
    gt = sb["topk"].cpu().numpy()
    n = wl.row_entries()
    o_ref = np.zeros((wl.R, wl.H, 512), np.float32)
    l_ref = np.zeros((wl.R, wl.H), np.float32)
    for r in range(wl.R):
        parity.check_topk_row(gt[r], scores[r], int(n[r]))
        o_ref[r], l_ref[r], _ = oracle.attention_row_rope(ref, wl.row_req[r], wl.row_pos[r], gt[r], q[r],
                                                          wl.softmax_scale, c["rope_cos"], c["rope_sin"])
    _check_rope_attention(wl, ref, gt, q, sb["out"].float().cpu().numpy(), sb["lse"].cpu().numpy(), o_ref, l_ref)


# ------------------------------------------------ two-level candidate filter (NEXT f-2)
@pytest.mark.parametrize("n", [1, 64, 65, 511, 700, 5000, 70000, 262144])
def test_topk_two_level_exact(n):
    g = np.random.default_rng(n + 5)
    R = 3
    ld = max(64, ((n + 63) // 64) * 64)
    sc = (g.integers(0, 400, (R, ld)) / 16).astype(np.float32)   # many exact ties
    sc[1] = -sc[1]
    sc[2, : n // 2] = 0.0
    sc[2, n // 3: n // 2] = -0.0
    nv = np.array([n, n, n], np.int32)
    nb = (n + 63) // 64
    d_sc, d_nv = torch.from_numpy(sc).cuda(), torch.from_numpy(nv).cuda()
    out = torch.empty((R, 512), dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for B in sorted({1, 7, 64, 128, min(nb, 128)}):
        csa.csa_topk_two_level(R, d_sc, ld, d_nv, n, B, out, ws)
        got = out.cpu().numpy()
        for r in range(R):
            assert np.array_equal(got[r], oracle.topk_two_level(sc[r], n, B)), (B, r)
    rc, flags = csa.csa_check_device_status(ws)
    assert rc == 0 and flags == 0


def test_decode_with_two_level_filter():
    """csa_decode_ex with candidate_blocks selects exactly what the standalone
    filter selects from the same scores, and attends over that selection."""
    ctx = [700, 9000, 30000, 2500, 64000, 129]
    wl = W.custom("two", 65, ctx, [1] * len(ctx), H=64, Hi=64, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    B = 32
    csa.csa_decode_ex(st.cache, st.window, s["rows"], wl.Hi, s["q_idx"], s["w"], wl.H, s["q"], wl.softmax_scale,
                      s["out"], s["lse"], s["topk"], csa.make_opts(candidate_blocks=B), s["ws"])
    rc, flags = csa.csa_check_device_status(s["ws"])
    assert rc == 0 and flags == 0, flags
    ld = ((wl.max_entries + 63) // 64) * 64
    scores = torch.full((wl.R, ld), float("nan"), device="cuda")
    ws = torch.zeros(csa.csa_workspace_size(csa.OP_INDEX_SCORE, wl.R, wl.max_entries, 16), dtype=torch.uint8,
                     device="cuda")
    csa.csa_index_score(st.cache, s["rows"], wl.Hi, s["q_idx"], s["w"], scores, ld, ws)
    n = torch.from_numpy(wl.row_entries()).cuda()
    want = torch.empty_like(s["topk"])
    csa.csa_topk_two_level(wl.R, scores, ld, n, wl.max_entries, B, want, ws)
    assert torch.equal(s["topk"], want)
    gt = s["topk"].cpu().numpy()
    sc = scores.cpu().numpy()
    nn = wl.row_entries()
    recall = []
    for r in range(wl.R):
        assert np.array_equal(gt[r], oracle.topk_two_level(sc[r], int(nn[r]), B)), r
        flat = set(oracle.topk_row(sc[r], int(nn[r])).tolist()) - {-1}
        recall.append(len(flat & set(gt[r].tolist())) / max(1, len(flat)))
    ref = oracle.build_cache(wl)
    _, _, q = wl.step_queries()
    o_ref = np.zeros((wl.R, wl.H, 512), np.float32)
    l_ref = np.zeros((wl.R, wl.H), np.float32)
    for r in range(wl.R):
        o_ref[r], l_ref[r] = oracle.attention_row(ref, wl.row_req[r], wl.row_pos[r], gt[r], q[r], wl.softmax_scale)
    parity.check_attention(s["out"].float().cpu().numpy(), o_ref, s["lse"].cpu().numpy(), l_ref)
    print("two-level B=32 recall of the flat top-512 per row:", [round(x, 3) for x in recall])
