"""Failure detection on the GPU without a GPU fault.

Faults only the device can see are planted from the host (a page id outside
the pool, a selected index outside the row's visible range, a row length
beyond the host bound): the kernel skips the unit, raises its flag in the
status word, and leaves every other output as a clean call writes it.  The
time-out path is exercised by a wait budget too small for the index score's
first page copies to land: the kernel stops, raises CSA_FLAG_TIMEOUT, drains
what it issued and returns, and the next call on the same stream is exact."""
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


def _state(name, seed, ctx, H=16, Hi=64):
    wl = W.custom(name, seed, ctx, [1] * len(ctx), H=H, Hi=Hi, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    return wl, st, s


def _score(st, s, wl, Hi=64):
    ld = ((wl.max_entries + 63) // 64) * 64
    scores = torch.full((wl.R, ld), float("nan"), device="cuda")
    ws = torch.zeros(csa.csa_workspace_size(csa.OP_INDEX_SCORE, wl.R, wl.max_entries, 16), dtype=torch.uint8,
                     device="cuda")
    csa.csa_index_score(st.cache, s["rows"], Hi, s["q_idx"], s["w"], scores, ld, ws)
    rc, flags = csa.csa_check_device_status(ws)
    return scores.cpu().numpy(), rc, flags


def test_score_wait_budget_runs_out_and_the_next_call_is_exact():
    wl, st, s = _state("tmo", 71, [20000, 30001, 9000, 64000])
    clean, rc, flags = _score(st, s, wl)
    assert rc == 0 and flags == 0
    try:
        csa.csa_set_wait_budget(200)                  # SM clocks: shorter than any page copy
        _, rc, flags = _score(st, s, wl)
        assert rc == 6 and (flags & csa.FLAG_TIMEOUT), (rc, flags)
    finally:
        csa.csa_set_wait_budget(0)                    # the default budget
    again, rc, flags = _score(st, s, wl)
    assert rc == 0 and flags == 0, flags
    assert np.array_equal(again.view(np.uint32), clean.view(np.uint32))


def test_score_flags_a_page_outside_the_pool():
    wl, st, s = _state("pgf", 72, [3000, 5001])
    clean, rc, flags = _score(st, s, wl)
    assert rc == 0 and flags == 0
    good = int(st.page_table[1, 3])
    st.page_table[1, 3] = wl.num_pages + 7            # entries 192..255 of request 1
    try:
        bad, rc, flags = _score(st, s, wl)
    finally:
        st.page_table[1, 3] = good
    assert rc == 5 and (flags & csa.FLAG_PAGE_OOB), (rc, flags)
    assert np.isneginf(bad[1, 192:256]).all()
    keep = np.ones_like(bad, dtype=bool)
    keep[1, 192:256] = False
    assert np.array_equal(bad[keep].view(np.uint32), clean[keep].view(np.uint32))


def _attn(st, s, wl, topk):
    out = torch.empty((wl.R, wl.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.R, wl.H), device="cuda")
    ws = torch.zeros(csa.csa_workspace_size(csa.OP_SPARSE_ATTN, wl.R, wl.max_entries, wl.H), dtype=torch.uint8,
                     device="cuda")
    csa.csa_sparse_attn(st.cache, st.window, s["rows"], topk, wl.H, s["q"], wl.softmax_scale, out, lse, ws)
    rc, flags = csa.csa_check_device_status(ws)
    return out, lse, rc, flags


def test_attention_skips_bad_entries_and_flags_them():
    """A selected index outside the row's visible range (CSA_FLAG_TOPK_OOB) and
    a selected entry whose page id is outside the pool (CSA_FLAG_PAGE_OOB)
    are skipped: the row attends to the rest, as the oracle does with those
    entries removed, and the other row is bit-equal to a clean call."""
    wl, st, s = _state("atf", 73, [3000, 4001])
    st.step_decode(s)
    rc, flags = csa.csa_check_device_status(s["ws"])
    assert rc == 0 and flags == 0
    topk = s["topk"].clone()
    out0, lse0, rc, flags = _attn(st, s, wl, topk)
    assert rc == 0 and flags == 0
    ref = oracle.build_cache(wl)
    _, _, q = wl.step_queries()
    n = wl.row_entries()
    tk = topk.cpu().numpy()

    # row 0: one index past the visible range
    bad = topk.clone()
    bad[0, 5] = int(n[0]) + 10
    out, lse, rc, flags = _attn(st, s, wl, bad)
    assert rc == 5 and (flags & csa.FLAG_TOPK_OOB), (rc, flags)
    assert torch.equal(out[1], out0[1]) and torch.equal(lse[1], lse0[1])
    sel = tk[0].copy()
    sel[5] = -1
    o_ref, l_ref = oracle.attention_row(ref, wl.row_req[0], wl.row_pos[0], sel, q[0], wl.softmax_scale)
    parity.check_attention(out[0].float().cpu().numpy(), o_ref, lse[0].cpu().numpy(), l_ref)

    # row 1: the page of its first selected entry points outside the pool
    lp = int(tk[1, 0]) // 64
    good = int(st.page_table[1, lp])
    st.page_table[1, lp] = wl.num_pages + 3
    try:
        out, lse, rc, flags = _attn(st, s, wl, topk)
    finally:
        st.page_table[1, lp] = good
    assert rc == 5 and (flags & csa.FLAG_PAGE_OOB), (rc, flags)
    assert torch.equal(out[0], out0[0]) and torch.equal(lse[0], lse0[0])
    sel = tk[1].copy()
    sel[(sel // 64) == lp] = -1
    o_ref, l_ref = oracle.attention_row(ref, wl.row_req[1], wl.row_pos[1], sel, q[1], wl.softmax_scale)
    parity.check_attention(out[1].float().cpu().numpy(), o_ref, lse[1].cpu().numpy(), l_ref)


def test_attention_tail_split_survives_a_flagged_row():
    """A tail row (rows past one wave of one CTA per SM, split over several
    CTAs that merge through the workspace) with a selected index outside its
    visible range: the row is flagged and merged without that entry, the other
    rows are bit-equal to a clean call, and a clean call on the same workspace
    afterwards is bit-equal again (every tail CTA counted itself in, so the
    arrival counters are back at zero)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    R = sms + 3
    ctx = [700 + 37 * i for i in range(R)]
    wl, st, s = _state("tlf", 74, ctx, H=16, Hi=16)
    st.step_decode(s)
    rc, flags = csa.csa_check_device_status(s["ws"])
    assert rc == 0 and flags == 0
    topk = s["topk"].clone()
    ws = torch.zeros(csa.csa_workspace_size(csa.OP_SPARSE_ATTN, wl.R, wl.max_entries, wl.H), dtype=torch.uint8,
                     device="cuda")
    assert ws.numel() > 256                              # the tail split's partials fit

    def run(tk):
        out = torch.full((wl.R, wl.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((wl.R, wl.H), float("nan"), device="cuda")
        csa.csa_sparse_attn(st.cache, st.window, s["rows"], tk, wl.H, s["q"], wl.softmax_scale, out, lse, ws)
        rc, flags = csa.csa_check_device_status(ws)
        return out, lse, rc, flags

    out0, lse0, rc, flags = run(topk)
    assert rc == 0 and flags == 0
    r = R - 1                                            # a row of the split last wave
    n = wl.row_entries()
    bad = topk.clone()
    bad[r, 7] = int(n[r]) + 5
    out, lse, rc, flags = run(bad)
    assert rc == 5 and (flags & csa.FLAG_TOPK_OOB), (rc, flags)
    assert torch.equal(out[:r], out0[:r]) and torch.equal(lse[:r], lse0[:r])
    ref = oracle.build_cache(wl)
    _, _, q = wl.step_queries()
    sel = topk[r].cpu().numpy().copy()
    sel[7] = -1
    o_ref, l_ref = oracle.attention_row(ref, wl.row_req[r], wl.row_pos[r], sel, q[r], wl.softmax_scale)
    parity.check_attention(out[r].float().cpu().numpy(), o_ref, lse[r].cpu().numpy(), l_ref)
    out2, lse2, rc, flags = run(topk)
    assert rc == 0 and flags == 0
    assert torch.equal(out2, out0) and torch.equal(lse2, lse0)


def test_topk_flags_a_row_longer_than_its_bound():
    g = np.random.default_rng(74)
    R, ld = 3, 4096
    sc = g.standard_normal((R, ld)).astype(np.float32)
    nv = np.array([1000, 4000, 2000], np.int32)          # row 1 exceeds max_n = 3000
    out = torch.empty((R, 512), dtype=torch.int32, device="cuda")
    ws = torch.zeros(csa.csa_workspace_size(csa.OP_TOPK, R, ld, 16), dtype=torch.uint8, device="cuda")
    csa.csa_topk(R, torch.from_numpy(sc).cuda(), ld, torch.from_numpy(nv).cuda(), 3000, 512, out, ws)
    rc, flags = csa.csa_check_device_status(ws)
    assert rc == 5 and (flags & csa.FLAG_ROW_INVALID), (rc, flags)
    got = out.cpu().numpy()
    assert np.array_equal(got[0], oracle.topk_row(sc[0], 1000))
    assert np.array_equal(got[1], oracle.topk_row(sc[1], 3000))      # clamped to the bound
    assert np.array_equal(got[2], oracle.topk_row(sc[2], 2000))
