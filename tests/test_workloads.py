"""Seeded workload generator: determinism, chunk independence, the shapes the
pages describe, and the constructed tie group of the unpooled config."""
import numpy as np

import oracle
from fp4_sparse_attention_csa_gb300 import workloads as W
from util import read_golden


def test_tokens_are_chunk_independent_and_deterministic():
    wl = W.config(3)
    x, y = wl.tokens(5, 100, 9000)
    x2, y2 = wl.tokens(5, 4000, 9000)
    assert np.array_equal(x[3900:], x2) and np.array_equal(y[3900:], y2)
    x3, _ = W.config(3).tokens(5, 100, 200)
    assert np.array_equal(x[:100], x3)


def test_bf16_rounding_is_nearest_even():
    # bf16 keeps 7 fraction bits: 1 + 2^-8 is a tie (-> 1.0, even), 1 + 3*2^-8
    # is a tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    v = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1.0 + 2**-8 + 2**-20], np.float32)
    b = W.f32_to_bf16_bits(v)
    assert list(W.bf16_bits_to_f32(b)) == [1.0, 1.0, 1.0 + 2**-6, -2.5, 1.0 + 2**-7]


def test_config_shapes_follow_the_pages():
    g = {k: int(v) for k, v in read_golden("page_constants.txt")}
    c3 = W.config(3)
    assert c3.B == 32 and c3.R == 32 * g["max_verify_rows"]
    assert (c3.hist_len >= 3072).all() and (c3.hist_len <= 5120 + 1024).all()
    assert all(np.all(np.diff(c3.row_pos[c3.row_req == b]) == 1) for b in range(c3.B))
    c4 = W.config(4)
    assert c4.R == 128 and c4.ctx_len.min() >= 4096 and c4.ctx_len.max() <= 131072
    used = c4.page_table[c4.page_table >= 0]
    assert np.array_equal(np.sort(used), np.arange(c4.num_pages))      # a permutation
    assert not np.array_equal(used, np.arange(c4.num_pages))           # shuffled
    c5 = W.config(5)
    assert c5.P == 1 and c5.max_entries == 262144
    c1 = W.config(1)
    assert c1.max_entries == 2048 and c1.H == c1.Hi == 16
    c2 = W.config(2)
    assert c2.max_entries == 16384 and len(c2._salient_entries(0)) == round(0.05 * 16384)


def test_tie_group_straddles_rank_512():
    """The constructed group of bitwise-identical indexer keys holds rank 512."""
    wl = W.config(5)
    cache = oracle.Cache(wl.num_pages, wl.page_table, 1, window=False)
    x, y = wl.tokens(0, 0, 262144)
    pos0 = np.zeros(4, np.int32)
    off = np.array([0, 262144, 262144, 262144, 262144], np.int32)
    assert cache.append(pos0, off, np.zeros_like(x), y, window=False) == 0
    q_idx, w, _ = wl.step_queries()
    sc = oracle.index_score(cache, wl.row_req[:1], wl.row_pos[:1], q_idx[:1], w[:1])[0]
    grp, _, _ = wl._tie_sets(0)
    assert len({sc[i] for i in grp}) == 1
    tie = sc[grp[0]]
    above = int((sc > tie).sum())
    assert above < 512 < above + len(grp)
    top = oracle.topk_row(sc, 262144)
    chosen_ties = sorted(set(top) & set(grp.tolist()))
    assert chosen_ties == sorted(grp.tolist())[:512 - above]
