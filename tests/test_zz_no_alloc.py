"""csa_index_score_noalloc: the index score for callers that cannot allocate
device memory -- a serving loop that reserved its memory at start-up and may
not call cudaMalloc while it decodes, or a C host with no device allocator.
The entry point uses the library's own fixed scratch array instead of a
caller workspace.  Through the C ABI, two calls in a row must give the same
scores as csa_index_score with a caller workspace; a size beyond the array is
rejected before any launch.  Device-detected faults land in the array's own
status word, which csa_check_device_status(NULL) reads.  This file runs last
(pytest collects it last)."""
import ctypes as C

import numpy as np
import pytest
import torch

import fp4_sparse_attention_csa_gb300 as csa
from fp4_sparse_attention_csa_gb300 import workloads as W
from fp4_sparse_attention_csa_gb300.session import DeviceState

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    csa.build.build()
    torch.cuda.set_device(0)
    wl = W.custom("noalloc", 77, [3000 + 6, 130 + 6, 9000 + 6], [6, 6, 6], H=16, Hi=64, shuffle=True)
    st = DeviceState(wl)
    st.build_history()
    s = st.step_inputs()
    st.step_append(s)
    ld = ((wl.max_entries + 63) // 64) * 64
    n = wl.row_entries()

    ref = torch.full((wl.R, ld), float("nan"), device="cuda")
    ws = torch.zeros(csa.csa_workspace_size(csa.OP_INDEX_SCORE, wl.R, wl.max_entries, 16), dtype=torch.uint8,
                     device="cuda")
    csa.csa_index_score(st.cache, s["rows"], wl.Hi, s["q_idx"], s["w"], ref, ld, ws)
    ref = ref.cpu().numpy()

    lib = csa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        got = torch.full((wl.R, ld), float("nan"), device="cuda")
        rc = lib.csa_index_score_noalloc(C.byref(st.cache), C.byref(s["rows"]), wl.Hi, s["q_idx"].data_ptr(),
                                         s["w"].data_ptr(), got.data_ptr(), ld, stream)
        assert rc == 0, (call, csa.STATUS_NAMES.get(rc, rc))
        rc, flags = csa.csa_check_device_status(None)      # the fixed array's status word
        assert rc == 0 and flags == 0, (call, rc, flags)
        g = got.cpu().numpy()
        for r in range(wl.R):
            # the same kernel on the same inputs: the same bits
            assert np.array_equal(g[r, :n[r]].view(np.uint32), ref[r, :n[r]].view(np.uint32)), (call, r)
            assert np.isnan(g[r, n[r]:]).all()


def test_noalloc_rejects_sizes_beyond_its_array():
    csa.build.build()
    torch.cuda.set_device(0)
    R = 2000                                                # 2000 rows x 128 heads x 68 B > 4 MiB
    req = torch.zeros(R, dtype=torch.int32, device="cuda")
    pos = torch.zeros(R, dtype=torch.int32, device="cuda")
    rows = csa.make_rows(req, pos, 64, R)
    pool = torch.zeros(18432, dtype=torch.uint8, device="cuda")
    ipool = torch.zeros(4352, dtype=torch.uint8, device="cuda")
    pt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    cache = csa.make_cache(pool, ipool, pt, 1, 2)
    q_idx = torch.zeros((R, 128, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((R, 128), device="cuda")
    sc = torch.zeros((R, 64), device="cuda")
    rc = csa.lib().csa_index_score_noalloc(C.byref(cache), C.byref(rows), 128, q_idx.data_ptr(), w.data_ptr(),
                                           sc.data_ptr(), 64, torch.cuda.current_stream().cuda_stream)
    assert rc == 3          # CSA_ERR_WORKSPACE_TOO_SMALL, nothing launched
