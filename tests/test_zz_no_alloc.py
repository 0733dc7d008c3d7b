"""The allocation-free variant of steps (2)+(3), step5_index_score_topk_noalloc, for
callers that cannot allocate device memory: it must pick the same regions, in the same
order, with the same scores as step5_index_score_topk given a caller workspace.

Two calls in a row with different row counts and summary capacities check that each
call clears what the previous one left in the shared fixed scratch.  Collected last
(file name) so that a failure here comes after every other test has run.
"""
import numpy as np
import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s5():
    import block_sparse_attention_step5_gb300 as s5
    s5.build()
    s5.load()
    return s5


def run_both(s5, w, t):
    geom = s5.STEP5_GEOMETRY
    dev = t["q"].device
    N, G = w.N, 4
    out = {}
    for kind in ("workspace", "noalloc"):
        ids = torch.full((N, G, 512), -7, dtype=torch.int32, device=dev)
        cnt = torch.full((N, G), -7, dtype=torch.int32, device=dev)
        sc = torch.full((N, G, w.r_cap), float("nan"), dtype=torch.float32, device=dev)
        ss = torch.empty((N, G, 512), dtype=torch.float32, device=dev)
        if kind == "workspace":
            ws = s5.Workspace.create(geom, N, w.r_cap, device=dev)
            s5.step5_index_score_topk(geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], t["cos"], t["sin"],
                                      t["summaries"], ids, cnt, ws.tensor, t_cap=w.t_cap, scores=sc, sel_scores=ss)
        else:
            s5.step5_index_score_topk_noalloc(geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], t["cos"],
                                              t["sin"], t["summaries"], ids, cnt, t_cap=w.t_cap, scores=sc,
                                              sel_scores=ss)
        torch.cuda.synchronize()
        out[kind] = (ids.cpu().numpy(), cnt.cpu().numpy(), sc.cpu().numpy(), ss.cpu().numpy())
    assert s5.step5_device_status() == 0
    return out


def test_noalloc_matches_workspace_call_twice(s5):
    geom = s5.STEP5_GEOMETRY
    for positions, B in (([90000, 70001, 5], 3), ([150000], 1)):
        w = S.workload({"positions": positions, "B": B}, seed=41)
        t = S.materialize(w, device="cuda", with_kv=False)
        # summaries of every completed region, built by the library
        s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["sum_begin"], t["sum_end"],
                                  t["summaries"], max_regions_per_seq=w.max_span)
        assert s5.step5_select_path_for(geom, w.N, w.r_cap) == 2   # the path that uses scratch
        r = run_both(s5, w, t)
        ids_a, cnt_a, sc_a, ss_a = r["workspace"]
        ids_b, cnt_b, sc_b, ss_b = r["noalloc"]
        assert np.array_equal(cnt_a, cnt_b)
        assert np.array_equal(ids_a, ids_b)
        for n in range(w.N):
            R = int(w.row_pos[n]) // 8
            assert np.array_equal(sc_a[n, :, :R], sc_b[n, :, :R])
        assert np.array_equal(ss_a, ss_b)


def test_noalloc_rejects_problems_beyond_its_scratch(s5):
    geom = s5.STEP5_GEOMETRY
    N, r_cap = 8, 131073
    assert s5.step5_workspace_bytes(geom, N, r_cap) > 4 << 20
    w = torch.zeros((N, 16), dtype=torch.float32, device="cuda")
    q = torch.zeros((N, 16, 64), dtype=torch.bfloat16, device="cuda")
    seq = torch.zeros(N, dtype=torch.int32, device="cuda")
    summ = torch.zeros((1, 4, r_cap, 64), dtype=torch.uint8, device="cuda")
    ids = torch.empty((N, 4, 512), dtype=torch.int32, device="cuda")
    cnt = torch.full((N, 4), -3, dtype=torch.int32, device="cuda")
    with pytest.raises(s5.Step5Error) as e:
        s5.step5_index_score_topk_noalloc(geom, q, w, seq, seq, None, None, summ, ids, cnt, t_cap=8 * r_cap)
    assert e.value.status == 3
    torch.cuda.synchronize()
    assert (cnt.cpu() == -3).all()   # nothing was enqueued
