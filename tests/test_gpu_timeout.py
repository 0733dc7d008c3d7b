"""A bounded device wait that gives up: the split selection path's wait on the
threshold word of a (row, group), made to run out on purpose.

The workspace is filled with 0xff bytes before the call, so every per-(row, group)
arrival counter starts at 2^32 - 1: the arrivals of the blocks then count
2^32 - 1, 0, 1, ..., and none of them sees itself as the last of its (row, group), so
no threshold is ever published (a flag that nothing sets).  Every block then polls the
threshold word until the poll limit (set small here) runs out, raises
STEP5_DEV_TIMEOUT and returns; no copy is in flight at that point and nothing faults.
After re-zeroing the workspace the same call gives the oracle's selection again.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s5():
    import block_sparse_attention_step5_gb300 as s5
    s5.build()
    s5.load()
    return s5


def test_threshold_wait_gives_up_and_the_next_call_recovers(s5):
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [40000, 30001], "B": 2}, seed=23)
    t = S.materialize(w, device="cuda")
    N, G = w.N, geom.num_kv_groups
    s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["sum_begin"], t["sum_end"],
                              t["summaries"], max_regions_per_seq=w.max_span)
    ws = s5.Workspace.create(geom, N, w.r_cap)
    sel_ids = torch.full((N, G, geom.top_k), -7, dtype=torch.int32, device="cuda")
    sel_count = torch.full((N, G), -7, dtype=torch.int32, device="cuda")
    scores = torch.zeros((N, G, w.r_cap), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0

    def call():
        s5.step5_index_score_topk(geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], t["cos"], t["sin"],
                                  t["summaries"], sel_ids, sel_count, ws.tensor, t_cap=w.t_cap, scores=scores)

    prev_path = s5.step5_set_select_path(2)
    prev_polls = s5.step5_set_wait_polls(256)
    try:
        ws.tensor.fill_(0xff)
        call()
        torch.cuda.synchronize()
        flags = s5.step5_device_status()
        assert flags & s5.DEV_TIMEOUT, f"expected the timeout bit, got flags {flags}"
        # no selection was written: the outputs keep their fill
        assert (sel_count == -7).all()
    finally:
        s5.step5_set_wait_polls(0)
        assert s5.step5_set_wait_polls(0) == prev_polls
        s5.step5_set_select_path(prev_path)

    # after re-zeroing, the default limit and the split path give the oracle's selection
    s5.step5_workspace_init(ws.tensor)
    s5.step5_set_select_path(2)
    try:
        call()
    finally:
        s5.step5_set_select_path(prev_path)
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    ids_o, cnt_o, _ = oracle.select_batch(scores.cpu().numpy(), w.row_pos, K=geom.top_k)
    assert np.array_equal(cnt_o, sel_count.cpu().numpy())
    assert np.array_equal(ids_o, sel_ids.cpu().numpy())
