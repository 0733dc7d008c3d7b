"""GPU: the whole step from host inputs to host output (step5_decode_step_host) gives
the same selection and output, bit for bit, as step5_decode_step on the same inputs in
device memory, eagerly and replayed from a CUDA graph, with the page-locked host buffers
read and written in place by the kernels and through copies."""
import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s5():
    import block_sparse_attention_step5_gb300 as s5
    s5.build()
    s5.load()
    torch.cuda.init()
    return s5


@pytest.mark.parametrize("copies", [0, 1])
@pytest.mark.parametrize("cfg", [0, {"positions": [30000, 4100, 70, 15], "B": 2}, 1])
def test_host_step_equals_device_step(s5, cfg, copies):
    geom = s5.STEP5_GEOMETRY
    w = S.workload(cfg, seed=89)
    t = S.materialize(w, device="cuda")
    dev = t["q"].device
    N, G, K = w.N, geom.num_kv_groups, geom.top_k
    pre = int((w.pre_end - w.pre_begin).max())
    if pre > 0:
        s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["pre_begin"], t["pre_end"],
                                  t["summaries"], max_regions_per_seq=pre)
    summ0 = t["summaries"].clone()
    ws = s5.Workspace.create(geom, N, w.r_cap, device=dev)
    ids_d = torch.empty((N, G, K), dtype=torch.int32, device=dev)
    cnt_d = torch.empty((N, G), dtype=torch.int32, device=dev)
    out_d = torch.empty((N, geom.num_q_heads, geom.head_dim), dtype=torch.bfloat16, device=dev)
    s5.step5_decode_step(geom, t, ws, ids_d, cnt_d, out_d, max_regions_per_seq=w.max_span)
    torch.cuda.synchronize()
    summ_d = t["summaries"].clone()
    t["summaries"].copy_(summ0)

    rows = s5.HostRows(geom, N, w.B, device=dev)
    for src, name in (("q", "q"), ("idx_q", "idx_q"), ("w", "w"), ("row_seq", "row_seq"), ("row_pos", "row_pos"),
                      ("sum_begin", "region_begin"), ("sum_end", "region_end")):
        rows.view(name).copy_(t[src].cpu())
    assert rows.h2d_bytes == rows.layout.total and rows.d2h_bytes == out_d.numel() * 2
    ws2 = s5.Workspace.create(geom, N, w.r_cap, device=dev)
    ids_h = torch.full_like(ids_d, -7)
    cnt_h = torch.full_like(cnt_d, -7)

    def call():
        prev = s5.step5_set_host_copies(copies)
        try:
            s5.step5_decode_step_host(geom, t, ws2, rows, ids_h, cnt_h, max_regions_per_seq=w.max_span)
        finally:
            s5.step5_set_host_copies(prev)

    call()
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    assert torch.equal(ids_h, ids_d) and torch.equal(cnt_h, cnt_d)
    assert torch.equal(t["summaries"], summ_d)
    assert torch.equal(rows.out_host.view(torch.int16), out_d.cpu().view(torch.int16))
    # in place: the device staging buffers were not used (page-locked memory is
    # device-addressable here); through copies: they hold the inputs and the output
    assert bool(rows.dev.any()) == bool(copies)
    assert bool(rows.out_dev.view(torch.int16).any()) == bool(copies)
    # replayed from a graph, from fresh host values
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        call()
    rows.out_host.fill_(float("nan"))
    t["summaries"].copy_(summ0)
    g.replay()
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    assert torch.equal(rows.out_host.view(torch.int16), out_d.cpu().view(torch.int16))
    # a changed host input reaches the device: all rows moved to sequence 0 at a lower
    # position give a different output
    rows.view("row_pos").fill_(9)
    rows.view("row_seq").fill_(0)
    rows.view("region_begin").fill_(0)
    rows.view("region_end").fill_(1)
    g.replay()
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    assert (cnt_h.cpu() == 1).all()
    assert not torch.equal(rows.out_host.view(torch.int16), out_d.cpu().view(torch.int16))


def test_host_step_with_pageable_buffers(s5):
    """Pageable host buffers give the same results: where the device can address them
    (on Grace, through the CPU's page tables) the kernels use them in place, elsewhere
    the call copies them through the device staging buffers."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [4100, 70], "B": 2}, seed=97)
    t = S.materialize(w, device="cuda")
    dev = t["q"].device
    N, G, K = w.N, geom.num_kv_groups, geom.top_k
    summ0 = t["summaries"].clone()
    ws = s5.Workspace.create(geom, N, w.r_cap, device=dev)
    ids_d = torch.empty((N, G, K), dtype=torch.int32, device=dev)
    cnt_d = torch.empty((N, G), dtype=torch.int32, device=dev)
    out_d = torch.empty((N, geom.num_q_heads, geom.head_dim), dtype=torch.bfloat16, device=dev)
    s5.step5_decode_step(geom, t, ws, ids_d, cnt_d, out_d, max_regions_per_seq=w.max_span)
    torch.cuda.synchronize()
    t["summaries"].copy_(summ0)
    rows = s5.HostRows(geom, N, w.B, device=dev)
    rows.host = torch.zeros(rows.host.shape, dtype=rows.host.dtype)  # pageable
    rows.out_host = torch.zeros(rows.out_host.shape, dtype=rows.out_host.dtype)
    assert not rows.host.is_pinned() and not rows.out_host.is_pinned()
    for src, name in (("q", "q"), ("idx_q", "idx_q"), ("w", "w"), ("row_seq", "row_seq"), ("row_pos", "row_pos"),
                      ("sum_begin", "region_begin"), ("sum_end", "region_end")):
        rows.view(name).copy_(t[src].cpu())
    ws2 = s5.Workspace.create(geom, N, w.r_cap, device=dev)
    ids_h = torch.full_like(ids_d, -7)
    cnt_h = torch.full_like(cnt_d, -7)
    s5.step5_decode_step_host(geom, t, ws2, rows, ids_h, cnt_h, max_regions_per_seq=w.max_span)
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    assert torch.equal(ids_h, ids_d) and torch.equal(cnt_h, cnt_d)
    assert torch.equal(rows.out_host.view(torch.int16), out_d.cpu().view(torch.int16))
