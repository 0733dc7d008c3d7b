"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same
seeded inputs.  See tests/parity.py for the comparison rules.

Cases cover several tiles and ragged tails: rows with no candidate region (p < 8), a
complete own region (p = 7 mod 8), just under / at / over 512 regions, several rows per
sequence, both selection paths, the geometry variants the boundary accepts, degenerate
all-equal scores (pure id order, including more tied candidates than the split path's
candidate list holds), injected exact ties, and repeated calls on one workspace.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from parity import (check_out, check_scores, check_selection_chain, check_selection_near_ties,
                    check_summaries, run_path, score_term_bound)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s5():
    import block_sparse_attention_step5_gb300 as s5
    s5.build()
    s5.load()
    torch.cuda.init()
    return s5


def host_inputs(t):
    out = {}
    for k, v in t.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = S.codes16(v)
        else:
            out[k] = v.cpu().numpy()
    return out


def oracle_chain(geom, w, h, summaries=None):
    """Oracle steps 1-4 from scratch on host inputs h."""
    if summaries is None:
        summ = h["summaries"].copy()
        summ, s64, _ = oracle.summarize_batch(h["idx_k"], h["idx_z"], h["cos"], h["sin"], w.sum_begin,
                                              w.sum_end, w.r_cap, geom.rope_dims, summ=summ,
                                              want_f64=True)
    else:
        summ, s64 = summaries, None
    scores, _ = oracle.score_batch(h["idx_q"], h["w"], w.row_seq, w.row_pos, summ,
                                   geom.num_kv_groups, geom.rope_dims, h["cos"], h["sin"])
    ids, cnt, _ = oracle.select_batch(scores, w.row_pos, K=geom.top_k)
    out, _ = oracle.attend_batch(h["q"], h["k_cache"], h["v_cache"], w.row_seq, w.row_pos, ids, cnt,
                                 geom.softmax_scale)
    return dict(summaries=summ, s64=s64, scores=scores, ids=ids, cnt=cnt, out=out)


def full_check(s5, geom, w, t, path=0, chain=True):
    """Every comparison of tests/parity.py on one workload; returns the GPU results."""
    h = host_inputs(t)
    g = run_path(s5, geom, w, t, path=path)
    assert g["status"] == 0, f"device status {g['status']}"
    G = geom.num_kv_groups
    hpg = geom.idx_heads // G
    # (1) summaries over the regions the step summarised
    ref_summ, ref_s64, _ = oracle.summarize_batch(h["idx_k"], h["idx_z"], h["cos"], h["sin"],
                                                  w.sum_begin, w.sum_end, w.r_cap, geom.rope_dims,
                                                  summ=h["summaries"].copy(), want_f64=True)
    for b in range(w.B):
        r0, r1 = int(w.sum_begin[b]), int(w.sum_end[b])
        if r1 <= r0:
            continue
        kreg = h["idx_k"][b, :, 8 * r0:8 * r1].reshape(G, r1 - r0, 8, 64)
        check_summaries(g["summaries"][b, :, r0:r1], g["summ_f32"][b, :, r0:r1],
                        ref_s64[b, :, r0:r1], kreg, geom.rope_dims if h["cos"] is not None else 0,
                        where=f"seq {b}")
    # (2) scores from the GPU's summaries (teacher forced)
    tf_scores, _ = oracle.score_batch(h["idx_q"], h["w"], w.row_seq, w.row_pos, g["summaries"], G,
                                      geom.rope_dims, h["cos"], h["sin"])
    for n in range(w.N):
        R = int(w.row_pos[n]) // 8
        b = int(w.row_seq[n])
        for gg in range(G):
            if R == 0:
                continue
            bound = score_term_bound(h["idx_q"][n, gg * hpg:(gg + 1) * hpg], h["w"][n, gg * hpg:(gg + 1) * hpg],
                                     int(w.row_pos[n]), geom.rope_dims, g["summaries"][b, gg, :R],
                                     h["cos"], h["sin"])
            check_scores(g["scores"][n, gg, :R], tf_scores[n, gg, :R], bound, where=f"row {n} group {gg}")
    # (3) selection from the GPU's scores (teacher forced): exact ids in order
    tf_ids, tf_cnt, _ = oracle.select_batch(g["scores"], w.row_pos, K=geom.top_k)
    assert np.array_equal(tf_cnt, g["sel_count"])
    assert np.array_equal(tf_ids, g["sel_ids"])
    # selection by the oracle fed the GPU's summaries (its own fp64 scores): near-ties only
    gs_ids, gs_cnt, _ = oracle.select_batch(tf_scores, w.row_pos, K=geom.top_k)
    for n in range(w.N):
        for gg in range(G):
            check_selection_near_ties(g["sel_ids"][n, gg], int(g["sel_count"][n, gg]), gs_ids[n, gg],
                                      int(gs_cnt[n, gg]), tf_scores[n, gg], where=f"row {n} group {gg}")
    # picked scores export
    for n in range(w.N):
        for gg in range(G):
            c = int(g["sel_count"][n, gg])
            assert np.array_equal(g["sel_scores"][n, gg, :c], g["scores"][n, gg, g["sel_ids"][n, gg, :c]])
            assert np.all(np.isneginf(g["sel_scores"][n, gg, c:]))
    # (4) attention on the GPU's selection (teacher forced)
    ref_out, _ = oracle.attend_batch(h["q"], h["k_cache"], h["v_cache"], w.row_seq, w.row_pos,
                                     g["sel_ids"], g["sel_count"], geom.softmax_scale)
    check_out(g["out"], ref_out, where="teacher-forced")
    if chain:
        ref = oracle_chain(geom, w, h)
        for n in range(w.N):
            for gg in range(G):
                R = int(w.row_pos[n]) // 8
                assert np.all((g["sel_ids"][n, gg, :g["sel_count"][n, gg]] >= 0) &
                              (g["sel_ids"][n, gg, :g["sel_count"][n, gg]] < R))
                b = int(w.row_seq[n])
                flipped = (g["summaries"][b, gg, :R] != ref["summaries"][b, gg, :R]).any(axis=-1)
                check_selection_chain(g["sel_ids"][n, gg], int(g["sel_count"][n, gg]), ref["ids"][n, gg],
                                      int(ref["cnt"][n, gg]), ref["scores"][n, gg, :R], flipped,
                                      where=f"row {n} group {gg}")
        check_out(g["out"], ref["out"], where="oracle chain")
    return g


SMALL_POS = [0, 1, 7, 8, 9, 15, 16, 17, 129, 4095, 4096, 4097, 4103, 4104, 4600]


@pytest.mark.parametrize("seed", [17, 41])
@pytest.mark.parametrize("path", [1, 2, 3])
def test_small_cases_every_path(s5, seed, path):
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": SMALL_POS, "B": 3}, seed=seed)
    t = S.materialize(w, device="cuda")
    full_check(s5, geom, w, t, path=path)


@pytest.mark.parametrize("cfg", [{"positions": [9000 + 7 * i for i in range(150)], "B": 1},
                                 {"positions": [3000 + 11 * i for i in range(96)] + [700, 12, 0], "B": 3}])
def test_tensor_core_scoring_many_rows(s5, cfg):
    """Path 3 on blocks of rows that share a sequence (a prefill chunk) and on blocks that
    mix three sequences (a pass per sequence), against the oracle: scores within the term
    tolerance, the selection of the GPU's scores exact, near-ties only against the
    oracle's own scores of the GPU's summaries."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload(cfg, seed=53)
    t = S.materialize(w, device="cuda")
    full_check(s5, geom, w, t, path=3, chain=False)


def test_bulk_and_decode_summary_forms_agree_bit_for_bit(s5):
    """Step (1) in one call over hundreds of regions per sequence (the vectorised bulk
    form) and over the same regions a few at a time (the one-dim-per-thread form) write
    the same codes and the same fp32 values, with and without rotation, and match the
    oracle within the summary tolerance."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [2500, 2100], "B": 2}, seed=29)
    t = S.materialize(w, device="cuda", with_kv=False)
    h = host_inputs(t)
    dev = t["idx_k"].device
    R = [int(p) // 8 for p in w.row_pos]
    for rope in (True, False):
        cos, sin = (t["cos"], t["sin"]) if rope else (None, None)
        outs = []
        for step in (max(R), 5):
            summ = torch.zeros_like(t["summaries"])
            f32 = torch.full(t["summaries"].shape, float("nan"), dtype=torch.float32, device=dev)
            for r0 in range(0, max(R), step):
                rb = torch.tensor([min(r0, R[b]) for b in range(w.B)], dtype=torch.int32, device=dev)
                re = torch.tensor([min(r0 + step, R[b]) for b in range(w.B)], dtype=torch.int32, device=dev)
                s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], cos, sin, rb, re, summ, f32,
                                          max_regions_per_seq=step)
            torch.cuda.synchronize()
            assert s5.step5_device_status() == 0
            outs.append((summ.cpu().numpy(), f32.cpu().numpy()))
        assert np.array_equal(outs[0][0], outs[1][0])
        assert np.array_equal(outs[0][1].view(np.uint32), outs[1][1].view(np.uint32))
        _, s64, _ = oracle.summarize_batch(h["idx_k"], h["idx_z"], h["cos"] if rope else None,
                                           h["sin"] if rope else None, np.zeros(w.B, np.int32),
                                           np.array(R, np.int32), w.r_cap, geom.rope_dims if rope else 0,
                                           want_f64=True)
        for b in range(w.B):
            kreg = h["idx_k"][b, :, :8 * R[b]].reshape(4, R[b], 8, 64)
            check_summaries(outs[0][0][b, :, :R[b]], outs[0][1][b, :, :R[b]], s64[b, :, :R[b]], kreg,
                            geom.rope_dims if rope else 0, where=f"bulk seq {b}")


def test_paths_agree(s5):
    """The three scoring paths on the same inputs: the e4m3 products are exact on the CUDA
    cores and on the tensor cores, so the scores agree to fp32 summation order (within
    the score tolerance of each other); the picks agree except where two regions' scores
    are within that tolerance, and each path's picks are exactly the oracle's selection
    of its own scores."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [5000, 9000, 12001, 700, 3], "B": 2}, seed=17)
    t = S.materialize(w, device="cuda")
    res = {path: run_path(s5, geom, w, t, path=path) for path in (1, 2, 3)}
    h = host_inputs(t)
    R = w.row_pos // 8
    hpg = geom.idx_heads // geom.num_kv_groups
    for path, g in res.items():
        assert g["status"] == 0
        ids, cnt, _ = oracle.select_batch(g["scores"], w.row_pos, K=geom.top_k)
        assert np.array_equal(ids, g["sel_ids"]) and np.array_equal(cnt, g["sel_count"]), path
    a = res[1]
    for path in (2, 3):
        b = res[path]
        assert np.array_equal(a["sel_count"], b["sel_count"])
        for n in range(w.N):
            bb = int(w.row_seq[n])
            for gg in range(geom.num_kv_groups):
                if R[n] == 0:
                    continue
                bound = score_term_bound(h["idx_q"][n, gg * hpg:(gg + 1) * hpg], h["w"][n, gg * hpg:(gg + 1) * hpg],
                                         int(w.row_pos[n]), geom.rope_dims, a["summaries"][bb, gg, :R[n]],
                                         h["cos"], h["sin"])
                check_scores(b["scores"][n, gg, :R[n]], a["scores"][n, gg, :R[n]].astype(np.float64), 2 * bound,
                             where=f"path {path} row {n} group {gg}")
                check_selection_near_ties(b["sel_ids"][n, gg], int(b["sel_count"][n, gg]), a["sel_ids"][n, gg],
                                          int(a["sel_count"][n, gg]), a["scores"][n, gg].astype(np.float64),
                                          where=f"path {path} row {n} group {gg}")
        check_out(b["out"], a["out"].astype(np.float64), where=f"path {path} vs 1")


@pytest.mark.parametrize("over", [
    dict(num_q_heads=16), dict(num_q_heads=64), dict(idx_heads=4), dict(idx_heads=8),
    dict(idx_heads=32), dict(rope_dims=0), dict(rope_dims=16), dict(rope_dims=48),
    dict(rope_dims=64), dict(top_k=64), dict(top_k=2048), dict(num_kv_groups=2, idx_heads=16),
    dict(num_kv_groups=8, num_q_heads=64, idx_heads=16),
])
def test_geometry_variants(s5, over):
    base = s5.STEP5_GEOMETRY
    geom = s5.Geometry.step5(**over)
    sg = S.Geometry(num_q_heads=geom.num_q_heads, num_kv_groups=geom.num_kv_groups, head_dim=128,
                    idx_heads=geom.idx_heads, idx_dim=64, rope_dims=geom.rope_dims, region_tokens=8,
                    top_k=geom.top_k, softmax_scale=base.softmax_scale)
    w = S.workload({"positions": [17, 600, 4100, 20000], "B": 2}, seed=41, geom=sg)
    t = S.materialize(w, device="cuda")
    for path in (1, 2, 3):
        full_check(s5, geom, w, t, path=path, chain=(path == 1))


def test_no_rotation_tables(s5):
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [4200, 33], "B": 2}, seed=17)
    t = S.materialize(w, device="cuda")
    t["cos"] = None
    t["sin"] = None
    full_check(s5, geom, w, t, path=0)


@pytest.mark.parametrize("path", [1, 2])
def test_all_equal_scores_pick_ids_in_order(s5, path):
    """w = 0 makes every score +0: the picks are regions 0..K-1 in id order.  The row
    with 24,000 regions puts more tied keys in the threshold bin than the split path's
    candidate list holds, which takes its exact full-scan route."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [4500, 192003, 30], "B": 3}, seed=17)
    t = S.materialize(w, device="cuda", with_kv=True)
    t["w"].zero_()
    g = run_path(s5, geom, w, t, path=path)
    assert g["status"] == 0
    for n in range(w.N):
        R = int(w.row_pos[n]) // 8
        k = min(R, geom.top_k)
        for gg in range(4):
            assert g["sel_count"][n, gg] == k
            assert np.array_equal(g["sel_ids"][n, gg, :k], np.arange(k))
            assert np.all(g["scores"][n, gg, :R] == 0) and not np.signbit(g["scores"][n, gg, :R]).any()


def test_injected_ties_order_by_id(s5):
    """Summaries built by the oracle on the CPU, 10% of each (sequence, group)'s regions
    overwritten with copies of others (exact score ties), uploaded; the step then only
    scores, selects and attends."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [40000, 24000], "B": 2}, seed=41)
    t = S.materialize(w, device="cuda")
    h = host_inputs(t)
    summ, _, _ = oracle.summarize_batch(h["idx_k"], h["idx_z"], h["cos"], h["sin"], w.sum_begin,
                                        w.sum_end, w.r_cap, geom.rope_dims)
    rng = np.random.default_rng(3)
    for b in range(w.B):
        R = int(w.row_pos[b]) // 8
        for gg in range(4):
            src = rng.integers(0, R, R // 10)
            dst = rng.integers(0, R, R // 10)
            summ[b, gg, dst] = summ[b, gg, src]
    t["summaries"].copy_(torch.from_numpy(summ))
    w.sum_end[:] = w.sum_begin
    t["sum_end"].copy_(t["sum_begin"])
    for path in (1, 2):
        full_check(s5, geom, w, t, path=path)


def _cluster_summaries(summ, w, rng, copy=0.55, nudge=0.40):
    """Most regions' summaries replaced by one base row (exact ties) or by the base row
    with one code moved to its neighbouring finite e4m3 code (scores a hair apart), the
    rest left as built: one (row, group)'s scores crowd into a sliver of their range."""
    for b in range(w.B):
        R = int(w.row_pos[w.row_seq == b].max()) // 8
        for gg in range(summ.shape[1]):
            base = summ[b, gg, 0].copy()
            u = rng.random(R)
            for r in range(1, R):
                if u[r] < copy:
                    summ[b, gg, r] = base
                elif u[r] < copy + nudge:
                    row = base.copy()
                    d = int(rng.integers(0, row.shape[0]))
                    c = int(row[d])
                    mag = c & 0x7F
                    row[d] = c + 1 if mag < 0x7E else c - 1  # never the NaN code 0x7F
                    summ[b, gg, r] = row


@pytest.mark.parametrize("case", ["fused_split", "tensor_core"])
def test_clustered_scores_deep_descent(s5, case):
    """Scores crowded into a sliver of their range with thousands of exact ties: the
    block top-k's first digit leaves more than 512 keys in the K-th key's bin, so its
    descent takes further levels (and, at a tie value, picks the smallest ids in order);
    every path's picks must equal the oracle's selection from the same scores."""
    geom = s5.STEP5_GEOMETRY
    if case == "fused_split":
        w = S.workload({"positions": [48001, 40003], "B": 2}, seed=43)
        paths = (1, 2)
    else:  # many rows of one sequence: the tensor-core scoring and the selection from scores
        w = S.workload({"positions": list(range(44000, 44032)), "B": 1}, seed=43)
        paths = (3,)
    t = S.materialize(w, device="cuda")
    h = host_inputs(t)
    summ, _, _ = oracle.summarize_batch(h["idx_k"], h["idx_z"], h["cos"], h["sin"], w.sum_begin,
                                        w.sum_end, w.r_cap, geom.rope_dims)
    _cluster_summaries(summ, w, np.random.default_rng(5))
    t["summaries"].copy_(torch.from_numpy(summ))
    w.sum_end[:] = w.sum_begin
    t["sum_end"].copy_(t["sum_begin"])
    for path in paths:
        g = full_check(s5, geom, w, t, path=path)
        # the crowding worked: many exact ties among each row's scores
        R = int(w.row_pos[0]) // 8
        sc = g["scores"][0, 0, :R]
        assert np.unique(sc).size < R // 4


def test_repeat_calls_reuse_workspace(s5):
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [30000, 4100, 70], "B": 3}, seed=17)
    t = S.materialize(w, device="cuda")
    dev = t["q"].device
    ws = s5.Workspace.create(geom, w.N, w.r_cap, device=dev)
    outs = []
    for path in (2, 2, 1, 2):
        prev = s5.step5_set_select_path(path)
        sel_ids = torch.empty((w.N, 4, 512), dtype=torch.int32, device=dev)
        sel_count = torch.empty((w.N, 4), dtype=torch.int32, device=dev)
        out = torch.empty((w.N, 32, 128), dtype=torch.bfloat16, device=dev)
        s5.decode_step(geom, t, ws, sel_ids, sel_count, out, max_regions_per_seq=w.max_span)
        s5.step5_set_select_path(prev)
        torch.cuda.synchronize()
        outs.append((sel_ids.cpu(), sel_count.cpu(), out.cpu()))
    assert s5.step5_device_status() == 0
    # the workspace is left zero where it must be
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)


def test_dense_equivalence_on_gpu(s5):
    """At most 512 regions: every region is picked and the output is dense causal
    attention over tokens 0..p (torch SDPA in fp64 on the CPU)."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [4095, 2000, 8, 0], "B": 4}, seed=41)
    t = S.materialize(w, device="cuda")
    g = run_path(s5, geom, w, t, path=0)
    h = host_inputs(t)
    for n in range(w.N):
        p, b = int(w.row_pos[n]), int(w.row_seq[n])
        assert np.all(g["sel_count"][n] == p // 8)
        for gg in range(4):
            assert sorted(g["sel_ids"][n, gg, :p // 8].tolist()) == list(range(p // 8))
            q = torch.from_numpy(oracle.bf16_values(h["q"][n, 8 * gg:8 * gg + 8]))
            k = torch.from_numpy(oracle.bf16_values(h["k_cache"][b, gg, :p + 1]))
            v = torch.from_numpy(oracle.bf16_values(h["v_cache"][b, gg, :p + 1]))
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[:, None], k[None].expand(8, -1, -1), v[None].expand(8, -1, -1),
                scale=geom.softmax_scale)[:, 0].numpy()
            check_out(g["out"][n, 8 * gg:8 * gg + 8], ref, where=f"dense row {n}")


def test_cache_rows_past_position_are_ignored(s5):
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [4101, 4099], "B": 2}, seed=17)
    t = S.materialize(w, device="cuda")
    a = run_path(s5, geom, w, t, path=0)
    for b, p in enumerate(w.row_pos):
        t["k_cache"][b, :, p + 1:] = float("nan")
        t["v_cache"][b, :, p + 1:] = float("inf")
    bres = run_path(s5, geom, w, t, path=0)
    assert np.array_equal(a["out"], bres["out"]) and np.array_equal(a["sel_ids"], bres["sel_ids"])


def test_out_of_range_row_sets_status_and_touches_nothing_else(s5):
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [300, 5000], "B": 2}, seed=17)
    t = S.materialize(w, device="cuda")
    good = run_path(s5, geom, w, t, path=0)
    t["row_pos"][0] = w.t_cap + 100     # violates row_pos < t_cap
    bad = run_path(s5, geom, w, t, path=0)
    assert bad["status"] & s5.DEV_RANGE
    assert np.array_equal(good["out"][1], bad["out"][1])
    assert np.array_equal(good["sel_ids"][1], bad["sel_ids"][1])
    assert s5.step5_device_status() == 0


def test_prologue_overlap_gives_identical_results(s5):
    """The opt-in overlap of the scoring prologue with the summary launch changes when
    inputs are read, never what is computed."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [30000, 41000, 4100, 70], "B": 3}, seed=23)
    t = S.materialize(w, device="cuda")
    dev = t["q"].device
    res = []
    for overlap in (0, 1):
        ws = s5.Workspace.create(geom, w.N, w.r_cap, device=dev)
        sel_ids = torch.empty((w.N, 4, 512), dtype=torch.int32, device=dev)
        sel_count = torch.empty((w.N, 4), dtype=torch.int32, device=dev)
        prev_path = s5.step5_set_select_path(2)
        s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["sum_begin"],
                                  t["sum_end"], t["summaries"], max_regions_per_seq=w.max_span)
        prev = s5.step5_set_prologue_overlap(overlap)
        s5.step5_index_score_topk(geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], t["cos"],
                                  t["sin"], t["summaries"], sel_ids, sel_count, ws.tensor,
                                  t_cap=t["idx_k"].shape[2])
        s5.step5_set_prologue_overlap(prev)
        s5.step5_set_select_path(prev_path)
        torch.cuda.synchronize()
        res.append((sel_ids.cpu(), sel_count.cpu()))
    assert s5.step5_device_status() == 0
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
    assert s5.step5_set_prologue_overlap(7) in (0, 1)  # out-of-range values are ignored


@pytest.mark.parametrize("positions,B", [
    ([100] * 150 + [9, 17], 5),   # many short rows: one block's share spans many (row, group)s
    ([20000] * 70 + [20007], 2),  # long shares: more regions per block than it keeps on chip
])
def test_split_path_share_shapes(s5, positions, B):
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": positions, "B": B}, seed=29)
    t = S.materialize(w, device="cuda")
    a = run_path(s5, geom, w, t, path=1)
    b = run_path(s5, geom, w, t, path=2)
    assert a["status"] == 0 and b["status"] == 0
    for k in ("sel_ids", "sel_count", "sel_scores", "out"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("cfg", [{"positions": [30000, 41000, 4100, 70], "B": 3}, 4])
def test_decode_step_entry_matches_the_three_calls(s5, cfg):
    """step5_decode_step (one call: the scoring kernel fetches the summary tiles clear of
    the regions being summarised before waiting for the summary kernel) gives the same
    selection and output as the three calls."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload(cfg, seed=31)
    dev = torch.device("cuda")
    res = []
    for fused_entry in (False, True):
        t = S.materialize(w, device=dev)
        pre = int((w.pre_end - w.pre_begin).max())
        if pre > 0:
            s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["pre_begin"],
                                      t["pre_end"], t["summaries"], max_regions_per_seq=pre)
        ws = s5.Workspace.create(geom, w.N, w.r_cap, device=dev)
        sel_ids = torch.empty((w.N, 4, 512), dtype=torch.int32, device=dev)
        sel_count = torch.empty((w.N, 4), dtype=torch.int32, device=dev)
        out = torch.empty((w.N, 32, 128), dtype=torch.bfloat16, device=dev)
        for _ in range(2):  # twice: the second call reuses the workspace
            if fused_entry:
                s5.step5_decode_step(geom, t, ws, sel_ids, sel_count, out, max_regions_per_seq=w.max_span)
            else:
                s5.decode_step(geom, t, ws, sel_ids, sel_count, out, max_regions_per_seq=w.max_span)
        torch.cuda.synchronize()
        assert s5.step5_device_status() == 0
        res.append((sel_ids.cpu(), sel_count.cpu(), out.cpu(), S.codes8(t["summaries"])))
        del t
    for a, b in zip(res[0][:3], res[1][:3]):
        assert torch.equal(a, b)
    assert np.array_equal(res[0][3], res[1][3])


@pytest.mark.parametrize("cfg", [{"positions": [30000, 41000, 4100, 70], "B": 3}, {"positions": [1016], "B": 1}])
def test_attention_split_over_blocks_and_single_block(s5, cfg):
    """With a workspace, few (row, group) pairs split their key list over several blocks
    that merge through it; without one, one block takes each pair.  Both agree with the
    oracle on the same selection, and the split result repeats bit for bit."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload(cfg, seed=37)
    t = S.materialize(w, device="cuda")
    g = run_path(s5, geom, w, t, path=0)
    assert g["status"] == 0
    h = host_inputs(t)
    ref_out, _ = oracle.attend_batch(h["q"], h["k_cache"], h["v_cache"], w.row_seq, w.row_pos,
                                     g["sel_ids"], g["sel_count"], geom.softmax_scale)
    dev = t["q"].device
    sel_ids = torch.from_numpy(g["sel_ids"]).to(dev)
    sel_count = torch.from_numpy(g["sel_count"]).to(dev)
    ws = s5.Workspace.create(geom, w.N, w.r_cap, device=dev)
    outs = []
    for workspace in (ws.tensor, None, ws.tensor):
        out = torch.full((w.N, geom.num_q_heads, geom.head_dim), float("nan"), dtype=torch.bfloat16, device=dev)
        s5.step5_sparse_attn(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"],
                             sel_ids, sel_count, out, workspace)
        torch.cuda.synchronize()
        outs.append(out.float().cpu().numpy())
    assert s5.step5_device_status() == 0
    for i, o in enumerate(outs):
        check_out(o, ref_out, where="one block" if i == 1 else "split")
    assert np.array_equal(outs[0], outs[2])


def test_attention_rejects_a_workspace_too_small(s5):
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [4100], "B": 1}, seed=37)
    t = S.materialize(w, device="cuda")
    dev = t["q"].device
    sel_ids = torch.full((1, 4, 512), -1, dtype=torch.int32, device=dev)
    sel_count = torch.zeros((1, 4), dtype=torch.int32, device=dev)
    out = torch.zeros((1, geom.num_q_heads, geom.head_dim), dtype=torch.bfloat16, device=dev)
    tiny = torch.zeros(256, dtype=torch.uint8, device=dev)
    with pytest.raises(s5.Step5Error) as e:
        s5.step5_sparse_attn(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"],
                             sel_ids, sel_count, out, tiny)
    assert e.value.status == 3
    torch.cuda.synchronize()
    assert (out.cpu() == 0).all()   # nothing was enqueued


def test_picks_clustered_in_one_share(s5):
    """The K best regions are the last 600 of a long row (equal scores; every other score
    is zero): one or two blocks of the split launch hold all the picks, and every score
    outside them ties at zero; twice on one workspace."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [320000], "B": 1}, seed=53)
    t = S.materialize(w, device="cuda")
    R = int(w.row_pos[0]) // 8
    summ = torch.zeros_like(t["summaries"])
    summ[0, :, R - 600:R, :] = 0x38  # e4m3 +1.0
    t["summaries"].copy_(summ)
    t["idx_q"].abs_()  # no rotation below: every head's dot product with +1.0 is positive
    t["w"].abs_()
    K = geom.top_k
    ws = s5.Workspace.create(geom, w.N, w.r_cap)
    ids = torch.empty((1, 4, K), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, 4), dtype=torch.int32, device="cuda")
    for _ in range(2):
        ids.fill_(-7)
        s5.step5_index_score_topk(geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], None, None,
                                  t["summaries"], ids, cnt, ws.tensor, t_cap=w.t_cap)
        torch.cuda.synchronize()
        assert s5.step5_device_status() == 0
        assert (cnt.cpu() == K).all()
        want = torch.arange(R - 600, R - 600 + K, dtype=torch.int32)
        for g in range(4):
            assert torch.equal(ids[0, g].cpu(), want)


@pytest.mark.parametrize("cfg", [{"positions": [30000, 4100, 70, 15], "B": 2},
                                 {"positions": [9000] * 40, "B": 5}])
def test_gated_attention_matches_the_oracle(s5, cfg):
    """step5_sparse_attn_gated: the per-head sigmoid output gate on the attention output,
    against the oracle (attention, then the gate, one rounding), with the split over
    blocks (workspace) and with one block per (row, group); a zero logit halves the
    ungated output bit for bit."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload(cfg, seed=59)
    t = S.materialize(w, device="cuda")
    g = run_path(s5, geom, w, t, path=0)
    assert g["status"] == 0
    dev = t["q"].device
    sel_ids = torch.from_numpy(g["sel_ids"]).to(dev)
    sel_count = torch.from_numpy(g["sel_count"]).to(dev)
    gen = torch.Generator().manual_seed(61)
    gate = (torch.randn((w.N, geom.num_q_heads), generator=gen) * 3).to(torch.bfloat16).to(dev)
    h = host_inputs(t)
    ref, _ = oracle.attend_batch(h["q"], h["k_cache"], h["v_cache"], w.row_seq, w.row_pos,
                                 g["sel_ids"], g["sel_count"], geom.softmax_scale)
    ref_gated = oracle.sigmoid_gate(ref, S.codes16(gate))
    ws = s5.Workspace.create(geom, w.N, w.r_cap, device=dev)
    for workspace in (ws.tensor, None):
        out = torch.full((w.N, geom.num_q_heads, geom.head_dim), float("nan"), dtype=torch.bfloat16, device=dev)
        s5.step5_sparse_attn_gated(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"],
                                   sel_ids, sel_count, gate, out, workspace)
        plain = torch.empty_like(out)
        s5.step5_sparse_attn(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"],
                             sel_ids, sel_count, plain, workspace)
        half = torch.empty_like(out)
        s5.step5_sparse_attn_gated(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"],
                                   sel_ids, sel_count, torch.zeros_like(gate), half, workspace)
        torch.cuda.synchronize()
        assert s5.step5_device_status() == 0
        check_out(out.float().cpu().numpy(), ref_gated, where="gated")
        assert torch.equal(half.float() * 2, plain.float())


def _bf16_ulps(a_codes, b_codes):
    """|a - b| in bf16 units of the last place (codes of finite values)."""
    a = a_codes.astype(np.int32)
    b = b_codes.astype(np.int32)
    a = np.where(a & 0x8000, 0x8000 - a, a)  # sign-magnitude to a monotone integer line
    b = np.where(b & 0x8000, 0x8000 - b, b)
    return np.abs(a - b)


@pytest.mark.parametrize("rope", [True, False])
def test_indexer_front_end(s5, rope):
    """step5_indexer_front against the oracle: normalised q and k within one bf16 step
    (fp32 against fp64 sums) and equal almost everywhere, z and every untouched cache
    row bit for bit, and the summaries of the regions that rows complete equal to the
    oracle's summary step over the caches the GPU wrote (e4m3 midpoint rule) and bit for
    bit to step5_region_summarize over the same caches."""
    geom = s5.STEP5_GEOMETRY
    G, H, D, B, t_cap, r_cap = 4, geom.idx_heads, 64, 3, 256, 32
    gen = torch.Generator().manual_seed(67)
    dev = torch.device("cuda")
    bf = lambda *shape, scale=1.0, shift=0.0: (torch.randn(shape, generator=gen) * scale + shift).to(torch.bfloat16)
    q_pre, k_pre, z_pre = bf(3, H, D, scale=2.0), bf(3, G, D, scale=1.5, shift=0.3), bf(3, G, D)
    qw, kw, kb = bf(D, scale=0.1), bf(D, scale=0.1, shift=1.0), bf(D, scale=0.1)
    k_cache, z_cache = bf(B, G, t_cap, D), bf(B, G, t_cap, D)
    summ = torch.zeros((B, G, r_cap, D), dtype=torch.uint8)
    ang = np.outer(np.arange(t_cap), 10000.0 ** (-np.arange(16) * 2 / 32))
    cos = torch.from_numpy(np.cos(ang)).to(torch.bfloat16) if rope else None
    sin = torch.from_numpy(np.sin(ang)).to(torch.bfloat16) if rope else None
    seqs = torch.tensor([2, 0, 1], dtype=torch.int32)
    pos = torch.tensor([15, 100, 255], dtype=torch.int32)  # rows 0 and 2 complete regions 1 and 31
    eps = 1e-6
    ref_q, ref_k, ref_z, ref_s = oracle.indexer_front(S.codes16(q_pre), S.codes16(k_pre), S.codes16(z_pre),
                                                      S.codes16(qw), S.codes16(kw), S.codes16(kb), seqs.numpy(),
                                                      pos.numpy(), None if cos is None else S.codes16(cos),
                                                      None if sin is None else S.codes16(sin), S.codes16(k_cache),
                                                      S.codes16(z_cache), summ.numpy(), eps=eps, rope_dims=32)
    d = {k: v.to(dev) for k, v in dict(q_pre=q_pre, k_pre=k_pre, z_pre=z_pre, qw=qw, kw=kw, kb=kb, kc=k_cache,
                                       zc=z_cache, summ=summ, seqs=seqs, pos=pos).items()}
    dcos = cos.to(dev) if rope else None
    dsin = sin.to(dev) if rope else None
    q_out = torch.empty_like(d["q_pre"])
    s5.step5_indexer_front(geom, d["q_pre"], d["k_pre"], d["z_pre"], d["qw"], d["kw"], d["kb"], eps, d["seqs"],
                           d["pos"], dcos, dsin, q_out, d["kc"], d["zc"], d["summ"])
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    gq, gk, gz, gs = S.codes16(q_out), S.codes16(d["kc"]), S.codes16(d["zc"]), d["summ"].cpu().numpy()
    for got, ref in ((gq, ref_q), (gk, ref_k)):
        ulps = _bf16_ulps(got, ref)
        assert ulps.max() <= 1 and (ulps > 0).mean() < 0.01
    assert np.array_equal(gz, ref_z)
    # the completed regions' summaries against the oracle's summary step run on the
    # caches the GPU wrote (teacher-forced): values through the e4m3 midpoint rule
    rb_h = np.array([0, 31, 1], dtype=np.int32)
    re_h = np.array([0, 32, 2], dtype=np.int32)
    _, s64, _ = oracle.summarize_batch(gk, gz, None if cos is None else S.codes16(cos),
                                       None if sin is None else S.codes16(sin), rb_h, re_h, r_cap,
                                       32 if rope else 0, want_f64=True)
    for b, r in ((1, 31), (2, 1)):
        k_reg = gk[b, :, 8 * r:8 * r + 8, :]
        check_summaries(gs[b, :, r], None, s64[b, :, r], k_reg, 32 if rope else 0, where=f"front seq {b}")
    # both front ends write the completed regions only
    untouched = np.ones(gs.shape[:3], bool)
    untouched[1, :, 31] = untouched[2, :, 1] = False
    assert not gs[untouched].any() and not ref_s[untouched].any()
    # and the summary kernel over the same (GPU) caches writes them bit for bit
    chk = torch.zeros_like(d["summ"])
    rb = torch.tensor([0, 0, 0], dtype=torch.int32, device=dev)
    re = torch.tensor([0, 0, 0], dtype=torch.int32, device=dev)
    rb[2], re[2], rb[1], re[1] = 1, 2, 31, 32
    s5.step5_region_summarize(geom, d["kc"], d["zc"], dcos, dsin, rb, re, chk, max_regions_per_seq=1)
    torch.cuda.synchronize()
    assert np.array_equal(gs, chk.cpu().numpy())
    assert gs[2, :, 1].any() and gs[1, :, 31].any() and not gs[0].any()
