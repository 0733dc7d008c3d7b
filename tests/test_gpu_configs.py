"""The five workloads at full size, in the launch configuration the benchmark times
(automatic selection path), against the oracle.

Small workloads (1 row at 4,608; 16 rows at 16K-32K) are checked on every row.  The
large ones are checked on sampled rows (prefill: 48 of 2,048 rows) with every score of a
checked row, and on every summarised region.  Cache rows the oracle needs are drawn on
the device (only those rows), so the 1M-token caches are never copied back whole; the
generator's CPU/GPU identity is checked in test_gpu_codecs.py.
"""
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
    return s5


def lazy_rows(tensor, flat_rows):
    """Host uint16 array of the tensor's full shape (lazily zero) holding only the given
    rows of its flattened leading dims, gathered on the device and copied back."""
    shape = tuple(tensor.shape)
    out = np.zeros(shape, dtype=np.uint16)
    rows = np.unique(np.asarray(flat_rows, dtype=np.int64))
    if rows.size:
        flat = tensor.view(-1, shape[-1])
        got = flat.index_select(0, torch.from_numpy(rows).to(tensor.device))
        out.reshape(-1, shape[-1])[rows] = S.codes16(got)
    return out


def token_rows(w, rows, sel_ids, sel_count, G):
    """Flat [B*G*t_cap] row indices of every key token the rows attend to; sel_ids and
    sel_count are indexed like ``rows`` (entry i belongs to row rows[i])."""
    out = []
    for i, n in enumerate(rows):
        b, p = int(w.row_seq[n]), int(w.row_pos[n])
        own = p // 8
        for g in range(G):
            base = (b * G + g) * w.t_cap
            regs = list(sel_ids[i, g, :sel_count[i, g]]) + [own]
            toks = (np.asarray(regs, dtype=np.int64)[:, None] * 8 + np.arange(8)[None, :]).ravel()
            out.append(base + toks)
    return np.concatenate(out)


def check_workload(s5, cfg, rows=None, seed=17):
    geom = s5.STEP5_GEOMETRY
    G = geom.num_kv_groups
    hpg = geom.idx_heads // G
    w = S.workload(cfg, seed=seed)
    t = S.materialize(w, device="cuda")
    pre = None
    if int((w.pre_end - w.pre_begin).max()) > 0:
        # prefix regions built once at set-up, by the kernel (they are inputs of the step)
        s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["pre_begin"],
                                  t["pre_end"], t["summaries"],
                                  max_regions_per_seq=int((w.pre_end - w.pre_begin).max()))
    summ_before = S.codes8(t["summaries"])
    g = run_path(s5, geom, w, t, path=0)
    assert g["status"] == 0
    rows = np.arange(w.N) if rows is None else np.asarray(rows)

    # host inputs: small tensors copied, caches drawn lazily for the rows they serve
    h = {k: S.codes16(t[k]) for k in ("q", "idx_q", "cos", "sin")}
    h["w"] = t["w"].cpu().numpy()
    # (1) summaries of the regions the step built
    for b in range(w.B):
        r0, r1 = int(w.sum_begin[b]), int(w.sum_end[b])
        if r1 <= r0:
            continue
        flat = ((b * G + np.arange(G))[:, None] * w.t_cap + np.arange(8 * r0, 8 * r1)[None, :]).ravel()
        ik = lazy_rows(t["idx_k"], flat)
        iz = lazy_rows(t["idx_z"], flat)
        rb = np.zeros(w.B, np.int32)
        re = np.zeros(w.B, np.int32)
        rb[b], re[b] = r0, r1
        _, s64, _ = oracle.summarize_batch(ik, iz, h["cos"], h["sin"], rb, re, w.r_cap, geom.rope_dims,
                                           summ=summ_before.copy(), want_f64=True)
        kreg = ik[b, :, 8 * r0:8 * r1].reshape(G, r1 - r0, 8, 64)
        check_summaries(g["summaries"][b, :, r0:r1], g["summ_f32"][b, :, r0:r1], s64[b, :, r0:r1], kreg,
                        geom.rope_dims, where=f"{w.name} seq {b}")
    # (2)-(3) scores and picks of the sampled rows, teacher forced
    sub_pos = w.row_pos[rows]
    sub_seq = w.row_seq[rows]
    tf_scores, _ = oracle.score_batch(h["idx_q"][rows], h["w"][rows], sub_seq, sub_pos, g["summaries"], G,
                                      geom.rope_dims, h["cos"], h["sin"])
    for i, n in enumerate(rows):
        R = int(w.row_pos[n]) // 8
        b = int(w.row_seq[n])
        for gg in range(G):
            bound = score_term_bound(h["idx_q"][n, gg * hpg:(gg + 1) * hpg], h["w"][n, gg * hpg:(gg + 1) * hpg],
                                     int(w.row_pos[n]), geom.rope_dims, g["summaries"][b, gg, :R],
                                     h["cos"], h["sin"])
            check_scores(g["scores"][n, gg, :R], tf_scores[i, gg, :R], bound, where=f"{w.name} row {n} g {gg}")
    tf_ids, tf_cnt, _ = oracle.select_batch(g["scores"][rows], sub_pos, K=geom.top_k)
    assert np.array_equal(tf_ids, g["sel_ids"][rows]) and np.array_equal(tf_cnt, g["sel_count"][rows])
    # the oracle fed the GPU's summaries, selecting on its own fp64 scores: near-ties only
    gs_ids, gs_cnt, _ = oracle.select_batch(tf_scores, sub_pos, K=geom.top_k)
    for i, n in enumerate(rows):
        for gg in range(G):
            check_selection_near_ties(g["sel_ids"][n, gg], int(g["sel_count"][n, gg]), gs_ids[i, gg],
                                      int(gs_cnt[i, gg]), tf_scores[i, gg], where=f"{w.name} row {n} g {gg}")
    # (4) attention of the sampled rows on the GPU's picks
    need = token_rows(w, rows, g["sel_ids"][rows], g["sel_count"][rows], G)
    kc = lazy_rows(t["k_cache"], need)
    vc = lazy_rows(t["v_cache"], need)
    ref_out, _ = oracle.attend_batch(h["q"][rows], kc, vc, sub_seq, sub_pos, g["sel_ids"][rows],
                                     g["sel_count"][rows], geom.softmax_scale)
    err_tf = check_out(g["out"][rows], ref_out, where=f"{w.name} teacher-forced")
    # the oracle's own chain: its summaries (initial summaries + its step-1 regions)
    ref_summ = summ_before.copy()
    if w.random_summaries:
        ref_summ = S.random_summaries(w).numpy()
    for b in range(w.B):
        for (r0, r1) in ((int(w.pre_begin[b]), int(w.pre_end[b])), (int(w.sum_begin[b]), int(w.sum_end[b]))):
            if r1 <= r0:
                continue
            flat = ((b * G + np.arange(G))[:, None] * w.t_cap + np.arange(8 * r0, 8 * r1)[None, :]).ravel()
            ik = lazy_rows(t["idx_k"], flat)
            iz = lazy_rows(t["idx_z"], flat)
            rb = np.zeros(w.B, np.int32)
            re = np.zeros(w.B, np.int32)
            rb[b], re[b] = r0, r1
            oracle.summarize_batch(ik, iz, h["cos"], h["sin"], rb, re, w.r_cap, geom.rope_dims, summ=ref_summ)
    ch_scores, _ = oracle.score_batch(h["idx_q"][rows], h["w"][rows], sub_seq, sub_pos, ref_summ, G,
                                      geom.rope_dims, h["cos"], h["sin"])
    ch_ids, ch_cnt, _ = oracle.select_batch(ch_scores, sub_pos, K=geom.top_k)
    swaps = 0
    for i, n in enumerate(rows):
        R = int(w.row_pos[n]) // 8
        b = int(w.row_seq[n])
        for gg in range(G):
            flipped = (g["summaries"][b, gg, :R] != ref_summ[b, gg, :R]).any(axis=-1)
            swaps += check_selection_chain(g["sel_ids"][n, gg], int(g["sel_count"][n, gg]), ch_ids[i, gg],
                                           int(ch_cnt[i, gg]), ch_scores[i, gg, :R], flipped,
                                           where=f"{w.name} row {n} g {gg}")
    need2 = token_rows(w, rows, ch_ids, ch_cnt, G)
    kc2 = lazy_rows(t["k_cache"], need2)
    vc2 = lazy_rows(t["v_cache"], need2)
    ch_out, _ = oracle.attend_batch(h["q"][rows], kc2, vc2, sub_seq, sub_pos, ch_ids, ch_cnt, geom.softmax_scale)
    err_ch = check_out(g["out"][rows], ch_out, where=f"{w.name} oracle chain")
    return dict(err_tf=err_tf, err_chain=err_ch, swaps=swaps)


def test_config0_decode_4608(s5):
    check_workload(s5, 0)


def test_config1_decode_16_ragged(s5):
    check_workload(s5, 1)


def test_config2_decode_4x128k_ties(s5):
    check_workload(s5, 2)


def test_config3_prefill_2048_on_64k_sampled(s5):
    rows = np.unique(np.concatenate([np.arange(0, 2048, 47), [0, 1, 7, 8, 2047]]))
    check_workload(s5, 3, rows=rows)


def test_config4_decode_1m(s5):
    check_workload(s5, 4)
