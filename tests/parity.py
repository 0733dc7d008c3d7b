"""Comparison rules between the CUDA path and the CPU oracle (shared by the GPU tests,
the smoke check and the benchmark's sanity check).

Tolerances (the method's stated parity bar):
  * summaries: fp32 values within 1e-5 relative to the size of their terms
    (|s_gpu - s_ref| <= 1e-5 * max_t |rot(k)_t[d]|, which bounds sum_t w_t |rot(k)_t[d]|);
    e4m3 codes equal, except where the reference lies within that tolerance of a
    rounding boundary of e4m3(bf16(.)) (an e4m3 "midpoint" case);
  * scores: within 1e-5 relative to their terms
    (|x_gpu - x_ref| <= 1e-5 * sum_h w_h sum_d |qe_hd * s_d| + 1e-30);
  * selection fed the GPU's own scores: ids and their order exactly equal;
  * selection by the oracle fed the GPU's summaries (its own fp64 scores): equal except
    at near-ties, where swapped regions' reference scores differ by < 1e-6 relative;
  * selection from the oracle's fully independent chain: as above, except that a
    region whose summary code flipped at an allowed e4m3 midpoint has a different
    score by construction, so such regions may move; every other difference must be a
    near-tie;
  * attention output (bf16): within 2e-2 absolute.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synthetic as S

SUMMARY_RTOL = 1e-5
SCORE_RTOL = 1e-5
NEAR_TIE = 1e-6
OUT_ATOL = 2e-2


def e4m3_of(values: np.ndarray) -> np.ndarray:
    """e4m3(bf16(v)) codes with the oracle's (pinned) codecs."""
    return oracle.bf16_codes_to_e4m3_codes(oracle.bf16_round_array(values))


def summary_bound(k_codes: np.ndarray, rope_dims: int) -> np.ndarray:
    """Per-dim bound on |rot(k)| over a region's tokens: k [..., 8, 64] -> [..., 64]."""
    kv = np.abs(oracle.bf16_values(k_codes))
    half = rope_dims // 2
    b = kv.copy()
    if half:
        pair = kv[..., :half] + kv[..., half:rope_dims]
        b[..., :half] = pair
        b[..., half:rope_dims] = pair
    return b.max(axis=-2)


def check_summaries(gpu_codes, gpu_f32, ref_f64, k_region_codes, rope_dims, where=""):
    """gpu_codes/ref arrays [..., 64] over the summarised regions; k_region_codes
    [..., 8, 64].  Returns (number of midpoint exemptions, number of values)."""
    bound = summary_bound(k_region_codes, rope_dims)
    tol = SUMMARY_RTOL * bound + 1e-30
    if gpu_f32 is not None:
        err = np.abs(gpu_f32.astype(np.float64) - ref_f64)
        bad = err > tol
        assert not bad.any(), f"{where} summary values off: max err/tol {np.max(err / tol):.3g}"
    ref_codes = e4m3_of(ref_f64)
    diff = gpu_codes != ref_codes
    if diff.any():
        lo = e4m3_of(ref_f64 - tol)
        hi = e4m3_of(ref_f64 + tol)
        near_boundary = (lo != hi) | (lo != ref_codes) | (hi != ref_codes)
        unexplained = diff & ~near_boundary
        assert not unexplained.any(), f"{where} {unexplained.sum()} summary codes differ away from a midpoint"
    return int(diff.sum()), int(diff.size)


def score_term_bound(q_codes_group, w_group, pos, rope_dims, summ_codes, cos, sin):
    """sum_h w_h sum_d |qe_hd s_d| for every region: q [hpg][64], summ [R][64]."""
    half = rope_dims // 2
    qe = []
    for h in range(q_codes_group.shape[0]):
        if cos is not None:
            rot = oracle.rotate_neox(q_codes_group[h], rope_dims, cos[pos], sin[pos])
        else:
            rot = oracle.bf16_values(q_codes_group[h])
        qe.append(oracle.e4m3_values(e4m3_of(rot)))
    qe = np.abs(np.stack(qe))                       # [hpg][64]
    sv = np.abs(oracle.e4m3_values(summ_codes))     # [R][64]
    return (sv @ qe.T) @ np.abs(w_group.astype(np.float64))


def check_scores(gpu_scores, ref_scores, bound, where=""):
    err = np.abs(gpu_scores.astype(np.float64) - ref_scores)
    tol = SCORE_RTOL * bound + 1e-30
    bad = err > tol
    assert not bad.any(), f"{where} scores off at {bad.sum()} regions, max err/tol {np.max(err / tol):.3g}"


def check_selection_near_ties(gpu_ids, gpu_cnt, ref_ids, ref_cnt, ref_scores, where=""):
    """Selection from an independent chain: equal except at near-ties (reference scores
    of the swapped regions within NEAR_TIE relative)."""
    assert gpu_cnt == ref_cnt, f"{where} count {gpu_cnt} != {ref_cnt}"
    a = gpu_ids[:gpu_cnt]
    b = ref_ids[:ref_cnt]
    if np.array_equal(a, b):
        return 0
    assert len(set(a.tolist())) == len(a), f"{where} repeated ids"
    sa = ref_scores[a]
    sb = ref_scores[b]
    # the multiset of reference scores at each rank must agree up to near-ties
    gap = np.abs(sa - sb)
    scale = np.maximum(np.abs(sa), np.abs(sb))
    ok = gap <= NEAR_TIE * scale
    assert ok.all(), (f"{where} selection differs beyond near-ties at ranks "
                      f"{np.nonzero(~ok)[0][:8]}: {sa[~ok][:4]} vs {sb[~ok][:4]}")
    return int((a != b).sum())


def check_selection_chain(gpu_ids, gpu_cnt, ref_ids, ref_cnt, ref_scores, flipped, where=""):
    """Selection from the oracle's independent chain.  ``flipped`` [R] marks regions
    whose summary code differs between the GPU and the oracle (allowed midpoint cases).
    With those regions taken out of both lists, the rest must agree rank by rank up to
    near-ties, and any extra tail entry of the GPU list must be the best region the
    oracle left out (up to a near-tie).  Returns the number of flipped regions involved."""
    assert gpu_cnt == ref_cnt, f"{where} count {gpu_cnt} != {ref_cnt}"
    a = np.asarray(gpu_ids[:gpu_cnt])
    b = np.asarray(ref_ids[:ref_cnt])
    if np.array_equal(a, b):
        return 0
    if not flipped.any():
        return check_selection_near_ties(gpu_ids, gpu_cnt, ref_ids, ref_cnt, ref_scores, where)
    a1 = a[~flipped[a]]
    b1 = b[~flipped[b]]
    m = min(len(a1), len(b1))
    sa, sb = ref_scores[a1[:m]], ref_scores[b1[:m]]
    ok = np.abs(sa - sb) <= NEAR_TIE * np.maximum(np.abs(sa), np.abs(sb))
    assert ok.all(), f"{where} chain selection differs beyond near-ties and flipped summaries"
    if len(a1) > m:
        R = len(ref_scores)
        left_out = np.setdiff1d(np.nonzero(~flipped)[0], b1)
        best = np.sort(ref_scores[left_out])[::-1][:len(a1) - m]
        got = np.sort(ref_scores[a1[m:]])[::-1]
        assert np.all(np.abs(got - best) <= NEAR_TIE * np.maximum(np.abs(got), np.abs(best))), \
            f"{where} extra picks are not the next-best regions"
        del R
    return int(flipped[a].sum() + flipped[b].sum())


def check_out(gpu_out, ref_out, where=""):
    err = np.abs(gpu_out.astype(np.float64) - ref_out)
    assert np.all(np.isfinite(gpu_out)), f"{where} non-finite outputs"
    assert err.max() <= OUT_ATOL, f"{where} attention output off by {err.max():.4g}"
    return float(err.max())


def run_path(s5, geom, w, t, path: int = 0, want_scores=True, want_summ_f32=True, stream=None):
    """One full pass on the GPU; returns a dict of host copies."""
    dev = t["q"].device
    N, G = w.N, geom.num_kv_groups
    ws = s5.Workspace.create(geom, N, w.r_cap, device=dev)
    sel_ids = torch.full((N, G, geom.top_k), -7, dtype=torch.int32, device=dev)
    sel_count = torch.full((N, G), -7, dtype=torch.int32, device=dev)
    sel_scores = torch.empty((N, G, geom.top_k), dtype=torch.float32, device=dev)
    scores = torch.full((N, G, w.r_cap), float("nan"), dtype=torch.float32, device=dev) if want_scores else None
    summ_f32 = (torch.full(t["summaries"].shape, float("nan"), dtype=torch.float32, device=dev)
                if want_summ_f32 else None)
    out = torch.empty((N, geom.num_q_heads, geom.head_dim), dtype=torch.bfloat16, device=dev)
    prev = s5.step5_set_select_path(path)
    try:
        s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["sum_begin"],
                                  t["sum_end"], t["summaries"], summ_f32, max_regions_per_seq=w.max_span)
        s5.step5_index_score_topk(geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], t["cos"],
                                  t["sin"], t["summaries"], sel_ids, sel_count, ws.tensor,
                                  t_cap=w.t_cap, scores=scores, sel_scores=sel_scores)
        s5.step5_sparse_attn(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"],
                             sel_ids, sel_count, out, ws.tensor)
    finally:
        s5.step5_set_select_path(prev)
    torch.cuda.synchronize()
    status = s5.step5_device_status()
    res = dict(sel_ids=sel_ids.cpu().numpy(), sel_count=sel_count.cpu().numpy(),
               sel_scores=sel_scores.cpu().numpy(), out=out.float().cpu().numpy(),
               summaries=S.codes8(t["summaries"]), status=status)
    if scores is not None:
        res["scores"] = scores.cpu().numpy()
    if summ_f32 is not None:
        res["summ_f32"] = summ_f32.cpu().numpy()
    return res
