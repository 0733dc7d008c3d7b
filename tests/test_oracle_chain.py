"""The oracle's four steps chained over a small synthetic workload.

Invariant from the CSA-indexer commit: a row with at most 512 candidate regions keeps
them all, so its attention is the dense one -- while a row has at most 512 completed
regions the selection is every region (in key order) and the output equals dense
causal attention (torch SDPA, fp64).  Above 512 regions the chain keeps exactly 512
ids, each the id of a completed region, none repeated, in non-increasing score order.
"""
import math

import numpy as np
import torch

import synthetic as S


def run_chain(orc, w, t):
    g = w.geom
    c16 = S.codes16
    summ, _, _ = orc.summarize_batch(c16(t["idx_k"]), c16(t["idx_z"]), c16(t["cos"]), c16(t["sin"]),
                                     w.sum_begin, w.sum_end, w.r_cap, g.rope_dims)
    scores, _ = orc.score_batch(c16(t["idx_q"]), t["w"].numpy(), w.row_seq, w.row_pos, summ,
                                g.num_kv_groups, g.rope_dims, c16(t["cos"]), c16(t["sin"]))
    ids, cnt, _ = orc.select_batch(scores, w.row_pos, K=g.top_k)
    out, _ = orc.attend_batch(c16(t["q"]), c16(t["k_cache"]), c16(t["v_cache"]), w.row_seq,
                              w.row_pos, ids, cnt, g.softmax_scale)
    return summ, scores, ids, cnt, out


def test_chain_dense_equivalence_small(orc):
    w = S.workload({"positions": [0, 7, 8, 9, 17, 129, 300], "B": 3}, seed=41)
    t = S.materialize(w)
    summ, scores, ids, cnt, out = run_chain(orc, w, t)
    g = w.geom
    hpg = g.num_q_heads // g.num_kv_groups
    for n in range(w.N):
        p, b = int(w.row_pos[n]), int(w.row_seq[n])
        R = p // 8
        for gg in range(g.num_kv_groups):
            assert cnt[n, gg] == R
            assert sorted(ids[n, gg, :R].tolist()) == list(range(R))
            assert np.all(ids[n, gg, R:] == -1)
            q = torch.from_numpy(orc.bf16_values(S.codes16(t["q"][n, gg * hpg:(gg + 1) * hpg])))
            k = torch.from_numpy(orc.bf16_values(S.codes16(t["k_cache"][b, gg, :p + 1])))
            v = torch.from_numpy(orc.bf16_values(S.codes16(t["v_cache"][b, gg, :p + 1])))
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[:, None, :], k[None].expand(hpg, -1, -1), v[None].expand(hpg, -1, -1),
                scale=g.softmax_scale)[:, 0]
            assert np.allclose(out[n, gg * hpg:(gg + 1) * hpg], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_chain_prunes_above_512(orc):
    w = S.workload({"positions": [4300], "B": 1}, seed=17)
    t = S.materialize(w)
    summ, scores, ids, cnt, out = run_chain(orc, w, t)
    R = 4300 // 8
    for gg in range(4):
        assert cnt[0, gg] == 512
        sel = ids[0, gg]
        assert len(set(sel.tolist())) == 512 and sel.min() >= 0 and sel.max() < R
        sc = scores[0, gg, sel]
        assert np.all(np.diff(sc) <= 0)
        # everything not picked scores no higher than the last pick
        rest = np.setdiff1d(np.arange(R), sel)
        assert scores[0, gg, rest].max() <= sc[-1]
    assert np.all(np.isfinite(out))
