"""Pins of the oracle's sequence-sharded decode: a row's regions split over S shards,
each shard picking its own top K, a merge of the picks, attention over each shard's
share of the keys and a combine of the partial softmax states.  Pinned against the
unsharded oracle (the selection over all regions, and dense attention over the union of
the keys, which the pages fix) on split points that cut regions, the own region and
empty shards, and by brute force on tiny lists.
"""
import numpy as np

import oracle


def test_merge_of_shard_picks_is_the_whole_rows_pick():
    rng = np.random.default_rng(1)
    R, K = 3000, 512
    scores = rng.standard_normal(R).astype(np.float32).astype(np.float64)
    scores[rng.integers(0, R, 300)] = scores[rng.integers(0, R, 300)]  # exact ties
    whole = oracle.select_topk(scores, K)
    for cuts in ([0, 1000, 2000, 3000], [0, 7, 2999, 3000], [0, 3000], [0, 1500, 1500, 3000]):
        S = len(cuts) - 1
        ids = np.full((S, K), -1, np.int32)
        sc = np.zeros((S, K))
        cnt = np.zeros(S, np.int32)
        for s in range(S):
            lo, hi = cuts[s], cuts[s + 1]
            pick = oracle.select_topk(scores[lo:hi], K) + lo if hi > lo else np.zeros(0, np.int32)
            cnt[s] = pick.size
            ids[s, :pick.size] = pick
            sc[s, :pick.size] = scores[pick]
        assert np.array_equal(oracle.merge_topk(ids, sc, cnt, K), whole)


def test_merge_brute_force_small():
    ids = np.array([[5, 2, -1], [9, 1, 7]], np.int32)
    sc = np.array([[3.0, 1.0, 0.0], [3.0, 2.0, 1.0]])
    cnt = np.array([2, 3], np.int32)
    # keys (-score, id): (-3,5) (-3,9) (-2,1) (-1,2) (-1,7)
    assert np.array_equal(oracle.merge_topk(ids, sc, cnt, 3), [5, 9, 1])
    assert np.array_equal(oracle.merge_topk(ids, sc, cnt, 8), [5, 9, 1, 2, 7])


def test_partial_attention_combines_to_the_whole():
    rng = np.random.default_rng(2)
    hq, D, t_cap, pos = 8, 128, 4096, 4000
    bf = lambda a: (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q = bf(rng.standard_normal((hq, D)))
    kc = bf(rng.standard_normal((t_cap, D)))
    vc = bf(rng.standard_normal((t_cap, D)))
    sel = np.sort(rng.choice(pos // 8, 300, replace=False)).astype(np.int32)
    scale = 1 / np.sqrt(128)
    whole = oracle.attend_group(q, kc, vc, sel, pos, 8, scale)
    for cuts in ([0, 1024, 2048, 3072, 4096], [0, 3, 4001, 4096], [0, 4096], [0, 2000, 2000, 4096]):
        parts = [oracle.attend_partial(q, kc, vc, sel, pos, cuts[s], cuts[s + 1], scale) for s in range(len(cuts) - 1)]
        for h in range(hq):
            m = np.array([p[0][h] for p in parts])
            l = np.array([p[1][h] for p in parts])
            o = np.stack([p[2][h] for p in parts])
            got = oracle.attn_combine(m, l, o)
            assert np.allclose(got, whole[h], rtol=1e-12, atol=1e-12)


def test_empty_shard_state():
    rng = np.random.default_rng(3)
    bf = lambda a: (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q = bf(rng.standard_normal((2, 128)))
    kc = bf(rng.standard_normal((64, 128)))
    m, l, o = oracle.attend_partial(q, kc, kc, np.array([0, 1], np.int32), 30, 40, 64, 0.1)
    assert np.all(np.isneginf(m)) and np.all(l == 0) and np.all(o == 0)
