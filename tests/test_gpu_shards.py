"""GPU parity of the sequence-sharded decode: a row's regions and KV cache split over S
shards at uneven token cuts, each shard scored, picked and attended on its own, the
picks merged and the softmax states combined.

The whole-row path is the reference for the selection (the shards' merged pick must
equal it exactly: same scores, same (-score, id) order); every shard's state is checked
against the oracle's partial attention over the same token range, and the combined
output against the oracle's attention over the whole row (and, with one shard, against
step5_sparse_attn bit for bit).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from parity import check_out, run_path

pytestmark = pytest.mark.gpu

SLOT = 130


@pytest.fixture(scope="module")
def s5():
    import block_sparse_attention_step5_gb300 as s5
    s5.build()
    s5.load()
    torch.cuda.init()
    return s5


def token_cuts(t_cap, n_shards, seed):
    """n_shards + 1 increasing multiples of 8 from 0 to t_cap, at uneven places."""
    rng = np.random.default_rng(seed)
    inner = np.sort(rng.choice(np.arange(1, t_cap // 8), size=n_shards - 1, replace=False)) * 8
    return [0, *inner.tolist(), t_cap]


def run_shards(s5, geom, w, t, cuts, sel_ids, sel_count, workspace=True):
    """Scores / picks of every shard, their merge, and every shard's attention state over
    the given (whole-row) pick; returns device tensors."""
    dev = t["q"].device
    N, G, K, Hq = w.N, geom.num_kv_groups, geom.top_k, geom.num_q_heads
    n = len(cuts) - 1
    ids = torch.full((n, N, G, K), -7, dtype=torch.int32, device=dev)
    cnt = torch.full((n, N, G), -7, dtype=torch.int32, device=dev)
    scs = torch.empty((n, N, G, K), dtype=torch.float32, device=dev)
    states = torch.full((n, N, Hq, SLOT), float("nan"), dtype=torch.float32, device=dev)
    for s in range(n):
        lo_t, hi_t = cuts[s], cuts[s + 1]
        lo, hi = lo_t // 8, min(hi_t // 8, w.r_cap)
        summ = t["summaries"][:, :, lo:hi].contiguous()
        ws = s5.Workspace.create(geom, N, hi - lo, device=dev).tensor if workspace else None
        s5.step5_index_score_topk_shard(geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], t["cos"], t["sin"],
                                        summ, lo, ids[s], cnt[s], scs[s], ws, t_cap=w.t_cap)
        kc = t["k_cache"][:, :, lo_t:hi_t].contiguous()
        vc = t["v_cache"][:, :, lo_t:hi_t].contiguous()
        s5.step5_sparse_attn_shard(geom, t["q"], kc, vc, lo_t, t["row_seq"], t["row_pos"], sel_ids, sel_count,
                                   states[s], ws)
    m_ids = torch.full((N, G, K), -7, dtype=torch.int32, device=dev)
    m_cnt = torch.full((N, G), -7, dtype=torch.int32, device=dev)
    m_sc = torch.empty((N, G, K), dtype=torch.float32, device=dev)
    s5.step5_merge_topk(geom, ids, scs, cnt, m_ids, m_cnt, m_sc)
    return dict(ids=ids, cnt=cnt, scs=scs, states=states, m_ids=m_ids, m_cnt=m_cnt, m_sc=m_sc)


CASES = [
    ({"positions": [30000, 4100, 70, 15], "B": 2}, 4, 71),
    ({"positions": [9000] * 6 + [4101, 4102], "B": 3}, 3, 73),
    ({"positions": [60007], "B": 1}, 8, 79),
]


@pytest.mark.parametrize("cfg,n_shards,seed", CASES)
def test_sharded_decode_matches_the_whole_row(s5, cfg, n_shards, seed):
    geom = s5.STEP5_GEOMETRY
    w = S.workload(cfg, seed=seed)
    t = S.materialize(w, device="cuda")
    g = run_path(s5, geom, w, t, path=0)
    assert g["status"] == 0
    dev = t["q"].device
    sel_ids = torch.from_numpy(g["sel_ids"]).to(dev)
    sel_count = torch.from_numpy(g["sel_count"]).to(dev)
    cuts = token_cuts(w.t_cap, n_shards, seed)
    r = run_shards(s5, geom, w, t, cuts, sel_ids, sel_count)
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    G, K, Hq = geom.num_kv_groups, geom.top_k, geom.num_q_heads
    hq_g = Hq // G
    ids, cnt, scs = r["ids"].cpu().numpy(), r["cnt"].cpu().numpy(), r["scs"].cpu().numpy()
    # each shard's pick: the shard's candidates, with the whole-row scores, in key order
    for s in range(n_shards):
        lo, hi = cuts[s] // 8, min(cuts[s + 1] // 8, w.r_cap)
        for n in range(w.N):
            R = int(w.row_pos[n]) // 8
            want = max(0, min(hi, R) - lo)
            for gg in range(G):
                c = int(cnt[s, n, gg])
                assert c == min(K, want)
                got = ids[s, n, gg, :c]
                assert np.all((got >= lo) & (got < min(hi, R)))
                assert np.array_equal(scs[s, n, gg, :c], g["scores"][n, gg, got])
                assert np.all(ids[s, n, gg, c:] == -1)
    # the merge equals the whole-row pick exactly, and the oracle's merge of the lists
    assert np.array_equal(r["m_cnt"].cpu().numpy(), g["sel_count"])
    assert np.array_equal(r["m_ids"].cpu().numpy(), g["sel_ids"])
    assert np.array_equal(r["m_sc"].cpu().numpy(), g["sel_scores"])
    for n in range(w.N):
        for gg in range(G):
            ref = oracle.merge_topk(ids[:, n, gg], scs[:, n, gg], cnt[:, n, gg], K)
            assert np.array_equal(ref, g["sel_ids"][n, gg, :g["sel_count"][n, gg]])
    # every shard's state against the oracle's partial attention over its tokens
    st = r["states"].cpu().numpy()
    q, kc, vc = S.codes16(t["q"]), S.codes16(t["k_cache"]), S.codes16(t["v_cache"])
    empty = 0
    for s in range(n_shards):
        for n in range(w.N):
            b, pos = int(w.row_seq[n]), int(w.row_pos[n])
            for gg in range(G):
                c = int(g["sel_count"][n, gg])
                m, l, o = oracle.attend_partial(q[n, gg * hq_g:(gg + 1) * hq_g], kc[b, gg], vc[b, gg],
                                                g["sel_ids"][n, gg, :c], pos, cuts[s], cuts[s + 1],
                                                geom.softmax_scale)
                x = st[s, n, gg * hq_g:(gg + 1) * hq_g]
                for h in range(hq_g):
                    if m[h] == -math.inf:
                        empty += 1
                        assert x[h, 0] == -math.inf and x[h, 1] == 0.0 and not x[h, 2:].any()
                        continue
                    assert abs(x[h, 0] * math.log(2.0) - m[h]) <= 1e-4 * max(1.0, abs(m[h]))
                    assert abs(x[h, 1] - l[h]) <= 1e-4 * l[h]
                    check_out((x[h, 2:] / x[h, 1])[None], (o[h] / l[h])[None], where=f"shard {s} row {n} head {h}")
    if cfg["positions"][-1] == 15:
        assert empty > 0  # the row at 15 has keys (tokens 0..15) in at most two shards
    # the combined output against the oracle's whole-row attention (with and without gate)
    out = torch.full((w.N, Hq, geom.head_dim), float("nan"), dtype=torch.bfloat16, device=dev)
    s5.step5_attn_combine(geom, r["states"], out)
    gen = torch.Generator().manual_seed(seed)
    gate = (torch.randn((w.N, Hq), generator=gen) * 3).to(torch.bfloat16).to(dev)
    gated = torch.empty_like(out)
    s5.step5_attn_combine(geom, r["states"], gated, gate=gate)
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    ref, _ = oracle.attend_batch(q, kc, vc, w.row_seq, w.row_pos, g["sel_ids"], g["sel_count"], geom.softmax_scale)
    check_out(out.float().cpu().numpy(), ref, where="combined")
    check_out(gated.float().cpu().numpy(), oracle.sigmoid_gate(ref, S.codes16(gate)), where="combined, gated")


@pytest.mark.parametrize("workspace", [True, False])
def test_one_shard_is_the_whole_row_bit_for_bit(s5, workspace):
    """One shard holding every token: the state, combined, is step5_sparse_attn's output
    bit for bit (the same blocks and merge order; the combine's weight is exactly 1) when
    the whole-row call takes the warp-level kernel the shard call takes (without a
    workspace the whole-row call would otherwise take the tensor-core kernel, whose fp32
    sums run in another order)."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [30000, 4100, 70, 15], "B": 2}, seed=83)
    t = S.materialize(w, device="cuda")
    g = run_path(s5, geom, w, t, path=0)
    dev = t["q"].device
    sel_ids = torch.from_numpy(g["sel_ids"]).to(dev)
    sel_count = torch.from_numpy(g["sel_count"]).to(dev)
    ws = s5.Workspace.create(geom, w.N, w.r_cap, device=dev).tensor if workspace else None
    states = torch.empty((1, w.N, geom.num_q_heads, SLOT), dtype=torch.float32, device=dev)
    s5.step5_sparse_attn_shard(geom, t["q"], t["k_cache"], t["v_cache"], 0, t["row_seq"], t["row_pos"], sel_ids,
                               sel_count, states[0], ws)
    out = torch.empty((w.N, geom.num_q_heads, geom.head_dim), dtype=torch.bfloat16, device=dev)
    s5.step5_attn_combine(geom, states, out)
    plain = torch.empty_like(out)
    prev = s5.step5_set_attention_path(1)
    try:
        s5.step5_sparse_attn(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"], sel_ids,
                             sel_count, plain, ws)
    finally:
        s5.step5_set_attention_path(prev)
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))


def test_merge_clamps_a_bad_count(s5):
    """A shard count outside [0, top_k] raises the range bit and is clamped."""
    geom = s5.STEP5_GEOMETRY
    dev = torch.device("cuda")
    K, G = geom.top_k, geom.num_kv_groups
    ids = torch.arange(2 * G * K, dtype=torch.int32, device=dev).view(2, 1, G, K)
    scs = torch.zeros((2, 1, G, K), dtype=torch.float32, device=dev)
    cnt = torch.tensor([[[-3] * G], [[K] * G]], dtype=torch.int32, device=dev)
    m_ids = torch.empty((1, G, K), dtype=torch.int32, device=dev)
    m_cnt = torch.empty((1, G), dtype=torch.int32, device=dev)
    s5.step5_merge_topk(geom, ids, scs, cnt, m_ids, m_cnt)
    torch.cuda.synchronize()
    assert s5.step5_device_status() == s5.DEV_RANGE
    assert (m_cnt.cpu() == K).all()
    assert torch.equal(m_ids.cpu(), ids[1].cpu())


@pytest.mark.parametrize("S_, K", [(1, 512), (8, 2048), (32, 512)])
def test_merge_at_its_limits(s5, S_, K):
    """The merge against the oracle's merge at one shard and at S * top_k = 16,384 keys
    (the most a merge block stages), with random scores, ties and short lists."""
    geom = s5.Geometry.step5(top_k=K)
    G = geom.num_kv_groups
    dev = torch.device("cuda")
    rng = np.random.default_rng(101 + S_)
    N = 2
    ids = np.full((S_, N, G, K), -1, dtype=np.int32)
    scs = np.full((S_, N, G, K), -np.inf, dtype=np.float32)
    cnt = np.zeros((S_, N, G), dtype=np.int32)
    for s in range(S_):
        for n in range(N):
            for g in range(G):
                c = int(rng.integers(0, K + 1)) if (s + n + g) % 3 else K
                pool = rng.choice(1 << 20, size=c, replace=False).astype(np.int32) * S_ + s  # distinct across shards
                sc = np.round(rng.standard_normal(c) * 4).astype(np.float32)  # many exact ties
                order = np.lexsort((pool, -sc.astype(np.float64)))
                ids[s, n, g, :c] = pool[order]
                scs[s, n, g, :c] = sc[order]
                cnt[s, n, g] = c
    d_ids, d_scs, d_cnt = (torch.from_numpy(x).to(dev) for x in (ids, scs, cnt))
    m_ids = torch.full((N, G, K), -7, dtype=torch.int32, device=dev)
    m_cnt = torch.full((N, G), -7, dtype=torch.int32, device=dev)
    m_sc = torch.empty((N, G, K), dtype=torch.float32, device=dev)
    s5.step5_merge_topk(geom, d_ids, d_scs, d_cnt, m_ids, m_cnt, m_sc)
    torch.cuda.synchronize()
    assert s5.step5_device_status() == 0
    got_ids, got_cnt, got_sc = m_ids.cpu().numpy(), m_cnt.cpu().numpy(), m_sc.cpu().numpy()
    for n in range(N):
        for g in range(G):
            ref = oracle.merge_topk(ids[:, n, g], scs[:, n, g], cnt[:, n, g], K)
            c = int(got_cnt[n, g])
            assert c == len(ref)
            assert np.array_equal(got_ids[n, g, :c], ref)
            assert np.all(got_ids[n, g, c:] == -1) and np.all(np.isneginf(got_sc[n, g, c:]))


@pytest.mark.parametrize("cfg,n_shards,seed", CASES[:2])
def test_merge_attend_composition_matches_the_two_calls(s5, cfg, n_shards, seed):
    """step5_merge_attend_shard (the merge, then the shard's attention, launched back to
    back with the attention waiting on the device) writes the merged pick and each shard's
    states bit for bit as step5_merge_topk and step5_sparse_attn_shard do."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload(cfg, seed=seed)
    t = S.materialize(w, device="cuda")
    g = run_path(s5, geom, w, t, path=0)
    dev = t["q"].device
    sel_ids = torch.from_numpy(g["sel_ids"]).to(dev)
    sel_count = torch.from_numpy(g["sel_count"]).to(dev)
    cuts = token_cuts(w.t_cap, n_shards, seed)
    r = run_shards(s5, geom, w, t, cuts, sel_ids, sel_count)
    N, G, K = w.N, geom.num_kv_groups, geom.top_k
    for s in range(n_shards):
        lo_t, hi_t = cuts[s], cuts[s + 1]
        kc = t["k_cache"][:, :, lo_t:hi_t].contiguous()
        vc = t["v_cache"][:, :, lo_t:hi_t].contiguous()
        ws = s5.Workspace.create(geom, N, w.r_cap, device=dev).tensor if s % 2 == 0 else None
        c_ids = torch.full((N, G, K), -7, dtype=torch.int32, device=dev)
        c_cnt = torch.full((N, G), -7, dtype=torch.int32, device=dev)
        c_states = torch.full((N, geom.num_q_heads, SLOT), float("nan"), dtype=torch.float32, device=dev)
        s5.step5_merge_attend_shard(geom, r["ids"], r["scs"], r["cnt"], t["q"], kc, vc, lo_t, t["row_seq"],
                                    t["row_pos"], c_ids, c_cnt, c_states, ws)
        # the reference states with the same workspace choice
        ref_states = torch.empty_like(c_states)
        s5.step5_sparse_attn_shard(geom, t["q"], kc, vc, lo_t, t["row_seq"], t["row_pos"], r["m_ids"], r["m_cnt"],
                                   ref_states, ws)
        torch.cuda.synchronize()
        assert s5.step5_device_status() == 0
        assert torch.equal(c_ids, r["m_ids"]) and torch.equal(c_cnt, r["m_cnt"])
        assert torch.equal(c_states.view(torch.int32), ref_states.view(torch.int32))
