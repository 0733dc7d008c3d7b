"""Step (4) on the two kernels that take a (row, KV group) in one CTA -- the tcgen05
tensor-core kernel and the warp-level MMA kernel -- against the oracle on the same
picks: several 16-region tiles with a ragged last tile, own regions of 1 to 8 tokens,
rows with no candidate region and rows with fewer than top_k, 4, 8 and 16 query heads per
KV group, picks in an arbitrary order, and NaN in the cache rows past the last position
of each sequence (never read into the result)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from parity import check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s5():
    import block_sparse_attention_step5_gb300 as s5
    s5.build()
    s5.load()
    return s5


def random_picks(w, K, seed):
    """min(K, R) distinct candidate regions per (row, group), in random order, -1 after."""
    rng = np.random.default_rng(seed)
    G = w.geom.num_kv_groups
    ids = np.full((w.N, G, K), -1, np.int32)
    cnt = np.zeros((w.N, G), np.int32)
    for n in range(w.N):
        R = int(w.row_pos[n]) // 8
        for g in range(G):
            k = min(K, R)
            ids[n, g, :k] = rng.choice(R, size=k, replace=False)
            cnt[n, g] = k
    return ids, cnt


def poison_past_positions(w, t):
    """NaN in every cache row past the last position of its sequence."""
    for b in range(w.B):
        last = int(w.row_pos[w.row_seq == b].max())
        t["k_cache"][b, :, last + 1:] = float("nan")
        t["v_cache"][b, :, last + 1:] = float("nan")


@pytest.mark.parametrize("hq", [16, 32, 64])
@pytest.mark.parametrize("cfg", [{"positions": [30000, 4100, 70, 15, 8, 0], "B": 3},
                                 {"positions": [9000 + 3 * i for i in range(40)], "B": 5}])
def test_one_cta_kernels_match_the_oracle(s5, hq, cfg):
    base = s5.STEP5_GEOMETRY
    geom = s5.Geometry.step5(num_q_heads=hq)
    sg = S.Geometry(num_q_heads=hq, num_kv_groups=4, head_dim=128, idx_heads=16, idx_dim=64, rope_dims=32,
                    region_tokens=8, top_k=base.top_k, softmax_scale=base.softmax_scale)
    w = S.workload(cfg, seed=43, geom=sg)
    t = S.materialize(w, device="cuda")
    poison_past_positions(w, t)
    ids, cnt = random_picks(w, geom.top_k, 5)
    h = {k: S.codes16(t[k]) for k in ("q", "k_cache", "v_cache")}
    ref, _ = oracle.attend_batch(h["q"], h["k_cache"], h["v_cache"], w.row_seq, w.row_pos, ids, cnt,
                                 geom.softmax_scale)
    dev = t["q"].device
    d_ids, d_cnt = torch.from_numpy(ids).to(dev), torch.from_numpy(cnt).to(dev)
    outs = {}
    for path in (2, 1, 2):
        prev = s5.step5_set_attention_path(path)
        try:
            out = torch.full((w.N, hq, 128), float("nan"), dtype=torch.bfloat16, device=dev)
            s5.step5_sparse_attn(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"], d_ids,
                                 d_cnt, out, None)
            torch.cuda.synchronize()
        finally:
            s5.step5_set_attention_path(prev)
        assert s5.step5_device_status() == 0
        o = out.float().cpu().numpy()
        check_out(o, ref, where=f"kernel {path}")
        if path in outs:
            assert np.array_equal(o, outs[path])  # repeats bit for bit
        outs[path] = o


def test_tensor_core_kernel_with_gate_and_selection_order(s5):
    """The gated output, and picks handed over in key order (as the selection writes them)
    rather than at random: the same result within rounding."""
    geom = s5.STEP5_GEOMETRY
    w = S.workload({"positions": [20000 + 5 * i for i in range(24)], "B": 4}, seed=47)
    t = S.materialize(w, device="cuda")
    ids, cnt = random_picks(w, geom.top_k, 9)
    h = {k: S.codes16(t[k]) for k in ("q", "k_cache", "v_cache")}
    ref, _ = oracle.attend_batch(h["q"], h["k_cache"], h["v_cache"], w.row_seq, w.row_pos, ids, cnt,
                                 geom.softmax_scale)
    gen = torch.Generator().manual_seed(3)
    gate = (torch.randn((w.N, geom.num_q_heads), generator=gen) * 3).to(torch.bfloat16).to("cuda")
    ref_gated = oracle.sigmoid_gate(ref, S.codes16(gate))
    sorted_ids = np.where(ids >= 0, np.sort(np.where(ids >= 0, ids, 1 << 30), axis=-1), -1).astype(np.int32)
    prev = s5.step5_set_attention_path(2)
    try:
        for pick in (ids, sorted_ids):
            d_ids = torch.from_numpy(pick).cuda()
            d_cnt = torch.from_numpy(cnt).cuda()
            out = torch.empty((w.N, geom.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
            s5.step5_sparse_attn_gated(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"], d_ids,
                                       d_cnt, gate, out, None)
            torch.cuda.synchronize()
            assert s5.step5_device_status() == 0
            check_out(out.float().cpu().numpy(), ref_gated, where="gated tensor-core kernel")
    finally:
        s5.step5_set_attention_path(prev)
