"""The C-ABI boundary without a GPU: the library loads, exports every function that
include/*.h declares, and rejects bad arguments on the host before anything is
enqueued (no CUDA call is reached on these paths).

Geometry rules follow the vLLM Step5 DSA validation (provider groups = KV groups,
indexer heads divisible into them, 4/8/16 query heads per KV group).
"""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def s5():
    import block_sparse_attention_step5_gb300 as s5
    s5.build()
    s5.load()
    return s5


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(step5_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_three_steps():
    names = declared_functions()
    for n in ("step5_region_summarize", "step5_index_score_topk", "step5_sparse_attn"):
        assert n in names


def test_library_exports_every_declared_symbol(s5):
    lib = ctypes.CDLL(s5.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), name
    binding = set(dir(s5))
    for name in declared_functions():
        assert name in binding, f"binding lacks {name}"


def test_library_links_no_oracle(s5):
    data = open(s5.library_path(), "rb").read()
    assert b"orc_" not in data and b"liboracle" not in data


def G(**over):
    import block_sparse_attention_step5_gb300 as s5
    return s5.Geometry.step5(**over)


@pytest.mark.parametrize("over,expect", [
    ({}, "ok"),
    ({"num_kv_groups": 3}, 2),          # 16 indexer heads do not divide into 3 groups
    ({"num_q_heads": 8}, 2),            # 2 q heads per group
    ({"num_q_heads": 128}, 2),          # 32 q heads per group
    ({"num_q_heads": 64}, "ok"),        # 16 per group
    ({"num_q_heads": 16}, "ok"),        # 4 per group
    ({"idx_heads": 48}, 2),             # 12 per group
    ({"idx_heads": 8}, "ok"),           # 2 per group
    ({"head_dim": 64}, 2),
    ({"idx_dim": 128}, 2),
    ({"rope_dims": 24}, 2),
    ({"rope_dims": 0}, "ok"),
    ({"region_tokens": 16}, 2),
    ({"top_k": 0}, 2),
    ({"top_k": 4096}, 2),
    ({"softmax_scale": 0.0}, 1),
    ({"softmax_scale": float("nan")}, 1),
    ({"num_kv_groups": 0}, 1),
])
def test_geometry_rules(s5, over, expect):
    g = G(**over)
    nbytes = s5.step5_workspace_bytes(g, 4, 1000)
    if expect == "ok":
        assert nbytes > 0
    else:
        assert nbytes == 0
        lib = s5.load()
        st = lib.step5_region_summarize(ctypes.byref(g), 1, 64, 8, 1, None, None, None, None, None,
                                        None, None, None, None)
        assert st == expect


def test_null_and_size_rejections(s5):
    lib = s5.load()
    g = G()
    fake = ctypes.c_void_p(0x10000)        # never dereferenced: rejected on the host
    odd = ctypes.c_void_p(0x10008)         # not 16-byte aligned
    # summarize: null required pointers, t_cap not a multiple of 8, misaligned
    assert lib.step5_region_summarize(ctypes.byref(g), 1, 64, 8, 1, None, fake, None, None, fake,
                                      fake, fake, None, None) == 1
    assert lib.step5_region_summarize(ctypes.byref(g), 1, 60, 8, 1, fake, fake, None, None, fake,
                                      fake, fake, None, None) == 1
    assert lib.step5_region_summarize(ctypes.byref(g), 1, 64, 8, 1, odd, fake, None, None, fake,
                                      fake, fake, None, None) == 1
    assert lib.step5_region_summarize(ctypes.byref(g), 1, 64, 8, 1, fake, fake, fake, None, fake,
                                      fake, fake, None, None) == 1   # cos without sin
    assert lib.step5_region_summarize(ctypes.byref(g), 0, 64, 8, 1, fake, fake, None, None, fake,
                                      fake, fake, None, None) == 1
    # score/select: missing workspace on the split path, null outputs
    s5.step5_set_select_path(2)
    try:
        assert lib.step5_index_score_topk(ctypes.byref(g), 1, 1, 64, 100000, fake, fake, fake, fake,
                                          None, None, fake, fake, fake, None, None, None, 0,
                                          None) == 3
        assert lib.step5_index_score_topk(ctypes.byref(g), 1, 1, 64, 100000, fake, fake, fake, fake,
                                          None, None, fake, fake, fake, None, None, fake, 16,
                                          None) == 3
    finally:
        s5.step5_set_select_path(0)
    assert lib.step5_index_score_topk(ctypes.byref(g), 1, 1, 64, 8, fake, fake, fake, fake, None,
                                      None, fake, None, fake, None, None, None, 0, None) == 1
    # attention: odd t_cap, misaligned cache, too many rows
    assert lib.step5_sparse_attn(ctypes.byref(g), 1, 1, 60, fake, fake, fake, fake, fake, fake,
                                 fake, fake, None, 0, None) == 1
    assert lib.step5_sparse_attn(ctypes.byref(g), 1, 1, 64, fake, odd, fake, fake, fake, fake,
                                 fake, fake, None, 0, None) == 1
    assert lib.step5_sparse_attn(ctypes.byref(g), 1 << 20, 1, 64, fake, fake, fake, fake, fake,
                                 fake, fake, fake, None, 0, None) == 2


def test_shard_call_rejections(s5):
    """The sequence-shard calls reject bad arguments on the host, before any launch."""
    lib = s5.load()
    g = G()
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    # shard scoring: negative region_lo, missing picked-score output
    assert lib.step5_index_score_topk_shard(ctypes.byref(g), 1, 1, 64, 8, -8, fake, fake, fake, fake, None,
                                            None, fake, fake, fake, fake, None, 0, None) == 1
    assert lib.step5_index_score_topk_shard(ctypes.byref(g), 1, 1, 64, 8, 0, fake, fake, fake, fake, None,
                                            None, fake, fake, fake, None, None, 0, None) == 1
    # merge: no shards, too many shards or keys, null inputs
    assert lib.step5_merge_topk(ctypes.byref(g), 0, 1, fake, fake, fake, fake, fake, None, None) == 1
    assert lib.step5_merge_topk(ctypes.byref(g), 33, 1, fake, fake, fake, fake, fake, None, None) == 2
    assert lib.step5_merge_topk(ctypes.byref(G(top_k=2048)), 9, 1, fake, fake, fake, fake, fake, None,
                                None) == 2
    assert lib.step5_merge_topk(ctypes.byref(g), 2, 1, None, fake, fake, fake, fake, None, None) == 1
    # shard attention: no states, token_lo off the region grid, misaligned states
    assert lib.step5_sparse_attn_shard(ctypes.byref(g), 1, 1, 64, 0, fake, fake, fake, fake, fake, fake,
                                       fake, None, None, 0, None) == 1
    assert lib.step5_sparse_attn_shard(ctypes.byref(g), 1, 1, 64, 4, fake, fake, fake, fake, fake, fake,
                                       fake, fake, None, 0, None) == 1
    assert lib.step5_sparse_attn_shard(ctypes.byref(g), 1, 1, 64, 8, fake, fake, fake, fake, fake, fake,
                                       fake, odd, None, 0, None) == 1
    # combine: no shards, too many, misaligned output
    assert lib.step5_attn_combine(ctypes.byref(g), 0, 1, fake, None, fake, None) == 1
    assert lib.step5_attn_combine(ctypes.byref(g), 33, 1, fake, None, fake, None) == 2
    assert lib.step5_attn_combine(ctypes.byref(g), 2, 1, fake, None, odd, None) == 1


def test_rows_layout_and_host_step_rejections(s5):
    """The packed per-row input layout (256-byte aligned arrays in the documented order,
    no overlap) and the host-buffer step's argument checks."""
    lib = s5.load()
    g = s5.STEP5_GEOMETRY
    for N, B in ((1, 1), (16, 16), (2048, 1), (3, 7)):
        lay = s5.step5_rows_layout_for(g, N, B)
        sizes = [N * g.num_q_heads * g.head_dim * 2, N * g.idx_heads * g.idx_dim * 2, N * g.idx_heads * 4,
                 N * 4, N * 4, B * 4, B * 4]
        offs = [lay.q, lay.idx_q, lay.w, lay.row_seq, lay.row_pos, lay.region_begin, lay.region_end, lay.total]
        assert offs[0] == 0
        for i, size in enumerate(sizes):
            assert offs[i] % 256 == 0 and offs[i] + size <= offs[i + 1] < offs[i] + size + 256
    with pytest.raises(s5.Step5Error):
        s5.step5_rows_layout_for(g, 0, 1)
    G_ = ctypes.byref(G())
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    args = lambda rows_host, rows_dev, out_host: (G_, 1, 1, 64, 8, 1, fake, fake, None, None, fake, fake, fake,
                                                  rows_host, rows_dev, out_host, fake, fake, fake, None, 0, None)
    assert lib.step5_decode_step_host(*args(None, fake, fake)) == 1
    assert lib.step5_decode_step_host(*args(fake, odd, fake)) == 1
    assert lib.step5_decode_step_host(*args(fake, fake, None)) == 1


def test_select_path_rule(s5):
    """The automatic scoring path at the measured points: fused for one row up to ~3,000
    regions and for sixteen rows at 16K-32K tokens, split for single rows beyond that and
    for the 128K / 1M decodes, tensor-core scoring for prefill chunks (many rows of one
    sequence), fused for many rows of as many sequences."""
    g = s5.STEP5_GEOMETRY
    prev = s5.step5_set_select_path(0)
    try:
        for N, B, r_cap, want in ((1, 1, 577, 1), (1, 1, 2051, 1), (1, 1, 3001, 2), (1, 1, 6001, 2),
                                  (4, 4, 6001, 2), (16, 16, 3842, 1), (16, 16, 4097, 1), (16, 16, 8000, 2),
                                  (4, 4, 16385, 2), (1, 1, 131073, 2), (2048, 1, 8449, 3), (2048, 2048, 8449, 1),
                                  (256, 32, 4000, 3), (256, 64, 4000, 1), (2048, 1, 16385, 2)):
            assert s5.step5_select_path_for(g, N, r_cap, B) == want, (N, B, r_cap)
    finally:
        s5.step5_set_select_path(prev)


def test_status_strings(s5):
    for code in range(6):
        assert isinstance(s5.step5_status_string(code), str)
    assert s5.step5_status_string(0) == "ok"


def test_workspace_grows_with_rows_and_regions(s5):
    g = G()
    a = s5.step5_workspace_bytes(g, 1, 131073)
    b = s5.step5_workspace_bytes(g, 4, 131073)
    c = s5.step5_workspace_bytes(g, 4, 16385)
    assert 0 < c < b and a < b


def test_select_path_switch_roundtrip(s5):
    prev = s5.step5_set_select_path(1)
    assert s5.step5_set_select_path(2) == 1
    assert s5.step5_set_select_path(prev) == 2
    assert s5.step5_set_select_path(3) == prev
    assert s5.step5_set_select_path(prev) == 3
    assert s5.step5_set_select_path(7) == prev   # out-of-range modes are ignored
    assert s5.step5_set_select_path(prev) == prev


def test_wait_polls_switch_roundtrip(s5):
    prev = s5.step5_set_wait_polls(1000)
    assert prev > 0
    assert s5.step5_set_wait_polls(0) == 1000      # 0 restores the default ...
    assert s5.step5_set_wait_polls(0) == prev      # ... which the next call reports
