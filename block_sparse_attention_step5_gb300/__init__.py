"""Python binding of libstep5sa: the Step-5 sparse-indexer attention on GB300 (sm_103a).

Thin ctypes marshalling over the C ABI declared in ``include/step5_sparse_attn.h``:
each function takes torch tensors that already live on the GPU, passes their device
pointers and the current CUDA stream, and raises ``Step5Error`` on a non-OK status.
Every step of the computation runs in the library's kernels; there is no other path.
If the library has not been built, the first call raises.

Steps (TensorFold PR #903, "Step-5-Preview on one 256 GB Mac", CSA-indexer commit):
  step5_region_summarize  -- e4m3 summary of each completed 8-token region
  step5_index_score_topk  -- sum_h relu(e4m3(q_h) . summary) * w_h, top-k by (-score, id)
  step5_sparse_attn       -- attention over the picked regions plus the row's own region
  step5_sparse_attn_gated -- the same, followed by the per-head sigmoid output gate
  step5_indexer_front     -- decode front end: q/k norms, k/z cache write, summary on completion
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

from ._build import LIB, build  # noqa: F401

__all__ = [
    "Step5Error", "Geometry", "STEP5_GEOMETRY", "library_path", "load",
    "step5_region_summarize", "step5_index_score_topk", "step5_sparse_attn", "step5_sparse_attn_gated",
    "step5_indexer_front",
    "step5_index_score_topk_noalloc",
    "step5_index_score_topk_shard", "step5_merge_topk", "step5_sparse_attn_shard", "step5_attn_combine",
    "step5_merge_attend_shard",
    "RowsLayout", "step5_rows_layout_for", "HostRows", "step5_decode_step_host", "step5_set_host_copies",
    "step5_workspace_bytes", "step5_workspace_init", "step5_device_status",
    "step5_set_select_path", "step5_set_wait_polls", "step5_set_attention_path", "step5_select_path_for", "step5_set_prologue_overlap", "step5_decode_step", "step5_status_string", "step5_convert_bf16_to_e4m3",
    "Workspace", "decode_step",
]

STATUS = {0: "STEP5_OK", 1: "STEP5_ERR_INVALID_ARGUMENT", 2: "STEP5_ERR_UNSUPPORTED",
          3: "STEP5_ERR_WORKSPACE", 4: "STEP5_ERR_CUDA", 5: "STEP5_ERR_TIMEOUT"}
DEV_RANGE, DEV_TIMEOUT = 1, 2


class Step5Error(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)}" + (f" ({detail})" if detail else ""))


class Geometry(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_groups", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("idx_heads", ctypes.c_int32),
                ("idx_dim", ctypes.c_int32), ("rope_dims", ctypes.c_int32),
                ("region_tokens", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float)]

    @classmethod
    def step5(cls, **over) -> "Geometry":
        vals = dict(num_q_heads=32, num_kv_groups=4, head_dim=128, idx_heads=16, idx_dim=64,
                    rope_dims=32, region_tokens=8, top_k=512, softmax_scale=1.0 / math.sqrt(128.0))
        vals.update(over)
        return cls(**vals)

    @classmethod
    def of(cls, g) -> "Geometry":
        if isinstance(g, Geometry):
            return g
        return cls(g.num_q_heads, g.num_kv_groups, g.head_dim, g.idx_heads, g.idx_dim,
                   g.rope_dims, g.region_tokens, g.top_k, g.softmax_scale)


STEP5_GEOMETRY = Geometry.step5()

_lib = None


def library_path() -> str:
    return LIB


def load():
    """Loads libstep5sa.so (raises if it is missing: build it with ``build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(f"{LIB} is not built; run block_sparse_attention_step5_gb300.build() "
                           "(nvcc, sm_103a) first")
    lib = ctypes.CDLL(LIB)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    G = ctypes.POINTER(Geometry)
    sigs = {
        "step5_region_summarize": (i32, [G, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P]),
        "step5_index_score_topk": (i32, [G, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P,
                                         P, sz, P]),
        "step5_sparse_attn": (i32, [G, i32, i32, i32, P, P, P, P, P, P, P, P, P, sz, P]),
        "step5_sparse_attn_gated": (i32, [G, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, sz, P]),
        "step5_indexer_front": (i32, [G, i32, i32, i32, i32, P, P, P, P, P, P, ctypes.c_float, P, P, P, P,
                                      P, P, P, P, P]),
        "step5_decode_step": (i32, [G, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                    P, P, P, P, sz, P]),
        "step5_index_score_topk_noalloc": (i32, [G, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P,
                                                 P, P, P]),
        "step5_index_score_topk_shard": (i32, [G, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P,
                                               P, P, sz, P]),
        "step5_merge_topk": (i32, [G, i32, i32, P, P, P, P, P, P, P]),
        "step5_sparse_attn_shard": (i32, [G, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, sz, P]),
        "step5_attn_combine": (i32, [G, i32, i32, P, P, P, P]),
        "step5_merge_attend_shard": (i32, [G, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P, P, sz, P]),
        "step5_rows_layout_for": (i32, [G, i32, i32, ctypes.POINTER(RowsLayout)]),
        "step5_decode_step_host": (i32, [G, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                         P, sz, P]),
        "step5_workspace_bytes": (sz, [G, i32, i32]),
        "step5_workspace_init": (i32, [P, sz, P]),
        "step5_device_status": (i32, [ctypes.POINTER(ctypes.c_uint32), P]),
        "step5_set_select_path": (i32, [i32]),
        "step5_set_wait_polls": (ctypes.c_uint32, [ctypes.c_uint32]),
        "step5_set_attention_path": (i32, [i32]),
        "step5_set_prologue_overlap": (i32, [i32]),
        "step5_set_host_copies": (i32, [i32]),
        "step5_select_path_for": (i32, [G, i32, i32, i32]),
        "step5_status_string": (ctypes.c_char_p, [i32]),
        "step5_convert_bf16_to_e4m3": (i32, [P, P, i64, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libstep5sa must be on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libstep5sa must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise Step5Error(fn, status)


def step5_status_string(status: int) -> str:
    return load().step5_status_string(status).decode()


def step5_set_select_path(mode: int) -> int:
    """0 = automatic, 1 = one block per (row, group), 2 = histogram split path, 3 =
    tensor-core scoring then one selecting block per (row, group)."""
    return load().step5_set_select_path(mode)


def step5_set_attention_path(mode: int) -> int:
    """Step (4) without a split: 0 = automatic, 1 = warp-level MMA kernel, 2 = tcgen05
    kernel; returns the previous value."""
    return load().step5_set_attention_path(mode)


def step5_set_wait_polls(polls: int) -> int:
    """Poll limit of the split selection path's waits on other blocks (0 = default);
    returns the previous limit."""
    return int(load().step5_set_wait_polls(polls))


def step5_set_prologue_overlap(enable: int) -> int:
    """1 = the scoring kernel reads its non-summary inputs before waiting for the launch
    before it (which must not write them); 0 = every read waits.  Returns the previous."""
    return load().step5_set_prologue_overlap(enable)


def step5_set_host_copies(always: int) -> int:
    """1: step5_decode_step_host always copies its host buffers; 0 (default): in place
    when they are device-addressable page-locked memory.  Returns the previous value."""
    return load().step5_set_host_copies(int(always))


def step5_select_path_for(geom, N: int, r_cap: int, B: int = None) -> int:
    """1 (fused), 2 (split) or 3 (tensor-core scoring, then selection) for N rows of B
    sequences (default: one row per sequence) and r_cap."""
    return load().step5_select_path_for(ctypes.byref(Geometry.of(geom)), N, N if B is None else B, r_cap)


def step5_workspace_bytes(geom, N: int, r_cap: int) -> int:
    return load().step5_workspace_bytes(ctypes.byref(Geometry.of(geom)), N, r_cap)


def step5_workspace_init(workspace: torch.Tensor, stream=None):
    _check("step5_workspace_init", load().step5_workspace_init(
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def step5_device_status(stream=None) -> int:
    """Reads and clears the device status word (synchronises the stream)."""
    v = ctypes.c_uint32(0)
    st = load().step5_device_status(ctypes.byref(v), _stream(stream))
    if st not in (0, 5):
        _check("step5_device_status", st)
    return v.value


def step5_convert_bf16_to_e4m3(x: torch.Tensor, out: torch.Tensor, stream=None):
    assert x.dtype == torch.bfloat16 and out.dtype == torch.uint8 and out.numel() == x.numel()
    _check("step5_convert_bf16_to_e4m3", load().step5_convert_bf16_to_e4m3(
        _ptr(x), _ptr(out), x.numel(), _stream(stream)))


def step5_region_summarize(geom, idx_k, idx_z, cos, sin, region_begin, region_end,
                           summaries, summaries_f32=None, max_regions_per_seq=None, stream=None):
    """idx_k/idx_z [B][G][t_cap][64] bf16, cos/sin [t_cap][rope/2] bf16 (or None),
    region_begin/end [B] int32, summaries [B][G][r_cap][64] uint8 (written)."""
    B, G, t_cap, _ = idx_k.shape
    r_cap = summaries.shape[2]
    if max_regions_per_seq is None:
        max_regions_per_seq = r_cap
    _check("step5_region_summarize", load().step5_region_summarize(
        ctypes.byref(Geometry.of(geom)), B, t_cap, r_cap, int(max_regions_per_seq),
        _ptr(idx_k), _ptr(idx_z), _ptr(cos), _ptr(sin), _ptr(region_begin), _ptr(region_end),
        _ptr(summaries), _ptr(summaries_f32), _stream(stream)))


def step5_index_score_topk(geom, idx_q, w, row_seq, row_pos, cos, sin, summaries, sel_ids,
                           sel_count, workspace, t_cap, scores=None, sel_scores=None, stream=None):
    """idx_q [N][idx_heads][64] bf16, w [N][idx_heads] fp32, row_seq/row_pos [N] int32,
    summaries [B][G][r_cap][64] uint8; writes sel_ids [N][G][top_k], sel_count [N][G]."""
    N = idx_q.shape[0]
    B, _, r_cap, _ = summaries.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("step5_index_score_topk", load().step5_index_score_topk(
        ctypes.byref(Geometry.of(geom)), N, B, int(t_cap), r_cap, _ptr(idx_q), _ptr(w),
        _ptr(row_seq), _ptr(row_pos), _ptr(cos), _ptr(sin), _ptr(summaries), _ptr(sel_ids),
        _ptr(sel_count), _ptr(scores), _ptr(sel_scores), _ptr(workspace), ws_bytes,
        _stream(stream)))


def step5_index_score_topk_noalloc(geom, idx_q, w, row_seq, row_pos, cos, sin, summaries, sel_ids,
                                   sel_count, t_cap, scores=None, sel_scores=None, stream=None):
    """step5_index_score_topk with the library's fixed static scratch (about 6.1 MiB: 4 MiB
    for this call's own scratch after the ~2.1 MiB any workspace keeps for step (4))
    instead of a caller workspace, for callers that cannot allocate device memory (see
    the header for the size limit and the sharing rules)."""
    N = idx_q.shape[0]
    B, _, r_cap, _ = summaries.shape
    _check("step5_index_score_topk_noalloc", load().step5_index_score_topk_noalloc(
        ctypes.byref(Geometry.of(geom)), N, B, int(t_cap), r_cap, _ptr(idx_q), _ptr(w),
        _ptr(row_seq), _ptr(row_pos), _ptr(cos), _ptr(sin), _ptr(summaries), _ptr(sel_ids),
        _ptr(sel_count), _ptr(scores), _ptr(sel_scores), _stream(stream)))


def step5_indexer_front(geom, q_pre, k_pre, z_pre, q_norm_w, k_norm_w, k_norm_b, eps, row_seq, row_pos,
                        cos, sin, idx_q_out, idx_k, idx_z, summaries, stream=None):
    """The indexer's decode front end: q RMSNorm (1 + w) into idx_q_out, k LayerNorm and z
    written at each row's position of the caches, and the summary of a region the row's
    token completes (see the header)."""
    N = q_pre.shape[0]
    B, _, t_cap, _ = idx_k.shape
    r_cap = summaries.shape[2]
    _check("step5_indexer_front", load().step5_indexer_front(
        ctypes.byref(Geometry.of(geom)), N, B, t_cap, r_cap, _ptr(q_pre), _ptr(k_pre), _ptr(z_pre),
        _ptr(q_norm_w), _ptr(k_norm_w), _ptr(k_norm_b), float(eps), _ptr(row_seq), _ptr(row_pos),
        _ptr(cos), _ptr(sin), _ptr(idx_q_out), _ptr(idx_k), _ptr(idx_z), _ptr(summaries), _stream(stream)))


def step5_sparse_attn_gated(geom, q, k_cache, v_cache, row_seq, row_pos, sel_ids, sel_count, gate,
                            out, workspace, stream=None):
    """step5_sparse_attn followed by the per-head sigmoid output gate: gate [N][Hq] bf16
    logits; every dim of head h of row n is scaled by sigmoid(gate[n][h]) before the
    output's rounding."""
    N = q.shape[0]
    B, _, t_cap, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("step5_sparse_attn_gated", load().step5_sparse_attn_gated(
        ctypes.byref(Geometry.of(geom)), N, B, t_cap, _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(row_seq), _ptr(row_pos), _ptr(sel_ids), _ptr(sel_count), _ptr(gate), _ptr(out),
        _ptr(workspace), ws_bytes, _stream(stream)))


def step5_sparse_attn(geom, q, k_cache, v_cache, row_seq, row_pos, sel_ids, sel_count, out,
                      workspace, stream=None):
    """q [N][Hq][128] bf16, k/v cache [B][G][t_cap][128] bf16 -> out [N][Hq][128] bf16."""
    N = q.shape[0]
    B, _, t_cap, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("step5_sparse_attn", load().step5_sparse_attn(
        ctypes.byref(Geometry.of(geom)), N, B, t_cap, _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(row_seq), _ptr(row_pos), _ptr(sel_ids), _ptr(sel_count), _ptr(out), _ptr(workspace),
        ws_bytes, _stream(stream)))


def step5_index_score_topk_shard(geom, idx_q, w, row_seq, row_pos, cos, sin, summaries, region_lo,
                                 sel_ids, sel_count, sel_scores, workspace, t_cap, stream=None):
    """Scoring and top-k of one sequence shard: summaries [B][G][r_cap_local][64] hold
    regions region_lo .. region_lo + r_cap_local - 1; writes the shard's pick with the
    rows' region ids, sel_scores required."""
    N = idx_q.shape[0]
    B, _, r_cap, _ = summaries.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("step5_index_score_topk_shard", load().step5_index_score_topk_shard(
        ctypes.byref(Geometry.of(geom)), N, B, int(t_cap), r_cap, int(region_lo), _ptr(idx_q), _ptr(w),
        _ptr(row_seq), _ptr(row_pos), _ptr(cos), _ptr(sin), _ptr(summaries), _ptr(sel_ids),
        _ptr(sel_count), _ptr(sel_scores), _ptr(workspace), ws_bytes, _stream(stream)))


def step5_merge_topk(geom, shard_ids, shard_scores, shard_counts, sel_ids, sel_count, sel_scores=None,
                     stream=None):
    """The rows' pick from S shards' picks: shard_ids / shard_scores [S][N][G][top_k],
    shard_counts [S][N][G] -> sel_ids [N][G][top_k], sel_count [N][G] (+ sel_scores)."""
    S, N = shard_ids.shape[0], shard_ids.shape[1]
    _check("step5_merge_topk", load().step5_merge_topk(
        ctypes.byref(Geometry.of(geom)), S, N, _ptr(shard_ids), _ptr(shard_scores), _ptr(shard_counts),
        _ptr(sel_ids), _ptr(sel_count), _ptr(sel_scores), _stream(stream)))


def step5_sparse_attn_shard(geom, q, k_cache, v_cache, token_lo, row_seq, row_pos, sel_ids, sel_count,
                            states, workspace, stream=None):
    """Attention of one sequence shard: k/v cache [B][G][t_cap_local][128] hold tokens
    token_lo .. token_lo + t_cap_local - 1; writes states [N][Hq][130] fp32 (m, l, o)."""
    N = q.shape[0]
    B, _, t_cap, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("step5_sparse_attn_shard", load().step5_sparse_attn_shard(
        ctypes.byref(Geometry.of(geom)), N, B, t_cap, int(token_lo), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(row_seq), _ptr(row_pos), _ptr(sel_ids), _ptr(sel_count), _ptr(states), _ptr(workspace),
        ws_bytes, _stream(stream)))


def step5_merge_attend_shard(geom, shard_ids, shard_scores, shard_counts, q, k_cache, v_cache, token_lo, row_seq,
                             row_pos, sel_ids, sel_count, states, workspace, stream=None):
    """The merge of S shards' picks [S][N][G][K] into sel_ids/sel_count, then this shard's
    attention states [N][Hq][130], in one call (see the header)."""
    S, N = shard_ids.shape[0], shard_ids.shape[1]
    B, _, t_cap, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("step5_merge_attend_shard", load().step5_merge_attend_shard(
        ctypes.byref(Geometry.of(geom)), S, N, B, t_cap, int(token_lo), _ptr(shard_ids), _ptr(shard_scores),
        _ptr(shard_counts), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(row_seq), _ptr(row_pos), _ptr(sel_ids),
        _ptr(sel_count), _ptr(states), _ptr(workspace), ws_bytes, _stream(stream)))


def step5_attn_combine(geom, states, out, gate=None, stream=None):
    """The output from S shards' states [S][N][Hq][130] -> out [N][Hq][128] bf16 (with the
    per-head sigmoid gate [N][Hq] when given)."""
    S, N = states.shape[0], states.shape[1]
    _check("step5_attn_combine", load().step5_attn_combine(
        ctypes.byref(Geometry.of(geom)), S, N, _ptr(states), _ptr(gate), _ptr(out), _stream(stream)))


def step5_decode_step(geom, t: dict, ws, sel_ids, sel_count, out, max_regions_per_seq, stream=None):
    """The whole step in one C-ABI call (summaries of [sum_begin, sum_end), score +
    select, attention), over the tensors of ``t`` (keys as produced by the synthetic
    workload module).  Same results as the three calls."""
    B, G, t_cap, _ = t["idx_k"].shape
    r_cap = t["summaries"].shape[2]
    N = t["idx_q"].shape[0]
    ws_t = None if ws is None else (ws.tensor if isinstance(ws, Workspace) else ws)
    ws_bytes = 0 if ws_t is None else ws_t.numel() * ws_t.element_size()
    _check("step5_decode_step", load().step5_decode_step(
        ctypes.byref(Geometry.of(geom)), N, B, t_cap, r_cap, int(max_regions_per_seq),
        _ptr(t["idx_k"]), _ptr(t["idx_z"]), _ptr(t["cos"]), _ptr(t["sin"]), _ptr(t["sum_begin"]),
        _ptr(t["sum_end"]), _ptr(t["summaries"]), _ptr(t["idx_q"]), _ptr(t["w"]), _ptr(t["row_seq"]),
        _ptr(t["row_pos"]), _ptr(t["q"]), _ptr(t["k_cache"]), _ptr(t["v_cache"]), _ptr(sel_ids),
        _ptr(sel_count), _ptr(out), _ptr(ws_t), ws_bytes, _stream(stream)))


class RowsLayout(ctypes.Structure):
    """Byte offsets of a step's per-row inputs packed in one buffer (step5_rows_layout_for)."""
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("q", "idx_q", "w", "row_seq", "row_pos", "region_begin", "region_end", "total")]


def step5_rows_layout_for(geom, N: int, B: int) -> RowsLayout:
    lay = RowsLayout()
    _check("step5_rows_layout_for", load().step5_rows_layout_for(ctypes.byref(Geometry.of(geom)), N, B,
                                                                 ctypes.byref(lay)))
    return lay


class HostRows:
    """A decode step's per-row inputs packed in one page-locked host buffer (filled by the
    caller through ``view``) and its device copy, plus the page-locked output; the buffers
    that step5_decode_step_host takes."""

    def __init__(self, geom, N: int, B: int, device="cuda"):
        g = Geometry.of(geom)
        self.N, self.B = N, B
        self.layout = step5_rows_layout_for(geom, N, B)
        self.host = torch.zeros(self.layout.total, dtype=torch.uint8, pin_memory=True)
        self.dev = torch.zeros(self.layout.total, dtype=torch.uint8, device=device)
        self.out_host = torch.zeros((N, g.num_q_heads, g.head_dim), dtype=torch.bfloat16, pin_memory=True)
        self.out_dev = torch.zeros((N, g.num_q_heads, g.head_dim), dtype=torch.bfloat16, device=device)
        self._shapes = {"q": ((N, g.num_q_heads, g.head_dim), torch.bfloat16),
                        "idx_q": ((N, g.idx_heads, g.idx_dim), torch.bfloat16),
                        "w": ((N, g.idx_heads), torch.float32), "row_seq": ((N,), torch.int32),
                        "row_pos": ((N,), torch.int32), "region_begin": ((B,), torch.int32),
                        "region_end": ((B,), torch.int32)}

    def view(self, name: str, on_device: bool = False) -> torch.Tensor:
        """The array ``name`` of the packed buffer (host, or its device copy)."""
        shape, dtype = self._shapes[name]
        off = getattr(self.layout, name)
        nbytes = math.prod(shape) * torch.tensor([], dtype=dtype).element_size()
        buf = self.dev if on_device else self.host
        return buf[off:off + nbytes].view(dtype).view(shape)

    @property
    def h2d_bytes(self) -> int:
        return int(self.layout.total)

    @property
    def d2h_bytes(self) -> int:
        return self.out_host.numel() * self.out_host.element_size()


def _hptr(t: torch.Tensor):
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("host buffers passed to libstep5sa must be contiguous CPU tensors")
    return ctypes.c_void_p(t.data_ptr())


def step5_decode_step_host(geom, t: dict, ws, rows: HostRows, sel_ids, sel_count, max_regions_per_seq,
                           stream=None):
    """The whole step from host inputs to host output in one C-ABI call: the step runs
    over rows.host's arrays (in place when the device can address them, else copied to
    rows.dev) and the device caches, summaries and tables of ``t``; the output lands in
    rows.out_host (valid after the stream reaches the end of the call's work)."""
    B, G, t_cap, _ = t["idx_k"].shape
    r_cap = t["summaries"].shape[2]
    ws_t = None if ws is None else (ws.tensor if isinstance(ws, Workspace) else ws)
    ws_bytes = 0 if ws_t is None else ws_t.numel() * ws_t.element_size()
    _check("step5_decode_step_host", load().step5_decode_step_host(
        ctypes.byref(Geometry.of(geom)), rows.N, B, t_cap, r_cap, int(max_regions_per_seq),
        _ptr(t["idx_k"]), _ptr(t["idx_z"]), _ptr(t["cos"]), _ptr(t["sin"]), _ptr(t["summaries"]),
        _ptr(t["k_cache"]), _ptr(t["v_cache"]), _hptr(rows.host), _ptr(rows.dev), _hptr(rows.out_host),
        _ptr(rows.out_dev), _ptr(sel_ids), _ptr(sel_count), _ptr(ws_t), ws_bytes, _stream(stream)))


@dataclass
class Workspace:
    """Device workspace for N rows and r_cap summary slots, zeroed once on creation."""
    tensor: torch.Tensor

    @classmethod
    def create(cls, geom, N: int, r_cap: int, device="cuda") -> "Workspace":
        nbytes = step5_workspace_bytes(geom, N, r_cap)
        if nbytes == 0:
            raise Step5Error("step5_workspace_bytes", 2, "unsupported geometry")
        t = torch.empty(nbytes, dtype=torch.uint8, device=device)
        step5_workspace_init(t)
        return cls(t)


def decode_step(geom, t: dict, ws: Workspace, sel_ids, sel_count, out, max_regions_per_seq,
                summarize: bool = True, stream=None):
    """One pass of the whole path over the tensors of ``t`` (keys as produced by the
    synthetic workload module): summarise [sum_begin, sum_end), score + select, attend."""
    if summarize:
        step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["sum_begin"],
                               t["sum_end"], t["summaries"],
                               max_regions_per_seq=max_regions_per_seq, stream=stream)
    # the launch just before the scoring call is the summary kernel (or, without it, the
    # previous step's attention), which writes none of the scoring inputs but summaries
    prev = step5_set_prologue_overlap(1 if summarize else 0)
    try:
        step5_index_score_topk(geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], t["cos"],
                               t["sin"], t["summaries"], sel_ids, sel_count, ws.tensor,
                               t_cap=t["idx_k"].shape[2], stream=stream)
    finally:
        step5_set_prologue_overlap(prev)
    step5_sparse_attn(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"],
                      sel_ids, sel_count, out, ws.tensor, stream=stream)
