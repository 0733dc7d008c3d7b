"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This module holds none of the method's arithmetic: it only draws random numbers and
lays them out in the shapes the Step-5 sparse-indexer layer uses.

Generator.  Every value is a pure function of (seed, stream, flat index): a
splitmix64 hash of the counter, done with 64-bit integer tensor ops, so a tensor drawn
on the GPU is bit-identical to the same tensor drawn on the CPU, and any single element
can be drawn on its own (the 1M-token caches are filled on the device; the oracle
draws only the rows it reads).
  * normal: the sum of twelve 16-bit uniforms, centred and divided by 65536 (the
    Irwin-Hall approximation of N(0,1), variance 1 - 2^-32, range +-6), exact in fp32,
    then rounded to bf16 by the tensor library's fp32 -> bf16 cast.
  * uniform: 24 random bits times 2^-24, exact in fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

MASK64 = (1 << 64) - 1


def _s64(u: int) -> int:
    """An unsigned 64-bit constant as the signed int64 torch stores."""
    u &= MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_M1 = _s64(0xBF58476D1CE4E5B9)
_M2 = _s64(0x94D049BB133111EB)


def _lsr(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor."""
    return torch.bitwise_and(torch.bitwise_right_shift(x, k), (1 << (64 - k)) - 1)


def _mix(x: torch.Tensor) -> torch.Tensor:
    x = x + _GOLDEN
    x = torch.bitwise_xor(x, _lsr(x, 30)) * _M1
    x = torch.bitwise_xor(x, _lsr(x, 27)) * _M2
    return torch.bitwise_xor(x, _lsr(x, 31))


def _key(seed: int, stream: int) -> int:
    """64-bit key of one (seed, stream) pair, computed with Python integers."""
    def mix(v):
        v = (v + 0x9E3779B97F4A7C15) & MASK64
        v = ((v ^ (v >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        v = ((v ^ (v >> 27)) * 0x94D049BB133111EB) & MASK64
        return v ^ (v >> 31)
    return _s64(mix(mix(seed) ^ (stream * 0xD1B54A32D192ED03)))


def hash64(idx: torch.Tensor, seed: int, stream: int) -> torch.Tensor:
    """splitmix64 of (key(seed, stream) xor counter) for an int64 counter tensor."""
    return _mix(torch.bitwise_xor(idx, _key(seed, stream)))


def normal_at(idx: torch.Tensor, seed: int, stream: int) -> torch.Tensor:
    """fp32 approximately N(0,1) values at int64 flat indices ``idx``."""
    total = torch.zeros(idx.shape, dtype=torch.int64, device=idx.device)
    base = idx * 3
    for j in range(3):
        h = hash64(base + j, seed, stream)
        for s in (0, 16, 32, 48):
            total += torch.bitwise_and(_lsr(h, s), 0xFFFF)
    # 12 uniforms on {0..65535}: mean 12*32767.5 = 393210, sd = sqrt(65536^2 - 1)
    return (total - 393210).to(torch.float32) * (1.0 / 65536.0)


def uniform_at(idx: torch.Tensor, seed: int, stream: int) -> torch.Tensor:
    """fp32 U[0,1) values at int64 flat indices ``idx`` (multiples of 2^-24)."""
    h = hash64(idx, seed, stream)
    return _lsr(h, 40).to(torch.float32) * (1.0 / 16777216.0)


def _chunked(numel: int, device, fn, out: torch.Tensor, chunk: int = 1 << 25):
    flat = out.view(-1)
    for start in range(0, numel, chunk):
        stop = min(numel, start + chunk)
        idx = torch.arange(start, stop, dtype=torch.int64, device=device)
        flat[start:stop] = fn(idx)
    return out


def normal_bf16(shape, seed: int, stream: int, scale: float = 1.0, device="cpu") -> torch.Tensor:
    """bf16 tensor of bf16(scale * N(0,1)); ``scale`` must be a power of two (exact)."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    numel = out.numel()
    _chunked(numel, device, lambda i: (normal_at(i, seed, stream) * scale).to(torch.bfloat16), out)
    return out


def normal_bf16_rows(shape, rows: np.ndarray, seed: int, stream: int, scale: float = 1.0) -> np.ndarray:
    """uint16 codes of the same tensor as ``normal_bf16(shape, ...)`` but only at the
    given rows of its flattened leading dims (shape[:-1]); the rest stays zero.
    Returns a lazily-zeroed numpy array of the full shape."""
    out = np.zeros(shape, dtype=np.uint16)
    width = shape[-1]
    rows = np.unique(np.asarray(rows, dtype=np.int64))
    if rows.size == 0:
        return out
    idx = torch.from_numpy(rows)[:, None] * width + torch.arange(width, dtype=torch.int64)[None, :]
    vals = (normal_at(idx, seed, stream) * scale).to(torch.bfloat16)
    flat = out.reshape(-1, width)
    flat[rows] = vals.view(torch.int16).numpy().view(np.uint16)
    return out


def uniform_f32(shape, seed: int, stream: int, device="cpu") -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.float32, device=device)
    _chunked(out.numel(), device, lambda i: uniform_at(i, seed, stream), out)
    return out


def randint_at(n: int, lo: int, hi: int, seed: int, stream: int) -> np.ndarray:
    """n integers uniform on [lo, hi] (inclusive), drawn on the CPU."""
    idx = torch.arange(n, dtype=torch.int64)
    h = _lsr(hash64(idx, seed, stream), 11).numpy().astype(np.uint64)
    span = np.uint64(hi - lo + 1)
    return (lo + (h % span).astype(np.int64)).astype(np.int64)


def rope_tables(t_cap: int, rope_dims: int, base: float = 10000.0):
    """bf16 cos/sin tables [t_cap][rope_dims/2] for NEOX rotation: angle of position
    p, pair i = p * base^(-2i/rope_dims), evaluated in fp64 and cast to bf16."""
    half = rope_dims // 2
    inv = base ** (-(np.arange(half, dtype=np.float64) * 2.0) / rope_dims)
    ang = np.arange(t_cap, dtype=np.float64)[:, None] * inv[None, :]
    cos = torch.from_numpy(np.cos(ang)).to(torch.float32).to(torch.bfloat16)
    sin = torch.from_numpy(np.sin(ang)).to(torch.float32).to(torch.bfloat16)
    return cos.contiguous(), sin.contiguous()


def codes16(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (copied to the host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def codes8(t: torch.Tensor) -> np.ndarray:
    """uint8 codes of an e4m3 / uint8 tensor (copied to the host)."""
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


# ----------------------------------------------------------------------------------
# Geometry and workloads
# ----------------------------------------------------------------------------------

@dataclass(frozen=True)
class Geometry:
    """Step-5 full-attention layer geometry (per layer, one GPU)."""
    num_q_heads: int = 32
    num_kv_groups: int = 4
    head_dim: int = 128
    idx_heads: int = 16
    idx_dim: int = 64
    rope_dims: int = 32
    region_tokens: int = 8
    top_k: int = 512
    softmax_scale: float = 1.0 / math.sqrt(128.0)


# stream ids: one per tensor
S_Q, S_K, S_V, S_IQ, S_IK, S_IZ, S_W, S_POS, S_SUMM, S_TIE_T, S_TIE_S = range(1, 12)


@dataclass
class Workload:
    name: str
    geom: Geometry
    B: int
    N: int
    t_cap: int
    r_cap: int
    row_seq: np.ndarray            # int32 [N]
    row_pos: np.ndarray            # int32 [N]
    sum_begin: np.ndarray          # int32 [B]: regions the step summarises
    sum_end: np.ndarray            # int32 [B]
    pre_begin: np.ndarray          # int32 [B]: regions built by summaries at set-up
    pre_end: np.ndarray            # int32 [B]
    random_summaries: bool         # summaries drawn directly as e4m3 (configs 2, 4)
    idx_q_scale: float = 1.0
    tie_fraction: float = 0.0
    seed: int = 17
    tensors: dict = field(default_factory=dict)

    @property
    def max_span(self) -> int:
        return int(max(1, (self.sum_end - self.sum_begin).max()))


def _align8(x: int) -> int:
    return (x + 7) // 8 * 8


def workload(cfg, seed: int = 17, geom: Optional[Geometry] = None) -> Workload:
    """Shapes and row positions of the five workloads, or of a small case.

    cfg: 0..4, or a dict {"positions": [...], "B": b (rows assigned round-robin)}.
      0: 1 decode row at context 4,608 (576 completed regions).
      1: 16 decode rows, one per sequence, contexts uniform on [16,384, 32,768].
      Configs 0 and 1 build the summaries of their earlier regions at set-up (pre_begin,
      pre_end) and summarise in the step only the region the previous token completed.
      2: 4 decode rows at 131,072 (16,384 regions), e4m3 summaries drawn directly,
         indexer q scaled by 4, 5% of regions per (sequence, group) copied from another
         region (exact score ties).
      3: chunked prefill: 2,048 rows at positions 65,536..67,583 of one sequence; the
         chunk's 256 regions are summarised by the step, the 8,192 before it at set-up.
      4: 1 decode row at 1,048,576 (131,072 regions), e4m3 summaries drawn directly.
    Decode rows sit at position p = context; the step summarises the region that the
    previous token completed (when p is a multiple of 8).
    """
    g = geom or Geometry()
    rt = g.region_tokens
    if isinstance(cfg, dict):
        pos = np.asarray(cfg["positions"], dtype=np.int64)
        B = int(cfg.get("B", len(pos)))
        N = len(pos)
        seq = np.arange(N) % B
        t_cap = _align8(int(pos.max()) + 1)
        r_cap = max(1, t_cap // rt)
        pre_end = np.zeros(B, dtype=np.int64)
        for n in range(N):
            pre_end[seq[n]] = max(pre_end[seq[n]], pos[n] // rt)
        w = Workload(cfg.get("name", "small"), g, B, N, t_cap, r_cap, seq.astype(np.int32),
                     pos.astype(np.int32), np.zeros(B, np.int32), pre_end.astype(np.int32),
                     np.zeros(B, np.int32), np.zeros(B, np.int32), False,
                     idx_q_scale=float(cfg.get("idx_q_scale", 1.0)), seed=seed)
        return w
    if cfg == 0:
        p = 4608
        t_cap = _align8(p + 1)
        R = p // rt
        return Workload("decode_1x4608", g, 1, 1, t_cap, t_cap // rt, np.zeros(1, np.int32),
                        np.array([p], np.int32), np.array([R - 1], np.int32),
                        np.array([R], np.int32), np.zeros(1, np.int32),
                        np.array([R - 1], np.int32), False, seed=seed)
    if cfg == 1:
        pos = randint_at(16, 16384, 32768, seed, S_POS)
        t_cap = _align8(int(pos.max()) + 1)
        R = pos // rt
        # the step summarises the region the previous token completed (p a multiple of 8);
        # every earlier region is summarised at set-up
        done = (pos % rt == 0)
        sb = np.where(done, R - 1, R)
        return Workload("decode_16x16k-32k", g, 16, 16, t_cap, t_cap // rt,
                        np.arange(16, dtype=np.int32), pos.astype(np.int32),
                        sb.astype(np.int32), R.astype(np.int32),
                        np.zeros(16, np.int32), sb.astype(np.int32), False, seed=seed)
    if cfg == 2:
        p = 131072
        t_cap = _align8(p + 1)
        R = p // rt
        return Workload("decode_4x128k", g, 4, 4, t_cap, t_cap // rt,
                        np.arange(4, dtype=np.int32), np.full(4, p, np.int32),
                        np.full(4, R - 1, np.int32), np.full(4, R, np.int32),
                        np.zeros(4, np.int32), np.zeros(4, np.int32), True,
                        idx_q_scale=4.0, tie_fraction=0.05, seed=seed)
    if cfg == 3:
        p0, chunk = 65536, 2048
        t_cap = p0 + chunk
        return Workload("prefill_2048_on_64k", g, 1, chunk, t_cap, t_cap // rt,
                        np.zeros(chunk, np.int32), (p0 + np.arange(chunk)).astype(np.int32),
                        np.array([p0 // rt], np.int32), np.array([(p0 + chunk) // rt], np.int32),
                        np.array([0], np.int32), np.array([p0 // rt], np.int32), False,
                        seed=seed)
    if cfg == 4:
        p = 1 << 20
        t_cap = _align8(p + 1)
        R = p // rt
        return Workload("decode_1x1m", g, 1, 1, t_cap, t_cap // rt, np.zeros(1, np.int32),
                        np.array([p], np.int32), np.array([R - 1], np.int32),
                        np.array([R], np.int32), np.zeros(1, np.int32),
                        np.zeros(1, np.int32), True, seed=seed)
    raise ValueError(f"unknown workload {cfg!r}")


def random_summaries(w: Workload) -> torch.Tensor:
    """uint8 e4m3 summaries [B][G][r_cap][idx_dim] drawn as e4m3(bf16(N(0,1))) on the
    CPU (the tensor library's bf16 -> float8_e4m3fn cast), with ``tie_fraction`` of the
    regions of each (sequence, group) overwritten by a copy of another region."""
    g = w.geom
    shape = (w.B, g.num_kv_groups, w.r_cap, g.idx_dim)
    x = normal_bf16(shape, w.seed, S_SUMM)
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8).clone()
    if w.tie_fraction > 0:
        R = int(w.row_pos.max()) // g.region_tokens
        ntie = int(round(w.tie_fraction * R))
        for b in range(w.B):
            for gg in range(g.num_kv_groups):
                base = (b * g.num_kv_groups + gg) * R
                # targets: the ntie regions with the smallest hash; sources: any region
                order = torch.argsort(hash64(torch.arange(R, dtype=torch.int64) + base,
                                             w.seed, S_TIE_T))
                tgt = order[:ntie]
                src = torch.from_numpy(randint_at(ntie, 0, R - 1, w.seed + base + 1, S_TIE_S))
                src = torch.where(src == tgt, (src + 1) % R, src)
                codes[b, gg, tgt] = codes[b, gg, src]
    return codes


def materialize(w: Workload, device="cpu", with_kv: bool = True) -> dict:
    """All input tensors of a workload on ``device`` (bf16 as torch.bfloat16, e4m3 as
    uint8).  Keys: q, k_cache, v_cache, idx_q, idx_k, idx_z, w, cos, sin, row_seq,
    row_pos, sum_begin, sum_end, pre_begin, pre_end, summaries (random or zeros)."""
    g = w.geom
    G = g.num_kv_groups
    t = {}
    t["q"] = normal_bf16((w.N, g.num_q_heads, g.head_dim), w.seed, S_Q, device=device)
    if with_kv:
        t["k_cache"] = normal_bf16((w.B, G, w.t_cap, g.head_dim), w.seed, S_K, device=device)
        t["v_cache"] = normal_bf16((w.B, G, w.t_cap, g.head_dim), w.seed, S_V, device=device)
    t["idx_q"] = normal_bf16((w.N, g.idx_heads, g.idx_dim), w.seed, S_IQ,
                             scale=w.idx_q_scale, device=device)
    t["idx_k"] = normal_bf16((w.B, G, w.t_cap, g.idx_dim), w.seed, S_IK, device=device)
    t["idx_z"] = normal_bf16((w.B, G, w.t_cap, g.idx_dim), w.seed, S_IZ, device=device)
    t["w"] = uniform_f32((w.N, g.idx_heads), w.seed, S_W, device=device)
    cos, sin = rope_tables(w.t_cap, g.rope_dims)
    t["cos"], t["sin"] = cos.to(device), sin.to(device)
    for name in ("row_seq", "row_pos", "sum_begin", "sum_end", "pre_begin", "pre_end"):
        t[name] = torch.from_numpy(np.ascontiguousarray(getattr(w, name), dtype=np.int32)).to(device)
    if w.random_summaries:
        t["summaries"] = random_summaries(w).to(device)
    else:
        t["summaries"] = torch.zeros((w.B, G, w.r_cap, g.idx_dim), dtype=torch.uint8, device=device)
    return t
