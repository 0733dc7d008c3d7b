"""Benchmark of the Step-5 sparse-indexer attention step on GB300.

A step is one pass of the whole path over one batch of rows: summarise the region the
previous token completed (step 1), score every candidate region and select the top 512
per KV group (steps 2-3), attend over the picks plus the own region (step 4).

Headline workload: one decode row at 1,048,576 tokens (131,072 regions x 4 KV groups,
e4m3 summaries, 2 GiB bf16 K/V); the 4-row 128K workload is reported beside it.  Inputs
are seeded synthetic tensors already resident in HBM; L2 is flushed (a 256 MiB write)
between timed steps, each step timed with CUDA events on the launching stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

``--impl reference`` times the CPU oracle (the reference implementation of this path) on
the host cores, on a bounded sample of the same workload, and prints the same line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn decode rows/sec at 128K and 1M ctx; achieved HBM GB/s vs peak"
UNIT = "rows/s"
FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20  # GB300's L2 (the device's own figure is used when torch reports it)
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "score_select_decode_1x1m.md")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=4, choices=[0, 1, 2, 3, 4],
                    help="workload: 4 (headline, 1 row at 1M), 2 (4 rows at 128K), 0, 1, 3")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rotate", action="store_true",
                    help="skip the rotated-inputs measurement (it holds up to 16 copies of the inputs)")
    ap.add_argument("--shards", type=int, default=4,
                    help="sequence shards of the headline row timed beside the step (0: none)")
    return ap.parse_args()


# --------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor throughput (TFLOP/s, burst) and where it comes from."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return float(json.load(open(path))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def attention_flops(w, geom):
    """Tensor FLOPs of step (4): per row and KV group, S = Q K^T and O = P V over the
    picked regions' tokens plus the own region's, for the group's query heads."""
    hq_g = geom.num_q_heads // geom.num_kv_groups
    f = 0
    for n in range(w.N):
        p = int(w.row_pos[n])
        R = p // 8
        keys = min(R, geom.top_k) * 8 + (p - 8 * R + 1)
        f += geom.num_kv_groups * hq_g * keys * geom.head_dim * 2 * 2
    return f


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_sha():
    """sha256 (first 16 hex digits) of the dominant kernel's sources with comments and
    blank lines removed, so that only a change of code retires a recorded profile."""
    src = os.path.join(ROOT, "block_sparse_attention_step5_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("score_select.cu", "common.cuh", "kernels.cuh"):
        text = open(os.path.join(src, name)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(line.rstrip() for line in text.split("\n") if line.strip()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if
    it was taken on the current source of that kernel (else None)."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    text = open(PROFILE_SUMMARY).read()
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != kernel_source_sha():
        return None
    return float(m_tr.group(1))


def step_bytes(w, geom):
    """Algorithmic bytes one step must move: summaries read by scoring, K/V of every
    picked and own-region token, the rows' q / indexer q / w, the output, and step 1's
    k/z/cos/sin of the summarised regions plus their summaries."""
    G = geom.num_kv_groups
    total = 0
    score = 0
    for n in range(w.N):
        p = int(w.row_pos[n])
        R = p // 8
        k = min(R, geom.top_k)
        own = p - 8 * R + 1
        score += R * G * geom.idx_dim
        total += G * (k * 8 + own) * geom.head_dim * 2 * 2
        total += geom.num_q_heads * geom.head_dim * 2 * 2          # q in, out
        total += geom.idx_heads * geom.idx_dim * 2 + geom.idx_heads * 4
    span = int((w.sum_end - w.sum_begin).sum())
    summ = span * G * (8 * geom.idx_dim * 2 * 2 + geom.idx_dim) + span * 8 * geom.rope_dims * 2
    score_call = score + w.N * (geom.idx_heads * geom.idx_dim * 2 + geom.idx_heads * 4) \
        + w.N * G * (geom.top_k * 4 + 4)
    return total + score + summ, score_call


# --------------------------------------------------------------------------- ranks

def max_over_ranks(values, dist, device):
    """Element-wise maximum of a list of floats over all ranks (the slowest rank sets
    the job's time); the values themselves without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    tt = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return [float(v) for v in tt.tolist()]


def whole_job_rate(rows_per_rank, world, ms):
    """Rows per second of the whole job: every rank's rows over the slowest rank's time."""
    return rows_per_rank * world / (ms / 1e3)


# --------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch

    import block_sparse_attention_step5_gb300 as s5
    import synthetic as S

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    s5.build()
    s5.load()
    geom = s5.STEP5_GEOMETRY
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def measure(cfg, steps, warmup, clocks=False, n_shards=0, bulk=False, rotate=False):
        w = S.workload(cfg, seed=17)
        t = S.materialize(w, device=dev)
        N, G = w.N, geom.num_kv_groups
        pre_span = int((w.pre_end - w.pre_begin).max())
        if pre_span > 0:  # summaries of the regions completed before the step (set-up)
            s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["pre_begin"],
                                      t["pre_end"], t["summaries"], max_regions_per_seq=pre_span)
            torch.cuda.synchronize()
        ws = s5.Workspace.create(geom, N, w.r_cap, device=dev)
        sel_ids = torch.empty((N, G, geom.top_k), dtype=torch.int32, device=dev)
        sel_count = torch.empty((N, G), dtype=torch.int32, device=dev)
        out = torch.empty((N, geom.num_q_heads, geom.head_dim), dtype=torch.bfloat16, device=dev)
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream()
        span = w.max_span
        path = s5.step5_select_path_for(geom, N, w.r_cap, w.B)
        launches_per_step = (1 if span > 0 else 0) + 1 + 1  # summarize, score + select, attention

        def call_sum():
            s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], t["sum_begin"],
                                      t["sum_end"], t["summaries"], max_regions_per_seq=span)

        def call_score():
            s5.step5_index_score_topk(geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], t["cos"],
                                      t["sin"], t["summaries"], sel_ids, sel_count, ws.tensor, t_cap=w.t_cap)

        def call_attn():
            s5.step5_sparse_attn(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"],
                                 sel_ids, sel_count, out, ws.tensor)

        # the per-head sigmoid output gate after attention (timed beside the step only)
        gate = (torch.randn((N, geom.num_q_heads), generator=torch.Generator().manual_seed(61)) * 3).to(
            torch.bfloat16).to(dev)

        out_gated = torch.empty_like(out)

        def call_attn_gated():
            s5.step5_sparse_attn_gated(geom, t["q"], t["k_cache"], t["v_cache"], t["row_seq"], t["row_pos"],
                                       sel_ids, sel_count, gate, out_gated, ws.tensor)

        # the indexer's decode front end (q/k norms, the row token's k/z write, a completed
        # region's summary), timed beside the step only: it writes token p of the caches
        # and, at p % 8 == 7, the summary of the row's own region, neither of which the
        # step reads
        fg = torch.Generator().manual_seed(71)
        front_in = [(torch.randn(shape, generator=fg) * sc + sh).to(torch.bfloat16).to(dev) for shape, sc, sh in
                    (((N, geom.idx_heads, 64), 2.0, 0.0), ((N, G, 64), 1.5, 0.3), ((N, G, 64), 1.0, 0.0),
                     ((64,), 0.1, 0.0), ((64,), 0.1, 1.0), ((64,), 0.1, 0.0))]
        q_front = torch.empty_like(front_in[0])

        def call_front():
            s5.step5_indexer_front(geom, *front_in, 1e-6, t["row_seq"], t["row_pos"], t["cos"], t["sin"], q_front,
                                   t["idx_k"], t["idx_z"], t["summaries"])

        def step():
            # the whole step in one C-ABI call (summaries, score + select, attention)
            s5.step5_decode_step(geom, t, ws, sel_ids, sel_count, out, max_regions_per_seq=span)

        # eager warm-up (sets kernel attributes, TMA descriptors), then the step and each
        # call captured as CUDA graphs: a replay issues the whole step at once, so the
        # device time is not bounded by the host's launch rate
        for _ in range(warmup):
            flush.zero_()
            step()
        torch.cuda.synchronize()
        assert s5.step5_device_status() == 0

        def capture(fn):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                fn()
            return g

        g_step = capture(step)
        for _ in range(warmup):
            flush.zero_()
            g_step.replay()
        torch.cuda.synchronize()
        assert s5.step5_device_status() == 0

        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        sampler = ClockSampler(local_rank) if clocks else None
        if sampler:
            sampler.__enter__()
        barrier()
        wall0 = time.perf_counter()
        for i in range(steps):
            flush.zero_()
            evs[i][0].record(stream)
            g_step.replay()
            evs[i][1].record(stream)
        barrier()
        wall = time.perf_counter() - wall0
        if sampler:
            sampler.__exit__(None, None, None)
        per_step = np.array([e[0].elapsed_time(e[1]) for e in evs])
        assert s5.step5_device_status() == 0
        ms = max_over_ranks([float(per_step.mean())], dist, dev)[0]

        # The same step with inputs larger than L2 instead of a flush: the graph replayed
        # round robin over `copies` independent copies of every input, so that the data a
        # step reads was last touched (copies - 1) steps earlier, behind more than twice
        # the L2 of other data, while the kernels' code stays in L2 as it does in a decode
        # loop.  (The flush also evicts the code, and the step then fetches each phase's
        # instructions from DRAM.)
        rotated = None
        if rotate:
            touched = max(1, step_bytes(w, geom)[0])
            l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_BYTES)
            copies = int(min(16, max(4, -(-2 * l2 // touched) + 1)))
            per_copy = sum(x.numel() * x.element_size() for x in t.values() if torch.is_tensor(x))
            free = torch.cuda.mem_get_info(dev)[0]
            if per_copy * (copies - 1) < 0.5 * free:
                sets = [t] + [{k: (x.clone() if torch.is_tensor(x) else x) for k, x in t.items()}
                              for _ in range(copies - 1)]

                def step_on(tc):
                    return lambda: s5.step5_decode_step(geom, tc, ws, sel_ids, sel_count, out,
                                                        max_regions_per_seq=span)

                graphs = [capture(step_on(tc)) for tc in sets]
                for _ in range(warmup):
                    for gr in graphs:
                        gr.replay()
                torch.cuda.synchronize()
                evr = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
                barrier()
                for i in range(steps):
                    evr[i][0].record(stream)
                    graphs[i % copies].replay()
                    evr[i][1].record(stream)
                barrier()
                assert s5.step5_device_status() == 0
                rot_ms = max_over_ranks([float(np.mean([e[0].elapsed_time(e[1]) for e in evr]))], dist, dev)[0]
                rotated = dict(ms=rot_ms, copies=copies, bytes_touched_per_step=touched)
                del graphs, sets
                torch.cuda.empty_cache()

        # per-kernel durations: the calls captured in one CUDA graph with timing event
        # nodes between them (the events keep the kernels from overlapping), so the events
        # bracket the kernels alone; without event nodes in graphs, eager calls behind a
        # 1 GiB write that covers their launch
        def time_calls(calls, reps):
            times = np.zeros((reps, len(calls)))
            try:
                evg = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(calls) + 1)]
                g_b = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_b, capture_error_mode="thread_local"):
                    evg[0].record()
                    for j, fn in enumerate(calls):
                        fn()
                        evg[j + 1].record()
                how = "CUDA graph with event nodes between the calls"
                barrier()
                for i in range(reps):
                    flush.zero_()
                    g_b.replay()
                    torch.cuda.synchronize()
                    times[i] = [evg[j].elapsed_time(evg[j + 1]) for j in range(len(calls))]
            except (TypeError, RuntimeError):
                how = "eager calls behind a 1 GiB write"
                hold = torch.empty(4 * FLUSH_BYTES, dtype=torch.uint8, device=dev)
                evb = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(reps)]
                barrier()
                for i in range(reps):
                    hold.zero_()
                    evb[i][0].record(stream)
                    for j, fn in enumerate(calls):
                        fn()
                        evb[i][j + 1].record(stream)
                barrier()
                times = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(len(calls))] for e in evb])
                del hold
            assert s5.step5_device_status() == 0
            return times, how

        steps_b = steps
        calls_b = (call_sum, call_score, call_attn, call_attn_gated, call_front)
        times_b, breakdown_how = time_calls(calls_b, steps_b)
        per_sum, per_score, per_attn, per_gated = times_b[:, 0], times_b[:, 1], times_b[:, 2], times_b[:, 3]
        per_front = times_b[:, 4]
        bytes_step, bytes_score = step_bytes(w, geom)
        res = dict(w=w, ms=ms, ms_min=float(per_step.min()), per_score=float(per_score.mean()),
                   breakdown_how=breakdown_how,
                   per_attn=float(per_attn.mean()), per_sum=float(per_sum.mean()),
                   per_gated=float(per_gated.mean()), per_front=float(per_front.mean()), bytes_step=bytes_step,
                   bytes_score=bytes_score, launches=launches_per_step * steps, path=path, wall=wall,
                   rotated=rotated,
                   clocks=sampler.summary() if sampler else None)

        # sequence shards of the rows (each shard's summaries and K/V a copy of its part,
        # as one GPU of a sharded deployment would hold them): each shard's score + pick,
        # the merge, each shard's attention and the combine, timed call by call on this
        # one GPU (the exchange of picks and states between GPUs is not part of it)
        if n_shards > 1:
            cuts = [w.t_cap // 8 * i // n_shards * 8 for i in range(n_shards)] + [w.t_cap]
            Hq, K = geom.num_q_heads, geom.top_k
            sh_ids = torch.empty((n_shards, N, G, K), dtype=torch.int32, device=dev)
            sh_cnt = torch.empty((n_shards, N, G), dtype=torch.int32, device=dev)
            sh_sc = torch.empty((n_shards, N, G, K), dtype=torch.float32, device=dev)
            sh_states = torch.empty((n_shards, N, Hq, 130), dtype=torch.float32, device=dev)
            m_ids = torch.empty_like(sel_ids)
            m_cnt = torch.empty_like(sel_count)
            out_sh = torch.empty_like(out)
            parts = []
            for i in range(n_shards):
                lo_t, hi_t = cuts[i], cuts[i + 1]
                lo, hi = lo_t // 8, min(hi_t // 8, w.r_cap)
                parts.append(dict(lo=lo, lo_t=lo_t, summ=t["summaries"][:, :, lo:hi].contiguous(),
                                  kc=t["k_cache"][:, :, lo_t:hi_t].contiguous(),
                                  vc=t["v_cache"][:, :, lo_t:hi_t].contiguous(),
                                  ws=s5.Workspace.create(geom, N, hi - lo, device=dev)))

            def shard_score(i):
                d = parts[i]
                return lambda: s5.step5_index_score_topk_shard(
                    geom, t["idx_q"], t["w"], t["row_seq"], t["row_pos"], t["cos"], t["sin"], d["summ"], d["lo"],
                    sh_ids[i], sh_cnt[i], sh_sc[i], d["ws"].tensor, t_cap=w.t_cap)

            def shard_attn(i):
                d = parts[i]
                return lambda: s5.step5_sparse_attn_shard(
                    geom, t["q"], d["kc"], d["vc"], d["lo_t"], t["row_seq"], t["row_pos"], m_ids, m_cnt,
                    sh_states[i], d["ws"].tensor)

            def shard_merge_attn(i):
                d = parts[i]
                return lambda: s5.step5_merge_attend_shard(
                    geom, sh_ids, sh_sc, sh_cnt, t["q"], d["kc"], d["vc"], d["lo_t"], t["row_seq"], t["row_pos"],
                    m_ids, m_cnt, sh_states[i], d["ws"].tensor)

            calls_s = ([shard_score(i) for i in range(n_shards)] +
                       [lambda: s5.step5_merge_topk(geom, sh_ids, sh_sc, sh_cnt, m_ids, m_cnt)] +
                       [shard_attn(i) for i in range(n_shards)] +
                       [lambda: s5.step5_attn_combine(geom, sh_states, out_sh)] +
                       [shard_merge_attn(i) for i in range(n_shards)])
            for _ in range(warmup):
                for fn in calls_s:
                    fn()
            torch.cuda.synchronize()
            assert s5.step5_device_status() == 0
            times_s, _ = time_calls(calls_s, steps_b)
            ts = times_s.mean(axis=0) * 1e3
            sc_us, at_us = ts[:n_shards], ts[n_shards + 1:2 * n_shards + 1]
            comb_us = ts[2 * n_shards + 1]
            ma_us = ts[2 * n_shards + 2:]
            res["shards"] = {
                "shards": n_shards, "tokens_per_shard": cuts[1] - cuts[0],
                "score_select_us": [round(float(x), 2) for x in sc_us],
                "merge_us": round(float(ts[n_shards]), 2),
                "attention_us": [round(float(x), 2) for x in at_us],
                "combine_us": round(float(comb_us), 2),
                "merge_attend_us": [round(float(x), 2) for x in ma_us],
                "per_gpu_critical_path_us": round(float(sc_us.max() + ma_us.max() + comb_us), 2),
                "per_gpu_critical_path_separate_calls_us": round(float(sc_us.max() + ts[n_shards] + at_us.max() +
                                                                       comb_us), 2),
                "picks_equal_whole_row": bool(torch.equal(m_ids, sel_ids) and torch.equal(m_cnt, sel_count)),
                "out_max_abs_diff_vs_whole_row": float((out_sh.float() - out.float()).abs().max()),
                "how": "calls timed one by one on one GPU; critical path = slowest shard's score + slowest "
                       "shard's step5_merge_attend_shard + combine, without the exchanges between GPUs"}
            del parts
            torch.cuda.empty_cache()

        # end to end through the C ABI with host buffers: step5_decode_step_host copies the
        # step's per-row inputs (packed in one page-locked buffer: q, indexer q, weights,
        # rows' sequences and positions, the summarised region ranges) to the device, runs
        # the step and copies the output back to page-locked memory, every step
        rows = s5.HostRows(geom, N, w.B, device=dev)
        for src, name in (("q", "q"), ("idx_q", "idx_q"), ("w", "w"), ("row_seq", "row_seq"),
                          ("row_pos", "row_pos"), ("sum_begin", "region_begin"), ("sum_end", "region_end")):
            rows.view(name).copy_(t[src].cpu())
        h2d, d2h = rows.h2d_bytes, rows.d2h_bytes

        def step_host():
            s5.step5_decode_step_host(geom, t, ws, rows, sel_ids, sel_count, max_regions_per_seq=span)

        for _ in range(warmup):
            step_host()
        torch.cuda.synchronize()
        assert torch.equal(rows.out_host.view(torch.int16), out.cpu().view(torch.int16))
        in_place = not bool(rows.dev.any())  # the device staging buffer stayed unused
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        barrier()
        for i in range(steps):
            flush.zero_()
            ev2[i][0].record(stream)
            step_host()
            ev2[i][1].record(stream)
        barrier()
        e2e_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev2]))
        # the same call captured once in a CUDA graph (copies and kernels) and replayed
        g_host = capture(step_host)
        for _ in range(warmup):
            g_host.replay()
        barrier()
        for i in range(steps):
            flush.zero_()
            ev2[i][0].record(stream)
            g_host.replay()
            ev2[i][1].record(stream)
        barrier()
        e2e_graph_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev2]))
        assert s5.step5_device_status() == 0
        e2e_ms, e2e_graph_ms = max_over_ranks([e2e_ms, e2e_graph_ms], dist, dev)
        res.update(e2e_ms=e2e_ms, e2e_graph_ms=e2e_graph_ms, h2d=h2d, d2h=d2h, in_place=in_place)

        # step (1) in bulk: the summaries of every completed region of every sequence (the
        # set-up pass of a long context, the vectorised form), into a buffer of its own,
        # timed behind an L2 flush
        if bulk:
            R_seq = np.zeros(w.B, np.int64)
            for n in range(N):
                R_seq[int(w.row_seq[n])] = max(R_seq[int(w.row_seq[n])], int(w.row_pos[n]) // 8)
            rb_bulk = torch.zeros(w.B, dtype=torch.int32, device=dev)
            re_bulk = torch.from_numpy(R_seq.astype(np.int32)).to(dev)
            out_bulk = torch.empty_like(t["summaries"])
            span_bulk = int(R_seq.max())

            def call_bulk():
                s5.step5_region_summarize(geom, t["idx_k"], t["idx_z"], t["cos"], t["sin"], rb_bulk, re_bulk,
                                          out_bulk, max_regions_per_seq=span_bulk)

            call_bulk()
            torch.cuda.synchronize()
            evb = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(5)]
            for i in range(5):
                flush.zero_()
                evb[i][0].record(stream)
                call_bulk()
                evb[i][1].record(stream)
            torch.cuda.synchronize()
            assert s5.step5_device_status() == 0
            bulk_us = float(np.mean([e[0].elapsed_time(e[1]) for e in evb])) * 1e3
            nreg = int(R_seq.sum())
            bulk_bytes = nreg * G * (8 * geom.idx_dim * 2 * 2 + geom.idx_dim) + nreg * 8 * geom.rope_dims * 2
            res["bulk"] = dict(regions=nreg, us=bulk_us, bytes=bulk_bytes)
            del out_bulk
        del t, flush
        torch.cuda.empty_cache()
        return res

    peak, peak_kind = peaks()
    head = measure(args.workload, args.steps, args.warmup, clocks=True, n_shards=args.shards, bulk=True,
                   rotate=not args.no_rotate)
    w = head["w"]
    rows = w.N * world
    value = whole_job_rate(w.N, world, head["ms"])
    score_gbs = head["bytes_score"] / (head["per_score"] / 1e3) / 1e9
    if head["path"] == 3:
        # many rows per sequence (prefill chunks): the attention dominates, on the tensor
        # cores; its rows share regions through L2, so per-row bytes exceed DRAM's
        tpeak, tkind = bf16_peak()
        attn_tf = attention_flops(w, geom) / (head["per_attn"] / 1e3) / 1e12
        roofline = {"kernel": "sparse_attn_tc_kernel (step5_sparse_attn, tcgen05 bf16)", "bound": "tensor",
                    "achieved": round(attn_tf, 2), "peak": tpeak, "unit": "TFLOP/s",
                    "frac": round(attn_tf / tpeak, 4), "peak_kind": f"{tkind} dense bf16 (burst)",
                    "algorithmic_flops_per_launch": attention_flops(w, geom), "traffic": None,
                    "note": "the gathers come from L2 (a chunk's rows share their sequence's regions)"}
    else:
        roofline = None
    step_gbs = head["bytes_step"] / (head["ms"] / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(head["ms"], 5), "ms_per_step_min": round(head["ms_min"], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3+bf16 (fp32 accumulate)", "data": "synthetic (seeded)",
        "config": {"workload": w.name, "rows_per_gpu": w.N, "context": int(w.row_pos.max()),
                   "regions_per_group": int(w.row_pos.max()) // 8, "kv_groups": 4, "q_heads": 32,
                   "idx_heads": 16, "top_k": 512, "select_path": {1: "fused", 2: "split", 3: "tensor-core"}[head["path"]],
                   "l2": "flushed between timed steps (256 MiB write, untimed)",
                   "timing": "CUDA events around a CUDA-graph replay of the whole step",
                   "parallelism": f"replicas x{world}"},
        "step_hbm": {"bytes_per_step": head["bytes_step"], "achieved_gbs": round(step_gbs, 1),
                     "peak_gbs": peak, "frac": round(step_gbs / peak, 4), "peak_kind": peak_kind,
                     **({"note": "bytes counted per row; a chunk's rows share regions through L2, so this "
                                 "exceeds what DRAM moves"} if head["path"] == 3 else {})},
        "breakdown_us": {"summarize": round(head["per_sum"] * 1e3, 2),
                         "score_select": round(head["per_score"] * 1e3, 2),
                         "attention": round(head["per_attn"] * 1e3, 2),
                         "attention_gated": round(head["per_gated"] * 1e3, 2),
                         "indexer_front": round(head["per_front"] * 1e3, 2),
                         "how": head["breakdown_how"]},
        "roofline": roofline or {"kernel": {1: "score_fused_kernel (step5_index_score_topk, fused path)",
                                2: "score_select_kernel (step5_index_score_topk, split path)",
                                3: "score_tc_kernel + score_fused_kernel<select> (step5_index_score_topk, "
                                   "tensor-core path)"}[head["path"]],
                     "bound": "hbm", "achieved": round(score_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(score_gbs / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "algorithmic_bytes_per_launch": head["bytes_score"],
                     # the committed capture is of the split kernel on the 1M decode row
                     "traffic": profiled_traffic() if (head["path"] == 2 and w.name == "decode_1x1m") else None},
        "e2e": {"value": round(rows / (head["e2e_ms"] / 1e3), 2), "unit": UNIT,
                "ms_per_step": round(head["e2e_ms"], 5), "h2d_bytes_per_step": head["h2d"],
                "d2h_bytes_per_step": head["d2h"],
                "how": "step5_decode_step_host (one C-ABI call, issued eagerly): the step's per-row inputs in one "
                       "page-locked host buffer, the output into page-locked host memory; " +
                       ("the kernels read and write the host buffers in place (device-addressable page-locked "
                        "memory over NVLink-C2C), no copy operations" if head["in_place"] else
                        "one host-to-device and one device-to-host copy"),
                "graph_value": round(rows / (head["e2e_graph_ms"] / 1e3), 2),
                "graph_ms_per_step": round(head["e2e_graph_ms"], 5)},
        "rotated_inputs": None if head["rotated"] is None else {
            "value": round(rows / (head["rotated"]["ms"] / 1e3), 2), "unit": UNIT,
            "ms_per_step": round(head["rotated"]["ms"], 5), "copies": head["rotated"]["copies"],
            "bytes_touched_per_step": head["rotated"]["bytes_touched_per_step"],
            "how": "no flush: the step's CUDA graph replayed round robin over independent copies of every input, "
                   "so each step's data was last read behind more than twice the L2 of other data (cold), while "
                   "the kernels' code stays in L2 as in a decode loop; the headline value flushes L2, which also "
                   "evicts the code"},
        "gpu_launches": head["launches"],
        "clocks": head["clocks"],
    }
    if "shards" in head:
        line["sharded_decode"] = head["shards"]
    if "bulk" in head:
        bk = head["bulk"]
        bgbs = bk["bytes"] / (bk["us"] / 1e6) / 1e9
        line["summarize_bulk"] = {
            "kernel": "summarize_bulk_kernel (step5_region_summarize over every completed region)",
            "regions_per_group": bk["regions"], "us": round(bk["us"], 2),
            "algorithmic_bytes": bk["bytes"], "achieved_gbs": round(bgbs, 1), "peak_gbs": peak,
            "frac": round(bgbs / peak, 4),
            "bytes_per_region_group": "2,048 k/z in + 64 out, plus 512 of cos/sin per region"}
    if not args.no_secondary:
        sec = measure(2 if args.workload == 4 else 4, max(20, args.steps // 2), args.warmup)
        sgbs = sec["bytes_step"] / (sec["ms"] / 1e3) / 1e9
        line["secondary"] = {"workload": sec["w"].name, "value": round(whole_job_rate(sec["w"].N, world, sec["ms"]), 2),
                             "unit": UNIT, "ms_per_step": round(sec["ms"], 5),
                             "achieved_gbs": round(sgbs, 1), "frac": round(sgbs / peak, 4),
                             "select_path": {1: "fused", 2: "split", 3: "tensor-core"}[sec["path"]],
                             "breakdown_us": {"summarize": round(sec["per_sum"] * 1e3, 2),
                                              "score_select": round(sec["per_score"] * 1e3, 2),
                                              "attention": round(sec["per_attn"] * 1e3, 2),
                                              "attention_gated": round(sec["per_gated"] * 1e3, 2),
                                              "indexer_front": round(sec["per_front"] * 1e3, 2)}}
        line["gpu_launches"] += sec["launches"]
    if rank == 0 and not args.no_cpu_baseline:
        cb = oracle_sample(args.workload, quarter=False)
        line["cpu_baseline"] = cb
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- oracle arm

def oracle_inputs(cfg):
    """Host inputs of one workload for the oracle, drawn on the CPU from the same
    generator (caches only at the rows the oracle reads)."""
    import synthetic as S
    w = S.workload(cfg, seed=17)
    g = w.geom
    G = g.num_kv_groups
    h = {}
    h["q"] = S.codes16(S.normal_bf16((w.N, g.num_q_heads, g.head_dim), w.seed, S.S_Q))
    h["idx_q"] = S.codes16(S.normal_bf16((w.N, g.idx_heads, g.idx_dim), w.seed, S.S_IQ, scale=w.idx_q_scale))
    h["w"] = S.uniform_f32((w.N, g.idx_heads), w.seed, S.S_W).numpy()
    cos, sin = S.rope_tables(w.t_cap, g.rope_dims)
    h["cos"], h["sin"] = S.codes16(cos), S.codes16(sin)
    if w.random_summaries:
        h["summaries"] = S.random_summaries(w).numpy()
    else:
        h["summaries"] = np.zeros((w.B, G, w.r_cap, g.idx_dim), np.uint8)
    rows = []
    for b in range(w.B):
        for (r0, r1) in ((int(w.pre_begin[b]), int(w.pre_end[b])), (int(w.sum_begin[b]), int(w.sum_end[b]))):
            if r1 > r0:
                rows.append(((b * G + np.arange(G))[:, None] * w.t_cap + np.arange(8 * r0, 8 * r1)[None, :]).ravel())
    rows = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    kshape = (w.B, G, w.t_cap, g.idx_dim)
    h["idx_k"] = S.normal_bf16_rows(kshape, rows, w.seed, S.S_IK)
    h["idx_z"] = S.normal_bf16_rows(kshape, rows, w.seed, S.S_IZ)
    if int((w.pre_end - w.pre_begin).max()) > 0:  # set-up summaries (untimed)
        import oracle
        oracle.summarize_batch(h["idx_k"], h["idx_z"], h["cos"], h["sin"], w.pre_begin, w.pre_end, w.r_cap,
                               g.rope_dims, summ=h["summaries"])
    return w, h


def oracle_kv(w, ids, cnt, rows_n):
    import synthetic as S
    g = w.geom
    G = g.num_kv_groups
    need = []
    for i, n in enumerate(rows_n):
        b, p = int(w.row_seq[n]), int(w.row_pos[n])
        for gg in range(G):
            regs = np.concatenate([ids[i, gg, :cnt[i, gg]], [p // 8]]).astype(np.int64)
            need.append((b * G + gg) * w.t_cap + (regs[:, None] * 8 + np.arange(8)).ravel())
    need = np.concatenate(need)
    shape = (w.B, G, w.t_cap, g.head_dim)
    return S.normal_bf16_rows(shape, need, w.seed, S.S_K), S.normal_bf16_rows(shape, need, w.seed, S.S_V)


def oracle_step(w, h, groups=None, nthreads=0):
    """The oracle's whole path for the workload's rows (optionally only some groups);
    returns (seconds, threads used).  K/V drawing is outside the timed span."""
    import oracle
    g = w.geom
    t0 = time.perf_counter()
    summ = h["summaries"].copy()
    _, _, th1 = oracle.summarize_batch(h["idx_k"], h["idx_z"], h["cos"], h["sin"], w.sum_begin, w.sum_end,
                                       w.r_cap, g.rope_dims, summ=summ, nthreads=nthreads)
    scores, th2 = oracle.score_batch(h["idx_q"], h["w"], w.row_seq, w.row_pos, summ, g.num_kv_groups,
                                     g.rope_dims, h["cos"], h["sin"], nthreads=nthreads)
    if groups is not None:
        keep = np.zeros(g.num_kv_groups, bool)
        keep[list(groups)] = True
        scores[:, ~keep] = 0.0
    ids, cnt, th3 = oracle.select_batch(scores, w.row_pos, K=g.top_k, nthreads=nthreads)
    t1 = time.perf_counter()
    kc, vc = oracle_kv(w, ids, cnt, range(w.N))
    t2 = time.perf_counter()
    out, th4 = oracle.attend_batch(h["q"], kc, vc, w.row_seq, w.row_pos, ids, cnt, g.softmax_scale,
                                   nthreads=nthreads)
    t3 = time.perf_counter()
    return (t1 - t0) + (t3 - t2), max(th1, th2, th3, th4)


def oracle_sample(cfg, quarter=False, budget=10.0, max_steps=400):
    """The oracle as it stands on the host cores: whole steps of the workload repeated
    for about `budget` seconds of oracle work (at most max_steps)."""
    import oracle
    oracle.build()
    w, h = oracle_inputs(cfg)
    times, th = [], 1
    while sum(times) < budget and len(times) < max_steps:
        sec, th = oracle_step(w, h)
        times.append(sec)
    sec = float(np.mean(times))
    return {"value": round(w.N / sec, 4), "unit": UNIT, "cores": int(th), "kind": "oracle",
            "sample": f"{len(times)} whole steps of {w.name} ({w.N} row(s), all 4 KV groups) on the host "
                      f"cores, {sum(times):.1f} s of oracle work", "cpu_count": os.cpu_count()}


def run_reference(args, rank, world):
    """The oracle timed on the host cores: each step is the oracle's whole path for the
    workload's row(s); rank 0 only."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    w, h = oracle_inputs(args.workload)
    for _ in range(min(args.warmup, 1)):
        oracle_step(w, h)
    times, th = [], 1
    budget = 150.0
    t_start = time.perf_counter()
    for i in range(args.steps):
        sec, th = oracle_step(w, h)
        times.append(sec)
        if time.perf_counter() - t_start > budget:
            break
    ms = float(np.mean(times)) * 1e3
    value = w.N / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "rows_per_gpu": w.N, "context": int(w.row_pos.max())},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": int(th), "kind": "oracle",
                             "sample": f"{len(times)} whole oracle steps of {w.name} (the steps requested, "
                                       f"cut at a {budget:.0f} s budget)"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
