"""Decode-step benchmark of the DeepSeek-V4 hybrid compressed-attention hot path on GB300.

One step = SWA insert + compressor update + Lightning-Indexer scoring/top-k + sparse MLA
attention (+ split merge) over one batch of synthetic decode tokens, inputs resident in HBM.
Default workload: CSA c4 bf16, batch 32, context 65536 (16384 compressed entries per sequence),
64 query heads, indexer 64 x 128, top-k 512.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Multi-GPU: each rank runs its own batch (sequences are independent; no collective on the data
path), so per-GPU work is fixed and `value` is the total tokens of all ranks / the slowest rank.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA/HCA decode tokens/s per GB300 and achieved HBM TB/s vs roofline"
DEFAULT_CONFIG = "csa_c4_bf16"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-extra", action="store_true", help="time the headline workload only")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def rank_config(cfg, rank):
    """Replicas: every rank decodes its own batch of the workload, drawn with the seed offset by the
    rank (sequences are independent, so no data crosses ranks)."""
    return dataclasses.replace(cfg, seed=cfg.seed + 1000 * rank)


def max_over_ranks(x, world, device):
    """The largest of the ranks' values of x, on every rank (the slowest rank sets the job's time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms_per_step):
    """Whole-job throughput: the tokens of every rank's step over the (slowest rank's) step time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------------------------------------
# algorithmic bytes (what the method must move, counted from the index sets actually used)
# ------------------------------------------------------------------------------------------------

def row_bytes(dtype, width):
    return {0: 4 * width, 1: 2 * width, 2: 656, 3: width + 4, 4: width // 2 + width // 32}[dtype]


def algorithmic_bytes(st, topk_idx=None):
    """Per-call algorithmic HBM bytes of one step: each row the method reads or writes, once."""
    import dsv4_inputs as I
    cfg = st.cfg
    T, H = cfg.T, cfg.H
    act = 4 if cfg.act_dtype == I.F32 else 2
    rb = row_bytes(cfg.cache_dtype, 576)
    pos = st.positions.astype(np.int64)
    qps = cfg.q_per_seq
    b = {}
    b["insert"] = T * 576 * act + T * 8 + T * rb
    H_att = H
    if getattr(cfg, "q_prep", False):  # the fused insert also reads the raw queries and writes the padded ones
        H_att = cfg.H_pad
        b["insert"] += T * H * 576 * act + T * H_att * 576 * act
    if cfg.ratio:
        coff = cfg.coff
        sw = 2 * coff * 576 * 4
        emit = [(int(p) + 1) % cfg.ratio == 0 for p in pos]
        fold_rows = cfg.ratio * coff
        b["compress"] = T * sw * 2 + sum(emit) * (fold_rows * sw // 1 + rb)
        if cfg.topk and getattr(cfg, "ik_store", False):  # index keys: the projection once, one key row per entry
            b["compress"] += cfg.d_I * 576 * 2 + sum(emit) * row_bytes(cfg.idx_dtype, cfg.d_I)
    if cfg.ratio and cfg.topk:
        ib = row_bytes(cfg.idx_dtype, cfg.d_I)
        nc_seq = (pos.reshape(cfg.B, qps)[:, -1] + 1) // cfg.ratio
        n_keys = int(nc_seq.sum())
        cb = getattr(cfg, "cand_block", 0)
        if cb and not cfg.cand_write:
            # a candidate consumer needs the keys of the blocks its tokens name (the increasing run of
            # each list), or every key of a token whose entries fit in the top-k
            n_keys = 0
            for s_ in range(cfg.B):
                need = set()
                for t in range(s_ * qps, s_ * qps + qps):
                    nc_t = (int(pos[t]) + 1) // cfg.ratio
                    if nc_t <= cfg.topk:
                        need |= set(range(nc_t))
                        continue
                    prev = -1
                    for blk in st.cand_in[t].tolist():
                        if blk <= prev:
                            break
                        need |= set(range(blk * cb, min((blk + 1) * cb, nc_t)))
                        prev = blk
                n_keys += len(need)
        b["indexer"] = n_keys * ib + T * cfg.I_h * cfg.d_I * act + T * cfg.I_h * 4 + T * cfg.topk * 8
        if cb:
            b["indexer"] += T * cfg.cand_topk * 4  # the candidate lists read or written
    # attention: q + out + SWA rows + compressed rows (union of the sequence's selections)
    rows = 0
    for s in range(cfg.B):
        p_last = int(pos[s * qps + qps - 1])
        p_first = int(pos[s * qps])
        rows += min(p_last + 1, 128) + (p_last - p_first)  # window rows of all the seq's queries
        if cfg.ratio:
            if cfg.topk:
                sel = set()
                for t in range(s * qps, s * qps + qps):
                    row = topk_idx[t]
                    sel |= set(row[row >= 0].tolist())
                rows += len(sel)
            else:
                rows += (p_last + 1) // cfg.ratio
    out_b = 4 if cfg.out_dtype == I.F32 else 2
    b["attention"] = rows * rb + T * H_att * 576 * act + T * H_att * 512 * out_b + T * H_att * 4
    return b


# ------------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="dsv4_clocks_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, pw = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": float(max(pw))}


# ------------------------------------------------------------------------------------------------
# CPU oracle leg
# ------------------------------------------------------------------------------------------------

def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
        return int(n)
    except Exception:
        return len(os.sched_getaffinity(0))


def oracle_throughput(st, seconds):
    """Times the oracle step on as many whole sequences as fit in ~`seconds` of CPU work."""
    from oracle import dsv4_oracle as O
    cfg = st.cfg
    done, t0 = 0, time.perf_counter()
    b = 0
    while True:
        O.decode_step(st, seqs=[b])
        done += 1
        b = (b + 1) % cfg.B
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    tokens = done * cfg.q_per_seq
    return tokens / el, (f"{done} single-sequence decode steps cycling over the {cfg.B} sequences of the workload "
                         f"({tokens} tokens, full step per sequence), {el:.1f} s")


# ------------------------------------------------------------------------------------------------

def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "deepseek_v4_hybrid_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(config, kernel_file, units):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[config]
        if e.get("source_hash") != kernel_source_hash([kernel_file, "dsv4_common.cuh"]):
            return None
        return float(e["dram_bytes_per_unit"]) * units
    except Exception:
        return None


L2_BYTES = 129 * 1024 * 1024  # GB300 L2 (bench uses the device's own figure when it can read it)


def replica_count(step_bytes, l2_bytes):
    """Device replicas of a workload to rotate so that, between two uses of one replica's inputs, at
    least twice the L2 of other inputs is read (every step then starts from a cold L2 without a
    flush kernel, whose dirty lines would be written back during the timed kernels)."""
    need = int(np.ceil(2.0 * l2_bytes / max(step_bytes, 1))) + 1
    return int(min(8, max(4, need)))


def rotating_call_us(torch, replays, reps):
    """GPU time of one replay: the given graphs replayed back to back in rotation, `reps` rounds,
    between two CUDA events on the launching stream, divided by the replays made."""
    stream = torch.cuda.current_stream()
    for f in replays:
        f()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        for f in replays:
            f()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (reps * len(replays))


def measure_workload(cfg, K, warmup, world, local, want_e2e):
    """Times one workload's decode step on this GPU: the step (CUDA-graph replay, CUDA events), each
    call alone, the end-to-end path through host buffers, and the roofline of the dominant call.
    L2: the step's inputs live in R device replicas used in rotation (R chosen so that each step's
    inputs were last touched R - 1 steps, at least twice the L2 of other inputs, earlier).
    Returns a dict of the JSON fields."""
    import torch
    import dsv4_inputs as I
    import deepseek_v4_hybrid_gb300 as M
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    st = I.make_step(cfg)
    ds0 = DeviceStep(st)
    stream = torch.cuda.current_stream()
    for _ in range(max(warmup, 3)):
        ds0.run()
    torch.cuda.synchronize()
    flags = M.dsv4_read_device_flags()
    if flags:
        raise SystemExit(f"kernels raised range/timeout flags {flags:#x} during warm-up of {cfg.name}; not timing")
    topk_host = ds0.topk_idx.cpu().numpy() if ds0.has_indexer else None
    alg = algorithmic_bytes(st, topk_host)
    try:
        l2 = int(torch.cuda.get_device_properties(local).L2_cache_size)
    except Exception:
        l2 = L2_BYTES
    R = replica_count(sum(alg.values()), l2)
    reps_ds = [ds0] + [DeviceStep(st) for _ in range(R - 1)]
    ctx_range = list(map(int, (st.ctx_len.min(), st.ctx_len.max())))
    del st

    calls = ["insert", "compress", "indexer", "attention"]
    # CUDA graphs: each replica's step alone, and the R replicas' steps back to back in one graph (the
    # replicas in rotation, as R layers of one model graph would run), so that consecutive steps are
    # not separated by host graph launches; each call likewise, CALL_ROUNDS rounds of the R replicas'
    # calls in one graph.  The library never synchronises, so nothing inside a graph waits on the host.
    CALL_ROUNDS = 4
    for ds in reps_ds:
        for _ in range(max(warmup, 3)):
            ds.run()
    torch.cuda.synchronize()
    graph_single = []
    launches_step = None  # the library's kernels in one step: its launch counter across one capture
    for ds in reps_ds:
        g = torch.cuda.CUDAGraph()
        n0 = M.dsv4_kernel_launches()
        with torch.cuda.graph(g):
            ds.run()
        if launches_step is None:
            launches_step = M.dsv4_kernel_launches() - n0
        graph_single.append(g)
    graph_multi = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_multi):
        for ds in reps_ds:
            ds.run()
    graph_call = {}
    for c in calls:
        gc = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gc):
            for _ in range(CALL_ROUNDS):
                for ds in reps_ds:
                    getattr(ds, c)()
        graph_call[c] = gc
    for _ in range(3):
        graph_multi.replay()
    torch.cuda.synchronize()
    # exactly K steps: K // R replays of the R-step graph, then K % R single steps
    plan = [graph_multi] * (K // R) + [graph_single[k] for k in range(K % R)]
    steps_of = [R] * (K // R) + [1] * (K % R)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(len(plan))]
    sampler = ClockSampler(local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)
    wall0 = time.perf_counter()
    for k, g in enumerate(plan):
        ev[k][0].record(stream)
        g.replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_per_step = sum(e[0].elapsed_time(e[1]) for e in ev) / sum(steps_of)
    ms_per_step = max_over_ranks(ms_per_step, world, "cuda")
    # per-call breakdown: each call's graph (CALL_ROUNDS x R calls, replicas in rotation), CUDA events
    # around a few replays, divided by the calls made
    reps = max(1, min(K, 400) // (R * CALL_ROUNDS))
    per_call_us = {c: rotating_call_us(torch, [graph_call[c].replay], reps) / (R * CALL_ROUNDS) for c in calls}

    res = {"ms_per_step": ms_per_step, "value": job_tokens_per_s(cfg.T, world, ms_per_step), "calls_us": per_call_us,
           "clocks": clocks, "wall_s_timed": wall, "gpu_launches": int(K * launches_step),
           "timing": (f"steps: CUDA graphs of the {R} replicas' steps back to back ({K // R} replays) + {K % R} "
                      f"single-step graphs; calls: graphs of {CALL_ROUNDS} x {R} calls"),
           "step_algorithmic_gbs": sum(alg.values()) / (ms_per_step * 1e-3) / 1e9,
           "config": {"workload": cfg.name, "batch_per_gpu": cfg.B, "q_per_seq": cfg.q_per_seq,
                      "context": ctx_range,
                      "heads": cfg.H, "ratio": cfg.ratio, "indexer": [cfg.I_h, cfg.d_I], "topk": cfg.topk, "page": 64,
                      "l2": (f"inputs larger than L2: {R} device replicas of the step's inputs used in rotation, "
                             f"so each step's inputs were last read {R - 1} steps earlier with >= 2x L2 "
                             f"({l2 // 2**20} MiB) of other inputs read since; no flush kernel")},
           "dtype": {0: "f32", 1: "bf16"}[cfg.act_dtype] + "/" + I.DTYPE_NAMES[cfg.cache_dtype]}

    if want_e2e:
        # end to end through host buffers: every step copies its inputs from pinned host memory into
        # its replica (H2D stream), runs the step graph (compute stream) and reads the output and top-k
        # back into pinned host memory (D2H stream).  The R replicas are R independent batches in
        # flight: batch k + 1's inputs upload while batch k computes.  Events keep each replica's
        # inputs until its step has read them and its outputs until they have been copied back.
        host_in = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in ds0.step_input_tensors().items()}
        for k, v in ds0.step_input_tensors().items():
            host_in[k].copy_(v)
        host_out = torch.empty_like(ds0.out, device="cpu").pin_memory()
        host_topk = torch.empty_like(ds0.topk_idx, device="cpu").pin_memory() if ds0.has_indexer else None
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = host_out.numel() * host_out.element_size() + (host_topk.numel() * 4 if host_topk is not None else 0)
        Ke = max(20, min(K, 400)) // R * R
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(Ke)]
        ev_comp = [torch.cuda.Event() for _ in range(Ke)]
        ev_out = [torch.cuda.Event() for _ in range(Ke)]
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e_start.record(h2d_s)
        for k in range(Ke):
            r = k % R
            ds = reps_ds[r]
            if k >= R:
                h2d_s.wait_event(ev_comp[k - R])  # step k - R has read this replica's inputs
            with torch.cuda.stream(h2d_s):
                for name, dev in ds.step_input_tensors().items():
                    dev.copy_(host_in[name], non_blocking=True)
                ev_in[k].record(h2d_s)
            stream.wait_event(ev_in[k])
            if k >= R:
                stream.wait_event(ev_out[k - R])  # step k - R's outputs of this replica are copied back
            graph_single[r].replay()
            ev_comp[k].record(stream)
            d2h_s.wait_event(ev_comp[k])
            with torch.cuda.stream(d2h_s):
                host_out.copy_(ds.out, non_blocking=True)
                if host_topk is not None:
                    host_topk.copy_(ds.topk_idx, non_blocking=True)
                ev_out[k].record(d2h_s)
        e_end.record(d2h_s)
        e_end.synchronize()
        e2e_ms = e_start.elapsed_time(e_end) / Ke
        e2e_ms = max_over_ranks(e2e_ms, world, "cuda")
        res["e2e"] = {"value": job_tokens_per_s(cfg.T, world, e2e_ms), "unit": "tokens/s",
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
                      "method": (f"{Ke} steps; per step pinned H2D of its inputs, the step graph, D2H of output and "
                                 f"top-k, on three streams with {R} batches in flight")}

    # roofline of the dominant call
    dom = max((c for c in calls if c in alg), key=lambda c: per_call_us[c])
    peak, peak_kind = peaks()
    achieved = alg[dom] / (per_call_us[dom] * 1e-6) / 1e9
    dom_file = {"indexer": "indexer_topk.cu", "attention": "attention.cu", "compress": "insert_compress.cu",
                "insert": "insert_compress.cu"}[dom]
    res["roofline"] = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                       "frac": achieved / peak, "peak_kind": peak_kind,
                       "traffic": traffic_from_profiles(cfg.name, dom_file, cfg.T),
                       "algorithmic_bytes": int(alg[dom]), "us_per_launch": per_call_us[dom]}
    res["calls_roofline"] = {c: {"algorithmic_bytes": int(alg[c]), "us": per_call_us[c],
                                 "frac": alg[c] / (per_call_us[c] * 1e-6) / 1e9 / peak if per_call_us[c] > 0 else None}
                             for c in calls if c in alg}
    del reps_ds, ds0, graph_single, graph_multi, graph_call
    torch.cuda.empty_cache()
    return res


def measure_prefill(name, K, warmup, local):
    """Times a chunked prefill (every position of every sequence from 0, four positions of each
    sequence a chunk, the chain's calls for each chunk) captured as one CUDA graph: CUDA events around
    each replay, an L2-sized buffer written before each (the prefill's caches fit in L2).  Value:
    prompt tokens per second."""
    import torch
    import dsv4_inputs as I
    import deepseek_v4_hybrid_gb300 as M
    from deepseek_v4_hybrid_gb300.step import PrefillRunner
    cfg, P = I.PREFILL_CONFIGS[name]
    pf = I.make_prefill(cfg, P)
    runner = PrefillRunner(pf, chunk=4)
    stream = torch.cuda.current_stream()
    for _ in range(max(warmup, 3)):
        runner.run()
    torch.cuda.synchronize()
    flags = M.dsv4_read_device_flags()
    if flags:
        raise SystemExit(f"kernels raised range/timeout flags {flags:#x} during warm-up of {name}; not timing")
    alg = 0
    for (p0, n), ds in zip(runner.spans, runner.steps):
        topk = ds.topk_idx.cpu().numpy() if ds.has_indexer else None
        alg += sum(algorithmic_bytes(pf.chunk(p0, n), topk).values())
    g = torch.cuda.CUDAGraph()
    n0 = M.dsv4_kernel_launches()
    with torch.cuda.graph(g):
        runner.run()
    launches = M.dsv4_kernel_launches() - n0
    l2 = int(torch.cuda.get_device_properties(local).L2_cache_size)
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device="cuda")
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    for k in range(K):
        flush.fill_(float(k))
        ev[k][0].record(stream)
        g.replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    peak, peak_kind = peaks()
    gbs = alg / (ms * 1e-3) / 1e9
    return {"metric": "prefill tokens/s per GB300", "value": cfg.B * P / (ms * 1e-3), "unit": "tokens/s",
            "ms_per_prefill": ms, "steps": K, "gpu_launches": int(K * launches), "clocks": clocks,
            "dtype": {0: "f32", 1: "bf16"}[cfg.act_dtype] + "/" + I.DTYPE_NAMES[cfg.cache_dtype],
            "algorithmic_gbs": gbs, "frac_of_hbm": gbs / peak, "peak_kind": peak_kind,
            "config": {"workload": name, "batch_per_gpu": cfg.B, "prompt": P, "chunk": 4, "chunks": len(runner.spans),
                       "heads": cfg.H, "ratio": cfg.ratio, "indexer": [cfg.I_h, cfg.d_I], "topk": cfg.topk,
                       "l2": f"a {2 * l2 // 2**20} MiB buffer written before each timed prefill"}}


PREFILL_WORKLOADS = ("prefill_c4_bf16",)

EXTRA_WORKLOADS = ("hca_c128_bf16", "csa_c4_fp8", "csa_c4_1m", "csa_c4_mxfp4", "csa_c4_cand", "csa_c4_src")


def run_ours(args):
    import torch
    import torch.distributed as dist
    import dsv4_inputs as I
    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    cfg = rank_config(I.ALL_CONFIGS[args.config], rank)
    K = args.steps
    head = measure_workload(cfg, K, args.warmup, world, local, want_e2e=True)
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic (seeded N(0,1)*0.1 rows, shuffled paged block tables)",
        "config": dict(head["config"], parallelism=f"replicas x{world} (per-sequence)"),
        "e2e": head["e2e"], "gpu_launches": head["gpu_launches"], "roofline": head["roofline"],
        "calls_us": head["calls_us"], "calls_roofline": head["calls_roofline"],
        "step_algorithmic_gbs": head["step_algorithmic_gbs"], "clocks": head["clocks"], "timing": head["timing"],
        "wall_s_timed": head["wall_s_timed"],
    }
    if world == 1 and not args.no_extra:
        # the other full-size workloads on the same GPU (the headline stays `config.workload`)
        extra = {}
        for name in EXTRA_WORKLOADS:
            if name == cfg.name:
                continue
            r = measure_workload(I.ALL_CONFIGS[name], min(K, 500), args.warmup, 1, local, want_e2e=False)
            extra[name] = {k: r[k] for k in ("value", "ms_per_step", "dtype", "config", "roofline", "calls_us",
                                             "calls_roofline", "step_algorithmic_gbs", "clocks", "gpu_launches",
                                             "timing")}
            extra[name]["unit"] = "tokens/s"
            extra[name]["steps"] = min(K, 500)
        for name in PREFILL_WORKLOADS:
            extra[name] = measure_prefill(name, max(3, min(K, 20)), args.warmup, local)
        line["extra_workloads"] = extra
    if rank == 0 and not args.no_cpu_baseline:
        st = I.make_step(cfg)
        v, sample = oracle_throughput(st, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": sample}
        one = oracle_single_core(args.config, args.cpu_seconds)
        if one is not None:
            line["cpu_baseline"]["single_core"] = one
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def oracle_single_core(config, seconds):
    """The same oracle sample in a child process limited to one core (BLAS threads 1, CPU affinity
    one core)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import os, sys, json; sys.path.insert(0, %r); os.sched_setaffinity(0, {min(os.sched_getaffinity(0))}); "
            "import bench, dsv4_inputs as I; st = I.make_step(I.ALL_CONFIGS[%r]); "
            "v, s = bench.oracle_throughput(st, %r); print(json.dumps({'value': v, 'sample': s}))"
            % (ROOT, config, float(seconds)))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        d = json.loads(r.stdout.strip().splitlines()[-1])
        return {"value": d["value"], "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": d["sample"]}
    except Exception:
        return None


def run_reference(args):
    """The CPU oracle as the reference arm, timed on this host's cores on a bounded sample."""
    import dsv4_inputs as I
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cfg = I.ALL_CONFIGS[args.config]
    st = I.make_step(cfg)
    from oracle import dsv4_oracle as O
    # one reference step = the oracle's whole decode step for one sequence; the run stops after K
    # steps or ~150 s of CPU time, whichever comes first, and reports the steps it ran
    for _ in range(min(args.warmup, 1)):
        O.decode_step(st, seqs=[0])
    tokens, el, b = 0, 0.0, 0
    K = 0
    while K < max(1, args.steps) and el < 150.0:
        t0 = time.perf_counter()
        O.decode_step(st, seqs=[b % cfg.B])
        el += time.perf_counter() - t0
        tokens += cfg.q_per_seq
        b += 1
        K += 1
    v = tokens / el
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64 (oracle)", "data": "synthetic", "impl": "reference",
            "config": {"workload": cfg.name, "batch_per_gpu": cfg.B},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{b} sequence steps over {el:.1f} s"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
