"""Benchmark of the fixed-size KV cache hot path on GB300.

One step = one pass of the whole path over one batch: snap_compress of every
sequence's prompt (window scoring, pooling, top-K, cache build), then D decode
steps over the fixed-size cache (snap_decode_step: ring append + split-KV attention).
Inputs are seeded synthetic tensors already resident in HBM (the prefill K/V/Q
of the batch and every decode step's q/k/v); they exceed the 129 MB L2 many
times over, so no L2 flush is needed between steps.

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  value = decoded tokens of all ranks / the
slowest rank's step time (compression included).  The line also carries the
decode-only throughput, the compression time, the uncompressed full-KV decode
baseline on the same GPU, the dominant kernel's roofline fraction, an
end-to-end figure through the C ABI with host buffers, and the CPU oracle timed
on a bounded sample.  --impl reference times the CPU oracle alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode tok/s + HBM GB/s (fixed cache vs full KV) at 128k ctx; compress ms"
L2_BYTES = 129 << 20
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0      # the ~8 TB/s nominal HBM3e figure decode is also reported against
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default="gqa_128k_b16")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling)")
    p.add_argument("--eager", action="store_true",
                   help="launch the decode steps one by one instead of replaying them as one captured "
                        "CUDA graph (the default: the decode loop has static shapes and no host sync)")
    p.add_argument("--graph", action="store_true", help=argparse.SUPPRESS)  # the default; kept for old commands
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-full-kv", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--prefill-only", type=int, default=0, metavar="S",
                   help="extra mode: only the prefill attention of one S-token prompt (profiling)")
    p.add_argument("--no-prefill", action="store_true",
                   help="skip the prefill-attention timing (compression as prefill overhead)")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the short runs of the other four workloads that the 128k line carries")
    p.add_argument("--capacity", type=float, default=0.0, metavar="GIB",
                   help="extra mode: the largest batch whose cache fits GIB of HBM, fixed-size cache vs full "
                        "KV, with decode tok/s measured at that batch (one JSON line per cache kind)")
    p.add_argument("--sweep", action="store_true",
                   help="extra mode: decode tok/s over context length (fixed C = S/4 vs full KV) and over "
                        "the cache composition (L_sink, K, L_recent) at 128k (one JSON line per case)")
    return p.parse_args()


# ----------------------------------------------------------------------------- peaks
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
        bf = d.get("bf16_tflops_sustained") or d.get("bf16_tflops")
        burst = d.get("bf16_tflops") or bf
        if hbm:
            return float(hbm), float(bf or FALLBACK_BF16_TFLOPS), float(burst or FALLBACK_BF16_TFLOPS), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"snap_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- workload
def replica_seed(seed, rank):
    """Each rank is an independent replica with its own inputs (weak scaling)."""
    return seed + 7919 * rank


def max_over_ranks(x, world, device):
    """The slowest rank's value (timings are reported as the max over ranks)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, max_ms):
    """Whole-job tokens per second: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / (max_ms / 1e3)


def make_batch(wl, seed, rank, device):
    import torch
    from fixed_size_kv_gb300 import inputs
    rs = replica_seed(seed, rank)
    lengths = inputs.prompt_lengths(wl, rs)
    pre = [inputs.gen_prefill(wl, S, seed=rs, seq=b, device=device)
           for b, S in enumerate(lengths)]
    qs, ks, vs = [], [], []
    for t in range(wl.decode_steps):
        tok = inputs.gen_decode(wl, wl.batch, step=t, seed=rs, device=device)
        qs.append(tok.q)
        ks.append(tok.k)
        vs.append(tok.v)
    q = torch.stack(qs)
    k = torch.stack(ks)
    v = torch.stack(vs) if wl.layout == 0 else None
    return lengths, pre, q, k, v


def window_lse(wl, K, Q):
    """Natural-log log-sum-exp of every observation row over its causal keys, fp32 [W][H_q]:
    what a prefill attention kernel already has (plain torch; set-up, not timed)."""
    import torch
    S = K.shape[0]
    pos = torch.arange(S - wl.W, S, device=K.device).view(-1, 1)
    keys = torch.arange(S, device=K.device).view(1, -1)
    out = torch.empty((wl.W, wl.n_q_heads), dtype=torch.float32, device=K.device)
    for i in range(wl.n_q_heads):
        h = i // wl.G
        s = wl.sm_scale * (Q[:, i, :] @ K[:, h, :].T).float()              # [W][S], fp32 accumulation
        out[:, i] = torch.logsumexp(s.masked_fill(keys > pos, float("-inf")), dim=1)
    return out.contiguous()


def algorithmic_decode_flop(wl, metas):
    """FLOP one decode-attention launch must do: per valid cache row and query head, the
    score (2 d_qk) and the weighted value sum (2 d_v)."""
    valid = 0
    for m in metas:
        S, T, R0, n_sink, n_mid = m
        valid += n_sink + n_mid + min(T - R0, wl.L_recent)
    return valid * wl.G * 2.0 * (wl.d_qk + wl.d_v) * wl.n_kv_heads


def issued_decode_flop(wl, metas):
    """FLOP the decode kernels' MMAs issue per launch.  GQA issues the algorithmic work.  The
    MLA kernel runs two CTAs per split, each computing the whole 576-wide score of all query
    heads and half of the value sum: per valid row 2 (2 d_qk) + 2 d_v per query head."""
    if wl.layout == 0:
        return algorithmic_decode_flop(wl, metas)
    valid = 0
    for m in metas:
        S, T, R0, n_sink, n_mid = m
        valid += n_sink + n_mid + min(T - R0, wl.L_recent)
    return valid * wl.G * 2.0 * (2 * wl.d_qk + wl.d_v) * wl.n_kv_heads


def algorithmic_decode_bytes(wl, metas):
    """Bytes one decode-attention launch must move: every valid cache row once
    (keys, plus values for GQA), the queries and the outputs."""
    row = wl.n_kv_heads * (wl.d_qk + (wl.d_v if wl.layout == 0 else 0)) * 2
    valid = 0
    for m in metas:
        S, T, R0, n_sink, n_mid = m
        valid += n_sink + n_mid + min(T - R0, wl.L_recent)
    n = len(metas)
    return valid * row + n * wl.n_q_heads * (wl.d_qk * 2 + wl.d_v * 4)


def workload_config(wl, B, lengths, world):
    """The workload description both arms print (the GPU arm and the oracle arm)."""
    return {"workload": wl.name, "batch": B, "prompt_len": max(lengths), "decode_steps": wl.decode_steps,
            "cache": f"{wl.L_sink}+{wl.K}+{wl.L_recent}={wl.C}", "W": wl.W, "P": wl.P,
            "heads": f"{wl.n_q_heads}/{wl.n_kv_heads}x{wl.d_qk}", "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (no flush)"}


def score_pass_flop(wl, lengths):
    """Algorithmic FLOP of one score GEMM pass per sequence (mean over the batch):
    2 R d S per KV head, R = G W observation rows (the compression's one dense contraction)."""
    return statistics.mean(2.0 * wl.G * wl.W * wl.d_qk * S * wl.n_kv_heads for S in lengths)


def compress_hbm_bytes(wl, lengths, passes):
    """Algorithmic HBM bytes of one compression call per sequence (mean over the batch):
    each score pass reads the prompt's keys once (S x Hkv x d_qk bf16) and the cache write
    reads and writes the kept rows (C x Hkv rows of d_qk + d_v bf16, MLA's one 576-wide
    row); the window queries and the column sums (a few MB) are left out."""
    row = wl.d_qk + (wl.d_v if wl.layout == 0 else 0)
    return statistics.mean(passes * 2.0 * S * wl.n_kv_heads * wl.d_qk + 2 * 2.0 * wl.n_kv_heads * wl.C * row
                           for S in lengths)


def gpu_head_start(stream, ms=1.0):
    """Enqueues about `ms` of device-side sleep on `stream`, so that the host has queued
    the launches that follow (and their events) before the GPU reaches them: the events
    then time the kernels, not the host's launch path."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 2.0e6))     # cycles at about 2 GHz


def time_compress_stages(cache, pre, stream, lses=None, reps=2):
    """Per-sequence CUDA-event times (ms) of each compression stage, each stage launched
    on its own between events (snap_compress_stages) behind a device-side head start;
    the last of `reps` passes."""
    import torch
    from fixed_size_kv_gb300 import snap
    stages = [("rows", snap.STAGE_ROWS), ("columns", snap.STAGE_COLUMNS), ("select", snap.STAGE_SELECT),
              ("write", snap.STAGE_WRITE)]
    B = len(pre)
    out = {}
    for _ in range(reps):
        evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in stages]
               for _ in range(B)]
        for b in range(B):
            p = pre[b]
            gpu_head_start(stream)
            for i, (_, bit) in enumerate(stages):
                evs[b][i][0].record(stream)
                cache.compress_stages(b, p.K, p.V, p.Q, bit, lse_obs=None if lses is None else lses[b],
                                      stream=stream)
                evs[b][i][1].record(stream)
        stream.synchronize()
        out = {name: statistics.mean(evs[b][i][0].elapsed_time(evs[b][i][1]) for b in range(B))
               for i, (name, _) in enumerate(stages)}
    return out


def measure(wl, args, steps, warmup, dev, stream, world, rank, full_run=True):
    """One workload on this GPU: `warmup` untimed steps, then `steps` timed steps of
    (compress every prompt, then every decode step of the batch, the decode loop
    replayed as one CUDA graph unless --eager).  Returns the JSON fields of the
    workload (without the CPU baseline and the end-to-end run)."""
    import torch

    from fixed_size_kv_gb300 import snap

    B, D = wl.batch, wl.decode_steps
    hbm_peak, bf16_sus, bf16_burst, peak_kind = peaks()
    with torch.cuda.stream(stream):
        lengths, pre, q_all, k_all, v_all = make_batch(wl, args.seed, rank, dev)
    stream.synchronize()
    cfg = snap.make_config(**wl.config_kwargs())
    cache = snap.SnapCache(cfg, max_batch=B, max_prompt=max(lengths), max_n=B, device=dev, stream=stream)
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    out = torch.empty((D, B, wl.n_q_heads, wl.d_v), dtype=torch.float32, device=dev)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def one_step(c, prefill, record=None):
        ev = record
        if ev is not None:
            ev["c0"].record(stream)
        for b in range(B):
            p = prefill[b]
            c.compress(b, p.K, p.V, p.Q, stream=stream)
        if ev is not None:
            ev["c1"].record(stream)
        for t in range(D):
            # one decode step: append the new token, then attend (snap_decode_step)
            if ev is not None:
                ev["a0"][t].record(stream)
            c.decode_step(slots, q_all[t], k_all[t], v_all[t] if v_all is not None else None, out=out[t],
                          stream=stream)
            if ev is not None:
                ev["a1"][t].record(stream)
        if ev is not None:
            ev["d1"].record(stream)

    def new_events():
        E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        return {"s0": E(), "c0": E(), "c1": E(), "d1": E(),
                "a0": [E() for _ in range(D)], "a1": [E() for _ in range(D)]}

    for _ in range(warmup):
        one_step(cache, pre)
    barrier()
    graph = None
    if not args.eager:
        # the decode loop has static shapes and no host synchronisation: capture it once
        graph = torch.cuda.CUDAGraph()
        for b in range(B):
            cache.compress(b, pre[b].K, pre[b].V, pre[b].Q, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for t in range(D):
                cache.decode_step(slots, q_all[t], k_all[t], v_all[t] if v_all is not None else None,
                                  out=out[t], stream=stream)
        stream.synchronize()
    st = cache.check_device(stream)
    if st != snap.SNAP_OK:
        raise RuntimeError(f"{wl.name}: device status after warm-up: {snap.status_string(st)}")
    metas = [tuple(r[:5]) for r in cache.meta().cpu().tolist()]
    # the decode launches see T = S .. S + D - 1; bytes at the middle step stand for all
    mid_metas = [(S, S + D // 2, R0, ns, nm) for (S, T, R0, ns, nm) in
                 [(m[0], m[1], m[2], m[3], m[4]) for m in metas]]
    attn_bytes = algorithmic_decode_bytes(wl, mid_metas)
    attn_flop = algorithmic_decode_flop(wl, mid_metas)
    attn_issued = issued_decode_flop(wl, mid_metas)

    # working set of one step: prompts, cache, decode inputs and outputs
    work_bytes = sum(p.K.numel() * 2 + (p.V.numel() * 2 if p.V is not None else 0) for p in pre)
    work_bytes += snap.cache_bytes(cfg, B) + q_all.numel() * 2 + k_all.numel() * 2 + out.numel() * 4
    flush = None
    if work_bytes < 4 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    clocks = ClockSampler(dev.index or 0) if full_run else None
    if clocks:
        clocks.start()
    evs = [new_events() for _ in range(steps)]
    barrier()
    t_wall = time.perf_counter()
    for i in range(steps):
        if flush is not None:  # evict the previous step's data from L2 (not timed)
            with torch.cuda.stream(stream):
                flush.fill_(i & 255)
        evs[i]["s0"].record(stream)
        if graph is None:
            one_step(cache, pre, evs[i])
        else:
            evs[i]["c0"].record(stream)
            for b in range(B):
                cache.compress(b, pre[b].K, pre[b].V, pre[b].Q, stream=stream)
            evs[i]["c1"].record(stream)
            with torch.cuda.stream(stream):  # replay on the stream the events are recorded on
                graph.replay()
            evs[i]["d1"].record(stream)
    barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop() if clocks else None
    step_ms = [evs[i]["s0"].elapsed_time(evs[i]["d1"]) for i in range(steps)]
    compress_ms = [evs[i]["c0"].elapsed_time(evs[i]["c1"]) for i in range(steps)]
    decode_ms = [evs[i]["c1"].elapsed_time(evs[i]["d1"]) for i in range(steps)]
    if graph is not None:
        # per-launch attention time from one more pass of the same calls, launched one by one
        ev = new_events()
        one_step(cache, pre, ev)
        stream.synchronize()
        evs = [ev]
    attn_ms = [sum(e["a0"][t].elapsed_time(e["a1"][t]) for t in range(D)) / D for e in evs]
    eager_launch_ms = statistics.mean(attn_ms)
    st = cache.check_device(stream)
    if st != snap.SNAP_OK:
        raise RuntimeError(f"{wl.name}: device status after timed steps: {snap.status_string(st)}")

    def reduce_max(x):
        return max_over_ranks(x, world, dev)

    total_ms = reduce_max(sum(step_ms))
    dec_ms = reduce_max(sum(decode_ms)) / steps
    cmp_ms = reduce_max(sum(compress_ms)) / steps
    # the decode step's device time: from the graph-replayed loop (back-to-back launches, as
    # the timed region runs them) when the loop is a graph, else per eager launch; a GQA step
    # is one kernel, an MLA step the attention kernel plus its merge
    attn_avg_ms = dec_ms / D if graph is not None else eager_launch_ms
    attn_gbs = attn_bytes / (attn_avg_ms / 1e3) / 1e9

    # ---------------------------------------------------------------- full-KV baseline
    full = None
    if not args.no_full_kv:
        full_wl = wl.replace(L_sink=0, K=0, L_recent=max(lengths) + D)
        fcfg = snap.make_config(**full_wl.config_kwargs())
        fcache = snap.SnapCache(fcfg, max_batch=B, max_prompt=1, max_n=B, device=dev, stream=stream)

        def f_decode():
            for t in range(D):
                fcache.decode_step(slots, q_all[t], k_all[t], v_all[t] if v_all is not None else None,
                                   out=out[t], stream=stream)

        fgraph = None
        if not args.eager:  # the same launch mode as the fixed cache's decode loop
            for b in range(B):
                fcache.compress(b, pre[b].K, pre[b].V, pre[b].Q, stream=stream)
            stream.synchronize()
            fgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(fgraph, stream=stream):
                f_decode()
            stream.synchronize()
        runs = []
        for rep in range(2):
            for b in range(B):
                fcache.compress(b, pre[b].K, pre[b].V, pre[b].Q, stream=stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea, eb = [], []
            e0.record(stream)
            for t in range(D):
                a, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fcache.decode_step(slots, q_all[t], k_all[t], v_all[t] if v_all is not None else None,
                                   out=out[t], stream=stream)
                bb.record(stream)
                ea.append(a)
                eb.append(bb)
            e1.record(stream)
            stream.synchronize()
            loop_ms = e0.elapsed_time(e1)
            if fgraph is not None:  # the loop time from a replay (the attention time above stays per launch)
                for b in range(B):
                    fcache.compress(b, pre[b].K, pre[b].V, pre[b].Q, stream=stream)
                e0.record(stream)
                with torch.cuda.stream(stream):
                    fgraph.replay()
                e1.record(stream)
                stream.synchronize()
                loop_ms = e0.elapsed_time(e1)
            runs.append((loop_ms, sum(x.elapsed_time(y) for x, y in zip(ea, eb)) / D))
        f_ms, f_attn = min(runs)
        fmetas = [(S, S + D // 2, 0, 0, 0) for S in lengths]
        f_bytes = algorithmic_decode_bytes(full_wl, fmetas)
        full = {"decode_tok_s": B * D * world / (f_ms / 1e3), "decode_ms_per_token_step": f_ms / D,
                "attn_ms": f_attn, "attn_hbm_gbs": f_bytes / (f_attn / 1e3) / 1e9,
                "attn_frac": f_bytes / (f_attn / 1e3) / 1e9 / hbm_peak,
                "cache_bytes": snap.cache_bytes(fcfg, B)}
        del fcache, fgraph
        torch.cuda.empty_cache()

    # ---------------------------------------------------------------- prefill attention of the first
    # prompt (GQA): its time, its tensor roofline, and the compression as overhead on it
    prefill = None
    lse0 = None
    if wl.layout == 0 and not args.no_prefill:
        from fixed_size_kv_gb300 import inputs
        p0 = pre[0]
        S0 = p0.K.shape[0]
        with torch.cuda.stream(stream):
            Qf = inputs.gen_prompt_queries(wl, p0, seed=replica_seed(args.seed, rank), seq=0, device=dev)
            Of = torch.empty_like(Qf)
            lse0 = torch.empty((wl.W, wl.n_q_heads), dtype=torch.float32, device=dev)
        pe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
        for e0_, e1_ in pe:
            e0_.record(stream)
            cache.prefill_attn(Qf, p0.K, p0.V, O=Of, lse_obs=lse0, stream=stream)
            e1_.record(stream)
        stream.synchronize()
        pre_ms = min(a_.elapsed_time(b_) for a_, b_ in pe[1:])
        pflop = 2.0 * wl.n_q_heads * wl.d_qk * S0 * (S0 + 1)      # QK^T and PV over the causal half
        prefill = {"prompt_len": S0, "ms": pre_ms, "flop": pflop,
                   "achieved_tflops": pflop / (pre_ms / 1e3) / 1e12,
                   "frac": pflop / (pre_ms / 1e3) / 1e12 / bf16_burst, "peak": bf16_burst,
                   "peak_kind": "bf16 burst", "kernel": "prefill_tc_kernel (snap_prefill_attn)"}
        del Qf, Of
    # ---------------------------------------------------------------- compression, stage by stage,
    # and with the prefill's log-sum-exp supplied (snap_compress_lse: no row pass)
    lses = [window_lse(wl, p.K, p.Q) for p in pre]
    if lse0 is not None:
        lses[0] = lse0              # the prefill kernel's own log-sum-exp for the first prompt
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for rep in range(2):
        gpu_head_start(stream)
        e0.record(stream)
        for b in range(B):
            cache.compress_lse(b, pre[b].K, pre[b].V, pre[b].Q, lses[b], stream=stream)
        e1.record(stream)
        stream.synchronize()
    cmp_lse_ms = e0.elapsed_time(e1) / B
    stage_ms = time_compress_stages(cache, pre, stream)
    if prefill is not None:
        gpu_head_start(stream)
        e0.record(stream)
        cache.compress_lse(0, pre[0].K, pre[0].V, pre[0].Q, lses[0], stream=stream)
        e1.record(stream)
        stream.synchronize()
        c_lse0 = e0.elapsed_time(e1)
        gpu_head_start(stream)
        e0.record(stream)
        cache.compress(0, pre[0].K, pre[0].V, pre[0].Q, stream=stream)
        e1.record(stream)
        stream.synchronize()
        c_full0 = e0.elapsed_time(e1)
        prefill["compress_with_prefill_lse_ms"] = c_lse0
        prefill["compress_both_passes_ms"] = c_full0
        prefill["overhead_frac"] = c_lse0 / prefill["ms"]
        prefill["overhead_frac_both_passes"] = c_full0 / prefill["ms"]
    del lses
    F = score_pass_flop(wl, lengths)
    tf = lambda ms: F / (ms / 1e3) / 1e12 if ms else None  # noqa: E731
    scored = any((max(wl.L_sink, S - wl.L_recent) if S > wl.L_sink else S) - min(S, wl.L_sink) > wl.K > 0
                 for S in lengths)
    compress_roofline = None
    if scored:
        compress_roofline = {
            "bound": "tensor", "unit": "TFLOP/s", "peak": bf16_burst,
            "peak_kind": "bf16 burst (each pass timed on its own)", "peak_source": peak_kind,
            "flop_per_pass_per_seq": F,
            "row_pass": {"ms": stage_ms["rows"], "achieved": tf(stage_ms["rows"]),
                         "frac": tf(stage_ms["rows"]) / bf16_burst,
                         "note": "row-statistics GEMM plus the small merge of its per-split partials"},
            "column_pass": {"ms": stage_ms["columns"], "achieved": tf(stage_ms["columns"]),
                            "frac": tf(stage_ms["columns"]) / bf16_burst},
            "select_ms": stage_ms["select"], "cache_write_ms": stage_ms["write"],
            "whole_call": {"ms": cmp_ms / B, "achieved": tf(cmp_ms / B), "frac": tf(cmp_ms / B) / bf16_burst,
                           "note": "snap_compress per sequence against one GEMM's FLOP"},
            "whole_call_with_prefill_lse": {"ms": cmp_lse_ms, "achieved": tf(cmp_lse_ms),
                                            "frac": tf(cmp_lse_ms) / bf16_burst},
            # on the FLOP the MMAs issue: two passes without the prefill's LSE, one with it
            "issued": {"whole_call": {"flop": 2 * F, "frac": 2 * tf(cmp_ms / B) / bf16_burst},
                       "whole_call_with_prefill_lse": {"flop": F, "frac": tf(cmp_lse_ms) / bf16_burst}},
        }

        def call_roofline(ms, passes):
            hb = compress_hbm_bytes(wl, lengths, passes)
            t_hbm = hb / (hbm_peak * 1e9) * 1e3              # ms at the measured copy peak
            t_tc = passes * F / (bf16_burst * 1e12) * 1e3    # ms at the measured bf16 burst
            floor = max(t_hbm, t_tc)
            return {"ms": ms, "hbm_bytes": hb, "flop": passes * F, "hbm_floor_ms": t_hbm,
                    "tensor_floor_ms": t_tc, "bound": "hbm" if t_hbm >= t_tc else "tensor",
                    "achieved_gbs": hb / (ms / 1e3) / 1e9, "frac": floor / ms}
        # the whole call against its own floor: the larger of its bytes at the HBM peak and
        # its GEMM FLOP at the bf16 burst (frac = floor / measured time)
        compress_roofline["call"] = {"with_prefill_lse": call_roofline(cmp_lse_ms, 1),
                                     "both_passes": call_roofline(cmp_ms / B, 2),
                                     "hbm_peak_gbs": hbm_peak, "bf16_peak_tflops": bf16_burst}
    cache_write_bytes = statistics.mean(2 * wl.n_kv_heads * wl.C * (wl.d_qk + (wl.d_v if wl.layout == 0 else 0)) * 2
                                        for _ in lengths)

    splits = cache.decode_attn_plan(B)[0]
    n_seq_launch = 5  # rowstat, lse merge, colsum, select, cache write (scored prompts)
    per_step_launches = 0
    for S in lengths:
        M = (max(wl.L_sink, S - wl.L_recent) if S > wl.L_sink else S) - min(S, wl.L_sink)
        per_step_launches += n_seq_launch if (M > wl.K and wl.K > 0) else 1
    per_step_launches += D * decode_launches_per_step(wl, splits)
    res = {
        "lengths": lengths, "pre": pre, "q_all": q_all, "k_all": k_all, "v_all": v_all, "cfg": cfg,
        "B": B, "D": D, "steps": steps, "graph": graph is not None, "flush": flush is not None,
        "splits": splits, "value": job_throughput(B * D * steps, world, total_ms),
        "ms_per_step": total_ms / steps, "clk": clk, "t_wall": t_wall,
        "fields": {
            "decode_tok_s": B * D * world / (dec_ms / 1e3),
            "decode_ms_per_token_step": dec_ms / D,
            "compress_ms_per_batch": cmp_ms,
            "compress_ms_per_seq": cmp_ms / B,
            "compress_with_prefill_lse_ms_per_seq": cmp_lse_ms,
            "compress_stage_ms_per_seq": stage_ms,
            "attn": {"ms": attn_avg_ms, "hbm_gbs": attn_gbs, "bytes_per_launch": attn_bytes,
                     "frac": attn_gbs / hbm_peak, "frac_of_nominal": attn_gbs / NOMINAL_HBM_GBS,
                     "nominal_gbs": NOMINAL_HBM_GBS,
                     # the same launch against the tensor roofline (bf16 sustained: the decode
                     # loop runs for a long time); it matters for the MLA layout, at the ridge
                     "tensor": {"flop_per_launch": attn_flop,
                                "achieved_tflops": attn_flop / (attn_avg_ms / 1e3) / 1e12,
                                "peak": bf16_sus,
                                "frac": attn_flop / (attn_avg_ms / 1e3) / 1e12 / bf16_sus,
                                # on the FLOP the MMAs issue (MLA: each CTA of a pair computes
                                # the whole score)
                                "issued_flop_per_launch": attn_issued,
                                "issued_frac": attn_issued / (attn_avg_ms / 1e3) / 1e12 / bf16_sus},
                     "eager_launch_ms": eager_launch_ms,
                     "timing": ("graph-replayed decode loop / steps" if graph is not None
                                else "CUDA events around each eager launch")},
            "full_kv": full,
            "speedup_vs_full_kv": (B * D * world / (dec_ms / 1e3)) / full["decode_tok_s"] if full else None,
            "cache_bytes": snap.cache_bytes(cfg, B),
            "cache_write": {"ms": stage_ms["write"], "bytes_per_seq": cache_write_bytes,
                            "hbm_gbs": cache_write_bytes / (stage_ms["write"] / 1e3) / 1e9,
                            "frac": cache_write_bytes / (stage_ms["write"] / 1e3) / 1e9 / hbm_peak},
            "roofline": {"bound": "hbm", "kernel": decode_kernel_name(wl),
                         "achieved": attn_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": attn_gbs / hbm_peak, "peak_source": peak_kind,
                         "traffic": traffic_record(wl.name)},
            "compress_roofline": compress_roofline,
            "prefill": prefill,
            "prefill_overhead_frac": prefill["overhead_frac"] if prefill else None,
            "gpu_launches": per_step_launches * steps,
        },
    }
    del cache
    return res


def decode_launches_per_step(wl, splits):
    """Kernels one snap_decode_step launches: GQA one (ring append, attention and split
    merge fused); MLA the attention (with the append) plus the merge when it splits."""
    if wl.layout == 0:
        return 1
    return 2 if splits > 1 else 1


def decode_kernel_name(wl):
    if wl.layout == 0:
        return "gqa_decode_kernel = snap_decode_step (ring append + split-KV attention + split merge), per launch"
    return "mla_decode_tc_kernel in snap_decode_step (ring append + split-KV attention; merge kernel after), per step"


SUB_WORKLOADS = ["gqa_2k_tiny", "gqa_16k32k_b8", "mla_128k_b8", "gqa_mixed_b64"]


def run_ours(args):
    import torch
    import torch.distributed as dist

    from fixed_size_kv_gb300 import inputs, snap

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    snap.load(build_if_missing=True)

    wl = inputs.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.replace(batch=args.batch)
    stream = torch.cuda.Stream(device=dev)
    r = measure(wl, args, args.steps, args.warmup, dev, stream, world, rank)
    B, lengths = r["B"], r["lengths"]

    # ---------------------------------------------------------------- end to end
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, lengths, r["pre"], r["q_all"], r["k_all"], r["v_all"], r["cfg"], dev, stream,
                      world, lambda x: max_over_ranks(x, world, dev))

    # ---------------------------------------------------------------- CPU oracle sample
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(wl, lengths, r["pre"], r["q_all"], r["k_all"], r["v_all"])
    for k in ("pre", "q_all", "k_all", "v_all"):
        r[k] = None
    torch.cuda.empty_cache()

    # ---------------------------------------------------------------- the other workloads, briefly
    workloads = None
    if not args.no_workloads and not args.batch and args.workload == "gqa_128k_b16":
        workloads = {}
        for name in SUB_WORKLOADS:
            swl = inputs.WORKLOADS[name]
            if swl.arrival_every > 0:
                workloads[name] = mixed_batch(swl, args, dev, world, full_run=False)
            else:
                sr = measure(swl, args, 2, 3, dev, stream, world, rank, full_run=False)
                workloads[name] = {"config": workload_config(swl, sr["B"], sr["lengths"], world),
                                   "steps": 2, "warmup": 3, "tok_s": sr["value"], "ms_per_step": sr["ms_per_step"],
                                   "decode_splits": sr["splits"], **sr["fields"]}
                del sr
            torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    config = workload_config(wl, B, lengths, world)
    if r["flush"]:
        config["l2"] = f"L2 flushed before each step ({2 * L2_BYTES >> 20} MiB write)"
    line = {
        "metric": METRIC,
        "value": r["value"],
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": r["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config,
        "launch": {"decode": "cuda graph" if r["graph"] else "eager", "decode_splits": r["splits"]},
        **r["fields"],
        "cpu_baseline": cpu,
        "e2e": e2e,
        "workloads": workloads,
        "clocks": r["clk"],
        "wall_s": r["t_wall"],
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# source file of each decode-attention kernel whose DRAM traffic is on record
KERNEL_SOURCES = {"gqa_decode_kernel": "k_decode.cu", "mla_decode_tc_kernel": "k_decode_mla_tc.cu"}


def traffic_record(workload):
    """DRAM bytes per decode-attention launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_attn_traffic.txt")
    try:
        for line in open(path):
            parts = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
            if parts.get("workload") != workload or parts.get("kernel") not in KERNEL_SOURCES:
                continue
            src = os.path.join(ROOT, "fixed_size_kv_gb300", "csrc", KERNEL_SOURCES[parts["kernel"]])
            digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
            if parts.get("src") == digest:
                return float(parts["bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def run_e2e(args, wl, lengths, pre, q_all, k_all, v_all, cfg, dev, stream, world, reduce_max):
    """The same job through the public API with pinned HOST inputs: every step copies
    its prompts and every decode step's q/k/v to the device and reads every decode output
    back, all inside the timed region.  The copies run on a second stream into two sets
    of device buffers: step i+1's inputs upload while step i computes (the first step's
    upload is not hidden), and within a step each compression waits for its own prompt
    only.  The outputs of a step's decode steps come back in one copy on the copy stream,
    overlapping the next step; the timed region ends when the last step's are on the host."""
    import torch
    from fixed_size_kv_gb300 import snap
    B, D = wl.batch, wl.decode_steps
    hK = [p.K.to("cpu").pin_memory() for p in pre]
    hV = [p.V.to("cpu").pin_memory() if p.V is not None else None for p in pre]
    hQ = [p.Q.to("cpu").pin_memory() for p in pre]
    hq, hk = q_all.to("cpu").pin_memory(), k_all.to("cpu").pin_memory()
    hv = v_all.to("cpu").pin_memory() if v_all is not None else None

    def buffers():
        return {"K": [torch.empty_like(p.K) for p in pre],
                "V": [torch.empty_like(p.V) if p.V is not None else None for p in pre],
                "Q": [torch.empty_like(p.Q) for p in pre],
                "q": torch.empty_like(q_all), "k": torch.empty_like(k_all),
                "v": torch.empty_like(v_all) if v_all is not None else None,
                "out": torch.empty((D, B, wl.n_q_heads, wl.d_v), dtype=torch.float32, device=dev),
                "hout": torch.empty((D, B, wl.n_q_heads, wl.d_v), dtype=torch.float32).pin_memory(),
                "up": [torch.cuda.Event() for _ in range(B)], "up_dec": torch.cuda.Event(),
                "done": torch.cuda.Event(), "read": torch.cuda.Event(), "used": False, "read_pending": False}

    sets = [buffers(), buffers()]
    cache = snap.SnapCache(cfg, max_batch=B, max_prompt=max(lengths), max_n=B, device=dev, stream=stream)
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    h2d = sum(x.numel() * 2 for x in hK + hQ) + sum(x.numel() * 2 for x in hV if x is not None)
    h2d += (q_all.numel() + k_all.numel() + (v_all.numel() if v_all is not None else 0)) * 2
    d2h = D * B * wl.n_q_heads * wl.d_v * 4
    copy = torch.cuda.Stream(device=dev)

    def upload(st):
        if st["used"]:
            copy.wait_event(st["done"])     # the step that last used this set has finished
        st["used"] = True
        with torch.cuda.stream(copy):
            for b in range(B):
                st["K"][b].copy_(hK[b], non_blocking=True)
                if st["V"][b] is not None:
                    st["V"][b].copy_(hV[b], non_blocking=True)
                st["Q"][b].copy_(hQ[b], non_blocking=True)
                st["up"][b].record(copy)
            st["q"].copy_(hq, non_blocking=True)
            st["k"].copy_(hk, non_blocking=True)
            if st["v"] is not None:
                st["v"].copy_(hv, non_blocking=True)
            st["up_dec"].record(copy)

    def compute(st):
        if st["read_pending"]:
            stream.wait_event(st["read"])   # this set's previous outputs are on the host
        for b in range(B):
            stream.wait_event(st["up"][b])
            cache.compress(b, st["K"][b], st["V"][b], st["Q"][b], stream=stream)
        stream.wait_event(st["up_dec"])
        for t in range(D):
            cache.decode_step(slots, st["q"][t], st["k"][t], st["v"][t] if st["v"] is not None else None,
                              out=st["out"][t], stream=stream)
        st["done"].record(stream)
        # the step's outputs go back on the copy stream, overlapping the next step
        copy.wait_event(st["done"])
        with torch.cuda.stream(copy):
            st["hout"].copy_(st["out"], non_blocking=True)
        st["read"].record(copy)
        st["read_pending"] = True

    # untimed warm-up of both buffer sets
    for w in range(2):
        upload(sets[w])
        compute(sets[w])
    stream.synchronize()
    copy.synchronize()
    # this host's pinned host->device bandwidth, on one prompt (explains the e2e number)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(copy)
    with torch.cuda.stream(copy):
        sets[0]["K"][0].copy_(hK[0], non_blocking=True)
    c1.record(copy)
    copy.synchronize()
    h2d_gbs = hK[0].numel() * 2 / (c0.elapsed_time(c1) / 1e3) / 1e9
    steps = max(1, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy.wait_stream(stream)                # the timed region starts before the first upload
    upload(sets[0])
    for i in range(steps):
        if i + 1 < steps:
            upload(sets[(i + 1) % 2])
        compute(sets[i % 2])
    stream.wait_stream(copy)                # the last step's outputs are on the host
    e1.record(stream)
    stream.synchronize()
    ms = reduce_max(e0.elapsed_time(e1))
    del cache
    return {"value": B * D * steps * world / (ms / 1e3), "unit": "tok/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "overlap": "double-buffered inputs",
            "h2d_gbs_one_copy": h2d_gbs}


# ----------------------------------------------------------------------------- oracle
def cpu_sample(wl, lengths, K0, V0, Q0, q1, k1, v1, threads=1):
    """Times the CPU oracle on a bounded sample and scales it to the whole step.

    Sample: the window scoring, max-pool and top-K of sequence 0's KV heads over a
    prompt prefix of at most 16384 tokens (the compression's cost, linear in prompt
    length), and one decode step (append + attention) over a cache of the workload's
    size.  threads == 1: one KV head's scoring and one sequence's decode, on one core.
    threads > 1: every KV head of sequence 0 scored at once and the decode of
    min(batch, threads) sequences at once, one oracle call per thread (the C oracle
    releases the GIL; the work per call is unchanged)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    B, D = wl.batch, wl.decode_steps
    oracle.build()
    S_full = lengths[0]
    S_s = min(S_full, 16384)
    G = wl.G
    one = wl.replace(n_q_heads=G, n_kv_heads=1)
    ocfg1 = oracle.Config(**one.config_kwargs())
    # scoring units: (KV head, group of query heads); MLA's 128 heads in groups of 8
    grp = 8 if G > 8 else G
    units = [(h, g0) for h in range(wl.n_kv_heads) for g0 in range(0, G, grp)]
    if threads == 1:
        units = units[:max(1, G // grp)]         # one KV head: all its query heads
    sub = oracle.Config(**wl.replace(n_q_heads=grp, n_kv_heads=1).config_kwargs())
    heads_per_unit_set = len(units) * grp / G       # KV heads covered by the sample
    K1 = [K0[:S_s, h:h + 1].contiguous() for h in range(wl.n_kv_heads)]

    def score(u):
        h, g0 = u
        return oracle.window_scores(sub, K1[h], Q0[:, h * G + g0:h * G + g0 + grp].contiguous())[1][0]

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        cols = list(ex.map(score, units))
    col = sum(cols[:max(1, G // grp)])
    pooled = oracle.maxpool(col[:S_s - wl.W], wl.P)
    oracle.select(pooled, wl.L_sink, S_s - wl.W, max(1, wl.K * S_s // S_full))  # K scaled to the prefix
    t_c = time.perf_counter() - t0
    compress_full = t_c * (S_full / S_s) * (wl.n_kv_heads / heads_per_unit_set) * B
    # decode: caches of the workload's size built by layout alone (no scoring needed)
    ocfg = oracle.Config(**wl.config_kwargs())
    keep = wl.L_sink + wl.K + wl.L_recent
    Kc = K0[:keep].contiguous()
    Vc = V0[:keep].contiguous() if V0 is not None else None
    n_dec = 1 if threads == 1 else min(B, threads)
    caches = [oracle.compress(ocfg, Kc, Vc, Q0) for _ in range(n_dec)]

    def dec(c):
        oracle.append(c, k1, v1)
        oracle.decode_attn(c, q1)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(dec, caches))
    t_d = time.perf_counter() - t0
    decode_full = t_d * (B / n_dec) * D
    total = compress_full + decode_full
    return {"value": B * D / total, "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": (f"window scoring + pool + top-K of {heads_per_unit_set:g} KV head(s) of sequence 0 over a "
                       f"{S_s}-token prefix ({t_c:.2f}s, scaled x{S_full / S_s:.0f} length, "
                       f"x{wl.n_kv_heads / heads_per_unit_set * B:g} heads/seqs) + 1 decode step of {n_dec} "
                       f"sequence(s) ({t_d:.2f}s, scaled x{B / n_dec * D:g}); C oracle in fp64 on {threads} "
                       f"thread(s)"),
            "seconds": t_c + t_d, "compress_s_est": compress_full, "decode_s_est": decode_full}


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def cpu_baseline(wl, lengths, pre, q_all, k_all, v_all):
    """The oracle on every host core (the reported baseline), with the one-core run beside it."""
    p0 = pre[0]
    args = (wl, lengths, p0.K.cpu(), p0.V.cpu() if p0.V is not None else None, p0.Q.cpu(),
            q_all[0, 0].cpu(), k_all[0, 0].cpu(), v_all[0, 0].cpu() if v_all is not None else None)
    n = host_cores()
    multi = cpu_sample(*args, threads=n)
    single = cpu_sample(*args, threads=1)
    multi["host_cores"] = n
    multi["single_thread"] = {"value": single["value"], "cores": 1, "sample": single["sample"]}
    return multi


def run_reference(args):
    """The CPU oracle as the reference arm: each step is one bounded sample of the
    workload (see cpu_sample), timed on every host core, scaled to tok/s."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from fixed_size_kv_gb300 import inputs
    wl = inputs.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.replace(batch=args.batch)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    lengths = inputs.prompt_lengths(wl, args.seed)
    S_s = min(lengths[0], 16384)
    keep = max(S_s, wl.C)
    pre = inputs.gen_prefill(wl, keep, seed=args.seed, seq=0)
    tok = inputs.gen_decode(wl, 1, step=0, seed=args.seed)
    n = host_cores()
    vals, secs = [], []
    for i in range(args.warmup + args.steps):
        r = cpu_sample(wl, [lengths[0]], pre.K, pre.V, pre.Q, tok.q[0], tok.k[0],
                       tok.v[0] if tok.v is not None else None, threads=n)
        if i >= args.warmup:
            vals.append(r["value"])
            secs.append(r["seconds"])
    value = statistics.mean(vals)
    B, D = wl.batch, wl.decode_steps
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": B * D / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(wl, B, lengths, world),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": n, "host_cores": n, "kind": "oracle",
                             "sample": r["sample"]},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "sample_seconds_per_step": statistics.mean(secs)}
    print(json.dumps(line), flush=True)


def mixed_batch(wl, args, dev, world, full_run=True):
    """Continuous batch with arrivals (the 64-slot mixed workload): every
    `arrival_every` decode steps, the slots whose request finished take new requests,
    which are compressed on a second stream while the first keeps decoding the
    others; a new request joins the decode batch at the next arrival boundary.
    value = decoded tokens / device time of the whole run (compressions included).
    Returns the fields of the workload's JSON record."""
    import torch
    from fixed_size_kv_gb300 import inputs, snap

    B, D, every = wl.batch, wl.decode_steps, wl.arrival_every
    sa, sb = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    n_req = B * 16
    lengths = inputs.prompt_lengths(wl, args.seed, n=n_req)
    outs = inputs.output_lengths(args.seed, n_req)
    # a pool of prompt buffers at the longest length; request i reads a prefix of pool[i % NP]
    NP = 8
    with torch.cuda.stream(sa):
        pool = [inputs.gen_prefill(wl, wl.prompt_max, seed=args.seed, seq=i, device=dev) for i in range(NP)]
        toks = [inputs.gen_decode(wl, B, step=t, seed=args.seed, device=dev) for t in range(64)]
    sa.synchronize()
    cfg = snap.make_config(**wl.config_kwargs())
    cache = snap.SnapCache(cfg, max_batch=B, max_prompt=wl.prompt_max, max_n=B, device=dev, stream=sa)
    out = torch.empty((B, wl.n_q_heads, wl.d_v), dtype=torch.float32, device=dev)

    # valid cache slots of each slot's request: min(S, C) (every prompt covers sinks + ring)
    valid = [0] * B
    row_bytes = wl.n_kv_heads * (wl.d_qk + (wl.d_v if wl.layout == 0 else 0)) * 2
    tok_bytes = wl.n_q_heads * (wl.d_qk * 2 + wl.d_v * 4)

    def compress(slot, req, stream):
        p = pool[req % NP]
        S = lengths[req]
        valid[slot] = min(S, wl.C)
        cache.compress(slot, p.K[:S], p.V[:S] if p.V is not None else None, p.Q, stream=stream)

    def run(steps, timed):
        next_req = 0
        remaining = [0] * B
        for slot in range(B):                    # initial fill, before the clock starts
            compress(slot, next_req, sa)
            remaining[slot] = outs[next_req]
            next_req += 1
        sa.synchronize()
        pending = {}                             # slot -> remaining, joining at the next boundary
        ev_b = None
        tokens = 0
        n_compress = 0
        dec_bytes = 0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(sa)
        active = [s for s in range(B) if remaining[s] > 0]
        slots_t = torch.tensor(active, dtype=torch.int32).to(dev, non_blocking=True)
        for t in range(steps):
            if t > 0 and t % every == 0:
                if pending:
                    sa.wait_event(ev_b)
                    for s, r in pending.items():
                        remaining[s] = r
                    pending = {}
                free = [s for s in range(B) if remaining[s] == 0]
                if free:
                    for s in free:
                        compress(s, next_req % n_req, sb)
                        pending[s] = outs[next_req % n_req]
                        next_req += 1
                        n_compress += 1
                    ev_b = torch.cuda.Event()
                    ev_b.record(sb)
                active = [s for s in range(B) if remaining[s] > 0]
                with torch.cuda.stream(sa):
                    slots_t = torch.tensor(active, dtype=torch.int32).to(dev, non_blocking=True)
            n = len(active)
            if n:
                tk = toks[t % 64]
                cache.decode_step(slots_t, tk.q[:n], tk.k[:n], tk.v[:n] if tk.v is not None else None,
                                  out=out[:n], stream=sa)
                tokens += n
                dec_bytes += sum(valid[s] for s in active) * row_bytes + n * tok_bytes
                done = False
                for s in active:
                    remaining[s] -= 1
                    done |= remaining[s] == 0
                if done:
                    active = [s for s in active if remaining[s] > 0]
                    with torch.cuda.stream(sa):
                        slots_t = torch.tensor(active, dtype=torch.int32).to(dev, non_blocking=True)
        e1.record(sa)
        torch.cuda.synchronize(dev)
        return tokens, e0.elapsed_time(e1), n_compress, dec_bytes

    run(min(D, 64), False)                       # warm-up
    clocks = ClockSampler(dev.index or 0) if full_run else None
    if clocks:
        clocks.start()
    tokens, ms, n_compress, dec_bytes = run(D, True)
    hbm_peak, _, _, peak_kind = peaks()
    achieved = dec_bytes / (ms / 1e3) / 1e9
    clk = clocks.stop() if clocks else None
    st = cache.check_device(sa)
    if st != snap.SNAP_OK:
        raise RuntimeError(f"device status: {snap.status_string(st)}")
    del cache, pool, toks
    return {"config": {"workload": wl.name, "slots": B, "prompt_len": f"U[{wl.prompt_min},{wl.prompt_max}]",
                       "decode_steps": D, "arrival_every": every,
                       "cache": f"{wl.L_sink}+{wl.K}+{wl.L_recent}={wl.C}", "W": wl.W, "P": wl.P,
                       "heads": f"{wl.n_q_heads}/{wl.n_kv_heads}x{wl.d_qk}",
                       "output_len": "U[32,1024]", "prompt_pool": NP, "parallelism": f"replicas x{world}"},
            "tok_s": tokens / (ms / 1e3), "ms": ms, "ms_per_step": ms / D,
            "decoded_tokens": tokens, "arrivals_compressed": n_compress,
            "roofline": {"bound": "hbm", "kernel": "snap_decode_step over the run (compressions overlap on a "
                         "second stream, so this is a lower bound)", "achieved": achieved, "peak": hbm_peak,
                         "unit": "GB/s", "frac": achieved / hbm_peak, "peak_source": peak_kind,
                         "traffic": None, "decode_bytes": dec_bytes},
            "clocks": clk}


def run_mixed(args):
    """The mixed continuous batch as its own JSON line (python bench.py --workload gqa_mixed_b64)."""
    import torch
    from fixed_size_kv_gb300 import inputs, snap
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    snap.load(build_if_missing=True)
    wl = inputs.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.replace(batch=args.batch)
    r = mixed_batch(wl, args, dev, 1)
    line = {"metric": METRIC, "value": r["tok_s"], "unit": "tok/s", "n_gpus": 1, "steps": wl.decode_steps,
            "warmup": 1, "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": r["config"],
            "decoded_tokens": r["decoded_tokens"], "arrivals_compressed": r["arrivals_compressed"],
            "roofline": r["roofline"], "clocks": r["clocks"]}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- extra modes
def _decode_rate(cache, wl, B, S_list, seed, dev, stream, steps=32, warm=4):
    """Decode tok/s of B sequences already compressed in `cache`: `steps` decode steps
    replayed as one CUDA graph after `warm` eager ones (inputs resident on the device)."""
    import torch
    from fixed_size_kv_gb300 import inputs
    slots = torch.arange(B, dtype=torch.int32, device=dev)
    toks = [inputs.gen_decode(wl, B, step=t, seed=seed, device=dev) for t in range(steps)]
    out = torch.empty((B, wl.n_q_heads, wl.d_v), dtype=torch.float32, device=dev)
    for t in range(warm):
        cache.decode_step(slots, toks[t].q, toks[t].k, toks[t].v, out=out, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for t in range(steps):
            cache.decode_step(slots, toks[t].q, toks[t].k, toks[t].v, out=out, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        graph.replay()
    e1.record(stream)
    stream.synchronize()
    return B * steps / (e0.elapsed_time(e1) / 1e3)


def _fill(cache, pool, B, stream):
    for b in range(B):
        p = pool[b % len(pool)]
        cache.compress(b, p.K, p.V, p.Q, stream=stream)
    stream.synchronize()


def run_capacity(args):
    """Capacity (the pages' "Max Batch Size Unlocked"): at a fixed HBM budget for the
    cache, the largest batch of the workload's prompt length for the fixed-size cache
    and for full KV, and the decode tok/s measured at that batch.  Sequences are filled
    from a pool of 4 seeded prompts (the decode cost depends on the cache, not on which
    prompt filled it)."""
    import torch
    from fixed_size_kv_gb300 import inputs, snap
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    snap.load(build_if_missing=True)
    stream = torch.cuda.Stream(device=dev)
    wl = inputs.WORKLOADS[args.workload]
    S = wl.prompt_max
    budget = int(args.capacity * (1 << 30))
    with torch.cuda.stream(stream):
        pool = [inputs.gen_prefill(wl, S, seed=args.seed, seq=i, device=dev) for i in range(4)]
    stream.synchronize()
    rates = {}
    for kind in ("fixed", "full_kv"):
        kwl = wl if kind == "fixed" else wl.replace(L_sink=0, K=0, L_recent=S + 64)
        cfg = snap.make_config(**kwl.config_kwargs())
        per_seq = snap.cache_bytes(cfg, 2) - snap.cache_bytes(cfg, 1)
        B = budget // per_seq
        if B < 1:
            print(json.dumps({"mode": "capacity", "cache": kind, "max_batch": 0, "budget_gib": args.capacity}))
            continue
        cache = snap.SnapCache(cfg, max_batch=B, max_prompt=S, max_n=B, device=dev, stream=stream)
        _fill(cache, pool, B, stream)
        rate = _decode_rate(cache, kwl, B, [S] * B, args.seed, dev, stream)
        rates[kind] = rate
        print(json.dumps({"mode": "capacity", "workload": wl.name, "cache": kind, "budget_gib": args.capacity,
                          "prompt_len": S, "cache_slots": kwl.C, "bytes_per_seq": per_seq, "max_batch": int(B),
                          "decode_tok_s": rate, "data": "synthetic"}), flush=True)
        del cache
        torch.cuda.empty_cache()
    if len(rates) == 2:
        print(json.dumps({"mode": "capacity", "workload": wl.name, "budget_gib": args.capacity,
                          "throughput_ratio_fixed_over_full": rates["fixed"] / rates["full_kv"]}), flush=True)


def run_sweep(args):
    """Speed sweep: decode tok/s of a batch of 16 GQA (Llama-3.1-8B shape) sequences
    (a) over context length with the cache at a quarter of the prompt (4 sinks, half
    recent) against full KV (the pages' "Throughput by Context Length"), and (b) over the
    cache composition (L_sink, K, L_recent) at 128k, K = 0 being StreamingLLM alone (the
    axes of the pages' hyperparameter ablation)."""
    import torch
    from fixed_size_kv_gb300 import inputs, snap
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    snap.load(build_if_missing=True)
    stream = torch.cuda.Stream(device=dev)
    base = inputs.WORKLOADS["gqa_128k_b16"]
    B = base.batch

    def measure(wl, S, pool, tag):
        cfg = snap.make_config(**wl.config_kwargs())
        cache = snap.SnapCache(cfg, max_batch=B, max_prompt=S, max_n=B, device=dev, stream=stream)
        _fill(cache, pool, B, stream)
        rate = _decode_rate(cache, wl, B, [S] * B, args.seed, dev, stream)
        del cache
        torch.cuda.empty_cache()
        return rate

    for S in (32768, 65536, 131072):
        with torch.cuda.stream(stream):
            pool = [inputs.gen_prefill(base, S, seed=args.seed, seq=i, device=dev) for i in range(B)]
        stream.synchronize()
        C = S // 4
        fixed = base.replace(L_sink=4, K=C // 2 - 4, L_recent=C // 2)
        r_fixed = measure(fixed, S, pool, "fixed")
        r_full = measure(base.replace(L_sink=0, K=0, L_recent=S + 64), S, pool, "full")
        print(json.dumps({"mode": "sweep", "axis": "context", "prompt_len": S, "batch": B,
                          "cache": f"4+{C // 2 - 4}+{C // 2}={C}", "decode_tok_s": r_fixed,
                          "full_kv_decode_tok_s": r_full, "speedup": r_fixed / r_full}), flush=True)
    S = 131072
    for (ls, k, lr) in ((4, 16380, 16384), (0, 16384, 16384), (64, 16320, 16384), (4, 8188, 24576),
                        (4, 24572, 8192), (4, 0, 32764)):
        wl = base.replace(L_sink=ls, K=k, L_recent=lr)
        r = measure(wl, S, pool, "mix")
        print(json.dumps({"mode": "sweep", "axis": "composition", "prompt_len": S, "batch": B,
                          "L_sink": ls, "K": k, "L_recent": lr, "decode_tok_s": r,
                          "note": "StreamingLLM only" if k == 0 else ""}), flush=True)


def run_prefill_only(args):
    """The prefill attention alone (profiling): snap_prefill_attn of one prompt of
    --prefill-only tokens of the workload (GQA), with the window rows' LSE, run three
    times; prints the CUDA-event time of the last two."""
    import torch
    from fixed_size_kv_gb300 import inputs, snap
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    snap.load(build_if_missing=True)
    wl = inputs.WORKLOADS[args.workload]
    S = args.prefill_only
    pre = inputs.gen_prefill(wl, S, seed=args.seed, device=dev)
    Q = inputs.gen_prompt_queries(wl, pre, seed=args.seed, device=dev)
    cache = snap.SnapCache(snap.make_config(**wl.config_kwargs()), max_batch=1, max_prompt=1, device=dev)
    lse = torch.empty((wl.W, wl.n_q_heads), dtype=torch.float32, device=dev)
    O = torch.empty_like(Q)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
    for a, b in ev:
        a.record()
        cache.prefill_attn(Q, pre.K, pre.V, O=O, lse_obs=lse)
        b.record()
    torch.cuda.synchronize()
    if cache.check_device() != snap.SNAP_OK:
        raise RuntimeError("device status after the prefill")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev[1:])
    flop = 2.0 * wl.n_q_heads * wl.d_qk * S * (S + 1)
    print(json.dumps({"mode": "prefill", "workload": wl.name, "prompt_len": S, "ms": ms,
                      "tflops": flop / (ms / 1e3) / 1e12}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.prefill_only:
        run_prefill_only(args)
        return
    if args.capacity > 0:
        run_capacity(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    from fixed_size_kv_gb300 import inputs
    if inputs.WORKLOADS[args.workload].arrival_every > 0:
        run_mixed(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
