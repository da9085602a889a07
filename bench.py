#!/usr/bin/env python
"""Benchmark of one fused DSA decode step on GB300.

Workload (default): batch 32 requests, 131072-token context each, indexer
64 heads x 128 dims in fp8 e4m3 with per-row scales, top-k 2048, sparse MLA
with 64 heads over 576-wide bf16 latent rows (Dv 512).  Synthetic, seeded
inputs.  One step = index score -> top-k -> sparse MLA (-> split combine) for
all 32 requests, through the C ABI entry point dsa_decode.

Timing: W warm-up steps, then K steps each bracketed by CUDA events on the
launching stream; between timed steps a 256 MiB buffer is written and a
second 256 MiB buffer is read, so the L2 holds neither step inputs nor dirty
lines whose write-back would be charged to the next step (the flush is
outside the events).  A GPU-side sleep ahead of each timed loop lets the host
queue its launches first, so host launch latency stays out of the events.
Beside these cold steps the line reports the same step warm (back to back,
no flush: `warm_us`) and captured once into a CUDA graph (`graph_us`, cold).
Multi-GPU runs (torchrun) are independent replicas: the path does not shard
across GPUs.

Prints one JSON line.  `--impl reference` times the CPU oracle instead (the
reference arm), on a bounded sample of the same workload.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA decode/prefill µs per step (score+topk+attn); % of GB300 HBM roofline"
UNIT = "us/step"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


def workload_config(B, N, k):
    return {"workload": "decode_b%d_n%d" % (B, N), "batch": B, "context": N, "topk": k,
            "heads": 64, "index_heads": 64, "index_dim": 128, "index_dtype": "fp8_e4m3",
            "kv_format": "bf16 latent 576 (Dv 512)",
            "l2": "flushed between timed steps (256 MiB write, then 256 MiB read); index-k sweep 553 MB > L2",
            "parallelism": "replicas"}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- ranks

def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over the ranks of the default process group (x itself
    for one rank).  Each rank serves its own batch of requests (weak
    scaling), so a step of the whole job takes as long as its slowest rank."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Seed of the synthetic request batch rank `rank` serves: the ranks'
    batches are different requests, not copies."""
    return int(rank)


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world):
    import torch
    from deepseek_sparse_attention_index_gb300 import build as B
    from deepseek_sparse_attention_index_gb300 import inputs as I
    from deepseek_sparse_attention_index_gb300 import ops

    if rank == 0 or not os.path.exists(B.LIB):
        B.build()
    if world > 1:
        torch.distributed.barrier()
    ops.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    Bsz, N, k = args.batch, args.context, 2048
    case = I.decode_sweep(Bsz, N, device=dev, seed=rank_seed(rank))
    ind = case.indexer
    H, Dv = case.H, case.Dv
    ws = ops.workspace(ops.dsa_decode_workspace_size(Bsz, N, k, H, Dv), dev)
    idx_out = torch.empty((Bsz, k), dtype=torch.int32, device=dev)
    out = torch.empty((Bsz, H, Dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Bsz, H), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def l2_flush(i):
        flush.fill_(i & 0xff)
        flush_rd.sum()
    stream = torch.cuda.current_stream()

    def step():
        ops.decode_case(case, ws=ws, idx_out=idx_out, out=out, lse=lse)

    # warm-up iterations are the timed ones untimed: the flush included (the
    # first launch of its kernels costs ~0.1 ms, which must not land in a
    # timed step)
    for i in range(args.warmup):
        l2_flush(i)
        step()
    torch.cuda.synchronize()

    # ---- timed region: K fused steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    torch.cuda._sleep(50_000_000)   # ~25 ms of GPU time while the host queues the steps
    for i in range(args.steps):
        l2_flush(i)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    us_per_step = total_ms * 1000.0 / args.steps

    # ---- beside the cold steps (the timed region above): the same fused step
    # back to back without the L2 flush (warm), and the step captured once
    # into a CUDA graph, each replay between events after an L2 flush
    warm_us = statistics.median(_timed(step, args.steps, 1, lambda i: None))
    graph_dev_us = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        gdev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gdev):
            step()
        graph_dev_us = statistics.median(_timed(gdev.replay, args.steps, 2, l2_flush))
        del gdev
    except RuntimeError as exc:    # reported, not fatal
        graph_dev_us = "capture failed: %s" % str(exc).splitlines()[0][:120]

    # ---- staged pass: the three stages as separate entry points, events around each
    rs = case.slot_base
    re = (case.slot_base + case.seq_lens).contiguous()
    ld = (N + 3) // 4 * 4
    scores = torch.empty((Bsz, ld), dtype=torch.float32, device=dev)
    tws = ops.workspace(ops.dsa_topk_workspace_size(Bsz, N, k), dev)
    mws = ops.workspace(ops.dsa_sparse_mla_workspace_size(Bsz, H, Dv, k, 0), dev)
    stage_ms = {"index_score": [], "topk": [], "sparse_mla": []}
    n_stage = max(3, min(args.steps, 10))
    stage_ev = []
    torch.cuda._sleep(50_000_000)
    for i in range(n_stage):
        l2_flush(i)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        ops.dsa_index_score(ind["q_idx"], ind["idx_dtype"], ind["q_scale"], ind["k_idx"],
                            ind["k_scale"], ind["w"], rs, re, N, scores=scores)
        e[1].record(stream)
        ops.dsa_topk(scores, case.seq_lens, k, N, index_base=case.slot_base, idx=idx_out, ws=tws)
        e[2].record(stream)
        ops.dsa_sparse_mla_fwd(case.q, case.softmax_scale, case.kv, idx_out, out=out, lse=lse,
                               ws=mws)
        e[3].record(stream)
        stage_ev.append(e)
    torch.cuda.synchronize()
    for e in stage_ev:
        stage_ms["index_score"].append(e[0].elapsed_time(e[1]))
        stage_ms["topk"].append(e[1].elapsed_time(e[2]))
        stage_ms["sparse_mla"].append(e[2].elapsed_time(e[3]))
    stage_us = {s: 1000.0 * statistics.median(v) for s, v in stage_ms.items()}

    # algorithmic bytes (per launch) of the dominant kernel, the index score:
    # per key 128 B fp8 + 4 B scale; per request the query's 64 x 128 fp8
    # head rows, their 64 scales and 64 weights (8704 B).  The score row the
    # kernel writes (4 B a key, re-read from L2 by the top-k) is workspace
    # traffic, not an input or output of the method: it is reported beside
    # the figure, not in it.
    hbm_gbs, _, peak_kind = measured_peaks()
    q_idx_bytes = 64 * 128 + 64 * 4 + 64 * 4
    idx_bytes = Bsz * N * (128 + 4) + Bsz * q_idx_bytes
    score_bytes = Bsz * N * 4
    idx_gbs = idx_bytes / (stage_us["index_score"] * 1e-6) / 1e9
    # whole-step algorithmic bytes: keys and scales, the gathered KV rows,
    # the indexer query, q, out and lse
    rows = Bsz * min(N, k)
    step_bytes = idx_bytes + rows * 1152 + Bsz * H * (576 * 2 + Dv * 2 + 4)
    step_gbs = step_bytes / (us_per_step * 1e-6) / 1e9
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "index_score_traffic.json")
    if os.path.exists(tfile):
        # the ncu counters hold only for the kernel source they were taken on
        import hashlib
        with open(tfile) as f:
            tr = json.load(f)
        h = hashlib.sha256(b"".join(open(os.path.join(ROOT, p), "rb").read()
                                    for p in tr["source_files"])).hexdigest()[:16]
        if h == tr.get("source_sha256_16"):
            traffic = tr.get("bytes_per_launch_full_size")

    # ---- e2e: host buffers through the C-ABI host-buffer entry point
    # (dsa_decode_host): per-step inputs copied in and results copied out
    # inside the call, on the library's streams
    pin = lambda t: t.detach().cpu().pin_memory()
    h_in = {"q_idx": pin(ind["q_idx"]), "q_scale": pin(ind["q_scale"]), "w": pin(ind["w"]),
            "q": pin(case.q), "seq_lens": pin(case.seq_lens), "slot_base": pin(case.slot_base)}
    h_out = {"idx": torch.empty_like(idx_out, device="cpu").pin_memory(),
             "out": torch.empty_like(out, device="cpu").pin_memory(),
             "lse": torch.empty_like(lse, device="cpu").pin_memory()}
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    hws = ops.workspace(ops.dsa_decode_host_workspace_size(
        Bsz, N, k, case.H_I, case.d_idx, ind["idx_dtype"], H, case.D, Dv), dev)

    def e2e_step():
        ops.dsa_decode_host(h_in["q_idx"], ind["idx_dtype"], h_in["q_scale"], ind["k_idx"],
                            ind["k_scale"], h_in["w"], h_in["seq_lens"], h_in["slot_base"], N, k,
                            h_in["q"], case.softmax_scale, case.kv, idx_out=h_out["idx"],
                            out=h_out["out"], lse=h_out["lse"], ws=hws)

    for i in range(max(2, args.warmup)):
        l2_flush(i)
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(args.steps):
        l2_flush(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        torch.cuda.synchronize()
        e2e_ms.append((time.perf_counter() - t0) * 1000.0)
    e2e_us = max_over_ranks(1000.0 * statistics.mean(e2e_ms), world, dev)

    # ---- the same step through dsa_decode_graph: captured once on the same
    # pinned buffers, one graph launch per step (copies and kernels inside)
    graph_us, graph_err = None, None
    try:
        gstep = ops.DecodeGraph(h_in["q_idx"], ind["idx_dtype"], h_in["q_scale"], ind["k_idx"],
                                ind["k_scale"], h_in["w"], h_in["seq_lens"], h_in["slot_base"], N,
                                k, h_in["q"], case.softmax_scale, case.kv, idx_out=h_out["idx"],
                                out=h_out["out"], lse=h_out["lse"], ws=hws)
        for i in range(max(2, args.warmup)):
            l2_flush(i)
            gstep.launch()
        torch.cuda.synchronize()
        g_ms = []
        for i in range(args.steps):
            l2_flush(i)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            gstep.launch()
            torch.cuda.synchronize()
            g_ms.append((time.perf_counter() - t0) * 1000.0)
        gstep.close()
        graph_us = 1000.0 * statistics.mean(g_ms)
    except ops.DsaError as exc:     # reported, not fatal: the line keeps the direct-call e2e
        graph_err = str(exc)
    # every rank joins the reduction (a failed capture on any rank voids the graph number)
    graph_us = max_over_ranks(graph_us if graph_us is not None else 1e30, world, dev)
    if graph_us >= 1e29:
        graph_us = None

    splits = 1 if ops.dsa_sparse_mla_workspace_size(Bsz, H, Dv, k, 0) == 0 else 2
    launches_per_step = 1 + 1 + 1 + 1 + (1 if splits > 1 else 0)

    res = {
        "metric": METRIC, "value": round(us_per_step, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us_per_step / 1000, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 indexer + bf16 attention (fp32 accumulate)", "data": "synthetic",
        "config": workload_config(Bsz, N, k),
        "roofline": {"bound": "hbm", "kernel": "index_score", "achieved": round(idx_gbs, 1),
                     "peak": hbm_gbs, "peak_kind": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)",
                     "unit": "GB/s", "frac": round(idx_gbs / hbm_gbs, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": idx_bytes,
                     "score_write_bytes_per_launch": score_bytes,
                     "launch_us": round(stage_us["index_score"], 2)},
        "step_roofline": {"achieved_gbs": round(step_gbs, 1), "frac": round(step_gbs / hbm_gbs, 4),
                          "algorithmic_bytes_per_step": step_bytes},
        "stages_us": {s: round(v, 2) for s, v in stage_us.items()},
        "warm_us": round(warm_us, 3),
        "graph_us": round(graph_dev_us, 3) if isinstance(graph_dev_us, float) else graph_dev_us,
        # e2e: the step through the library's public API from pinned host
        # buffers -- the captured step (dsa_decode_graph, one launch a step,
        # the way a decode loop runs it) and, beside it, the direct call
        "e2e": {"value": round(graph_us if graph_us is not None else e2e_us, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "dsa_decode_graph" if graph_us is not None else "dsa_decode_host",
                "note": "per-step inputs from pinned host memory, results back to host memory, "
                        "the copies inside the timed step; the index-k cache and KV pool stay "
                        "resident in HBM as model state"},
        "e2e_direct": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "path": "dsa_decode_host",
                       "graph_error": graph_err},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }
    return res


# ---------------------------------------------------------------- other workloads

def _timed(fn, steps, warmup, flush_fn):
    """Device µs of fn() per call: W warm-up calls, then K calls each between
    CUDA events on the current stream, the L2 flushed before each (outside the
    events, and before each warm-up call too); all launches queued behind a
    GPU-side sleep."""
    import torch
    for i in range(warmup):
        flush_fn(i)
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = []
    torch.cuda._sleep(50_000_000)
    for i in range(steps):
        flush_fn(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    return [1000.0 * a.elapsed_time(b) for a, b in ev]


def run_workload(args):
    """Secondary measurements (one JSON line each): the other configurations
    of the scope table, timed like the default line.  Not the default line."""
    import torch
    from deepseek_sparse_attention_index_gb300 import build as B
    from deepseek_sparse_attention_index_gb300 import inputs as I
    from deepseek_sparse_attention_index_gb300 import ops
    B.build()
    ops.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm_gbs, bf16_tflops, peak_kind = measured_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def l2_flush(i):
        flush.fill_(i & 0xff)
        flush_rd.sum()

    clocks = ClockSampler(0)
    res = {"metric": METRIC, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
           "warmup": args.warmup, "higher_is_better": False, "scaling": "weak",
           "vs_baseline": None, "data": "synthetic", "e2e": None, "gpu_launches": None}
    w = args.workload
    if w == "bwd":
        # the attention's backward over a causal prefill's selections: T tokens,
        # 64 heads, k = 2048 bf16 rows each (the forward's lse as input)
        T, H = args.context, args.heads
        case = I.prefill_case([T], k=2048, H=H, device=dev)
        ind = case.indexer
        ld = (T + 3) // 4 * 4
        scores = torch.empty((T, ld), dtype=torch.float32, device=dev)
        rl = (case.row_end - case.row_start).contiguous()
        tws = ops.workspace(ops.dsa_topk_workspace_size(T, T, case.k), dev)
        idx = torch.empty((T, case.k), dtype=torch.int32, device=dev)
        ops.dsa_index_score_prefill(ind["q_idx"], ind["idx_dtype"], ind["q_scale"], ind["k_idx"],
                                    ind["k_scale"], ind["w"], case.row_start, case.row_end, T,
                                    scores=scores)
        ops.dsa_topk(scores, rl, case.k, T, index_base=case.row_start, idx=idx, ws=tws)
        out, lse = ops.dsa_sparse_mla_fwd(case.q, case.softmax_scale, case.kv, idx)
        dout = I.to_bf16(torch.randn(out.shape, generator=torch.Generator(device=dev).manual_seed(1),
                                     device=dev))
        dq = torch.empty((T, H, 576), dtype=torch.float32, device=dev)
        dkv = torch.zeros((int(case.kv.rows), 576), dtype=torch.float32, device=dev)
        fn = lambda: ops.dsa_sparse_mla_bwd(case.q, case.softmax_scale, case.kv, idx, lse, dout,
                                            dq=dq, dkv=dkv)
        clocks.start()
        us = _timed(fn, args.steps, args.warmup, l2_flush)
        clk = clocks.stop()
        v = statistics.median(us)
        rows = int((idx >= 0).sum())
        # the backward's products: dS (q.K and dout.V) and dq, dK, dV, about
        # 2.5 times the forward's 2 * H * 1088 flops per (token, row)
        flop = 2.5 * 2.0 * H * 1088 * rows
        res.update({"value": round(v, 3), "ms_per_step": round(v / 1000, 6),
                    "dtype": "bf16 operands on the tensor cores (P and dS as bf16 hi + lo terms), fp32 accumulate",
                    "config": {"workload": "sparse_mla_bwd_T%d_H%d" % (T, H), "tokens": T,
                               "heads": H, "topk": case.k},
                    "roofline": {"bound": "tensor", "unit": "TFLOP/s",
                                 "achieved": round(flop / (v * 1e-6) / 1e12, 2),
                                 "peak": bf16_tflops, "peak_kind": "measured bf16 dense",
                                 "frac": round(flop / (v * 1e-6) / 1e12 / bf16_tflops, 4),
                                 "flop": flop},
                    "clocks": clk})
    elif w == "paged":
        # the decode step on paged caches: pages of 64 slots, shuffled over the
        # pool, positions reached through the block table
        case = I.paged_decode(args.batch, args.context, page=args.page, device=dev)
        N = args.context
        ws = ops.workspace(ops.dsa_decode_workspace_size(case.B, N, case.k, case.H, case.Dv), dev)
        fn = lambda: ops.decode_case(case, ws=ws)
        clocks.start()
        us = _timed(fn, args.steps, args.warmup, l2_flush)
        clk = clocks.stop()
        v = statistics.median(us)
        nbytes = case.B * N * (128 + 4 + 4) + case.B * 64 * (128 + 8) + \
            case.B * min(N, case.k) * 1152 + case.B * case.H * (576 * 2 + 512 * 2 + 4)
        res.update({"value": round(v, 3), "ms_per_step": round(v / 1000, 6),
                    "dtype": "fp8_e4m3 indexer + bf16 attention (fp32 accumulate)",
                    "config": {"workload": case.name, "batch": case.B, "context": N,
                               "page_size": args.page, "topk": case.k, "heads": case.H},
                    "step_roofline": {"bound": "hbm", "algorithmic_bytes_per_step": nbytes,
                                      "achieved_gbs": round(nbytes / (v * 1e-6) / 1e9, 1),
                                      "frac": round(nbytes / (v * 1e-6) / 1e9 / hbm_gbs, 4),
                                      "peak": hbm_gbs, "peak_kind": peak_kind},
                    "clocks": clk})
    elif w == "mtp":
        # two new tokens per request (speculative verification): B*2 rows of the
        # fused decode, a request's rows sharing its context
        Bq, Q, N = args.batch, 2, args.context
        case = I.multi_token_decode(Bq, Q, N, device=dev)
        ws = ops.workspace(ops.dsa_decode_workspace_size(case.B, N, case.k, case.H, case.Dv), dev)
        # the step as a request's rows paired (rows_per_request = 2: one read of
        # the request's keys for both rows), and beside it every row on its own
        fn = lambda: ops.decode_case(case, ws=ws, rows_per_request=2)
        fn1 = lambda: ops.decode_case(case, ws=ws)
        clocks.start()
        us = _timed(fn, args.steps, args.warmup, l2_flush)
        clk = clocks.stop()
        v = statistics.median(us)
        v1 = statistics.median(_timed(fn1, args.steps, args.warmup, l2_flush))
        # unique bytes: each request's keys and scales once, the selected rows of
        # every token, q/out/lse of every row (the paired step reads a request's
        # keys once; one row at a time, Q times)
        nbytes = Bq * N * (128 + 4) + case.B * N * 4 + case.B * 2048 * 1152 + \
            case.B * case.H * (576 * 2 + 512 * 2 + 4)
        res.update({"value": round(v, 3), "ms_per_step": round(v / 1000, 6),
                    "dtype": "fp8_e4m3 indexer + bf16 attention (fp32 accumulate)",
                    "config": {"workload": case.name, "requests": Bq, "tokens_per_request": Q,
                               "context": N, "topk": case.k, "heads": case.H,
                               "rows_per_request": 2},
                    "single_rows_us": round(v1, 3),
                    "step_roofline": {"bound": "hbm", "algorithmic_bytes_per_step": nbytes,
                                      "achieved_gbs": round(nbytes / (v * 1e-6) / 1e9, 1),
                                      "frac": round(nbytes / (v * 1e-6) / 1e9 / hbm_gbs, 4),
                                      "peak": hbm_gbs, "peak_kind": peak_kind},
                    "clocks": clk})
    elif w in ("tiny", "packed_1m"):
        case = I.tiny_decode(device=dev) if w == "tiny" else I.packed_long_decode(device=dev)
        k_swa = 0 if case.idx_swa is None else case.idx_swa.shape[1]
        ws = ops.workspace(ops.dsa_decode_workspace_size(case.B, case.max_seq_len, case.k,
                                                         case.H, case.Dv, k_swa), dev)
        fn = lambda: ops.decode_case(case, ws=ws)
        clocks.start()
        us = _timed(fn, args.steps, args.warmup, l2_flush)
        clk = clocks.stop()
        N = case.max_seq_len
        if w == "tiny":
            nbytes = N * 64 * 2 + min(N, case.k) * 1152 + case.H * (576 * 2 + 512 * 2 + 4)
            dtype = "bf16 indexer + bf16 attention"
        else:
            nbytes = N * (128 + 4 + 4) + (case.k + k_swa) * 584 + case.H * (512 * 2 + 448 * 2 + 4)
            dtype = "fp8_e4m3 indexer + fp8_ds_mla attention (fp32 accumulate)"
        v = statistics.median(us)
        res.update({"value": round(v, 3), "ms_per_step": round(v / 1000, 6), "dtype": dtype,
                    "config": {"workload": case.name, "batch": case.B, "context": N,
                               "topk": case.k, "swa": k_swa, "heads": case.H},
                    "step_roofline": {"bound": "hbm", "algorithmic_bytes_per_step": nbytes,
                                      "achieved_gbs": round(nbytes / (v * 1e-6) / 1e9, 1),
                                      "frac": round(nbytes / (v * 1e-6) / 1e9 / hbm_gbs, 4),
                                      "peak": hbm_gbs, "peak_kind": peak_kind},
                    "clocks": clk})
    elif w == "uniform_fp8":
        case = I.uniform_fp8_swa_topk_case(device=dev)
        n = case.idx.shape[1]
        ws = ops.workspace(ops.dsa_sparse_mla_workspace_size(case.T, case.H, case.Dv, n, 0), dev)
        fn = lambda: ops.dsa_sparse_mla_fwd(case.q, case.softmax_scale, case.kv, case.idx, ws=ws)
        clocks.start()
        us = _timed(fn, args.steps, args.warmup, l2_flush)
        clk = clocks.stop()
        valid = int((case.idx >= 0).sum())
        nbytes = valid * (512 + 32) + case.T * case.H * (512 * 2 + 448 * 2 + 4) + case.idx.numel() * 4
        v = statistics.median(us)
        res.update({"value": round(v, 3), "ms_per_step": round(v / 1000, 6),
                    "dtype": "fp8_e4m3 pool (1x64 fp32 scales) + bf16 q, fp32 accumulate",
                    "config": {"workload": case.name, "batch": case.T, "entries": n,
                               "heads": case.H, "D": case.D, "Dv": case.Dv},
                    "step_roofline": {"bound": "hbm", "algorithmic_bytes_per_step": nbytes,
                                      "achieved_gbs": round(nbytes / (v * 1e-6) / 1e9, 1),
                                      "frac": round(nbytes / (v * 1e-6) / 1e9 / hbm_gbs, 4),
                                      "peak": hbm_gbs, "peak_kind": peak_kind},
                    "clocks": clk})
    elif w == "prefill":
        T, H = args.context, args.heads
        # one causal sequence of T tokens, or a packed batch of segments with
        # lengths drawn U[1, 8192] (two 1-token segments first) summing to T
        seg = [T] if args.segments == "single" else I.packed_segment_lengths(T)
        case = I.prefill_case(seg, k=2048, H=H, device=dev)
        ind = case.indexer
        lens = (case.row_end - case.row_start).cpu()
        maxL = int(lens.max())
        ld = (maxL + 3) // 4 * 4
        scores = torch.empty((T, ld), dtype=torch.float32, device=dev)
        rl = (case.row_end - case.row_start).contiguous()
        tws = ops.workspace(ops.dsa_topk_workspace_size(T, maxL, case.k), dev)
        mws = ops.workspace(ops.dsa_sparse_mla_workspace_size(T, H, 512, case.k, 0), dev)
        idx = torch.empty((T, case.k), dtype=torch.int32, device=dev)
        f_idx = lambda: ops.dsa_index_score_prefill(ind["q_idx"], 1, ind["q_scale"], ind["k_idx"],
                                                    ind["k_scale"], ind["w"], case.row_start,
                                                    case.row_end, maxL, scores=scores)
        f_topk = lambda: ops.dsa_topk(scores, rl, case.k, maxL, index_base=case.row_start,
                                      idx=idx, ws=tws)
        f_mla = lambda: ops.dsa_sparse_mla_fwd(case.q, case.softmax_scale, case.kv, idx, ws=mws)
        clocks.start()
        st = {"index_score": statistics.median(_timed(f_idx, args.steps, args.warmup, l2_flush)),
              "topk": statistics.median(_timed(f_topk, args.steps, args.warmup, l2_flush)),
              "sparse_mla": statistics.median(_timed(f_mla, args.steps, args.warmup, l2_flush))}
        clk = clocks.stop()
        R = int(lens.clamp(max=case.k).sum())
        mla_flop = 2.0 * H * R * 1088
        idx_flop = 2.0 * 64 * 128 * int(lens.sum())
        v = sum(st.values())
        fp8_tflops = 2.0 * bf16_tflops   # the fp8 dense rate is twice bf16's
        res.update({"value": round(v, 3), "ms_per_step": round(v / 1000, 6),
                    "dtype": "fp8_e4m3 indexer + bf16 attention (fp32 accumulate)",
                    "config": {"workload": "prefill_%sT%d_H%d" % ("" if len(seg) == 1 else "packed_", T, H),
                               "tokens": T, "heads": H, "topk": case.k, "segments": len(seg)},
                    "stages_us": {k: round(x, 2) for k, x in st.items()},
                    "roofline": {"sparse_mla": {"bound": "tensor", "unit": "TFLOP/s",
                                                "achieved": round(mla_flop / (st["sparse_mla"] * 1e-6) / 1e12, 1),
                                                "peak": bf16_tflops, "peak_kind": peak_kind + " bf16 dense",
                                                "frac": round(mla_flop / (st["sparse_mla"] * 1e-6) / 1e12 / bf16_tflops, 4),
                                                "flop": mla_flop,
                                                # beside it, the row gather: R rows of 1152 B
                                                # (served from L2: the pool is resident), against
                                                # the measured HBM copy rate for scale
                                                "gather": {"bytes": R * 1152,
                                                           "achieved_gbs": round(R * 1152 / (st["sparse_mla"] * 1e-6) / 1e9, 1),
                                                           "frac_of_hbm_copy": round(R * 1152 / (st["sparse_mla"] * 1e-6) / 1e9 / hbm_gbs, 4)}},
                                 "index_score": {"bound": "tensor", "unit": "TFLOP/s",
                                                 "achieved": round(idx_flop / (st["index_score"] * 1e-6) / 1e12, 1),
                                                 "peak": fp8_tflops, "peak_kind": peak_kind + " bf16 x 2 (fp8 dense)",
                                                 "frac": round(idx_flop / (st["index_score"] * 1e-6) / 1e12 / fp8_tflops, 4),
                                                 "flop": idx_flop}},
                    "clocks": clk})
    elif w in ("index", "topk", "mla"):
        # one stage of the decode step on decode_sweep(batch, context) inputs
        Bsz, N, k = args.batch, args.context, 2048
        case = I.decode_sweep(Bsz, N, device=dev)
        ind = case.indexer
        rs = case.slot_base
        re = (case.slot_base + case.seq_lens).contiguous()
        ld = (N + 3) // 4 * 4
        scores = torch.empty((Bsz, ld), dtype=torch.float32, device=dev)
        idx = torch.empty((Bsz, k), dtype=torch.int32, device=dev)
        f_idx = lambda: ops.dsa_index_score(ind["q_idx"], ind["idx_dtype"], ind["q_scale"],
                                            ind["k_idx"], ind["k_scale"], ind["w"], rs, re, N,
                                            scores=scores)
        tws = ops.workspace(ops.dsa_topk_workspace_size(Bsz, N, k), dev)
        f_topk = lambda: ops.dsa_topk(scores, case.seq_lens, k, N, index_base=case.slot_base,
                                      idx=idx, ws=tws)
        mws = ops.workspace(ops.dsa_sparse_mla_workspace_size(Bsz, case.H, case.Dv, k, 0), dev)
        f_mla = lambda: ops.dsa_sparse_mla_fwd(case.q, case.softmax_scale, case.kv, idx, ws=mws)
        f_idx()
        f_topk()
        torch.cuda.synchronize()
        fn = {"index": f_idx, "topk": f_topk, "mla": f_mla}[w]
        clocks.start()
        v = statistics.median(_timed(fn, args.steps, args.warmup, l2_flush))
        clk = clocks.stop()
        nbytes = {"index": Bsz * N * (128 + 4 + 4) + Bsz * 64 * (128 + 8),
                  "topk": Bsz * N * 4 + Bsz * k * 4,
                  "mla": Bsz * min(N, k) * (1152 + 4) + Bsz * case.H * (576 * 2 + 512 * 2 + 4)}[w]
        res.update({"value": round(v, 3), "ms_per_step": round(v / 1000, 6),
                    "dtype": "fp8_e4m3 indexer + bf16 attention (fp32 accumulate)",
                    "config": {"workload": "%s_b%d_n%d" % (w, Bsz, N), "batch": Bsz, "context": N,
                               "topk": k},
                    "step_roofline": {"bound": "hbm", "algorithmic_bytes_per_step": nbytes,
                                      "achieved_gbs": round(nbytes / (v * 1e-6) / 1e9, 1),
                                      "frac": round(nbytes / (v * 1e-6) / 1e9 / hbm_gbs, 4),
                                      "peak": hbm_gbs, "peak_kind": peak_kind},
                    "clocks": clk})
    print(json.dumps(res), flush=True)


# ---------------------------------------------------------------- oracle (CPU)
#
# The oracle is plain numpy in float64, one request at a time.  It is timed
# on the host's cores as a pool of worker processes (spawned, so no CUDA
# state is inherited), each with one BLAS thread and its own request of the
# workload; a barrier starts a round of requests on every worker at once, and
# a round lasts as long as its slowest request.

_OW = {}


def _oracle_init(N, barrier):
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        os.environ[v] = "1"
    _OW["N"], _OW["barrier"] = N, barrier


def _oracle_round(seed):
    """One request of the decode workload through the oracle; returns its
    seconds.  The worker builds its request once (context N, its own seed)."""
    import torch
    torch.set_num_threads(1)
    import oracle.dsa_oracle as O
    from deepseek_sparse_attention_index_gb300 import inputs as I
    from tests.helpers import decode_case_np
    if "case" not in _OW:
        _OW["case"] = decode_case_np(I.decode_sweep(1, _OW["N"], device="cpu", seed=100 + seed))
    _OW["barrier"].wait()
    t0 = time.perf_counter()
    O.decode_request(0, _OW["case"])
    return time.perf_counter() - t0


class OraclePool:
    """`workers` processes timing the oracle on requests of context N."""

    def __init__(self, N, workers):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.workers = workers
        self.barrier = ctx.Barrier(workers)
        self.pool = ctx.Pool(workers, initializer=_oracle_init, initargs=(N, self.barrier))

    def round(self):
        """Seconds of one round: `workers` requests at once, one per worker."""
        return max(self.pool.map(_oracle_round, range(self.workers), chunksize=1))

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(B, N, rounds=1):
    """The oracle on the host cores for a (B, N) decode step: all cores (one
    request per core at once, scaled to the batch) and one thread (one
    request, scaled to the batch)."""
    cores = cpu_cores()
    pool = OraclePool(N, cores)
    pool.round()                                   # builds each worker's request
    t_all = statistics.mean(pool.round() for _ in range(rounds))
    pool.close()
    one = OraclePool(N, 1)
    one.round()
    t_one = statistics.mean(one.round() for _ in range(rounds))
    one.close()
    return {"value": round(t_all * B / cores * 1e6, 1), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": "%d requests of context %d at once, one per core (1 BLAS thread each), "
                      "the round's time scaled x%d/%d to the batch of %d" % (cores, N, B, cores, B),
            "one_thread": {"value": round(t_one * B * 1e6, 1), "unit": UNIT, "cores": 1,
                           "sample": "1 request of context %d, scaled x%d" % (N, B)}}


def run_reference(args):
    """The reference arm: the CPU oracle on this host's cores, on the default
    decode workload.  Each step is one round of requests on every core at once
    (one request per core), scaled to the batch."""
    Bsz, N = args.batch, args.context
    cores = cpu_cores()
    pool = OraclePool(N, cores)
    for _ in range(args.warmup):                   # the first round builds the requests
        pool.round()
    per = [pool.round() for _ in range(args.steps)]
    pool.close()
    us = statistics.mean(per) * Bsz / cores * 1e6
    sample = ("each step: %d requests of context %d at once, one per core (1 BLAS thread each), "
              "the round's time scaled x%d/%d to the batch of %d (extrapolated from the sample)"
              % (cores, N, Bsz, cores, Bsz))
    res = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1000, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(Bsz, N, 2048),
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "extrapolated": {"timed_requests_per_step": cores, "batch": Bsz,
                         "timed_s_per_step": round(statistics.mean(per), 3)},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=32)
    ap.add_argument("--context", type=int, default=131072)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "tiny", "uniform_fp8", "packed_1m", "prefill",
                             "index", "topk", "mla", "mtp", "paged", "bwd"],
                    help="decode (default): the driver's line; the others are secondary "
                         "measurements of the remaining configurations")
    ap.add_argument("--heads", type=int, default=64, help="prefill: attention heads")
    ap.add_argument("--segments", default="single", choices=["single", "packed"],
                    help="prefill: one causal sequence, or packed segments of U[1, 8192] tokens")
    ap.add_argument("--page", type=int, default=64, help="paged: slots per page (a multiple of 64)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.gpus != world:
        # one process per GPU: N GPUs need N ranks (torchrun --nproc-per-node N)
        sys.exit("bench.py: --gpus %d but WORLD_SIZE=%d; launch N > 1 GPUs with "
                 "python -m torch.distributed.run --nproc-per-node N bench.py --gpus N"
                 % (args.gpus, world))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if args.workload != "decode":
        if rank == 0:
            run_workload(args)
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.batch, args.context)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
