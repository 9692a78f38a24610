"""Benchmark of the CSA layer hot path (decode step of the 128K-context
workload: 64 sequences, 32768 compressed entries each, top-k 512, window 128).

One step = one csa_layer_decode_with_keys call over the batch: the new
token's window row into the ring, block-boundary emission of the new
indexer key (from the key compressor's staging ring) and of the new
compressed entry, lightning indexer over every visible entry, top-k, and the
sparse attention.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun, one process per GPU) every rank decodes its own batch
of 64 sequences (weak scaling; no data exchange); the time is the maximum
over ranks.  `--impl reference` times the CPU oracle (the only reference this
method has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA-layer decode queries/s & indexer HBM GB/s, attn TC util vs GB300 peak"
QSETS = 4
UNIT = "queries/s"


GRAPH_STEPS = 16  # decode steps per captured CUDA graph


def pick_launch(eager_ms, eager_steps, graph_ms, graph_steps):
    """The faster of the two timed launch forms of the decode loop, per step:
    (steps, total ms, description, graph chosen).  graph_ms is None when no
    graph ran."""
    if graph_ms is not None and graph_steps > 0 and graph_ms / graph_steps < eager_ms / eager_steps:
        return graph_steps, graph_ms, "CUDA graphs of %d steps, replayed" % GRAPH_STEPS, True
    return eager_steps, eager_ms, "eager stream launches", False


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2, help="decode workload id (1, 2 or 3)")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (profiling captures only)")
    ap.add_argument("--no-extras", action="store_true", help="skip e2e, stage trace and CPU baseline")
    ap.add_argument("--section", choices=["decode", "reindex", "fp4_index", "compressor", "prefill", "hca"],
                    default="decode",
                    help="reindex: only the hierarchical indexer's Reindex layer on --workload (4 Full-layer "
                         "calls make the pools, then --warmup and --steps Reindex calls; for profiling); "
                         "fp4_index: only the FP4 indexer section on --workload; compressor: only the bulk "
                         "compressor section; prefill: only --warmup and --steps calls of the self-contained "
                         "prefill layer call on the 64K-context chunk, the first --queries queries of it; hca: "
                         "only the HCA section (dense attention at 128K and 1M, the single-stream compressor)")
    ap.add_argument("--queries", type=int, default=4096, help="prefill section: queries of the chunk (a multiple "
                                                              "of 4, for profiling captures of fewer)")
    return ap.parse_args()


def rank_config(config: int, rank: int) -> int:
    """Seed base of a rank's inputs: every rank decodes its own sequences."""
    return config + 100 * rank


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (all ranks call this)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, batch: int, steps: int, ms: float) -> float:
    """Whole-job queries/s: every rank's batch, per step, over the slowest rank's time."""
    return world * batch * steps / (ms / 1e3)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def bf16_sustained():
    """The sustained dense bf16 rate (a kernel inside a long call), measured
    copy if present, else the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1700.0, "fallback"


def fp8_peak(torch, dev):
    """Dense FP8 E4M3 GEMM rate on this GPU, measured here: torch._scaled_mm
    of 8192^3 (2*N^3 flops, unit scales, bf16 output), best of 10 after 3
    warm-up calls.  None if the library call is unavailable."""
    try:
        n = 8192
        g = torch.Generator(device=dev).manual_seed(5)
        a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn).t()  # column-major operand
        one = torch.ones((), device=dev)
        mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            mm()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(10):
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        time.sleep(0.05)

    def summary(self):
        rows = []
        for ts, line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((ts, float(f[1]), float(f[2]), f))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        t0, t1 = (self.marks + [0, 0])[:2] if len(self.marks) >= 2 else (0, 0)
        inside = [r for r in rows if t0 <= r[0] <= t1 + 0.05] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3][5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import compressed_sparse_attention_02_gb300 as csa
    import synthetic as syn

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = syn.WORKLOADS[args.workload]
    if args.batch:
        w = syn.Workload(w.name, w.config, w.kind, B=args.batch, t=w.t, topk=w.topk, n_cap=w.n_cap,
                         hadamard_kI=w.hadamard_kI)
    assert w.kind == "decode"
    B = w.B
    # each rank's batch is its own slice of sequences (seeded per sequence)
    x = syn.decode_inputs(syn.Workload(w.name, rank_config(w.config, rank), w.kind, B=B, t=w.t, topk=w.topk,
                                       n_cap=w.n_cap, hadamard_kI=w.hadamard_kI), device=dev)
    # Consecutive steps use different queries (QSETS sets, rotated), so each
    # step selects and gathers different cache rows: the selected rows of one
    # step are not left in L2 for the next.
    qsets = [syn.indexer_query(rank_config(w.config, rank) + 1000 * r, B, 1, device=dev) for r in range(QSETS)]
    for r, qs in enumerate(qsets):
        qs["q"] = syn.main_query(rank_config(w.config, rank) + 1000 * r, B, 1, device=dev)
    p = csa.csa_default_params(topk=w.topk)
    kv = x["kv"]
    idx = torch.empty(B, w.topk, dtype=torch.int32, device=dev)
    out = torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, 64, dtype=torch.float32, device=dev)
    ws = csa.workspace(csa.CSA_OP_LAYER_DECODE, p, B, 1, w.n_cap, device=dev)
    stream = torch.cuda.current_stream()
    counter = [0]
    keys = csa.index_key_src(x["ring_CIa"], x["ring_ZIa"], x["ring_CIb"], x["ring_ZIb"], x["BIa"], x["BIb"],
                             x["rms_wI"])
    swa_new = x["swa"][:, w.t % w.W].contiguous()

    def step():
        qs = qsets[counter[0] % QSETS]
        counter[0] += 1
        csa.csa_layer_decode_with_keys(p, B, x["q_pos"], swa_new, keys, x["ring_Ca"], x["ring_Za"], x["ring_Cb"],
                                       x["ring_Zb"], x["Ba"], x["Bb"], x["rms_w"], kv, w.n_cap, x["kI"], qs["qI"],
                                       qs["wI"], qs["q"], x["swa"], x["sink"], idx, out, lse, ws)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = csa.csa_check_status()
    if st != 0:
        raise RuntimeError("device status after warm-up: " + csa.csa_status_string(st))

    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark()
    launches0 = csa.csa_launch_count()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    launches = csa.csa_launch_count() - launches0
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1)
    # A serving loop replays captured steps: GRAPH_STEPS consecutive decode
    # steps (their query sets rotating as above) in one CUDA graph, replayed
    # for the same number of steps; the faster of the two launch forms counts.
    graph_ms, graph_why, g_steps = None, None, 0
    reps = args.steps // GRAPH_STEPS
    if reps >= 1:
        try:
            cap = torch.cuda.Stream()
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                for _ in range(3):
                    step()
            cap.synchronize()
            graph = torch.cuda.CUDAGraph()
            lc0 = csa.csa_launch_count()
            with torch.cuda.graph(graph, stream=cap):
                for _ in range(GRAPH_STEPS):
                    step()
            per_step = (csa.csa_launch_count() - lc0) / GRAPH_STEPS
            with torch.cuda.stream(stream):
                graph.replay()
            torch.cuda.synchronize()
            barrier()
            e0.record(stream)
            with torch.cuda.stream(stream):
                for _ in range(reps):
                    graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            graph_ms, g_steps = e0.elapsed_time(e1), reps * GRAPH_STEPS
            g_launches = int(round(per_step * g_steps))
            del graph
        except Exception as exc:  # keep the eager number
            graph_why = "graph capture failed: %s" % str(exc).splitlines()[0][:120]
    if clocks:
        clocks.mark()
    barrier()
    eager_ms = max_over_ranks(eager_ms, world, dev)
    if graph_ms is not None:
        graph_ms = max_over_ranks(graph_ms, world, dev)
    steps_timed, ms, launch, graph_chosen = pick_launch(eager_ms, args.steps, graph_ms, g_steps)
    if graph_chosen:
        launches = g_launches
    if clocks:
        clocks.stop()
    result = {
        "metric": METRIC, "value": job_value(world, B, steps_timed, ms), "unit": UNIT, "n_gpus": world,
        "steps": steps_timed, "warmup": args.warmup, "ms_per_step": ms / steps_timed, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16+e4m3",
        "data": "synthetic (seeded N(0,1) inputs in the pages' shapes; no trained weights)",
        "config": {"workload": w.name, "batch_per_gpu": B, "context_tokens": w.t + 1,
                   "compressed_entries": w.n_cap, "topk": w.topk, "swa_window": w.W, "m": w.m,
                   "l2": "inputs larger than L2 (K^I %d MiB + KV cache %d MiB per GPU); queries rotate over "
                         "%d sets so consecutive steps gather different rows"
                         % (B * w.n_cap * 128 >> 20, B * w.n_cap * 1024 >> 20, QSETS)},
        "gpu_launches": launches,
        "launch": launch,
        "eager_ms_per_step": eager_ms / args.steps,
        "graph_ms_per_step": graph_ms / g_steps if graph_ms is not None else graph_why,
    }
    if clocks:
        result["clocks"] = clocks.summary()
    if rank == 0 and not args.no_extras:
        # step time over 20 separately timed batches: median and p10 / p90
        nb = max(args.steps // 20, 50)
        per = []
        for _ in range(20):
            e0.record(stream)
            for _ in range(nb):
                step()
            e1.record(stream)
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) / nb)
        per.sort()
        result["step_ms_quantiles"] = {"p10": per[1], "p50": (per[9] + per[10]) / 2, "p90": per[17],
                                       "batches": 20, "steps_per_batch": nb}
        result.update(stage_profile(csa, torch, w, x, p, B, step, kv, out, idx, lse, ws, stream, args))
        result["attn"].update(attn_warm_l2(csa, torch, w, x, p, B, kv, out, idx, lse, stream))
        result["prefill"] = prefill_profile(csa, torch, dev)
        result["compressor"] = compressor_profile(csa, torch, dev)
        result["hierarchical"] = [hierarchical_profile(csa, torch, dev, cfg) for cfg in (2, 3)]
        result["hca"] = hca_profile(csa, torch, dev)
        result["fp4_cache"] = fp4_profile(csa, torch, dev, x, w)
        result["bf16_scores"] = [scores_profile(csa, torch, dev, cfg) for cfg in (2, 3)]
        result["fp4_index"] = [index_fp4_profile(csa, torch, dev, cfg,
                                                 x=x if cfg == args.workload and B == w.B else None)
                               for cfg in (2, 3)]
        result["e2e"] = end_to_end(csa, torch, w, x, qsets, p, B, kv, out, idx, lse, ws, stream, args)
        result["cpu_baseline"] = cpu_baseline(w, x, seconds=12.0)
    return result


def stage_profile(csa, torch, w, x, p, B, step, kv, out, idx, lse, ws, stream, args):
    """Live stage durations of the same decode step (events recorded between
    the layer call's kernels on its stream), and the roofline of the
    dominant kernel (the indexer score kernel)."""
    n = min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):
        csa.csa_set_trace_events(evs[i])
        step()
    csa.csa_set_trace_events(None)
    torch.cuda.synchronize()
    stage = [[evs[i][s].elapsed_time(evs[i][s + 1]) for i in range(n)] for s in range(4)]
    mean = [sum(v) / n for v in stage]
    hbm, bf16, src = peaks()
    V = (w.t + 1) // w.m
    idx_bytes = B * (V * 128 + 64 * 128 + 64 * 2)
    idx_ms = mean[1]
    achieved = idx_bytes / (idx_ms * 1e-3) / 1e9
    n_rows = min(w.W, w.t + 1) + min(w.topk, V)
    attn_flops = B * 4.0 * 64 * 512 * n_rows
    attn_bytes = B * (n_rows * 1024 + 2 * 64 * 1024)
    attn_ms = mean[3]
    traffic = _traffic_from_profile()
    return {
        "roofline": {"bound": "hbm", "kernel": "index_score_kernel", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic, "peak_source": src,
                     "frac_of_nominal_8000": achieved / 8000.0,
                     "algorithmic_bytes_per_launch": idx_bytes, "avg_launch_ms": idx_ms},
        # the decode step's compressor entry rides in the top-k launch (m <= 4),
        # so its own stage is empty and "topk" includes it
        "stages_ms": {"compress_emit": mean[0], "index_scores": mean[1], "topk": mean[2], "sparse_attn": mean[3],
                      "traced_steps": n, "note": "events between stages break the programmatic overlap"},
        "attn": {"binding_roofline_frac": max(attn_bytes / (hbm * 1e9), attn_flops / (bf16 * 1e12)) / (attn_ms * 1e-3),
                 "tflops": attn_flops / (attn_ms * 1e-3) / 1e12, "tc_frac_of_bf16_peak":
                 attn_flops / (attn_ms * 1e-3) / 1e12 / bf16, "gbs": attn_bytes / (attn_ms * 1e-3) / 1e9,
                 "hbm_frac": attn_bytes / (attn_ms * 1e-3) / 1e9 / hbm},
        "index_topk_gbs": idx_bytes / ((mean[1] + mean[2]) * 1e-3) / 1e9,
    }


def attn_warm_l2(csa, torch, w, x, p, B, kv, out, idx, lse, stream):
    """The sparse attention alone, repeated on the same selection, so its rows
    (40 MiB) are L2-resident: the warm-L2 counterpart of the in-step number."""
    hbm, bf16, _ = peaks()
    wsa = csa.workspace(csa.CSA_OP_SPARSE_ATTN, p, B, 1, w.n_cap, device=kv.device)

    def attn():
        csa.csa_sparse_attn(p, B, 1, x["q_pos"], x["q"], kv, w.n_cap, idx, x["swa"], 0, w.W, None, x["sink"], out,
                            lse, wsa)
    for _ in range(5):
        attn()
    torch.cuda.synchronize()
    n = 200
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        attn()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    V = (w.t + 1) // w.m
    n_rows = min(w.W, w.t + 1) + min(w.topk, V)
    flops = B * 4.0 * 64 * 512 * n_rows
    return {"warm_l2_ms": ms, "warm_l2_tflops": flops / (ms * 1e-3) / 1e12,
            "warm_l2_tc_frac_of_bf16_peak": flops / (ms * 1e-3) / 1e12 / bf16}


def prefill_profile(csa, torch, dev):
    """The chunked-prefill layer call of the 64K-context workload (4096 queries
    at positions 61440..65535 over 16384 entries), the self-contained form that
    also writes the chunk's indexer keys: stage durations, whole-call time, and
    the tensor-core rates of its two contractions (prefill is where the tensor
    peaks are the meaningful rooflines): the attention against the sustained
    bf16 rate (a kernel inside a call of about 2 ms), the indexer's scoring
    against an FP8 GEMM measured in this process."""
    import synthetic as syn
    hbm, bf16, _ = peaks()
    bf16_s, bf16_s_src = bf16_sustained()
    fp8 = fp8_peak(torch, dev)
    w = syn.WORKLOADS[4]
    B, Q = w.B, w.Q
    x = syn.prefill_inputs(w, device=dev)
    p = csa.csa_default_params(topk=w.topk)
    kv = x["kv"].clone()
    idx = torch.empty(B, Q, p.topk, dtype=torch.int32, device=dev)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Q, 64, dtype=torch.float32, device=dev)
    ws = csa.workspace(csa.CSA_OP_LAYER_PREFILL, p, B, Q, x["n_cap"], device=dev)
    keys_src = csa.index_key_src(x["CIa"], x["ZIa"], x["CIb"], x["ZIb"], x["BIa"], x["BIb"], x["rms_wI"],
                                 x["CIb_prev"], x["ZIb_prev"])

    def step():
        csa.csa_layer_prefill_with_keys(p, B, Q, w.pos0, x["Ca"], x["Za"], x["Cb"], x["Zb"], x["Cb_prev"],
                                        x["Zb_prev"], x["Ba"], x["Bb"], x["rms_w"], keys_src, kv, x["n_cap"],
                                        x["kI"], x["qI"], x["wI"], x["q"], x["swa"], x["sink"], idx, out, lse, ws)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    if csa.csa_check_status() != 0:
        raise RuntimeError("device status after prefill warm-up")
    n = 10
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
    for i in range(n):
        csa.csa_set_trace_events(evs[i])
        step()
    csa.csa_set_trace_events(None)
    torch.cuda.synchronize()
    st = [sum(evs[i][s].elapsed_time(evs[i][s + 1]) for i in range(n)) / n for s in range(4)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    # every query attends its 128 window rows and min(k, V(t)) selected entries
    rows = sum(min(w.W, t + 1) + min(w.topk, (t + 1) // w.m) for t in range(w.pos0, w.pos0 + Q))
    attn_flops = B * 4.0 * 64 * 512 * rows
    pairs = sum(min(x["n_cap"], (t + 1) // w.m) for t in range(w.pos0, w.pos0 + Q))
    index_flops = B * 2.0 * 64 * 128 * pairs
    attn_tf = attn_flops / (st[3] * 1e-3) / 1e12
    index_tf = index_flops / (st[1] * 1e-3) / 1e12
    n_new = Q // w.m
    res = {"workload": w.name, "tokens_per_s": B * Q / (ms * 1e-3), "ms_per_call": ms,
           "stages_ms": {"compress_and_keys": st[0], "index_scores": st[1], "topk": st[2], "sparse_attn": st[3]},
           "attn_tflops": attn_tf,
           "attn_tc_frac_of_bf16_peak": attn_tf / bf16,
           "attn_tc_frac_of_bf16_sustained": attn_tf / bf16_s, "bf16_sustained_tflops": bf16_s,
           "bf16_sustained_source": bf16_s_src,
           "index_fp8_tflops": index_tf,
           "fp8_peak_tflops": fp8, "fp8_peak_source": "torch._scaled_mm e4m3 8192^3, best of 10, this process",
           "index_fp8_frac": (index_tf / fp8) if fp8 else None,
           "compress_and_keys": {"entries": B * n_new, "bytes": B * n_new * (4 * w.m * (512 + 128) * 2 + 1024 + 128),
                                 "note": "main entries (bf16) and indexer keys (E4M3) of the chunk in one launch; "
                                         "stage time includes the first kernel (counters cleared)"}}
    del x, kv, idx, out, lse, ws
    torch.cuda.empty_cache()
    return res


def compressor_profile(csa, torch, dev):
    """The overlapped compressor in bulk form on v4flash-decode-b32-8k: 32
    sequences of 8192 tokens into 2048 entries each.  Algorithmic bytes: every
    input row read once (C^a, Z^a, C^b, Z^b: 4 x 8192 rows of 1 KiB per
    sequence, 1 GiB in all, larger than L2) and every entry written once."""
    import synthetic as syn
    hbm, _, _ = peaks()
    w = syn.WORKLOADS[1]
    B, T, m = w.B, w.t + 1, w.m
    n_new = T // m
    rows = syn.compressor_rows(w.config, B, T, device=dev)
    sp = syn.shared_params(w.config, m, dev)
    kv = torch.empty(B, n_new, 512, dtype=torch.bfloat16, device=dev)
    p = csa.csa_default_params(topk=w.topk, m=m)

    def call(i):
        csa.csa_compress(p, B, n_new, 0, rows["Ca"], rows["Za"], rows["Cb"], rows["Zb"], None, None, sp["Ba"],
                         sp["Bb"], sp["rms_w"], kv, n_new * 512)
    ms = _ms_per_call(torch, call, 20, warm=3)
    if csa.csa_check_status() != 0:
        raise RuntimeError("device status after the compressor section")
    byts = B * (4 * T + n_new) * 1024
    res = {"workload": w.name, "tokens": B * T, "entries": B * n_new, "ms": ms, "bytes": byts,
           "gbs": byts / (ms * 1e-3) / 1e9, "hbm_frac": byts / (ms * 1e-3) / 1e9 / hbm}
    del rows, kv
    torch.cuda.empty_cache()
    return res


def hierarchical_profile(csa, torch, dev, cfg, pool_blocks=2048, sets=4):
    """The hierarchical indexer on a decode workload ("DeepSeek-V4 CSA/HCA 与
    DeepSeek-V4.1 CSA2" §11): a Full layer (indexer + top-k + pool of 2048
    blocks, 16384 candidates) against the plain indexer + top-k, and a
    Reindex layer over the pool.  Query sets rotate (4 sets, each with its own
    pool), so consecutive calls gather different key blocks."""
    import synthetic as syn
    hbm, _, _ = peaks()
    w = syn.WORKLOADS[cfg]
    B = w.B
    kI = syn.indexer_keys(w.config, B, w.n_cap, device=dev, hadamard_rows=w.hadamard_kI)
    pos = torch.full((B, 1), w.t, dtype=torch.int32, device=dev)
    p = csa.csa_default_params(topk=w.topk)
    qs = [syn.indexer_query(w.config + 2000 + 100 * r, B, 1, device=dev) for r in range(sets)]
    q2 = [syn.indexer_query(w.config + 3000 + 100 * r, B, 1, device=dev) for r in range(sets)]
    idx = torch.empty(B, 1, w.topk, dtype=torch.int32, device=dev)
    pools = [torch.empty(B, 1, pool_blocks, dtype=torch.int32, device=dev) for _ in range(sets)]
    ws_full = csa.workspace(csa.CSA_OP_INDEX_TOPK_POOL, p, B, 1, w.n_cap, device=dev)
    ws_plain = csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, 1, w.n_cap, device=dev)
    ws_re = csa.workspace(csa.CSA_OP_REINDEX_TOPK, p, B, 1, w.n_cap, device=dev)

    def full(i):
        q = qs[i % sets]
        csa.csa_index_topk_pool(p, B, 1, pos, q["qI"], q["wI"], kI, w.n_cap, idx, None, pool_blocks,
                                pools[i % sets], ws_full)

    def plain(i):
        q = qs[i % sets]
        csa.csa_index_topk(p, B, 1, pos, q["qI"], q["wI"], kI, w.n_cap, idx, None, ws_plain)

    def reindex(i):
        q = q2[i % sets]
        csa.csa_reindex_topk(p, B, 1, pos, q["qI"], q["wI"], kI, w.n_cap, pools[i % sets], pool_blocks, idx, None,
                             ws_re)

    def timed(fn, n=200):
        for i in range(2 * sets):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n):
            fn(i)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def stages(fn, n=100):  # indexer kernel / top-k launches, from the call's trace events
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
        for i in range(n):
            csa.csa_set_trace_events(evs[i])
            fn(i)
        csa.csa_set_trace_events(None)
        torch.cuda.synchronize()
        return [sum(evs[i][s].elapsed_time(evs[i][s + 1]) for i in range(n)) / n for s in (1, 2)]

    res = {"workload": w.name, "pool_blocks": pool_blocks, "candidates": pool_blocks * 8,
           "full_layer_ms": timed(full), "index_topk_ms": timed(plain), "reindex_ms": timed(reindex)}
    res["full_layer_stages_ms"] = dict(zip(("index_scores", "topk_and_pool"), stages(full)))
    res["reindex_stages_ms"] = dict(zip(("index_scores", "topk"), stages(reindex)))
    if csa.csa_check_status() != 0:
        raise RuntimeError("device status after the hierarchical indexer")
    V = (w.t + 1) // w.m
    cand = min(pool_blocks, (V + 7) // 8) * 8
    rbytes = B * (cand * 128 + 64 * 128 + 64 * 2)
    res["reindex_gbs"] = rbytes / (res["reindex_ms"] * 1e-3) / 1e9
    res["reindex_hbm_frac"] = res["reindex_gbs"] / hbm
    kms = res["reindex_stages_ms"]["index_scores"]
    res["reindex_kernel_gbs"] = rbytes / (kms * 1e-3) / 1e9
    res["reindex_kernel_hbm_frac"] = res["reindex_kernel_gbs"] / hbm
    res["reindex_bytes"] = rbytes
    res["note"] = ("reindex bytes = the pool's key rows (1 KiB blocks gathered) + q^I + w^I per query; "
                   "full_layer_ms includes the block-score top-k; *_stages_ms from events between the "
                   "launches (which break their programmatic overlap); reindex_kernel_* = the indexer "
                   "kernel alone")
    del kI, qs, q2, pools, ws_full, ws_plain, ws_re
    torch.cuda.empty_cache()
    return res


def fp4_profile(csa, torch, dev, x, w, sets=4):
    """The FP4 cache ("DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §16.1, 288 B
    per entry) on the decode workload: the quantizer over the whole cache, and
    the sparse attention alone over the bf16 and the FP4 cache with the same
    selections (4 sets of 512 random entries per query, rotated)."""
    hbm, bf16, _ = peaks()
    B, n_cap, k = w.B, w.n_cap, w.topk
    kv = x["kv"]
    fp4 = torch.empty(B, n_cap, 288, dtype=torch.uint8, device=dev)

    def quant():
        csa.csa_quantize_kv_fp4(B * n_cap, kv, 512, fp4, 288)
    quant()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        quant()
    e1.record()
    torch.cuda.synchronize()
    qms = e0.elapsed_time(e1) / 10
    qbytes = B * n_cap * (1024 + 288)
    g = torch.Generator().manual_seed(7)
    sels = [torch.stack([torch.sort(torch.randperm(n_cap, generator=g)[:k])[0] for _ in range(B)])
            .to(torch.int32).view(B, 1, k).to(dev) for _ in range(sets)]
    qs = [syn_main_query(w, B, r, dev) for r in range(sets)]
    out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=dev)
    res = {"workload": w.name, "quantize": {"entries": B * n_cap, "ms": qms, "gbs": qbytes / (qms * 1e-3) / 1e9,
                                            "hbm_frac": qbytes / (qms * 1e-3) / 1e9 / hbm}}
    for fmt, cache in (("bf16", kv), ("fp4", fp4)):
        p = csa.csa_default_params(topk=k, kv_format=1 if fmt == "fp4" else 0)

        def attn(i):
            csa.csa_sparse_attn(p, B, 1, x["q_pos"], qs[i % sets], cache, n_cap, sels[i % sets], x["swa"], 0, w.W,
                                None, x["sink"], out, None)
        for i in range(8):
            attn(i)
        torch.cuda.synchronize()
        e0.record()
        for i in range(200):
            attn(i)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 200
        row = 288 if fmt == "fp4" else 1024
        byts = B * (k * row + w.W * 1024 + 2 * 64 * 1024)
        res["attention_" + fmt] = {"ms": ms, "gbs": byts / (ms * 1e-3) / 1e9, "bytes": byts}
    # the whole decode step (csa_layer_decode) over each cache, the same query rotation
    for fmt, cache in (("bf16", kv.clone()), ("fp4", fp4)):
        p = csa.csa_default_params(topk=k, kv_format=1 if fmt == "fp4" else 0)
        idx = torch.empty(B, k, dtype=torch.int32, device=dev)
        ws = csa.workspace(csa.CSA_OP_LAYER_DECODE, p, B, 1, n_cap, device=dev)
        qi = [syn_indexer_query(w, B, r, dev) for r in range(sets)]

        def step(i):
            qq = qi[i % sets]
            csa.csa_layer_decode(p, B, x["q_pos"], x["ring_Ca"], x["ring_Za"], x["ring_Cb"], x["ring_Zb"], x["Ba"],
                                 x["Bb"], x["rms_w"], cache, n_cap, x["kI"], qq["qI"], qq["wI"], qs[i % sets],
                                 x["swa"], x["sink"], idx, out.view(B, 64, 512), None, ws)
        for i in range(8):
            step(i)
        torch.cuda.synchronize()
        e0.record()
        for i in range(200):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        res["layer_step_ms_" + fmt] = e0.elapsed_time(e1) / 200
        del ws, qi
    res["cache_bytes_per_entry"] = {"bf16": 1024, "fp4": 288}
    if csa.csa_check_status() != 0:
        raise RuntimeError("device status after the FP4 section")
    del fp4, sels, qs, out
    torch.cuda.empty_cache()
    return res


def scores_profile(csa, torch, dev, cfg, sets=4):
    """The indexer + top-k with fp32 and with bf16 scores ([KV 压缩] §7: BF16
    scores for the selector): stage durations from the call's trace events
    (indexer kernel, top-k launch) and the whole call, query sets rotated."""
    import synthetic as syn
    w = syn.WORKLOADS[cfg]
    B = w.B
    kI = syn.indexer_keys(w.config, B, w.n_cap, device=dev, hadamard_rows=w.hadamard_kI)
    pos = torch.full((B, 1), w.t, dtype=torch.int32, device=dev)
    qs = [syn.indexer_query(w.config + 4000 + 100 * r, B, 1, device=dev) for r in range(sets)]
    idx = torch.empty(B, 1, w.topk, dtype=torch.int32, device=dev)
    res = {"workload": w.name}
    for name, flag in (("fp32", 0), ("bf16", 1)):
        p = csa.csa_default_params(topk=w.topk, bf16_scores=flag)
        ws = csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, 1, w.n_cap, device=dev)

        def call(i):
            q = qs[i % sets]
            csa.csa_index_topk(p, B, 1, pos, q["qI"], q["wI"], kI, w.n_cap, idx, None, ws)
        for i in range(8):
            call(i)
        torch.cuda.synchronize()
        n = 100
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n):
            call(i)
        e1.record()
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
        for i in range(n):
            csa.csa_set_trace_events(evs[i])
            call(i)
        csa.csa_set_trace_events(None)
        torch.cuda.synchronize()
        st = [sum(evs[i][s].elapsed_time(evs[i][s + 1]) for i in range(n)) / n for s in (1, 2)]
        res[name] = {"call_ms": e0.elapsed_time(e1) / n, "index_scores_ms": st[0], "topk_ms": st[1]}
        del ws
    if csa.csa_check_status() != 0:
        raise RuntimeError("device status after the score-format section")
    del kI, qs, idx
    torch.cuda.empty_cache()
    return res


def _ms_per_call(torch, fn, n, warm=8):
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def _index_stages(csa, torch, fn, n):
    """Mean indexer-kernel and top-k durations of n calls, from the calls'
    trace events (csa_set_trace_events: events 1-2 bracket the indexer, 2-3
    the top-k)."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
    for i in range(n):
        csa.csa_set_trace_events(evs[i])
        fn(i)
    csa.csa_set_trace_events(None)
    torch.cuda.synchronize()
    return [sum(evs[i][s].elapsed_time(evs[i][s + 1]) for i in range(n)) / n for s in (1, 2)]


def index_fp4_profile(csa, torch, dev, cfg, x=None, sets=4, n=100):
    """The FP4 indexer ("DeepSeek-V4 CSA/HCA 与 DeepSeek-V4.1 CSA2" §16.2:
    68-byte keys, E2M1 with an E8M0 scale per 32 values; "DeepSeek-V4 的 KV
    压缩" §7.2: FP4 QK path and BF16 scores for the selector) beside the E4M3
    indexer on the same workload: the key quantizer, the indexer kernel and
    the top-k from the calls' trace events, the indexer's algorithmic HBM
    rate, the whole call, and (given the decode inputs x) the whole decode
    step with either indexer format.  Query sets rotate."""
    import synthetic as syn
    hbm, _, _ = peaks()
    w = syn.WORKLOADS[cfg]
    B, n_cap, t, k = w.B, w.n_cap, w.t, w.topk
    kbf = syn.indexer_keys_bf16(w.config, B, n_cap, device=dev)
    k4 = torch.empty(csa.index_keys_fp4_bytes(B, n_cap), dtype=torch.uint8, device=dev)
    qms = _ms_per_call(torch, lambda i: csa.csa_quantize_index_keys_fp4(B, n_cap, 0, kbf, n_cap * 128, k4, n_cap),
                       10, warm=1)
    del kbf
    k8 = syn.indexer_keys(w.config, B, n_cap, device=dev, hadamard_rows=w.hadamard_kI)
    pos = torch.full((B, 1), t, dtype=torch.int32, device=dev)
    qsets = []
    for r in range(sets):
        qb = syn.indexer_query_bf16(w.config + 4000 + 100 * r, B, 1, device=dev)
        q4 = torch.empty(csa.index_query_fp4_bytes(B), dtype=torch.uint8, device=dev)
        csa.csa_quantize_index_query_fp4(B, qb["qI"], q4)
        qsets.append({"e4m3": qb["qI"].to(torch.float8_e4m3fn), "fp4": q4, "wI": qb["wI"]})
    idx = torch.empty(B, 1, k, dtype=torch.int32, device=dev)
    V = min((t + 1) // w.m, n_cap)
    nbytes = {"e4m3": B * (V * 128 + 64 * 128 + 64 * 2),
              "fp4": B * (V * 64 + (V + 127) // 128 * 512 + 4608 + 64 * 2)}
    res = {"workload": w.name, "key_bytes_per_entry": {"e4m3": 128, "fp4": 68},
           "quantize_keys": {"entries": B * n_cap, "ms": qms,
                             "gbs": B * n_cap * (256 + 68) / (qms * 1e-3) / 1e9}}
    for name, fmt, sflag in (("e4m3", "e4m3", 0), ("fp4", "fp4", 0), ("fp4_bf16_scores", "fp4", 1)):
        p = csa.csa_default_params(topk=k, index_format=1 if fmt == "fp4" else 0, bf16_scores=sflag)
        ws = csa.workspace(csa.CSA_OP_INDEX_TOPK, p, B, 1, n_cap, device=dev)
        kI = k4 if fmt == "fp4" else k8

        def call(i):
            q = qsets[i % sets]
            csa.csa_index_topk(p, B, 1, pos, q[fmt], q["wI"], kI, n_cap, idx, None, ws)
        call_ms = _ms_per_call(torch, call, n)
        st = _index_stages(csa, torch, call, n)
        gbs = nbytes[fmt] / (st[0] * 1e-3) / 1e9
        res[name] = {"call_ms": call_ms, "index_scores_ms": st[0], "topk_ms": st[1], "index_bytes": nbytes[fmt],
                     "index_gbs": gbs, "index_hbm_frac": gbs / hbm}
        del ws
    # the hierarchical indexer with either key format: Full layers make one
    # 2048-block pool per query set, then Reindex layers with other queries
    nb = 2048
    pools = [torch.empty(B, 1, nb, dtype=torch.int32, device=dev) for _ in range(sets)]
    cand = min(nb, (V + 7) // 8) * 8
    for fmt in ("e4m3", "fp4"):
        p = csa.csa_default_params(topk=k, index_format=1 if fmt == "fp4" else 0)
        kI = k4 if fmt == "fp4" else k8
        ws_full = csa.workspace(csa.CSA_OP_INDEX_TOPK_POOL, p, B, 1, n_cap, device=dev)
        ws_re = csa.workspace(csa.CSA_OP_REINDEX_TOPK, p, B, 1, n_cap, device=dev)

        def full(i):
            q = qsets[i % sets]
            csa.csa_index_topk_pool(p, B, 1, pos, q[fmt], q["wI"], kI, n_cap, idx, None, nb, pools[i % sets],
                                    ws_full)

        def reindex(i):
            q = qsets[(i + 1) % sets]
            csa.csa_reindex_topk(p, B, 1, pos, q[fmt], q["wI"], kI, n_cap, pools[i % sets], nb, idx, None, ws_re)
        full_ms = _ms_per_call(torch, full, n)
        re_ms = _ms_per_call(torch, reindex, n)
        re_st = _index_stages(csa, torch, reindex, n)
        rbytes = B * (cand * (68 if fmt == "fp4" else 128) + (4608 if fmt == "fp4" else 8192) + 64 * 2)
        res["hierarchical_" + fmt] = {"full_layer_ms": full_ms, "reindex_ms": re_ms, "reindex_index_ms": re_st[0],
                                      "reindex_topk_ms": re_st[1], "reindex_bytes": rbytes,
                                      "reindex_kernel_gbs": rbytes / (re_st[0] * 1e-3) / 1e9,
                                      "reindex_kernel_hbm_frac": rbytes / (re_st[0] * 1e-3) / 1e9 / hbm}
        del ws_full, ws_re
    del pools
    if x is not None:  # the whole decode step (csa_layer_decode) with either indexer format
        qs = [syn_main_query(w, B, r, dev) for r in range(sets)]
        out = torch.empty(B, 64, 512, dtype=torch.bfloat16, device=dev)
        idx2 = torch.empty(B, k, dtype=torch.int32, device=dev)
        kv = x["kv"].clone()
        for fmt in ("e4m3", "fp4"):
            p = csa.csa_default_params(topk=k, index_format=1 if fmt == "fp4" else 0)
            ws = csa.workspace(csa.CSA_OP_LAYER_DECODE, p, B, 1, n_cap, device=dev)
            kI = k4 if fmt == "fp4" else k8

            def step(i):
                q = qsets[i % sets]
                csa.csa_layer_decode(p, B, x["q_pos"], x["ring_Ca"], x["ring_Za"], x["ring_Cb"], x["ring_Zb"],
                                     x["Ba"], x["Bb"], x["rms_w"], kv, n_cap, kI, q[fmt], q["wI"], qs[i % sets],
                                     x["swa"], x["sink"], idx2, out, None, ws)
            res["layer_step_ms_" + fmt] = _ms_per_call(torch, step, 200)
            del ws
        del qs, out, kv
    if csa.csa_check_status() != 0:
        raise RuntimeError("device status after the FP4 indexer section")
    del k4, k8, qsets, idx
    torch.cuda.empty_cache()
    return res


def syn_indexer_query(w, B, r, dev):
    import synthetic as syn
    return syn.indexer_query(w.config + 5000 + 1000 * r, B, 1, device=dev)


def syn_main_query(w, B, r, dev):
    import synthetic as syn
    return syn.main_query(w.config + 5000 + 1000 * r, B, 1, device=dev)


def hca_profile(csa, torch, dev, m=128):
    """The HCA layer's path (block size 128, no indexer): dense decode
    attention over the window and every visible compressed entry at 128K
    (64 sequences, 1024 entries) and 1M (8 sequences, 8192 entries) context,
    and the single-stream compressor over a prefill chunk.  Query sets rotate
    (4), caches are larger than L2 at 1M."""
    import synthetic as syn
    hbm, bf16, _ = peaks()
    p = csa.csa_default_params(m=m)
    res = {"block": m, "attention": []}
    for name, B, t in (("hca-decode-b64-128k", 64, 131071), ("hca-decode-b8-1m", 8, 1048575)):
        n_cap = (t + 1) // m
        kv = syn.cache_rows(100, B, n_cap, device=dev)
        swa = syn.cache_rows(100, B, 128, device=dev, name="swa")
        sink = syn.normal((64,), 100000, "sink", dev).float()
        qs = [syn.main_query(100 + 1000 * r, B, 1, device=dev) for r in range(4)]
        pos = torch.full((B, 1), t, dtype=torch.int32, device=dev)
        out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device=dev)

        wsa = csa.workspace(csa.CSA_OP_SPARSE_ATTN, p, B, 1, n_cap, device=dev)  # split-KV partials (B <= 16)

        def attn(i):
            csa.csa_sparse_attn(p, B, 1, pos, qs[i % 4], kv, n_cap, None, swa, 0, 128, None, sink, out, None, wsa)
        for i in range(8):
            attn(i)
        torch.cuda.synchronize()
        n = 100
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n):
            attn(i)
        e1.record()
        torch.cuda.synchronize()
        if csa.csa_check_status() != 0:
            raise RuntimeError("device status after the HCA attention")
        ms = e0.elapsed_time(e1) / n
        rows = 128 + n_cap
        flops = B * 4.0 * 64 * 512 * rows
        byts = B * (rows * 1024 + 2 * 64 * 1024)
        entry = {"workload": name, "batch": B, "entries": n_cap, "rows_per_query": rows, "ms": ms,
                 "queries_per_s": B / (ms * 1e-3), "gbs": byts / (ms * 1e-3) / 1e9,
                 "hbm_frac": byts / (ms * 1e-3) / 1e9 / hbm, "tflops": flops / (ms * 1e-3) / 1e12,
                 "binding_roofline_frac": max(byts / (hbm * 1e9), flops / (bf16 * 1e12)) / (ms * 1e-3)}
        # the whole HCA decode step (csa_hca_layer_decode): the compressor
        # state update (this position closes a block, so the entry is
        # written every step) and the dense attention
        x1 = syn.single_stream_inputs(102, B, 1, m, True, device=dev)
        state = torch.zeros(B, 3, 512, dtype=torch.float32, device=dev)
        wsl = csa.workspace(csa.CSA_OP_HCA_LAYER_DECODE, p, B, 1, n_cap, device=dev)
        C1, Z1 = x1["C"][:, 0].contiguous(), x1["Z"][:, 0].contiguous()

        def layer(i):
            csa.csa_hca_layer_decode(p, B, pos, C1, Z1, x1["B"], x1["rms_w"], state, kv, n_cap, qs[i % 4], swa, sink,
                                     out, None, wsl)
        for i in range(8):
            layer(i)
        torch.cuda.synchronize()
        e0.record()
        for i in range(n):
            layer(i)
        e1.record()
        torch.cuda.synchronize()
        lms = e0.elapsed_time(e1) / n
        entry["layer_step_ms"] = lms
        entry["layer_queries_per_s"] = B / (lms * 1e-3)
        res["attention"].append(entry)
        del kv, swa, qs, out, wsa, wsl, state
    # the compressor over a 16384-token chunk of 8 sequences: 128 entries each
    B, T = 8, 16384
    x = syn.single_stream_inputs(101, B, T, m, True, device=dev)
    kvc = torch.empty(B, T // m, 512, dtype=torch.bfloat16, device=dev)

    def comp():
        csa.csa_compress_single(p, B, T // m, 0, x["C"], x["Z"], x["B"], x["rms_w"], kvc, (T // m) * 512)
    for _ in range(3):
        comp()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(20):
        comp()
    e1.record()
    torch.cuda.synchronize()
    cms = e0.elapsed_time(e1) / 20
    cbytes = B * T * 2 * 1024 + B * (T // m) * 1024
    res["compressor"] = {"workload": "hca-compress-b8-16k-tokens", "entries": B * T // m, "ms": cms,
                         "gbs": cbytes / (cms * 1e-3) / 1e9, "hbm_frac": cbytes / (cms * 1e-3) / 1e9 / hbm}
    del x, kvc
    torch.cuda.empty_cache()
    return res


def reindex_section(args, pool_blocks=2048, sets=4):
    """The Reindex layer alone (for profiling captures): the Full layer makes
    one pool per query set (4 calls), then warm-up and timed Reindex calls
    rotate over the sets."""
    import torch

    import compressed_sparse_attention_02_gb300 as csa
    import synthetic as syn
    dev = torch.device("cuda", 0)
    w = syn.WORKLOADS[args.workload]
    B = args.batch or w.B
    kI = syn.indexer_keys(w.config, B, w.n_cap, device=dev, hadamard_rows=w.hadamard_kI)
    pos = torch.full((B, 1), w.t, dtype=torch.int32, device=dev)
    p = csa.csa_default_params(topk=w.topk)
    qs = [syn.indexer_query(w.config + 2000 + 100 * r, B, 1, device=dev) for r in range(sets)]
    q2 = [syn.indexer_query(w.config + 3000 + 100 * r, B, 1, device=dev) for r in range(sets)]
    idx = torch.empty(B, 1, w.topk, dtype=torch.int32, device=dev)
    pools = [torch.empty(B, 1, pool_blocks, dtype=torch.int32, device=dev) for _ in range(sets)]
    ws_full = csa.workspace(csa.CSA_OP_INDEX_TOPK_POOL, p, B, 1, w.n_cap, device=dev)
    ws_re = csa.workspace(csa.CSA_OP_REINDEX_TOPK, p, B, 1, w.n_cap, device=dev)
    for r in range(sets):
        csa.csa_index_topk_pool(p, B, 1, pos, qs[r]["qI"], qs[r]["wI"], kI, w.n_cap, idx, None, pool_blocks, pools[r],
                                ws_full)

    def reindex(i):
        q = q2[i % sets]
        csa.csa_reindex_topk(p, B, 1, pos, q["qI"], q["wI"], kI, w.n_cap, pools[i % sets], pool_blocks, idx, None,
                             ws_re)
    for i in range(args.warmup):
        reindex(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        reindex(i)
    e1.record()
    torch.cuda.synchronize()
    if csa.csa_check_status() != 0:
        raise RuntimeError("device status after the Reindex calls")
    return {"section": "reindex", "workload": w.name, "batch": B, "pool_blocks": pool_blocks,
            "ms_per_call": e0.elapsed_time(e1) / max(args.steps, 1)}


def prefill_section(args):
    """Timed calls of csa_layer_prefill_with_keys on the first --queries
    queries of the 64K-context chunk (positions 61440..): for profiling."""
    import torch

    import compressed_sparse_attention_02_gb300 as csa
    import synthetic as syn
    dev = torch.device("cuda", 0)
    w0 = syn.WORKLOADS[4]
    Q = max(4, args.queries // 4 * 4)
    w = syn.Workload(w0.name, w0.config, w0.kind, B=w0.B, t=w0.pos0 + Q - 1, topk=w0.topk, n_cap=w0.n_cap, Q=Q,
                     pos0=w0.pos0)
    x = syn.prefill_inputs(w, device=dev)
    p = csa.csa_default_params(topk=w.topk)
    B = w.B
    idx = torch.empty(B, Q, p.topk, dtype=torch.int32, device=dev)
    out = torch.empty(B, Q, 64, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Q, 64, dtype=torch.float32, device=dev)
    ws = csa.workspace(csa.CSA_OP_LAYER_PREFILL, p, B, Q, x["n_cap"], device=dev)
    keys = csa.index_key_src(x["CIa"], x["ZIa"], x["CIb"], x["ZIb"], x["BIa"], x["BIb"], x["rms_wI"], x["CIb_prev"],
                             x["ZIb_prev"])

    def step():
        csa.csa_layer_prefill_with_keys(p, B, Q, w.pos0, x["Ca"], x["Za"], x["Cb"], x["Zb"], x["Cb_prev"],
                                        x["Zb_prev"], x["Ba"], x["Bb"], x["rms_w"], keys, x["kv"], x["n_cap"],
                                        x["kI"], x["qI"], x["wI"], x["q"], x["swa"], x["sink"], idx, out, lse, ws)
    for _ in range(args.warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    if csa.csa_check_status() != 0:
        raise RuntimeError("device status after the prefill calls")
    return {"section": "prefill", "workload": w.name, "queries": Q,
            "ms_per_call": e0.elapsed_time(e1) / max(args.steps, 1)}


def _traffic_from_profile():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary (scaled from the captured batch to the full launch), or None when
    the kernel source has changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "index_score_kernel_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        with open(os.path.join(ROOT, d["source_file"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != d["source_sha256"]:
                return None
        return d.get("dram_bytes_per_full_launch")
    except Exception:
        return None


def end_to_end(csa, torch, w, x, qsets, p, B, kv, out, idx, lse, ws, stream, args):
    """Same metric through the same C-ABI call with every step's inputs in
    pinned host memory and its results read back: the step's queries, indexer
    queries and weights, positions, the staging rows of both compressors and
    the new token's window row travel host -> device in one packed copy (the
    layer call's first kernel stores the row into the window ring and
    computes the new entry's indexer key), and the attention output and the
    selection travel back.
    The copies run on their own streams one step ahead of / behind the layer
    call (two staging buffers and two output buffers), as a serving loop
    would overlap them; the timed region spans every step's copies."""
    stream = torch.cuda.Stream()  # a stream of its own (the legacy default stream cannot be captured)
    torch.cuda.synchronize()
    names = ["q", "qI", "wI", "q_pos", "ring_Ca", "ring_Za", "ring_Cb", "ring_Zb", "ring_CIa", "ring_ZIa",
             "ring_CIb", "ring_ZIb", "swa_row"]
    slot = w.t % w.W
    parts = {k: x[k] for k in names[:12]}
    parts["swa_row"] = x["swa"][:, slot].contiguous()
    layout, off = {}, 0
    for k in names:
        t = parts[k]
        layout[k] = (off, t.dtype, tuple(t.shape))
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    total = off

    def pack(src):
        buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        for k in names:
            o, dt, shape = layout[k]
            t = src.get(k, parts[k]).contiguous().cpu()
            buf[o:o + t.numel() * t.element_size()].copy_(t.view(-1).view(torch.uint8))
        return buf

    def views(buf):
        v = {}
        for k in names:
            o, dt, shape = layout[k]
            n = 1
            for d in shape:
                n *= d
            v[k] = buf[o:o + n * torch.empty((), dtype=dt).element_size()].view(dt).view(shape)
        return v

    hsets = [pack({k: qs[k] for k in ("q", "qI", "wI")}) for qs in qsets]
    stage = [torch.empty(total, dtype=torch.uint8, device=kv.device) for _ in range(2)]
    sviews = [views(b) for b in stage]
    vkeys = [csa.index_key_src(v["ring_CIa"], v["ring_ZIa"], v["ring_CIb"], v["ring_ZIb"], x["BIa"], x["BIb"],
                               x["rms_wI"]) for v in sviews]
    outs = [out, torch.empty_like(out)]
    idxs = [idx, torch.empty_like(idx)]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    idx_h = torch.empty(idx.shape, dtype=idx.dtype).pin_memory()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, stage_free, out_ready, out_free = ([ev(), ev()] for _ in range(4))
    h2d = total
    d2h = out_h.numel() * out_h.element_size() + idx_h.numel() * idx_h.element_size()

    def copy_in(i):
        s_ = i % 2
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(stage_free[s_])
            stage[s_].copy_(hsets[i % len(hsets)], non_blocking=True)
            in_ready[s_].record(h2d_s)

    def compute(i):
        s_ = i % 2
        v = sviews[s_]
        with torch.cuda.stream(stream):
            stream.wait_event(in_ready[s_])
            if i >= 2:
                stream.wait_event(out_free[s_])
            csa.csa_layer_decode_with_keys(p, B, v["q_pos"], v["swa_row"], vkeys[s_], v["ring_Ca"], v["ring_Za"],
                                           v["ring_Cb"], v["ring_Zb"], x["Ba"], x["Bb"], x["rms_w"], kv, w.n_cap,
                                           x["kI"], v["qI"], v["wI"], v["q"], x["swa"], x["sink"], idxs[s_],
                                           outs[s_], lse, ws)
            stage_free[s_].record(stream)
            out_ready[s_].record(stream)

    def copy_out(i):
        s_ = i % 2
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(out_ready[s_])
            out_h.copy_(outs[s_], non_blocking=True)
            idx_h.copy_(idxs[s_], non_blocking=True)
            out_free[s_].record(d2h_s)

    def run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
            copy_out(i)
        done = torch.cuda.Event()
        done.record(d2h_s)
        stream.wait_event(done)

    run(3)
    torch.cuda.synchronize()

    def timed(fn, n_steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_s.wait_event(e0)
        d2h_s.wait_event(e0)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return B * n_steps / (e0.elapsed_time(e1) / 1e3)

    n = min(args.steps, 512)
    eager = timed(lambda: run(n), n)
    # A serving loop replays captured steps: G consecutive steps (their copies
    # and the overlap between neighbours included) in one CUDA graph.
    G = 16
    graph, why = None, None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
            fork = torch.cuda.Event()
            fork.record(stream)
            h2d_s.wait_event(fork)
            d2h_s.wait_event(fork)
            run(G)
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
    except Exception as exc:  # report the eager loop alone
        graph, why = None, "graph capture failed: %s" % str(exc).splitlines()[0][:120]
    res = {"unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "copies": "one packed H2D and two D2H per step, on two copy streams overlapping the neighbouring "
                     "steps' layer calls", "eager_value": eager}
    if graph is not None:
        reps = max(n // G, 1)

        def replay():  # on the stream the timing events are recorded on
            with torch.cuda.stream(stream):
                for _ in range(reps):
                    graph.replay()
        g_val = timed(replay, reps * G)
        res["graph_value"] = g_val
        # a serving loop takes the faster of the two launch forms
        if g_val >= eager:
            res.update({"value": g_val, "steps": reps * G,
                        "launch": "CUDA graphs of %d steps (copies included), replayed" % G})
        else:
            res.update({"value": eager, "steps": n,
                        "launch": "eager stream launches (faster here than CUDA graphs of %d steps)" % G})
    else:
        res.update({"value": eager, "steps": n, "launch": "eager: " + why})
    if csa.csa_check_status() != 0:
        raise RuntimeError("device status after the end-to-end section")
    return res


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def _oracle_step_inputs(w, x, b):
    b16 = lambda t: __import__("synthetic").bits(t)
    return dict(t=w.t, ring_Ca=b16(x["ring_Ca"][b]), ring_Za=b16(x["ring_Za"][b]), ring_Cb=b16(x["ring_Cb"][b]),
                ring_Zb=b16(x["ring_Zb"][b]), Ba=b16(x["Ba"]), Bb=b16(x["Bb"]), rms_w=b16(x["rms_w"]),
                kv_comp=b16(x["kv"][b]), kI=b16(x["kI"][b]), qI=b16(x["qI"][b, 0]), wI=b16(x["wI"][b, 0]),
                q=b16(x["q"][b, 0]), swa_ring=b16(x["swa"][b]), sink=b16(x["sink"]),
                key_ring={k: b16(x["ring_" + k][b]) for k in ("CIa", "ZIa", "CIb", "ZIb")},
                key_params={k: b16(x[k]) for k in ("BIa", "BIb", "rms_wI")})


def _host_cores():
    """CPUs this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _oracle_units(w, inputs, threads):
    """Runs the oracle's full decode step of each input (one sequence) as one
    task, `threads` at a time: the oracle's C parts release the interpreter
    lock, so the independent units run on separate host cores.  A step that
    completes a block first computes the new entry's indexer key from the key
    compressor's ring (as the GPU step does) and indexes with it."""
    import concurrent.futures

    import oracle
    oracle.build()  # loaded before the workers start

    def unit(a):
        a = dict(a)
        t, ring, kp = a.pop("t"), a.pop("key_ring"), a.pop("key_params")
        if (t + 1) % w.m == 0 and (t + 1) // w.m - 1 < len(a["kI"]):
            i, m = (t + 1) // w.m - 1, w.m
            sa = [(m * i + r) % (2 * m) for r in range(m)]
            sb = [(m * (i - 1) + r) % (2 * m) for r in range(m)]
            _, codes = oracle.index_key_entry(i, ring["CIa"][sa], ring["ZIa"][sa], ring["CIb"][sb], ring["ZIb"][sb],
                                              kp["BIa"], kp["BIb"], kp["rms_wI"])
            a["kI"] = a["kI"].copy()
            a["kI"][i] = codes
        oracle.layer_decode_one(t, **a, m=w.m, topk_k=w.topk, W=w.W)
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(unit, inputs))


def cpu_baseline(w, x, seconds):
    """The oracle's full decode step for the sequences of the batch, one unit
    per host core at a time, in rounds until the batch or about `seconds` is
    used up."""
    cores = max(1, min(_host_cores(), w.B))
    done, t0 = 0, time.perf_counter()
    while done < w.B and (done == 0 or time.perf_counter() - t0 < seconds):
        n = min(cores, w.B - done)
        _oracle_units(w, [_oracle_step_inputs(w, x, b) for b in range(done, done + n)], cores)
        done += n
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d of the %d sequences of one decode step (full step each: key and entry emission, indexer over %d "
                      "entries, top-%d, attention over %d rows), fp64, one sequence per thread on %d threads"
                      % (done, w.B, (w.t + 1) // w.m, w.topk, min(w.W, w.t + 1) + w.topk, cores)}


def run_reference(args):
    """The CPU oracle as it stands, on this workload's inputs.  Each step
    decodes a bounded sample: P sequences of the decode step (one per host
    core, up to 16, in parallel), each restricted to h of the 64 query heads
    and h of the 64 indexer heads (work per head is identical, so the rate
    scales by h/64); h is chosen so the whole run stays within a few
    minutes."""
    import synthetic as syn

    w = syn.WORKLOADS[args.workload]
    P = max(1, min(_host_cores(), 16, w.B))
    x = syn.decode_inputs(syn.Workload(w.name, w.config, w.kind, B=P, t=w.t, topk=w.topk, n_cap=w.n_cap,
                                       hadamard_kI=w.hadamard_kI), device="cpu")
    seqs = [_oracle_step_inputs(w, x, b) for b in range(P)]

    def one(h):
        _oracle_units(w, [dict(a, qI=a["qI"][:h], wI=a["wI"][:h], q=a["q"][:h], sink=a["sink"][:h]) for a in seqs],
                      P)

    t0 = time.perf_counter()
    one(1)
    per_head = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    h = int(max(1, min(64, budget / max(per_head, 1e-6))))
    for _ in range(args.warmup):
        one(h)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one(h)
    dt = time.perf_counter() - t0
    value = args.steps * P * (h / 64.0) / dt
    sample = ("per step: %d sequences of the decode step in parallel (one per thread) on %d of 64 query heads "
              "and %d of 64 indexer heads (value scaled by %d/64), fp64 oracle" % (P, h, h, h))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "batch_per_gpu": w.B},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": P, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.section == "reindex":
        if rank == 0:
            print(json.dumps(reindex_section(args)), flush=True)
        return
    if args.section == "fp4_index":
        if rank == 0:
            import torch

            import compressed_sparse_attention_02_gb300 as csa
            print(json.dumps(index_fp4_profile(csa, torch, torch.device("cuda", 0), args.workload,
                                               n=max(args.steps, 1))), flush=True)
        return
    if args.section == "prefill":
        if rank == 0:
            print(json.dumps(prefill_section(args)), flush=True)
        return
    if args.section == "hca":
        if rank == 0:
            import torch

            import compressed_sparse_attention_02_gb300 as csa
            print(json.dumps(hca_profile(csa, torch, torch.device("cuda", 0))), flush=True)
        return
    if args.section == "compressor":
        if rank == 0:
            import torch

            import compressed_sparse_attention_02_gb300 as csa
            print(json.dumps(compressor_profile(csa, torch, torch.device("cuda", 0))), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
