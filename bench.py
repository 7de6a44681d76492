"""Benchmark of the DSA decode step (Lightning Indexer + Top-K + Sparse Flash Attention).

Default workload: BF16 decode, batch 32, context 32768, 64-token pages randomly placed,
indexer 64 heads x d128, top-K 2048, SFA 128 heads x 576 (bf16).  One step = one
dsa_fused_decode call: one new token for each of the 32 sequences.

Prints one JSON line:
  value   decode tokens/s over the timed steps (device clock, inputs resident in HBM)
  e2e     the same through host buffers (pinned H2D of the step's queries, weights and
          page metadata + D2H of indices and attention output inside the timed region)
  roofline  the dominant kernel's algorithmic bytes per launch over its event-timed
          average duration, against the measured HBM copy bandwidth
  cpu_baseline  the float64 oracle on the host cores over a bounded sample
Use --impl reference to time the float64 oracle itself (the reference arm).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dsa_workloads as W  # noqa: E402

METRIC = "decode tokens/s and µs/step (indexer+SFA) at 1 GB300; % HBM / tensor roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ---------------------------------------------------------------------------------------
# Algorithmic work per launch (bytes that must move at least once; flops of the math)
# ---------------------------------------------------------------------------------------
def _visible(wl):
    lens = wl.seq_lens.astype(np.int64)
    return np.minimum(wl.q_pos.astype(np.int64) + 1, lens[wl.q_seq]).clip(min=0)


def algorithmic(wl, act="identity"):
    s = wl.spec
    vis = _visible(wl)
    T = wl.n_tokens
    k_elem = 2 if s.idx_dtype == "bf16" else 1
    k_row = s.idx_dim * k_elem + (4 if s.idx_scale == "per_token" else (s.idx_dim // 32 if s.idx_scale == "mx" else 0))
    if s.mode == "decode":
        key_tokens = int(vis.sum())            # every visible key row read once
    elif s.mode == "multi":
        key_tokens = int(wl.seq_lens.sum())    # each sequence's keys read once for all its draft tokens
    else:
        key_tokens = int(wl.seq_lens[0])       # the prefix is read once (shared by all rows)
    q_bytes = T * s.idx_heads * s.idx_dim * k_elem + T * s.idx_heads * 4
    if s.idx_scale == "per_token":
        q_bytes += T * 4
    elif s.idx_scale == "mx":
        q_bytes += T * s.idx_heads * s.idx_dim // 32
    sel = np.minimum(vis, s.topk)
    idx_bytes = T * s.topk * 4
    score_flops = 2.0 * s.idx_heads * s.idx_dim * float(vis.sum())
    gather_rows = int(sel.sum())
    kv_row = 1152 if s.kv_format == "bf16" else 512 + 4 * 4 + 64 * 2   # FP8: codes, 4 tile scales, bf16 rope
    sfa_bytes = gather_rows * kv_row + T * s.sfa_heads * 576 * 2 + T * s.sfa_heads * 512 * 2 + idx_bytes
    sfa_flops = 2.0 * s.sfa_heads * (576 + 512) * float(sel.sum())
    meta = wl.block_table.nbytes + wl.seq_lens.nbytes
    # The row-blocked scorer (a prefill; a sequence's draft tokens) folds the head sum into
    # the query: per block of up to 21 rows and 128-key tile it runs one M = 128, N = 64
    # (21 rows x 3 split terms), K = d MMA.  Its executed tensor work, not the per-head
    # definition's, is what its tensor fraction is measured on.
    blk_flops = 0.0
    if s.mode in ("prefill", "multi") and s.idx_heads and T >= 2 and act == "identity":
        seg = T if s.mode == "prefill" else s.tokens_per_seq
        for s0 in range(0, T, seg):
            for r0 in range(s0, s0 + seg, 21):
                mv = int(vis[r0:min(r0 + 21, s0 + seg)].max(initial=0))
                blk_flops += 2.0 * 128 * 64 * s.idx_dim * ((mv + 127) // 128)
    return {
        "indexer_score": {"bytes": key_tokens * k_row + q_bytes + meta, "flops": score_flops,
                          "executed_flops": blk_flops},
        "indexer_topk": {"bytes": idx_bytes, "flops": 0.0},
        "sfa": {"bytes": sfa_bytes, "flops": sfa_flops},
        "hist_clear": {"bytes": T * 4096 * 4, "flops": 0.0},
        "step": {"bytes": key_tokens * k_row + q_bytes + meta + sfa_bytes, "flops": score_flops + sfa_flops},
    }


# ---------------------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"dsa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------
# Traffic measured by ncu (profiles/traffic.json), used only while the kernel source is
# unchanged since the capture.
# ---------------------------------------------------------------------------------------
KERNEL_SOURCES = {"indexer_score": "indexer_tc.cu", "indexer_topk": "topk.cu", "sfa": "sfa_tc.cu"}


def _src_sha(kernel):
    path = os.path.join(ROOT, "sparse_attention_decode_dsa_gb300", "csrc", KERNEL_SOURCES[kernel])
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def _traffic(kernel, workload, units):
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d or d.get("src_sha") != _src_sha(kernel) or d.get("workload") != workload:
        return None
    # bytes per unit (key token or gathered row) from the capture, scaled to this launch
    return d["bytes_per_unit"] * units


def max_over_ranks(ms, dist=None, device=None):
    """The slowest rank's time in ms (all ranks get it); the local time without a group."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, ms):
    """Units all ranks processed (replicas: each rank the same count) per second, over
    the slowest rank's time."""
    return world * units_per_rank / (ms * 1e-3)


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_sample(wl, budget_s):
    """Time the float64 oracle over whole query tokens until the budget is spent."""
    from oracle import dsa_oracle as O
    n, t0 = 0, time.perf_counter()
    order = np.random.default_rng(0).permutation(wl.n_tokens)
    while n < len(order):
        O.step(wl, int(order[n]))
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return n, time.perf_counter() - t0


# ---------------------------------------------------------------------------------------
def run_prolog(args):
    """The index prolog on its own: dsa_quantize_mxfp8 over the 8192-token prefill query
    (8192 x 64 heads x 128 bf16, 134 MB: larger than L2) and dsa_index_cache_append_mxfp8
    of one decode step's 32 new keys into a 16384-page MXFP8 cache.  Inputs resident in
    HBM; CUDA events on the launch stream around K back-to-back launches."""
    import torch
    import sparse_attention_decode_dsa_gb300 as dsa
    torch.manual_seed(0)
    dev = torch.device("cuda", 0)
    rows, dim = 8192 * 64, 128
    x = (torch.randn(rows, dim, device=dev) * 4).to(torch.bfloat16)
    codes = torch.empty(rows, dim, dtype=torch.uint8, device=dev)
    scales = torch.empty(rows, dim // 32, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        dsa.quantize_mxfp8(x, codes, scales)
    torch.cuda.synchronize()
    b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b.record(stream)
    for _ in range(args.steps):
        dsa.quantize_mxfp8(x, codes, scales)
    e.record(stream)
    torch.cuda.synchronize()
    q_us = b.elapsed_time(e) * 1e3 / args.steps
    q_bytes = rows * dim * 2 + rows * dim + rows * dim // 32  # bf16 in, e4m3 + E8M0 out
    # append: B = 32 sequences of 32768 positions over a 16384-page pool
    B, L, pool = 32, 32768, 16384
    maxp = L // 64
    bt = torch.randperm(pool, device=dev).to(torch.int32).view(B, maxp)
    lens_h = torch.full((B,), L, dtype=torch.int32)
    lens = lens_h.to(dev)
    cc = torch.zeros(pool, 64, dim, dtype=torch.uint8, device=dev)
    cs = torch.zeros(pool, 64, dim // 32, dtype=torch.uint8, device=dev)
    k_new = (torch.randn(B, dim, device=dev) * 4).to(torch.bfloat16)
    ws = dsa.alloc_workspace(256)
    for _ in range(max(3, args.warmup)):
        dsa.index_cache_append_mxfp8(k_new, cc, cs, bt, lens, lens_h, ws)
    torch.cuda.synchronize()
    b.record(stream)
    for _ in range(args.steps):
        dsa.index_cache_append_mxfp8(k_new, cc, cs, bt, lens, lens_h, ws)
    e.record(stream)
    torch.cuda.synchronize()
    a_us = b.elapsed_time(e) * 1e3 / args.steps
    assert dsa.read_device_error(ws) == 0

    def time_calls(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        b.record(stream)
        for _ in range(args.steps):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        assert dsa.read_device_error(ws) == 0
        return b.elapsed_time(e) * 1e3 / args.steps

    # the other appends of one decode step (32 new tokens): K-index rows bf16 and e4m3 +
    # per-token scale, latent rows bf16 and FP8 (tiles of 128)
    kb = torch.zeros(pool, 64, dim, dtype=torch.bfloat16, device=dev)
    kf = torch.zeros(pool, 64, dim, dtype=torch.uint8, device=dev)
    kfs = torch.zeros(pool, 64, dtype=torch.float32, device=dev)
    lat_new = torch.randn(B, 576, device=dev).to(torch.bfloat16)
    lb = torch.zeros(pool, 64, 576, dtype=torch.bfloat16, device=dev)
    lc = torch.zeros(pool, 64, 512, dtype=torch.uint8, device=dev)
    lsc = torch.zeros(pool, 64, 4, dtype=torch.float32, device=dev)
    lr = torch.zeros(pool, 64, 64, dtype=torch.bfloat16, device=dev)
    appends = {
        "index_bf16_us": time_calls(lambda: dsa.index_cache_append(k_new, kb, None, bt, lens, lens_h, ws)),
        "index_fp8_per_token_us": time_calls(lambda: dsa.index_cache_append(k_new, kf, kfs, bt, lens, lens_h, ws)),
        "latent_bf16_us": time_calls(lambda: dsa.latent_cache_append(lat_new, lb, bt, lens, lens_h, ws)),
        "latent_fp8_us": time_calls(lambda: dsa.latent_cache_append(lat_new, lc, bt, lens, lens_h, ws, cache_scale=lsc,
                                                                    cache_rope=lr)),
    }
    peak, _, _, peak_src = _peaks()
    achieved = q_bytes / (q_us * 1e-6) / 1e9
    print(json.dumps({
        "metric": "index prolog: MXFP8 quantisation GB/s (8192 x 64 x 128 bf16 rows)", "value": achieved,
        "unit": "GB/s", "higher_is_better": True, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "quantize_us": q_us, "append_32_keys_us": a_us, "appends_32_tokens": appends, "dtype": "bf16 -> e4m3 + E8M0",
        "roofline": {"kernel": "mxfp8_quant", "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "algorithmic_bytes": q_bytes,
                     "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback"},
        "config": {"workload": "index_prolog", "rows": rows, "dim": dim, "group": 32,
                   "append": {"batch": B, "context": L, "pool_pages": pool},
                   "l2": "no flush: 134 MB in + 71 MB out per launch > L2"},
        "data": "synthetic (torch.randn * 4, seeded)"}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="bf16_decode", choices=sorted(W.ALL))
    ap.add_argument("--batch", type=int, default=0, help="override the batch (smaller capture cases)")
    ap.add_argument("--act", default="identity", choices=["identity", "relu"],
                    help="per-head activation of the indexer (relu: the per-head path in every mode)")
    ap.add_argument("--e2e-steps", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prolog", action="store_true",
                    help="time the index prolog instead (MXFP8 quantisation, K-index append)")
    args = ap.parse_args()
    if args.prolog:
        return run_prolog(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    spec = W.ALL[args.workload]
    if args.batch:
        assert spec.mode == "decode"
        lens = spec.seq_lens[:args.batch] if spec.seq_lens else ()
        spec = W.replace(spec, batch=args.batch, seq_lens=lens, pool_pages=0 if spec.seq_lens else spec.pool_pages)
    config = {"workload": spec.name, "batch": spec.batch,
              "context": int(max(spec.seq_lens)) if spec.seq_lens else f"log-uniform{list(spec.len_loguniform)}",
              "top_k": spec.topk, "index_heads": spec.idx_heads, "index_dim": spec.idx_dim,
              "index_dtype": spec.idx_dtype + ("" if spec.idx_scale == "none" else "+" + spec.idx_scale),
              "sfa_heads": spec.sfa_heads, "kv_dim": 576, "page_size": 64, "seed": spec.seed}
    if spec.kv_format != "bf16":
        config["kv_format"] = spec.kv_format
    if spec.mode == "multi":
        config["tokens_per_seq"] = spec.tokens_per_seq

    if args.impl == "reference":
        return run_reference(args, spec, config, world, rank)

    import torch
    import sparse_attention_decode_dsa_gb300 as dsa
    from dsa_workloads.device import to_device

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    wl = W.make(spec)
    d = to_device(wl, dev)
    if args.act == "relu":
        d.act = dsa.DSA_ACT_RELU
        config["act"] = "relu"
    plan = dsa.Plan(d)
    T, K, H = wl.n_tokens, spec.topk, spec.sfa_heads
    out_idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    ws = dsa.alloc_workspace(plan.ws_fused(), dev)
    stream = torch.cuda.current_stream(dev)
    work = algorithmic(wl, args.act)
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    input_bytes = sum(int(t.numel() * t.element_size()) for t in
                      [d.idx_k, d.kv, d.kv_codes, d.kv_scale, d.kv_rope, d.idx_q, d.sfa_q, d.head_w, d.block_table]
                      if t is not None)

    def step(trace=None):
        dsa.fused_decode(plan, out_idx, out, ws, stream=stream, trace=trace)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert dsa.read_device_error(ws) == 0

    # Per-launch events.  Events recorded between two launches would turn the overlapped
    # (programmatic dependent) launches of a step back into serialised ones, so the timed
    # region runs untraced and the per-kernel durations come from a traced pass of the
    # same steps right after it.
    traces = []
    for _ in range(args.steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * dsa.DSA_TRACE_MAX)]
        for e in evs:       # torch creates the CUDA event lazily, on its first record
            e.record(stream)
        tr = dsa.Trace()
        for i in range(dsa.DSA_TRACE_MAX):
            tr.begin[i] = evs[2 * i].cuda_event
            tr.end[i] = evs[2 * i + 1].cuda_event
            assert tr.begin[i] and tr.end[i]
        traces.append((tr, evs))
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local_rank)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(t_begin.elapsed_time(t_end), dist, dev)
    assert dsa.read_device_error(ws) == 0

    # traced pass (per-kernel durations)
    t_tb = torch.cuda.Event(enable_timing=True)
    t_te = torch.cuda.Event(enable_timing=True)
    t_tb.record(stream)
    for tr, _ in traces:
        step(tr)
    t_te.record(stream)
    torch.cuda.synchronize()
    traced_ms = t_tb.elapsed_time(t_te)
    assert dsa.read_device_error(ws) == 0

    per_kernel = {}
    launches = 0
    for tr, evs in traces:
        for i in range(tr.n_recorded):
            name = tr.name[i].decode()
            per_kernel.setdefault(name, []).append(evs[2 * i].elapsed_time(evs[2 * i + 1]))
            launches += 1
    kstats = {k: {"launches": len(v), "avg_us": 1e3 * sum(v) / len(v), "total_ms": sum(v)}
              for k, v in per_kernel.items()}
    ktotal = sum(s["total_ms"] for s in kstats.values())
    for s in kstats.values():
        s["share"] = s["total_ms"] / ktotal if ktotal else None
    dom = max(kstats, key=lambda k: kstats[k]["total_ms"])
    hbm_gbs, bf16_tf, bf16_tf_sust, peak_src = _peaks()
    dom_work = work.get(dom, {"bytes": 0, "flops": 0})
    avg_s = kstats[dom]["avg_us"] * 1e-6
    units = int(_visible(wl).sum()) if dom == "indexer_score" else int(np.minimum(_visible(wl), K).sum())
    traffic = _traffic(dom, spec.name, units)
    roofline = {"kernel": dom, "bound": "hbm", "achieved": dom_work["bytes"] / avg_s / 1e9, "peak": hbm_gbs,
                "unit": "GB/s", "frac": dom_work["bytes"] / avg_s / 1e9 / hbm_gbs,
                "traffic": traffic, "algorithmic_bytes": dom_work["bytes"],
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst copy)" if peak_src == "measured" else "fallback 6.8 TB/s",
                "frac_of_8TBps_nominal": dom_work["bytes"] / avg_s / 1e9 / 8000.0}
    if spec.mode == "prefill" and dom_work["flops"] > 0:
        # prefill is bound by the tensor cores: the kernel's algorithmic flops against the
        # measured sustained bf16 rate (it runs for milliseconds inside the step)
        ach = dom_work["flops"] / avg_s / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": bf16_tf_sust, "unit": "TFLOP/s",
                    "frac": ach / bf16_tf_sust, "traffic": traffic, "algorithmic_flops": dom_work["flops"],
                    "peak_source": f"{peak_src} (MEASURED_PEAKS.json bf16_tflops_sustained)" if peak_src == "measured"
                    else "fallback 1.7 PFLOP/s sustained"}

    # every kernel against its own bound: HBM bytes for all; tensor flops for the attention
    # and the row-blocked scorer
    kroof = {}
    for k, st in kstats.items():
        wk = work.get(k)
        if not wk or st["avg_us"] <= 0:
            continue
        a_s = st["avg_us"] * 1e-6
        r = {"algorithmic_bytes": wk["bytes"], "achieved_gbs": wk["bytes"] / a_s / 1e9,
             "frac_hbm": wk["bytes"] / a_s / 1e9 / hbm_gbs}
        fl = wk.get("executed_flops") or (wk["flops"] if k == "sfa" or (k == "indexer_score" and spec.mode == "prefill")
                                          else 0.0)
        if fl:
            r["tensor_tflops"] = fl / a_s / 1e12
            r["frac_tensor"] = fl / a_s / 1e12 / bf16_tf
            if k == "indexer_score":
                r["flops_note"] = "executed by the row-blocked (head-folded) scorer, not the per-head definition's"
        kroof[k] = r

    ms_per_step = total_ms / args.steps
    value = whole_job_rate(world, T * args.steps, total_ms)

    # ---- the same step replayed from a CUDA graph (host launch cost taken out) ----------
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            dsa.fused_decode(plan, out_idx, out, ws, stream=cap)
        torch.cuda.synchronize()
        for _ in range(max(3, args.warmup)):
            g.replay()
        torch.cuda.synchronize()
        g_b = torch.cuda.Event(enable_timing=True)
        g_e = torch.cuda.Event(enable_timing=True)
        g_b.record()
        for _ in range(args.steps):
            g.replay()
        g_e.record()
        torch.cuda.synchronize()
        g_ms = g_b.elapsed_time(g_e) / args.steps  # this rank's (no collective inside the try)
        graph = {"us_per_step": 1e3 * g_ms, "value": whole_job_rate(world, T, g_ms), "unit": UNIT,
                 "note": "one dsa_fused_decode captured once, replayed back to back"}
        assert dsa.read_device_error(ws) == 0
    except Exception as ex:  # report, do not fail the bench line
        graph = {"unavailable": f"{type(ex).__name__}: {ex}"[:200]}

    # ---- end to end through host buffers ----------------------------------------------
    # A serving loop: step i's inputs go up (pinned host -> device) on a copy stream while
    # step i - 1 computes, and step i's indices and outputs come back on another stream
    # while step i + 1 computes: two input / output sets with a plan each over the same
    # caches and workspace, events ordering every reuse.  Every step still pays its own
    # H2D and D2H copies inside the timed region.
    import dataclasses
    e2e_steps = args.e2e_steps or max(10, args.steps // 4)
    # Each input set is one device arena (the step's queries, weights and page metadata,
    # 256-byte aligned views) filled by ONE copy from one pinned host arena; the outputs
    # (indices, attention) are one device arena read back by ONE copy.
    in_names = [n for n in ("idx_q", "head_w", "sfa_q", "block_table", "seq_lens", "idx_q_scale")
                if getattr(d, n) is not None]

    def arena(tensors, device):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(n, dtype=torch.uint8, device=device) if device is not None else \
            torch.empty(n, dtype=torch.uint8).pin_memory()
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
        return buf, views

    h_in, h_in_views = arena([getattr(d, n) for n in in_names], None)
    for v, n in zip(h_in_views, in_names):
        v.copy_(getattr(d, n).cpu())
    sets = []
    for k in range(2):
        dv_buf, dv_views = arena([getattr(d, n) for n in in_names], dev)
        dk = dataclasses.replace(d, **dict(zip(in_names, dv_views)))
        o_buf, (o_idx, o_out) = arena([out_idx, out], dev)
        h_out, h_out_views = arena([out_idx, out], None)
        sets.append({"dv": dv_buf, "plan": dsa.Plan(dk), "out_idx": o_idx, "out": o_out, "o_buf": o_buf,
                     "h_out": h_out, "h_out_idx": h_out_views[0],
                     "up": torch.cuda.Event(), "comp": torch.cuda.Event(), "down": torch.cuda.Event()})
    h2d = h_in.numel()
    d2h = sets[0]["h_out"].numel()
    up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    e_b = torch.cuda.Event(enable_timing=True)
    e_e = torch.cuda.Event(enable_timing=True)
    e_b.record(stream)
    up_s.wait_event(e_b)
    for i in range(e2e_steps):
        st = sets[i % 2]
        with torch.cuda.stream(up_s):
            if i >= 2:
                up_s.wait_event(st["comp"])  # step i - 2 has consumed this set's inputs
            st["dv"].copy_(h_in, non_blocking=True)
            st["up"].record(up_s)
        stream.wait_event(st["up"])
        if i >= 2:
            stream.wait_event(st["down"])  # step i - 2's outputs of this set are on the host
        dsa.fused_decode(st["plan"], st["out_idx"], st["out"], ws, stream=stream)
        st["comp"].record(stream)
        with torch.cuda.stream(down_s):
            down_s.wait_event(st["comp"])
            st["h_out"].copy_(st["o_buf"], non_blocking=True)
            st["down"].record(down_s)
    stream.wait_stream(down_s)
    e_e.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_b.elapsed_time(e_e), dist, dev)
    e2e_val = whole_job_rate(world, T * e2e_steps, e2e_ms)
    assert dsa.read_device_error(ws) == 0
    assert torch.equal(sets[(e2e_steps - 1) % 2]["h_out_idx"], out_idx.cpu()), "end-to-end indices differ"

    # ---- oracle on the host cores --------------------------------------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, secs = _oracle_sample(wl, args.cpu_budget)
        cpu = {"value": n / secs, "unit": UNIT, "cores": _cores(), "kind": "oracle",
               "sample": f"{n} of {T} query tokens of {spec.name} (whole indexer + top-K + attention "
                         f"per token), float64 NumPy, {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_step": 1e3 * ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; integer-valued indexer inputs, N(0,1) bf16 latent KV)",
            "config": {**config, "l2": f"no flush: per-step inputs {input_bytes / 1e6:.0f} MB > L2 {l2_bytes / 1e6:.0f} MB",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline,
            "kernels": kstats,
            "kernel_rooflines": kroof,
            "kernel_timing": "per-launch CUDA events on the launch stream, in a traced pass of the same "
                             f"{args.steps} steps right after the timed region (events between launches "
                             "serialise them; that pass took " + f"{1e3 * traced_ms / args.steps:.1f} us/step)",
            "gpu_launches": launches,
            "step_algorithmic_bytes": work["step"]["bytes"],
            "step_frac_hbm": work["step"]["bytes"] / (ms_per_step * 1e-3) / 1e9 / hbm_gbs,
            "graph_replay": graph,
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps},
            "cpu_baseline": cpu,
            "clocks": clk,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def run_reference(args, spec, config, world, rank):
    """The reference arm: the float64 oracle on the host cores, a bounded sample per step."""
    if rank != 0:
        return
    wl = W.make(spec)
    from oracle import dsa_oracle as O
    order = np.random.default_rng(0).permutation(wl.n_tokens)
    per_step = max(1, min(wl.n_tokens, int(os.environ.get("DSA_REF_TOKENS_PER_STEP", "1"))))
    times = []
    k = 0
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for _ in range(per_step):
            O.step(wl, int(order[k % len(order)]))
            k += 1
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = per_step * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": config,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                             "sample": f"{per_step} query token(s) of {spec.name} per step (whole indexer + "
                                       f"top-K + attention), float64 NumPy"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
