#!/usr/bin/env python
"""Benchmark of the dynamic-mask sparse attention hot path on one B300.

A step is one pass of the whole prefill hot path -- dma_score_keys,
dma_select_topk (FULL), dma_sparse_attn_prefill -- over the 64K-token workload
(B=1, H=32, Hkv=8, S=65536, D=128, bf16, keep w=4096 plus a 512-token window,
5% salient rows).  The headline value is effective TFLOP/s counted on kept
(query, key) pairs: 4 * D flop per kept pair (QK^T and PV), the exact pair
count taken from the selection's output, divided by the whole step's time.
The decode workload (B=64 sequences, 32K-token caches, keep 2048 plus the last
64) is measured too and reported under "decode": GB/s of selected K and V rows.

Rules kept here: W >= 3 untimed warm-up steps; inputs larger than L2 (Q, K, V
and O of one step are 805 MB against a 126 MB L2); CUDA events on the launching
stream with a synchronize and a barrier on both sides; max over ranks; clocks
sampled by nvidia-smi during the timed region.

Multi-GPU: the path shards by independent (batch, KV head) units with no data
exchange, so N ranks each run the full workload (weak scaling) and value is the
sum of their work over the slowest rank's time.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (a slow, plain program: a reported baseline).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dma_workloads as wl  # noqa: E402

METRIC = "prefill eff. TFLOP/s on kept pairs @64K; decode selected-KV GB/s (% of peak)"
PREFILL_WL = "prefill_s64k_bf16"
DECODE_WL = "decode_b64_l32k_bf16"
LAUNCHES_SELECT_TOKEN = 19  # 4 x (hist, scan, scatter) + rank + table + prefix + boundary + walk + compact + tiles
LAUNCHES_PER_DECODE_STEP = 4  # score (new key) + update + decode partial + merge

# DRAM bytes (read + write) of one prefill attention launch on the 64K workload, from an ncu
# capture of that launch itself (metrics dram__bytes_read.sum and dram__bytes_write.sum only, one
# pass): 939,489,280 bytes read + 522,981,632 bytes written.  The compulsory bytes are 805 MB read
# (Q 537 MB, K and V 268 MB) and 545 MB written (O 537 MB, lse 8 MB); the extra 134 MB of reads
# are gathered K/V rows fetched again after leaving L2, and the writes fall short of the
# compulsory bytes by what is still dirty in L2 when the kernel ends.  Valid only for the kernel
# source it was taken on: reported as null once that source changes.
PREFILL_TRAFFIC = {"workload": "prefill_s64k_bf16", "bytes": 939489280 + 522981632,
                   "source_sha256": "aa33f5941c9a734a06391d252bafd9817379dbe7ac5ef958efdf045c4e7fd89b"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples of this GPU's clocks and throttle reasons (read only)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        try:
            p = torch.cuda.get_device_properties(device)
            self.gpu_id = "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            self.gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[device]

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------- dist ---

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    # NCCL reduces device tensors; other backends (gloo, in the CPU tests) host tensors
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ kept pairs ----

def prefill_traffic(workload: str):
    import hashlib
    src = os.path.join(ROOT, "content_aware_dynamic_dma_b300", "csrc", "prefill_tc.cu")
    try:
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    if workload != PREFILL_TRAFFIC["workload"] or sha != PREFILL_TRAFFIC["source_sha256"]:
        return None
    return PREFILL_TRAFFIC["bytes"]


def kept_pairs(expiry: torch.Tensor, S: int, window: int, block: int, G: int) -> int:
    """Sum over (b, query head, row i) of |kept set of row i|, from the per-key
    top-set intervals: key j is kept by rows [j, j+window) (window) united with
    [lo_j, expiry_j) (top set), clipped to [j, S)."""
    j = torch.arange(S, device=expiry.device, dtype=torch.int64)
    lo = j if block <= 1 else (j // block) * block + block - 1
    e = expiry.to(torch.int64)
    wa, wb = j, torch.clamp(j + window, max=S)                   # window rows [wa, wb)
    ta, tb = lo, torch.maximum(torch.minimum(e, torch.tensor(S, device=e.device)), lo)  # top rows [ta, tb)
    lw = (wb - wa).clamp(min=0)
    lt = (tb - ta).clamp(min=0)
    inter = (torch.minimum(wb, tb) - torch.maximum(wa, ta)).clamp(min=0)
    return int((lw + lt - inter).sum().item()) * G


# --------------------------------------------------------------- prefill ----

def bench_prefill(args, world, rank, peaks, clocks):
    import content_aware_dynamic_dma_b300 as dma
    cfg = wl.WORKLOADS[args.workload]
    inp = wl.make_workload(cfg)
    dev = torch.device("cuda")
    Q, K, V = inp["Q"].to(dev), inp["K"].to(dev), inp["V"].to(dev)
    W = inp["W"].to(dev)
    A = None
    B, S, H, Hkv, D = cfg.B, cfg.S, cfg.H, cfg.Hkv, cfg.D
    scores = torch.empty((B, Hkv, S), dtype=torch.float32, device=dev)
    kept = dma.Kept(B, Hkv, S, cfg.w, cfg.window, cfg.block, dma.ROWWISE, device=dev)
    O = torch.empty_like(Q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        dma.dma_score_keys(V, W, A, scores, stream=stream)
        dma.dma_select_topk(scores, kept, dma.FULL, stream=stream)
        dma.dma_sparse_attn_prefill(Q, K, V, scores, kept, O, lse, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    pairs = kept_pairs(kept.expiry, S, cfg.window, cfg.block, H // Hkv)
    flops = 4.0 * D * pairs

    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(n):
        ev[s][0].record(stream)
        dma.dma_score_keys(V, W, A, scores, stream=stream)
        ev[s][1].record(stream)
        dma.dma_select_topk(scores, kept, dma.FULL, stream=stream)
        ev[s][2].record(stream)
        dma.dma_sparse_attn_prefill(Q, K, V, scores, kept, O, lse, stream=stream)
        ev[s][3].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    assert dma.dma_get_device_status() == 0
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    ms = total_ms / n
    score_ms = statistics.mean(ev[s][0].elapsed_time(ev[s][1]) for s in range(n))
    select_ms = statistics.mean(ev[s][1].elapsed_time(ev[s][2]) for s in range(n))
    attn_ms = statistics.mean(ev[s][2].elapsed_time(ev[s][3]) for s in range(n))

    # e2e: host (pinned) inputs, copies inside the timed region, read back O
    e2e = None
    if not args.no_e2e:
        hQ, hK, hV = inp["Q"].pin_memory(), inp["K"].pin_memory(), inp["V"].pin_memory()
        hW = inp["W"].pin_memory()
        hO = torch.empty(O.shape, dtype=O.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hQ, hK, hV, hW))
        d2h = hO.numel() * hO.element_size()

        def e2e_step():
            Q.copy_(hQ, non_blocking=True)
            K.copy_(hK, non_blocking=True)
            V.copy_(hV, non_blocking=True)
            W.copy_(hW, non_blocking=True)
            step()
            hO.copy_(O, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        ne = max(3, min(n, 5))
        barrier(world)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(ne):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a.elapsed_time(b), world) / ne
        e2e = {"value": round(flops * world / (e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 3),
               "steps": ne}
    attn_tflops = flops / (attn_ms * 1e-3) / 1e12
    res = {
        "cfg": cfg, "pairs": pairs, "flops": flops, "ms": ms, "score_ms": score_ms, "select_ms": select_ms,
        "attn_ms": attn_ms, "attn_tflops": attn_tflops, "clocks": clk, "e2e": e2e,
        "launches": n * (1 + LAUNCHES_SELECT_TOKEN + (2 if cfg.block > 1 else 0) + 1),
        "sparsity": 1.0 - pairs / (B * H * S * (S + 1) / 2.0),
    }
    return res


# ---------------------------------------------------------------- decode ----

def bench_decode(args, world):
    import dataclasses
    import content_aware_dynamic_dma_b300 as dma
    cfg = wl.WORKLOADS[DECODE_WL]
    if args.decode_batch != cfg.B:
        cfg = dataclasses.replace(cfg, B=args.decode_batch)
    B, L, H, Hkv, D = cfg.B, cfg.S, cfg.H, cfg.Hkv, cfg.D
    n = args.steps
    nq = args.warmup + n
    d = wl.make_workload(cfg, n_queries=nq, device="cuda")
    st = dma.DecodeState(B, L, H, Hkv, D, cfg.w, cfg.window)
    L0 = L - nq
    st.full_select(d["Kc"], d["Vc"], d["W"], length=L0)
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    lens = [torch.full((B,), L0 + k + 1, dtype=torch.int32, device="cuda") for k in range(nq)]
    stream = torch.cuda.current_stream()
    j = torch.arange(cfg.w, device="cuda")

    def rows_kept(pos):
        # kept rows of row `pos` per (b, KV head): top keys outside the window plus the window
        tc = st.kept.top_count.to(torch.int64)
        valid = (j.view(1, 1, -1) < tc.unsqueeze(-1)) & (st.kept.top_idx[:, :, :cfg.w] < pos + 1 - cfg.window)
        return valid.sum() + B * Hkv * min(cfg.window, pos + 1)

    for k in range(args.warmup):
        pos = L0 + k
        st.step(d["q"][k], d["Kc"], d["Vc"], d["W"], lens[k], pos, o, lse, stream=stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    rows = []
    barrier(world)
    torch.cuda.synchronize()
    for s in range(n):
        k = args.warmup + s
        pos = L0 + k
        ev[s][0].record(stream)
        dma.dma_score_keys(d["Vc"], d["W"], None, st.scores, pos, pos + 1, stream=stream)
        dma.dma_select_topk(st.scores, st.kept, dma.UPDATE, seq_len=lens[k], stream=stream)
        ev[s][1].record(stream)
        dma.dma_sparse_attn_decode(d["q"][k], d["Kc"], d["Vc"], st.scores, st.kept, o, st.ws, lse, lens[k],
                                   stream=stream)
        ev[s][2].record(stream)
        rows.append(rows_kept(pos))  # enqueued after the step's last event: outside the step timings
    torch.cuda.synchronize()
    barrier(world)
    assert dma.dma_get_device_status() == 0
    step_ms = max_over_ranks(sum(ev[s][0].elapsed_time(ev[s][2]) for s in range(n)), world) / n
    dec_ms = [ev[s][1].elapsed_time(ev[s][2]) for s in range(n)]
    upd_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(n)]
    kv_bytes = [int(r.item()) * 2 * D * 2 for r in rows]
    gbs = sum(kv_bytes) / (sum(dec_ms) * 1e-3) / 1e9
    return {"workload": DECODE_WL if cfg.B == wl.WORKLOADS[DECODE_WL].B else "%s_b%d" % (DECODE_WL, cfg.B), "gbs": gbs, "decode_ms": statistics.mean(dec_ms),
            "score_update_ms": statistics.mean(upd_ms), "step_ms": step_ms,
            "selected_kv_bytes_per_step": statistics.mean(kv_bytes)}


# ----------------------------------------------------------- CPU oracle -----

def oracle_sample(cfg, n_rows: int, seed: int = 0):
    """Times the fp64 oracle on the host: full score + full select, then dense
    masked attention on n_rows sampled rows of every (b, query head); the
    attention time is scaled to all S rows.  Returns (TFLOP/s on kept pairs,
    seconds spent, description, threads)."""
    import oracle
    inp = wl.make_workload(cfg)
    t0 = time.perf_counter()
    sc = oracle.score(inp["V"], inp["W"], inp["A"])
    t1 = time.perf_counter()
    ex = oracle.select(sc, cfg.w, cfg.block)
    t2 = time.perf_counter()
    rows = wl.sample_rows(cfg.S, n_rows, cfg.seed + seed, cfg.w)
    oracle.attend_rows(inp["Q"], inp["K"], inp["V"], sc, ex, rows, cfg.window, cfg.block)
    t3 = time.perf_counter()
    pairs = kept_pairs(ex, cfg.S, cfg.window, cfg.block, cfg.H // cfg.Hkv)
    est = (t1 - t0) + (t2 - t1) + (t3 - t2) * cfg.S / len(rows)
    value = 4.0 * cfg.D * pairs / est / 1e12
    desc = ("full score (%.2fs) + full select (%.2fs) + dense masked attention on %d sampled rows of every "
            "(b, query head) (%.2fs), attention scaled to all %d rows" % (t1 - t0, t2 - t1, len(rows), t3 - t2,
                                                                          cfg.S))
    return value, t3 - t0, desc, oracle.num_threads()


def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = wl.WORKLOADS[args.workload]
    vals, secs = [], []
    desc, thr = "", 1
    for s in range(args.warmup + args.steps):
        v, t, desc, thr = oracle_sample(cfg, args.ref_rows, seed=s)
        if s >= args.warmup:
            vals.append(v)
            secs.append(t)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "B": cfg.B, "S": cfg.S, "H": cfg.H, "Hkv": cfg.Hkv, "D": cfg.D,
                       "w": cfg.w, "window": cfg.window, "block": cfg.block, "mode": "rowwise"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main ----

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=PREFILL_WL,
                    choices=[PREFILL_WL, "prefill_s64k_block64_bf16", "prefill_s16k_bf16", "prefill_s4k_gqa_bf16"],
                    help="prefill workload of a step (the smaller ones serve profiling runs)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode only (a profiling aid: the line then carries no prefill metric)")
    ap.add_argument("--decode-batch", type=int, default=wl.WORKLOADS[DECODE_WL].B,
                    help="sequences of the decode workload (smaller values serve profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=4096, help="rows per (b, head) in the CPU-baseline sample")
    ap.add_argument("--ref-rows", type=int, default=256, help="rows per (b, head) per reference-arm step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        run_reference(args, world, rank)
        return

    world, rank, local = dist_setup()
    peaks = load_peaks()
    clocks = ClockSampler(local)
    if args.no_prefill:
        dec = bench_decode(args, world)
        if rank == 0:
            print(json.dumps({"metric": "decode selected-KV GB/s", "value": round(dec["gbs"], 2), "unit": "GB/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "decode": dec}), flush=True)
        return
    pf = bench_prefill(args, world, rank, peaks, clocks)
    dec = None if args.no_decode else bench_decode(args, world)

    if rank != 0:
        return
    cfg = pf["cfg"]
    value = pf["flops"] * world / (pf["ms"] * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(pf["ms"], 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "B": cfg.B, "S": cfg.S, "H": cfg.H, "Hkv": cfg.Hkv, "D": cfg.D, "w": cfg.w,
                   "window": cfg.window, "block": cfg.block, "mode": "rowwise", "parallelism": "replicas x%d" % world,
                   "l2": "inputs larger than L2 (Q+K+V+O = %.0f MB per step vs 126 MB)" % (
                       (2 * cfg.B * cfg.S * cfg.H * cfg.D * 2 + 2 * cfg.B * cfg.S * cfg.Hkv * cfg.D * 2) / 1e6),
                   "kept_pairs": pf["pairs"], "sparsity_vs_dense_causal": round(pf["sparsity"], 4)},
        "roofline": {"bound": "tensor", "kernel": "dma_sparse_attn_prefill", "achieved": round(pf["attn_tflops"], 3),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(pf["attn_tflops"] / peak, 4),
                     "frac_of_sustained": round(pf["attn_tflops"] / peaks["bf16_tflops_sustained"], 4)
                     if peaks.get("bf16_tflops_sustained") else None,
                     "peak_source": peaks["source"] + " bf16 dense (burst)", "traffic": prefill_traffic(cfg.name),
                     "traffic_unit": "bytes per launch (DRAM read + write)",
                     "algorithmic": "4*D flop per kept (query, key) pair, exact pair count from the selection"},
        "kernels_ms": {"score": round(pf["score_ms"], 4), "select": round(pf["select_ms"], 4),
                       "attention": round(pf["attn_ms"], 4)},
        "e2e": pf["e2e"],
        "gpu_launches": pf["launches"] + (0 if dec is None else LAUNCHES_PER_DECODE_STEP * args.steps),
        "clocks": pf["clocks"],
    }
    if dec is not None:
        line["decode"] = {"workload": dec["workload"], "value": round(dec["gbs"], 2), "unit": "GB/s",
                          "frac_of_hbm": round(dec["gbs"] / peaks["hbm_gbs"], 4), "peak_gbs": peaks["hbm_gbs"],
                          "decode_kernel_ms": round(dec["decode_ms"], 4),
                          "score_and_update_ms": round(dec["score_update_ms"], 4),
                          "step_ms": round(dec["step_ms"], 4),
                          "selected_kv_bytes_per_step": dec["selected_kv_bytes_per_step"]}
    if not args.no_cpu_baseline and world == 1:
        v, secs, desc, thr = oracle_sample(cfg, args.cpu_rows)
        line["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                "sample": desc, "seconds": round(secs, 2)}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
