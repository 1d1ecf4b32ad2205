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
Every other seeded workload -- the tiny fp32 one, 4K with GQA, 16K, and 64K with
64-key block selection -- is timed as well and reported under "per_config",
with FULL selection next to UPDATE for decode.  The rows the CPU baseline
computes with the fp64 oracle are compared with the timed 64K prefill's output
in the same run ("parity").

Rules kept here: W >= 3 untimed warm-up steps; inputs larger than L2 (Q, K, V
and O of one step are 1342 MB against a 126 MB L2); CUDA events on the launching
stream with a synchronize and a barrier on both sides; max over ranks; clocks
sampled by nvidia-smi during the timed regions (prefill, per-config and decode).

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
# launches of one FULL selection: 4 x (histogram, scatter) + count table + table prefix +
# boundary + walk + list count + list write + tile lists; block units add the block maxima and
# the expansion to keys; more than 64 query tiles (S > 8192) add the super-group lists
LAUNCHES_SELECT_TOKEN = 15
LAUNCHES_SELECT_BLOCK_EXTRA = 2
LAUNCHES_SELECT_SUPER_GROUPS = 1
LAUNCHES_PER_DECODE_STEP = 4  # score (new key) + update + decode partial + merge

# DRAM bytes (read + write) of one prefill attention launch on the 64K workload, from an ncu
# capture of that launch itself (metrics dram__bytes_read.sum and dram__bytes_write.sum only,
# one pass).  Valid only for the kernel source it was taken on: reported as null once that
# source changes.
PREFILL_TRAFFIC = {"workload": "prefill_s64k_bf16", "bytes": 897375232 + 510041600,
                   "source_sha256": "a07b9592472bb1a84f4ba0787d8b8ba56e035a12100a5483ac65c8e83da5c849"}


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
    if PREFILL_TRAFFIC["bytes"] is None:
        return None
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


def config_keys(cfg, pairs, world=1):
    """The `config` object of a JSON line: the workload and its sizes (the same keys in both
    arms)."""
    return {"workload": cfg.name, "B": cfg.B, "S": cfg.S, "H": cfg.H, "Hkv": cfg.Hkv, "D": cfg.D, "w": cfg.w,
            "window": cfg.window, "block": cfg.block, "mode": "rowwise", "parallelism": "replicas x%d" % world,
            "l2": "inputs larger than L2 (Q+K+V+O = %.0f MB per step vs 126 MB)" % (
                (2 * cfg.B * cfg.S * cfg.H * cfg.D * 2 + 2 * cfg.B * cfg.S * cfg.Hkv * cfg.D * 2) / 1e6),
            "kept_pairs": pairs, "sparsity_vs_dense_causal": round(1.0 - pairs / (cfg.B * cfg.H * cfg.S *
                                                                                  (cfg.S + 1) / 2.0), 4)}


# --------------------------------------------------------------- prefill ----

class Prefill:
    """Device buffers and the three calls of one prefill step for a workload."""

    def __init__(self, dma, cfg, inp=None, block=None, form=0, w_head=None):
        self.dma, self.cfg = dma, cfg
        self.form = form
        inp = wl.make_workload(cfg) if inp is None else inp
        self.inp = inp
        dev = torch.device("cuda")
        self.Q, self.K, self.V = inp["Q"].to(dev), inp["K"].to(dev), inp["V"].to(dev)
        self.W = inp["W"].to(dev)
        self.A = None if inp["A"] is None else inp["A"].to(dev)
        self.block = cfg.block if block is None else block
        B, S, H, Hkv = cfg.B, cfg.S, cfg.H, cfg.Hkv
        self.scores = torch.empty((B, Hkv, S), dtype=torch.float32, device=dev)
        # the logits' bias: the scores themselves, or delta = exp(s) in its own array
        self.bias = self.scores if form == dma.BIAS_LOG else torch.empty_like(self.scores)
        self.w_head = None if w_head is None else torch.tensor(w_head, dtype=torch.int32, device=dev)
        self.kept = dma.Kept(B, Hkv, S, cfg.w, cfg.window, self.block, dma.ROWWISE, device=dev)
        self.O = torch.empty_like(self.Q)
        self.lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
        self.launches = (1 + LAUNCHES_SELECT_TOKEN + (LAUNCHES_SELECT_BLOCK_EXTRA if self.block > 1 else 0) +
                         (LAUNCHES_SELECT_SUPER_GROUPS if S > 64 * 128 else 0) + 1)

    def calls(self, stream, ev=None):
        d = self.dma
        if ev:
            ev[0].record(stream)
        if self.form == d.BIAS_LOG:
            d.dma_score_keys(self.V, self.W, self.A, self.scores, stream=stream)
        else:
            d.dma_score_keys_bias(self.V, self.W, self.A, self.form, self.scores, self.bias, stream=stream)
        if ev:
            ev[1].record(stream)
        if self.w_head is None:
            d.dma_select_topk(self.scores, self.kept, d.FULL, stream=stream)
        else:
            d.dma_select_topk_heads(self.scores, self.kept, self.w_head, d.FULL, stream=stream)
        if ev:
            ev[2].record(stream)
        d.dma_sparse_attn_prefill(self.Q, self.K, self.V, self.bias, self.kept, self.O, self.lse, stream=stream)
        if ev:
            ev[3].record(stream)

    def pairs(self):
        return kept_pairs(self.kept.expiry, self.cfg.S, self.cfg.window, self.block, self.cfg.H // self.cfg.Hkv)

    def timed(self, steps, warmup, world=1):
        """Mean per-kernel times and the whole-step time over `steps` timed steps."""
        stream = torch.cuda.current_stream()
        for _ in range(warmup):
            self.calls(stream)
        torch.cuda.synchronize()
        assert self.dma.dma_get_device_status() == 0
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        t0.record(stream)
        for s in range(steps):
            self.calls(stream, ev[s])
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        assert self.dma.dma_get_device_status() == 0
        total_ms = max_over_ranks(t0.elapsed_time(t1), world)
        k = [statistics.mean(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(steps)) for i in range(3)]
        return {"ms": total_ms / steps, "score_ms": k[0], "select_ms": k[1], "attn_ms": k[2]}

    def e2e(self, steps):
        """The same step with Q, K, V, W copied in from pinned host memory and O copied back
        every step.  Two device buffer sets let the copies of one step overlap the compute of
        the step before (host-to-device, compute and device-to-host on three streams)."""
        d = self.dma
        hQ, hK, hV = self.inp["Q"].pin_memory(), self.inp["K"].pin_memory(), self.inp["V"].pin_memory()
        hW = self.inp["W"].pin_memory()
        hO = [torch.empty(self.O.shape, dtype=self.O.dtype).pin_memory() for _ in range(2)]
        bufs = [(self.Q, self.K, self.V, self.W, self.O),
                (torch.empty_like(self.Q), torch.empty_like(self.K), torch.empty_like(self.V),
                 torch.empty_like(self.W), torch.empty_like(self.O))]
        h2d_b = sum(t.numel() * t.element_size() for t in (hQ, hK, hV, hW))
        d2h_b = hO[0].numel() * hO[0].element_size()
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        in_done = [torch.cuda.Event() for _ in range(2)]
        cmp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def run(n):
            for i in range(n):
                k = i & 1
                Q, K, V, W, O = bufs[k]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(cmp_done[k])  # step i - 2 is done reading these inputs
                    Q.copy_(hQ, non_blocking=True)
                    K.copy_(hK, non_blocking=True)
                    V.copy_(hV, non_blocking=True)
                    W.copy_(hW, non_blocking=True)
                    in_done[k].record(s_in)
                s_cmp.wait_event(in_done[k])
                if i >= 2:
                    s_cmp.wait_event(out_done[k])  # O of step i - 2 has been read back
                d.dma_score_keys(V, W, self.A, self.scores, stream=s_cmp)
                d.dma_select_topk(self.scores, self.kept, d.FULL, stream=s_cmp)
                d.dma_sparse_attn_prefill(Q, K, V, self.scores, self.kept, O, self.lse, stream=s_cmp)
                cmp_done[k].record(s_cmp)
                s_out.wait_event(cmp_done[k])
                with torch.cuda.stream(s_out):
                    hO[k].copy_(O, non_blocking=True)
                    out_done[k].record(s_out)

        run(2)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        run(steps)
        s_in.wait_stream(s_out)
        b.record(s_in)
        torch.cuda.synchronize()
        assert d.dma_get_device_status() == 0
        return a.elapsed_time(b) / steps, h2d_b, d2h_b


# -------------------------------------------------------------- backward ----

LAUNCHES_BACKWARD = 5  # delta/zero prep, row kernel, key kernel, score backward, its finalize (bf16)


class Backward:
    """The backward calls over a forward's kept sets (dQ, dK, dV, ds, then dW, dA and the score's
    share of dV), with a seeded upstream gradient.  The forward's O, lse and selection must be in
    place (Prefill.calls has run)."""

    def __init__(self, dma, pf, seed=7):
        self.dma, self.pf = dma, pf
        cfg = pf.cfg
        B, S, H, Hkv, D = cfg.B, cfg.S, cfg.H, cfg.Hkv, cfg.D
        g = torch.Generator(device="cuda").manual_seed(seed)
        self.dO = torch.randn(pf.Q.shape, generator=g, device="cuda").to(pf.Q.dtype)
        f32 = dict(dtype=torch.float32, device="cuda")
        self.dQ = torch.empty((B, S, H, D), **f32)
        self.dK = torch.empty((B, S, Hkv, D), **f32)
        self.dV = torch.empty((B, S, Hkv, D), **f32)
        self.ds = torch.empty((B, Hkv, S), **f32)
        self.dW = torch.empty((Hkv, D), **f32)
        self.dA = torch.empty((Hkv,), **f32) if pf.A is not None else None
        self.ws = torch.empty((dma.dma_backward_workspace_size(B, S, H, Hkv, D),), dtype=torch.uint8, device="cuda")

    def calls(self, stream, ev=None):
        d, pf = self.dma, self.pf
        if ev:
            ev[0].record(stream)
        d.dma_sparse_attn_prefill_backward(pf.Q, pf.K, pf.V, pf.scores, pf.kept, pf.O, pf.lse, self.dO, self.dQ,
                                           self.dK, self.dV, self.ds, ws=self.ws, stream=stream)
        if ev:
            ev[1].record(stream)
        d.dma_score_keys_backward(pf.V, pf.W, pf.A, self.ds, self.dV, self.dW, self.dA, ws=self.ws, stream=stream)
        if ev:
            ev[2].record(stream)

    def timed(self, steps, warmup, world=1):
        stream = torch.cuda.current_stream()
        self.pf.calls(stream)
        for _ in range(warmup):
            self.calls(stream)
        torch.cuda.synchronize()
        assert self.dma.dma_get_device_status() == 0
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize()
        for s in range(steps):
            self.calls(stream, ev[s])
        torch.cuda.synchronize()
        barrier(world)
        assert self.dma.dma_get_device_status() == 0
        a = max_over_ranks(statistics.mean(ev[s][0].elapsed_time(ev[s][1]) for s in range(steps)), world)
        b = max_over_ranks(statistics.mean(ev[s][1].elapsed_time(ev[s][2]) for s in range(steps)), world)
        return {"attn_bwd_ms": a, "score_bwd_ms": b, "ms": a + b}


def backward_entry(pf, r, peaks, steps):
    """The backward's numbers for a workload: FLOPs by the usual convention of 2.5 times the
    forward (S recomputed once, then dP, dQ, dK and dV: 10 D flop per kept pair)."""
    cfg = pf.cfg
    pairs = pf.pairs()
    flops = 10.0 * cfg.D * pairs
    tf = flops / (r["ms"] * 1e-3) / 1e12
    ent = {"ms": round(r["ms"], 4), "attention_backward_ms": round(r["attn_bwd_ms"], 4),
           "score_backward_ms": round(r["score_bwd_ms"], 4), "tflops": round(tf, 3),
           "algorithmic": "10*D flop per kept (query, key) pair (5 products of 2*D; the kernels form "
                          "S and dP in both the row and the key kernel: 14*D of tensor work)",
           "gpu_launches": LAUNCHES_BACKWARD * steps}
    if cfg.dtype != "f32":
        ent["frac_of_bf16_peak"] = round(tf / peaks["bf16_tflops"], 4)
        ent["tensor_work_frac_of_bf16_peak"] = round(tf * 1.4 / peaks["bf16_tflops"], 4)
    return ent


# ---------------------------------------------------------------- decode ----

def decode_parity(cfg, nq, st, o, lse, sample):
    """The timed decode's last step (row L - 1 of every cache) against the oracle on the sampled
    sequences, regenerated from their own seeds: the top sets compared exactly except near-tie
    swaps (a KV head with one is left out of the output check), outputs with the tests' bound
    (2e-2 on the arithmetic plus half a bf16 ulp for the output's rounding)."""
    import numpy as np
    import oracle
    L, Hkv, H = cfg.S, cfg.Hkv, cfg.H
    G = H // Hkv
    h_inp = {k: (None if v is None else v.cpu())
             for k, v in wl.make_workload(cfg, n_queries=nq, device="cuda", batches=sample).items()}
    sc = oracle.score(h_inp["Vc"], h_inp["W"], None)
    o_ref, lse_ref = oracle.decode(h_inp["q"][nq - 1], h_inp["Kc"], h_inp["Vc"], [L] * len(sample), sc, cfg.w,
                                   cfg.window)
    ex = oracle.select(sc, cfg.w)
    keep = torch.ones((len(sample), H), dtype=torch.bool)
    swaps = 0
    for r, b in enumerate(sample):
        for h in range(Hkv):
            got = set(st.kept.top_idx[b, h, :int(st.kept.top_count[b, h])].tolist())
            want = set(torch.nonzero(ex[r, h] >= L).flatten().tolist())
            if got != want:
                s32 = sc[r, h].numpy().astype(np.float32).astype(np.float64)
                cut = min(s32[list(want)])
                if any(abs(s32[j] - cut) > 1e-5 for j in got ^ want):
                    return {"sequences": sample, "ok": False, "reason": "kept set differs beyond a near tie"}
                keep[r, h * G:(h + 1) * G] = False
                swaps += 1
    g = o[sample].double().cpu()
    _, e = torch.frexp(o_ref.abs())
    half_ulp = torch.ldexp(torch.ones_like(o_ref), (e - 9).to(torch.int32))
    err = (g - o_ref).abs().amax(dim=-1)
    ex_half = ((g - o_ref).abs() - half_ulp).amax(dim=-1)
    lse_err = (lse[sample].double().cpu() - lse_ref).abs()
    return {"sequences": sample, "kv_heads_left_out_near_ties": swaps,
            "max_abs_err": round(float(err[keep].max()), 5), "max_err_less_half_ulp": round(float(ex_half[keep].max()), 5),
            "lse_max_abs_err": round(float(lse_err[keep].max()), 6),
            "ok": bool(float(ex_half[keep].max()) <= 2e-2 and float(lse_err[keep].max()) <= 2e-2)}


def bench_decode(args, world, check=False):
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
    stream = torch.cuda.current_stream()
    # FULL selection over the score cache (the decode set-up, and c5's FULL figure)
    st.full_select(d["Kc"], d["Vc"], d["W"], length=L0)
    full = dma.Kept(B, Hkv, L0, cfg.w, cfg.window, 1, dma.ROWWISE, tiles=False)
    sc0 = st.scores[:, :, :L0].contiguous()
    for _ in range(2):
        dma.dma_select_topk(sc0, full, dma.FULL, stream=stream)
    torch.cuda.synchronize()
    fe = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    fe[0].record(stream)
    for i in range(3):
        dma.dma_select_topk(sc0, full, dma.FULL, stream=stream)
        fe[i + 1].record(stream)
    torch.cuda.synchronize()
    full_ms = statistics.median(fe[i].elapsed_time(fe[i + 1]) for i in range(3))
    del full, sc0
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    lens = [torch.full((B,), L0 + k + 1, dtype=torch.int32, device="cuda") for k in range(nq)]
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
    out = {"workload": DECODE_WL if cfg.B == wl.WORKLOADS[DECODE_WL].B else "%s_b%d" % (DECODE_WL, cfg.B),
           "gbs": gbs, "decode_ms": statistics.mean(dec_ms), "score_update_ms": statistics.mean(upd_ms),
           "step_ms": step_ms, "selected_kv_bytes_per_step": statistics.mean(kv_bytes),
           "full_select_ms": full_ms, "full_select_keys": B * Hkv * L0}
    if check:  # kept for the CPU-baseline leg, which checks this step against the oracle
        out["_last_step"] = (cfg, nq, st, o, lse)
    return out


def bench_nsa(dma, pf, peaks, steps, warmup, world=1):
    """The NSA-style three-branch step on the prefill workload's inputs: score, 64-key block
    selection, block compression, the compressed, selected and sliding attentions, and the gated
    sum.  TFLOP/s counts 4*D per kept pair over the three branches (exact counts: the compressed
    blocks each row sees, the selection's intervals, the window band)."""
    cfg = pf.cfg
    B, S, H, Hkv, D = cfg.B, cfg.S, cfg.H, cfg.Hkv, cfg.D
    G, c = wl.make_nsa_gates(H, D, cfg.seed)
    G, c = G.cuda(), c.cuda()
    st = dma.NsaPrefill(B, S, H, Hkv, D, cfg.w, cfg.window, dtype=pf.Q.dtype)
    O = torch.empty_like(pf.Q)
    stream = torch.cuda.current_stream()
    names = ["score", "select", "compress", "attn_compressed", "attn_selected", "attn_window", "combine"]

    def step(ev=None):
        calls = [lambda: dma.dma_score_keys(pf.V, pf.W, pf.A, st.scores, stream=stream),
                 lambda: dma.dma_select_topk(st.scores, st.kept_slc, dma.FULL, stream=stream),
                 lambda: dma.dma_nsa_compress(pf.K, pf.V, st.Kc, st.Vc, stream=stream),
                 lambda: dma.dma_sparse_attn_prefill(pf.Q, st.Kc, st.Vc, st.zero, st.kept_cmp, st.o_cmp, None,
                                                     stream=stream),
                 lambda: dma.dma_sparse_attn_prefill(pf.Q, pf.K, pf.V, st.zero, st.kept_slc, st.o_slc, None,
                                                     stream=stream),
                 lambda: dma.dma_sparse_attn_prefill(pf.Q, pf.K, pf.V, st.zero, st.kept_win, st.o_win, None,
                                                     stream=stream),
                 lambda: dma.dma_nsa_combine(pf.Q, st.o_cmp, st.o_slc, st.o_win, G, c, O, stream=stream)]
        for i, call in enumerate(calls):
            if ev:
                ev[i].record(stream)
            call()
        if ev:
            ev[len(calls)].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for s_ in range(steps):
        step(ev[s_])
    torch.cuda.synchronize()
    barrier(world)
    assert dma.dma_get_device_status() == 0
    k_ms = {n: statistics.mean(ev[s_][i].elapsed_time(ev[s_][i + 1]) for s_ in range(steps))
            for i, n in enumerate(names)}
    total = max_over_ranks(statistics.mean(ev[s_][0].elapsed_time(ev[s_][-1]) for s_ in range(steps)), world)
    G_ = H // Hkv
    i = torch.arange(S, dtype=torch.int64)
    p_cmp = int(((i + 1) // 64).sum()) * B * H
    p_slc = kept_pairs(st.kept_slc.expiry, S, 0, 64, G_)
    p_win = int(torch.clamp(i + 1, max=cfg.window).sum()) * B * H
    pairs = p_cmp + p_slc + p_win
    fl = 4.0 * D

    def tf(p, ms):
        return round(fl * p / (ms * 1e-3) / 1e12, 3)
    comb_bytes = 5 * B * S * H * D * pf.Q.element_size()
    ent = {"workload": cfg.name + "_nsa3", "B": B, "S": S, "H": H, "Hkv": Hkv, "D": D, "w": cfg.w,
           "window": cfg.window, "block": 64, "kept_pairs": {"compressed": p_cmp, "selected": p_slc,
                                                            "window": p_win},
           "kernels_ms": {n: round(v, 4) for n, v in k_ms.items()}, "step_ms": round(total, 4),
           "step_tflops": tf(pairs, total),
           "attention_tflops": {"compressed": tf(p_cmp, k_ms["attn_compressed"]),
                                "selected": tf(p_slc, k_ms["attn_selected"]),
                                "window": tf(p_win, k_ms["attn_window"])},
           "combine_gbs": round(comb_bytes / (k_ms["combine"] * 1e-3) / 1e9, 1),
           "combine_frac_of_hbm": round(comb_bytes / (k_ms["combine"] * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
           "compress_gbs": round(2 * B * S * Hkv * D * pf.Q.element_size() / (k_ms["compress"] * 1e-3) / 1e9, 1),
           "gates": "random-init G ~ N(0, 0.01), c ~ N(0, 1) (no trained gates)",
           "fixed_patterns": "the compressed and window kept structures depend on S and the window only: "
                             "built once, outside the timed steps"}
    ent["attention_frac_of_bf16_peak"] = {k: round(v / peaks["bf16_tflops"], 4)
                                          for k, v in ent["attention_tflops"].items()}
    del st
    torch.cuda.empty_cache()
    return ent


def bench_decode_nsa(args, world):
    """The NSA-style three-branch decode on the decode workload: each step scores the new key
    (and its 64-key block), compresses a block when the step completes one, selects the blocks
    of the decode row, runs the compressed, selected and sliding decodes and the gated sum.
    GB/s counts the K/V rows the three decodes read (compressed rows, selected blocks, window)."""
    import dataclasses
    import content_aware_dynamic_dma_b300 as dma
    cfg = wl.WORKLOADS[DECODE_WL]
    if args.decode_batch != cfg.B:
        cfg = dataclasses.replace(cfg, B=args.decode_batch)
    B, L, H, Hkv, D = cfg.B, cfg.S, cfg.H, cfg.Hkv, cfg.D
    n = args.steps
    nq = args.warmup + n
    d = wl.make_workload(cfg, n_queries=nq, device="cuda")
    G, c = wl.make_nsa_gates(H, D, cfg.seed)
    G, c = G.cuda(), c.cuda()
    st = dma.NsaDecode(B, L, H, Hkv, D, cfg.w, cfg.window)
    L0 = L - nq
    stream = torch.cuda.current_stream()
    st.prepare(d["Kc"], d["Vc"], d["W"], torch.full((B,), L0, dtype=torch.int32, device="cuda"), L0,
               stream=stream)
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    lens = [torch.full((B,), L0 + k + 1, dtype=torch.int32, device="cuda") for k in range(nq)]
    for k in range(args.warmup):
        st.step(d["q"][k], d["Kc"], d["Vc"], d["W"], lens[k], L0 + k, G, c, o, stream=stream)
    torch.cuda.synchronize()
    # the step's calls, as NsaDecode.step makes them, with events between the parts
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
    rows = []
    ks = st.kept_slc
    barrier(world)
    torch.cuda.synchronize()
    for s_ in range(n):
        k = args.warmup + s_
        pos = L0 + k
        q = d["q"][k]
        ev[s_][0].record(stream)
        dma.dma_score_keys_paged(st._pages(d["Vc"]), st.block_table, d["W"], None, st.scores, st.page_scores,
                                 lens[k], pos, pos + 1, stream=stream)
        if (pos + 1) % 64 == 0:
            dma.dma_nsa_compress(d["Kc"], d["Vc"], st.Kc, st.Vc, pos // 64, pos // 64 + 1, stream=stream)
            dma.dma_nsa_kept_pattern(dma.NSA_COMPRESSED, st.kept_cmp, lens[k], stream=stream)
        dma.dma_select_pages(st.page_scores, 64, cfg.w, ks.top_idx, ks.top_count, lens[k], stream=stream)
        ev[s_][1].record(stream)
        dma.dma_sparse_attn_decode(q, st.Kc, st.Vc, st.zero, st.kept_cmp, st.o_cmp, st.ws, None, lens[k],
                                   stream=stream)
        ev[s_][2].record(stream)
        dma.dma_sparse_attn_decode(q, d["Kc"], d["Vc"], st.zero, ks, st.o_slc, st.ws, None, lens[k], stream=stream)
        dma.dma_sparse_attn_decode(q, d["Kc"], d["Vc"], st.zero, st.kept_win, st.o_win, st.ws, None, lens[k],
                                   stream=stream)
        ev[s_][3].record(stream)
        dma.dma_nsa_combine(q, st.o_cmp, st.o_slc, st.o_win, G, c, o, stream=stream)
        ev[s_][4].record(stream)
        Lk = pos + 1
        # rows read: the compressed rows, the selected blocks' keys and the window (all heads)
        rows.append((ks.top_count.sum(), B * Hkv * (Lk // 64), B * Hkv * min(cfg.window, Lk)))
    torch.cuda.synchronize()
    barrier(world)
    assert dma.dma_get_device_status() == 0

    def mean_ms(i0, i1):
        return statistics.mean(ev[s_][i0].elapsed_time(ev[s_][i1]) for s_ in range(n))
    t = max_over_ranks(mean_ms(0, 4), world)
    row_b = 2 * D * 2
    b_cmp = statistics.mean(int(r[1]) * row_b for r in rows)
    b_sw = statistics.mean((int(r[0].item()) + int(r[2])) * row_b for r in rows)
    dec_ms = mean_ms(1, 3)
    return {"step_ms": round(t, 4), "kv_rows_bytes_per_step": b_cmp + b_sw,
            "gbs": round((b_cmp + b_sw) / (t * 1e-3) / 1e9, 1),
            "kernels_ms": {"score_block_score_select": round(mean_ms(0, 1), 4),
                           "decode_compressed": round(mean_ms(1, 2), 4),
                           "decode_selected_and_window": round(mean_ms(2, 3), 4),
                           "gated_sum": round(mean_ms(3, 4), 4)},
            "decode_gbs": round((b_cmp + b_sw) / (dec_ms * 1e-3) / 1e9, 1),
            "note": "gbs: the whole step against the K/V bytes the three decodes read; decode_gbs: the three "
                    "decode launches alone"}


def bench_decode_paged(args, world, page_size=64):
    """The decode workload over a paged cache (pages of `page_size` tokens in random physical
    order): each step scores the new key and its page, selects the pages, and attends."""
    import dataclasses
    import content_aware_dynamic_dma_b300 as dma
    cfg = wl.WORKLOADS[DECODE_WL]
    if args.decode_batch != cfg.B:
        cfg = dataclasses.replace(cfg, B=args.decode_batch)
    B, L, H, Hkv, D = cfg.B, cfg.S, cfg.H, cfg.Hkv, cfg.D
    n = args.steps
    nq = args.warmup + n
    d = wl.make_workload(cfg, n_queries=nq, device="cuda")
    Kp, bt = wl.paginate(d.pop("Kc"), page_size, seed=cfg.seed)
    Vp, _ = wl.paginate(d.pop("Vc"), page_size, seed=cfg.seed)
    torch.cuda.empty_cache()
    st = dma.PagedDecodeState(B, bt.shape[1], page_size, H, Hkv, D, cfg.w, cfg.window)
    L0 = L - nq
    stream = torch.cuda.current_stream()
    st.full_score(Vp, bt, d["W"], cache_len=torch.full((B,), L0, dtype=torch.int32, device="cuda"))
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    lens = [torch.full((B,), L0 + k + 1, dtype=torch.int32, device="cuda") for k in range(nq)]
    j = torch.arange(st.top_cap, device="cuda")

    def rows_kept(pos):
        # kept rows per (b, KV head): keys of the kept pages outside the window, plus the window
        tc = st.top_count.to(torch.int64)
        valid = (j.view(1, 1, -1) < tc.unsqueeze(-1)) & (st.top_idx < pos + 1 - cfg.window)
        return valid.sum() + B * Hkv * min(cfg.window, pos + 1)

    for k in range(args.warmup):
        st.step(d["q"][k], Kp, Vp, bt, d["W"], lens[k], L0 + k, o, lse, stream=stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    rows = []
    barrier(world)
    torch.cuda.synchronize()
    for s in range(n):
        k = args.warmup + s
        pos = L0 + k
        ev[s][0].record(stream)
        dma.dma_score_keys_paged(Vp, bt, d["W"], None, st.scores, st.page_scores, lens[k], pos, pos + 1,
                                 stream=stream)
        dma.dma_select_pages(st.page_scores, page_size, cfg.w, st.top_idx, st.top_count, lens[k], stream=stream)
        ev[s][1].record(stream)
        dma.dma_sparse_attn_decode_paged(d["q"][k], Kp, Vp, bt, st.scores, st.top_idx, st.top_count, cfg.window, o,
                                         st.ws, lse, lens[k], stream=stream)
        ev[s][2].record(stream)
        rows.append(rows_kept(pos))
    torch.cuda.synchronize()
    barrier(world)
    assert dma.dma_get_device_status() == 0
    step_ms = max_over_ranks(sum(ev[s][0].elapsed_time(ev[s][2]) for s in range(n)), world) / n
    dec_ms = [ev[s][1].elapsed_time(ev[s][2]) for s in range(n)]
    sel_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(n)]
    kv_bytes = [int(r.item()) * 2 * D * 2 for r in rows]
    return {"page_size": page_size, "gbs": sum(kv_bytes) / (sum(dec_ms) * 1e-3) / 1e9,
            "decode_ms": statistics.mean(dec_ms), "score_and_select_pages_ms": statistics.mean(sel_ms),
            "step_ms": step_ms, "selected_kv_bytes_per_step": statistics.mean(kv_bytes)}


# ----------------------------------------------------------- CPU oracle -----

def oracle_sample(cfg, n_rows: int, seed: int = 0, out=None):
    """Times the fp64 oracle on the host: full score + full select, then dense
    masked attention on n_rows sampled rows of every (b, query head); the
    attention time is scaled to all S rows.  Returns (TFLOP/s on kept pairs,
    seconds spent, description, threads, kept pairs); with `out` a dict, also
    leaves the sampled rows and the oracle's results there."""
    import oracle
    inp = wl.make_workload(cfg)
    t0 = time.perf_counter()
    sc = oracle.score(inp["V"], inp["W"], inp["A"])
    t1 = time.perf_counter()
    ex = oracle.select(sc, cfg.w, cfg.block)
    t2 = time.perf_counter()
    rows = wl.sample_rows(cfg.S, n_rows, cfg.seed + seed, cfg.w)
    O_ref, lse_ref = oracle.attend_rows(inp["Q"], inp["K"], inp["V"], sc, ex, rows, cfg.window, cfg.block)
    t3 = time.perf_counter()
    if out is not None:
        out.update(rows=rows, O_ref=O_ref, lse_ref=lse_ref, expiry=ex)
    pairs = kept_pairs(ex, cfg.S, cfg.window, cfg.block, cfg.H // cfg.Hkv)
    est = (t1 - t0) + (t2 - t1) + (t3 - t2) * cfg.S / len(rows)
    value = 4.0 * cfg.D * pairs / est / 1e12
    desc = ("full score (%.2fs) + full select (%.2fs) + dense masked attention on %d sampled rows of every "
            "(b, query head) (%.2fs), attention scaled to all %d rows" % (t1 - t0, t2 - t1, len(rows), t3 - t2,
                                                                          cfg.S))
    return value, t3 - t0, desc, oracle.num_threads(), pairs


def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = wl.WORKLOADS[args.workload]
    vals, secs = [], []
    desc, thr, pairs = "", 1, 0
    for s in range(args.warmup + args.steps):
        v, t, desc, thr, pairs = oracle_sample(cfg, args.ref_rows, seed=s)
        if s >= args.warmup:
            vals.append(v)
            secs.append(t)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_keys(cfg, pairs, world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main ----

PER_CONFIG = ["prefill_tiny_s256_fp32", "prefill_s4k_gqa_bf16", "prefill_s16k_bf16", "prefill_s64k_block64_bf16"]
# a non-uniform allocation over the 8 KV heads of the 64K workload (at most its w = 4096)
PER_HEAD_BUDGETS = [512, 1024, 2048, 4096, 4096, 2048, 1024, 512]


def parity_vs_oracle(pf, ref):
    """The timed 64K prefill against the oracle rows of the CPU-baseline sample: per-key
    intervals compared exactly; outputs on the sampled rows with the tests' bound (2e-2 on bf16
    arithmetic plus half a bf16 ulp for the output's rounding), leaving out the rows of a
    KV-head group whose kept set a near-tie swap changed (a key whose expiry differs)."""
    cfg = pf.cfg
    G = cfg.H // cfg.Hkv
    rows = ref["rows"]
    ge = pf.kept.expiry.cpu().to(torch.int64)
    oe = ref["expiry"].to(torch.int64)
    j = torch.arange(cfg.S)
    lo = j if pf.block <= 1 else (j // pf.block) * pf.block + pf.block - 1
    keep = torch.ones((cfg.B, len(rows), cfg.H), dtype=torch.bool)
    rt = torch.tensor(rows, dtype=torch.int64)
    n_diff = 0
    for b in range(cfg.B):
        for h in range(cfg.Hkv):
            bad = torch.nonzero(ge[b, h] != oe[b, h]).flatten()
            n_diff += len(bad)
            for jj in bad.tolist():
                a0 = max(int(lo[jj]), int(min(ge[b, h, jj], oe[b, h, jj])))
                a1 = int(max(ge[b, h, jj], oe[b, h, jj]))
                hit = (rt >= a0) & (rt < a1)
                keep[b, hit, h * G:(h + 1) * G] = False
    g = pf.O.double().cpu()[:, rows]
    O_ref = ref["O_ref"]
    _, e = torch.frexp(O_ref.abs())
    half_ulp = torch.ldexp(torch.ones_like(O_ref), (e - 9).to(torch.int32))
    err = ((g - O_ref).abs()).amax(dim=-1)
    ex_half = ((g - O_ref).abs() - half_ulp).amax(dim=-1)
    lse_err = (pf.lse.double().cpu()[:, :, rows] - ref["lse_ref"]).abs().permute(0, 2, 1)
    k = keep
    return {"rows_per_head": len(rows), "expiry_keys_differing": n_diff,
            "row_heads_left_out_near_ties": int((~k).sum()),
            "max_abs_err": round(float(err[k].max()), 5), "max_err_less_half_ulp": round(float(ex_half[k].max()), 5),
            "lse_max_abs_err": round(float(lse_err[k].max()), 6),
            "ok": bool(float(ex_half[k].max()) <= 2e-2 and float(lse_err[k].max()) <= 2e-2)}


def per_config_entry(pf, r, peaks):
    cfg = pf.cfg
    pairs = pf.pairs()
    flops = 4.0 * cfg.D * pairs
    attn = flops / (r["attn_ms"] * 1e-3) / 1e12
    ent = {"dtype": "f32" if cfg.dtype == "f32" else "bf16", "B": cfg.B, "S": cfg.S, "H": cfg.H, "Hkv": cfg.Hkv,
           "D": cfg.D, "w": cfg.w, "window": cfg.window, "block": pf.block, "kept_pairs": pairs,
           "kernels_ms": {"score": round(r["score_ms"], 4), "select": round(r["select_ms"], 4),
                          "attention": round(r["attn_ms"], 4)},
           "step_ms": round(r["ms"], 4), "step_tflops": round(flops / (r["ms"] * 1e-3) / 1e12, 3),
           "attention_tflops": round(attn, 3)}
    if cfg.dtype == "f32":
        ent["roofline"] = "fp32 SIMT path (TF32 would break the 1e-4 bound): no tensor-core peak applies"
    else:
        ent["attention_frac_of_bf16_peak"] = round(attn / peaks["bf16_tflops"], 4)
    return ent


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
    ap.add_argument("--nsa-only", action="store_true",
                    help="the NSA-style three-branch step on the --workload inputs only (a profiling aid)")
    ap.add_argument("--decode-batch", type=int, default=wl.WORKLOADS[DECODE_WL].B,
                    help="sequences of the decode workload (smaller values serve profiling runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
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
    import content_aware_dynamic_dma_b300 as dma
    if args.no_prefill:
        dec = bench_decode(args, world)
        if rank == 0:
            print(json.dumps({"metric": "decode selected-KV GB/s", "value": round(dec["gbs"], 2), "unit": "GB/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "decode": dec}), flush=True)
        return
    cfg = wl.WORKLOADS[args.workload]
    pf = Prefill(dma, cfg)
    if args.nsa_only:
        nsa = bench_nsa(dma, pf, peaks, args.steps, args.warmup, world)
        if rank == 0:
            print(json.dumps({"metric": "NSA-style three-branch step TFLOP/s", "value": nsa["step_tflops"],
                              "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "nsa": nsa}), flush=True)
        return
    clocks.start()
    r = pf.timed(args.steps, args.warmup, world)
    pairs = pf.pairs()
    flops = 4.0 * cfg.D * pairs
    e2e = None
    if not args.no_e2e:
        ne = max(3, min(args.steps, 5))
        e_ms, h2d, d2h = pf.e2e(ne)
        e_ms = max_over_ranks(e_ms, world)
        e2e = {"value": round(flops * world / (e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 3), "steps": ne,
               "overlap": "copies of one step overlap the compute of the step before (two buffer sets, "
                          "three streams)"}
    bwd = None
    if not args.no_backward:
        bw = Backward(dma, pf)
        bwd = backward_entry(pf, bw.timed(args.steps, args.warmup, world), peaks, args.steps)
        bwd["workload"] = cfg.name
        del bw
        torch.cuda.empty_cache()
    per_config = {}
    if not args.no_per_config:
        for name in PER_CONFIG:
            c = wl.WORKLOADS[name]
            if name == "prefill_s64k_block64_bf16" and cfg.name == PREFILL_WL:
                p = Prefill(dma, c, inp=pf.inp, block=64)  # the same 64K inputs, 64-key block units
            else:
                p = Prefill(dma, c)
            per_config[name] = per_config_entry(p, p.timed(args.steps, args.warmup, world), peaks)
            if not args.no_backward and name != "prefill_s64k_block64_bf16":
                bw = Backward(dma, p)
                per_config[name]["backward"] = backward_entry(p, bw.timed(args.steps, args.warmup, world), peaks,
                                                              args.steps)
                del bw
            del p
            torch.cuda.empty_cache()
        if cfg.name == PREFILL_WL:
            # the two variants on the same 64K inputs: the exp-form bias, and a budget per KV head
            for key, kw in (("prefill_s64k_bf16_exp_bias", dict(form=dma.BIAS_EXP)),
                            ("prefill_s64k_bf16_per_head_budgets", dict(w_head=PER_HEAD_BUDGETS))):
                p = Prefill(dma, cfg, inp=pf.inp, **kw)
                per_config[key] = per_config_entry(p, p.timed(args.steps, args.warmup, world), peaks)
                per_config[key].update({"bias": "exp(s)" if "form" in kw else "s",
                                        "w_head": kw.get("w_head", [cfg.w] * cfg.Hkv)})
                del p
                torch.cuda.empty_cache()
            nsa = bench_nsa(dma, pf, peaks, args.steps, args.warmup, world)
            per_config[nsa["workload"]] = nsa
    dec = None if args.no_decode else bench_decode(args, world, check=(rank == 0 and not args.no_cpu_baseline))
    pdec = None if (args.no_decode or args.no_per_config) else bench_decode_paged(args, world)
    ndec = None if (args.no_decode or args.no_per_config) else bench_decode_nsa(args, world)
    clk = clocks.stop()

    if rank != 0:
        return
    value = flops * world / (r["ms"] * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    attn_tflops = flops / (r["attn_ms"] * 1e-3) / 1e12
    launches = args.steps * pf.launches
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(r["ms"], 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_keys(cfg, pairs, world),
        "roofline": {"bound": "tensor", "kernel": "dma_sparse_attn_prefill", "achieved": round(attn_tflops, 3),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(attn_tflops / peak, 4),
                     "frac_of_sustained": round(attn_tflops / peaks["bf16_tflops_sustained"], 4)
                     if peaks.get("bf16_tflops_sustained") else None,
                     "peak_source": peaks["source"] + " bf16 dense (burst)", "traffic": prefill_traffic(cfg.name),
                     "traffic_unit": "bytes per launch (DRAM read + write)",
                     "algorithmic": "4*D flop per kept (query, key) pair, exact pair count from the selection"},
        "kernels_ms": {"score": round(r["score_ms"], 4), "select": round(r["select_ms"], 4),
                       "attention": round(r["attn_ms"], 4)},
        "e2e": e2e,
        "gpu_launches": launches + (0 if dec is None else LAUNCHES_PER_DECODE_STEP * args.steps),
        "clocks": clk,
    }
    if bwd is not None:
        line["backward"] = bwd
    if dec is not None:
        line["decode"] = {"workload": dec["workload"], "value": round(dec["gbs"], 2), "unit": "GB/s",
                          "frac_of_hbm": round(dec["gbs"] / peaks["hbm_gbs"], 4), "peak_gbs": peaks["hbm_gbs"],
                          "decode_kernel_ms": round(dec["decode_ms"], 4),
                          "score_and_update_ms": round(dec["score_update_ms"], 4),
                          "step_ms": round(dec["step_ms"], 4),
                          "selected_kv_bytes_per_step": dec["selected_kv_bytes_per_step"]}

        per_config[dec["workload"]] = {
            "update_select_and_score_ms": round(dec["score_update_ms"], 4),
            "full_select_ms": round(dec["full_select_ms"], 4), "full_select_keys": dec["full_select_keys"],
            "decode_kernel_ms": round(dec["decode_ms"], 4), "decode_gbs": round(dec["gbs"], 2),
            "decode_frac_of_hbm": round(dec["gbs"] / peaks["hbm_gbs"], 4)}
    if pdec is not None:
        per_config[DECODE_WL + "_paged%d" % pdec["page_size"]] = {
            "page_size": pdec["page_size"], "score_and_select_pages_ms": round(pdec["score_and_select_pages_ms"], 4),
            "decode_kernel_ms": round(pdec["decode_ms"], 4), "decode_gbs": round(pdec["gbs"], 2),
            "decode_frac_of_hbm": round(pdec["gbs"] / peaks["hbm_gbs"], 4), "step_ms": round(pdec["step_ms"], 4),
            "selected_kv_bytes_per_step": pdec["selected_kv_bytes_per_step"],
            "layout": "K/V pages [n_pages][page_size][Hkv][D] in random physical order behind a block table"}
    if ndec is not None:
        ndec["frac_of_hbm"] = round(ndec["gbs"] / peaks["hbm_gbs"], 4)
        ndec["decode_frac_of_hbm"] = round(ndec["decode_gbs"] / peaks["hbm_gbs"], 4)
        per_config[DECODE_WL + "_nsa3"] = ndec
    if per_config:
        line["per_config"] = per_config
    if not args.no_cpu_baseline and world == 1:
        ref = {}
        v, secs, desc, thr, _ = oracle_sample(cfg, args.cpu_rows, out=ref)
        line["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                "sample": desc, "seconds": round(secs, 2)}
        # the oracle rows of that sample, against the timed run's output
        line["parity"] = parity_vs_oracle(pf, ref)
        if dec is not None and "_last_step" in dec:
            # the oracle's decode of three sampled sequences, timed, against the timed decode's last step
            dcfg, nq, dst, do, dlse = dec["_last_step"]
            sample = sorted({0, dcfg.B // 2, dcfg.B - 1})
            t0 = time.perf_counter()
            dpar = decode_parity(dcfg, nq, dst, do, dlse, sample)
            secs = time.perf_counter() - t0
            line["cpu_baseline"]["decode"] = {
                "sample": "%d of %d sequences: score, select and decode row of %d cached tokens" % (
                    len(sample), dcfg.B, dcfg.S), "seconds": round(secs, 2),
                "value": round(dec["selected_kv_bytes_per_step"] * len(sample) / dcfg.B / secs / 1e9, 6),
                "unit": "GB/s of selected K/V (the oracle also scores and selects)"}
            line["decode"]["parity"] = dpar
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
