"""The CUDA backward against the fp64 oracle's backward, through the C ABI (needs a B300).

Each case runs the forward (score, select, attend) on seeded inputs, draws a seeded
upstream gradient dO, then calls dma_sparse_attn_prefill_backward (dQ, dK, dV, ds) and
dma_score_keys_backward (dW, dA and the score's share of dV).  The oracle selects its own
kept sets from its own scores and computes the same gradients from their definitions.
Bound per gradient tensor (parity.check_grad): max |g - ref| <= TOL * max(1, max |ref|),
TOL = 1e-4 for fp32 inputs, 2e-2 for bf16 inputs.  Rows whose kept set differs by a
near-tie (parity.check_expiry) are left out, with every key such a row keeps.
"""
import pytest
import torch

import dma_workloads as wl
import oracle
import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dma():
    import content_aware_dynamic_dma_b300 as d
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return d


def _dev(inp):
    return {k: (None if v is None else v.to("cuda")) for k, v in inp.items()}


def gpu_backward(dma, d, dO, w, window, block=1, mode=0, simt=False, score_path=True):
    """Forward and backward on the GPU; returns the gradients and the forward's kept sets."""
    B, S, H, D = d["Q"].shape
    Hkv = d["K"].shape[2]
    f32 = dict(dtype=torch.float32, device="cuda")
    old = dma.dma_set_prefill_kernel(1 if simt else 0)
    try:
        O, lse, scores, kept = dma.prefill(d["Q"], d["K"], d["V"], d["W"], d["A"], w, window, block, mode)
        dQ = torch.empty((B, S, H, D), **f32)
        dK = torch.empty((B, S, Hkv, D), **f32)
        dV = torch.empty((B, S, Hkv, D), **f32)
        ds = torch.empty((B, Hkv, S), **f32)
        dma.dma_sparse_attn_prefill_backward(d["Q"], d["K"], d["V"], scores, kept, O, lse, dO.to("cuda"), dQ, dK,
                                             dV, ds)
        dVt = dV.clone()
        dW = torch.empty((Hkv, D), **f32)
        dA = torch.empty((Hkv,), **f32) if d["A"] is not None else None
        if score_path:
            dma.dma_score_keys_backward(d["V"], d["W"], d["A"], ds, dVt, dW, dA)
        torch.cuda.synchronize()
    finally:
        dma.dma_set_prefill_kernel(old)
    assert dma.dma_get_device_status() == 0
    return dict(dQ=dQ, dK=dK, dV=dV, ds=ds, dVt=dVt, dW=dW, dA=dA, kept=kept)


def run_backward_case(dma, inp, w, window, block=1, mode=0, seed=1, segment=None, rows=None, keys=None,
                      simt=False, score_path=True):
    Q = inp["Q"]
    B, S, H, D = Q.shape
    Hkv = inp["K"].shape[2]
    G = H // Hkv
    dt = Q.dtype
    dO = wl.make_grad(Q.shape, dt, seed)
    r = gpu_backward(dma, _dev(inp), dO, w, window, block, mode, simt, score_path)
    sc = oracle.score(inp["V"], inp["W"], inp["A"])
    ex = oracle.select(sc, w, block, mode)
    affected = parity.check_expiry(r["kept"].expiry, ex, sc, w, block, mode)
    ref = oracle.attend_backward(inp["Q"], inp["K"], inp["V"], sc, ex, dO, window, block, segment=segment,
                                 rows=rows, keys=keys)
    gex = r["kept"].expiry.cpu()
    segs = range(B * Hkv) if segment is None else [segment]
    row_idx = list(range(S)) if rows is None else list(rows)
    key_idx = list(range(S)) if keys is None else list(keys)
    row_mask = torch.zeros((B, S, H), dtype=torch.bool)
    key_mask = torch.zeros((B, S, Hkv), dtype=torch.bool)
    ds_mask = torch.zeros((B, Hkv, S), dtype=torch.bool)
    dropped_rows = dropped_keys = 0
    for seg in segs:
        b, h = divmod(seg, Hkv)
        bad_rows = affected.get((b, h), set())
        bad_keys = set()
        for i in bad_rows:
            bad_keys |= oracle.kept_set(ex[b, h], i, window, block) | oracle.kept_set(gex[b, h], i, window, block)
        rr = [i for i in row_idx if i not in bad_rows]
        kk = [j for j in key_idx if j not in bad_keys]
        dropped_rows += len(row_idx) - len(rr)
        dropped_keys += len(key_idx) - len(kk)
        if rr:
            row_mask[b, torch.tensor(rr), h * G:(h + 1) * G] = True
        if kk:
            key_mask[b, torch.tensor(kk), h] = True
            ds_mask[b, h, torch.tensor(kk)] = True
    stats = [parity.check_grad("dQ", r["dQ"], ref[0], dt, row_mask),
             parity.check_grad("dK", r["dK"], ref[1], dt, key_mask),
             parity.check_grad("dV", r["dV"], ref[2], dt, key_mask),
             parity.check_grad("ds", r["ds"], ref[3], dt, ds_mask)]
    if score_path:
        assert not affected, "the score path is compared only without near-tie swaps"
        dV2, dW_ref, dA_ref = oracle.score_backward(inp["V"], inp["W"], inp["A"], ref[3])
        stats.append(parity.check_grad("dV_total", r["dVt"], ref[2] + dV2, dt))
        stats.append(parity.check_grad("dW", r["dW"], dW_ref, dt))
        if r["dA"] is not None:
            stats.append(parity.check_grad("dA", r["dA"], dA_ref, dt))
    print("backward parity", dict(S=S, H=H, Hkv=Hkv, D=D, w=w, window=window, block=block, mode=mode, simt=simt,
                                  dropped_rows=dropped_rows, dropped_keys=dropped_keys), stats)
    r.update(stats=stats, ref=ref, affected=affected, dropped_rows=dropped_rows, dropped_keys=dropped_keys)
    return r


# ------------------------------------------------------------ workloads -----

def test_backward_tiny_fp32(dma):
    cfg = wl.WORKLOADS["prefill_tiny_s256_fp32"]
    run_backward_case(dma, wl.make_workload(cfg), cfg.w, cfg.window, seed=cfg.seed)


def test_backward_s4k_gqa_bf16_all_elements(dma):
    cfg = wl.WORKLOADS["prefill_s4k_gqa_bf16"]
    r = run_backward_case(dma, wl.make_workload(cfg), cfg.w, cfg.window, seed=cfg.seed)
    assert r["dropped_rows"] == 0 and r["dropped_keys"] == 0


def test_backward_s16k_bf16_one_segment(dma):
    """One (batch, KV head) segment of the 16K workload: dQ on 256 sampled rows (every query
    head of the group), dK, dV and ds on sampled keys plus the 16 best-scored keys of the
    segment (kept by thousands of rows)."""
    cfg = wl.WORKLOADS["prefill_s16k_bf16"]
    inp = wl.make_workload(cfg)
    seg = 1  # b = 0, KV head 1
    rows = wl.sample_rows(cfg.S, 256, cfg.seed, cfg.w)
    sc = oracle.score(inp["V"], inp["W"], inp["A"])
    best = torch.argsort(sc[0, seg], descending=True)[:16].tolist()
    keys = sorted(set(wl.sample_rows(cfg.S, 240, cfg.seed + 1, cfg.w)) | set(best))
    run_backward_case(dma, inp, cfg.w, cfg.window, seed=cfg.seed, segment=seg, rows=rows, keys=keys,
                      score_path=False)


# ------------------------------------------------------------ edge cases ----

EDGE = [
    # B, S, H, Hkv, D, dtype, w, window, block, mode
    (1, 1, 2, 1, 128, torch.bfloat16, 4, 0, 1, 0),        # one row
    (2, 260, 2, 2, 64, torch.bfloat16, 40, 0, 1, 0),      # one query head per KV head, D = 64
    (1, 333, 3, 1, 128, torch.bfloat16, 64, 16, 1, 0),    # odd group, ragged tail
    (1, 517, 8, 1, 128, torch.bfloat16, 200, 50, 1, 0),   # group of 8
    (1, 200, 4, 2, 64, torch.bfloat16, 0, 0, 1, 0),       # nothing kept: every gradient is 0
    (1, 384, 4, 2, 128, torch.bfloat16, 0, 100, 1, 0),    # window only
    (1, 450, 4, 2, 128, torch.bfloat16, 30, 0, 1, 1),     # global mode, empty early rows
    (1, 1100, 4, 2, 64, torch.bfloat16, 256, 64, 64, 0),  # 64-key blocks
    (1, 2048, 2, 2, 128, torch.bfloat16, 512, 64, 1, 0),  # more key blocks than the metadata ring
    (1, 129, 2, 2, 64, torch.float32, 129, 0, 1, 0),      # w >= S: dense causal
    (2, 333, 4, 1, 64, torch.float32, 37, 5, 1, 1),       # fp32, global mode, ragged tail
    (1, 700, 4, 2, 128, torch.float32, 130, 70, 64, 0),   # fp32, 64-key blocks
]


@pytest.mark.parametrize("simt", [False, True], ids=["default", "simt"])
@pytest.mark.parametrize("case", EDGE, ids=[str(i) for i in range(len(EDGE))])
def test_backward_edge_cases(dma, case, simt):
    B, S, H, Hkv, D, dtype, w, window, block, mode = case
    inp = wl.make_prefill(B, S, H, Hkv, D, dtype, seed=2000 + S + w, salient=True, with_gate=(S % 2 == 1))
    r = run_backward_case(dma, inp, w, window, block, mode, seed=S + w, simt=simt)
    if w == 0 and window == 0:
        for name in ("dQ", "dK", "dV", "ds", "dW"):
            assert float(r[name].abs().max()) == 0.0, name


def test_backward_never_kept_keys_get_zero(dma):
    """Without a window, a key that never enters the top set receives exactly zero dK, dV
    and ds on the GPU (DMA summary §五: the skipped positions' gradient is exactly 0)."""
    S, w = 1500, 48
    inp = wl.make_prefill(1, S, 4, 2, 128, torch.bfloat16, seed=2101, salient=True)
    dO = wl.make_grad(inp["Q"].shape, torch.bfloat16, 3)
    r = gpu_backward(dma, _dev(inp), dO, w, 0, score_path=False)
    ex = r["kept"].expiry.cpu()
    never = ex <= torch.arange(S)
    assert int(never.sum()) > 1000
    for h in range(2):
        idx = torch.nonzero(never[0, h]).flatten().cuda()
        assert float(r["dK"][0, idx, h].abs().max()) == 0.0
        assert float(r["dV"][0, idx, h].abs().max()) == 0.0
        assert float(r["ds"][0, h, idx].abs().max()) == 0.0


def test_backward_repeatable(dma):
    """dQ is written once per element (no atomics): bit-identical across runs.  The SIMT
    path gives every output one writer: all of it is bit-identical."""
    inp = wl.make_prefill(1, 1000, 8, 2, 128, torch.bfloat16, seed=2102, salient=True)
    dO = wl.make_grad(inp["Q"].shape, torch.bfloat16, 4)
    d = _dev(inp)
    a = gpu_backward(dma, d, dO, 96, 32)
    b = gpu_backward(dma, d, dO, 96, 32)
    assert torch.equal(a["dQ"], b["dQ"])
    s1 = gpu_backward(dma, d, dO, 96, 32, simt=True)
    s2 = gpu_backward(dma, d, dO, 96, 32, simt=True)
    for name in ("dQ", "dK", "dV", "ds", "dW"):
        assert torch.equal(s1[name], s2[name]), name
