"""Per-KV-head budgets and the exp form of the bias, CUDA path against the fp64 oracle
through the C ABI (needs a B300).

Per-head budgets (dma_select_topk_heads, dma_select_pages_heads): the oracle selects
each KV head with its own budget; the comparison is that of the uniform selection
(expiry exact except near-cutoff ties, tile lists and bitmaps exact, outputs within
2e-2 / 1e-4).  A budget list that repeats one value gives the uniform selection's
arrays bit for bit.

Exp form (dma_score_keys_bias with DMA_BIAS_EXP, dma_score_keys_backward_bias): the
logits get delta = exp(s).  The bias is checked against the oracle's exp(s) with the
bound that the score's own bound implies, |delta/delta_ref - 1| <= expm1(e_s) + 4e-7
with e_s = 5e-5 + 1e-5 |s| (the score's fp32 bound, plus a few ulps of expf).  A logit
error of delta * e_s grows with delta, so the exp-form workloads keep delta moderate
(s below about 4.5): the unit-variance weights of the 4K workload, smaller ones for fp32.
"""
import math

import numpy as np
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


def _wh(lst):
    return torch.tensor(lst, dtype=torch.int32, device="cuda")


def check_bias(bias_gpu, sc_ref):
    """The exp-form bias against exp of the oracle's score, with the bound the score implies."""
    g = bias_gpu.double().cpu()
    ref = torch.exp(sc_ref)
    e_s = parity.SCORE_ATOL + parity.SCORE_RTOL * sc_ref.abs()
    rel = (g / ref - 1.0).abs()
    bound = torch.expm1(e_s) + 4e-7
    assert bool((rel <= bound).all()), "bias error %.3g above its bound" % float((rel - bound).max())


def run_case(dma, inp, w, window, block=1, mode=0, w_head=None, form="log", rows=None, check_tiles=True,
             tiles=None):
    """Score, select and attend on the GPU; compare with the oracle.  Returns the GPU arrays."""
    Q = inp["Q"]
    B, S, H, D = Q.shape
    Hkv = inp["K"].shape[2]
    d = _dev(inp)
    O, lse, bias, kept = dma.prefill(d["Q"], d["K"], d["V"], d["W"], d["A"], w, window, block, mode,
                                     form=dma.BIAS_EXP if form == "exp" else dma.BIAS_LOG,
                                     w_head=None if w_head is None else _wh(w_head))
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    sc = oracle.score(inp["V"], inp["W"], inp["A"])
    ex = oracle.select(sc, w if w_head is None else w_head, block, mode)
    affected = parity.check_expiry(kept.expiry, ex, sc, w, block, mode)
    if form == "exp":
        check_bias(bias, sc)
    if check_tiles:
        lists, bitmaps = parity.expected_tiles(ex, window, block, tiles=tiles)
        tc, ti = kept.tile_cnt.cpu().numpy(), kept.tile_idx.cpu().numpy()
        bm = kept.bitmap.cpu().numpy().view(np.uint32)
        gs = dma_scores(dma, d)
        for (b, h, t), (want_full, want_part) in lists.items():
            if (b, h) in affected:
                continue
            parity.check_tile_list(ti[b, h, t, :tc[b, h, t]], want_full, want_part, gs[b, h], block)
            assert np.array_equal(bm[b, h, t], bitmaps[(b, h, t)]), (b, h, t)
    rows = list(range(S)) if rows is None else rows
    bias_ref = sc if form == "log" else oracle.score(inp["V"], inp["W"], inp["A"], form="exp")
    O_ref, lse_ref = oracle.attend_rows(inp["Q"], inp["K"], inp["V"], bias_ref, ex, rows, window, block)
    parity.check_outputs(O, O_ref, lse, lse_ref, rows, Q.dtype, H, Hkv, affected)
    return dict(O=O, lse=lse, bias=bias, kept=kept, sc=sc, ex=ex, affected=affected)


def filled_kept(dma, *args, **kw):
    """A Kept whose arrays start at -1, so that two selections compare element by element."""
    k = dma.Kept(*args, device="cuda", **kw)
    for name in ("expiry", "tile_idx", "top_idx"):
        getattr(k, name).fill_(-1)
    return k


def dma_scores(dma, d):
    """The GPU's ranking scores (the tile lists are ordered by them)."""
    B, S, Hkv, D = d["V"].shape
    s = torch.empty((B, Hkv, S), dtype=torch.float32, device="cuda")
    dma.dma_score_keys(d["V"], d["W"], d["A"], s)
    torch.cuda.synchronize()
    return s.cpu().numpy()


# ---------------------------------------------------------- per-head budgets --

def test_per_head_prefill_rowwise_bf16(dma):
    """Budgets 0, 100, 512 and 333 on four KV heads, every row against the oracle."""
    inp = wl.make_prefill(1, 3000, 8, 4, 128, torch.bfloat16, seed=3001, salient=True, with_gate=True)
    r = run_case(dma, inp, 512, 64, w_head=[0, 100, 512, 333])
    ex = r["kept"].expiry.cpu()
    assert torch.all(ex[0, 0] == torch.arange(3000))  # a budget of 0 keeps nothing beyond the window


def test_per_head_prefill_global_fp32(dma):
    inp = wl.make_prefill(2, 700, 4, 2, 64, torch.float32, seed=3002, salient=True)
    run_case(dma, inp, 200, 16, mode=1, w_head=[37, 200])


@pytest.mark.parametrize("mode", [0, 1])
def test_per_head_prefill_blocks_bf16(dma, mode):
    """64-key blocks: budgets of 10, 2, 1 (65 keys) and 0 (63 keys) blocks."""
    inp = wl.make_prefill(1, 2100, 8, 4, 128, torch.bfloat16, seed=3003 + mode, salient=True)
    run_case(dma, inp, 640, 64, block=64, mode=mode, w_head=[640, 128, 65, 63])


def test_per_head_prefill_s64k_sampled_rows(dma):
    """The 64K workload with budgets 512 .. 4096 over its eight KV heads (the bench's per-head
    configuration): 128 sampled rows, six tiles' lists."""
    cfg = wl.WORKLOADS["prefill_s64k_bf16"]
    rows = wl.sample_rows(cfg.S, 128, cfg.seed, cfg.w)
    run_case(dma, wl.make_workload(cfg), cfg.w, cfg.window, w_head=[512, 1024, 2048, 4096, 4096, 2048, 1024, 512],
             rows=rows, tiles=[0, 31, 32, 33, 255, 511])


@pytest.mark.parametrize("block,mode", [(1, 0), (1, 1), (64, 0), (64, 1)])
def test_uniform_budget_list_equals_one_budget(dma, block, mode):
    """w_head = [w] * Hkv writes the same arrays as dma_select_topk, bit for bit."""
    B, S, Hkv, w, window = 2, 3000, 4, 512, 64
    inp = wl.make_prefill(B, S, 8, Hkv, 128, torch.bfloat16, seed=3005, salient=True)
    d = _dev(inp)
    scores = torch.empty((B, Hkv, S), dtype=torch.float32, device="cuda")
    dma.dma_score_keys(d["V"], d["W"], None, scores)
    k1 = filled_kept(dma, B, Hkv, S, w, window, block, mode)
    k2 = filled_kept(dma, B, Hkv, S, w, window, block, mode)
    dma.dma_select_topk(scores, k1)
    dma.dma_select_topk_heads(scores, k2, _wh([w] * Hkv))
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    for name in ("expiry", "tile_cnt", "tile_idx", "bitmap", "top_idx", "top_count"):
        assert torch.equal(getattr(k1, name), getattr(k2, name)), name


def test_budget_out_of_range_is_reported_and_clamped(dma):
    """Entries below 0 or above the layout's budget are recorded as DMA_ERR_DEVICE_CHECK and
    clamped: the selection equals the one with [0, w]."""
    B, S, Hkv, w = 1, 1500, 2, 200
    inp = wl.make_prefill(B, S, 4, Hkv, 64, torch.bfloat16, seed=3006)
    d = _dev(inp)
    scores = torch.empty((B, Hkv, S), dtype=torch.float32, device="cuda")
    dma.dma_score_keys(d["V"], d["W"], None, scores)
    k1 = filled_kept(dma, B, Hkv, S, w, 0)
    k2 = filled_kept(dma, B, Hkv, S, w, 0)
    dma.dma_select_topk_heads(scores, k1, _wh([-5, w + 10]))
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == dma.DMA_ERR_DEVICE_CHECK
    assert dma.dma_get_device_status() == 0
    dma.dma_select_topk_heads(scores, k2, _wh([0, w]))
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    assert torch.equal(k1.expiry, k2.expiry) and torch.equal(k1.tile_idx, k2.tile_idx)


def test_per_head_decode_update_and_oracle(dma):
    """Decode with budgets 40 and 160: FULL at L - n then n UPDATE steps gives the top sets of
    a FULL selection at L, and the output of the oracle's per-head decode."""
    B, L, H, Hkv, D, window, n = 3, 1200, 8, 2, 128, 32, 12
    w_head = [40, 160]
    gen = lambda bs: wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=3007, n_queries=n, device="cuda",
                                    batches=bs)
    d = gen(None)
    st = dma.DecodeState(B, L, H, Hkv, D, 160, window, w_head=_wh(w_head))
    st.full_select(d["Kc"], d["Vc"], d["W"], length=L - n)
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    for k in range(n):
        pos = L - n + k
        st.step(d["q"][k], d["Kc"], d["Vc"], d["W"], torch.full((B,), pos + 1, dtype=torch.int32, device="cuda"),
                pos, o, lse)
    full = dma.DecodeState(B, L, H, Hkv, D, 160, window, w_head=_wh(w_head))
    full.full_select(d["Kc"], d["Vc"], d["W"])
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    assert torch.equal(st.kept.top_count, full.kept.top_count)
    assert st.kept.top_count[:, 0].eq(40).all() and st.kept.top_count[:, 1].eq(160).all()
    for b in range(B):
        for h in range(Hkv):
            c = int(full.kept.top_count[b, h])
            assert torch.equal(st.kept.top_idx[b, h, :c], full.kept.top_idx[b, h, :c])
    inp = {k: (None if v is None else v.cpu()) for k, v in gen(None).items()}
    sc = oracle.score(inp["Vc"], inp["W"], None)
    o_ref, lse_ref = oracle.decode(inp["q"][n - 1], inp["Kc"], inp["Vc"], [L] * B, sc, w_head, window)
    ex = oracle.select(sc, w_head)
    keep = torch.ones((B, H), dtype=torch.bool)
    for b in range(B):
        for h in range(Hkv):
            got = set(st.kept.top_idx[b, h, :int(st.kept.top_count[b, h])].tolist())
            want = {j for j in range(L) if ex[b, h, j] >= L}
            if got != want:
                s32 = sc[b, h].numpy().astype(np.float32).astype(np.float64)
                cut = min(s32[list(want)])
                for j in got ^ want:
                    assert abs(s32[j] - cut) <= parity.TIE_TOL, (b, h, j)
                keep[b, h * (H // Hkv):(h + 1) * (H // Hkv)] = False
    err = ((o.double().cpu() - o_ref).abs() - parity.out_tol(o_ref, torch.bfloat16)).amax(dim=-1)
    assert float(torch.where(keep, err, torch.full_like(err, -1.0)).max()) <= 0
    assert float(torch.where(keep, (lse.double().cpu() - lse_ref).abs(), torch.zeros_like(lse_ref)).max()) <= 2e-2


def test_per_head_page_selection(dma):
    """Paged decode selection with budgets 0, 130 (2 pages of 64) and 512 (8 pages): the kept
    pages of each head against the oracle's; a uniform list equals dma_select_pages."""
    B, L, H, Hkv, D, P, window = 3, 1500, 6, 3, 128, 64, 16
    dd = wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=3008, device="cuda")
    lens = [1500, 900, 200]
    Vp, bt = wl.paginate(dd["Vc"], P, 9, 2)
    w_head = [0, 130, 512]
    st = dma.PagedDecodeState(B, bt.shape[1], P, H, Hkv, D, 512, window, w_head=_wh(w_head))
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    st.full_score(Vp, bt, dd["W"], cache_len=cl)
    st.select(cl)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    sc = oracle.score(dd["Vc"].cpu(), dd["W"].cpu(), None)
    want = oracle.select_pages(sc, lens, P, w_head)
    for b in range(B):
        for h in range(Hkv):
            keys = st.top_idx[b, h, :int(st.top_count[b, h])].cpu().tolist()
            pages = sorted(set(j // P for j in keys))
            assert keys == [p * P + e for p in pages for e in range(P)]
            if pages != want[(b, h)]:
                pm = [float(np.float32(sc[b, h, p * P:(p + 1) * P].max())) for p in range(lens[b] // P)]
                cut = sorted(pm, reverse=True)[len(want[(b, h)]) - 1]
                for p in set(pages) ^ set(want[(b, h)]):
                    assert abs(pm[p] - cut) <= parity.TIE_TOL, (b, h, p)
    ti2 = torch.zeros_like(st.top_idx)
    tc2 = torch.zeros_like(st.top_count)
    dma.dma_select_pages_heads(st.page_scores, P, 512, _wh([512] * Hkv), ti2, tc2, cl)
    ti1 = torch.zeros_like(st.top_idx)
    tc1 = torch.zeros_like(st.top_count)
    dma.dma_select_pages(st.page_scores, P, 512, ti1, tc1, cl)
    torch.cuda.synchronize()
    assert torch.equal(ti1, ti2) and torch.equal(tc1, tc2)


# ------------------------------------------------------------------ exp form --

def test_exp_bias_array(dma):
    """dma_score_keys_bias: the scores are dma_score_keys' bits; LOG copies them into the
    bias, EXP writes exp(s) within the bound derived from the score's."""
    inp = wl.make_prefill(2, 1000, 4, 2, 128, torch.bfloat16, seed=3010, with_gate=True)
    d = _dev(inp)
    shp = (2, 2, 1000)
    s0, s1, b1, s2, b2 = (torch.full(shp, -7.0, device="cuda") for _ in range(5))
    dma.dma_score_keys(d["V"], d["W"], d["A"], s0)
    dma.dma_score_keys_bias(d["V"], d["W"], d["A"], dma.BIAS_LOG, s1, b1)
    dma.dma_score_keys_bias(d["V"], d["W"], d["A"], dma.BIAS_EXP, s2, b2, key_begin=100, key_end=900)
    torch.cuda.synchronize()
    assert torch.equal(s0, s1) and torch.equal(s0, b1)
    assert torch.equal(s2[..., 100:900], s0[..., 100:900])
    assert bool((s2[..., :100] == -7).all() and (b2[..., 900:] == -7).all())
    sc = oracle.score(inp["V"], inp["W"], inp["A"])
    check_bias(b2[..., 100:900], sc[..., 100:900])


def test_exp_prefill_s4k_bf16(dma):
    """The 4K workload with the exp-form bias, every row (rows with a near-tie swap aside)."""
    cfg = wl.WORKLOADS["prefill_s4k_gqa_bf16"]
    run_case(dma, wl.make_workload(cfg), cfg.w, cfg.window, form="exp")


@pytest.mark.parametrize("block,mode", [(1, 0), (1, 1), (64, 0)])
def test_exp_prefill_fp32(dma, block, mode):
    inp = wl.make_prefill(1, 900, 4, 2, 64, torch.float32, seed=3011, w_std=0.05, with_gate=True)
    run_case(dma, inp, 256, 32, block=block, mode=mode, form="exp")


def test_exp_prefill_per_head_bf16(dma):
    """Both variants at once: exp-form bias and per-head budgets, 64-key blocks."""
    inp = wl.make_prefill(1, 2000, 8, 2, 128, torch.bfloat16, seed=3012)
    run_case(dma, inp, 512, 64, block=64, w_head=[192, 512], form="exp")


@pytest.mark.parametrize("dt,simt", [(torch.float32, False), (torch.bfloat16, False), (torch.bfloat16, True)],
                         ids=["fp32", "bf16", "bf16-simt"])
def test_exp_backward(dma, dt, simt):
    """Gradients with the exp-form bias against the oracle: dQ, dK, dV, ds (now dL/d delta) from
    the attention backward given delta, and dV_total, dW, dA through delta = exp(s)."""
    S, H, Hkv, D, w, window = (300, 4, 2, 64, 60, 8) if dt == torch.float32 else (1000, 8, 2, 128, 200, 32)
    inp = wl.make_prefill(1, S, H, Hkv, D, dt, seed=3013, w_std=0.05 if dt == torch.float32 else 0.06,
                          with_gate=True)
    d = _dev(inp)
    dO = wl.make_grad(inp["Q"].shape, dt, 11)
    old = dma.dma_set_prefill_kernel(1 if simt else 0)
    try:
        O, lse, bias, kept = dma.prefill(d["Q"], d["K"], d["V"], d["W"], d["A"], w, window, form=dma.BIAS_EXP)
        f32 = dict(dtype=torch.float32, device="cuda")
        dQ, dK, dV = (torch.empty(t.shape, **f32) for t in (d["Q"], d["K"], d["V"]))
        ds = torch.empty((1, Hkv, S), **f32)
        dma.dma_sparse_attn_prefill_backward(d["Q"], d["K"], d["V"], bias, kept, O, lse, dO.to("cuda"), dQ, dK, dV,
                                             ds)
        dVt = dV.clone()
        dW = torch.empty((Hkv, D), **f32)
        dA = torch.empty((Hkv,), **f32)
        dma.dma_score_keys_backward_bias(d["V"], d["W"], d["A"], dma.BIAS_EXP, ds, dVt, dW, dA)
        torch.cuda.synchronize()
    finally:
        dma.dma_set_prefill_kernel(old)
    assert dma.dma_get_device_status() == 0
    sc = oracle.score(inp["V"], inp["W"], inp["A"])
    ex = oracle.select(sc, w)
    assert not parity.check_expiry(kept.expiry, ex, sc, w, 1, 0), "the case is chosen without near-tie swaps"
    delta = oracle.score(inp["V"], inp["W"], inp["A"], form="exp")
    ref = oracle.attend_backward(inp["Q"], inp["K"], inp["V"], delta, ex, dO, window)
    dV2, dW_ref, dA_ref = oracle.score_backward(inp["V"], inp["W"], inp["A"], ref[3], form="exp")
    stats = [parity.check_grad("dQ", dQ, ref[0], dt), parity.check_grad("dK", dK, ref[1], dt),
             parity.check_grad("dV", dV, ref[2], dt), parity.check_grad("ds", ds, ref[3], dt),
             parity.check_grad("dV_total", dVt, ref[2] + dV2, dt), parity.check_grad("dW", dW, dW_ref, dt),
             parity.check_grad("dA", dA, dA_ref, dt)]
    print("exp-form backward parity", dict(S=S, dtype=str(dt), simt=simt), stats)
    # the composition: the same calls (bit-identical where every sum has a fixed order, the fp32
    # and SIMT paths; the tensor-core path sums ds with atomics in scheduling order)
    old = dma.dma_set_prefill_kernel(1 if simt else 0)
    try:
        g = dma.prefill_backward(d["Q"], d["K"], d["V"], d["W"], d["A"], O, lse, bias, kept, dO.to("cuda"),
                                 form=dma.BIAS_EXP)
        torch.cuda.synchronize()
    finally:
        dma.dma_set_prefill_kernel(old)
    if dt == torch.float32 or simt:
        assert torch.equal(g[3], dW) and torch.equal(g[4], dA)
    parity.check_grad("dW", g[3], dW_ref, dt)
    parity.check_grad("dA", g[4], dA_ref, dt)


def test_exp_decode_update(dma):
    """Decode with the exp-form bias: UPDATE steps, the top set and output against the oracle's
    decode given delta as the bias."""
    B, L, H, Hkv, D, w, window, n = 2, 1000, 8, 2, 128, 128, 16, 6
    gen = lambda bs: wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=3014, n_queries=n, salient=False,
                                    device="cuda", batches=bs)
    d = gen(None)
    st = dma.DecodeState(B, L, H, Hkv, D, w, window, form=dma.BIAS_EXP)
    st.full_select(d["Kc"], d["Vc"], d["W"], length=L - n)
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    for k in range(n):
        pos = L - n + k
        st.step(d["q"][k], d["Kc"], d["Vc"], d["W"], torch.full((B,), pos + 1, dtype=torch.int32, device="cuda"),
                pos, o, lse)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    inp = {k: (None if v is None else v.cpu()) for k, v in gen(None).items()}
    sc = oracle.score(inp["Vc"], inp["W"], None)
    check_bias(st.bias, sc)
    ex = oracle.select(sc, w)
    for b in range(B):
        for h in range(Hkv):
            got = set(st.kept.top_idx[b, h, :int(st.kept.top_count[b, h])].tolist())
            assert got == {j for j in range(L) if ex[b, h, j] >= L}, (b, h)
    delta = oracle.score(inp["Vc"], inp["W"], None, form="exp")
    o_ref, lse_ref = oracle.decode(inp["q"][n - 1], inp["Kc"], inp["Vc"], [L] * B, sc, w, window, bias=delta)
    assert float(((o.double().cpu() - o_ref).abs() - parity.out_tol(o_ref, torch.bfloat16)).max()) <= 0
    assert float((lse.double().cpu() - lse_ref).abs().max()) <= 2e-2


def test_exp_paged_decode(dma):
    """The exp form over a paged cache: the bias array beside the scores, the page selection on
    the scores, the decode against the oracle's decode given delta as the bias (block = page)."""
    B, L, H, Hkv, D, w, window, P = 3, 1000, 8, 2, 128, 256, 32, 64
    dd = wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=3015, salient=False, device="cuda")
    lens = [1000, 700, 130]
    Kp, bt = wl.paginate(dd["Kc"], P, 7, 2)
    Vp, _ = wl.paginate(dd["Vc"], P, 7, 2)
    st = dma.PagedDecodeState(B, bt.shape[1], P, H, Hkv, D, w, window, form=dma.BIAS_EXP)
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    st.full_score(Vp, bt, dd["W"], cache_len=cl)
    st.select(cl)
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    dma.dma_sparse_attn_decode_paged(dd["q"][0], Kp, Vp, bt, st.bias, st.top_idx, st.top_count, window, o, st.ws,
                                     None, cl)
    ref = torch.zeros((B, Hkv, L), dtype=torch.float32, device="cuda")
    dma.dma_score_keys(dd["Vc"], dd["W"], None, ref)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    for b in range(B):
        assert torch.equal(st.scores[b, :, :lens[b]], ref[b, :, :lens[b]])
    h = {k: (None if v is None else v.cpu()) for k, v in dd.items()}
    sc = oracle.score(h["Vc"], h["W"], None)
    for b in range(B):
        check_bias(st.bias[b:b + 1, :, :lens[b]], sc[b:b + 1, :, :lens[b]])
    want = oracle.select_pages(sc, lens, P, w)
    keep = torch.ones((B, H), dtype=torch.bool)
    for b in range(B):
        for hh in range(Hkv):
            keys = st.top_idx[b, hh, :int(st.top_count[b, hh])].cpu().tolist()
            pages = sorted(set(j // P for j in keys))
            if pages != want[(b, hh)]:
                # only a near tie may swap a page: its fp32 page score within 1e-5 of the cutoff
                pm = [float(np.float32(sc[b, hh, p * P:(p + 1) * P].max())) for p in range(lens[b] // P)]
                cut = sorted(pm, reverse=True)[len(want[(b, hh)]) - 1]
                for p in set(pages) ^ set(want[(b, hh)]):
                    assert abs(pm[p] - cut) <= parity.TIE_TOL, (b, hh, p)
                keep[b, hh * (H // Hkv):(hh + 1) * (H // Hkv)] = False
    delta = oracle.score(h["Vc"], h["W"], None, form="exp")
    o_ref, _ = oracle.decode(h["q"][0], h["Kc"], h["Vc"], lens, sc, w, window, block=P, bias=delta)
    err = ((o.double().cpu() - o_ref).abs() - parity.out_tol(o_ref, torch.bfloat16)).amax(dim=-1)
    assert float(torch.where(keep, err, torch.full_like(err, -1.0)).max()) <= 0
