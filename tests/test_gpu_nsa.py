"""The NSA-style three-branch fusion on the CUDA path against the fp64 oracle, through the
C ABI (needs a B300).

  compression   rows 64 beta + 63 of Kc, Vc against the oracle's block means: fp32 within
                1e-6 relative (an fp32 sum of 64 terms), bf16 within half a bf16 ulp of
                the mean plus that; every other row untouched
  patterns      the compressed and window kept structures equal, array for array, those
                of the selection path on scores that rank the compressed keys first (global
                mode, w = S / 64) and of a selection with w = 0
  branches      o_cmp, o_slc, o_win within the output bounds (2e-2 bf16, 1e-4 fp32, plus
                half a bf16 ulp); the selected branch's kept blocks as in the uniform parity
                tests (near-tie rows left out)
  fused O       the same bound plus, in bf16, each branch's half ulp weighted by its gate:
                the branch outputs are rounded to bf16 before the gated sum
  decode        steps across a block boundary, against the last row of the oracle's
                prefill over each sequence's prefix
"""
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


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_compress_block_range(dma, dt):
    B, S, Hkv, D = 2, 64 * 7 + 20, 4, 128
    inp = wl.make_prefill(B, S, 4, Hkv, D, dt, seed=71, salient=True)
    d = _dev(inp)
    Kc = torch.full_like(d["K"], 7.0)
    Vc = torch.full_like(d["V"], 7.0)
    dma.dma_nsa_compress(d["K"], d["V"], Kc, Vc, 2, 5)
    torch.cuda.synchronize()
    kr, vr = oracle.nsa_compress(inp["K"], inp["V"])
    rows = [64 * b + 63 for b in range(2, 5)]
    for got, ref in ((Kc, kr), (Vc, vr)):
        g = got.double().cpu()
        want = ref[:, 2:5]
        err = (g[:, rows] - want).abs()
        bound = 1e-6 * want.abs() + 1e-7
        if dt == torch.bfloat16:
            bound = bound + parity.bf16_half_ulp(want)
        assert bool((err <= bound).all()), float((err - bound).max())
        mask = torch.ones(S, dtype=torch.bool)
        mask[rows] = False
        assert bool((g[:, mask] == 7.0).all())


@pytest.mark.parametrize("S", [64 * 40, 64 * 33 + 50])
def test_patterns_equal_the_selection_path(dma, S):
    """The compressed pattern is the global selection of the S/64 best keys under scores that
    rank the keys 64 beta + 63 first; the window pattern is a selection with w = 0."""
    B, Hkv, window = 2, 3, 100
    nb = S // 64
    ind = torch.zeros((B, Hkv, S), dtype=torch.float32, device="cuda")
    ind[:, :, 63:nb * 64:64] = 1.0
    a = dma.Kept(B, Hkv, S, nb, 0, 1, dma.GLOBAL)
    p = dma.Kept(B, Hkv, S, nb, 0, 1, dma.GLOBAL)
    for k in (a, p):
        for name in ("expiry", "idx", "top_idx", "tile_idx"):
            getattr(k, name).fill_(-1)
    dma.dma_select_topk(ind, a)
    dma.dma_nsa_kept_pattern(dma.NSA_COMPRESSED, p)
    wa = dma.Kept(B, Hkv, S, 0, window, 1, dma.ROWWISE)
    wp = dma.Kept(B, Hkv, S, 0, window, 1, dma.ROWWISE)
    for k in (wa, wp):
        for name in ("expiry", "tile_idx"):
            getattr(k, name).fill_(-1)
    dma.dma_select_topk(torch.randn((B, Hkv, S), device="cuda"), wa)
    dma.dma_nsa_kept_pattern(dma.NSA_WINDOW, wp)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    for name in ("expiry", "count", "top_count", "tile_cnt", "bitmap"):
        assert torch.equal(getattr(a, name), getattr(p, name)), name
    assert torch.equal(a.idx[..., :nb], p.idx[..., :nb]) and torch.equal(a.top_idx[..., :nb], p.top_idx[..., :nb])
    tc = a.tile_cnt.cpu()
    ta, tp = a.tile_idx.cpu(), p.tile_idx.cpu()
    for b in range(B):
        for h in range(Hkv):
            for t in range(a.t.n_qt):
                n = int(tc[b, h, t])
                assert torch.equal(ta[b, h, t, :n], tp[b, h, t, :n]), (b, h, t)
    for name in ("expiry", "tile_cnt", "bitmap", "top_count"):
        assert torch.equal(getattr(wa, name), getattr(wp, name)), name


def run_nsa(dma, inp, G, c, w, window, rows=None, check_branches=True):
    B, S, H, D = inp["Q"].shape
    Hkv = inp["K"].shape[2]
    dt = inp["Q"].dtype
    d = _dev(inp)
    st = dma.NsaPrefill(B, S, H, Hkv, D, w, window, dtype=dt)
    O = torch.empty_like(d["Q"])
    gates = torch.empty((B, S, H, 3), dtype=torch.float32, device="cuda")
    st.run(d["Q"], d["K"], d["V"], d["W"], d["A"], G.cuda(), c.cuda(), O, gates)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    rows = list(range(S)) if rows is None else rows
    ref = oracle.nsa_prefill(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], G, c, w, window, rows=rows)
    affected = parity.check_expiry(st.kept_slc.expiry, ref["expiry"], ref["scores"], w, 64, 0)
    rt = torch.tensor(rows)
    g_gpu = gates.double().cpu()[:, rt]
    assert float((g_gpu - ref["gates"]).abs().max()) <= 1e-5
    if check_branches:
        for name, got in (("o_cmp", st.o_cmp), ("o_slc", st.o_slc), ("o_win", st.o_win)):
            print(name, end=": ")
            parity.check_outputs(got, ref[name], None, None, rows, dt, H, Hkv,
                                 affected if name == "o_slc" else None)
    # the fused output: each branch output is rounded to dt before the gated sum, so the bound
    # grants half an ulp of each branch (weighted by its gate) on top of the output's own
    tol = parity.out_tol(ref["O"], dt)
    if dt == torch.bfloat16:
        for b_i, name in enumerate(("o_cmp", "o_slc", "o_win")):
            tol = tol + ref["gates"][..., b_i:b_i + 1] * parity.bf16_half_ulp(ref[name])
    err = ((O.double().cpu()[:, rt] - ref["O"]).abs() - tol).amax(dim=-1)
    keep = torch.ones(err.shape, dtype=torch.bool)
    G_ = H // Hkv
    for (b, h), rs in affected.items():
        for r_i, i in enumerate(rows):
            if i in rs:
                keep[b, r_i, h * G_:(h + 1) * G_] = False
    worst = float(torch.where(keep, err, torch.full_like(err, -1.0)).max())
    print("O: fused output parity", dict(rows=len(rows), excess=worst, row_heads_dropped_near_tie=int((~keep).sum())))
    assert worst <= 0, "fused output error exceeds its bound by %.3g" % worst
    return st, O, ref


def test_nsa_prefill_tiny_fp32_ragged(dma):
    """S = 300: the last 44 keys form no complete block; rows below 63 see no block."""
    inp = wl.make_prefill(1, 300, 4, 2, 64, torch.float32, seed=72, salient=True, with_gate=True)
    G, c = wl.make_nsa_gates(4, 64, 72)
    run_nsa(dma, inp, G, c, 128, 32)


def test_nsa_prefill_s4k_bf16_all_rows(dma):
    cfg = wl.WORKLOADS["prefill_s4k_gqa_bf16"]
    inp = wl.make_workload(cfg)
    G, c = wl.make_nsa_gates(cfg.H, cfg.D, cfg.seed)
    run_nsa(dma, inp, G, c, cfg.w, cfg.window)


def test_nsa_prefill_s16k_bf16_sampled_rows(dma):
    cfg = wl.WORKLOADS["prefill_s16k_bf16"]
    inp = wl.make_workload(cfg)
    G, c = wl.make_nsa_gates(cfg.H, cfg.D, cfg.seed)
    rows = wl.sample_rows(cfg.S, 128, cfg.seed, cfg.w)
    run_nsa(dma, inp, G, c, cfg.w, cfg.window, rows=rows)


def test_nsa_prefill_s64k_bf16_sampled_rows(dma):
    """The bench's three-branch configuration: the 64K inputs, 64 sampled rows."""
    cfg = wl.WORKLOADS["prefill_s64k_bf16"]
    inp = wl.make_workload(cfg)
    G, c = wl.make_nsa_gates(cfg.H, cfg.D, cfg.seed)
    rows = wl.sample_rows(cfg.S, 64, cfg.seed, cfg.w)
    run_nsa(dma, inp, G, c, cfg.w, cfg.window, rows=rows)


@pytest.mark.parametrize("dt,D", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16", "fp32"])
def test_nsa_decode_steps_across_a_block_boundary(dma, dt, D):
    """Steps from L = 1000 to 1030 (the block ending at key 1023 completes on the way); the
    final output against the oracle's last row over each sequence's prefix."""
    B, Lmax, H, Hkv, w, window = 3, 1088, 8, 2, 256, 32
    L0, L1 = 1000, 1030
    n = L1 - L0
    dd = wl.make_decode(B, Lmax, H, Hkv, D, dt, seed=73, n_queries=n, device="cuda")
    G, c = wl.make_nsa_gates(H, D, 73)
    Gd, cd = G.cuda(), c.cuda()
    st = dma.NsaDecode(B, Lmax, H, Hkv, D, w, window, dtype=dt)
    st.prepare(dd["Kc"], dd["Vc"], dd["W"], torch.full((B,), L0, dtype=torch.int32, device="cuda"), L0)
    o = torch.empty((B, H, D), dtype=dt, device="cuda")
    for k in range(n):
        pos = L0 + k
        cl = torch.full((B,), pos + 1, dtype=torch.int32, device="cuda")
        st.step(dd["q"][k], dd["Kc"], dd["Vc"], dd["W"], cl, pos, Gd, cd, o)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    L = L1
    # the oracle: the prefill of each prefix, row L - 1, with that step's query in its place
    Kc, Vc = dd["Kc"].cpu(), dd["Vc"].cpu()
    q = dd["q"][n - 1].cpu()
    for b in range(B):
        Q = torch.zeros((1, L, H, D), dtype=dt)
        Q[0, L - 1] = q[b]
        ref = oracle.nsa_prefill(Q, Kc[b:b + 1, :L], Vc[b:b + 1, :L], dd["W"].cpu(), None, G, c, w, window,
                                 rows=[L - 1])
        got = o[b].double().cpu()
        want = ref["O"][0, 0]
        # the selected blocks of every KV head against the oracle's; a sequence with a near-tie
        # swap (block maxima within 1e-5 of the cutoff) is left out of the output check
        ex = ref["expiry"]
        swapped = False
        for h in range(Hkv):
            sel = {j // 64 for j in st.kept_slc.top_idx[b, h, :int(st.kept_slc.top_count[b, h])].tolist()}
            want_sel = {j // 64 for j in range(L) if oracle.top_lo(j, 64) <= L - 1 < int(ex[0, h, j])}
            if sel != want_sel:
                sc = ref["scores"][0, h].numpy().astype(np.float32).astype(np.float64)
                bmax = [sc[64 * k:64 * k + 64].max() for k in range(L // 64)]
                cut = min(bmax[k] for k in want_sel)
                for k in sel ^ want_sel:
                    assert abs(bmax[k] - cut) <= parity.TIE_TOL, (b, h, k)
                swapped = True
        if swapped:
            continue
        tol = parity.out_tol(want, dt)
        if dt == torch.bfloat16:  # each branch output is rounded to bf16 before the gated sum
            for b_i, name in enumerate(("o_cmp", "o_slc", "o_win")):
                tol = tol + ref["gates"][0, 0, :, b_i:b_i + 1] * parity.bf16_half_ulp(ref[name][0, 0])
        err = ((got - want).abs() - tol).max()
        assert float(err) <= 0, (b, float(err))
