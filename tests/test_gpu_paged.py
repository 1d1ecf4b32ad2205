"""Page-granular decode over a paged KV cache against the fp64 oracle (needs a B300).

The cache is laid out in pages [n_pages][page_size][Hkv][D] behind a block table with the
physical pages in seeded random order.  The oracle sees the same rows as a contiguous logical
cache: its page selection (oracle.select_pages, pinned against the block-unit selection) and
its decode with block = page size give the expected kept keys and outputs.
  scores       bit-identical to dma_score_keys on the contiguous cache
  page scores  exactly the max of the GPU's key scores of each page
  kept keys    the oracle's kept pages, except pages whose fp32 score is within 1e-5 of the
               cutoff (those (b, KV head) segments are left out of the output check)
  o            max-abs 2e-2 plus half a bf16 ulp (reading of the output rounding)
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


def to_pages(Kc, page_size, seed, extra_pages=3):
    """A paged copy of the contiguous cache (seeded random physical page order, spare pages)."""
    return wl.paginate(Kc, page_size, seed, extra_pages)


def run_paged(dma, d, page_size, w, window, lens, seed=3):
    """The paged score, page selection and decode on the GPU; returns the state and outputs."""
    B, L, Hkv, D = d["Kc"].shape
    H = d["q"].shape[2]
    Kp, bt = to_pages(d["Kc"], page_size, seed)
    Vp, bt2 = to_pages(d["Vc"], page_size, seed)
    assert torch.equal(bt, bt2)
    st = dma.PagedDecodeState(B, bt.shape[1], page_size, H, Hkv, D, w, window)
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    st.full_score(Vp, bt, d["W"], cache_len=cl)
    dma.dma_select_pages(st.page_scores, page_size, w, st.top_idx, st.top_count, cl)
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    dma.dma_sparse_attn_decode_paged(d["q"][0], Kp, Vp, bt, st.scores, st.top_idx, st.top_count, window, o, st.ws,
                                     lse, cl)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    return st, o, lse, Kp, Vp, bt, cl


def gpu_kept(st, b, h):
    n = int(st.top_count[b, h])
    return st.top_idx[b, h, :n].cpu().tolist()


def check_against_oracle(st, o, lse, h_inp, lens, page_size, w, window, batches=None):
    """h_inp: the CPU copy of the sequences in `batches` (all when None)."""
    B_all = st.B
    batches = list(range(B_all)) if batches is None else batches
    Hkv = st.Hkv
    G = st.H // Hkv
    sc = oracle.score(h_inp["Vc"], h_inp["W"], None)
    lens_b = [lens[b] for b in batches]
    want = oracle.select_pages(sc, lens_b, page_size, w)
    ps_ref = oracle.page_scores(sc, lens_b, page_size)
    keep_heads = torch.ones((len(batches), st.H), dtype=torch.bool)
    swapped = 0
    for r, b in enumerate(batches):
        for h in range(Hkv):
            got_keys = gpu_kept(st, b, h)
            got_pages = sorted(set(j // page_size for j in got_keys))
            assert got_keys == [p * page_size + e for p in got_pages for e in range(page_size)]
            if got_pages != want[(r, h)]:
                # only near-ties may differ: every differing page within 1e-5 of the cutoff
                vals = ps_ref[r, h].numpy().astype(np.float32).astype(np.float64)
                n_c = lens[b] // page_size
                order = sorted(range(n_c), key=lambda p: (-vals[p], p))
                cut = vals[order[len(want[(r, h)]) - 1]]
                for p in set(got_pages) ^ set(want[(r, h)]):
                    assert abs(vals[p] - cut) <= parity.TIE_TOL, (b, h, p, vals[p], cut)
                keep_heads[r, h * G:(h + 1) * G] = False
                swapped += 1
    o_ref, lse_ref = oracle.decode(h_inp["q"][0], h_inp["Kc"], h_inp["Vc"], lens_b, sc, w, window, block=page_size)
    og = o.double().cpu()[batches]
    err = ((og - o_ref).abs() - parity.out_tol(o_ref, torch.bfloat16)).amax(dim=-1)
    err = torch.where(keep_heads, err, torch.full_like(err, -1.0))
    assert float(err.max()) <= 0, "paged decode error exceeds its bound by %.3g" % float(err.max())
    lg = lse.double().cpu()[batches]
    assert float(torch.where(keep_heads, (lg - lse_ref).abs(), torch.zeros_like(lg)).max()) <= 2e-2
    return swapped


@pytest.mark.parametrize("page_size", [16, 64])
def test_paged_decode_against_oracle(dma, page_size):
    B, L, H, Hkv, D, w, window = 4, 2000, 8, 2, 128, 256, 32
    dd = wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=41, device="cuda")
    lens = [2000, 1500, 777, 64]
    st, o, lse, *_ = run_paged(dma, dd, page_size, w, window, lens)
    h_inp = {k: (None if v is None else v.cpu()) for k, v in dd.items()}
    swapped = check_against_oracle(st, o, lse, h_inp, lens, page_size, w, window)
    print("paged decode parity", dict(page_size=page_size, segments_with_near_tie_swaps=swapped))


def test_paged_scores_and_page_maxima(dma):
    B, L, H, Hkv, D = 3, 1000, 4, 2, 128
    dd = wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=42, device="cuda")
    lens = [1000, 999, 130]
    st, *_ , bt, cl = run_paged(dma, dd, 64, 128, 16, lens)
    ref = torch.zeros((B, Hkv, L), dtype=torch.float32, device="cuda")
    dma.dma_score_keys(dd["Vc"], dd["W"], None, ref)
    torch.cuda.synchronize()
    for b in range(B):
        assert torch.equal(st.scores[b, :, :lens[b]], ref[b, :, :lens[b]])
        for p in range((lens[b] + 63) // 64):
            want = ref[b, :, p * 64:min(lens[b], (p + 1) * 64)].max(dim=-1).values
            assert torch.equal(st.page_scores[b, :, p], want)


def test_paged_equals_contiguous_decode(dma):
    """The same kept keys over a contiguous cache and over its paged copy: the same kernel code
    except for the row addressing, so the outputs are bit-identical."""
    B, L, H, Hkv, D, w, window = 4, 1536, 16, 4, 128, 384, 64
    dd = wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=43, device="cuda")
    lens = [1536, 1000, 1200, 65]
    st, o_p, lse_p, Kp, Vp, bt, cl = run_paged(dma, dd, 32, w, window, lens)
    kept = dma.Kept(B, Hkv, L, st.top_cap, window, 1, dma.ROWWISE, device="cuda", tiles=False)
    kept.top_idx.copy_(st.top_idx)
    kept.top_count.copy_(st.top_count)
    ws = torch.empty((dma.dma_decode_workspace_size(B, H, Hkv, D, kept.t.top_cap, window),), dtype=torch.uint8,
                     device="cuda")
    o_c = torch.empty_like(o_p)
    lse_c = torch.empty_like(lse_p)
    scores_c = st.scores[:, :, :L].contiguous()
    dma.dma_sparse_attn_decode(dd["q"][0], dd["Kc"], dd["Vc"], scores_c, kept, o_c, ws, lse_c, cl)
    torch.cuda.synchronize()
    assert torch.equal(o_c, o_p) and torch.equal(lse_c, lse_p)


def test_paged_steps_equal_full_recompute(dma):
    """Appending tokens one at a time (score the new key, update its page score, select, attend)
    gives the page scores and the output of a full recompute at the final length."""
    B, L, H, Hkv, D, w, window, P = 2, 700, 8, 2, 128, 128, 16, 16
    n_new = 20
    dd = wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=44, n_queries=n_new, device="cuda")
    Kp, bt = to_pages(dd["Kc"], P, 5)
    Vp, _ = to_pages(dd["Vc"], P, 5)
    st = dma.PagedDecodeState(B, bt.shape[1], P, H, Hkv, D, w, window)
    st.full_score(Vp, bt, dd["W"], cache_len=torch.full((B,), L - n_new, dtype=torch.int32, device="cuda"))
    o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    for k in range(n_new):
        pos = L - n_new + k
        cl = torch.full((B,), pos + 1, dtype=torch.int32, device="cuda")
        st.step(dd["q"][k], Kp, Vp, bt, dd["W"], cl, pos, o)
    torch.cuda.synchronize()
    full = dma.PagedDecodeState(B, bt.shape[1], P, H, Hkv, D, w, window)
    cl = torch.full((B,), L, dtype=torch.int32, device="cuda")
    full.full_score(Vp, bt, dd["W"], cache_len=cl)
    dma.dma_select_pages(full.page_scores, P, w, full.top_idx, full.top_count, cl)
    o_full = torch.empty_like(o)
    dma.dma_sparse_attn_decode_paged(dd["q"][n_new - 1], Kp, Vp, bt, full.scores, full.top_idx, full.top_count,
                                     window, o_full, full.ws, None, cl)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    assert torch.equal(st.page_scores, full.page_scores)
    assert torch.equal(st.top_idx, full.top_idx) and torch.equal(st.top_count, full.top_count)
    assert torch.equal(o, o_full)


def test_paged_bad_block_table_entry_is_reported(dma):
    """A block-table entry outside [0, n_pages) is recorded as DMA_ERR_DEVICE_CHECK and its rows
    are not read (the bounds check runs before any access)."""
    B, L, H, Hkv, D = 1, 256, 4, 1, 64
    dd = wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=45, device="cuda")
    Vp, bt = to_pages(dd["Vc"], 64, 6)
    bt[0, 1] = Vp.shape[0] + 5
    scores = torch.zeros((B, Hkv, L), dtype=torch.float32, device="cuda")
    dma.dma_score_keys_paged(Vp, bt, dd["W"], None, scores)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == dma.DMA_ERR_DEVICE_CHECK
    assert dma.dma_get_device_status() == 0


def test_paged_decode_b64_l32k(dma):
    """The decode workload (64 sequences of 32K cached tokens) in 64-token pages: three sampled
    sequences against the oracle."""
    cfg = wl.WORKLOADS["decode_b64_l32k_bf16"]
    B, L, H, Hkv, D, w, window = cfg.B, cfg.S, cfg.H, cfg.Hkv, cfg.D, cfg.w, cfg.window
    dd = wl.make_workload(cfg, device="cuda")
    lens = [L] * B
    st, o, lse, *_ = run_paged(dma, dd, 64, w, window, lens)
    sample = [0, 31, 63]
    # each sequence draws from its own generator on the device that holds it: regenerated there
    h_inp = {k: (None if v is None else v.cpu()) for k, v in wl.make_workload(cfg, device="cuda", batches=sample).items()}
    assert torch.equal(h_inp["Kc"][-1], dd["Kc"][sample[-1]].cpu())
    swapped = check_against_oracle(st, o, lse, h_inp, lens, 64, w, window, batches=sample)
    print("paged decode parity b64 l32k", dict(segments_with_near_tie_swaps=swapped))


def _pages_by_definition(ps, n_c, k):
    """The k best of the first n_c pages under (score descending, page index ascending), in page
    order: Python's sort of the page scores, as fp32 values."""
    vals = [float(np.float32(x)) for x in ps[:n_c]]
    return sorted(sorted(range(n_c), key=lambda p: (-vals[p], p))[:k])


@pytest.mark.parametrize("max_pages,n_levels", [(512, 2), (700, 3), (700, 1), (1024, 3), (1500, 4), (2500, 3)])
def test_page_selection_with_exact_ties(dma, max_pages, n_levels):
    """Page scores drawn from a few exact values (n_levels = 1: all equal), so that the cutoff
    falls inside a run of equal scores: the kept pages are those of the definition, ties to the
    lower page index.  Sequences of different lengths put the cutoff at different places.
    Tables of up to 512 and up to 1024 pages take the two instantiations of the
    one-warp-per-segment select; 1500 and 2500 pages take the one-CTA-per-segment kernel (its sort
    above 1024 complete pages, its counting rank below).
    Per-head budgets too: the uniform list and an uneven one with a zero budget."""
    B, Hkv, P, w = 3, 4, 16, 16 * 300
    gen = torch.Generator().manual_seed(90 + max_pages + n_levels)
    levels = torch.tensor([0.25 * (1 + e) for e in range(n_levels)], dtype=torch.float32)
    ps = levels[torch.randint(0, n_levels, (B, Hkv, max_pages), generator=gen)]
    ps[1, 2, :] = levels[-1]  # one segment wholly tied
    lens = [max_pages * P, (max_pages // 2) * P + 5, 301 * P]
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ps_d = ps.cuda()
    top_cap = (w // P) * P
    for w_head in (None, [w, w // 3, P * 7, 0]):
        top_idx = torch.full((B, Hkv, top_cap), -7, dtype=torch.int32, device="cuda")
        top_count = torch.full((B, Hkv), -7, dtype=torch.int32, device="cuda")
        if w_head is None:
            dma.dma_select_pages(ps_d, P, w, top_idx, top_count, cl)
        else:
            wh = torch.tensor(w_head, dtype=torch.int32, device="cuda")
            dma.dma_select_pages_heads(ps_d, P, w, wh, top_idx, top_count, cl)
        torch.cuda.synchronize()
        assert dma.dma_get_device_status() == 0
        for b in range(B):
            n_c = min(lens[b] // P, max_pages)
            for h in range(Hkv):
                budget = w if w_head is None else w_head[h]
                k = min(budget // P, n_c)
                want = _pages_by_definition(ps[b, h].tolist(), n_c, k)
                n = int(top_count[b, h])
                got = top_idx[b, h, :n].cpu().tolist()
                assert got == [p * P + e for p in want for e in range(P)], (max_pages, n_levels, w_head, b, h)
