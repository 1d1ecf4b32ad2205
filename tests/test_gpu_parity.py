"""CUDA path against the fp64 oracle, through the C ABI (needs a B300).

Every case runs the three prefill calls (score, select, attend) or the decode
calls on seeded inputs and compares, element by element:
  scores   within 5e-5 + 1e-5 |s| (fp32 accumulation of D products);
  expiry   exactly, except near-cutoff ties (see parity.py);
  tiles    per-tile gathered key lists and occupancy bitmaps exactly;
  O, lse   max-abs 1e-4 (fp32 inputs) / 2e-2 (bf16 inputs).
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
    out = {}
    for k, v in inp.items():
        out[k] = None if v is None else v.to("cuda")
    return out


def gpu_prefill(dma, inp, w, window, block=1, mode=0):
    d = _dev(inp)
    O, lse, scores, kept = dma.prefill(d["Q"], d["K"], d["V"], d["W"], d["A"], w, window, block, mode)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    return O, lse, scores, kept


def run_prefill_case(dma, inp, w, window, block=1, mode=0, rows=None, tiles=None, check_tile_lists=True):
    Q = inp["Q"]
    B, S, H, D = Q.shape
    Hkv = inp["K"].shape[2]
    O, lse, scores, kept = gpu_prefill(dma, inp, w, window, block, mode)
    sc = oracle.score(inp["V"], inp["W"], inp["A"])
    parity.check_scores(scores, sc)
    ex = oracle.select(sc, w, block, mode)
    affected = parity.check_expiry(kept.expiry, ex, sc, w, block, mode)
    if check_tile_lists:
        lists, bitmaps = parity.expected_tiles(ex, window, block, tiles=tiles)
        tc = kept.tile_cnt.cpu().numpy()
        ti = kept.tile_idx.cpu().numpy()
        bm = kept.bitmap.cpu().numpy().view(np.uint32)
        gs = scores.cpu().numpy()
        for (b, h, t), (want_full, want_part) in lists.items():
            if (b, h) in affected:
                continue
            got = ti[b, h, t, :tc[b, h, t]]
            parity.check_tile_list(got, want_full, want_part, gs[b, h], block)
            assert np.array_equal(bm[b, h, t], bitmaps[(b, h, t)]), (b, h, t)
    rows = list(range(S)) if rows is None else rows
    O_ref, lse_ref = oracle.attend_rows(inp["Q"], inp["K"], inp["V"], sc, ex, rows, window, block)
    skipped = parity.check_outputs(O, O_ref, lse, lse_ref, rows, Q.dtype, H, Hkv, affected)
    return dict(O=O, lse=lse, scores=scores, kept=kept, sc=sc, ex=ex, skipped=skipped)


# ------------------------------------------------------------ workloads -----

def test_tiny_prefill_fp32_rowwise(dma):
    cfg = wl.WORKLOADS["prefill_tiny_s256_fp32"]
    run_prefill_case(dma, wl.make_workload(cfg), cfg.w, cfg.window)


def test_tiny_prefill_fp32_global(dma):
    cfg = wl.WORKLOADS["prefill_tiny_s256_fp32"]
    run_prefill_case(dma, wl.make_workload(cfg), cfg.w, cfg.window, mode=1)


def test_s4k_gqa_bf16_all_rows(dma):
    cfg = wl.WORKLOADS["prefill_s4k_gqa_bf16"]
    r = run_prefill_case(dma, wl.make_workload(cfg), cfg.w, cfg.window)
    assert r["skipped"] == 0


def test_s16k_bf16_sampled_rows(dma):
    cfg = wl.WORKLOADS["prefill_s16k_bf16"]
    rows = wl.sample_rows(cfg.S, 256, cfg.seed, cfg.w)
    run_prefill_case(dma, wl.make_workload(cfg), cfg.w, cfg.window, rows=rows, tiles=[0, 15, 16, 17, 100, 127])


@pytest.mark.parametrize("block", [1, 64])
def test_s64k_bf16_sampled_rows(dma, block):
    cfg = wl.WORKLOADS["prefill_s64k_bf16"]
    rows = wl.sample_rows(cfg.S, 256, cfg.seed, cfg.w, block=64)
    run_prefill_case(dma, wl.make_workload(cfg), cfg.w, cfg.window, block=block, rows=rows,
                     tiles=[0, 31, 32, 33, 255, 511])


# ------------------------------------------------------------ edge cases ----

EDGE = [
    # B, S, H, Hkv, D, dtype, w, window, block, mode
    (1, 1, 1, 1, 64, torch.float32, 4, 0, 1, 0),
    (1, 5, 2, 1, 128, torch.float32, 2, 1, 1, 0),
    (2, 127, 4, 2, 64, torch.bfloat16, 16, 0, 1, 0),
    (1, 128, 4, 4, 128, torch.float32, 0, 9, 1, 0),       # window only: sliding window
    (1, 129, 2, 2, 64, torch.float32, 129, 0, 1, 0),      # w >= S: dense causal
    (1, 300, 8, 2, 128, torch.bfloat16, 1000, 300, 1, 0), # window >= S
    (2, 333, 4, 1, 64, torch.float32, 37, 5, 1, 1),       # global mode, ragged tail
    (1, 300, 2, 2, 64, torch.float32, 20, 0, 1, 1),       # global mode, empty early rows
    (1, 700, 4, 2, 128, torch.bfloat16, 130, 70, 64, 0),  # block units, partial last block
    (1, 640, 2, 1, 64, torch.float32, 200, 0, 64, 1),     # block units, global
    (1, 200, 2, 2, 64, torch.float32, 63, 16, 64, 0),     # block budget 0: window only
    (3, 1000, 6, 3, 128, torch.bfloat16, 100, 33, 1, 0),
    # bf16 cases for the tensor-core kernel: GQA group sizes 1, 3 and 8 (one query head per
    # pass, an odd last pass, four passes), one row, nothing kept at all, window only,
    # global mode with empty rows, D = 64 blocks
    (2, 260, 2, 2, 64, torch.bfloat16, 40, 0, 1, 0),
    (1, 333, 3, 1, 128, torch.bfloat16, 64, 16, 1, 0),
    (1, 517, 8, 1, 128, torch.bfloat16, 200, 50, 1, 0),
    (1, 1, 2, 1, 128, torch.bfloat16, 4, 0, 1, 0),
    (1, 200, 4, 2, 64, torch.bfloat16, 0, 0, 1, 0),
    (1, 384, 4, 2, 128, torch.bfloat16, 0, 100, 1, 0),
    (1, 450, 4, 2, 128, torch.bfloat16, 30, 0, 1, 1),
    (1, 1100, 4, 2, 64, torch.bfloat16, 256, 64, 64, 0),
    # one query head per KV head, and an odd group, each with more key blocks than the
    # metadata ring holds (the idle M-tile's share of the ring's releases)
    (1, 2048, 2, 2, 128, torch.bfloat16, 512, 64, 1, 0),
    (1, 1500, 3, 1, 128, torch.bfloat16, 400, 100, 1, 0),
]


@pytest.mark.parametrize("case", EDGE, ids=[str(i) for i in range(len(EDGE))])
def test_edge_cases(dma, case):
    B, S, H, Hkv, D, dtype, w, window, block, mode = case
    inp = wl.make_prefill(B, S, H, Hkv, D, dtype, seed=1000 + S + w, salient=True, with_gate=(S % 2 == 1))
    run_prefill_case(dma, inp, w, window, block, mode)


def test_ties_and_zero_weights(dma):
    """W = 0: every score is ln 2, the tie-break alone selects keys 0..w-1."""
    inp = wl.make_prefill(1, 500, 4, 2, 64, torch.float32, seed=77)
    inp["W"] = torch.zeros_like(inp["W"])
    r = run_prefill_case(dma, inp, 50, 7)
    ex = r["kept"].expiry.cpu()
    assert torch.all(ex[..., :50] == 500)
    assert torch.all(ex[..., 50:] == torch.arange(50, 500, dtype=torch.int32))


def test_masked_keys_are_never_read(dma):
    """Skipped positions contribute exactly nothing (DMA summary §五): changing
    the K rows of keys that never enter the top set, in the first half of the
    sequence, leaves every row from (last changed key + window) on
    bit-identical.  K does not enter the scores, so the selection is unchanged."""
    S, w, win = 600, 24, 8
    inp = wl.make_prefill(1, S, 4, 2, 64, torch.bfloat16, seed=78, salient=True)
    O1, lse1, _, kept = gpu_prefill(dma, inp, w, win)
    ex = kept.expiry.cpu()
    j = torch.arange(S)
    never = (ex <= j) & (j < S // 2)
    assert int(never.sum()) > 100
    K2 = inp["K"].clone()
    for h in range(2):
        K2[0, torch.nonzero(never[0, h]).flatten(), h] += 7.0
    inp2 = dict(inp)
    inp2["K"] = K2
    O2, lse2, _, kept2 = gpu_prefill(dma, inp2, w, win)
    assert torch.equal(kept2.expiry.cpu(), ex)
    r0 = int(torch.nonzero(never).max(dim=0).values[-1]) + win
    assert torch.equal(O1[:, r0:], O2[:, r0:]) and torch.equal(lse1[:, :, r0:], lse2[:, :, r0:])
    assert not torch.equal(O1[:, :r0], O2[:, :r0])  # the window did see the changed rows


def test_block_mode_full_budget_is_dense_causal(dma):
    """64-key blocks with a budget of every block and a 64-key window keep all of 0..i for
    every row: the GPU path against the oracle's dense causal attention with key bias."""
    S = 1000
    inp = wl.make_prefill(1, S, 8, 2, 128, torch.bfloat16, seed=801, w_std=0.3)
    O, lse, scores, kept = gpu_prefill(dma, inp, S, 64, block=64)
    sc = oracle.score(inp["V"], inp["W"], inp["A"])
    ex = oracle.select(sc, S, 64)
    rows = list(range(0, S, 7)) + [S - 1]
    O_ref, lse_ref = oracle.attend_rows(inp["Q"], inp["K"], inp["V"], sc, ex, rows, 64, 64)
    dense_ref, dense_lse = oracle.attend_rows(inp["Q"], inp["K"], inp["V"], sc,
                                              torch.full_like(ex, S + 1), rows, S, 1)
    assert torch.allclose(O_ref, dense_ref, atol=1e-12, rtol=0)
    parity.check_outputs(O, dense_ref, lse, dense_lse, rows, torch.bfloat16, 8, 2)


def test_per_head_masks_on_the_gpu(dma):
    """Changing the weights of KV head 1 leaves KV head 0's kept sets and the outputs of its
    query heads bit-identical on the GPU path, and changes head 1's."""
    B, S, H, Hkv, D, w, window = 1, 2000, 8, 2, 128, 256, 32
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.bfloat16, seed=802, w_std=0.3)
    O, lse, scores, kept = gpu_prefill(dma, inp, w, window)
    inp2 = dict(inp)
    W2 = inp["W"].clone()
    W2[1] = -W2[1]
    inp2["W"] = W2
    O2, lse2, scores2, kept2 = gpu_prefill(dma, inp2, w, window)
    assert torch.equal(kept2.expiry[:, 0], kept.expiry[:, 0])
    assert not torch.equal(kept2.expiry[:, 1], kept.expiry[:, 1])
    G = H // Hkv
    assert torch.equal(O2[:, :, :G], O[:, :, :G]) and torch.equal(lse2[:, :G], lse[:, :G])
    assert not torch.equal(O2[:, :, G:], O[:, :, G:])


def test_simt_and_default_kernels_agree(dma):
    cfg = wl.WORKLOADS["prefill_s4k_gqa_bf16"]
    inp = wl.make_workload(cfg)
    old = dma.dma_set_prefill_kernel(1)
    try:
        O1, lse1, _, _ = gpu_prefill(dma, inp, cfg.w, cfg.window)
    finally:
        dma.dma_set_prefill_kernel(old)
    O2, lse2, _, _ = gpu_prefill(dma, inp, cfg.w, cfg.window)
    assert float((O1.float() - O2.float()).abs().max()) <= 2e-2
    assert float((lse1 - lse2).abs().max()) <= 2e-2


# ---------------------------------------------------------------- decode ----

def _decode_gpu(dma, d, B, L, H, Hkv, D, w, window, n_update, lens=None):
    """FULL selection at length L - n_update, then n_update UPDATE steps, then decode."""
    st = dma.DecodeState(B, L, H, Hkv, D, w, window)
    st.full_select(d["Kc"], d["Vc"], d["W"], length=L - n_update)
    o = torch.empty((B, H, D), dtype=d["Kc"].dtype, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    for k in range(n_update):
        pos = L - n_update + k
        cl = torch.full((B,), pos + 1, dtype=torch.int32, device="cuda")
        st.step(d["q"][k], d["Kc"], d["Vc"], d["W"], cl, pos, o, lse)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    return st, o, lse


def _check_decode(dma, gen, B, L, H, Hkv, D, w, window, n_update, sample=None):
    """gen(batches) -> decode inputs on the GPU for those sequences (None = all).
    The GPU runs all B sequences; the oracle checks the sequences in `sample`."""
    d = gen(None)
    st, o, lse = _decode_gpu(dma, d, B, L, H, Hkv, D, w, window, n_update)
    sample = list(range(B)) if sample is None else sample
    inp = {k: (None if v is None else v.cpu()) for k, v in gen(sample).items()}
    assert torch.equal(inp["Kc"][-1], d["Kc"][sample[-1]].cpu())
    sc = oracle.score(inp["Vc"], inp["W"], None)
    parity.check_scores(st.scores[sample], sc)
    o_ref, lse_ref = oracle.decode(inp["q"][n_update - 1], inp["Kc"], inp["Vc"], [L] * len(sample), sc, w, window)
    o_g = o[sample].double().cpu()
    lse_g = lse[sample].double().cpu()
    # top set of the last row against the oracle's
    ex = oracle.select(sc, w)
    tc = st.kept.top_count[sample].cpu()
    ti = st.kept.top_idx[sample].cpu()
    bad = 0
    for r in range(len(sample)):
        for h in range(Hkv):
            got = set(ti[r, h, :tc[r, h]].tolist())
            want = {j for j in range(L) if ex[r, h, j] >= L}
            if got != want:
                s32 = sc[r, h].numpy().astype(np.float32).astype(np.float64)
                cut = min(s32[list(want)])
                for j in got ^ want:
                    assert abs(s32[j] - cut) <= parity.TIE_TOL, (r, h, j)
                bad += 1
                # a near-tie swapped one key: this group's rows are left out of the output check
                g0, g1 = h * (H // Hkv), (h + 1) * (H // Hkv)
                o_ref[r, g0:g1] = o_g[r, g0:g1]
                lse_ref[r, g0:g1] = lse_g[r, g0:g1]
    dt = d["q"].dtype
    assert float(((o_g - o_ref).abs() - parity.out_tol(o_ref, dt)).max()) <= 0
    assert float((lse_g - lse_ref).abs().max()) <= parity.TOL[dt]
    return bad


def test_decode_small_fp32(dma):
    B, L, H, Hkv, D, w, window = 3, 300, 4, 2, 64, 40, 9
    gen = lambda bs: wl.make_decode(B, L, H, Hkv, D, torch.float32, seed=501, n_queries=5, device="cuda", batches=bs)
    assert _check_decode(dma, gen, B, L, H, Hkv, D, w, window, 5) == 0


def test_decode_small_bf16_gqa8(dma):
    B, L, H, Hkv, D, w, window = 2, 1000, 16, 2, 128, 128, 64
    gen = lambda bs: wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=502, n_queries=3, device="cuda",
                                    batches=bs)
    _check_decode(dma, gen, B, L, H, Hkv, D, w, window, 3)


def test_decode_b1_long_list_bf16(dma):
    """One sequence with a long kept list: 33 splits per (sequence, KV head) (the 64-row chunk limit)."""
    B, L, H, Hkv, D, w, window = 1, 8192, 8, 2, 128, 2048, 64
    gen = lambda bs: wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=505, n_queries=2, device="cuda",
                                    batches=bs)
    _check_decode(dma, gen, B, L, H, Hkv, D, w, window, 2)


def test_decode_b32_split8_bf16(dma):
    """32 sequences: eight splits per (sequence, KV head)."""
    B, L, H, Hkv, D, w, window = 32, 4096, 32, 8, 128, 512, 64
    gen = lambda bs: wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=506, n_queries=2, device="cuda",
                                    batches=bs)
    _check_decode(dma, gen, B, L, H, Hkv, D, w, window, 2, sample=[0, 13, 31])


def test_decode_b64_short_list_bf16(dma):
    """Short kept lists (256 rows): as many splits as 64-row chunks, most of them only partly filled."""
    B, L, H, Hkv, D, w, window = 64, 1024, 32, 8, 128, 192, 64
    gen = lambda bs: wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=507, n_queries=2, device="cuda",
                                    batches=bs)
    _check_decode(dma, gen, B, L, H, Hkv, D, w, window, 2, sample=[0, 40, 63])


def test_decode_b64_l32k_bf16(dma):
    """The full decode workload on the GPU; the oracle checks three sampled sequences."""
    cfg = wl.WORKLOADS["decode_b64_l32k_bf16"]
    gen = lambda bs: wl.make_workload(cfg, n_queries=2, device="cuda", batches=bs)
    _check_decode(dma, gen, cfg.B, cfg.S, cfg.H, cfg.Hkv, cfg.D, cfg.w, cfg.window, 2, sample=[0, 17, 63])


def test_update_replay_equals_full(dma):
    """FULL at L - n followed by n UPDATE steps gives the FULL top set at L."""
    B, L, H, Hkv, D, w, window, n = 2, 2000, 4, 2, 64, 100, 16, 40
    d = wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=503, n_queries=n, device="cuda")
    st, _, _ = _decode_gpu(dma, d, B, L, H, Hkv, D, w, window, n)
    full = dma.DecodeState(B, L, H, Hkv, D, w, window)
    full.full_select(d["Kc"], d["Vc"], d["W"])
    torch.cuda.synchronize()
    assert torch.equal(st.kept.top_count, full.kept.top_count)
    for b in range(B):
        for h in range(Hkv):
            c = int(full.kept.top_count[b, h])
            assert torch.equal(st.kept.top_idx[b, h, :c], full.kept.top_idx[b, h, :c])


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_decode_varying_cache_len(dma, dt):
    """Per-sequence cache lengths: each sequence attends over its own prefix (its own window
    band and top set), on the fp32 kernel and on the pipelined bf16 kernel."""
    B, Lmax, w, window = 3, 400, 30, 5
    H, Hkv, D = (4, 1, 64) if dt == torch.float32 else (8, 2, 128)
    inp = wl.make_decode(B, Lmax, H, Hkv, D, dt, seed=504)
    d = _dev(inp)
    lens = [400, 257, 64]
    sc = oracle.score(inp["Vc"], inp["W"], None)
    o = torch.empty((B, H, D), dtype=dt, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    scores = torch.zeros((B, Hkv, Lmax), dtype=torch.float32, device="cuda")
    dma.dma_score_keys(d["Vc"], d["W"], None, scores)
    kept = dma.Kept(B, Hkv, Lmax, w, window, tiles=False)
    # per-sequence FULL selection, written into one kept struct
    for b, L in enumerate(lens):
        sub = dma.Kept(1, Hkv, L, w, window, tiles=False)
        dma.dma_select_topk(scores[b:b + 1, :, :L].contiguous(), sub)
        kept.top_idx[b, :, :sub.t.top_cap].copy_(sub.top_idx[0])
        kept.top_count[b].copy_(sub.top_count[0])
    ws = torch.empty((dma.dma_decode_workspace_size(B, H, Hkv, D, kept.t.top_cap, window),), dtype=torch.uint8,
                     device="cuda")
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q = (torch.stack([inp["Kc"][b, lens[b] - 1, 0, :].float().repeat(H, 1) for b in range(B)]) * 0.3).to(dt)
    dma.dma_sparse_attn_decode(q.to("cuda"), d["Kc"], d["Vc"], scores, kept, o, ws, lse, cl)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(q, inp["Kc"], inp["Vc"], lens, sc, w, window)
    assert float(((o.double().cpu() - o_ref).abs() - parity.out_tol(o_ref, dt)).max()) <= 0
    assert float((lse.double().cpu() - lse_ref).abs().max()) <= parity.TOL[dt]
    assert dma.dma_get_device_status() == 0


def test_full_select_on_a_side_stream(dma):
    """DecodeState.full_select with a prefix length runs every step -- scoring, the prefix's
    FULL selection and the copies of its top set -- on the stream it is given."""
    B, L, H, Hkv, D, w, window = 2, 1500, 8, 2, 128, 100, 16
    d = wl.make_decode(B, L, H, Hkv, D, torch.bfloat16, seed=508, n_queries=1, device="cuda")
    ref = dma.DecodeState(B, L, H, Hkv, D, w, window)
    ref.full_select(d["Kc"], d["Vc"], d["W"], length=L - 7)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    st = dma.DecodeState(B, L, H, Hkv, D, w, window)
    torch.cuda.synchronize()
    st.full_select(d["Kc"], d["Vc"], d["W"], length=L - 7, stream=side)
    side.synchronize()
    assert torch.equal(st.kept.top_count, ref.kept.top_count)
    assert torch.equal(st.kept.top_idx, ref.kept.top_idx)
