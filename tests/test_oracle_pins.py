"""Pins for the fp64 CPU oracle (no GPU).

Each test ties the oracle to something other than itself: high-precision
closed forms (mpmath), brute-force enumeration of every candidate subset,
Python's own sort, torch's fp64 scaled_dot_product_attention, or an
invariant stated by the method (Dynamic Mask Attention summary, §四/§五:
masked positions have weight exactly 0 and skipping them changes nothing; each
head attends to at most k historical positions at every time step).
"""
import itertools
import math
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import dma_workloads as wl

mpmath.mp.dps = 50


def mp_softplus(x: float) -> float:
    """log(1 + e^x) at 400 significant digits, enough to resolve e^x near 1e-324."""
    with mpmath.workdps(400):
        return float(mpmath.log(1 + mpmath.exp(mpmath.mpf(x))))


# ------------------------------------------------------------------ scoring --

def test_score_zero_weights_is_ln2_times_gate(oracle_mod):
    """W = 0 gives v.w = 0 for every key, so s = A * softplus(0) = A ln 2."""
    inp = wl.make_prefill(2, 37, 2, 2, 64, torch.float32, seed=11, with_gate=True)
    W = torch.zeros_like(inp["W"])
    s = oracle_mod.score(inp["V"], W, inp["A"])
    expect = inp["A"].double().view(1, 2, 1) * float(mpmath.log(2))
    assert torch.allclose(s, expect.expand_as(s), rtol=0, atol=1e-15)


@pytest.mark.parametrize("x", [0.0, 1.5, -3.25, 20.0, -20.0, 100.0, -100.0, 700.0, -745.0])
def test_score_softplus_special_values(oracle_mod, x):
    """A one-hot weight makes v.w = x exactly; compare with 400-digit log(1+e^x)."""
    D, Hkv = 64, 2
    V = torch.zeros(1, 3, Hkv, D)
    V[0, :, 1, 5] = torch.tensor([x, 0.5 * x, 2.0], dtype=torch.float32)
    W = torch.zeros(Hkv, D)
    W[1, 5] = 1.0
    s = oracle_mod.score(V, W, None)
    for j, xv in enumerate([x, 0.5 * x, 2.0]):
        want = mp_softplus(float(np.float32(xv)))
        got = s[0, 1, j].item()
        assert math.isclose(got, want, rel_tol=1e-14, abs_tol=1e-300), (j, got, want)
    # the other head saw an all-zero weight row: ln 2
    assert torch.allclose(s[0, 0], torch.full((3,), math.log(2), dtype=torch.float64), atol=1e-15)


def test_score_random_against_numpy_dot_and_mpmath(oracle_mod):
    """Layout and indexing: every (b, h, j) against numpy's dot and mpmath softplus."""
    inp = wl.make_prefill(2, 19, 4, 2, 64, torch.bfloat16, seed=3, with_gate=True, w_std=0.5)
    V = inp["V"].float().numpy().astype(np.float64)
    W = inp["W"].numpy().astype(np.float64)
    A = inp["A"].numpy().astype(np.float64)
    s = oracle_mod.score(inp["V"], inp["W"], inp["A"]).numpy()
    for b in range(2):
        for h in range(2):
            for j in range(19):
                want = A[h] * mp_softplus(float(np.dot(V[b, j, h], W[h])))
                assert math.isclose(s[b, h, j], want, rel_tol=1e-12), (b, h, j)


def test_score_key_range_and_negative_gate(oracle_mod):
    inp = wl.make_prefill(1, 16, 2, 2, 64, torch.float32, seed=5)
    A = torch.tensor([-1.0, 2.0])
    s = oracle_mod.score(inp["V"], inp["W"], A, key_begin=4, key_end=9)
    assert torch.all(s[..., :4] == 0) and torch.all(s[..., 9:] == 0)
    assert torch.all(s[0, 0, 4:9] < 0) and torch.all(s[0, 1, 4:9] > 0)
    full = oracle_mod.score(inp["V"], inp["W"], A)
    assert torch.equal(s[..., 4:9], full[..., 4:9])


# ---------------------------------------------------------------- selection --

def _val(scores_1d):
    """Rank values as the method's kernels see them: fp32."""
    return [float(np.float32(x)) for x in scores_1d]


def _beats(val, a, b):
    return val[a] > val[b] or (val[a] == val[b] and a < b)


def _brute_top(val, cands, k):
    """The unique k-subset of `cands` whose every member beats every non-member."""
    found = []
    for sub in itertools.combinations(cands, k):
        rest = [c for c in cands if c not in sub]
        if all(_beats(val, a, b) for a in sub for b in rest):
            found.append(set(sub))
    assert len(found) == 1
    return found[0]


def _score_sets(kind, S, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "random":
        return torch.rand(S, generator=g, dtype=torch.float64) * 4
    if kind == "ties":
        return torch.randint(0, 3, (S,), generator=g).double()
    if kind == "equal":
        return torch.full((S,), 0.7, dtype=torch.float64)
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["random", "ties", "equal"])
@pytest.mark.parametrize("w", [0, 1, 3, 5, 16])
def test_select_rowwise_brute_force(oracle_mod, kind, w):
    """Row i keeps the min(w, i+1) best of keys 0..i (causal mask, then top-k)."""
    S = 12
    sc = _score_sets(kind, S, seed=100 + w)
    ex = oracle_mod.select(sc.view(1, 1, S), w)[0, 0]
    val = _val(sc.tolist())
    for i in range(S):
        k = min(w, i + 1)
        want = _brute_top(val, list(range(i + 1)), k)
        assert oracle_mod.top_set(ex, i) == want, (i, kind, w)


@pytest.mark.parametrize("kind", ["random", "ties"])
@pytest.mark.parametrize("w", [0, 2, 5, 12])
def test_select_global_brute_force(oracle_mod, kind, w):
    """Global mode: row i keeps the keys j <= i among the w best of all keys."""
    S = 11
    sc = _score_sets(kind, S, seed=200 + w)
    ex = oracle_mod.select(sc.view(1, 1, S), w, mode=oracle_mod.GLOBAL)[0, 0]
    val = _val(sc.tolist())
    winners = _brute_top(val, list(range(S)), min(w, S))
    for i in range(S):
        assert oracle_mod.top_set(ex, i) == {j for j in winners if j <= i}


@pytest.mark.parametrize("kind", ["random", "ties"])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("w", [0, 4, 8, 13])
def test_select_block_brute_force(oracle_mod, kind, mode, w):
    """Block units (block = 4 here): block score = max of its keys; row i ranks
    complete blocks only and keeps the best floor(w/4) (row-wise) or the
    complete ones among the globally best floor(w/4) (global)."""
    S, blk = 18, 4
    sc = _score_sets(kind, S, seed=300 + w + 7 * mode)
    ex = oracle_mod.select(sc.view(1, 1, S), w, block=blk, mode=mode)[0, 0]
    val = _val(sc.tolist())
    nb = S // blk
    bval = [max(val[b * blk:(b + 1) * blk]) for b in range(nb)]
    wb = w // blk
    glob = _brute_top(bval, list(range(nb)), min(wb, nb))
    for i in range(S):
        complete = [b for b in range(nb) if b * blk + blk - 1 <= i]
        if mode == 0:
            blocks = _brute_top(bval, complete, min(wb, len(complete)))
        else:
            blocks = {b for b in glob if b in complete}
        want = {j for b in blocks for j in range(b * blk, b * blk + blk)}
        assert oracle_mod.top_set(ex, i, block=blk) == want, (i, w, mode)


def test_select_rowwise_against_python_sort_and_invariants(oracle_mod):
    """Larger S: Python's sort on sampled rows, plus the step-to-step invariants."""
    S, w = 1500, 97
    g = torch.Generator().manual_seed(9)
    sc = torch.randn(2, 3, S, generator=g, dtype=torch.float64)
    sc[0, 1, ::7] = 0.25  # a run of exact ties
    ex = oracle_mod.select(sc, w)
    for b, h in [(0, 0), (0, 1), (1, 2)]:
        val = _val(sc[b, h].tolist())
        prev = set()
        for i in range(S):
            top = oracle_mod.top_set(ex[b, h], i)
            assert len(top) == min(w, i + 1)
            assert top <= prev | {i}
            prev = top
            if i % 97 in (0, 96) or i == S - 1:
                ranked = sorted(range(i + 1), key=lambda j: (-val[j], j))
                assert top == set(ranked[:min(w, i + 1)])


def test_select_equal_scores_keep_the_first_keys(oracle_mod):
    """All-equal scores: the tie-break alone decides, so Top_i = {0..min(w,i+1)-1}."""
    S, w = 300, 40
    sc = torch.full((1, 2, S), math.log(2), dtype=torch.float64)
    ex = oracle_mod.select(sc, w)
    for i in range(S):
        assert oracle_mod.top_set(ex[0, 1], i) == set(range(min(w, i + 1)))


def test_select_last_row_rowwise_equals_global(oracle_mod):
    S, w = 700, 50
    g = torch.Generator().manual_seed(4)
    sc = torch.randn(1, 2, S, generator=g, dtype=torch.float64)
    e2 = oracle_mod.select(sc, w)
    e1 = oracle_mod.select(sc, w, mode=oracle_mod.GLOBAL)
    for h in range(2):
        assert oracle_mod.top_set(e2[0, h], S - 1) == oracle_mod.top_set(e1[0, h], S - 1)


def test_select_expiry_encoding(oracle_mod):
    """Never-kept keys are written as min(lo, S); kept ones end in (lo, S]."""
    S, w, blk = 200, 64, 16
    g = torch.Generator().manual_seed(5)
    sc = torch.randn(1, 1, S, generator=g, dtype=torch.float64)
    for block in (1, blk):
        ex = oracle_mod.select(sc, w, block=block)[0, 0].tolist()
        for j, e in enumerate(ex):
            lo = oracle_mod.top_lo(j, block)
            assert e <= S
            if e <= lo:
                assert e == min(lo, S)


# ---------------------------------------------------------------- attention --

def _sdpa_masked(Q, K, V, mask_bias, scale):
    """torch fp64 SDPA per (b, hq) with an additive float mask [B][Hkv][S][S]."""
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    G = H // Hkv
    q = Q.double().permute(0, 2, 1, 3)
    k = K.double().permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    v = V.double().permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    m = mask_bias.repeat_interleave(G, dim=1)
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)
    logits = (q @ k.transpose(-1, -2)) * scale + m
    lse = torch.logsumexp(logits, dim=-1)
    return o.permute(0, 2, 1, 3), lse


def _bias_mask(scores, keep):
    """keep [B][Hkv][S][S] bool -> additive mask: s_j where kept, -inf elsewhere."""
    m = scores.unsqueeze(-2).expand(keep.shape).clone()
    m[~keep] = -math.inf
    return m


def _keep_from_sort(scores, w, window):
    """Kept sets built from Python's sort (independent of the oracle's heap)."""
    B, Hkv, S = scores.shape
    keep = torch.zeros(B, Hkv, S, S, dtype=torch.bool)
    for b in range(B):
        for h in range(Hkv):
            val = _val(scores[b, h].tolist())
            for i in range(S):
                ranked = sorted(range(i + 1), key=lambda j: (-val[j], j))
                for j in ranked[:min(w, i + 1)]:
                    keep[b, h, i, j] = True
                for j in range(max(0, i - window + 1), i + 1):
                    keep[b, h, i, j] = True
    return keep


def test_attention_full_budget_is_dense_causal(oracle_mod):
    """w >= S, no window, W = 0: constant bias, so plain causal attention."""
    inp = wl.make_prefill(1, 48, 4, 2, 64, torch.float32, seed=21)
    W = torch.zeros_like(inp["W"])
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], W, None, w=48, window=0)
    q = inp["Q"].double().permute(0, 2, 1, 3)
    k = inp["K"].double().permute(0, 2, 1, 3).repeat_interleave(2, dim=1)
    v = inp["V"].double().permute(0, 2, 1, 3).repeat_interleave(2, dim=1)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=1 / 8.0).permute(0, 2, 1, 3)
    assert torch.allclose(O, ref, atol=1e-12, rtol=0)


def test_attention_full_budget_with_bias(oracle_mod):
    """w >= S with real weights: SDPA with the score as an additive key bias."""
    inp = wl.make_prefill(2, 40, 4, 2, 64, torch.bfloat16, seed=22, w_std=0.5, with_gate=True)
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], w=64, window=0)
    S = 40
    causal = torch.tril(torch.ones(S, S, dtype=torch.bool)).expand(2, 2, S, S)
    ref, ref_lse = _sdpa_masked(inp["Q"], inp["K"], inp["V"], _bias_mask(sc, causal), 1 / 8.0)
    assert torch.allclose(O, ref, atol=1e-12, rtol=0)
    assert torch.allclose(lse, ref_lse, atol=1e-12, rtol=0)


def test_attention_window_only_is_sliding_window(oracle_mod):
    """w = 0, window = 7, W = 0: sliding-window attention."""
    S, win = 50, 7
    inp = wl.make_prefill(1, S, 2, 2, 64, torch.float32, seed=23)
    W = torch.zeros_like(inp["W"])
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], W, None, w=0, window=win)
    i = torch.arange(S).view(S, 1)
    j = torch.arange(S).view(1, S)
    band = ((j <= i) & (j > i - win)).expand(1, 2, S, S)
    ref, ref_lse = _sdpa_masked(inp["Q"], inp["K"], inp["V"], _bias_mask(sc, band), 1 / 8.0)
    assert torch.allclose(O, ref, atol=1e-12, rtol=0)
    assert torch.allclose(lse, ref_lse, atol=1e-12, rtol=0)


def test_attention_block_mode_full_budget_with_window_is_dense_causal(oracle_mod):
    """64-key blocks, a budget of every block and a window >= 64: each row keeps every complete
    past block plus its own (incomplete) block through the window, i.e. all of 0..i: causal
    attention with the score as an additive key bias."""
    S = 150
    inp = wl.make_prefill(1, S, 4, 2, 64, torch.float32, seed=24, w_std=0.5)
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], inp["W"], None, w=S, window=64, block=64)
    causal = torch.tril(torch.ones(S, S, dtype=torch.bool)).expand(1, 2, S, S)
    ref, ref_lse = _sdpa_masked(inp["Q"], inp["K"], inp["V"], _bias_mask(sc, causal), 1 / 8.0)
    assert torch.allclose(O, ref, atol=1e-12, rtol=0)
    assert torch.allclose(lse, ref_lse, atol=1e-12, rtol=0)


def test_per_head_masks_depend_only_on_their_own_weights(oracle_mod):
    """Each KV head's kept sets and outputs follow its own weights w_h: changing w_1 changes
    head 1's kept sets and leaves head 0's sets and its query heads' outputs bit-identical."""
    S, w, win = 64, 12, 3
    inp = wl.make_prefill(1, S, 4, 2, 64, torch.float32, seed=25, w_std=1.0)
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], inp["W"], None, w=w, window=win)
    W2 = inp["W"].clone()
    W2[1] = -W2[1] + 0.3
    O2, lse2, sc2, ex2 = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], W2, None, w=w, window=win)
    assert torch.equal(ex2[:, 0], ex[:, 0])
    assert not torch.equal(ex2[:, 1], ex[:, 1])
    assert torch.equal(O2[:, :, :2], O[:, :, :2]) and torch.equal(lse2[:, :2], lse[:, :2])
    assert not torch.equal(O2[:, :, 2:], O[:, :, 2:])


@pytest.mark.parametrize("w,window", [(5, 0), (9, 4), (3, 20)])
def test_attention_general_against_sdpa_with_sorted_sets(oracle_mod, w, window):
    """Top-w (by Python's sort) united with the window, as an SDPA float mask."""
    S = 36
    inp = wl.make_prefill(1, S, 4, 2, 64, torch.bfloat16, seed=24 + w, salient=True)
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], inp["W"], None, w=w, window=window)
    keep = _keep_from_sort(sc, w, window)
    ref, ref_lse = _sdpa_masked(inp["Q"], inp["K"], inp["V"], _bias_mask(sc, keep), 1 / 8.0)
    assert torch.allclose(O, ref, atol=1e-12, rtol=0)
    assert torch.allclose(lse, ref_lse, atol=1e-12, rtol=0)


def test_attention_rows_sum_to_one(oracle_mod):
    """V = 1 everywhere: O = sum_j p_ij = 1 for every non-empty row."""
    inp = wl.make_prefill(1, 64, 2, 1, 64, torch.float32, seed=25)
    ones = torch.ones_like(inp["V"])
    sc = oracle_mod.score(inp["V"], inp["W"])
    ex = oracle_mod.select(sc, 9)
    O, _ = oracle_mod.attend_rows(inp["Q"], inp["K"], ones, sc, ex, list(range(64)), window=3)
    assert torch.allclose(O, torch.ones_like(O), atol=1e-14, rtol=0)


def test_attention_masked_keys_do_not_matter(oracle_mod):
    """Perturbing the K/V rows of keys a row does not keep leaves it bit-identical."""
    S, w, win = 80, 6, 5
    inp = wl.make_prefill(1, S, 2, 1, 64, torch.float32, seed=26)
    sc = oracle_mod.score(inp["V"], inp["W"])
    ex = oracle_mod.select(sc, w)
    rows = [79, 60, 41]
    O, lse = oracle_mod.attend_rows(inp["Q"], inp["K"], inp["V"], sc, ex, rows, window=win)
    kept = oracle_mod.kept_set(ex[0, 0], 79, win) | oracle_mod.kept_set(ex[0, 0], 60, win) | \
        oracle_mod.kept_set(ex[0, 0], 41, win)
    K2, V2 = inp["K"].clone(), inp["V"].clone()
    for j in range(S):
        if j not in kept:
            K2[0, j, 0] += 5.0
            V2[0, j, 0] -= 3.0
    O2, lse2 = oracle_mod.attend_rows(inp["Q"], K2, V2, sc, ex, rows, window=win)
    assert torch.equal(O, O2) and torch.equal(lse, lse2)


def test_attention_gqa_equals_repeated_kv_heads(oracle_mod):
    S = 40
    inp = wl.make_prefill(1, S, 4, 2, 64, torch.float32, seed=27)
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], inp["W"], None, w=7, window=3)
    K4 = inp["K"].repeat_interleave(2, dim=2)
    V4 = inp["V"].repeat_interleave(2, dim=2)
    W4 = inp["W"].repeat_interleave(2, dim=0)
    O4, lse4, _, _ = oracle_mod.prefill(inp["Q"], K4, V4, W4, None, w=7, window=3)
    assert torch.equal(O, O4) and torch.equal(lse, lse4)


def test_attention_empty_rows(oracle_mod):
    """Global mode with no window can leave early rows with nothing kept:
    O = 0 and lse = -inf, never NaN."""
    S = 30
    inp = wl.make_prefill(1, S, 2, 2, 64, torch.float32, seed=28)
    sc = torch.zeros(1, 2, S, dtype=torch.float64)
    sc[0, :, 20:] = 1.0  # the 3 winners are keys 20, 21, 22
    ex = oracle_mod.select(sc, 3, mode=oracle_mod.GLOBAL)
    O, lse = oracle_mod.attend_rows(inp["Q"], inp["K"], inp["V"], sc, ex, list(range(S)), window=0)
    assert torch.all(O[0, :20] == 0) and torch.all(torch.isneginf(lse[0, :, :20]))
    assert torch.all(torch.isfinite(lse[0, :, 20:]))


def test_decode_equals_last_prefill_row(oracle_mod):
    """Same rule in training and inference: decode over a cache of length L is
    the last row of prefill at S = L."""
    B, L, H, Hkv, D = 2, 70, 4, 2, 64
    inp = wl.make_prefill(B, L, H, Hkv, D, torch.bfloat16, seed=29, salient=True)
    for block, w in [(1, 11), (8, 24)]:
        O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], inp["W"], None, w=w, window=5,
                                            block=block, rows=[L - 1])
        q = inp["Q"][:, L - 1]
        o, l = oracle_mod.decode(q, inp["K"], inp["V"], [L, L], sc, w=w, window=5, block=block)
        assert torch.equal(o, O[:, 0]) and torch.equal(l, lse[:, :, 0])


def test_decode_shorter_cache_uses_its_own_prefix(oracle_mod):
    """cache_len < Lmax: selection and attention see only the first L keys."""
    B, Lmax, H, Hkv, D = 1, 64, 2, 1, 64
    inp = wl.make_prefill(B, Lmax, H, Hkv, D, torch.float32, seed=30)
    sc = oracle_mod.score(inp["V"], inp["W"])
    L = 41
    o, l = oracle_mod.decode(inp["Q"][:, L - 1], inp["K"], inp["V"], [L], sc, w=6, window=2)
    O, lse, _, _ = oracle_mod.prefill(inp["Q"][:, :L], inp["K"][:, :L], inp["V"][:, :L], inp["W"], None, w=6,
                                      window=2, rows=[L - 1])
    assert torch.allclose(o, O[:, 0], atol=1e-14) and torch.allclose(l, lse[:, :, 0], atol=1e-14)


def test_select_ranks_at_fp32_precision(oracle_mod):
    """Scores equal after rounding to fp32 tie, and the lower index wins even
    when its fp64 score is the smaller one (ranking is decided in the kernel's
    precision, fp32)."""
    S = 6
    sc = torch.tensor([[[1.0, 1.0 + 1e-12, 0.5, 1.0 + 2e-12, 0.25, 3.0]]], dtype=torch.float64)
    assert float(np.float32(sc[0, 0, 1])) == float(np.float32(sc[0, 0, 0]))
    ex = oracle_mod.select(sc, 1)[0, 0]
    # row 1: keys 0 and 1 tie in fp32 -> key 0 stays, key 1 never enters
    assert oracle_mod.top_set(ex, 1) == {0}
    assert oracle_mod.top_set(ex, 3) == {0}
    assert oracle_mod.top_set(ex, 5) == {5}


def _golden(name):
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)
    V, O = {}, {}
    for line in open(path):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "V":
            V[int(f[1])] = [float(Fraction(x)) for x in f[2:4]]
        elif f[0] == "O":
            O[int(f[1])] = ([float(Fraction(x)) for x in f[2:4]], int(f[4]))
    return V, O


@pytest.mark.parametrize("mode", [0, 1])
def test_golden_equal_scores_uniform_weights(oracle_mod, mode):
    """The hand-derived example in tests/golden/equal_scores_uniform_weights.txt."""
    V, O = _golden("equal_scores_uniform_weights.txt")
    S = len(V)
    v = torch.tensor([V[j] for j in range(S)], dtype=torch.float64).view(1, S, 1, 2)
    q = torch.randn(1, S, 1, 2, dtype=torch.float64, generator=torch.Generator().manual_seed(5))
    k = torch.zeros(1, S, 1, 2, dtype=torch.float64)
    W = torch.zeros(1, 2, dtype=torch.float64)
    out, lse, sc, ex = oracle_mod.prefill(q, k, v, W, None, w=2, window=1, mode=mode)
    assert torch.allclose(sc, torch.full_like(sc, math.log(2.0)), atol=1e-15, rtol=0)
    for i in range(S):
        want, n = O[i]
        assert torch.allclose(out[0, i, 0], torch.tensor(want, dtype=torch.float64), atol=1e-12, rtol=0), i
        assert abs(float(lse[0, 0, i]) - (math.log(2.0) + math.log(n))) < 1e-12, i


# ------------------------------------------------------------- paged pages --

@pytest.mark.parametrize("page_size", [16, 64])
def test_select_pages_is_block_selection_of_the_last_row(oracle_mod, page_size):
    """Page selection of the decode row L-1 equals the block-unit selection (block = page size)
    of that row, computed by the pinned selection oracle on the first L keys; the page score is
    the maximum of the page's key scores (checked against numpy's max)."""
    B, Hkv, Lmax, w = 3, 2, 700, 200
    g = torch.Generator().manual_seed(17)
    scores = torch.randn((B, Hkv, Lmax), generator=g, dtype=torch.float64)
    scores[0, 0, 100:300] = 0.5  # ties across pages
    lens = [700, 513, page_size * 3 - 1]
    ps = oracle_mod.page_scores(scores, lens, page_size)
    kept = oracle_mod.select_pages(scores, lens, page_size, w)
    for b in range(B):
        L = lens[b]
        ex = oracle_mod.select(scores[b:b + 1, :, :L], w, block=page_size)
        for h in range(Hkv):
            for p in range((L + page_size - 1) // page_size):
                want = np.max(scores[b, h, p * page_size:min(L, (p + 1) * page_size)].numpy())
                assert float(ps[b, h, p]) == float(want)
            top = oracle_mod.top_set(ex[0, h], L - 1, block=page_size)
            keys = sorted(j for p in kept[(b, h)] for j in range(p * page_size, (p + 1) * page_size))
            assert keys == sorted(top), (b, h)
            assert len(kept[(b, h)]) == min(w // page_size, L // page_size)


def test_select_pages_cutoff_inside_exact_ties(oracle_mod):
    """Equal page scores decide by page index alone: with every key score equal the kept pages are
    0 .. k-1; with two score levels the higher pages all go in first and the tied lower ones
    fill the rest from page 0 up."""
    P, w = 16, 16 * 5
    scores = torch.full((1, 2, 16 * 12), 0.75, dtype=torch.float64)
    high = [3, 8]
    for p in high:
        scores[0, 1, p * P + 7] = 2.0  # one key raises the page's maximum
    kept = oracle_mod.select_pages(scores, [16 * 12], P, w)
    assert kept[(0, 0)] == [0, 1, 2, 3, 4]
    assert kept[(0, 1)] == sorted(high + [0, 1, 2])
