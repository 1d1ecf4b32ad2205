"""Pins for two variants of the fp64 oracle (no GPU): per-KV-head budgets and the exp form
of the bias.

Per-head budgets (Sparse Frontier summary, budget allocation: uniform vs adaptive across
heads): head h keeps w_h keys at every time step.  Pinned by brute-force enumeration of
every candidate subset and by Python's sort, head by head.

Exp form (DMA summary §五 writes the dynamic weight as delta = exp(tau(v Delta) A)): the
logits get delta itself as their bias instead of log delta = A softplus(v . w).  Pinned by
the closed form delta = (1 + e^x)^A at high precision, by torch's fp64 masked attention
and autograd with the bias written as that power, and by the invariant that ranking by
delta and by log delta keeps the same sets.
"""
import itertools
import math

import mpmath
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import dma_workloads as wl


def _val(scores_1d):
    return [float(np.float32(x)) + 0.0 for x in scores_1d]


def _brute_top(val, cands, k):
    """The unique k-subset of `cands` whose every member beats every non-member."""
    beats = lambda a, b: val[a] > val[b] or (val[a] == val[b] and a < b)
    found = [set(sub) for sub in itertools.combinations(cands, k)
             if all(beats(a, b) for a in sub for b in cands if b not in sub)]
    assert len(found) == 1
    return found[0]


def _keep_from_sort(scores, w_head, window):
    """Kept sets [B][Hkv][S][S] from Python's sort with head h's own budget w_head[h]."""
    B, Hkv, S = scores.shape
    keep = torch.zeros(B, Hkv, S, S, dtype=torch.bool)
    for b in range(B):
        for h in range(Hkv):
            val = _val(scores[b, h].tolist())
            for i in range(S):
                ranked = sorted(range(i + 1), key=lambda j: (-val[j], j))
                for j in ranked[:min(w_head[h], i + 1)]:
                    keep[b, h, i, j] = True
                for j in range(max(0, i - window + 1), i + 1):
                    keep[b, h, i, j] = True
    return keep


def _delta(V, W, A):
    """The exp-form bias written as a power, (1 + e^u)^A, u = v . w (fp64 torch)."""
    u = torch.einsum("bjhd,hd->bhj", V.double(), W.double())
    a = torch.ones(W.shape[0], dtype=torch.float64) if A is None else A.double()
    return torch.pow(1.0 + torch.exp(u), a.view(1, -1, 1))


def _dense(Q, K, V, bias, keep, scale):
    """softmax(scale Q K^T + bias_j over the kept keys) V, fp64, O = 0 on empty rows."""
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    G = H // Hkv
    logits = scale * torch.einsum("bihd,bjhd->bhij", Q, K.repeat_interleave(G, dim=2))
    logits = logits + bias.repeat_interleave(G, dim=1).unsqueeze(2)
    m = keep.repeat_interleave(G, dim=1)
    logits = logits.masked_fill(~m, float("-inf"))
    empty = ~m.any(dim=-1, keepdim=True)
    p = torch.softmax(logits.masked_fill(empty, 0.0), dim=-1).masked_fill(empty | ~m, 0.0)
    return torch.einsum("bhij,bjhd->bihd", p, V.repeat_interleave(G, dim=2))


# ---------------------------------------------------------- per-head budgets --

@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("kind", ["random", "ties"])
def test_select_per_head_brute_force(oracle_mod, kind, mode):
    """Head h keeps the min(w_h, i+1) best of keys 0..i (row-wise) or the w_h best of the
    whole segment from their own position on (global), budgets 0, 1, 4 and 20 > S."""
    S, w_head = 11, [0, 1, 4, 20]
    g = torch.Generator().manual_seed(7 + mode)
    if kind == "random":
        sc = torch.rand((2, 4, S), generator=g, dtype=torch.float64) * 3
    else:
        sc = torch.randint(0, 3, (2, 4, S), generator=g).double()
    ex = oracle_mod.select(sc, w_head, mode=mode)
    for b in range(2):
        for h in range(4):
            val = _val(sc[b, h].tolist())
            top_all = _brute_top(val, list(range(S)), min(w_head[h], S)) if mode == 1 else None
            for i in range(S):
                if mode == 0:
                    want = _brute_top(val, list(range(i + 1)), min(w_head[h], i + 1))
                else:
                    want = {j for j in top_all if j <= i}
                assert oracle_mod.top_set(ex[b, h], i) == want, (b, h, i)


def test_select_per_head_uniform_list_equals_one_budget(oracle_mod):
    """A list holding the same budget for every head gives the uniform selection; a budget
    of 0 on one head empties exactly that head."""
    g = torch.Generator().manual_seed(9)
    sc = torch.randn((2, 3, 300), generator=g, dtype=torch.float64)
    for block in (1, 64):
        assert torch.equal(oracle_mod.select(sc, [128] * 3, block), oracle_mod.select(sc, 128, block))
    ex = oracle_mod.select(sc, [0, 128, 128])
    assert torch.all(ex[:, 0] == torch.arange(300))       # every key expires where it enters: never kept
    assert torch.equal(ex[:, 1:], oracle_mod.select(sc[:, 1:], 128))


def test_select_per_head_sizes(oracle_mod):
    """Each head's top set of row i has min(w_h, i+1) keys (DMA summary §五: at most k historical
    positions per head per time step, with k now the head's own)."""
    g = torch.Generator().manual_seed(10)
    sc = torch.randn((1, 4, 200), generator=g, dtype=torch.float64)
    w_head = [3, 50, 199, 1000]
    ex = oracle_mod.select(sc, w_head)
    for h, w in enumerate(w_head):
        for i in (0, 2, 3, 49, 50, 150, 199):
            assert len(oracle_mod.top_set(ex[0, h], i)) == min(w, i + 1)


def test_select_pages_per_head(oracle_mod):
    """Page selection with a budget per KV head: floor(w_h / P) best complete pages, by Python's
    sort of numpy page maxima."""
    B, Hkv, L, P = 2, 3, 500, 16
    g = torch.Generator().manual_seed(12)
    scores = torch.randn((B, Hkv, L), generator=g, dtype=torch.float64)
    w_head = [0, 40, 10 ** 4]
    lens = [500, 333]
    kept = oracle_mod.select_pages(scores, lens, P, w_head)
    for b in range(B):
        n_c = lens[b] // P
        for h in range(Hkv):
            pm = [float(np.float32(np.max(scores[b, h, p * P:(p + 1) * P].numpy()))) + 0.0 for p in range(n_c)]
            order = sorted(range(n_c), key=lambda p: (-pm[p], p))
            assert kept[(b, h)] == sorted(order[:w_head[h] // P]), (b, h)


def test_attention_per_head_budgets_against_sdpa(oracle_mod):
    """Prefill with per-head budgets: each head's output against a dense fp64 softmax whose mask
    is that head's own top-w_h (Python's sort) united with the window."""
    B, S, H, Hkv, D = 1, 40, 6, 3, 32
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=33, salient=True, with_gate=True)
    w_head, window = [2, 9, 40], 3
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], w_head, window, scale=0.2)
    keep = _keep_from_sort(sc, w_head, window)
    want = _dense(inp["Q"].double(), inp["K"].double(), inp["V"].double(), sc, keep, 0.2)
    assert torch.allclose(O, want, rtol=0, atol=1e-12)


def test_decode_per_head_budgets_equals_uniform_and_prefill(oracle_mod):
    """The decode with a budget list takes the prefix route; with equal budgets it equals the
    C decode with one budget, and with different ones the last prefill row of each prefix."""
    B, Lmax, H, Hkv, D = 3, 150, 4, 2, 64
    d = wl.make_decode(B, Lmax, H, Hkv, D, torch.float32, seed=34)
    sc = oracle_mod.score(d["Vc"], d["W"], None)
    lens = [150, 97, 5]
    o1, l1 = oracle_mod.decode(d["q"][0], d["Kc"], d["Vc"], lens, sc, 40, 8)
    o2, l2 = oracle_mod.decode(d["q"][0], d["Kc"], d["Vc"], lens, sc, [40, 40], 8)
    assert torch.allclose(o1, o2, rtol=0, atol=1e-13) and torch.allclose(l1, l2, rtol=0, atol=1e-13)
    o3, _ = oracle_mod.decode(d["q"][0], d["Kc"], d["Vc"], lens, sc, [7, 120], 8)
    for b, L in enumerate(lens):
        keep = _keep_from_sort(sc[b:b + 1, :, :L], [7, 120], 8)
        Q = torch.zeros((1, L, H, D), dtype=torch.float64)
        Q[0, L - 1] = d["q"][0, b].double()
        want = _dense(Q, d["Kc"][b:b + 1, :L].double(), d["Vc"][b:b + 1, :L].double(), sc[b:b + 1, :, :L], keep,
                      1 / math.sqrt(D))
        assert torch.allclose(o3[b], want[0, L - 1], rtol=0, atol=1e-12), b


# ------------------------------------------------------------------ exp form --

@pytest.mark.parametrize("x", [0.0, 1.5, -3.25, 4.0, -20.0])
@pytest.mark.parametrize("a", [1.0, 0.5, 2.0, -1.0])
def test_exp_score_closed_form(oracle_mod, x, a):
    """A one-hot weight makes v . w = x exactly: delta = (1 + e^x)^A at 50 digits."""
    D, Hkv = 64, 2
    V = torch.zeros(1, 2, Hkv, D)
    V[0, 0, 1, 3] = x
    W = torch.zeros(Hkv, D)
    W[1, 3] = 1.0
    A = torch.tensor([1.0, a])
    s = oracle_mod.score(V, W, A, form="exp")
    with mpmath.workdps(50):
        want = float(mpmath.power(1 + mpmath.exp(mpmath.mpf(x)), a))
        want0 = float(mpmath.power(2, a))      # v . w = 0 on key 1
    assert math.isclose(float(s[0, 1, 0]), want, rel_tol=1e-14)
    assert math.isclose(float(s[0, 1, 1]), want0, rel_tol=1e-14)
    assert math.isclose(float(s[0, 0, 0]), 2.0, rel_tol=1e-15)   # head 0: W row 0, A = 1


def test_exp_score_key_range(oracle_mod):
    inp = wl.make_prefill(1, 16, 2, 2, 64, torch.float32, seed=35, with_gate=True)
    s = oracle_mod.score(inp["V"], inp["W"], inp["A"], key_begin=3, key_end=10, form="exp")
    assert torch.all(s[..., :3] == 0) and torch.all(s[..., 10:] == 0)
    full = oracle_mod.score(inp["V"], inp["W"], inp["A"], form="exp")
    assert torch.equal(s[..., 3:10], full[..., 3:10])
    want = _delta(inp["V"], inp["W"], inp["A"])
    assert torch.allclose(full, want, rtol=1e-13, atol=0)


def test_exp_form_ranks_like_log_form(oracle_mod):
    """exp is strictly increasing: ranking delta or log delta keeps the same sets (inputs whose
    fp32 values of delta have no ties that log delta lacks)."""
    inp = wl.make_prefill(2, 300, 4, 2, 64, torch.float32, seed=36, salient=True, with_gate=True)
    s_log = oracle_mod.score(inp["V"], inp["W"], inp["A"])
    s_exp = oracle_mod.score(inp["V"], inp["W"], inp["A"], form="exp")
    for b in range(2):
        for h in range(2):
            assert len(set(_val(s_exp[b, h].tolist()))) == len(set(_val(s_log[b, h].tolist())))
    for mode in (0, 1):
        for block in (1, 64):
            assert torch.equal(oracle_mod.select(s_log, 50, block, mode), oracle_mod.select(s_exp, 50, block, mode))


@pytest.mark.parametrize("w,window", [(10 ** 6, 0), (7, 3)])
def test_exp_form_prefill_against_sdpa(oracle_mod, w, window):
    """Prefill with the exp-form bias against a dense fp64 softmax whose bias is (1 + e^u)^A."""
    B, S, H, Hkv, D = 2, 30, 4, 2, 16
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=37, salient=True, w_std=0.6, with_gate=True)
    w = min(w, S)
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], w, window, scale=0.3,
                                        form="exp")
    keep = _keep_from_sort(sc, [w] * Hkv, window)
    want = _dense(inp["Q"].double(), inp["K"].double(), inp["V"].double(), _delta(inp["V"], inp["W"], inp["A"]),
                  keep, 0.3)
    assert torch.allclose(O, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("w,window,gate", [(10 ** 6, 0, True), (6, 2, False), (5, 0, True)])
def test_exp_form_backward_against_autograd(oracle_mod, w, window, gate):
    """Every gradient with the exp-form bias against torch fp64 autograd of the dense masked
    attention whose bias is (1 + e^u)^A, u = V W: the score path's chain through delta."""
    B, S, H, Hkv, D = 1, 29, 4, 2, 16
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=38 + w % 13, salient=True, w_std=0.6,
                          with_gate=gate)
    w = min(w, S)
    dO = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(8))
    sc = oracle_mod.score(inp["V"], inp["W"], inp["A"])
    keep = _keep_from_sort(sc, [w] * Hkv, window)
    Q, K, V = (inp[k].double().clone().requires_grad_(True) for k in ("Q", "K", "V"))
    Wt = inp["W"].double().clone().requires_grad_(True)
    At = None if inp["A"] is None else inp["A"].double().clone().requires_grad_(True)
    O = _dense(Q, K, V, _delta(V, Wt, At), keep, 0.25)
    (O * dO.double()).sum().backward()
    want = [Q.grad, K.grad, V.grad, Wt.grad, None if At is None else At.grad]
    got = oracle_mod.backward(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], w, window, dO, scale=0.25,
                              form="exp")
    for name, a, b in zip(["dQ", "dK", "dV", "dW", "dA"], got, want):
        if b is None:
            continue
        assert torch.allclose(a, b, rtol=0, atol=1e-11 * max(1.0, float(b.abs().max()))), \
            (name, float((a - b).abs().max()))


def test_exp_form_decode_equals_last_prefill_row(oracle_mod):
    """The decode with the exp-form bias equals row L-1 of the exp-form prefill over the prefix."""
    B, L, H, Hkv, D = 1, 90, 4, 2, 32
    inp = wl.make_prefill(B, L, H, Hkv, D, torch.float32, seed=39, salient=True, with_gate=True)
    O, lse, sc, ex = oracle_mod.prefill(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], 20, 4, form="exp")
    bias = oracle_mod.score(inp["V"], inp["W"], inp["A"], form="exp")
    o, l = oracle_mod.decode(inp["Q"][:, L - 1], inp["K"], inp["V"], [L], sc, 20, 4, bias=bias)
    assert torch.allclose(o[0], O[0, L - 1], rtol=0, atol=1e-13)
    assert torch.allclose(l[0], lse[0, :, L - 1], rtol=0, atol=1e-13)
