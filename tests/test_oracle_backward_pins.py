"""Pins for the fp64 CPU oracle's backward pass (no GPU).

The backward (DMA summary, §四/§五/§七: the same mask in training and
inference, differentiable in the kept positions, the selection itself piecewise
constant, skipped positions with exactly zero gradient) is tied to things other
than itself:
  - torch's fp64 autograd through a dense masked softmax attention whose bias is
    s = A * softplus(V W) and whose mask comes from Python's sort;
  - central finite differences of the (pinned) forward oracle;
  - exact identities of the softmax backward: per (batch, KV head) the score
    gradients sum to 0, the key gradients sum to 0, and the value gradients sum
    to the output gradients of every row with a non-empty kept set;
  - skipped keys receive exactly zero gradient and do not change anyone else's;
  - GQA equals repeated KV heads with the key-side gradients summed.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import dma_workloads as wl


def _val(scores_row):
    """The selection's ranking value: the score rounded to fp32 (-0 is +0)."""
    return [float(np.float32(x)) + 0.0 for x in scores_row]


def _keep_from_sort(scores, w, window):
    """Kept sets from Python's sort (independent of the oracle's heap): [B][Hkv][S][S]."""
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


def _dense_forward(Q, K, V, W, A, keep, scale):
    """O = softmax(scale Q K^T + s, masked to `keep`) V with s = A_h softplus(V_j . W_h); fp64
    tensors that may require grad.  Rows with nothing kept give O = 0."""
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    G = H // Hkv
    u = torch.einsum("bjhd,hd->bhj", V, W)
    a = torch.ones(Hkv, dtype=torch.float64) if A is None else A
    s = a.view(1, Hkv, 1) * F.softplus(u)                              # [B][Hkv][S]
    Kr = K.repeat_interleave(G, dim=2)
    Vr = V.repeat_interleave(G, dim=2)
    logits = scale * torch.einsum("bihd,bjhd->bhij", Q, Kr) + s.repeat_interleave(G, dim=1).unsqueeze(2)
    m = keep.repeat_interleave(G, dim=1)
    logits = logits.masked_fill(~m, float("-inf"))
    empty = ~m.any(dim=-1, keepdim=True)
    p = torch.softmax(logits.masked_fill(empty, 0.0), dim=-1).masked_fill(empty | ~m, 0.0)
    return torch.einsum("bhij,bjhd->bihd", p, Vr)


def _autograd(inp, keep, dO, scale):
    Q, K, V = (inp[k].double().clone().requires_grad_(True) for k in ("Q", "K", "V"))
    W = inp["W"].double().clone().requires_grad_(True)
    A = None if inp["A"] is None else inp["A"].double().clone().requires_grad_(True)
    O = _dense_forward(Q, K, V, W, A, keep, scale)
    (O * dO.double()).sum().backward()
    return Q.grad, K.grad, V.grad, W.grad, (None if A is None else A.grad)


@pytest.mark.parametrize("w,window,gate", [(10**6, 0, False), (10**6, 0, True), (7, 0, True), (9, 4, False),
                                           (3, 11, True)])
def test_backward_matches_dense_autograd(oracle_mod, w, window, gate):
    """Every gradient -- Q, K, V (attention and score paths), W, A -- against torch fp64 autograd
    of a dense masked attention; the mask is the full causal one (w >= S) or top-w by Python's
    sort united with the window."""
    B, S, H, Hkv, D = 2, 33, 4, 2, 16
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=900 + window + (w % 97), salient=True,
                          w_std=0.6, with_gate=gate)
    g = torch.Generator().manual_seed(5)
    dO = torch.randn(B, S, H, D, generator=g).float()
    scale = 0.3
    sc = oracle_mod.score(inp["V"], inp["W"], inp["A"])
    keep = _keep_from_sort(sc, min(w, S), window)
    want = _autograd(inp, keep, dO, scale)
    got = oracle_mod.backward(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], min(w, S), window, dO, scale=scale)
    names = ["dQ", "dK", "dV", "dW", "dA"]
    for name, a, b in zip(names, got, want):
        if b is None:
            continue
        tol = 1e-11 * max(1.0, float(b.abs().max()))
        assert torch.allclose(a, b, rtol=0, atol=tol), (name, float((a - b).abs().max()))


def test_backward_block_units_against_autograd(oracle_mod):
    """64-key block selection (every complete block kept) with a 64-key window keeps all of 0..i:
    the dense causal autograd gradients."""
    B, S, H, Hkv, D = 1, 150, 2, 1, 16
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=931, w_std=0.5)
    dO = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(6))
    keep = torch.tril(torch.ones(S, S, dtype=torch.bool)).view(1, 1, S, S)
    want = _autograd(inp, keep, dO, 0.25)
    got = oracle_mod.backward(inp["Q"], inp["K"], inp["V"], inp["W"], None, S, 64, dO, block=64, scale=0.25)
    for a, b in zip(got[:4], want[:4]):
        assert torch.allclose(a, b, rtol=0, atol=1e-11 * max(1.0, float(b.abs().max())))


def test_backward_finite_differences(oracle_mod):
    """Central differences of L = sum(O * R) computed by the forward oracle, for every element
    of Q, K, V, W and A of a tiny problem.  The perturbation is a power of two, so x +- h is an
    exact fp32 value for these magnitudes; an element whose perturbation would change the
    selection is skipped (none is, for this seed)."""
    B, S, H, Hkv, D, w, window = 1, 12, 2, 1, 4, 4, 2
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=941, w_std=0.8, with_gate=True)
    R = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(7))
    scale = 0.5
    got = dict(zip(["Q", "K", "V", "W", "A"],
                   oracle_mod.backward(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], w, window, R,
                                       scale=scale)))
    base_ex = oracle_mod.select(oracle_mod.score(inp["V"], inp["W"], inp["A"]), w)

    def loss(d):
        O, _, sc, ex = oracle_mod.prefill(d["Q"], d["K"], d["V"], d["W"], d["A"], w, window, scale=scale)
        return float((O * R.double()).sum()), ex

    h = 2.0 ** -12
    skipped = 0
    for name in ("Q", "K", "V", "W", "A"):
        flat = inp[name].reshape(-1)
        fd = torch.zeros(flat.numel(), dtype=torch.float64)
        for e in range(flat.numel()):
            vals = []
            for sgn in (1.0, -1.0):
                d = dict(inp)
                t = inp[name].clone().reshape(-1)
                t[e] = t[e] + sgn * h
                d[name] = t.reshape(inp[name].shape)
                L, ex = loss(d)
                vals.append((L, ex))
            if not (torch.equal(vals[0][1], base_ex) and torch.equal(vals[1][1], base_ex)):
                skipped += 1
                fd[e] = got[name].reshape(-1)[e]
                continue
            fd[e] = (vals[0][0] - vals[1][0]) / (2 * h)
        g = got[name].reshape(-1)
        tol = 1e-6 + 1e-5 * float(g.abs().max())
        assert torch.allclose(fd, g, rtol=0, atol=tol), (name, float((fd - g).abs().max()))
    assert skipped == 0


def test_backward_sum_identities(oracle_mod):
    """Per (batch, KV head): sum_j ds_j = 0 and sum_j dK_j = 0 (each row's softmax gradient sums
    to zero), and sum_j dV_j (attention part) = the sum of dO over the rows of the group's query
    heads that keep at least one key (each such row's weights sum to one)."""
    B, S, H, Hkv, D, w, window = 2, 300, 6, 3, 32, 40, 8
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.bfloat16, seed=951, salient=True)
    dO = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(8))
    sc = oracle_mod.score(inp["V"], inp["W"], None)
    ex = oracle_mod.select(sc, w)
    dQ, dK, dV, ds = oracle_mod.attend_backward(inp["Q"], inp["K"], inp["V"], sc, ex, dO, window)
    G = H // Hkv
    for b in range(B):
        for h in range(Hkv):
            assert abs(float(ds[b, h].sum())) < 1e-10
            assert float(dK[b, :, h].sum(dim=0).abs().max()) < 1e-10
            want = dO[b, :, h * G:(h + 1) * G].double().sum(dim=(0, 1))
            assert torch.allclose(dV[b, :, h].sum(dim=0), want, rtol=0, atol=1e-10)


def test_backward_skipped_keys(oracle_mod):
    """Without a window, keys that never enter the top set get exactly zero gradient, and
    changing their K rows leaves every other gradient bit-identical."""
    B, S, H, Hkv, D, w = 1, 200, 4, 2, 16, 12
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=961, salient=True)
    dO = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(9))
    sc = oracle_mod.score(inp["V"], inp["W"], None)
    ex = oracle_mod.select(sc, w)
    j = torch.arange(S)
    never = ex <= j.view(1, 1, S)
    assert int(never.sum()) > 100
    g1 = oracle_mod.attend_backward(inp["Q"], inp["K"], inp["V"], sc, ex, dO, 0)
    dQ, dK, dV, ds = g1
    for h in range(Hkv):
        idx = torch.nonzero(never[0, h]).flatten()
        assert float(dK[0, idx, h].abs().max()) == 0.0
        assert float(dV[0, idx, h].abs().max()) == 0.0
        assert float(ds[0, h, idx].abs().max()) == 0.0
    K2 = inp["K"].clone()
    for h in range(Hkv):
        K2[0, torch.nonzero(never[0, h]).flatten(), h] += 5.0
    g2 = oracle_mod.attend_backward(inp["Q"], K2, inp["V"], sc, ex, dO, 0)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_backward_gqa_equals_repeated_kv_heads(oracle_mod):
    """Query heads sharing a KV head: the same as one KV head per query head (K, V, scores and
    kept sets repeated) with the key-side gradients summed over the repeats."""
    B, S, H, Hkv, D, w, window = 1, 90, 4, 2, 16, 10, 3
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=971, salient=True)
    dO = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(10))
    sc = oracle_mod.score(inp["V"], inp["W"], None)
    ex = oracle_mod.select(sc, w)
    dQ, dK, dV, ds = oracle_mod.attend_backward(inp["Q"], inp["K"], inp["V"], sc, ex, dO, window)
    G = H // Hkv
    Kr = inp["K"].repeat_interleave(G, dim=2)
    Vr = inp["V"].repeat_interleave(G, dim=2)
    dQ2, dK2, dV2, ds2 = oracle_mod.attend_backward(inp["Q"], Kr, Vr, sc.repeat_interleave(G, dim=1),
                                                    ex.repeat_interleave(G, dim=1), dO, window)
    assert torch.allclose(dQ, dQ2, rtol=0, atol=1e-12)
    assert torch.allclose(dK, dK2.view(B, S, Hkv, G, D).sum(dim=3), rtol=0, atol=1e-12)
    assert torch.allclose(dV, dV2.view(B, S, Hkv, G, D).sum(dim=3), rtol=0, atol=1e-12)
    assert torch.allclose(ds, ds2.view(B, Hkv, G, S).sum(dim=2), rtol=0, atol=1e-12)


def test_backward_single_segment_equals_all(oracle_mod):
    """Computing one (batch, KV head) segment alone gives that segment's gradients exactly."""
    B, S, H, Hkv, D, w, window = 2, 120, 4, 2, 16, 15, 5
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.bfloat16, seed=981, salient=True)
    dO = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(11))
    sc = oracle_mod.score(inp["V"], inp["W"], None)
    ex = oracle_mod.select(sc, w)
    full = oracle_mod.attend_backward(inp["Q"], inp["K"], inp["V"], sc, ex, dO, window)
    b, h = 1, 0
    one = oracle_mod.attend_backward(inp["Q"], inp["K"], inp["V"], sc, ex, dO, window, segment=b * Hkv + h)
    G = H // Hkv
    assert torch.equal(one[0][b, :, h * G:(h + 1) * G], full[0][b, :, h * G:(h + 1) * G])
    assert torch.equal(one[1][b, :, h], full[1][b, :, h])
    assert torch.equal(one[2][b, :, h], full[2][b, :, h])
    assert torch.equal(one[3][b, h], full[3][b, h])


def test_backward_sampled_rows_and_keys_equal_all(oracle_mod):
    """dQ limited to some rows and dK, dV, ds limited to some keys are those rows' and keys'
    values of the full computation, bit for bit; everything else is left at zero."""
    B, S, H, Hkv, D, w, window = 1, 150, 4, 2, 16, 12, 6
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=991, salient=True)
    dO = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(12))
    sc = oracle_mod.score(inp["V"], inp["W"], None)
    ex = oracle_mod.select(sc, w)
    full = oracle_mod.attend_backward(inp["Q"], inp["K"], inp["V"], sc, ex, dO, window)
    rows, keys = [0, 7, 64, 149], [0, 3, 100, 148, 149]
    part = oracle_mod.attend_backward(inp["Q"], inp["K"], inp["V"], sc, ex, dO, window, rows=rows, keys=keys)
    assert torch.equal(part[0][:, rows], full[0][:, rows])
    assert torch.equal(part[1][:, keys], full[1][:, keys])
    assert torch.equal(part[2][:, keys], full[2][:, keys])
    assert torch.equal(part[3][:, :, keys], full[3][:, :, keys])
    other = [i for i in range(S) if i not in rows]
    assert float(part[0][:, other].abs().max()) == 0.0
