"""Pins for the fp64 oracle of the NSA-style three-branch fusion (no GPU).

NSA post (news.news), §03: attention over compressed blocks, over selected blocks and
over a sliding window, mixed per token by gates from a small network.  The oracle's
readings -- block means, block-causal visibility of complete blocks, the method's
64-key block selection without a window, no bias, sigmoid gates of the query row --
are pinned by closed forms (an arithmetic ramp, equal keys), torch's fp64
scaled_dot_product_attention with masks built here from Python's sort, and gate
values at chosen points.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import dma_workloads as wl


def _val(row):
    return [float(np.float32(x)) + 0.0 for x in row]


def test_compress_is_block_mean_of_a_ramp(oracle_mod):
    """K[j] = j + 1000 h + d / 2: the mean of block beta is 64 beta + 31.5 + 1000 h + d / 2;
    an incomplete last block is left out."""
    B, S, Hkv, D = 2, 64 * 5 + 17, 3, 16
    j = torch.arange(S, dtype=torch.float32).view(1, S, 1, 1)
    h = torch.arange(Hkv, dtype=torch.float32).view(1, 1, Hkv, 1)
    d = torch.arange(D, dtype=torch.float32).view(1, 1, 1, D)
    K = (j + 1000 * h + d / 2).expand(B, S, Hkv, D).contiguous()
    V = -K
    Kc, Vc = oracle_mod.nsa_compress(K, V)
    assert Kc.shape == (B, 5, Hkv, D)
    beta = torch.arange(5, dtype=torch.float64).view(1, 5, 1, 1)
    want = 64 * beta + 31.5 + 1000 * h.double() + d.double() / 2
    assert torch.equal(Kc, want.expand_as(Kc)) and torch.equal(Vc, -want.expand_as(Vc))


def test_compressed_attention_against_sdpa(oracle_mod):
    """Rows >= 63 against torch SDPA over torch's block means with the block-causal mask
    (block beta seen iff 64 beta + 63 <= i); rows below 63 see no block: O = 0, lse = -inf."""
    B, S, H, Hkv, D = 1, 64 * 6 + 30, 4, 2, 32
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=61)
    Kc, Vc = oracle_mod.nsa_compress(inp["K"], inp["V"])
    rows = list(range(S))
    O, lse = oracle_mod.nsa_compressed_rows(inp["Q"], Kc, Vc, rows, scale=0.2)
    nb = S // 64
    kp = inp["K"].double()[:, :nb * 64].reshape(B, nb, 64, Hkv, D).mean(dim=2)
    vp = inp["V"].double()[:, :nb * 64].reshape(B, nb, 64, Hkv, D).mean(dim=2)
    G = H // Hkv
    q = inp["Q"].double().permute(0, 2, 1, 3)
    k = kp.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    v = vp.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vis = torch.tensor([[64 * bb + 63 <= i for bb in range(nb)] for i in range(S)])
    m = torch.zeros(S, nb, dtype=torch.float64).masked_fill(~vis, -math.inf)
    lo = 63
    o_ref = F.scaled_dot_product_attention(q[:, :, lo:], k, v, attn_mask=m[lo:], scale=0.2).permute(0, 2, 1, 3)
    assert torch.allclose(O[:, lo:], o_ref, rtol=0, atol=1e-12)
    lse_ref = torch.logsumexp(0.2 * q[:, :, lo:] @ k.transpose(-1, -2) + m[lo:], dim=-1)
    assert torch.allclose(lse[:, :, lo:], lse_ref, rtol=0, atol=1e-12)
    assert torch.all(O[:, :lo] == 0) and torch.all(torch.isneginf(lse[:, :, :lo]))


def test_compressed_attention_with_equal_keys_averages_values(oracle_mod):
    """K = 0: every compressed logit is 0, so row i averages the block means it sees, which is
    the plain mean of V over keys 0 .. 64 nv - 1 (nv = (i + 1) // 64)."""
    B, S, H, Hkv, D = 1, 300, 2, 1, 16
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=62)
    K = torch.zeros_like(inp["K"])
    Kc, Vc = oracle_mod.nsa_compress(K, inp["V"])
    rows = [63, 64, 127, 128, 200, 255, 256, 299]
    O, _ = oracle_mod.nsa_compressed_rows(inp["Q"], Kc, Vc, rows)
    for r, i in enumerate(rows):
        nv = (i + 1) // 64
        want = inp["V"].double()[0, :64 * nv, 0].mean(dim=0)
        for h in range(H):
            assert torch.allclose(O[0, r, h], want, rtol=0, atol=1e-13), (i, h)


def test_gates_at_chosen_points(oracle_mod):
    """G = 0 with c = (ln 3, 0, -ln 3) gives (3/4, 1/2, 1/4); a one-hot G reads q's entry."""
    B, S, H, D = 1, 5, 2, 8
    Q = torch.randn(B, S, H, D, generator=torch.Generator().manual_seed(1))
    G = torch.zeros(H, 3, D)
    c = torch.tensor([[math.log(3), 0.0, -math.log(3)]] * H)
    g = oracle_mod.nsa_gates(Q, G, c)
    want = torch.tensor([0.75, 0.5, 0.25], dtype=torch.float64)
    assert torch.allclose(g, want.expand_as(g), rtol=0, atol=1e-7)   # c is fp32
    G = torch.zeros(H, 3, D)
    G[1, 2, 5] = 1.0
    g = oracle_mod.nsa_gates(Q, G, torch.zeros(H, 3))
    x = Q[0, :, 1, 5].double()
    assert torch.allclose(g[0, :, 1, 2], 1 / (1 + torch.exp(-x)), rtol=0, atol=1e-15)
    assert torch.all(g[0, :, 0] == 0.5)


def _fused_torch(inp, G, c, w, window, scale):
    """The fused output built from torch pieces: masks from Python's sort of fp32 block
    maxima, torch block means, SDPA per branch, torch.sigmoid gates."""
    Q, K, V = (inp[k].double() for k in ("Q", "K", "V"))
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    Gq = H // Hkv
    u = torch.einsum("bjhd,hd->bhj", V, inp["W"].double())
    a = torch.ones(Hkv, dtype=torch.float64) if inp["A"] is None else inp["A"].double()
    s = a.view(1, Hkv, 1) * F.softplus(u)
    nb = S // 64
    slc = torch.zeros(B, Hkv, S, S, dtype=torch.bool)
    for b in range(B):
        for h in range(Hkv):
            val = _val(s[b, h].tolist())
            bmax = [max(val[64 * bb:64 * bb + 64]) for bb in range(nb)]
            for i in range(S):
                cand = [bb for bb in range(nb) if 64 * bb + 63 <= i]
                top = sorted(cand, key=lambda bb: (-bmax[bb], bb))[:w // 64]
                for bb in top:
                    slc[b, h, i, 64 * bb:64 * bb + 64] = True
    ii = torch.arange(S).view(S, 1)
    jj = torch.arange(S).view(1, S)
    win = ((jj <= ii) & (jj > ii - window)).expand(B, Hkv, S, S)

    def attend(mask, k, v):
        m = mask.repeat_interleave(Gq, dim=1)
        logits = scale * torch.einsum("bihd,bjhd->bhij", Q, k.repeat_interleave(Gq, dim=2))
        logits = logits.masked_fill(~m, float("-inf"))
        empty = ~m.any(dim=-1, keepdim=True)
        p = torch.softmax(logits.masked_fill(empty, 0.0), dim=-1).masked_fill(empty | ~m, 0.0)
        return torch.einsum("bhij,bjhd->bihd", p, v.repeat_interleave(Gq, dim=2))

    kp = K[:, :nb * 64].reshape(B, nb, 64, Hkv, D).mean(dim=2)
    vp = V[:, :nb * 64].reshape(B, nb, 64, Hkv, D).mean(dim=2)
    vis = torch.tensor([[64 * bb + 63 <= i for bb in range(nb)] for i in range(S)]).expand(B, Hkv, S, nb)
    o_cmp = attend(vis, kp, vp)
    o_slc = attend(slc, K, V)
    o_win = attend(win, K, V)
    g = torch.sigmoid(torch.einsum("bihd,hgd->bihg", Q, G.double()) + c.double())
    return g[..., 0:1] * o_cmp + g[..., 1:2] * o_slc + g[..., 2:3] * o_win, (o_cmp, o_slc, o_win)


@pytest.mark.parametrize("w,window", [(128, 16), (192, 0), (64, 40)])
def test_fused_prefill_against_torch(oracle_mod, w, window):
    B, S, H, Hkv, D = 1, 64 * 5 + 21, 4, 2, 32
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=63 + w, salient=True, with_gate=True)
    gen = torch.Generator().manual_seed(64)
    G = torch.randn(H, 3, D, generator=gen) * 0.2
    c = torch.randn(H, 3, generator=gen)
    r = oracle_mod.nsa_prefill(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], G, c, w, max(window, 1),
                               scale=0.25)
    want, parts = _fused_torch(inp, G, c, w, max(window, 1), 0.25)
    assert torch.allclose(r["O"], want, rtol=0, atol=1e-12)
    for name, p in zip(("o_cmp", "o_slc", "o_win"), parts):
        assert torch.allclose(r[name], p, rtol=0, atol=1e-12), name


def test_saturated_gates_pick_one_branch(oracle_mod):
    """c = (-60, 60, -60): the output is the selected branch alone, which is the method's
    64-key block attention without a window and with a zero bias."""
    B, S, H, Hkv, D = 1, 400, 2, 1, 32
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=65)
    G = torch.zeros(H, 3, D)
    c = torch.tensor([[-60.0, 60.0, -60.0]] * H)
    r = oracle_mod.nsa_prefill(inp["Q"], inp["K"], inp["V"], inp["W"], inp["A"], G, c, 128, 8)
    sc = oracle_mod.score(inp["V"], inp["W"], inp["A"])
    ex = oracle_mod.select(sc, 128, 64)
    o, _ = oracle_mod.attend_rows(inp["Q"], inp["K"], inp["V"], torch.zeros_like(sc), ex, list(range(S)), 0, 64)
    assert torch.allclose(r["O"], o, rtol=0, atol=1e-20)
