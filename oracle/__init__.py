"""fp64 CPU oracle for dynamic-mask sparse attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it, and
it shares no code with the CUDA path: the arithmetic lives in ``dma_oracle.c``
(plain C, fp64, OpenMP over independent (batch, head) segments), compiled by
``build()`` with gcc and loaded through ctypes.

Functions (all take CPU torch tensors; floating inputs are widened to fp32
exactly -- bf16 is a subset of fp32 -- and every result is fp64):

* ``score(V, W, A)``            importance s = A_h * softplus(v . w_h); form "exp": delta = e^s
* ``select(scores, w, ...)``    per-key top-set interval end ("expiry"); w per KV head or one
* ``attend_rows(...)``          dense masked softmax attention for listed rows
* ``decode(...)``               the last row of a cache of length L
* ``attend_backward(...)``      gradients through the kept pairs (dQ, dK, dV, d score)
* ``score_backward(...)``       gradients through the score (dV, dW, dA)
* ``backward(...)``             both, for a whole score -> select -> attend pass
* ``kept_set(...)``             the kept key set of one row, from an expiry array
* ``nsa_compress``, ``nsa_gates``, ``nsa_compressed_rows``, ``nsa_prefill``
                                the NSA-style three-branch fusion (NSA post, §03)

Method source: Dynamic Mask Attention summary (lsdiaocha.cn), §四 and §五.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dma_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

ROWWISE = 0
GLOBAL = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no fast-math) into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-o", tmp, _SRC,
                               "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_score.argtypes = [P, P, P, I, I, I, I, I, I, P]
        lib.oracle_select.argtypes = [P, I, I, I, I, I, I, P]
        lib.oracle_attend_rows.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double, I, P, P, P]
        lib.oracle_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, ctypes.c_double, P, P]
        lib.oracle_attend_backward.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double, I, P, I, P,
                                               I, P, P, P, P]
        lib.oracle_score_backward.argtypes = [P, P, P, P, I, I, I, I, P, P, P]
        lib.oracle_num_threads.restype = I
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def _f32(t: torch.Tensor) -> np.ndarray:
    return np.ascontiguousarray(t.detach().to("cpu", torch.float32).numpy())


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def score(V: torch.Tensor, W: torch.Tensor, A: Optional[torch.Tensor] = None, key_begin: int = 0,
          key_end: Optional[int] = None, form: str = "log") -> torch.Tensor:
    """s[b,h,j] = A_h * softplus(<V[b,j,h,:], W[h,:]>), fp64 [B][Hkv][S].

    form "exp" returns the dynamic weight itself, delta = exp(s) (DMA summary §五 writes
    delta = exp(tau(v Delta) A)), for the variant that adds delta rather than log delta = s
    to the logits.  Keys outside [key_begin, key_end) are left at 0.
    """
    if form not in ("log", "exp"):
        raise ValueError("form must be 'log' or 'exp'")
    B, S, Hkv, D = V.shape
    key_end = S if key_end is None else key_end
    v, w = _f32(V), _f32(W)
    a = None if A is None else _f32(A)
    out = np.zeros((B, Hkv, S), dtype=np.float64)
    _load().oracle_score(_ptr(v), _ptr(w), _ptr(a), B, S, Hkv, D, key_begin, key_end, _ptr(out))
    if form == "exp":
        out[:, :, key_begin:key_end] = np.exp(out[:, :, key_begin:key_end])
    return torch.from_numpy(out)


def select(scores: torch.Tensor, w, block: int = 1, mode: int = ROWWISE) -> torch.Tensor:
    """Per-key top-set interval end ("expiry"), int32 [B][Hkv][S].

    Key j is in the top set of rows lo_j <= i < expiry_j (lo_j = j for tokens,
    the block's last key for blocks); expiry_j = min(lo_j, S) means never.
    w is one budget for every head, or a sequence of Hkv budgets (Sparse Frontier
    summary, budget allocation across heads): KV head h of every sequence then
    keeps w[h] keys, selected exactly as a uniform budget of w[h] on that head alone.
    """
    B, Hkv, S = scores.shape
    if not isinstance(w, (int, np.integer)):
        w = [int(x) for x in w]
        if len(w) != Hkv:
            raise ValueError("w needs one budget per KV head")
        return torch.cat([select(scores[:, h:h + 1], w[h], block, mode) for h in range(Hkv)], dim=1)
    s = np.ascontiguousarray(scores.to(torch.float64).numpy())
    out = np.zeros((B, Hkv, S), dtype=np.int32)
    _load().oracle_select(_ptr(s), B, Hkv, S, int(w), block, mode, _ptr(out))
    return torch.from_numpy(out)


def attend_rows(Q, K, V, scores, expiry, rows: Sequence[int], window: int, block: int = 1,
                scale: Optional[float] = None):
    """Dense masked softmax attention for the listed rows of every (b, hq).

    Returns (O [B][n_rows][H][D], lse [B][H][n_rows]) in fp64.
    """
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    q, k, v = _f32(Q), _f32(K), _f32(V)
    s = np.ascontiguousarray(scores.to(torch.float64).numpy())
    e = np.ascontiguousarray(expiry.to(torch.int32).numpy())
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    O = np.zeros((B, len(r), H, D), dtype=np.float64)
    lse = np.zeros((B, H, len(r)), dtype=np.float64)
    _load().oracle_attend_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(e), B, S, H, Hkv, D, window, block,
                               float(scale), len(r), _ptr(r), _ptr(O), _ptr(lse))
    return torch.from_numpy(O), torch.from_numpy(lse)


def prefill(Q, K, V, W, A, w, window: int, block: int = 1, mode: int = ROWWISE, rows=None, scale=None,
            form: str = "log"):
    """Score, select and attend in one call.  Returns (O, lse, scores, expiry); the selection
    ranks the log-form scores, and form "exp" adds delta = e^s to the logits instead of s."""
    S = Q.shape[1]
    sc = score(V, W, A)
    ex = select(sc, w, block, mode)
    bias = sc if form == "log" else score(V, W, A, form=form)
    rows = list(range(S)) if rows is None else rows
    O, lse = attend_rows(Q, K, V, bias, ex, rows, window, block, scale)
    return O, lse, sc, ex


def decode(q, Kc, Vc, cache_len, scores, w, window: int, block: int = 1, mode: int = ROWWISE, scale=None,
           bias=None):
    """Attention of one new query row per sequence over its cache of length
    cache_len[b].  q [B][H][D]; Kc, Vc [B][Lmax][Hkv][D]; scores fp64
    [B][Hkv][Lmax].  Returns (o [B][H][D], lse [B][H]) in fp64.

    With per-head budgets (w a sequence) or a separate ``bias`` (the logits' bias, e.g. the
    exp form delta, while ``scores`` ranks), each sequence is the last row of a prefill over
    its own prefix: selection of that prefix, then attention of row L-1."""
    B, H, D = q.shape
    Lmax, Hkv = Kc.shape[1], Kc.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if bias is not None or not isinstance(w, (int, np.integer)):
        bias = scores if bias is None else bias
        o = torch.zeros((B, H, D), dtype=torch.float64)
        lse = torch.zeros((B, H), dtype=torch.float64)
        for b in range(B):
            L = int(cache_len[b])
            ex = select(scores[b:b + 1, :, :L], w, block, mode)
            Qb = torch.zeros((1, L, H, D), dtype=torch.float32)
            Qb[0, L - 1] = q[b].float()
            ob, lb = attend_rows(Qb, Kc[b:b + 1, :L], Vc[b:b + 1, :L], bias[b:b + 1, :, :L], ex, [L - 1], window,
                                 block, scale)
            o[b], lse[b] = ob[0, 0], lb[0, :, 0]
        return o, lse
    qq, k, v = _f32(q), _f32(Kc), _f32(Vc)
    cl = np.ascontiguousarray(np.asarray(cache_len, dtype=np.int32))
    s = np.ascontiguousarray(scores.to(torch.float64).numpy())
    o = np.zeros((B, H, D), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    _load().oracle_decode(_ptr(qq), _ptr(k), _ptr(v), _ptr(cl), _ptr(s), B, Lmax, H, Hkv, D, w, window, block,
                          mode, float(scale), _ptr(o), _ptr(lse))
    return torch.from_numpy(o), torch.from_numpy(lse)


def attend_backward(Q, K, V, scores, expiry, dO, window: int, block: int = 1, scale: Optional[float] = None,
                    segment: Optional[int] = None, rows=None, keys=None):
    """Gradients through the kept pairs of the prefill attention, given dO = dL/dO.

    Returns (dQ [B][S][H][D], dK and dV [B][S][Hkv][D], ds [B][Hkv][S]) in fp64: ds is the
    gradient of the score (the logits' bias).  With ``segment`` = b * Hkv + h, only that
    (batch, KV head) segment -- its keys and its G query heads' rows -- is computed; ``rows``
    (ascending) limits dQ to those rows and ``keys`` limits dK, dV and ds to those keys.
    Everything not computed is zero."""
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    q, k, v, do = _f32(Q), _f32(K), _f32(V), _f32(dO)
    s = np.ascontiguousarray(scores.to(torch.float64).numpy())
    e = np.ascontiguousarray(expiry.to(torch.int32).numpy())
    dQ = np.zeros((B, S, H, D), dtype=np.float64)
    dK = np.zeros((B, S, Hkv, D), dtype=np.float64)
    dV = np.zeros((B, S, Hkv, D), dtype=np.float64)
    ds = np.zeros((B, Hkv, S), dtype=np.float64)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    kk = None if keys is None else np.ascontiguousarray(np.asarray(keys, dtype=np.int32))
    _load().oracle_attend_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(e), _ptr(do), B, S, H, Hkv, D, window,
                                   block, float(scale), -1 if segment is None else int(segment), _ptr(r),
                                   0 if r is None else len(r), _ptr(kk), 0 if kk is None else len(kk), _ptr(dQ),
                                   _ptr(dK), _ptr(dV), _ptr(ds))
    return torch.from_numpy(dQ), torch.from_numpy(dK), torch.from_numpy(dV), torch.from_numpy(ds)


def score_backward(V, W, A, ds, form: str = "log"):
    """Through s = A_h * softplus(v . w_h): returns (dV from the score [B][S][Hkv][D], dW [Hkv][D],
    dA [Hkv]) in fp64, given ds = dL/ds [B][Hkv][S].  form "exp": ds is the gradient of the
    added bias delta = exp(s), so dL/ds = ds * delta (chain rule) before the same steps."""
    B, S, Hkv, D = V.shape
    v, w = _f32(V), _f32(W)
    a = None if A is None else _f32(A)
    if form == "exp":
        ds = ds.to(torch.float64) * score(V, W, A, form="exp")
    elif form != "log":
        raise ValueError("form must be 'log' or 'exp'")
    g = np.ascontiguousarray(ds.to(torch.float64).numpy())
    dV = np.zeros((B, S, Hkv, D), dtype=np.float64)
    dW = np.zeros((Hkv, D), dtype=np.float64)
    dA = np.zeros((Hkv,), dtype=np.float64)
    _load().oracle_score_backward(_ptr(v), _ptr(w), _ptr(a), _ptr(g), B, S, Hkv, D, _ptr(dV), _ptr(dW), _ptr(dA))
    return torch.from_numpy(dV), torch.from_numpy(dW), torch.from_numpy(dA)


def backward(Q, K, V, W, A, w, window: int, dO, block: int = 1, mode: int = ROWWISE, scale=None,
             form: str = "log"):
    """The whole backward of score -> select -> attend: returns (dQ, dK, dV, dW, dA) in fp64,
    dV holding both the attention's and the score's part.  The selection ranks s (form "exp"
    adds delta = e^s to the logits: the same order, hence the same kept sets)."""
    sc = score(V, W, A)
    ex = select(sc, w, block, mode)
    bias = sc if form == "log" else score(V, W, A, form=form)
    dQ, dK, dV, ds = attend_backward(Q, K, V, bias, ex, dO, window, block, scale)
    dV2, dW, dA = score_backward(V, W, A, ds, form)
    return dQ, dK, dV + dV2, dW, dA


def page_scores(scores, cache_len, page_size: int) -> torch.Tensor:
    """Page score of a paged cache (Sparse Frontier summary, decode findings: page-level
    selection; the page's score is the maximum of its keys' scores, as for 64-key blocks):
    ps[b][h][p] = max of scores[b][h][j] over the keys j < cache_len[b] of logical page p
    (keys p*page_size .. p*page_size + page_size - 1); -inf for a page with none.  fp64."""
    B, Hkv, Lmax = scores.shape
    n_pages = (Lmax + page_size - 1) // page_size
    out = torch.full((B, Hkv, n_pages), -math.inf, dtype=torch.float64)
    s = scores.to(torch.float64)
    for b in range(B):
        L = int(cache_len[b])
        for p in range((L + page_size - 1) // page_size):
            out[b, :, p] = s[b, :, p * page_size:min(L, (p + 1) * page_size)].max(dim=-1).values
    return out


def select_pages(scores, cache_len, page_size: int, w):
    """Kept pages of the decode row L-1 (L = cache_len[b]) for every (b, KV head): among the
    complete pages (last key <= L-1), the floor(w / page_size) with the highest page score,
    ties to the lower page index; scores compared as fp32 (-0 equals +0), as the selection
    does.  w: one budget, or one per KV head.  Returns {(b, h): sorted list of kept page
    indices}."""
    B, Hkv, _ = scores.shape
    wh = [int(w)] * Hkv if isinstance(w, (int, np.integer)) else [int(x) for x in w]
    out = {}
    for b in range(B):
        L = int(cache_len[b])
        n_c = L // page_size
        for h in range(Hkv):
            k = wh[h] // page_size
            vals = []
            for p in range(n_c):
                v = max(float(np.float32(x)) + 0.0 for x in scores[b, h, p * page_size:(p + 1) * page_size].tolist())
                vals.append((-v, p))
            vals.sort()
            out[(b, h)] = sorted(p for _, p in vals[:k])
    return out


def top_lo(j, block: int):
    """First row at which key j may enter the top set (its block's last key)."""
    if block <= 1:
        return j
    return (j // block) * block + block - 1


def kept_set(expiry_seg: torch.Tensor, i: int, window: int, block: int = 1) -> set:
    """Kept keys of row i for one (b, h) segment: top interval or local window."""
    ex = expiry_seg.tolist()
    out = set()
    for j in range(i + 1):
        if j > i - window or (top_lo(j, block) <= i < ex[j]):
            out.add(j)
    return out


def top_set(expiry_seg: torch.Tensor, i: int, block: int = 1) -> set:
    """Top-set keys of row i (no window) for one (b, h) segment."""
    ex = expiry_seg.tolist()
    return {j for j in range(i + 1) if top_lo(j, block) <= i < ex[j]}


# ------------------------------------------------------- NSA-style fusion --
#
# NSA post (news.news), §03: three branches run side by side -- attention over compressed
# blocks (a coarse global view), over selected blocks (the important content) and over a
# sliding window (local context) -- and a small gating network gives every token three
# fusion weights.  Readings: a compressed block is the mean of the K (V) rows of a complete
# 64-key block; the selected branch is the block-unit selection of this method (block
# score = max of the key scores) with no window; no branch adds a bias; the gate of query
# head h is sigmoid(<q, G[h, b]> + c[h, b]) for the branches b = compressed, selected,
# window, and the output is the gate-weighted sum of the three branch outputs.

NSA_BLOCK = 64


def nsa_compress(K, V, block: int = NSA_BLOCK):
    """Means of the complete blocks: (Kc, Vc) fp64 [B][S // block][Hkv][D]."""
    B, S, Hkv, D = K.shape
    nb = S // block
    k = _f32(K).astype(np.float64)[:, :nb * block].reshape(B, nb, block, Hkv, D)
    v = _f32(V).astype(np.float64)[:, :nb * block].reshape(B, nb, block, Hkv, D)
    out_k = np.zeros((B, nb, Hkv, D), dtype=np.float64)
    out_v = np.zeros((B, nb, Hkv, D), dtype=np.float64)
    for t in range(block):           # the sum in key order, then one division
        out_k += k[:, :, t]
        out_v += v[:, :, t]
    return torch.from_numpy(out_k / block), torch.from_numpy(out_v / block)


def nsa_gates(Q, G, c):
    """sigmoid(<Q[b, i, h], G[h, branch]> + c[h, branch]), fp64 [B][S][H][3]."""
    q = _f32(Q).astype(np.float64)
    g = _f32(G).astype(np.float64)
    x = np.einsum("bihd,hgd->bihg", q, g) + _f32(c).astype(np.float64)[None, None]
    return torch.from_numpy(1.0 / (1.0 + np.exp(-x)))


def nsa_compressed_rows(Q, Kc, Vc, rows, block: int = NSA_BLOCK, scale: Optional[float] = None):
    """Attention of the listed rows over the compressed blocks they see (block beta is seen by
    row i iff its last key block * beta + block - 1 <= i); no bias.  Returns (O [B][n_rows][H][D],
    lse [B][H][n_rows]) in fp64; a row that sees no block gets O = 0, lse = -inf."""
    B, S, H, D = Q.shape
    Hkv = Kc.shape[2]
    G = H // Hkv
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    q = _f32(Q).astype(np.float64)
    kc = Kc.to(torch.float64).numpy()
    vc = Vc.to(torch.float64).numpy()
    O = np.zeros((B, len(rows), H, D), dtype=np.float64)
    lse = np.full((B, H, len(rows)), -np.inf, dtype=np.float64)
    for r, i in enumerate(rows):
        nv = (i + 1) // block    # blocks 0 .. nv-1 are complete by row i
        if nv == 0:
            continue
        for b in range(B):
            for h in range(H):
                x = scale * (kc[b, :nv, h // G] @ q[b, i, h])
                m = x.max()
                p = np.exp(x - m)
                l = p.sum()
                O[b, r, h] = (p @ vc[b, :nv, h // G]) / l
                lse[b, h, r] = m + math.log(l)
    return torch.from_numpy(O), torch.from_numpy(lse)


def nsa_prefill(Q, K, V, W, A, G, c, w, window: int, rows=None, scale: Optional[float] = None):
    """The three branches and their gated sum for the listed rows.  Returns a dict with O (the
    fused output, [B][n_rows][H][D]), the branch outputs o_cmp, o_slc, o_win and their lse, the
    gates [B][n_rows][H][3], the scores and the selected branch's expiry; fp64."""
    B, S, H, D = Q.shape
    rows = list(range(S)) if rows is None else list(rows)
    sc = score(V, W, A)
    zero = torch.zeros_like(sc)
    ex_slc = select(sc, w, NSA_BLOCK, ROWWISE)
    o_slc, l_slc = attend_rows(Q, K, V, zero, ex_slc, rows, 0, NSA_BLOCK, scale)
    never = torch.arange(S, dtype=torch.int32).expand(sc.shape).contiguous()
    o_win, l_win = attend_rows(Q, K, V, zero, never, rows, window, 1, scale)
    Kc, Vc = nsa_compress(K, V)
    o_cmp, l_cmp = nsa_compressed_rows(Q, Kc, Vc, rows, NSA_BLOCK, scale)
    g = nsa_gates(Q[:, rows], G, c)
    O = g[..., 0:1] * o_cmp + g[..., 1:2] * o_slc + g[..., 2:3] * o_win
    return {"O": O, "o_cmp": o_cmp, "o_slc": o_slc, "o_win": o_win, "lse_cmp": l_cmp, "lse_slc": l_slc,
            "lse_win": l_win, "gates": g, "scores": sc, "expiry": ex_slc}
