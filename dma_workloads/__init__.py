"""Seeded synthetic workloads for dynamic-mask sparse attention.

This module only draws random numbers and lays them out.  It holds none of the
method's arithmetic (no scoring, no selection, no attention), so both the fp64
oracle and the CUDA path can read the very same host arrays from it.

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)`` in
a fixed order -- W, Q, K, V, then the salient-row mask -- and cast to the
workload's dtype afterwards.  bf16 values are exact in fp32, so a consumer that
upcasts reads the same numbers the GPU reads.

Workloads (the shapes of the Dynamic Mask Attention setting: per-KV-head
importance weights, a keep budget ``w`` and an optional local window):

========================  ==  ===  ===  =====  ===  =====  ====  ======  ========
name                      B   H    Hkv  S      D    dtype  w     window  salient
========================  ==  ===  ===  =====  ===  =====  ====  ======  ========
prefill_tiny_s256_fp32    1   2    2    256    64   f32    64    0       no
prefill_s4k_gqa_bf16      1   16   4    4096   128  bf16   1024  128     no
prefill_s16k_bf16         2   32   8    16384  128  bf16   2048  256     yes
prefill_s64k_bf16         1   32   8    65536  128  bf16   4096  512     yes
decode_b64_l32k_bf16      64  32   8    32768  128  bf16   2048  64      yes
========================  ==  ===  ===  =====  ===  =====  ====  ======  ========

Salient rows: a Bernoulli(0.05) mask over (batch, position, KV head) scales
that row of both K and V by 3, which gives the importance scores a heavy tail.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    H: int
    Hkv: int
    S: int          # sequence length (prefill) or cache length L (decode)
    D: int
    dtype: str      # "f32" or "bf16"
    w: int          # keep budget (tokens)
    window: int     # local window length
    salient: bool
    decode: bool = False
    block: int = 1  # selection unit: 1 = token, 64 = 64-key block

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "prefill_tiny_s256_fp32": Workload("prefill_tiny_s256_fp32", 1, 1, 2, 2, 256, 64, "f32", 64, 0, False),
    "prefill_s4k_gqa_bf16": Workload("prefill_s4k_gqa_bf16", 2, 1, 16, 4, 4096, 128, "bf16", 1024, 128, False),
    "prefill_s16k_bf16": Workload("prefill_s16k_bf16", 3, 2, 32, 8, 16384, 128, "bf16", 2048, 256, True),
    "prefill_s64k_bf16": Workload("prefill_s64k_bf16", 4, 1, 32, 8, 65536, 128, "bf16", 4096, 512, True),
    "prefill_s64k_block64_bf16": Workload("prefill_s64k_block64_bf16", 4, 1, 32, 8, 65536, 128, "bf16", 4096, 512,
                                          True, block=64),
    "decode_b64_l32k_bf16": Workload("decode_b64_l32k_bf16", 5, 64, 32, 8, 32768, 128, "bf16", 2048, 64, True,
                                     decode=True),
}


def _randn(g: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32)


def _apply_salient(g: torch.Generator, K: torch.Tensor, V: torch.Tensor, frac: float = 0.05, scale: float = 3.0):
    """Scale a Bernoulli(frac) set of (batch, position, KV head) rows of K and V."""
    B, S, Hkv, _ = K.shape
    mask = torch.rand((B, S, Hkv), generator=g) < frac
    K[mask] *= scale
    V[mask] *= scale
    return mask


def make_prefill(B: int, S: int, H: int, Hkv: int, D: int, dtype: torch.dtype, seed: int,
                 salient: bool = False, w_std: Optional[float] = None, with_gate: bool = False):
    """Seeded prefill inputs on the CPU.

    Returns a dict with
      W  [Hkv][D] fp32, ~N(0, 1/D) unless ``w_std`` is given;
      A  [Hkv] fp32 gate or None (``with_gate`` draws A ~ U(0.5, 1.5) after V);
      Q  [B][S][H][D], K and V [B][S][Hkv][D] in ``dtype``.
    """
    g = torch.Generator().manual_seed(seed)
    std = (1.0 / D) ** 0.5 if w_std is None else w_std
    W = _randn(g, (Hkv, D)) * std
    Q = _randn(g, (B, S, H, D))
    K = _randn(g, (B, S, Hkv, D))
    V = _randn(g, (B, S, Hkv, D))
    if salient:
        _apply_salient(g, K, V)
    A = None
    if with_gate:
        A = torch.rand((Hkv,), generator=g) + 0.5
    return {"W": W.contiguous(), "A": A, "Q": Q.to(dtype).contiguous(), "K": K.to(dtype).contiguous(),
            "V": V.to(dtype).contiguous()}


def make_decode(B: int, L: int, H: int, Hkv: int, D: int, dtype: torch.dtype, seed: int, salient: bool = True,
                n_queries: int = 1, device="cpu", batches=None):
    """Seeded decode inputs: ``n_queries`` new query rows per sequence.

    Returns W [Hkv][D] fp32, q [n_queries][B'][H][D] and the caches Kc, Vc
    [B'][L][Hkv][D] in ``dtype``, on ``device``.  Position ``L - n_queries + k``
    of the cache holds the key/value of the token that query ``k`` belongs to.

    Each sequence b draws from its own generator (seed * 7919 + b + 1; order q,
    K, V, salient mask), so ``batches`` -- a subset of range(B) -- regenerates
    exactly those sequences (B' = len(batches)) without drawing the others.
    The values depend on ``device`` (CPU and CUDA generators differ).
    """
    g = torch.Generator().manual_seed(seed)
    W = _randn(g, (Hkv, D)) * (1.0 / D) ** 0.5
    batches = list(range(B)) if batches is None else list(batches)
    nb = len(batches)
    q = torch.empty((n_queries, nb, H, D), dtype=dtype, device=device)
    Kc = torch.empty((nb, L, Hkv, D), dtype=dtype, device=device)
    Vc = torch.empty((nb, L, Hkv, D), dtype=dtype, device=device)
    for r, b in enumerate(batches):
        gb = torch.Generator(device=device).manual_seed(seed * 7919 + b + 1)
        q[:, r] = torch.randn((n_queries, H, D), generator=gb, device=device).to(dtype)
        k = torch.randn((L, Hkv, D), generator=gb, device=device)
        v = torch.randn((L, Hkv, D), generator=gb, device=device)
        if salient:
            mask = torch.rand((L, Hkv), generator=gb, device=device) < 0.05
            k[mask] *= 3.0
            v[mask] *= 3.0
        Kc[r] = k.to(dtype)
        Vc[r] = v.to(dtype)
    return {"W": W.contiguous().to(device), "A": None, "q": q, "Kc": Kc, "Vc": Vc}


def make_grad(shape, dtype: torch.dtype, seed: int) -> torch.Tensor:
    """A seeded upstream gradient dL/dO ~ N(0, 1) on the CPU, in ``dtype``."""
    g = torch.Generator().manual_seed(seed * 104729 + 17)
    return _randn(g, tuple(shape)).to(dtype).contiguous()


def make_nsa_gates(H: int, D: int, seed: int, g_std: float = 0.1):
    """Seeded gate parameters of the three-branch fusion: G [H][3][D] ~ N(0, g_std^2) and
    c [H][3] ~ N(0, 1), fp32 on the CPU (random-init weights: no trained gates exist here)."""
    g = torch.Generator().manual_seed(seed * 7907 + 3)
    G = _randn(g, (H, 3, D)) * g_std
    c = _randn(g, (H, 3))
    return G.contiguous(), c.contiguous()


def paginate(Kc: torch.Tensor, page_size: int, seed: int, extra_pages: int = 0):
    """A paged copy of a contiguous cache Kc [B][L][Hkv][D]: pages [n_pages][page_size][Hkv][D]
    with the physical pages in seeded random order (plus `extra_pages` unused ones), and the
    block table [B][ceil(L / page_size)] int32; both on Kc's device."""
    B, L, Hkv, D = Kc.shape
    max_pages = (L + page_size - 1) // page_size
    n_pages = B * max_pages + extra_pages
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n_pages, generator=g)[:B * max_pages].view(B, max_pages)
    pages = torch.zeros((n_pages, page_size, Hkv, D), dtype=Kc.dtype, device=Kc.device)
    idx = perm.flatten().to(Kc.device)
    if L == max_pages * page_size:
        pages[idx] = Kc.reshape(B * max_pages, page_size, Hkv, D)
    else:
        pad = torch.zeros((B, max_pages * page_size, Hkv, D), dtype=Kc.dtype, device=Kc.device)
        pad[:, :L] = Kc
        pages[idx] = pad.view(B * max_pages, page_size, Hkv, D)
    return pages.contiguous(), perm.to(torch.int32).to(Kc.device).contiguous()


def make_workload(wl: Workload, n_queries: int = 1, device="cpu", batches=None):
    if wl.decode:
        return make_decode(wl.B, wl.S, wl.H, wl.Hkv, wl.D, wl.torch_dtype, wl.seed, wl.salient, n_queries,
                           device=device, batches=batches)
    return make_prefill(wl.B, wl.S, wl.H, wl.Hkv, wl.D, wl.torch_dtype, wl.seed, wl.salient)


def sample_rows(S: int, n: int, seed: int, w: int = 0, block: int = 64):
    """A seeded, sorted set of query rows that always contains the edge rows.

    Edge rows: 0, w-1, w, S-1 and the rows just after block boundaries near the
    start and end; the rest are uniform draws.  Used where evaluating every row
    on the CPU would take too long.
    """
    g = torch.Generator().manual_seed(seed + 7919)
    edges = {0, S - 1, max(0, w - 1), min(S - 1, w), min(S - 1, block - 1), min(S - 1, block),
             min(S - 1, 2 * block - 1), max(0, S - block - 1), max(0, S - block)}
    rows = set(r for r in edges if 0 <= r < S)
    if n > len(rows):
        draw = torch.randint(0, S, (4 * n,), generator=g).tolist()
        for r in draw:
            if len(rows) >= n:
                break
            rows.add(int(r))
    return sorted(rows)
