"""Comparison rules between the CUDA path and the fp64 oracle (test infrastructure).

* Kept sets match exactly, except keys whose fp32 ranking value lies within
  ``TIE_TOL`` of that row's cutoff (the smallest ranking value in the oracle's
  top set; for global mode the global cutoff).  fp32 scores computed in a
  different summation order can swap such near-ties, which is the only freedom
  the comparison grants.  Rows touched by a swap are left out of the output
  comparison (the oracle is never fed a GPU-derived set).
* Outputs match within a max-abs error of 1e-4 (fp32 inputs) or 2e-2 (bf16),
  for O and for lse.  A bf16 output is rounded once (round-to-nearest-even) from
  the fp32 result; the bound applies to the arithmetic before that rounding, so
  each bf16 element is also granted half a bf16 ulp of the reference value
  (above |O| = 8 that half ulp alone is 0.031, more than 2e-2).
* Gradients (the backward) match within TOL[dtype] times the gradient tensor's
  own scale, max(1, max |reference|): the forward's bound, stated for outputs of
  magnitude about 1, applied to a tensor whose entries are sums of up to
  thousands of terms (dK, dV of a long-kept key).  The bf16 path rounds p and
  dx to bf16 as tensor-core operands (relative 2^-9 each) and the forward's O to
  bf16 (which enters Delta = <dO, O>), so its errors scale with the tensor's
  magnitude, not with each entry's.
"""
from __future__ import annotations

import numpy as np
import torch

TIE_TOL = 1e-5
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
SCORE_ATOL = 5e-5
SCORE_RTOL = 1e-5


def bf16_half_ulp(x: torch.Tensor) -> torch.Tensor:
    """Half the bf16 spacing at |x| (8 significant bits): |x| in [2^(e-1), 2^e)
    has spacing 2^(e-8)."""
    _, e = torch.frexp(x.double().abs())
    return torch.ldexp(torch.ones_like(x, dtype=torch.float64), (e - 9).to(torch.int32))


def out_tol(ref: torch.Tensor, dtype) -> torch.Tensor:
    """Per-element bound for an output of `dtype` against fp64 `ref`."""
    t = torch.full_like(ref, TOL[dtype], dtype=torch.float64)
    if dtype == torch.bfloat16:
        t = t + bf16_half_ulp(ref)
    return t


def top_lo(S: int, block: int) -> np.ndarray:
    j = np.arange(S)
    return j if block <= 1 else (j // block) * block + block - 1


def unit_values(scores32: np.ndarray, block: int) -> np.ndarray:
    """Ranking value of each key's unit: its fp32 score, or its block's max."""
    if block <= 1:
        return scores32
    S = scores32.shape[-1]
    nb = S // block
    out = np.full(S, -np.inf, dtype=np.float64)
    if nb:
        bm = scores32[:nb * block].reshape(nb, block).max(axis=1)
        out[:nb * block] = np.repeat(bm, block)
    return out


def check_scores(gpu: torch.Tensor, ref: torch.Tensor, key_begin: int = 0, key_end=None):
    g = gpu.double().cpu()[..., key_begin:key_end]
    r = ref[..., key_begin:key_end]
    err = (g - r).abs()
    bound = SCORE_ATOL + SCORE_RTOL * r.abs()
    assert bool((err <= bound).all()), "score error %.3g > bound" % float((err - bound).max())


def check_expiry(gpu_ex: torch.Tensor, or_ex: torch.Tensor, or_scores: torch.Tensor, w: int, block: int,
                 mode: int, max_rows: int = 5000):
    """Compares per-key top-set intervals.  Returns {(b, h): set of rows whose
    kept set differs by a near-tie}; raises on any other difference."""
    g = gpu_ex.cpu().numpy()
    o = or_ex.cpu().numpy()
    s32 = or_scores.cpu().numpy().astype(np.float32).astype(np.float64)
    B, Hkv, S = o.shape
    lo = top_lo(S, block)
    affected = {}
    checked = 0
    for b in range(B):
        for h in range(Hkv):
            bad = np.nonzero(g[b, h] != o[b, h])[0]
            if len(bad) == 0:
                continue
            val = unit_values(s32[b, h], block)
            if mode == 1:
                win = (o[b, h] >= S) & (lo < S)
                gcut = val[win].min() if win.any() else np.inf
            rows = set()
            for j in bad:
                a, c = sorted((int(g[b, h, j]), int(o[b, h, j])))
                r0, r1 = max(a, int(lo[j])), min(c, S)
                for i in range(r0, r1):
                    checked += 1
                    assert checked <= max_rows, "too many rows differ"
                    if mode == 1:
                        cut = gcut
                    else:
                        in_top = (lo <= i) & (i < o[b, h]) & (np.arange(S) <= i)
                        cut = val[in_top].min() if in_top.any() else np.inf
                    assert abs(val[j] - cut) <= TIE_TOL, \
                        "key %d (b=%d h=%d) row %d: expiry gpu %d oracle %d, value %.9g cutoff %.9g" % (
                            j, b, h, i, g[b, h, j], o[b, h, j], val[j], cut)
                    rows.add(i)
            affected[(b, h)] = rows
    return affected


def expected_tiles(or_ex: torch.Tensor, window: int, block: int, q_tile: int = 128, tiles=None):
    """Per (b, h, tile): the keys of the gathered list kept by every row of the
    tile and those kept by only some of its rows (two ascending arrays: the
    kernel emits each group in rank order, which check_tile_list verifies
    separately), and the 64-key occupancy bitmap, all derived from the oracle's
    intervals by their definitions."""
    o = or_ex.cpu().numpy()
    B, Hkv, S = o.shape
    lo = top_lo(S, block)
    j = np.arange(S)
    n_qt = (S + q_tile - 1) // q_tile
    words = ((S + 63) // 64 + 31) // 32
    lists, bitmaps = {}, {}
    for b in range(B):
        for h in range(Hkv):
            e = o[b, h]
            for t in (range(n_qt) if tiles is None else tiles):
                q0, q1 = t * q_tile, min(S, (t + 1) * q_tile) - 1
                lim = q0 - window if window > 0 else q1
                top = (lo <= q1) & (e > q0) & (np.maximum(q0, lo) <= np.minimum(q1, e - 1))
                sel = top & (j <= lim)
                every_row = (lo <= q0) & (e > q1)
                lists[(b, h, t)] = (j[sel & every_row], j[sel & ~every_row])
                occ = top.copy()
                if window > 0:
                    occ |= (j <= q1) & (j > q0 - window)
                bits = np.zeros(words, dtype=np.uint32)
                blk = np.unique(j[occ] // 64)
                np.bitwise_or.at(bits, blk // 32, (np.uint32(1) << (blk % 32).astype(np.uint32)))
                bitmaps[(b, h, t)] = bits
    return lists, bitmaps


def rank_sort_key(scores32: np.ndarray) -> np.ndarray:
    """The selection's order as a sortable integer per score: larger is better,
    -0 equals +0, NaN ranks below every number."""
    s = np.where(scores32 == 0, np.float32(0), scores32).astype(np.float32)
    u = s.view(np.uint32).astype(np.int64)
    neg = (u >> 31) == 1
    key = np.where(neg, -(u & 0x7FFFFFFF), u)  # monotone in the float value
    return np.where(np.isnan(s), np.iinfo(np.int64).min, key)


def check_tile_list(got: np.ndarray, want_full: np.ndarray, want_part: np.ndarray, gpu_scores32: np.ndarray,
                    block: int):
    """A gathered list holds exactly the expected keys, every-row keys first;
    inside each group the units run best first by the scores the GPU ranked
    (ties to the lower unit index) and a block's keys ascend."""
    nf = len(want_full)
    assert len(got) == nf + len(want_part), (len(got), nf, len(want_part))
    assert np.array_equal(np.sort(got[:nf]), want_full)
    assert np.array_equal(np.sort(got[nf:]), want_part)
    val = rank_sort_key(unit_values(gpu_scores32, block)) if block > 1 else rank_sort_key(gpu_scores32)
    bs = max(1, block)
    for part in (got[:nf], got[nf:]):
        if len(part) < 2:
            continue
        a, c = part[:-1], part[1:]
        ua, uc = a // bs, c // bs
        ok = (val[a] > val[c]) | ((val[a] == val[c]) & (ua < uc)) | ((ua == uc) & (c == a + 1))
        assert bool(ok.all()), "tile list out of rank order at %s" % (np.nonzero(~ok)[0][:5],)


def check_outputs(O_gpu: torch.Tensor, O_ref: torch.Tensor, lse_gpu, lse_ref, rows, dtype, H: int, Hkv: int,
                  affected=None):
    """O_gpu [B][S][H][D] (all rows), O_ref [B][n_rows][H][D] for `rows`;
    lse_gpu [B][H][S], lse_ref [B][H][n_rows]."""
    tol = TOL[dtype]
    G = H // Hkv
    rows_t = torch.tensor(rows, dtype=torch.long)
    g = O_gpu.double().cpu()[:, rows_t]
    keep = torch.ones(g.shape[0], len(rows), H, dtype=torch.bool)
    if affected:
        for (b, h), rs in affected.items():
            for r_i, i in enumerate(rows):
                if i in rs:
                    keep[b, r_i, h * G:(h + 1) * G] = False
    diff = (g - O_ref).abs()
    err = (diff - out_tol(O_ref, dtype)).amax(dim=-1)
    err = torch.where(keep, err, torch.full_like(err, -1.0))
    assert float(err.max()) <= 0, "max |O - O_ref| exceeds its bound by %.3g" % float(err.max())
    km = keep.unsqueeze(-1).expand_as(diff)
    stats = {"rows": len(rows), "dtype": str(dtype).replace("torch.", ""), "bound": tol,
             "max_err_before_half_ulp": float(diff[km].max()) if bool(km.any()) else 0.0,
             "elements": int(km.sum()), "elements_needing_half_ulp": int(((diff > tol) & km).sum()),
             "row_heads_dropped_near_tie": int((~keep).sum())}
    print("output parity", stats)
    if lse_gpu is not None:
        lg = lse_gpu.double().cpu()[:, :, rows_t]
        kl = keep.permute(0, 2, 1)
        both_inf = torch.isneginf(lg) & torch.isneginf(lse_ref)
        assert bool((both_inf | ~torch.isneginf(lse_ref) | ~kl).all()), "empty rows differ"
        d = torch.where(both_inf | ~kl, torch.zeros_like(lg), (lg - lse_ref).abs())
        assert float(d.max()) <= tol, "max |lse - lse_ref| = %.3g" % float(d.max())
    return int((~keep).sum())


def check_grad(name: str, got: torch.Tensor, ref: torch.Tensor, dtype, select=None) -> dict:
    """Gradient `got` (GPU, fp32) against the fp64 `ref` on the entries `select` (an index or
    boolean mask over the leading dimensions; None = all).  Returns the statistics."""
    g = got.double().cpu()
    r = ref.double()
    if select is not None:
        g, r = g[select], r[select]
    if r.numel() == 0:
        return dict(name=name, n=0)
    scale = max(1.0, float(r.abs().max()))
    err = float((g - r).abs().max())
    bound = TOL[dtype] * scale
    rms_ref = float(r.pow(2).mean().sqrt())
    rel_rms = float((g - r).pow(2).mean().sqrt()) / rms_ref if rms_ref > 0 else 0.0
    stats = dict(name=name, n=int(r.numel()), max_err=err, bound=bound, scale=scale, rel_rms=rel_rms)
    assert err <= bound, "%s: max error %.4g > bound %.4g (scale %.4g, rel rms %.3g)" % (name, err, bound, scale,
                                                                                          rel_rms)
    return stats
