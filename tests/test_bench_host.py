"""Host-side logic of bench.py that needs no GPU: the kept-pair count behind the
headline TFLOP/s, against brute-force enumeration of the keep rule."""
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import dma_workloads as wl  # noqa: E402


def _brute_pairs(expiry, S, window, block, G):
    """Count (b, query head, i, j) with j kept by row i: j <= i and (i - window < j, or
    lo_j <= i < expiry_j), lo_j = j for tokens and the last key of j's block for blocks."""
    e = expiry.numpy().astype(np.int64)
    j = np.arange(S)
    lo = j if block <= 1 else (j // block) * block + block - 1
    i = np.arange(S).reshape(S, 1)
    total = 0
    for b in range(e.shape[0]):
        for h in range(e.shape[1]):
            keep = (j <= i) & ((i - j < window) | ((i >= lo) & (i < e[b, h])))
            total += int(keep.sum())
    return total * G


@pytest.mark.parametrize("w,window,block,mode", [(7, 0, 1, 0), (7, 5, 1, 0), (0, 9, 1, 0), (300, 4, 1, 0),
                                                 (11, 3, 1, 1), (128, 64, 64, 0), (192, 0, 64, 0),
                                                 (64, 70, 64, 1)])
def test_kept_pairs_matches_enumeration(oracle_mod, w, window, block, mode):
    B, S, H, Hkv, D = 2, 200, 6, 3, 64
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.float32, seed=31, w_std=0.7)
    sc = oracle_mod.score(inp["V"], inp["W"], inp["A"])
    ex = oracle_mod.select(sc, w, block, mode)
    G = H // Hkv
    assert bench.kept_pairs(ex, S, window, block, G) == _brute_pairs(ex, S, window, block, G)
