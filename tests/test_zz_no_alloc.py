"""Decode without allocation (collected last on purpose).

dma_sparse_attn_decode_noalloc serves callers that may not call cudaMalloc: it
keeps its split-K partials in a fixed device array inside the library instead
of a workspace the caller allocates.  Its output must match
dma_sparse_attn_decode's on the same inputs, on two calls in a row (the array
keeps the previous call's contents, which must not leak into the next result).
The test passes alone in a fresh process and after the other tests.
"""
import pytest
import torch

import dma_workloads as wl
import parity

pytestmark = pytest.mark.gpu


def test_decode_noalloc_matches_workspace_decode():
    import content_aware_dynamic_dma_b300 as dma
    assert torch.cuda.is_available()
    B, L, H, Hkv, D, w, window = 4, 3000, 16, 4, 128, 256, 64
    dt = torch.bfloat16
    inp = wl.make_decode(B, L, H, Hkv, D, dt, seed=601, n_queries=2, device="cuda")
    st = dma.DecodeState(B, L, H, Hkv, D, w, window)
    st.full_select(inp["Kc"], inp["Vc"], inp["W"])
    cl = torch.full((B,), L, dtype=torch.int32, device="cuda")
    for call in range(2):
        q = inp["q"][call]
        o_ref = torch.empty((B, H, D), dtype=dt, device="cuda")
        lse_ref = torch.empty((B, H), dtype=torch.float32, device="cuda")
        dma.dma_sparse_attn_decode(q, inp["Kc"], inp["Vc"], st.scores, st.kept, o_ref, st.ws, lse_ref, cl)
        o = torch.full((B, H, D), float("nan"), dtype=dt, device="cuda")
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        dma.dma_sparse_attn_decode_noalloc(q, inp["Kc"], inp["Vc"], st.scores, st.kept, o, lse, cl)
        torch.cuda.synchronize()
        assert dma.dma_get_device_status() == 0
        # the same kernels on the same inputs: bit for bit the same result (which also keeps it
        # within the parity tolerance of bf16 outputs)
        assert torch.equal(o, o_ref), call
        assert torch.equal(lse, lse_ref), call
        assert float((o.float() - o_ref.float()).abs().max()) <= parity.TOL[dt], call


def test_decode_noalloc_rejects_oversize_before_launch():
    import content_aware_dynamic_dma_b300 as dma
    # 512 sequences x 64 heads x a 32K budget would need far more than the fixed scratch
    B, L, H, Hkv, D, w = 512, 40000, 64, 8, 128, 32768
    kept_t, _ = dma.dma_kept_layout(B, Hkv, L, w, 64, 1, dma.ROWWISE)
    f = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = f.data_ptr()
    import ctypes
    st = dma._lib.dma_sparse_attn_decode_noalloc(ctypes.c_void_p(p), ctypes.c_void_p(p), ctypes.c_void_p(p),
                                                  dma.DMA_BF16, B, L, None, H, Hkv, D, ctypes.c_void_p(p),
                                                  ctypes.byref(kept_t), 0.0, ctypes.c_void_p(p), None, None)
    assert st == dma.DMA_ERR_UNSUPPORTED
    assert "scratch" in dma._lib.dma_last_error_message().decode()
