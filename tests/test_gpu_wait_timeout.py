"""Failure detection on the GPU without a GPU fault.

Every wait inside the tensor-core prefill kernel has a time limit.  With the
fault-injection switch DMA_FAULT_DROP_ARRIVE, CTA 0 withholds the copy warps'
completion signal for the K rows of its first key block, so the MMA warp's wait
for them runs out: the kernel must record DMA_ERR_TIMEOUT in the device status
word, end on its own (every warp leaves, the copies in flight land), and leave
the CUDA context usable, so that the next launch, without injection, returns
the same output as before.  Nothing here faults, traps or hangs a GPU; the
injected wait ends after a 50 ms limit.
"""
import time

import pytest
import torch

import dma_workloads as wl

pytestmark = pytest.mark.gpu


def test_prefill_wait_timeout_is_reported_and_the_context_survives():
    import content_aware_dynamic_dma_b300 as dma
    assert torch.cuda.is_available()
    B, S, H, Hkv, D, w, window = 1, 1000, 4, 1, 128, 96, 32
    inp = wl.make_prefill(B, S, H, Hkv, D, torch.bfloat16, seed=701)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    O_ref, lse_ref, scores, kept = dma.prefill(d["Q"], d["K"], d["V"], d["W"], d["A"], w, window)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0

    O = torch.zeros_like(O_ref)
    old_limit = dma.dma_set_wait_limit_ns(50_000_000)
    old_mode = dma.dma_set_fault_injection(dma.DMA_FAULT_DROP_ARRIVE)
    try:
        t0 = time.monotonic()
        dma.dma_sparse_attn_prefill(d["Q"], d["K"], d["V"], scores, kept, O)
        torch.cuda.synchronize()
        elapsed = time.monotonic() - t0
    finally:
        dma.dma_set_fault_injection(old_mode)
        dma.dma_set_wait_limit_ns(old_limit)
    assert dma.dma_get_device_status() == dma.DMA_ERR_TIMEOUT
    assert elapsed < 10.0

    # the context is usable and the kernel is unchanged: the same output as before
    O2 = torch.empty_like(O_ref)
    lse2 = torch.empty_like(lse_ref)
    dma.dma_sparse_attn_prefill(d["Q"], d["K"], d["V"], scores, kept, O2, lse2)
    torch.cuda.synchronize()
    assert dma.dma_get_device_status() == 0
    assert torch.equal(O2, O_ref)
    assert torch.equal(lse2, lse_ref)
