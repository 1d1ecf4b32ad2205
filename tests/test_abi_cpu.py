"""The C ABI without a GPU: the library loads, exports every declared entry
point, computes layouts, and rejects bad arguments before touching the device."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dma():
    import __graft_entry__
    __graft_entry__.build()
    import content_aware_dynamic_dma_b300 as d
    return d


def _declared():
    src = open(os.path.join(ROOT, "include", "dma.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dma_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(dma):
    names = _declared()
    assert "dma_score_keys" in names and "dma_sparse_attn_decode" in names
    lib = ctypes.CDLL(dma.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(dma.EXPORTED) == names


def test_kept_struct_layout_matches_header(dma):
    # 13 int32 fields, 4 bytes of padding, 8 pointers
    assert ctypes.sizeof(dma.KeptT) == 13 * 4 + 4 + 8 * 8
    assert dma.KeptT.expiry.offset == 56


def test_kept_layout_geometry(dma):
    k, ws = dma.dma_kept_layout(1, 8, 65536, 4096, 512, 1, dma.ROWWISE)
    assert (k.B, k.Hkv, k.S, k.w, k.window, k.block, k.mode) == (1, 8, 65536, 4096, 512, 1, 0)
    assert k.q_tile == 128 and k.n_qt == 512 and k.cap == 65536
    assert k.top_cap == 4096
    assert k.tile_stride >= 4096 + 128 and k.tile_stride % 4 == 0
    assert k.bitmap_words == 32
    assert ws > 8 * 65536 * 16
    k, _ = dma.dma_kept_layout(2, 4, 300, 1000, 0, 1, dma.GLOBAL)
    assert k.n_qt == 3 and k.top_cap == 300 and k.tile_stride <= 304 and k.bitmap_words == 1
    k, _ = dma.dma_kept_layout(1, 1, 1000, 200, 64, 64, dma.ROWWISE)
    assert k.top_cap == 192  # floor(200 / 64) blocks of 64
    k, _ = dma.dma_kept_layout(1, 1, 10, 0, 0, 1, dma.ROWWISE)
    assert k.top_cap == 1  # storage for an empty set is still one entry


@pytest.mark.parametrize("args,status", [
    ((0, 1, 16, 4, 0, 1, 0), 1),      # B = 0
    ((1, 1, 16, -1, 0, 1, 0), 1),     # w < 0
    ((1, 1, 16, 4, -2, 1, 0), 1),     # window < 0
    ((1, 1, 16, 4, 0, 32, 0), 2),     # block 32 unsupported
    ((1, 1, 16, 4, 0, 1, 7), 1),      # bad mode
])
def test_kept_layout_rejects(dma, args, status):
    k = dma.KeptT()
    n = ctypes.c_size_t()
    assert dma._lib.dma_kept_layout(*args, ctypes.byref(k), ctypes.byref(n)) == status
    assert dma._lib.dma_last_error_message().decode() != ""


def test_score_rejects_before_launch(dma):
    lib = dma._lib
    fake = ctypes.c_void_p(0x10000)
    # NULL V
    assert lib.dma_score_keys(None, 1, 1, 16, 2, 128, 0, 16, fake, None, fake, None) == dma.DMA_ERR_INVALID_ARG
    # D = 96
    assert lib.dma_score_keys(fake, 1, 1, 16, 2, 96, 0, 16, fake, None, fake, None) == dma.DMA_ERR_UNSUPPORTED
    # misaligned V
    assert lib.dma_score_keys(ctypes.c_void_p(0x10008), 1, 1, 16, 2, 128, 0, 16, fake, None, fake,
                              None) == dma.DMA_ERR_INVALID_ARG
    # key range past S
    assert lib.dma_score_keys(fake, 1, 1, 16, 2, 128, 4, 17, fake, None, fake, None) == dma.DMA_ERR_INVALID_ARG
    # bad dtype
    assert lib.dma_score_keys(fake, 5, 1, 16, 2, 128, 0, 16, fake, None, fake, None) == dma.DMA_ERR_INVALID_ARG
    assert "key range" not in lib.dma_last_error_message().decode()
    # more KV heads than one scoring CTA's rows
    assert lib.dma_score_keys(fake, 1, 1, 16, 129, 64, 0, 16, fake, None, fake, None) == dma.DMA_ERR_UNSUPPORTED
    assert "128 KV heads" in lib.dma_last_error_message().decode()


def test_select_rejects_before_launch(dma):
    lib = dma._lib
    k, ws = dma.dma_kept_layout(1, 2, 256, 64, 0, 1, dma.ROWWISE)
    fake = 0x10000
    k.expiry = k.idx = k.count = fake
    sc = ctypes.c_void_p(fake)
    # workspace too small
    assert lib.dma_select_topk(sc, 1, 2, 256, 64, 0, 1, 0, 0, None, ctypes.byref(k), ctypes.c_void_p(fake), ws - 1,
                               None) == dma.DMA_ERR_WORKSPACE
    # NULL workspace
    assert lib.dma_select_topk(sc, 1, 2, 256, 64, 0, 1, 0, 0, None, ctypes.byref(k), None, ws,
                               None) == dma.DMA_ERR_WORKSPACE
    # w differs from the layout
    assert lib.dma_select_topk(sc, 1, 2, 256, 65, 0, 1, 0, 0, None, ctypes.byref(k), ctypes.c_void_p(fake), ws,
                               None) == dma.DMA_ERR_INVALID_ARG
    # S differs from the layout
    assert lib.dma_select_topk(sc, 1, 2, 255, 64, 0, 1, 0, 0, None, ctypes.byref(k), ctypes.c_void_p(fake), ws,
                               None) == dma.DMA_ERR_INVALID_ARG
    # seq_len with FULL
    assert lib.dma_select_topk(sc, 1, 2, 256, 64, 0, 1, 0, 0, ctypes.c_void_p(fake), ctypes.byref(k),
                               ctypes.c_void_p(fake), ws, None) == dma.DMA_ERR_UNSUPPORTED
    # UPDATE without a top set
    assert lib.dma_select_topk(sc, 1, 2, 256, 64, 0, 1, 0, 1, None, ctypes.byref(k), None, 0,
                               None) == dma.DMA_ERR_INVALID_ARG
    # tampered geometry
    k.tile_stride += 4
    assert lib.dma_select_topk(sc, 1, 2, 256, 64, 0, 1, 0, 0, None, ctypes.byref(k), ctypes.c_void_p(fake), ws,
                               None) == dma.DMA_ERR_INVALID_ARG


def test_prefill_and_decode_reject_before_launch(dma):
    lib = dma._lib
    k, ws = dma.dma_kept_layout(1, 2, 256, 64, 0, 1, dma.ROWWISE)
    f = ctypes.c_void_p(0x10000)
    # H not a multiple of Hkv
    assert lib.dma_sparse_attn_prefill(f, f, f, 1, 1, 256, 3, 2, 64, f, ctypes.byref(k), 0.0, f, None,
                                       None) == dma.DMA_ERR_INVALID_ARG
    # kept arrays missing
    assert lib.dma_sparse_attn_prefill(f, f, f, 1, 1, 256, 4, 2, 64, f, ctypes.byref(k), 0.0, f, None,
                                       None) == dma.DMA_ERR_INVALID_ARG
    # decode: workspace too small
    k.top_idx = k.top_count = 0x10000
    need = dma.dma_decode_workspace_size(1, 4, 2, 64, k.top_cap, k.window)
    assert lib.dma_sparse_attn_decode(f, f, f, 1, 1, 256, None, 4, 2, 64, f, ctypes.byref(k), 0.0, f, None, f,
                                      need - 1, None) == dma.DMA_ERR_WORKSPACE
    # decode: more than 16 query heads per KV head
    assert lib.dma_sparse_attn_decode(f, f, f, 1, 1, 256, None, 34, 2, 64, f, ctypes.byref(k), 0.0, f, None, f,
                                      need, None) == dma.DMA_ERR_UNSUPPORTED


def test_variant_entries_reject_before_launch(dma):
    """Per-head budgets, the bias form and the NSA-style calls check their arguments on the
    host and return before any launch."""
    lib = dma._lib
    f = ctypes.c_void_p(0x10000)
    k, ws = dma.dma_kept_layout(1, 2, 256, 64, 0, 1, dma.ROWWISE)
    k.expiry = k.idx = k.count = 0x10000
    # per-head selection without the budget array
    assert lib.dma_select_topk_heads(f, 1, 2, 256, 64, None, 0, 1, 0, 0, None, ctypes.byref(k), f, ws,
                                     None) == dma.DMA_ERR_INVALID_ARG
    # misaligned budget array
    assert lib.dma_select_topk_heads(f, 1, 2, 256, 64, ctypes.c_void_p(0x10002), 0, 1, 0, 0, None, ctypes.byref(k),
                                     f, ws, None) == dma.DMA_ERR_INVALID_ARG
    # the bias array must be its own array, and the form one of the two
    assert lib.dma_score_keys_bias(f, 1, 1, 16, 2, 128, 0, 16, f, None, 1, f, f, None) == dma.DMA_ERR_INVALID_ARG
    assert lib.dma_score_keys_bias(f, 1, 1, 16, 2, 128, 0, 16, f, None, 1, f, None, None) == dma.DMA_ERR_INVALID_ARG
    assert lib.dma_score_keys_bias(f, 1, 1, 16, 2, 128, 0, 16, f, None, 7, f,
                                   ctypes.c_void_p(0x20000), None) == dma.DMA_ERR_INVALID_ARG
    assert lib.dma_score_keys_backward_bias(f, 1, 1, 16, 2, 128, f, None, 7, f, f, f, None, f, 1 << 20,
                                            None) == dma.DMA_ERR_INVALID_ARG
    # page selection per head without the budget array
    assert lib.dma_select_pages_heads(f, 1, 2, 8, 64, None, 128, None, f, f, 128, None) == dma.DMA_ERR_INVALID_ARG
    # NSA: a block range past the complete blocks, and Kc aliasing K
    assert lib.dma_nsa_compress(f, ctypes.c_void_p(0x20000), 1, 1, 300, 2, 128, 0, 5, ctypes.c_void_p(0x30000),
                                ctypes.c_void_p(0x40000), None) == dma.DMA_ERR_INVALID_ARG
    assert lib.dma_nsa_compress(f, ctypes.c_void_p(0x20000), 1, 1, 300, 2, 128, 0, 4, f, ctypes.c_void_p(0x40000),
                                None) == dma.DMA_ERR_INVALID_ARG
    # NSA patterns: the compressed pattern takes the layout (S / 64, window 0, block 1, global)
    kc, _ = dma.dma_kept_layout(1, 2, 256, 4, 0, 1, dma.GLOBAL)
    kc.expiry = 0x10000
    kr, _ = dma.dma_kept_layout(1, 2, 256, 4, 0, 1, dma.ROWWISE)
    kr.expiry = 0x10000
    assert lib.dma_nsa_kept_pattern(dma.NSA_COMPRESSED, None, ctypes.byref(kr), None) == dma.DMA_ERR_INVALID_ARG
    kw, _ = dma.dma_kept_layout(1, 2, 256, 0, 32, 1, dma.ROWWISE)
    assert lib.dma_nsa_kept_pattern(dma.NSA_WINDOW, None, ctypes.byref(kw), None) == dma.DMA_ERR_INVALID_ARG  # no expiry
    assert lib.dma_nsa_kept_pattern(dma.NSA_WINDOW, None, ctypes.byref(kc), None) == dma.DMA_ERR_INVALID_ARG  # w != 0
    assert lib.dma_nsa_kept_pattern(5, None, ctypes.byref(kc), None) == dma.DMA_ERR_INVALID_ARG
    # the gated sum: D = 96 and NULL gate weights
    assert lib.dma_nsa_combine(f, f, f, f, 1, 1, 16, 4, 96, f, f, f, None, None) == dma.DMA_ERR_UNSUPPORTED
    assert lib.dma_nsa_combine(f, f, f, f, 1, 1, 16, 4, 128, None, f, f, None, None) == dma.DMA_ERR_INVALID_ARG


def test_status_strings(dma):
    names = [dma._lib.dma_status_string(i).decode() for i in range(7)]
    assert names == ["DMA_OK", "DMA_ERR_INVALID_ARG", "DMA_ERR_UNSUPPORTED", "DMA_ERR_WORKSPACE", "DMA_ERR_CUDA",
                     "DMA_ERR_TIMEOUT", "DMA_ERR_DEVICE_CHECK"]
    assert dma.dma_version() >= 1


def test_wait_limit_and_fault_injection_setters(dma):
    """The setters return the previous value; 0 restores the default limit; unknown modes are refused."""
    old = dma.dma_set_wait_limit_ns(12345)
    assert dma.dma_set_wait_limit_ns(0) == 12345
    assert dma.dma_set_wait_limit_ns(old) == 2_000_000_000 or old != 2_000_000_000
    assert dma.dma_set_fault_injection(7) == -1
    m = dma.dma_set_fault_injection(dma.DMA_FAULT_DROP_ARRIVE)
    assert dma.dma_set_fault_injection(m) == dma.DMA_FAULT_DROP_ARRIVE


def test_wait_limit_and_fault_injection_defaults_from_environment(dma):
    """DMA_TIMEOUT_NS and DMA_FAULT_INJECT, read when the library loads (a fresh process)."""
    code = ("import ctypes; lib = ctypes.CDLL(%r); lib.dma_set_wait_limit_ns.restype = ctypes.c_uint64; "
            "lib.dma_set_wait_limit_ns.argtypes = [ctypes.c_uint64]; "
            "print(lib.dma_set_wait_limit_ns(1), lib.dma_set_fault_injection(0))" % dma.LIB_PATH)
    env = dict(os.environ, DMA_TIMEOUT_NS="7777", DMA_FAULT_INJECT="drop_arrive")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["7777", "1"]
    env = {k: v for k, v in os.environ.items() if k not in ("DMA_TIMEOUT_NS", "DMA_FAULT_INJECT")}
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["2000000000", "0"]
