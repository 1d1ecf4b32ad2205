"""Dynamic-mask sparse attention on B300 (sm_103a): Python binding of libdma.

This module only marshals arguments into the C ABI declared in
``include/dma.h``; every step of the computation runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  If ``libdma.so`` is not
built, importing this package raises ImportError: there is no fallback.

The functions carry the C names:

* ``dma_score_keys``          s[b,h,j] = A_h * softplus(<V[b,j,h,:], W[h,:]>)
* ``dma_score_keys_bias``     the same plus the logits' bias: s, or delta = exp(s)
* ``dma_select_topk``         causal top-w selection (FULL or UPDATE)
* ``dma_select_topk_heads``   the same with a budget per KV head
* ``dma_sparse_attn_prefill`` masked softmax attention over the kept keys
* ``dma_sparse_attn_decode``  the same for one new query row per sequence
* ``dma_sparse_attn_prefill_backward``  dQ, dK, dV and ds over the kept pairs
* ``dma_score_keys_backward``  ds -> dW, dA and the score's share of dV
  (``dma_score_keys_backward_bias``: for either form of the bias)
* ``dma_score_keys_paged``, ``dma_select_pages`` (``dma_select_pages_heads``),
  ``dma_sparse_attn_decode_paged``: page-granular decode over a paged KV cache
* ``dma_nsa_compress``, ``dma_nsa_kept_pattern``, ``dma_nsa_combine``: the NSA-style
  three-branch fusion (compressed blocks, selected blocks, sliding window)

plus ``Kept`` (the caller-owned kept-key arrays, allocated with torch) and the
compositions ``prefill``, ``prefill_backward``, ``DecodeState``, ``PagedDecodeState``,
``NsaPrefill`` and ``NsaDecode`` for the common call sequences.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdma.so")

DMA_OK = 0
DMA_ERR_INVALID_ARG = 1
DMA_ERR_UNSUPPORTED = 2
DMA_ERR_WORKSPACE = 3
DMA_ERR_CUDA = 4
DMA_ERR_TIMEOUT = 5
DMA_ERR_DEVICE_CHECK = 6

DMA_F32 = 0
DMA_BF16 = 1
ROWWISE = 0
GLOBAL = 1
FULL = 0
UPDATE = 1
BIAS_LOG = 0
BIAS_EXP = 1
NSA_COMPRESSED = 0
NSA_WINDOW = 1
NSA_BLOCK = 64
Q_TILE = 128


class DmaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (_status_name(status), msg))
        self.status = status


class KeptT(ctypes.Structure):
    """Mirror of dma_kept_t (include/dma.h)."""
    _fields_ = [(n, ctypes.c_int32) for n in
                ("B", "Hkv", "S", "w", "window", "block", "mode", "q_tile", "n_qt", "cap", "top_cap",
                 "tile_stride", "bitmap_words")] + \
               [(n, ctypes.c_void_p) for n in
                ("expiry", "idx", "count", "top_idx", "top_count", "tile_cnt", "tile_idx", "bitmap")]


EXPORTED = ("dma_score_keys", "dma_kept_layout", "dma_select_topk", "dma_sparse_attn_prefill",
            "dma_decode_workspace_size", "dma_sparse_attn_decode", "dma_sparse_attn_decode_noalloc",
            "dma_get_device_status", "dma_status_string", "dma_last_error_message", "dma_set_prefill_kernel",
            "dma_set_wait_limit_ns", "dma_set_fault_injection", "dma_version", "dma_backward_workspace_size",
            "dma_sparse_attn_prefill_backward", "dma_score_keys_backward", "dma_score_keys_paged",
            "dma_select_pages", "dma_sparse_attn_decode_paged", "dma_score_keys_bias", "dma_select_topk_heads",
            "dma_select_pages_heads", "dma_score_keys_backward_bias", "dma_nsa_compress", "dma_nsa_kept_pattern",
            "dma_nsa_combine", "dma_score_keys_paged_bias")


def _load_lib():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libdma.so is not built (%s); run: python content_aware_dynamic_dma_b300/build.py"
                          % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    PK = ctypes.POINTER(KeptT)
    sig = {
        "dma_score_keys": [P, I, I, I, I, I, I, I, P, P, P, P],
        "dma_kept_layout": [I, I, I, I, I, I, I, PK, ctypes.POINTER(Z)],
        "dma_select_topk": [P, I, I, I, I, I, I, I, I, P, PK, P, Z, P],
        "dma_sparse_attn_prefill": [P, P, P, I, I, I, I, I, I, P, PK, F, P, P, P],
        "dma_decode_workspace_size": [I, I, I, I, I, I, ctypes.POINTER(Z)],
        "dma_sparse_attn_decode": [P, P, P, I, I, I, P, I, I, I, P, PK, F, P, P, P, Z, P],
        "dma_sparse_attn_decode_noalloc": [P, P, P, I, I, I, P, I, I, I, P, PK, F, P, P, P],
        "dma_get_device_status": [P, ctypes.POINTER(I)],
        "dma_status_string": [I],
        "dma_last_error_message": [],
        "dma_set_prefill_kernel": [I],
        "dma_set_wait_limit_ns": [ctypes.c_uint64],
        "dma_set_fault_injection": [I],
        "dma_version": [],
        "dma_backward_workspace_size": [I, I, I, I, I, ctypes.POINTER(Z)],
        "dma_sparse_attn_prefill_backward": [P, P, P, I, I, I, I, I, I, P, PK, F, P, P, P, P, P, P, P, P, Z, P],
        "dma_score_keys_backward": [P, I, I, I, I, I, P, P, P, P, P, P, P, Z, P],
        "dma_score_keys_paged": [P, I, I, P, I, I, I, P, I, I, I, I, P, P, P, P, P],
        "dma_select_pages": [P, I, I, I, I, P, I, P, P, I, P],
        "dma_sparse_attn_decode_paged": [P, P, P, I, I, P, I, I, I, P, I, I, I, P, P, P, I, I, F, P, P, P, Z, P],
        "dma_score_keys_bias": [P, I, I, I, I, I, I, I, P, P, I, P, P, P],
        "dma_select_topk_heads": [P, I, I, I, I, P, I, I, I, I, P, PK, P, Z, P],
        "dma_select_pages_heads": [P, I, I, I, I, P, I, P, P, P, I, P],
        "dma_score_keys_backward_bias": [P, I, I, I, I, I, P, P, I, P, P, P, P, P, Z, P],
        "dma_nsa_compress": [P, P, I, I, I, I, I, I, I, P, P, P],
        "dma_nsa_kept_pattern": [I, P, PK, P],
        "dma_nsa_combine": [P, P, P, P, I, I, I, I, I, P, P, P, P, P],
        "dma_score_keys_paged_bias": [P, I, I, P, I, I, I, P, I, I, I, I, P, P, I, P, P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I
    lib.dma_set_wait_limit_ns.restype = ctypes.c_uint64
    lib.dma_status_string.restype = ctypes.c_char_p
    lib.dma_last_error_message.restype = ctypes.c_char_p
    return lib


_lib = _load_lib()


def _status_name(s: int) -> str:
    return _lib.dma_status_string(s).decode()


def _check(status: int):
    if status != DMA_OK:
        raise DmaError(status, _lib.dma_last_error_message().decode())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DMA_F32
    if t.dtype == torch.bfloat16:
        return DMA_BF16
    raise TypeError("tensor dtype %s: expected float32 or bfloat16" % t.dtype)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------- C names ----

def dma_score_keys(V: torch.Tensor, W: torch.Tensor, A: Optional[torch.Tensor], scores: torch.Tensor,
                   key_begin: int = 0, key_end: Optional[int] = None, stream=None) -> None:
    B, S, Hkv, D = V.shape
    key_end = S if key_end is None else key_end
    _check(_lib.dma_score_keys(_ptr(V), _dtype(V), B, S, Hkv, D, key_begin, key_end, _ptr(W), _ptr(A), _ptr(scores),
                               _stream(stream)))


def dma_score_keys_bias(V: torch.Tensor, W: torch.Tensor, A: Optional[torch.Tensor], form: int,
                        scores: torch.Tensor, bias: torch.Tensor, key_begin: int = 0, key_end: Optional[int] = None,
                        stream=None) -> None:
    """scores (the ranking key s) and bias (s for BIAS_LOG, exp(s) for BIAS_EXP), [B][Hkv][S] fp32."""
    B, S, Hkv, D = V.shape
    key_end = S if key_end is None else key_end
    _check(_lib.dma_score_keys_bias(_ptr(V), _dtype(V), B, S, Hkv, D, key_begin, key_end, _ptr(W), _ptr(A), form,
                                    _ptr(scores), _ptr(bias), _stream(stream)))


def dma_kept_layout(B: int, Hkv: int, S: int, w: int, window: int, block: int = 1, mode: int = ROWWISE):
    k = KeptT()
    ws = ctypes.c_size_t(0)
    _check(_lib.dma_kept_layout(B, Hkv, S, w, window, block, mode, ctypes.byref(k), ctypes.byref(ws)))
    return k, ws.value


class Kept:
    """Caller-owned kept-key arrays (torch device tensors) and their dma_kept_t."""

    def __init__(self, B: int, Hkv: int, S: int, w: int, window: int, block: int = 1, mode: int = ROWWISE,
                 device="cuda", tiles: bool = True, top: bool = True, bitmap: bool = True):
        self.t, self.select_ws_bytes = dma_kept_layout(B, Hkv, S, w, window, block, mode)
        t = self.t
        i32 = dict(dtype=torch.int32, device=device)
        self.expiry = torch.empty((B, Hkv, S), **i32)
        self.idx = torch.empty((B, Hkv, t.cap), **i32)
        self.count = torch.zeros((B, Hkv), **i32)
        self.top_idx = torch.empty((B, Hkv, t.top_cap), **i32) if top else None
        self.top_count = torch.zeros((B, Hkv), **i32) if top else None
        self.tile_cnt = torch.zeros((B, Hkv, t.n_qt), **i32) if tiles else None
        self.tile_idx = torch.empty((B, Hkv, t.n_qt, t.tile_stride), **i32) if tiles else None
        self.bitmap = (torch.zeros((B, Hkv, t.n_qt, t.bitmap_words), dtype=torch.int32, device=device)
                       if (tiles and bitmap) else None)
        self.ws = torch.empty((max(self.select_ws_bytes, 16),), dtype=torch.uint8, device=device)
        for name in ("expiry", "idx", "count", "top_idx", "top_count", "tile_cnt", "tile_idx", "bitmap"):
            ten = getattr(self, name)
            setattr(t, name, ten.data_ptr() if ten is not None else None)

    @property
    def B(self):
        return self.t.B

    @property
    def Hkv(self):
        return self.t.Hkv

    @property
    def S(self):
        return self.t.S

    @property
    def w(self):
        return self.t.w

    @property
    def window(self):
        return self.t.window

    @property
    def block(self):
        return self.t.block

    @property
    def mode(self):
        return self.t.mode


def dma_select_topk(scores: torch.Tensor, kept: Kept, op: int = FULL, seq_len: Optional[torch.Tensor] = None,
                    ws: Optional[torch.Tensor] = None, stream=None) -> None:
    B, Hkv, S = scores.shape
    t = kept.t
    ws = kept.ws if ws is None else ws
    _check(_lib.dma_select_topk(_ptr(scores), B, Hkv, S, t.w, t.window, t.block, t.mode, op, _ptr(seq_len),
                                ctypes.byref(t), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def dma_select_topk_heads(scores: torch.Tensor, kept: Kept, w_head: torch.Tensor, op: int = FULL,
                          seq_len: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    """w_head: device int32 [Hkv], 0 <= w_head[h] <= kept.w (the layout's budget)."""
    B, Hkv, S = scores.shape
    t = kept.t
    ws = kept.ws if ws is None else ws
    _check(_lib.dma_select_topk_heads(_ptr(scores), B, Hkv, S, t.w, _ptr(w_head), t.window, t.block, t.mode, op,
                                      _ptr(seq_len), ctypes.byref(t), _ptr(ws), ws.numel() * ws.element_size(),
                                      _stream(stream)))


def dma_sparse_attn_prefill(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scores: torch.Tensor, kept: Kept,
                            O: torch.Tensor, lse: Optional[torch.Tensor] = None, scale: float = 0.0,
                            stream=None) -> None:
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    _check(_lib.dma_sparse_attn_prefill(_ptr(Q), _ptr(K), _ptr(V), _dtype(Q), B, S, H, Hkv, D, _ptr(scores),
                                        ctypes.byref(kept.t), float(scale), _ptr(O), _ptr(lse), _stream(stream)))


def dma_decode_workspace_size(B: int, H: int, Hkv: int, D: int, top_cap: int, window: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.dma_decode_workspace_size(B, H, Hkv, D, top_cap, window, ctypes.byref(n)))
    return n.value


def dma_sparse_attn_decode(q: torch.Tensor, Kc: torch.Tensor, Vc: torch.Tensor, scores: torch.Tensor, kept: Kept,
                           o: torch.Tensor, ws: torch.Tensor, lse: Optional[torch.Tensor] = None,
                           cache_len: Optional[torch.Tensor] = None, scale: float = 0.0, stream=None) -> None:
    B, H, D = q.shape
    Lmax, Hkv = Kc.shape[1], Kc.shape[2]
    _check(_lib.dma_sparse_attn_decode(_ptr(q), _ptr(Kc), _ptr(Vc), _dtype(q), B, Lmax, _ptr(cache_len), H, Hkv, D,
                                       _ptr(scores), ctypes.byref(kept.t), float(scale), _ptr(o), _ptr(lse),
                                       _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def dma_sparse_attn_decode_noalloc(q: torch.Tensor, Kc: torch.Tensor, Vc: torch.Tensor, scores: torch.Tensor,
                                   kept: Kept, o: torch.Tensor, lse: Optional[torch.Tensor] = None,
                                   cache_len: Optional[torch.Tensor] = None, scale: float = 0.0,
                                   stream=None) -> None:
    """dma_sparse_attn_decode for callers that cannot allocate: its scratch is a
    fixed 64 MiB device array inside the library, shared by all calls on a
    device (serialise calls that could overlap on the GPU)."""
    B, H, D = q.shape
    Lmax, Hkv = Kc.shape[1], Kc.shape[2]
    _check(_lib.dma_sparse_attn_decode_noalloc(_ptr(q), _ptr(Kc), _ptr(Vc), _dtype(q), B, Lmax, _ptr(cache_len), H,
                                               Hkv, D, _ptr(scores), ctypes.byref(kept.t), float(scale), _ptr(o),
                                               _ptr(lse), _stream(stream)))


def dma_backward_workspace_size(B: int, S: int, H: int, Hkv: int, D: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.dma_backward_workspace_size(B, S, H, Hkv, D, ctypes.byref(n)))
    return n.value


def _bwd_ws(ws, B, S, H, Hkv, D, device):
    if ws is None:
        ws = torch.empty((dma_backward_workspace_size(B, S, H, Hkv, D),), dtype=torch.uint8, device=device)
    return ws


def dma_sparse_attn_prefill_backward(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scores: torch.Tensor,
                                     kept: Kept, O: torch.Tensor, lse: torch.Tensor, dO: torch.Tensor,
                                     dQ: torch.Tensor, dK: torch.Tensor, dV: torch.Tensor, ds: torch.Tensor,
                                     scale: float = 0.0, ws: Optional[torch.Tensor] = None, stream=None) -> None:
    """dQ [B][S][H][D], dK and dV [B][S][Hkv][D], ds [B][Hkv][S] (all fp32) are written."""
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    for name, t in (("dQ", dQ), ("dK", dK), ("dV", dV), ("ds", ds), ("lse", lse)):
        if t.dtype != torch.float32:
            raise TypeError("%s must be float32" % name)
    ws = _bwd_ws(ws, B, S, H, Hkv, D, Q.device)
    _check(_lib.dma_sparse_attn_prefill_backward(
        _ptr(Q), _ptr(K), _ptr(V), _dtype(Q), B, S, H, Hkv, D, _ptr(scores), ctypes.byref(kept.t), float(scale),
        _ptr(O), _ptr(lse), _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ds), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def dma_score_keys_backward(V: torch.Tensor, W: torch.Tensor, A: Optional[torch.Tensor], ds: torch.Tensor,
                            dV: torch.Tensor, dW: torch.Tensor, dA: Optional[torch.Tensor] = None,
                            ws: Optional[torch.Tensor] = None, stream=None) -> None:
    """Adds the score path's share to dV; writes dW [Hkv][D] and dA [Hkv] (fp32)."""
    B, S, Hkv, D = V.shape
    ws = _bwd_ws(ws, B, S, Hkv, Hkv, D, V.device)
    _check(_lib.dma_score_keys_backward(_ptr(V), _dtype(V), B, S, Hkv, D, _ptr(W), _ptr(A), _ptr(ds), _ptr(dV),
                                        _ptr(dW), _ptr(dA), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)))


def dma_score_keys_backward_bias(V: torch.Tensor, W: torch.Tensor, A: Optional[torch.Tensor], form: int,
                                 ds: torch.Tensor, dV: torch.Tensor, dW: torch.Tensor,
                                 dA: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                                 stream=None) -> None:
    """dma_score_keys_backward for a bias of form BIAS_LOG or BIAS_EXP (ds = dL/d bias)."""
    B, S, Hkv, D = V.shape
    ws = _bwd_ws(ws, B, S, Hkv, Hkv, D, V.device)
    _check(_lib.dma_score_keys_backward_bias(_ptr(V), _dtype(V), B, S, Hkv, D, _ptr(W), _ptr(A), form, _ptr(ds),
                                             _ptr(dV), _ptr(dW), _ptr(dA), _ptr(ws), ws.numel() * ws.element_size(),
                                             _stream(stream)))


def dma_score_keys_paged(V_pages: torch.Tensor, block_table: torch.Tensor, W: torch.Tensor, A: Optional[torch.Tensor],
                         scores: torch.Tensor, page_scores: Optional[torch.Tensor] = None,
                         cache_len: Optional[torch.Tensor] = None, key_begin: int = 0, key_end: Optional[int] = None,
                         stream=None) -> None:
    """V_pages [n_pages][page_size][Hkv][D]; block_table [B][max_pages] int32; scores
    [B][Hkv][max_pages * page_size]; page_scores [B][Hkv][max_pages] (fp32)."""
    n_pages, P, Hkv, D = V_pages.shape
    B, max_pages = block_table.shape
    key_end = max_pages * P if key_end is None else key_end
    _check(_lib.dma_score_keys_paged(_ptr(V_pages), _dtype(V_pages), n_pages, _ptr(block_table), B, max_pages, P,
                                     _ptr(cache_len), Hkv, D, key_begin, key_end, _ptr(W), _ptr(A), _ptr(scores),
                                     _ptr(page_scores), _stream(stream)))


def dma_score_keys_paged_bias(V_pages: torch.Tensor, block_table: torch.Tensor, W: torch.Tensor,
                              A: Optional[torch.Tensor], form: int, scores: torch.Tensor, bias: torch.Tensor,
                              page_scores: Optional[torch.Tensor] = None, cache_len: Optional[torch.Tensor] = None,
                              key_begin: int = 0, key_end: Optional[int] = None, stream=None) -> None:
    """dma_score_keys_paged plus the bias array (s, or exp(s) for BIAS_EXP) for the paged decode."""
    n_pages, P, Hkv, D = V_pages.shape
    B, max_pages = block_table.shape
    key_end = max_pages * P if key_end is None else key_end
    _check(_lib.dma_score_keys_paged_bias(_ptr(V_pages), _dtype(V_pages), n_pages, _ptr(block_table), B, max_pages,
                                          P, _ptr(cache_len), Hkv, D, key_begin, key_end, _ptr(W), _ptr(A), form,
                                          _ptr(scores), _ptr(page_scores), _ptr(bias), _stream(stream)))


def dma_select_pages(page_scores: torch.Tensor, page_size: int, w: int, top_idx: torch.Tensor,
                     top_count: torch.Tensor, cache_len: Optional[torch.Tensor] = None, stream=None) -> None:
    B, Hkv, max_pages = page_scores.shape
    _check(_lib.dma_select_pages(_ptr(page_scores), B, Hkv, max_pages, page_size, _ptr(cache_len), w, _ptr(top_idx),
                                 _ptr(top_count), top_idx.shape[-1], _stream(stream)))


def dma_select_pages_heads(page_scores: torch.Tensor, page_size: int, w: int, w_head: torch.Tensor,
                           top_idx: torch.Tensor, top_count: torch.Tensor, cache_len: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    B, Hkv, max_pages = page_scores.shape
    _check(_lib.dma_select_pages_heads(_ptr(page_scores), B, Hkv, max_pages, page_size, _ptr(cache_len), w,
                                       _ptr(w_head), _ptr(top_idx), _ptr(top_count), top_idx.shape[-1],
                                       _stream(stream)))


def dma_sparse_attn_decode_paged(q: torch.Tensor, K_pages: torch.Tensor, V_pages: torch.Tensor,
                                 block_table: torch.Tensor, scores: torch.Tensor, top_idx: torch.Tensor,
                                 top_count: torch.Tensor, window: int, o: torch.Tensor, ws: torch.Tensor,
                                 lse: Optional[torch.Tensor] = None, cache_len: Optional[torch.Tensor] = None,
                                 scale: float = 0.0, stream=None) -> None:
    B, H, D = q.shape
    n_pages, P, Hkv, _ = K_pages.shape
    max_pages = block_table.shape[1]
    _check(_lib.dma_sparse_attn_decode_paged(
        _ptr(q), _ptr(K_pages), _ptr(V_pages), _dtype(q), n_pages, _ptr(block_table), B, max_pages, P,
        _ptr(cache_len), H, Hkv, D, _ptr(scores), _ptr(top_idx), _ptr(top_count), top_idx.shape[-1], window,
        float(scale), _ptr(o), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def dma_get_device_status(stream=None) -> int:
    v = ctypes.c_int(0)
    _check(_lib.dma_get_device_status(_stream(stream), ctypes.byref(v)))
    return v.value


def dma_set_prefill_kernel(which: int) -> int:
    """0 = automatic (tensor-core kernels for bf16, forward and backward), 1 = SIMT kernels."""
    return _lib.dma_set_prefill_kernel(which)


DMA_FAULT_NONE = 0
DMA_FAULT_DROP_ARRIVE = 1


def dma_set_wait_limit_ns(ns: int) -> int:
    """Limit of the kernels' bounded waits for later launches (0 = the default); returns the old one."""
    return _lib.dma_set_wait_limit_ns(ns)


def dma_set_fault_injection(mode: int) -> int:
    """DMA_FAULT_NONE or DMA_FAULT_DROP_ARRIVE (test aid); returns the old mode, -1 if unknown."""
    return _lib.dma_set_fault_injection(mode)


def dma_version() -> int:
    return _lib.dma_version()


# ------------------------------------------------------------ compositions ---

def prefill(Q, K, V, W, A, w: int, window: int, block: int = 1, mode: int = ROWWISE, scale: float = 0.0,
            kept: Optional[Kept] = None, with_lse: bool = True, stream=None, form: int = BIAS_LOG,
            w_head: Optional[torch.Tensor] = None):
    """Score, select and attend: the whole prefill hot path in three library calls.

    form BIAS_EXP adds delta = exp(s) to the logits instead of s; w_head (device int32 [Hkv],
    each at most w) gives every KV head its own budget.  Returns (O, lse, bias, kept): bias is
    the array the logits got, which the backward and decode calls take as their scores --
    the ranking scores themselves for BIAS_LOG."""
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    scores = torch.empty((B, Hkv, S), dtype=torch.float32, device=Q.device)
    bias = scores
    if form == BIAS_LOG:
        dma_score_keys(V, W, A, scores, stream=stream)
    else:
        bias = torch.empty_like(scores)
        dma_score_keys_bias(V, W, A, form, scores, bias, stream=stream)
    if kept is None:
        kept = Kept(B, Hkv, S, w, window, block, mode, device=Q.device)
    if w_head is None:
        dma_select_topk(scores, kept, FULL, stream=stream)
    else:
        dma_select_topk_heads(scores, kept, w_head, FULL, stream=stream)
    O = torch.empty_like(Q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=Q.device) if with_lse else None
    dma_sparse_attn_prefill(Q, K, V, bias, kept, O, lse, scale, stream=stream)
    return O, lse, bias, kept


def prefill_backward(Q, K, V, W, A, O, lse, bias, kept: Kept, dO, scale: float = 0.0, stream=None,
                     form: int = BIAS_LOG):
    """Backward of ``prefill`` through the same kept sets (``bias`` as prefill returned it):
    returns (dQ, dK, dV, dW, dA), fp32, with dV holding both the attention's and the score's
    share (dA is None when A is None)."""
    B, S, H, D = Q.shape
    Hkv = K.shape[2]
    dev = Q.device
    f32 = dict(dtype=torch.float32, device=dev)
    dQ = torch.empty((B, S, H, D), **f32)
    dK = torch.empty((B, S, Hkv, D), **f32)
    dV = torch.empty((B, S, Hkv, D), **f32)
    ds = torch.empty((B, Hkv, S), **f32)
    dW = torch.empty((Hkv, D), **f32)
    dA = torch.empty((Hkv,), **f32) if A is not None else None
    ws = _bwd_ws(None, B, S, H, Hkv, D, dev)
    dma_sparse_attn_prefill_backward(Q, K, V, bias, kept, O, lse, dO, dQ, dK, dV, ds, scale, ws, stream)
    if form == BIAS_LOG:
        dma_score_keys_backward(V, W, A, ds, dV, dW, dA, ws, stream)
    else:
        dma_score_keys_backward_bias(V, W, A, form, ds, dV, dW, dA, ws, stream)
    return dQ, dK, dV, dW, dA


class DecodeState:
    """Decode-side buffers: the score cache, the kept top set and the workspace.  form BIAS_EXP
    keeps a second cache, the bias delta = exp(s) the logits get; w_head (device int32 [Hkv],
    each at most w) gives every KV head its own budget."""

    def __init__(self, B: int, Lmax: int, H: int, Hkv: int, D: int, w: int, window: int, device="cuda",
                 form: int = BIAS_LOG, w_head: Optional[torch.Tensor] = None):
        self.B, self.Lmax, self.H, self.Hkv, self.D = B, Lmax, H, Hkv, D
        self.form, self.w_head = form, w_head
        self.scores = torch.zeros((B, Hkv, Lmax), dtype=torch.float32, device=device)
        self.bias = self.scores if form == BIAS_LOG else torch.zeros_like(self.scores)
        self.kept = Kept(B, Hkv, Lmax, w, window, 1, ROWWISE, device=device, tiles=False)
        self.ws = torch.empty((dma_decode_workspace_size(B, H, Hkv, D, self.kept.t.top_cap, window),),
                              dtype=torch.uint8, device=device)

    def _score(self, Vc, W, A, key_begin, key_end, stream):
        if self.form == BIAS_LOG:
            dma_score_keys(Vc, W, A, self.scores, key_begin, key_end, stream=stream)
        else:
            dma_score_keys_bias(Vc, W, A, self.form, self.scores, self.bias, key_begin, key_end, stream=stream)

    def _select(self, scores, kept, op, seq_len=None, stream=None):
        if self.w_head is None:
            dma_select_topk(scores, kept, op, seq_len=seq_len, stream=stream)
        else:
            dma_select_topk_heads(scores, kept, self.w_head, op, seq_len=seq_len, stream=stream)

    def full_select(self, Kc, Vc, W, A=None, length: Optional[int] = None, stream=None):
        """Scores the first ``length`` cache rows and selects the top set of row length-1.

        Everything runs on ``stream`` (torch's current stream when None), the copies of the
        prefix selection included."""
        length = self.Lmax if length is None else length
        stream = torch.cuda.current_stream() if stream is None else stream
        self._score(Vc, W, A, 0, length, stream)
        if length == self.Lmax:
            self._select(self.scores, self.kept, FULL, stream=stream)
            return
        with torch.cuda.stream(stream):
            sub = Kept(self.B, self.Hkv, length, self.kept.w, self.kept.window, 1, ROWWISE,
                       device=self.scores.device, tiles=False)
            sc = self.scores[:, :, :length].contiguous()
            self._select(sc, sub, FULL, stream=stream)
            self.kept.top_idx[:, :, :sub.t.top_cap].copy_(sub.top_idx)
            self.kept.top_count.copy_(sub.top_count)

    def step(self, q, Kc, Vc, W, cache_len: torch.Tensor, new_pos: int, o, lse=None, A=None, scale: float = 0.0,
             stream=None):
        """One decode step for a token already appended at ``new_pos`` (= cache_len - 1)."""
        self._score(Vc, W, A, new_pos, new_pos + 1, stream)
        self._select(self.scores, self.kept, UPDATE, seq_len=cache_len, stream=stream)
        dma_sparse_attn_decode(q, Kc, Vc, self.bias, self.kept, o, self.ws, lse, cache_len, scale, stream=stream)


class PagedDecodeState:
    """Decode-side buffers for a paged KV cache: the key and page score caches, the kept keys of
    the selected pages and the workspace."""

    def __init__(self, B: int, max_pages: int, page_size: int, H: int, Hkv: int, D: int, w: int, window: int,
                 device="cuda", w_head: Optional[torch.Tensor] = None, form: int = BIAS_LOG):
        self.B, self.max_pages, self.page_size, self.H, self.Hkv, self.D = B, max_pages, page_size, H, Hkv, D
        self.w, self.window, self.w_head, self.form = w, window, w_head, form
        f32 = dict(dtype=torch.float32, device=device)
        self.scores = torch.zeros((B, Hkv, max_pages * page_size), **f32)
        self.bias = self.scores if form == BIAS_LOG else torch.zeros_like(self.scores)
        self.page_scores = torch.full((B, Hkv, max_pages), float("-inf"), **f32)
        self.top_cap = max(1, (w // page_size) * page_size)
        self.top_idx = torch.zeros((B, Hkv, self.top_cap), dtype=torch.int32, device=device)
        self.top_count = torch.zeros((B, Hkv), dtype=torch.int32, device=device)
        self.ws = torch.empty((dma_decode_workspace_size(B, H, Hkv, D, self.top_cap, window),), dtype=torch.uint8,
                              device=device)

    def _score(self, V_pages, block_table, W, A, cache_len, key_begin, key_end, stream):
        if self.form == BIAS_LOG:
            dma_score_keys_paged(V_pages, block_table, W, A, self.scores, self.page_scores, cache_len, key_begin,
                                 key_end, stream=stream)
        else:
            dma_score_keys_paged_bias(V_pages, block_table, W, A, self.form, self.scores, self.bias,
                                      self.page_scores, cache_len, key_begin, key_end, stream=stream)

    def full_score(self, V_pages, block_table, W, A=None, cache_len=None, length: Optional[int] = None, stream=None):
        """Scores every key below ``length`` (all of the cache when None) and its page scores."""
        length = self.max_pages * self.page_size if length is None else length
        self._score(V_pages, block_table, W, A, cache_len, 0, length, stream)

    def select(self, cache_len=None, stream=None):
        """The kept pages of every sequence's decode row, from the page scores."""
        if self.w_head is None:
            dma_select_pages(self.page_scores, self.page_size, self.w, self.top_idx, self.top_count, cache_len,
                             stream=stream)
        else:
            dma_select_pages_heads(self.page_scores, self.page_size, self.w, self.w_head, self.top_idx,
                                   self.top_count, cache_len, stream=stream)

    def step(self, q, K_pages, V_pages, block_table, W, cache_len: torch.Tensor, new_pos: int, o, lse=None, A=None,
             scale: float = 0.0, stream=None):
        """One decode step for a token already written at logical position ``new_pos``
        (= cache_len - 1): score it, update its page's score, select the pages, attend."""
        self._score(V_pages, block_table, W, A, cache_len, new_pos, new_pos + 1, stream)
        self.select(cache_len, stream)
        dma_sparse_attn_decode_paged(q, K_pages, V_pages, block_table, self.bias, self.top_idx, self.top_count,
                                     self.window, o, self.ws, lse, cache_len, scale, stream=stream)


# ------------------------------------------------------- NSA-style fusion --

def dma_nsa_compress(K: torch.Tensor, V: torch.Tensor, Kc: torch.Tensor, Vc: torch.Tensor, block_begin: int = 0,
                     block_end: Optional[int] = None, stream=None) -> None:
    """Means of the complete 64-key blocks, written at row 64 beta + 63 of Kc, Vc (shaped like K)."""
    B, S, Hkv, D = K.shape
    block_end = S // NSA_BLOCK if block_end is None else block_end
    _check(_lib.dma_nsa_compress(_ptr(K), _ptr(V), _dtype(K), B, S, Hkv, D, block_begin, block_end, _ptr(Kc),
                                 _ptr(Vc), _stream(stream)))


def dma_nsa_kept_pattern(pattern: int, kept: Kept, seq_len: Optional[torch.Tensor] = None, stream=None) -> None:
    _check(_lib.dma_nsa_kept_pattern(pattern, _ptr(seq_len), ctypes.byref(kept.t), _stream(stream)))


def dma_nsa_combine(Q: torch.Tensor, O_cmp: torch.Tensor, O_slc: torch.Tensor, O_win: torch.Tensor,
                    G: torch.Tensor, c: torch.Tensor, O: torch.Tensor, gates: Optional[torch.Tensor] = None,
                    stream=None) -> None:
    """Q and the outputs [B][S][H][D] ([B][H][D] for decode); G [H][3][D], c [H][3] fp32."""
    if Q.dim() == 3:
        B, H, D = Q.shape
        S = 1
    else:
        B, S, H, D = Q.shape
    _check(_lib.dma_nsa_combine(_ptr(Q), _ptr(O_cmp), _ptr(O_slc), _ptr(O_win), _dtype(Q), B, S, H, D, _ptr(G),
                                _ptr(c), _ptr(O), _ptr(gates), _stream(stream)))


class NsaPrefill:
    """Buffers of the NSA-style three-branch prefill for one shape: the selected branch's
    kept keys (64-key blocks, no window), the two fixed patterns (built once here), the
    compressed K/V arrays, an all-zero bias and the three branch outputs."""

    def __init__(self, B: int, S: int, H: int, Hkv: int, D: int, w: int, window: int, dtype=torch.bfloat16,
                 device="cuda", stream=None):
        self.B, self.S, self.H, self.Hkv, self.D, self.w, self.window = B, S, H, Hkv, D, w, window
        f32 = dict(dtype=torch.float32, device=device)
        self.scores = torch.empty((B, Hkv, S), **f32)
        self.zero = torch.zeros((B, Hkv, S), **f32)
        self.kept_slc = Kept(B, Hkv, S, w, 0, NSA_BLOCK, ROWWISE, device=device)
        self.kept_cmp = Kept(B, Hkv, S, S // NSA_BLOCK, 0, 1, GLOBAL, device=device)
        self.kept_win = Kept(B, Hkv, S, 0, window, 1, ROWWISE, device=device)
        dma_nsa_kept_pattern(NSA_COMPRESSED, self.kept_cmp, stream=stream)
        dma_nsa_kept_pattern(NSA_WINDOW, self.kept_win, stream=stream)
        self.Kc = torch.zeros((B, S, Hkv, D), dtype=dtype, device=device)
        self.Vc = torch.zeros((B, S, Hkv, D), dtype=dtype, device=device)
        self.o_cmp, self.o_slc, self.o_win = (torch.empty((B, S, H, D), dtype=dtype, device=device)
                                              for _ in range(3))

    def run(self, Q, K, V, W, A, G, c, O, gates=None, scale: float = 0.0, stream=None):
        """Score, select (64-key blocks), compress, the three attentions, the gated sum into O."""
        dma_score_keys(V, W, A, self.scores, stream=stream)
        dma_select_topk(self.scores, self.kept_slc, FULL, stream=stream)
        dma_nsa_compress(K, V, self.Kc, self.Vc, stream=stream)
        dma_sparse_attn_prefill(Q, self.Kc, self.Vc, self.zero, self.kept_cmp, self.o_cmp, None, scale, stream=stream)
        dma_sparse_attn_prefill(Q, K, V, self.zero, self.kept_slc, self.o_slc, None, scale, stream=stream)
        dma_sparse_attn_prefill(Q, K, V, self.zero, self.kept_win, self.o_win, None, scale, stream=stream)
        dma_nsa_combine(Q, self.o_cmp, self.o_slc, self.o_win, G, c, O, gates, stream=stream)


class NsaDecode:
    """The NSA-style fusion for one new query row per sequence over caches [B][Lmax][Hkv][D]
    (Lmax a multiple of 64).  The selected branch takes the decode row's 64-key blocks by page
    selection over the contiguous cache viewed as 64-key pages (block table b * Lmax/64 + p),
    the block-unit rule on the last row."""

    def __init__(self, B: int, Lmax: int, H: int, Hkv: int, D: int, w: int, window: int, dtype=torch.bfloat16,
                 device="cuda"):
        if Lmax % NSA_BLOCK:
            raise ValueError("Lmax must be a multiple of 64")
        self.B, self.Lmax, self.H, self.Hkv, self.D, self.w, self.window = B, Lmax, H, Hkv, D, w, window
        f32 = dict(dtype=torch.float32, device=device)
        npg = Lmax // NSA_BLOCK
        self.block_table = torch.arange(B * npg, dtype=torch.int32, device=device).view(B, npg)
        self.scores = torch.zeros((B, Hkv, Lmax), **f32)
        self.page_scores = torch.full((B, Hkv, npg), float("-inf"), **f32)
        self.zero = torch.zeros((B, Hkv, Lmax), **f32)
        self.kept_slc = Kept(B, Hkv, Lmax, w, 0, NSA_BLOCK, ROWWISE, device=device, tiles=False)
        self.kept_cmp = Kept(B, Hkv, Lmax, npg, 0, 1, GLOBAL, device=device, tiles=False)
        self.kept_win = Kept(B, Hkv, Lmax, 0, window, 1, ROWWISE, device=device, tiles=False)
        dma_nsa_kept_pattern(NSA_WINDOW, self.kept_win)
        self.Kc = torch.zeros((B, Lmax, Hkv, D), dtype=dtype, device=device)
        self.Vc = torch.zeros((B, Lmax, Hkv, D), dtype=dtype, device=device)
        cap = max(k.t.top_cap for k in (self.kept_slc, self.kept_cmp, self.kept_win))
        self.ws = torch.empty((dma_decode_workspace_size(B, H, Hkv, D, cap, window),), dtype=torch.uint8,
                              device=device)
        self.o_cmp, self.o_slc, self.o_win = (torch.empty((B, H, D), dtype=dtype, device=device) for _ in range(3))

    def _pages(self, X):
        return X.view(self.B * (self.Lmax // NSA_BLOCK), NSA_BLOCK, self.Hkv, self.D)

    def prepare(self, Kc, Vc, W, cache_len: torch.Tensor, length: int, A=None, stream=None):
        """Scores, block scores and compressed blocks of the caches (keys below cache_len[b]; length
        = the largest cache length), and the compressed branch's kept blocks."""
        dma_score_keys_paged(self._pages(Vc), self.block_table, W, A, self.scores, self.page_scores, cache_len, 0,
                             length, stream=stream)
        dma_nsa_compress(Kc, Vc, self.Kc, self.Vc, 0, length // NSA_BLOCK, stream=stream)
        dma_nsa_kept_pattern(NSA_COMPRESSED, self.kept_cmp, cache_len, stream=stream)

    def step(self, q, Kc, Vc, W, cache_len: torch.Tensor, new_pos: int, G, c, o, A=None, scale: float = 0.0,
             stream=None):
        """One decode step for a token already written at ``new_pos`` (= cache_len - 1): its score
        and block score; when it completes a block, that block's means and the compressed
        branch's kept blocks; then the three branches and the gated sum into o."""
        dma_score_keys_paged(self._pages(Vc), self.block_table, W, A, self.scores, self.page_scores, cache_len,
                             new_pos, new_pos + 1, stream=stream)
        if (new_pos + 1) % NSA_BLOCK == 0:
            beta = new_pos // NSA_BLOCK
            dma_nsa_compress(Kc, Vc, self.Kc, self.Vc, beta, beta + 1, stream=stream)
            dma_nsa_kept_pattern(NSA_COMPRESSED, self.kept_cmp, cache_len, stream=stream)
        self.attend(q, Kc, Vc, cache_len, G, c, o, scale, stream)

    def attend(self, q, Kc, Vc, cache_len, G, c, o, scale: float = 0.0, stream=None):
        """The block selection of the decode row cache_len[b] - 1, the three branches and their
        gated sum."""
        ks = self.kept_slc
        dma_select_pages(self.page_scores, NSA_BLOCK, self.w, ks.top_idx, ks.top_count, cache_len, stream=stream)
        dma_sparse_attn_decode(q, self.Kc, self.Vc, self.zero, self.kept_cmp, self.o_cmp, self.ws, None, cache_len,
                               scale, stream=stream)
        dma_sparse_attn_decode(q, Kc, Vc, self.zero, ks, self.o_slc, self.ws, None, cache_len, scale, stream=stream)
        dma_sparse_attn_decode(q, Kc, Vc, self.zero, self.kept_win, self.o_win, self.ws, None, cache_len, scale,
                               stream=stream)
        dma_nsa_combine(q, self.o_cmp, self.o_slc, self.o_win, G, c, o, stream=stream)
