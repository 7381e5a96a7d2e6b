"""Thin Python binding of the IndexCache C ABI (``include/indexcache.h``).

Argument marshalling only: shapes and device pointers are read from torch
tensors and handed to ``libindexcache.so``; every step of the computation
runs in the library's CUDA kernels.  There is no CPU path: tensors must live
on a CUDA device, and a missing library raises at load time.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libindexcache.so")

IC_OK, IC_ERR_PATTERN, IC_ERR_ARG, IC_ERR_UNSUPPORTED, IC_ERR_CUDA, IC_ERR_DEVICE_TIMEOUT = range(6)
IC_BF16, IC_E4M3 = 0, 1

EXPORTED = ("ic_workspace_size", "ic_indexer_topk", "ic_sparse_attn", "ic_forward_pattern",
            "ic_forward_pattern_traced", "ic_trace_create", "ic_trace_destroy", "ic_trace_read",
            "ic_stream_status", "ic_last_error", "ic_abi_version", "ic_indexer_topk_noalloc",
            "ic_overlap", "ic_greedy_full_layers", "ic_debug_set_wait_limit_ns", "ic_decode_append",
            "ic_indexer_topk_fp8")


class IndexCacheError(RuntimeError):
    """A CUDA-side failure reported by the library."""


class DeviceTimeoutError(IndexCacheError):
    """A bounded device-side wait gave up (IC_ERR_DEVICE_TIMEOUT)."""


class PatternError(ValueError):
    """The F/S pattern was refused (IC_ERR_PATTERN)."""


class UnsupportedError(ValueError):
    """Sizes outside what the kernels cover (IC_ERR_UNSUPPORTED)."""


class ICDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("S", ctypes.c_int), ("S_cap", ctypes.c_int),
                ("H", ctypes.c_int), ("D", ctypes.c_int), ("k", ctypes.c_int), ("q_pos0", ctypes.c_int),
                ("k_dtype", ctypes.c_int), ("Hq", ctypes.c_int), ("Dh", ctypes.c_int), ("scale", ctypes.c_float)]


class ICLayer(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("kI", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("w", ctypes.c_void_p), ("Q", ctypes.c_void_p), ("K", ctypes.c_void_p),
                ("V", ctypes.c_void_p), ("O", ctypes.c_void_p)]


class ICAppendSrc(ctypes.Structure):
    _fields_ = [("kI", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("K", ctypes.c_void_p), ("V", ctypes.c_void_p)]


# double (*)(const char* pattern, void* user)
LOSS_FN = ctypes.CFUNCTYPE(ctypes.c_double, ctypes.c_char_p, ctypes.c_void_p)

_lib = None


def load(path: str = LIB_PATH):
    """Load the library once and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libindexcache.so is not built (run `python -m cross_layer_top_indexer_b300.build`)")
    lib = ctypes.CDLL(path)
    vp, i, sz, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    lib.ic_workspace_size.argtypes = [ctypes.POINTER(ICDims)]
    lib.ic_workspace_size.restype = sz
    lib.ic_indexer_topk.argtypes = [i, i, i, i, i, i, i, i, vp, vp, i, vp, vp, vp, vp, sz, vp]
    lib.ic_indexer_topk.restype = i
    lib.ic_indexer_topk_noalloc.argtypes = [i, i, i, i, i, i, i, i, vp, vp, i, vp, vp, vp, vp]
    lib.ic_indexer_topk_fp8.argtypes = [i, i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp]
    lib.ic_indexer_topk_fp8.restype = i
    lib.ic_indexer_topk_noalloc.restype = i
    lib.ic_sparse_attn.argtypes = [i, i, i, i, i, i, i, vp, vp, vp, vp, f, vp, vp, sz, vp]
    lib.ic_sparse_attn.restype = i
    lib.ic_forward_pattern.argtypes = [ctypes.c_char_p, i, ctypes.POINTER(ICLayer), ctypes.POINTER(ICDims), vp,
                                       ctypes.POINTER(i), vp, sz, vp]
    lib.ic_forward_pattern.restype = i
    lib.ic_forward_pattern_traced.argtypes = lib.ic_forward_pattern.argtypes + [vp]
    lib.ic_forward_pattern_traced.restype = i
    lib.ic_trace_create.argtypes = [i, i, ctypes.POINTER(vp)]
    lib.ic_trace_create.restype = i
    lib.ic_trace_destroy.argtypes = [vp]
    lib.ic_trace_destroy.restype = i
    lib.ic_trace_read.argtypes = [vp, ctypes.POINTER(i), ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]
    lib.ic_trace_read.restype = i
    lib.ic_stream_status.argtypes = [vp]
    lib.ic_stream_status.restype = i
    lib.ic_last_error.argtypes = []
    lib.ic_last_error.restype = ctypes.c_char_p
    lib.ic_abi_version.argtypes = []
    lib.ic_abi_version.restype = i
    lib.ic_debug_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.ic_debug_set_wait_limit_ns.restype = i
    lib.ic_decode_append.argtypes = [ctypes.c_char_p, i, ctypes.POINTER(ICLayer), ctypes.POINTER(ICAppendSrc),
                                     ctypes.POINTER(ICDims), i, vp]
    lib.ic_decode_append.restype = i
    lib.ic_overlap.argtypes = [i, i, vp, vp, vp, vp, vp]
    lib.ic_overlap.restype = i
    lib.ic_greedy_full_layers.argtypes = [i, i, LOSS_FN, vp, ctypes.c_char_p, ctypes.POINTER(ctypes.c_longlong)]
    lib.ic_greedy_full_layers.restype = i
    _lib = lib
    return lib


def _raise(code: int):
    if code == IC_OK:
        return
    msg = load().ic_last_error().decode(errors="replace")
    if code == IC_ERR_PATTERN:
        raise PatternError(msg)
    if code == IC_ERR_ARG:
        raise ValueError(msg)
    if code == IC_ERR_UNSUPPORTED:
        raise UnsupportedError(msg)
    if code == IC_ERR_DEVICE_TIMEOUT:
        raise DeviceTimeoutError(msg)
    raise IndexCacheError("%s (status %d)" % (msg, code))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device (this library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _kdtype(kI: torch.Tensor) -> int:
    if kI.dtype == torch.bfloat16:
        return IC_BF16
    if kI.dtype in (torch.float8_e4m3fn, torch.uint8):
        return IC_E4M3
    raise ValueError("kI must be bf16 or e4m3 (float8_e4m3fn / uint8 bytes)")


def make_dims(B, T, S, H, D, k, Hq, Dh, q_pos0=0, k_dtype=IC_BF16, S_cap=0, scale=0.0) -> ICDims:
    return ICDims(B, T, S, S_cap, H, D, k, q_pos0, k_dtype, Hq, Dh, float(scale))


def workspace_size(dims: ICDims) -> int:
    n = load().ic_workspace_size(ctypes.byref(dims))
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid dims")
    return n


def _workspace(nbytes: int, ws: Optional[torch.Tensor], device) -> tuple:
    if nbytes == 0:
        return (None if ws is None else ws.data_ptr()), (0 if ws is None else ws.numel() * ws.element_size())
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return ws.data_ptr(), ws.numel() * ws.element_size()


def indexer_topk(q: torch.Tensor, kI: torch.Tensor, w: torch.Tensor, k: int, q_pos0: int = 0,
                 kscale: Optional[torch.Tensor] = None, S: Optional[int] = None,
                 idx_out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None):
    """ic_indexer_topk: q [B,T,H,D] bf16, kI [B,S_cap,D] bf16/e4m3, w [B,T,H] fp32 -> idx [B,T,k] int32."""
    lib = load()
    B, T, H, D = q.shape
    S_cap = kI.shape[1]
    S = q_pos0 + T if S is None else S
    if idx_out is None:
        idx_out = torch.empty((B, T, k), dtype=torch.int32, device=q.device)
    dims = make_dims(B, T, S, H, D, k, 1, 64, q_pos0, _kdtype(kI), S_cap)
    wsp, wsb = _workspace(workspace_size(dims), ws, q.device)
    code = lib.ic_indexer_topk(B, T, S, S_cap, H, D, k, q_pos0, _ptr(q), _ptr(kI), _kdtype(kI), _ptr(kscale),
                               _ptr(w), _ptr(idx_out), wsp, wsb, _stream(stream))
    _raise(code)
    return idx_out


def indexer_topk_fp8(q8: torch.Tensor, q_scale: torch.Tensor, kI: torch.Tensor, kscale: torch.Tensor,
                     w: torch.Tensor, k: int, q_pos0: int = 0, S: Optional[int] = None,
                     idx_out: Optional[torch.Tensor] = None, stream=None):
    """ic_indexer_topk_fp8: q8 [B,T,H,D] e4m3, q_scale [B,T,H], kI [B,S_cap,D] e4m3, kscale [B,S_cap]."""
    lib = load()
    B, T, H, D = q8.shape
    S_cap = kI.shape[1]
    S = q_pos0 + T if S is None else S
    if idx_out is None:
        idx_out = torch.empty((B, T, k), dtype=torch.int32, device=q8.device)
    code = lib.ic_indexer_topk_fp8(B, T, S, S_cap, H, D, k, q_pos0, _ptr(q8), _ptr(q_scale), _ptr(kI), _ptr(kscale),
                                   _ptr(w), _ptr(idx_out), _stream(stream))
    _raise(code)
    return idx_out


def indexer_topk_noalloc(q: torch.Tensor, kI: torch.Tensor, w: torch.Tensor, k: int, q_pos0: int = 0,
                         kscale: Optional[torch.Tensor] = None, S: Optional[int] = None,
                         idx_out: Optional[torch.Tensor] = None, stream=None):
    """ic_indexer_topk_noalloc: the few-rows indexer with no workspace (scratch
    is a fixed device array inside the library)."""
    lib = load()
    B, T, H, D = q.shape
    S_cap = kI.shape[1]
    S = q_pos0 + T if S is None else S
    if idx_out is None:
        idx_out = torch.empty((B, T, k), dtype=torch.int32, device=q.device)
    code = lib.ic_indexer_topk_noalloc(B, T, S, S_cap, H, D, k, q_pos0, _ptr(q), _ptr(kI), _kdtype(kI),
                                       _ptr(kscale), _ptr(w), _ptr(idx_out), _stream(stream))
    _raise(code)
    return idx_out


def sparse_attn(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, idx: torch.Tensor, scale: float = 0.0,
                S: Optional[int] = None, O: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                stream=None):
    """ic_sparse_attn: Q [B,T,Hq,Dh], K/V [B,S_cap,Dh] bf16, idx [B,T,k] int32 -> O [B,T,Hq,Dh] bf16."""
    lib = load()
    B, T, Hq, Dh = Q.shape
    S_cap = K.shape[1]
    S = S_cap if S is None else S
    k = idx.shape[-1]
    if O is None:
        O = torch.empty_like(Q)
    dims = make_dims(B, T, S, 1, 32, k, Hq, Dh, 0, IC_BF16, S_cap, scale)
    wsp, wsb = _workspace(workspace_size(dims), ws, Q.device)
    code = lib.ic_sparse_attn(B, T, S, S_cap, Hq, Dh, k, _ptr(Q), _ptr(K), _ptr(V), _ptr(idx), float(scale),
                              _ptr(O), wsp, wsb, _stream(stream))
    _raise(code)
    return O


class Trace:
    """Per-layer CUDA-event timing of traced forwards (ic_trace_*)."""

    def __init__(self, n_layers: int, max_forwards: int):
        self.n_layers = n_layers
        h = ctypes.c_void_p()
        _raise(load().ic_trace_create(n_layers, max_forwards, ctypes.byref(h)))
        self.handle = h

    def read(self):
        """(n_forwards, indexer_ms[n_layers], attn_ms[n_layers]) summed over the traced forwards."""
        n = ctypes.c_int(0)
        a = (ctypes.c_float * self.n_layers)()
        b = (ctypes.c_float * self.n_layers)()
        _raise(load().ic_trace_read(self.handle, ctypes.byref(n), a, b))
        return n.value, list(a), list(b)

    def close(self):
        if self.handle:
            load().ic_trace_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Forward:
    """A prepared F/S forward: marshals the layer table once, then each call
    is a single ic_forward_pattern (or traced) launch sequence."""

    def __init__(self, pattern: str, layers: Sequence[dict], k: int, q_pos0: int = 0, S: Optional[int] = None,
                 index_cache: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                 scale: float = 0.0, alloc_outputs: bool = True):
        load()
        n = len(layers)
        Q0 = layers[0]["Q"]
        B_, T, Hq, Dh = Q0.shape
        S_cap = layers[0]["K"].shape[1]
        S = q_pos0 + T if S is None else S
        f0 = next((L for L, c in zip(layers, pattern) if c == "F" and L.get("q") is not None), None)
        H, D, kd = (f0["q"].shape[2], f0["q"].shape[3], _kdtype(f0["kI"])) if f0 is not None else (1, 32, IC_BF16)
        self.dims = make_dims(B_, T, S, H, D, k, Hq, Dh, q_pos0, kd, S_cap, scale)
        self.arr = (ICLayer * n)()
        for l, L in enumerate(layers):
            if alloc_outputs and L.get("O") is None:
                L["O"] = torch.empty_like(L["Q"])
            self.arr[l] = ICLayer(_ptr(L.get("q")), _ptr(L.get("kI")), _ptr(L.get("kscale")), _ptr(L.get("w")),
                                  _ptr(L["Q"]), _ptr(L["K"]), _ptr(L["V"]), _ptr(L.get("O")))
        self.layers = layers
        self.n = n
        self.pattern = pattern.encode() if isinstance(pattern, str) else pattern
        self.index_cache = index_cache if index_cache is not None else \
            torch.empty((B_, T, k), dtype=torch.int32, device=Q0.device)
        need = workspace_size(self.dims)
        self.ws = ws if (ws is not None or need == 0) else torch.empty(need, dtype=torch.uint8, device=Q0.device)
        self.wsp = None if self.ws is None else self.ws.data_ptr()
        self.wsb = 0 if self.ws is None else self.ws.numel() * self.ws.element_size()

    def __call__(self, stream=None, trace: Optional[Trace] = None) -> int:
        calls = ctypes.c_int(0)
        args = (self.pattern, self.n, self.arr, ctypes.byref(self.dims), _ptr(self.index_cache),
                ctypes.byref(calls), self.wsp, self.wsb, _stream(stream))
        if trace is None:
            code = load().ic_forward_pattern(*args)
        else:
            code = load().ic_forward_pattern_traced(*args, trace.handle)
        _raise(code)
        return calls.value


def forward_pattern(pattern: str, layers: Sequence[dict], k: int, q_pos0: int = 0, S: Optional[int] = None,
                    index_cache: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                    scale: float = 0.0, stream=None, alloc_outputs: bool = True):
    """ic_forward_pattern over ``layers`` (dicts of q, kI, kscale, w, Q, K, V, O tensors).

    Returns (index_cache, indexer_calls).  Missing ``O`` entries are allocated
    when ``alloc_outputs`` is true.
    """
    lib = load()
    n = len(layers)
    Q0 = layers[0]["Q"]
    B, T, Hq, Dh = Q0.shape
    S_cap = layers[0]["K"].shape[1]
    S = q_pos0 + T if S is None else S
    f0 = next((L for L, c in zip(layers, pattern) if c == "F" and L.get("q") is not None), None)
    H, D, kd = (f0["q"].shape[2], f0["q"].shape[3], _kdtype(f0["kI"])) if f0 is not None else (1, 32, IC_BF16)
    dims = make_dims(B, T, S, H, D, k, Hq, Dh, q_pos0, kd, S_cap, scale)
    arr = (ICLayer * n)()
    for l, L in enumerate(layers):
        if alloc_outputs and L.get("O") is None:
            L["O"] = torch.empty_like(L["Q"])
        arr[l] = ICLayer(_ptr(L.get("q")), _ptr(L.get("kI")), _ptr(L.get("kscale")), _ptr(L.get("w")),
                         _ptr(L["Q"]), _ptr(L["K"]), _ptr(L["V"]), _ptr(L.get("O")))
    if index_cache is None:
        index_cache = torch.empty((B, T, k), dtype=torch.int32, device=Q0.device)
    need = workspace_size(dims)
    wsp, wsb = _workspace(need, ws, Q0.device)
    calls = ctypes.c_int(0)
    code = lib.ic_forward_pattern(pattern.encode() if isinstance(pattern, str) else pattern, n, arr,
                                  ctypes.byref(dims), _ptr(index_cache), ctypes.byref(calls), wsp, wsb,
                                  _stream(stream))
    _raise(code)
    return index_cache, calls.value


def overlap(idx_a: torch.Tensor, idx_b: torch.Tensor, k: Optional[int] = None, counts: bool = False,
            stream=None):
    """ic_overlap: per-row |I_a ∩ I_b| / k of two index tensors [..., k] int32.

    Returns the fp32 ratios (shape of the leading axes), and the int32 counts
    too when ``counts`` is true."""
    lib = load()
    if idx_a.shape != idx_b.shape or idx_a.dtype != torch.int32 or idx_b.dtype != torch.int32:
        raise ValueError("idx_a and idx_b must be int32 tensors of one shape")
    k = idx_a.shape[-1] if k is None else k
    R = idx_a.numel() // idx_a.shape[-1]
    ratio = torch.empty(idx_a.shape[:-1], dtype=torch.float32, device=idx_a.device)
    cnt = torch.empty(idx_a.shape[:-1], dtype=torch.int32, device=idx_a.device) if counts else None
    _raise(lib.ic_overlap(R, k, _ptr(idx_a), _ptr(idx_b), _ptr(ratio), _ptr(cnt), _stream(stream)))
    return (ratio, cnt) if counts else ratio


def greedy_full_layers(n_layers: int, removals: int, evaluate_loss) -> tuple:
    """ic_greedy_full_layers with a Python loss: ``evaluate_loss(pattern: str)
    -> float`` runs the caller's model under the pattern.  Returns (pattern,
    number of loss evaluations).  An exception in the loss stops the search
    and is re-raised."""
    lib = load()
    failure = []

    def cb(pat, _user):
        try:
            return float(evaluate_loss(pat.decode()))
        except BaseException as ex:  # reported after the C call returns
            failure.append(ex)
            return float("nan")

    fn = LOSS_FN(cb)
    out = ctypes.create_string_buffer(max(n_layers, 0) + 1)
    fw = ctypes.c_longlong(0)
    code = lib.ic_greedy_full_layers(int(n_layers), int(removals), fn, None, out, ctypes.byref(fw))
    if failure:
        raise failure[0]
    _raise(code)
    return out.value.decode(), fw.value


class DecodeAppend:
    """ic_decode_append prepared once: ``caches`` are the stack's layer dicts
    (kI, kscale, K, V, ...), ``new_rows`` per-layer dicts of the new token's
    rows (kI [B,D], kscale [B], K [B,Dh], V [B,Dh]).  Each call appends them
    at row ``pos`` of every sequence, in one launch."""

    def __init__(self, pattern: str, caches: Sequence[dict], new_rows: Sequence[dict], k_dtype: int):
        load()
        n = len(caches)
        self.pattern = pattern.encode() if isinstance(pattern, str) else pattern
        self.n = n
        self.arr = (ICLayer * n)()
        self.src = (ICAppendSrc * n)()
        for l, (L, R) in enumerate(zip(caches, new_rows)):
            self.arr[l] = ICLayer(_ptr(L.get("q")), _ptr(L.get("kI")), _ptr(L.get("kscale")), _ptr(L.get("w")),
                                  _ptr(L["Q"]), _ptr(L["K"]), _ptr(L["V"]), _ptr(L.get("O")))
            self.src[l] = ICAppendSrc(_ptr(R.get("kI")), _ptr(R.get("kscale")), _ptr(R["K"]), _ptr(R["V"]))
        K0 = caches[0]["K"]
        f0 = next((L for L, c in zip(caches, pattern) if c == "F"), caches[0])
        D = f0["kI"].shape[-1] if f0.get("kI") is not None else 32
        self.dims = make_dims(K0.shape[0], 1, K0.shape[1], 1, D, 1, 1, K0.shape[-1], 0, k_dtype, K0.shape[1])
        self._keep = (caches, new_rows)

    def __call__(self, pos: int, stream=None) -> None:
        _raise(load().ic_decode_append(self.pattern, self.n, self.arr, self.src, ctypes.byref(self.dims), int(pos),
                                       _stream(stream)))


def stream_status(stream=None) -> None:
    """Wait for the stream and raise if a bounded device wait gave up."""
    _raise(load().ic_stream_status(_stream(stream)))
