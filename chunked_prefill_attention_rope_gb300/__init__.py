"""Python binding of libcpa.so: chunked prefill attention with past for GB300.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of libcpa.so; there is no fallback, and every call raises if the
library has not been built.  torch supplies device memory and the current
stream.  The entry points mirror include/cpa.h:

    chunk_prefill_attn   one chunk of C rows against the KV cache
    chunk_prefill_attn_append
                         the same, and the chunk appended to a global cache
    decode_step          the C = 1 case
    kv_append            append the chunk (rotated K, V) to the cache
    kv_snapshot_padded_append / kv_rollback_padded_append
                         make a padded append to a sliding-window cache
                         byte-identical to an unpadded one
    tail_plan            padded chunk or one-token steps for a prompt tail
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "CpaError", "KVCache", "load_library", "lib_path", "using_library", "chunk_prefill_attn", "chunk_prefill_attn_noalloc",
    "decode_step", "chunk_prefill_attn_append",
    "kv_append", "kv_snapshot_padded_append", "kv_rollback_padded_append",
    "PreparedCall", "prepare_chunk_prefill_attn", "prepare_chunk_prefill_attn_append", "prepare_kv_append",
    "attn_workspace_size", "attn_workspace_size_mask", "cache_scratch_size", "new_error_word", "EBIT", "GLOBAL", "SLIDING",
    "tail_plan", "TAIL_SCALAR", "TAIL_PADDED", "TAIL_AUTO", "TAIL_FORCE_SCALAR", "TAIL_FORCE_PADDED",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
GLOBAL, SLIDING = 0, 1
TAIL_SCALAR, TAIL_PADDED = 0, 1
TAIL_AUTO, TAIL_FORCE_SCALAR, TAIL_FORCE_PADDED = 0, 1, 2
EBIT = dict(CAPACITY=1, PAST_GT_SPAN=2, NREAL_GT_C=4, SLIDING_N=8, SNAPSHOT=16, TIMEOUT=32, BOUNDS=64)


class CpaError(RuntimeError):
    """A cpa_status other than CPA_OK."""

    def __init__(self, status: int, text: str):
        super().__init__(f"cpa status {status}: {text}")
        self.status = status


class _Cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("stride_b", ctypes.c_int64),
                ("stride_h", ctypes.c_int64), ("stride_s", ctypes.c_int64), ("len", ctypes.c_void_p),
                ("cap", ctypes.c_int32), ("kind", ctypes.c_int32), ("window", ctypes.c_int32),
                ("sink", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class _AttnArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
                ("C", ctypes.c_int), ("P", ctypes.c_int), ("scale", ctypes.c_float),
                ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("cos", ctypes.c_void_p), ("sin", ctypes.c_void_p), ("cache", ctypes.POINTER(_Cache)),
                ("mask", ctypes.c_void_p), ("past_len", ctypes.c_void_p), ("n_real", ctypes.c_void_p),
                ("window", ctypes.c_int), ("causal", ctypes.c_int), ("sel_row", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("out_sel", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("err", ctypes.c_void_p),
                ("sm_budget", ctypes.c_int)]


_LIBS = {}
_VARIANT = "default"
_LIB_FILES = {"default": "libcpa.so", "checked": "libcpa_checked.so"}


def lib_path(variant: Optional[str] = None) -> str:
    return os.path.join(_HERE, _LIB_FILES[variant or _VARIANT])


@contextlib.contextmanager
def using_library(variant: str):
    """Route the calls inside the block to one build of the library:
    "default" (libcpa.so) or "checked" (libcpa_checked.so, the bounds-checked
    build with its test hooks)."""
    global _VARIANT
    if variant not in _LIB_FILES:
        raise ValueError(f"unknown library variant {variant!r}")
    old = _VARIANT
    _VARIANT = variant
    try:
        yield load_library(variant)
    finally:
        _VARIANT = old


def load_library(variant: Optional[str] = None):
    """Load the library (raises if it is missing: run build() first)."""
    v = variant or _VARIANT
    if v in _LIBS:
        return _LIBS[v]
    path = lib_path(v)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "chunked_prefill_attention_rope_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.cpa_chunk_prefill_attn.argtypes = [ctypes.POINTER(_AttnArgs), vp]
    lib.cpa_decode_step.argtypes = [ctypes.POINTER(_AttnArgs), vp]
    lib.cpa_chunk_prefill_attn_noalloc.argtypes = [ctypes.POINTER(_AttnArgs), vp]
    lib.cpa_chunk_prefill_attn_append.argtypes = [ctypes.POINTER(_AttnArgs), vp, vp]
    lib.cpa_attn_workspace_size.argtypes = [i32] * 6
    lib.cpa_attn_workspace_size.restype = sz
    lib.cpa_attn_workspace_size_mask.argtypes = [i32] * 6
    lib.cpa_attn_workspace_size_mask.restype = sz
    lib.cpa_kv_append.argtypes = [ctypes.POINTER(_Cache), vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, sz, vp, vp]
    lib.cpa_cache_scratch_size.argtypes = [ctypes.POINTER(_Cache), i32, i32, i32, i32]
    lib.cpa_cache_scratch_size.restype = sz
    lib.cpa_kv_snapshot_padded_append.argtypes = [ctypes.POINTER(_Cache), vp, i32, i32, i32, i32, vp, sz, vp, vp]
    lib.cpa_kv_rollback_padded_append.argtypes = [ctypes.POINTER(_Cache), i32, i32, i32, i32, vp, sz, vp, vp]
    lib.cpa_tail_plan.argtypes = [i32, i32, i32, i32, vp, i32, i32, i32, vp, vp]
    lib.cpa_status_str.argtypes = [i32]
    lib.cpa_status_str.restype = ctypes.c_char_p
    lib.cpa_version.restype = ctypes.c_char_p
    for f in ("cpa_chunk_prefill_attn", "cpa_decode_step", "cpa_chunk_prefill_attn_noalloc",
              "cpa_chunk_prefill_attn_append", "cpa_kv_append",
              "cpa_kv_snapshot_padded_append", "cpa_kv_rollback_padded_append", "cpa_tail_plan"):
        getattr(lib, f).restype = i32
    if v == "checked":
        lib.cpa_test_drop_tile.argtypes = [i32]
        lib.cpa_test_drop_tile.restype = None
    _LIBS[v] = lib
    return lib


def _check(status: int):
    if status != 0:
        raise CpaError(status, load_library().cpa_status_str(status).decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device: torch.device) -> Optional[int]:
    """The cudaStream_t of `stream`, or of torch's current stream on `device`."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(device.index if device.index is not None else torch.cuda.current_device())
        return torch.cuda.current_stream(device).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def new_error_word(device="cuda") -> torch.Tensor:
    """A zeroed device int32 word for the library's CPA_EBIT_* flags."""
    return torch.zeros(4, dtype=torch.int32, device=device)


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if t.dtype is not dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


class KVCache:
    """One layer's KV cache: k, v bf16 or fp16 [B, Hkv, cap, D] (strided views
    allowed, last dim contiguous), len int32 [B] on the device, and its kind."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor, length: torch.Tensor, kind: int = GLOBAL,
                 window: int = 0, sink: int = 0):
        if k.dtype not in (torch.bfloat16, torch.float16) or v.dtype != k.dtype:
            raise TypeError("cache k/v must both be bf16 or both fp16")
        if k.shape != v.shape or k.stride() != v.stride() or k.dim() != 4 or k.stride(3) != 1:
            raise ValueError("cache k/v: same [B, Hkv, cap, D] shape and strides, last dim contiguous")
        _need(length, "len", torch.int32, (k.shape[0],))
        self.k, self.v, self.len = k, v, length
        self.kind, self.window, self.sink = kind, window, sink
        self.B, self.Hkv, self.cap, self.D = k.shape
        # the C struct is built once: a KVCache describes fixed tensors
        self._struct = _Cache(k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1), k.stride(2), length.data_ptr(),
                              self.cap, kind, window, sink, 1 if k.dtype == torch.float16 else 0)
        self._ref = ctypes.byref(self._struct)

    def struct(self) -> _Cache:
        return self._struct


def attn_workspace_size(B, Hq, Hkv, D, C, P) -> int:
    return int(load_library().cpa_attn_workspace_size(B, Hq, Hkv, D, C, P))


def attn_workspace_size_mask(B, Hq, Hkv, D, C, P) -> int:
    """Workspace for a call with an explicit mask (room for the mask's bit copy)."""
    return int(load_library().cpa_attn_workspace_size_mask(B, Hq, Hkv, D, C, P))


def cache_scratch_size(cache: KVCache, C: int) -> int:
    return int(load_library().cpa_cache_scratch_size(cache._ref, cache.B, cache.Hkv, cache.D, C))


class PreparedCall:
    """One library call whose arguments were checked and marshalled once.
    Calling it enqueues the call again on the same tensors, whose contents may
    change between calls but which must stay where they are; it returns the
    call's outputs.  For drivers that keep their buffers in place (a model's
    layer loop run eagerly): a call then costs the C entry point alone."""

    __slots__ = ("_fn", "_args", "_dev", "_keep", "outputs")

    def __init__(self, fn, args, dev, keep, outputs):
        self._fn, self._args, self._dev, self._keep, self.outputs = fn, args, dev, keep, outputs

    def __call__(self, stream=None):
        _check(self._fn(*self._args, _stream(stream, self._dev)))
        return self.outputs


def _attn_build(entry: str, q, k_new, v_new, cos, sin, cache: KVCache, P: int, past_len=None, n_real=None,
                window: int = 0, causal: bool = True, mask=None, scale: float = 0.0, sel_row=None,
                out=None, out_sel=None, want_sel: bool = False, workspace=None, err=None,
                alloc_workspace: bool = True, append_rows=None, sm_budget: int = 0):
    """Checks the arguments of an attention entry point and marshals them:
    (function, leading C arguments, device, tensors to keep alive, outputs)."""
    lib = load_library()
    B, Hq, C, D = q.shape
    Hkv = k_new.shape[1]
    dev = q.device
    bf16, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    kv_shape, tab_shape, row_shape = (B, Hkv, C, D), (B, C, D), (B,)
    _need(q, "q", bf16)
    _need(k_new, "k_new", bf16, kv_shape)
    _need(v_new, "v_new", bf16, kv_shape)
    _need(cos, "cos", f32, tab_shape)
    _need(sin, "sin", f32, tab_shape)
    if mask is not None:
        _need(mask, "mask", f32, (B, Hq, C, P + C))
    if past_len is not None:
        _need(past_len, "past_len", i32, row_shape)
    if n_real is not None:
        _need(n_real, "n_real", i32, row_shape)
    if sel_row is not None:
        _need(sel_row, "sel_row", i32, row_shape)
    if out is None:
        out = torch.empty((B, Hq, C, D), dtype=bf16, device=dev)
    else:
        _need(out, "out", bf16, q.shape)
    if out_sel is None and want_sel:
        out_sel = torch.empty((B, Hq * D), dtype=f32, device=dev)
    if workspace is None and alloc_workspace:
        size = lib.cpa_attn_workspace_size_mask if mask is not None else lib.cpa_attn_workspace_size
        need = size(B, Hq, Hkv, D, C, P)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if err is None:
        err = new_error_word(dev)
    a = _AttnArgs(B, Hq, Hkv, D, C, P, float(scale), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                  cos.data_ptr(), sin.data_ptr(), ctypes.pointer(cache._struct),
                  None if mask is None else mask.data_ptr(), None if past_len is None else past_len.data_ptr(),
                  None if n_real is None else n_real.data_ptr(), int(window), 1 if causal else 0,
                  None if sel_row is None else sel_row.data_ptr(), out.data_ptr(),
                  None if out_sel is None else out_sel.data_ptr(),
                  None if workspace is None else workspace.data_ptr(),
                  0 if workspace is None else workspace.numel(), err.data_ptr(), int(sm_budget))
    args = (ctypes.byref(a),)
    if append_rows is not None:
        _need(append_rows, "n_rows", i32, row_shape)
        args = (ctypes.byref(a), append_rows.data_ptr())
    keep = (a, cache, q, k_new, v_new, cos, sin, mask, past_len, n_real, sel_row, workspace, err, append_rows)
    return getattr(lib, entry), args, dev, keep, (out, out_sel)


def _attn(entry: str, *a, stream=None, **kw):
    fn, args, dev, _keep, outs = _attn_build(entry, *a, **kw)
    _check(fn(*args, _stream(stream, dev)))
    return outs


def prepare_chunk_prefill_attn(q, k_new, v_new, cos, sin, cache: KVCache, P: int, **kw) -> PreparedCall:
    """chunk_prefill_attn with its arguments bound once: calling the result
    runs the call again and returns (out, out_sel)."""
    return PreparedCall(*_attn_build("cpa_chunk_prefill_attn", q, k_new, v_new, cos, sin, cache, P, **kw))


def prepare_chunk_prefill_attn_append(q, k_new, v_new, cos, sin, cache: KVCache, P: int, n_rows,
                                      **kw) -> PreparedCall:
    """chunk_prefill_attn_append with its arguments bound once."""
    return PreparedCall(*_attn_build("cpa_chunk_prefill_attn_append", q, k_new, v_new, cos, sin, cache, P,
                                     append_rows=n_rows, **kw))


def chunk_prefill_attn(q, k_new, v_new, cos, sin, cache: KVCache, P: int, **kw):
    """Attention of one chunk (q [B,Hq,C,D], k_new/v_new [B,Hkv,C,D] bf16, cos/sin
    [B,C,D] fp32) over cache slots [0, P) plus the chunk.  Returns (out, out_sel)."""
    return _attn("cpa_chunk_prefill_attn", q, k_new, v_new, cos, sin, cache, P, **kw)


def chunk_prefill_attn_noalloc(q, k_new, v_new, cos, sin, cache: KVCache, P: int, **kw):
    """chunk_prefill_attn without a caller workspace: for callers that cannot
    allocate device memory (graph capture, statically planned runtimes,
    framework plugins).  Split-KV partials use the library's fixed 16 MiB
    array; sizes needing more raise CpaError (CPA_ERR_WORKSPACE)."""
    kw["workspace"] = None
    return _attn("cpa_chunk_prefill_attn_noalloc", q, k_new, v_new, cos, sin, cache, P,
                 alloc_workspace=False, **kw)


def chunk_prefill_attn_append(q, k_new, v_new, cos, sin, cache: KVCache, P: int, n_rows, **kw):
    """chunk_prefill_attn then kv_append(cache, k_new, v_new, cos, sin, n_rows) in one
    call (cpa_chunk_prefill_attn_append): the RoPE pre-pass writes the new cache rows,
    len advances after the attention.  GLOBAL caches only."""
    return _attn("cpa_chunk_prefill_attn_append", q, k_new, v_new, cos, sin, cache, P, append_rows=n_rows, **kw)


def decode_step(q, k_new, v_new, cos, sin, cache: KVCache, P: int, **kw):
    """One-token decode (C = 1).  Returns (out, out_sel)."""
    kw.setdefault("causal", False)
    return _attn("cpa_decode_step", q, k_new, v_new, cos, sin, cache, P, **kw)


def kv_append(cache: KVCache, k_new, v_new, cos, sin, n_rows, scratch=None, err=None, stream=None):
    """Append rows [0, n_rows[b]) of the chunk (K rotated, V copied) to the cache."""
    fn, args, dev, _keep, err = _append_build(cache, k_new, v_new, cos, sin, n_rows, scratch, err)
    _check(fn(*args, _stream(stream, dev)))
    return err


def prepare_kv_append(cache: KVCache, k_new, v_new, cos, sin, n_rows, scratch=None, err=None) -> PreparedCall:
    """kv_append with its arguments bound once: calling the result runs the
    append again (the cache's length advances each time) and returns err."""
    return PreparedCall(*_append_build(cache, k_new, v_new, cos, sin, n_rows, scratch, err))


def _append_build(cache: KVCache, k_new, v_new, cos, sin, n_rows, scratch, err):
    lib = load_library()
    B, Hkv, C, D = k_new.shape
    kv_shape, tab_shape = (B, Hkv, C, D), (B, C, D)
    _need(k_new, "k_new", torch.bfloat16)
    _need(v_new, "v_new", torch.bfloat16, kv_shape)
    _need(cos, "cos", torch.float32, tab_shape)
    _need(sin, "sin", torch.float32, tab_shape)
    _need(n_rows, "n_rows", torch.int32, (B,))
    dev = k_new.device
    if err is None:
        err = new_error_word(dev)
    if scratch is None and cache.kind == SLIDING:
        scratch = torch.empty(cache_scratch_size(cache, C), dtype=torch.uint8, device=dev)
    args = (cache._ref, k_new.data_ptr(), v_new.data_ptr(), cos.data_ptr(), sin.data_ptr(), n_rows.data_ptr(),
            B, Hkv, D, C, None if scratch is None else scratch.data_ptr(), 0 if scratch is None else scratch.numel(),
            err.data_ptr())
    return lib.cpa_kv_append, args, dev, (cache, k_new, v_new, cos, sin, n_rows, scratch, err), err


def kv_snapshot_padded_append(cache: KVCache, n_real, C: int, scratch, err=None, stream=None):
    """Save the rows a padded append of C rows would over-evict (sliding caches)."""
    lib = load_library()
    _need(n_real, "n_real", torch.int32, (cache.B,))
    if err is None:
        err = new_error_word(n_real.device)
    _check(lib.cpa_kv_snapshot_padded_append(cache._ref, n_real.data_ptr(), cache.B, cache.Hkv,
                                             cache.D, C, scratch.data_ptr(), scratch.numel(),
                                             err.data_ptr(), _stream(stream, n_real.device)))
    return err


def kv_rollback_padded_append(cache: KVCache, C: int, scratch, err=None, stream=None):
    """Drop the pad rows and reinsert the saved rows after a padded append."""
    lib = load_library()
    if err is None:
        err = new_error_word(cache.len.device)
    _check(lib.cpa_kv_rollback_padded_append(cache._ref, cache.B, cache.Hkv, cache.D, C,
                                             scratch.data_ptr(), scratch.numel(), err.data_ptr(),
                                             _stream(stream, cache.len.device)))
    return err


def tail_plan(t: int, C: int, window: int = 0, sink: int = 0, buckets=None, crossover: int = 0,
              force: int = TAIL_AUTO):
    """(mode, c_pad) for a prompt tail of t real tokens: TAIL_SCALAR with c_pad = t,
    or TAIL_PADDED with the chunk rows to pad to (cpa_tail_plan)."""
    lib = load_library()
    arr = None
    n = 0
    if buckets:
        n = len(buckets)
        arr = (ctypes.c_int32 * n)(*buckets)
    mode, c_pad = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.cpa_tail_plan(t, C, window, sink, arr, n, crossover, force, ctypes.byref(mode), ctypes.byref(c_pad)))
    return mode.value, c_pad.value
