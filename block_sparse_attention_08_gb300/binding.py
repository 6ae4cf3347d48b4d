"""Thin ctypes binding of libmsa (include/msa.h).

Argument marshalling only: shapes, dtypes and devices are checked, raw
pointers and the current CUDA stream are passed to the C ABI, and a non-OK
status raises :class:`MsaError`.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback path.  Output and workspace
tensors are allocated with torch when the caller does not pass them.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import _build

H, G, D, DI, BLOCK = 64, 4, 128, 128, 128
MSA_ERR_CUDA = 6  # msa_status for a failed CUDA call
MODE_DECODE, MODE_PREFILL, MODE_PACK, MODE_PREFILL_BWD = 0, 1, 2, 3
INDEX_DTYPES = {"bf16": 0, "e4m3": 1}
DEVICE_ERRORS = {0: "none", 1: "page id outside the pool", 2: "block id outside the query's range",
                 3: "sequence length out of range", 4: "bounded on-chip wait gave up",
                 5: "prefill attention score outside the fixed-reference range"}


class MsaError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: {text} (status {status})")
        self.status = status
        self.bad_index = -1


class msa_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_q_heads", "num_kv_heads", "head_dim", "num_index_heads", "index_dim", "block_size",
        "topk", "init_blocks", "local_blocks", "index_dtype")]


_lib = None
_lock = threading.Lock()
P, I, I64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
CFG = ctypes.POINTER(msa_config)
_SIGS = {
    "msa_config_default": [CFG],
    "msa_config_check": [CFG],
    "msa_workspace_size": [CFG, I, I64, I, ctypes.POINTER(SZ)],
    "msa_workspace_init": [P, SZ, P],
    "msa_read_device_error": [P, P, ctypes.POINTER(I), ctypes.POINTER(I64)],
    "msa_select_blocks_decode": [CFG, P, P, P, P, P, I, I, I64, P, P, SZ, P],
    "msa_sparse_attend_decode": [CFG, P, P, P, P, P, P, P, I, I, I64, F, P, P, SZ, P],
    "msa_sparse_attend_decode_mxfp8": [CFG, P, P, P, P, P, P, P, I, I, I64, F, P, P, P, SZ, P],
    "msa_sparse_attend_decode_fp8kv": [CFG, P, P, P, F, F, P, P, P, P, I, I, I64, F, P, P, SZ, P],
    "msa_select_blocks_prefill": [CFG, P, P, P, I, I64, I, P, P, SZ, P],
    "msa_sparse_attend_prefill": [CFG, P, P, P, P, P, I, I64, I, F, P, P, SZ, P],
    "msa_sparse_attend_prefill_lse": [CFG, P, P, P, P, P, I, I64, I, F, P, P, P, SZ, P],
    "msa_sparse_attend_prefill_backward": [CFG, P, P, P, P, P, I, I64, I, F, P, P, P, P, P, P, P, SZ, P],
    "msa_pack_metadata": [P, I, I, P, P, ctypes.POINTER(I), ctypes.POINTER(I64), ctypes.POINTER(I),
                          ctypes.POINTER(I64), P, SZ, P],
    "msa_pack": [P, P, I64, I64, P, P],
    "msa_unpack": [P, P, I64, I64, I64, P, P],
    "msa_check_bounded_wait": [P, P, ctypes.POINTER(I64)],
    "msa_index_produce_prefill": [CFG, P, P, P, I, I64, P, P, P, P, I, I64, P, SZ, P],
    "msa_index_produce_decode": [CFG, P, P, P, P, P, I, I, I64, P, P, P, SZ, P],
}
EXPORTS = tuple(_SIGS) + ("msa_status_string", "msa_last_cuda_error", "msa_cuda_error_string")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libmsa.so (building it first when it is missing or stale).  Raises
    when the library cannot be built or loaded: there is no other path."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libmsa not built: {path} is missing")
            lib = ctypes.CDLL(path)
            for name, args in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.msa_status_string.argtypes = [ctypes.c_int]
            lib.msa_status_string.restype = ctypes.c_char_p
            lib.msa_last_cuda_error.argtypes = []
            lib.msa_last_cuda_error.restype = ctypes.c_int
            lib.msa_cuda_error_string.argtypes = [ctypes.c_int]
            lib.msa_cuda_error_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _call(name: str, *args):
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        text = lib.msa_status_string(st).decode()
        if st == MSA_ERR_CUDA:
            code = lib.msa_last_cuda_error()
            text += f": {lib.msa_cuda_error_string(code).decode()} (cudaError {code})"
        raise MsaError(name, st, text)
    return st


def make_config(topk: int = 16, init_blocks: int = 0, local_blocks: int = 1, index_dtype="bf16",
                **overrides) -> msa_config:
    cfg = msa_config()
    _call("msa_config_default", ctypes.byref(cfg))
    cfg.topk, cfg.init_blocks, cfg.local_blocks = topk, init_blocks, local_blocks
    cfg.index_dtype = INDEX_DTYPES[index_dtype] if isinstance(index_dtype, str) else int(index_dtype)
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None:
        if t.dim() != len(shape) or any(b is not None and a != b for a, b in zip(t.shape, shape)):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    return t


def _index_dtype(t):
    if t.dtype == torch.bfloat16:
        return "bf16"
    if t.dtype == torch.float8_e4m3fn:
        return "e4m3"
    raise ValueError(f"index tensors must be bf16 or float8_e4m3fn, got {t.dtype}")


def workspace_size(cfg: msa_config, mode: int, n: int, max_blocks: int) -> int:
    out = ctypes.c_size_t()
    _call("msa_workspace_size", ctypes.byref(cfg), mode, n, max_blocks, ctypes.byref(out))
    return out.value


class Workspace:
    """Caller-owned scratch for the library's calls; zeroed once at creation."""

    def __init__(self, nbytes: int, device=None):
        self.nbytes = int(nbytes)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        _call("msa_workspace_init", _ptr(self.buf), self.nbytes, _stream(self.buf.device))

    def grow(self, nbytes: int):
        if nbytes > self.nbytes:
            self.__init__(nbytes, self.buf.device)
        return self

    def read_device_error(self):
        code, detail = ctypes.c_int(), ctypes.c_int64()
        _call("msa_read_device_error", _ptr(self.buf), _stream(self.buf.device), ctypes.byref(code),
              ctypes.byref(detail))
        return code.value, detail.value


_WS: dict = {}


def _workspace(key, nbytes, device, ws):
    if ws is not None:
        if ws.nbytes < nbytes:
            raise ValueError(f"workspace too small: {ws.nbytes} < {nbytes}")
        return ws
    w = _WS.get((key, str(device)))
    if w is None:
        w = _WS[(key, str(device))] = Workspace(nbytes, device)
    return w.grow(nbytes)


# ---- decode -----------------------------------------------------------------------

def msa_select_blocks_decode(index_q, index_k_cache, seq_lens, page_table=None, cu_seqlens_k=None, *,
                             max_blocks=None, topk=16, init_blocks=0, local_blocks=1, q2k=None,
                             workspace=None):
    """q2k int32 [4, batch, topk] for one decode query per request (C: msa_select_blocks_decode)."""
    B = index_q.shape[0]
    dt = _index_dtype(index_q)
    _need(index_q, "index_q", (torch.bfloat16, torch.float8_e4m3fn), (B, G, DI))
    _need(index_k_cache, "index_k_cache", index_q.dtype, (None, 1, DI))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if page_table is not None:
        _need(page_table, "page_table", torch.int32, (B, None))
        mb = page_table.shape[1]
    else:
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int64, (B + 1,))
        mb = max_blocks
    if mb is None:
        raise ValueError("max_blocks is required with a contiguous cache")
    cfg = make_config(topk, init_blocks, local_blocks, dt)
    dev = index_q.device
    if q2k is None:
        q2k = torch.empty((G, B, topk), dtype=torch.int32, device=dev)
    _need(q2k, "q2k", torch.int32, (G, B, topk))
    ws = _workspace("decode", workspace_size(cfg, MODE_DECODE, B, mb), dev, workspace)
    _call("msa_select_blocks_decode", ctypes.byref(cfg), _ptr(index_q), _ptr(index_k_cache), _ptr(seq_lens),
          _ptr(page_table), _ptr(cu_seqlens_k if page_table is None else None), B, mb,
          index_k_cache.shape[0], _ptr(q2k), _ptr(ws.buf), ws.nbytes, _stream(dev))
    return q2k


def msa_sparse_attend_decode(q, k_cache, v_cache, q2k, seq_lens, page_table=None, cu_seqlens_k=None, *,
                             max_blocks=None, scale=None, out=None, workspace=None):
    """bf16 out [batch, 64, 128] (C: msa_sparse_attend_decode)."""
    B = q.shape[0]
    _need(q, "q", torch.bfloat16, (B, H, D))
    _need(k_cache, "k_cache", torch.bfloat16, (None, G, D))
    _need(v_cache, "v_cache", torch.bfloat16, tuple(k_cache.shape))
    _need(q2k, "q2k", torch.int32, (G, B, None))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if page_table is not None:
        _need(page_table, "page_table", torch.int32, (B, None))
        mb = page_table.shape[1]
    else:
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int64, (B + 1,))
        mb = max_blocks
    if mb is None:
        raise ValueError("max_blocks is required with a contiguous cache")
    cfg = make_config(q2k.shape[2], 0, 0)
    dev = q.device
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B, H, D))
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    ws = _workspace("decode", workspace_size(cfg, MODE_DECODE, B, mb), dev, workspace)
    _call("msa_sparse_attend_decode", ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(q2k),
          _ptr(seq_lens), _ptr(page_table), _ptr(cu_seqlens_k if page_table is None else None), B, mb,
          k_cache.shape[0], scale, _ptr(out), _ptr(ws.buf), ws.nbytes, _stream(dev))
    return out


def msa_sparse_attend_decode_mxfp8(q, k_cache, v_cache, q2k, seq_lens, page_table=None, cu_seqlens_k=None, *,
                                   max_blocks=None, scale=None, out_q=None, out_scale=None, workspace=None):
    """The decode attention with the output as MXFP8: (E4M3 bytes uint8 [batch, 64 * 128], E8M0 scale
    bytes uint8 [batch, 256]) (C: msa_sparse_attend_decode_mxfp8)."""
    B = q.shape[0]
    _need(q, "q", torch.bfloat16, (B, H, D))
    _need(k_cache, "k_cache", torch.bfloat16, (None, G, D))
    _need(v_cache, "v_cache", torch.bfloat16, tuple(k_cache.shape))
    _need(q2k, "q2k", torch.int32, (G, B, None))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if page_table is not None:
        _need(page_table, "page_table", torch.int32, (B, None))
        mb = page_table.shape[1]
    else:
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int64, (B + 1,))
        mb = max_blocks
    if mb is None:
        raise ValueError("max_blocks is required with a contiguous cache")
    cfg = make_config(q2k.shape[2], 0, 0)
    dev = q.device
    out_q = torch.empty((B, H * D), dtype=torch.uint8, device=dev) if out_q is None else out_q
    out_scale = torch.empty((B, H * D // 32), dtype=torch.uint8, device=dev) if out_scale is None else out_scale
    _need(out_q, "out_q", torch.uint8, (B, H * D))
    _need(out_scale, "out_scale", torch.uint8, (B, H * D // 32))
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    ws = _workspace("decode", workspace_size(cfg, MODE_DECODE, B, mb), dev, workspace)
    _call("msa_sparse_attend_decode_mxfp8", ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(q2k),
          _ptr(seq_lens), _ptr(page_table), _ptr(cu_seqlens_k if page_table is None else None), B, mb,
          k_cache.shape[0], scale, _ptr(out_q), _ptr(out_scale), _ptr(ws.buf), ws.nbytes, _stream(dev))
    return out_q, out_scale


def msa_sparse_attend_decode_fp8kv(q, k_cache, v_cache, q2k, seq_lens, page_table=None, cu_seqlens_k=None, *,
                                   k_scale=1.0, v_scale=1.0, max_blocks=None, scale=None, out=None,
                                   workspace=None):
    """bf16 out [batch, 64, 128] over FP8 (E4M3) K/V caches standing for k_scale * k and
    v_scale * v (C: msa_sparse_attend_decode_fp8kv)."""
    B = q.shape[0]
    _need(q, "q", torch.bfloat16, (B, H, D))
    _need(k_cache, "k_cache", (torch.float8_e4m3fn, torch.uint8), (None, G, D))
    _need(v_cache, "v_cache", k_cache.dtype, tuple(k_cache.shape))
    _need(q2k, "q2k", torch.int32, (G, B, None))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if page_table is not None:
        _need(page_table, "page_table", torch.int32, (B, None))
        mb = page_table.shape[1]
    else:
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int64, (B + 1,))
        mb = max_blocks
    if mb is None:
        raise ValueError("max_blocks is required with a contiguous cache")
    cfg = make_config(q2k.shape[2], 0, 0)
    dev = q.device
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B, H, D))
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    ws = _workspace("decode", workspace_size(cfg, MODE_DECODE, B, mb), dev, workspace)
    _call("msa_sparse_attend_decode_fp8kv", ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache),
          float(k_scale), float(v_scale), _ptr(q2k), _ptr(seq_lens), _ptr(page_table),
          _ptr(cu_seqlens_k if page_table is None else None), B, mb, k_cache.shape[0], scale, _ptr(out),
          _ptr(ws.buf), ws.nbytes, _stream(dev))
    return out


# ---- prefill ----------------------------------------------------------------------

def msa_select_blocks_prefill(index_q, index_k, cu_seqlens, max_seqlen, *, topk=16, init_blocks=0,
                              local_blocks=1, q2k=None, workspace=None):
    """q2k int32 [4, tokens, topk] for packed documents (C: msa_select_blocks_prefill)."""
    T = index_q.shape[0]
    idt = _index_dtype(index_q)
    _need(index_q, "index_q", index_q.dtype, (T, G, DI))
    _need(index_k, "index_k", index_q.dtype, (T, 1, DI))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (None,))
    cfg = make_config(topk, init_blocks, local_blocks, idt)
    dev = index_q.device
    if q2k is None:
        q2k = torch.empty((G, T, topk), dtype=torch.int32, device=dev)
    _need(q2k, "q2k", torch.int32, (G, T, topk))
    mt = (int(max_seqlen) + BLOCK - 1) // BLOCK
    ws = _workspace("prefill", workspace_size(cfg, MODE_PREFILL, T, mt), dev, workspace)
    _call("msa_select_blocks_prefill", ctypes.byref(cfg), _ptr(index_q), _ptr(index_k), _ptr(cu_seqlens),
          cu_seqlens.shape[0] - 1, T, int(max_seqlen), _ptr(q2k), _ptr(ws.buf), ws.nbytes, _stream(dev))
    return q2k


def msa_sparse_attend_prefill(q, k, v, q2k, cu_seqlens, max_seqlen, *, scale=None, out=None, lse=None,
                              workspace=None):
    """bf16 out [tokens, 64, 128] for packed documents (C: msa_sparse_attend_prefill).  With ``lse``
    (fp32 [tokens, 64]) the call also writes the log-sum-exp the backward needs
    (C: msa_sparse_attend_prefill_lse)."""
    T = q.shape[0]
    _need(q, "q", torch.bfloat16, (T, H, D))
    _need(k, "k", torch.bfloat16, (T, G, D))
    _need(v, "v", torch.bfloat16, (T, G, D))
    _need(q2k, "q2k", torch.int32, (G, T, None))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (None,))
    cfg = make_config(q2k.shape[2], 0, 0)
    dev = q.device
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (T, H, D))
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    mt = (int(max_seqlen) + BLOCK - 1) // BLOCK
    ws = _workspace("prefill", workspace_size(cfg, MODE_PREFILL, T, mt), dev, workspace)
    if lse is None:
        _call("msa_sparse_attend_prefill", ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(q2k),
              _ptr(cu_seqlens), cu_seqlens.shape[0] - 1, T, int(max_seqlen), scale, _ptr(out), _ptr(ws.buf),
              ws.nbytes, _stream(dev))
    else:
        _need(lse, "lse", torch.float32, (T, H))
        _call("msa_sparse_attend_prefill_lse", ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(q2k),
              _ptr(cu_seqlens), cu_seqlens.shape[0] - 1, T, int(max_seqlen), scale, _ptr(out), _ptr(lse),
              _ptr(ws.buf), ws.nbytes, _stream(dev))
    return out


def msa_sparse_attend_prefill_backward(q, k, v, q2k, cu_seqlens, max_seqlen, out, lse, grad_out, *, scale=None,
                                       dq=None, dk=None, dv=None, workspace=None):
    """(dq [tokens, 64, 128], dk [tokens, 4, 128], dv [tokens, 4, 128]) bf16 from the forward's
    out and lse and grad_out (C: msa_sparse_attend_prefill_backward)."""
    T = q.shape[0]
    _need(q, "q", torch.bfloat16, (T, H, D))
    _need(k, "k", torch.bfloat16, (T, G, D))
    _need(v, "v", torch.bfloat16, (T, G, D))
    _need(q2k, "q2k", torch.int32, (G, T, None))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (None,))
    _need(out, "out", torch.bfloat16, (T, H, D))
    _need(lse, "lse", torch.float32, (T, H))
    _need(grad_out, "grad_out", torch.bfloat16, (T, H, D))
    cfg = make_config(q2k.shape[2], 0, 0)
    dev = q.device
    dq = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev) if dq is None else dq
    dk = torch.empty((T, G, D), dtype=torch.bfloat16, device=dev) if dk is None else dk
    dv = torch.empty((T, G, D), dtype=torch.bfloat16, device=dev) if dv is None else dv
    _need(dq, "dq", torch.bfloat16, (T, H, D))
    _need(dk, "dk", torch.bfloat16, (T, G, D))
    _need(dv, "dv", torch.bfloat16, (T, G, D))
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    mt = (int(max_seqlen) + BLOCK - 1) // BLOCK
    ws = _workspace("prefill_bwd", workspace_size(cfg, MODE_PREFILL_BWD, T, mt), dev, workspace)
    _call("msa_sparse_attend_prefill_backward", ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(q2k),
          _ptr(cu_seqlens), cu_seqlens.shape[0] - 1, T, int(max_seqlen), scale, _ptr(out), _ptr(lse),
          _ptr(grad_out), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws.buf), ws.nbytes, _stream(dev))
    return dq, dk, dv


class _SparseAttention(torch.autograd.Function):
    """NeMo ``_SparseAttention``: the prefill sparse attention as an autograd
    function (forward: msa_sparse_attend_prefill_lse; backward:
    msa_sparse_attend_prefill_backward).  q, k and v receive gradients; q2k and
    the document layout do not."""

    @staticmethod
    def forward(ctx, q, k, v, q2k, cu_seqlens, max_seqlen, scale):
        T = q.shape[0]
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
        out = msa_sparse_attend_prefill(q, k, v, q2k, cu_seqlens, max_seqlen, scale=scale, lse=lse)
        ctx.save_for_backward(q, k, v, q2k, cu_seqlens, out, lse)
        ctx.max_seqlen, ctx.scale = max_seqlen, scale
        return out

    @staticmethod
    def backward(ctx, grad_out):
        q, k, v, q2k, cu_seqlens, out, lse = ctx.saved_tensors
        dq, dk, dv = msa_sparse_attend_prefill_backward(q, k, v, q2k, cu_seqlens, ctx.max_seqlen, out, lse,
                                                        grad_out.contiguous(), scale=ctx.scale)
        return dq, dk, dv, None, None, None, None


def sparse_attention(q, k, v, q2k, cu_seqlens, max_seqlen, *, scale=None):
    """Differentiable prefill sparse attention (NeMo ``sparse_attention``): bf16 out
    [tokens, 64, 128]; q, k and v receive gradients through the library's backward."""
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    return _SparseAttention.apply(q, k, v, q2k, cu_seqlens, int(max_seqlen), scale)


# ---- index producer -----------------------------------------------------------------

_INDEX_TORCH = {"bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}


def _produce_ws(device, workspace):
    return _workspace("produce", 256, device, workspace)


def msa_index_produce_prefill(index_q, index_k, cu_seqlens, *, index_dtype="bf16", index_k_cache=None,
                              page_table=None, q_out=None, k_out=None, write_k_out=True, workspace=None):
    """Normalised index tensors for a packed prefill (C: msa_index_produce_prefill): returns
    (index_q_out [T, 4, 128], index_k_out [T, 1, 128] or None) in ``index_dtype``; with
    ``index_k_cache`` and ``page_table`` ([docs, max_blocks]) every token's key is also
    written into the paged cache."""
    T = index_q.shape[0]
    _need(index_q, "index_q", torch.bfloat16, (T, G, DI))
    _need(index_k, "index_k", torch.bfloat16, (T, 1, DI))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (None,))
    dt = _INDEX_TORCH[index_dtype]
    cfg = make_config(index_dtype=index_dtype)
    dev = index_q.device
    q_out = torch.empty((T, G, DI), dtype=dt, device=dev) if q_out is None else q_out
    _need(q_out, "q_out", dt, (T, G, DI))
    if write_k_out:
        k_out = torch.empty((T, 1, DI), dtype=dt, device=dev) if k_out is None else k_out
        _need(k_out, "k_out", dt, (T, 1, DI))
    else:
        k_out = None
    mb, ns = 0, 0
    if index_k_cache is not None:
        _need(index_k_cache, "index_k_cache", dt, (None, 1, DI))
        _need(page_table, "page_table", torch.int32, (cu_seqlens.shape[0] - 1, None))
        mb, ns = page_table.shape[1], index_k_cache.shape[0]
    ws = _produce_ws(dev, workspace)
    _call("msa_index_produce_prefill", ctypes.byref(cfg), _ptr(index_q), _ptr(index_k), _ptr(cu_seqlens),
          cu_seqlens.shape[0] - 1, T, _ptr(q_out), _ptr(k_out), _ptr(index_k_cache), _ptr(page_table), mb, ns,
          _ptr(ws.buf), ws.nbytes, _stream(dev))
    return q_out, k_out


def msa_index_produce_decode(index_q, index_k, index_k_cache, seq_lens, page_table=None, cu_seqlens_k=None, *,
                             max_blocks=None, q_out=None, workspace=None):
    """Normalised index queries [batch, 4, 128] in the cache's dtype, with each request's new
    normalised key written into ``index_k_cache`` at the slot of position seq_lens[r] - 1
    (C: msa_index_produce_decode)."""
    B = index_q.shape[0]
    _need(index_q, "index_q", torch.bfloat16, (B, G, DI))
    _need(index_k, "index_k", torch.bfloat16, (B, 1, DI))
    dtn = _index_dtype(index_k_cache)
    _need(index_k_cache, "index_k_cache", index_k_cache.dtype, (None, 1, DI))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    if page_table is not None:
        _need(page_table, "page_table", torch.int32, (B, None))
        mb = page_table.shape[1]
    else:
        _need(cu_seqlens_k, "cu_seqlens_k", torch.int64, (B + 1,))
        mb = max_blocks if max_blocks is not None else 1
    cfg = make_config(index_dtype=dtn)
    dev = index_q.device
    q_out = torch.empty((B, G, DI), dtype=index_k_cache.dtype, device=dev) if q_out is None else q_out
    _need(q_out, "q_out", index_k_cache.dtype, (B, G, DI))
    ws = _produce_ws(dev, workspace)
    _call("msa_index_produce_decode", ctypes.byref(cfg), _ptr(index_q), _ptr(index_k), _ptr(seq_lens),
          _ptr(page_table), _ptr(cu_seqlens_k if page_table is None else None), B, mb, index_k_cache.shape[0],
          _ptr(q_out), _ptr(index_k_cache), _ptr(ws.buf), ws.nbytes, _stream(dev))
    return q_out


# ---- packing ----------------------------------------------------------------------

def msa_pack_metadata(doc_ids, *, workspace=None):
    """(cu_seqlens int32 [docs+1], token_rows int64 [tokens], max_seqlen) of a [batch, seq]
    int64 document map (C: msa_pack_metadata; one device-to-host synchronisation)."""
    _need(doc_ids, "doc_ids", torch.int64)
    if doc_ids.dim() != 2:
        raise ValueError("doc_ids must be [batch, seq]")
    b, s = doc_ids.shape
    dev = doc_ids.device
    n = max(b * s, 1)
    cu = torch.empty(n + 1, dtype=torch.int32, device=dev)
    rows = torch.empty(n, dtype=torch.int64, device=dev)
    nd, nt, mx, bad = ctypes.c_int(), ctypes.c_int64(), ctypes.c_int(), ctypes.c_int64()
    wsp, wsn = None, 0
    if b > 0 and s > 0:
        ws = _workspace("pack", workspace_size(make_config(), MODE_PACK, b * s, b), dev, workspace)
        wsp, wsn = _ptr(ws.buf), ws.nbytes
    st = load().msa_pack_metadata(_ptr(doc_ids), b, s, _ptr(cu), _ptr(rows), ctypes.byref(nd), ctypes.byref(nt),
                                  ctypes.byref(mx), ctypes.byref(bad), wsp, wsn, _stream(dev))
    if st != 0:
        err = MsaError("msa_pack_metadata", st, load().msa_status_string(st).decode())
        err.bad_index = bad.value
        raise err
    return cu[: nd.value + 1], rows[: nt.value], mx.value


def msa_pack(external, token_rows):
    """Gather external[batch, seq, ...] -> [tokens, ...] (C: msa_pack)."""
    _need(external, "external")
    _need(token_rows, "token_rows", torch.int64, (None,))
    feat = tuple(external.shape[2:])
    row_bytes = external[0, 0].numel() * external.element_size()
    out = torch.empty((token_rows.shape[0],) + feat, dtype=external.dtype, device=external.device)
    _call("msa_pack", _ptr(external), _ptr(token_rows), token_rows.shape[0], row_bytes, _ptr(out),
          _stream(external.device))
    return out


def msa_unpack(packed, token_rows, batch, seq):
    """Scatter packed[tokens, ...] -> [batch, seq, ...] with zero padding (C: msa_unpack)."""
    _need(packed, "packed")
    _need(token_rows, "token_rows", torch.int64, (packed.shape[0],))
    feat = tuple(packed.shape[1:])
    row_bytes = packed[0].numel() * packed.element_size() if packed.shape[0] else 16
    out = torch.empty((batch, seq) + feat, dtype=packed.dtype, device=packed.device)
    _call("msa_unpack", _ptr(packed), _ptr(token_rows), packed.shape[0], batch * seq, row_bytes, _ptr(out),
          _stream(packed.device))
    return out


def msa_check_bounded_wait(workspace=None, device=None):
    """Run the bounded-wait diagnostic (C: msa_check_bounded_wait) on a
    256-byte workspace; returns ((first_wait_ns, second_wait_ns), (code, detail))."""
    ws = workspace if workspace is not None else Workspace(256, device)
    waits = (I64 * 2)()
    _call("msa_check_bounded_wait", _ptr(ws.buf), _stream(ws.buf.device), waits)
    return (waits[0], waits[1]), ws.read_device_error()
