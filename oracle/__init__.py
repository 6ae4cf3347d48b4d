"""CPU oracle for MiniMax-M3 block-sparse attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never touches it, and it never touches the product path.

The arithmetic lives in ``msa_oracle.c`` (plain C, fp64, OpenMP over queries);
this module compiles it with gcc and wraps it with ctypes over numpy arrays.
Inputs are raw element bits (bf16 as uint16, E4M3 as uint8) so the oracle
decodes every element itself.

Which statement on the pages each function follows:
  * ``select_prefill`` / ``select_decode`` -- block scores (max over causal,
    document-local keys of the unscaled index dot product) and top-k with forced
    init/local blocks: TensorRT-LLM "MiniMaxM3SparseAttentionConfig" (class
    description; fields sparse_topk_blocks, sparse_init_blocks,
    sparse_local_blocks, sparse_score_type, indexer_kv_dtype) and NeMo AutoModel
    "...minimax_m3_vl.msa" (MSAMicrobatch.select_blocks, _SelectionPlan).
  * ``attend_prefill`` / ``attend_decode`` -- sparse GQA attention over the
    selected blocks: the TensorRT-LLM class description and NeMo
    ``sparse_attention`` / ``_SparseAttention.forward``.
  * ``attend_decode_fp8`` -- the decode attention over an FP8 (E4M3) main K/V
    cache with one dequantisation scale per cache (TensorRT-LLM field
    fuse_qkv_index_projection: "an FP8 main KV cache"; the scale rule is a
    reading, see the C source).
  * ``attend_prefill_backward`` -- gradients of the sparse attention (NeMo
    ``_SparseAttention.backward``: grad_out -> dq, dk, dv), written out from
    the forward; ``attend_loss_f64`` -- the forward on fp64 inputs reduced to
    sum(out * dout), whose finite differences pin the backward.
  * ``mxfp8_quantize`` -- the MXFP8 emission of the output (vLLM page,
    forward_decode_mxfp8: E4M3 values, E8M0 scales per 32 elements), after the
    OCP MX block rule, which the page names but does not print.
  * ``pack_metadata`` / ``pack`` / ``unpack`` -- NeMo layout-from-doc_ids
    constructor, ``_contiguous_runs``, ``MSAMicrobatch.pack`` / ``unpack``.
  * ``index_normalize`` / ``index_produce_prefill`` / ``index_produce_decode``
    -- the index producer: L2 norm, storage cast (bf16 or unscaled E4M3) and
    insertion of index-K into the paged side cache (TensorRT-LLM fields
    fuse_qkv_index_projection and indexer_kv_dtype, the class description's
    paged index-K cache; NeMo select_blocks takes index tensors "post norm").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()

H, G, D, DI, BLOCK = 64, 4, 128, 128, 128
PACK_ERRORS = {
    1: "negative document id",
    2: "interrupted document",
    3: "no real token",
    4: "empty map",
    5: "coordinates past int32",
}


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2, OpenMP, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c11",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            Dbl = ctypes.c_double
            lib.oracle_select_prefill.argtypes = [P, P, I, P, I, P, I64, I, I, I, P, P, P, I]
            lib.oracle_attend_prefill.argtypes = [P, P, P, P, I, P, I64, P, I, Dbl, P]
            lib.oracle_select_decode.argtypes = [P, P, I, P, P, P, I, P, I64, I, I, I, P, P, P, I]
            lib.oracle_attend_decode.argtypes = [P, P, P, P, P, P, I, P, I64, P, I, Dbl, P]
            lib.oracle_pack_metadata.argtypes = [P, I64, I64, P, P, P, P, P, P]
            lib.oracle_attend_prefill_backward.argtypes = [P, P, P, P, P, I, I64, P, I, Dbl, P, P, P]
            lib.oracle_attend_loss_f64.argtypes = [P, P, P, P, P, I, I64, P, I, Dbl]
            lib.oracle_attend_loss_f64.restype = Dbl
            lib.oracle_mxfp8_quantize.argtypes = [P, I64, P, P]
            lib.oracle_index_normalize.argtypes = [P, I64, I, P]
            lib.oracle_attend_decode_fp8.argtypes = [P, P, P, Dbl, Dbl, P, P, P, I, P, I64, P, I, Dbl, P]
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = Dbl
            for f in (lib.oracle_select_prefill, lib.oracle_attend_prefill,
                      lib.oracle_select_decode, lib.oracle_attend_decode,
                      lib.oracle_pack_metadata):
                f.restype = I
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(x):
    """numpy view of raw element bits: bf16 -> uint16, e4m3 -> uint8."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            if x.dtype == torch.float8_e4m3fn:
                return x.view(torch.uint8).numpy()
            return x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x)


def _dtype_code(a):
    if a.dtype == np.uint16:
        return 0
    if a.dtype == np.uint8:
        return 1
    raise TypeError("index tensors must be bf16 (uint16 bits) or e4m3 (uint8 bits)")


def _i32(x):
    return np.ascontiguousarray(_bits(x), dtype=np.int32)


def _i64(x):
    return np.ascontiguousarray(_bits(x), dtype=np.int64)


def e4m3_value(byte: int) -> float:
    return _load().oracle_e4m3_value(byte)


def select_prefill(index_q, index_k, cu_seqlens, tokens, topk=16, init=0, local=1,
                   return_scores=False):
    """q2k int32 [G, n, topk] and relative top-k gap [G, n] for compact tokens."""
    lib = _load()
    iq, ik = _bits(index_q), _bits(index_k)
    code = _dtype_code(iq)
    cu = _i32(cu_seqlens)
    tok = _i64(tokens)
    n = tok.shape[0]
    q2k = np.full((G, n, topk), -7, dtype=np.int32)
    gap = np.zeros((G, n), dtype=np.float64)
    scores = None
    max_nb = 0
    if return_scores:
        lens = np.diff(cu.astype(np.int64))
        max_nb = int((lens.max() + BLOCK - 1) // BLOCK)
        scores = np.full((n, G, max_nb), np.nan)
    rc = lib.oracle_select_prefill(_ptr(iq), _ptr(ik), code, _ptr(cu), cu.shape[0] - 1, _ptr(tok), n,
                                   topk, init, local, _ptr(q2k), _ptr(gap), _ptr(scores), max_nb)
    if rc:
        raise ValueError("oracle_select_prefill failed")
    return (q2k, gap, scores) if return_scores else (q2k, gap)


def attend_prefill(q, k, v, cu_seqlens, tokens, q2k, scale):
    """fp64 out [n, H, D] for compact tokens, given their q2k rows [G, n, topk]."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cu = _i32(cu_seqlens)
    tok = _i64(tokens)
    n = tok.shape[0]
    q2k = _i32(q2k)
    topk = q2k.shape[2]
    out = np.zeros((n, H, D), dtype=np.float64)
    lib.oracle_attend_prefill(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), cu.shape[0] - 1, _ptr(tok), n,
                              _ptr(q2k), topk, float(scale), _ptr(out))
    return out


def attend_prefill_backward(q, k, v, dout, cu_seqlens, q2k, scale):
    """fp64 (dq [T, H, D], dk [T, G, D], dv [T, G, D]) for every compact token,
    given bf16 q, k, v, grad_out and the q2k rows of all tokens [G, T, topk]."""
    lib = _load()
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    cu = _i32(cu_seqlens)
    q2k = _i32(q2k)
    T, topk = q2k.shape[1], q2k.shape[2]
    dq = np.zeros((T, H, D), dtype=np.float64)
    dk = np.zeros((T, G, D), dtype=np.float64)
    dv = np.zeros((T, G, D), dtype=np.float64)
    lib.oracle_attend_prefill_backward(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(db), _ptr(cu), cu.shape[0] - 1, T,
                                       _ptr(q2k), topk, float(scale), _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


def attend_loss_f64(q, k, v, dout, cu_seqlens, q2k, scale):
    """sum(out * dout) of the forward on fp64 numpy inputs q [T, H, D],
    k / v [T, G, D], dout [T, H, D] (no bf16 rounding anywhere)."""
    lib = _load()
    q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, dout))
    cu = _i32(cu_seqlens)
    q2k = _i32(q2k)
    return lib.oracle_attend_loss_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(cu), cu.shape[0] - 1,
                                      q2k.shape[1], _ptr(q2k), q2k.shape[2], float(scale))


def mxfp8_quantize(x):
    """(E4M3 bytes uint8 [..., n], E8M0 scale bytes uint8 [..., n / 32]) of a bf16 tensor whose
    last dimension is a multiple of 32: the OCP MX block rule (see the C source)."""
    lib = _load()
    xb = np.ascontiguousarray(_bits(x))
    shape = xb.shape
    n = xb.size
    q = np.zeros(n, dtype=np.uint8)
    sc = np.zeros(n // 32, dtype=np.uint8)
    if lib.oracle_mxfp8_quantize(_ptr(xb), n, _ptr(q), _ptr(sc)):
        raise ValueError("the element count must be a multiple of 32")
    return q.reshape(shape), sc.reshape(shape[:-1] + (shape[-1] // 32,))


def select_decode(index_q, index_k_cache, seq_lens, page_table=None, cu_seqlens_k=None,
                  requests=None, topk=16, init=0, local=1, return_scores=False):
    """q2k int32 [G, n, topk] and gap [G, n] for the listed requests (and, with
    ``return_scores``, the fp64 block scores [n, G, max_nb], NaN past a request's
    blocks)."""
    lib = _load()
    iq, ik = _bits(index_q), _bits(index_k_cache)
    code = _dtype_code(iq)
    sl = _i32(seq_lens)
    pt = None if page_table is None else _i32(page_table)
    cuk = None if cu_seqlens_k is None else _i64(cu_seqlens_k)
    if pt is None and cuk is None:
        raise ValueError("need page_table or cu_seqlens_k")
    req = _i64(np.arange(sl.shape[0]) if requests is None else requests)
    n = req.shape[0]
    max_pages = 0 if pt is None else pt.shape[1]
    q2k = np.full((G, n, topk), -7, dtype=np.int32)
    gap = np.zeros((G, n), dtype=np.float64)
    scores, max_nb = None, 0
    if return_scores:
        max_nb = int((sl[req].max() + BLOCK - 1) // BLOCK) if n else 0
        scores = np.full((n, G, max(max_nb, 1)), np.nan)
    rc = lib.oracle_select_decode(_ptr(iq), _ptr(ik), code, _ptr(sl), _ptr(pt), _ptr(cuk), max_pages,
                                  _ptr(req), n, topk, init, local, _ptr(q2k), _ptr(gap), _ptr(scores), max_nb)
    if rc:
        raise ValueError("oracle_select_decode failed")
    return (q2k, gap, scores) if return_scores else (q2k, gap)


def attend_decode(q, k_cache, v_cache, seq_lens, q2k, scale, page_table=None, cu_seqlens_k=None,
                  requests=None):
    """fp64 out [n, H, D] for the listed requests, given their q2k rows [G, n, topk]."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    sl = _i32(seq_lens)
    pt = None if page_table is None else _i32(page_table)
    cuk = None if cu_seqlens_k is None else _i64(cu_seqlens_k)
    req = _i64(np.arange(sl.shape[0]) if requests is None else requests)
    n = req.shape[0]
    q2k = _i32(q2k)
    topk = q2k.shape[2]
    max_pages = 0 if pt is None else pt.shape[1]
    out = np.zeros((n, H, D), dtype=np.float64)
    lib.oracle_attend_decode(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(sl), _ptr(pt), _ptr(cuk), max_pages,
                             _ptr(req), n, _ptr(q2k), topk, float(scale), _ptr(out))
    return out


def attend_decode_fp8(q, k_cache, v_cache, seq_lens, q2k, scale, k_scale=1.0, v_scale=1.0, page_table=None,
                      cu_seqlens_k=None, requests=None):
    """fp64 out [n, H, D] over E4M3 K/V caches (raw bytes or float8_e4m3fn tensors) standing for
    k_scale * k and v_scale * v, for the listed requests given their q2k rows [G, n, topk]."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    if kb.dtype != np.uint8 or vb.dtype != np.uint8:
        raise TypeError("the K/V caches must be E4M3 bytes")
    sl = _i32(seq_lens)
    pt = None if page_table is None else _i32(page_table)
    cuk = None if cu_seqlens_k is None else _i64(cu_seqlens_k)
    req = _i64(np.arange(sl.shape[0]) if requests is None else requests)
    n = req.shape[0]
    q2k = _i32(q2k)
    out = np.zeros((n, H, D), dtype=np.float64)
    lib.oracle_attend_decode_fp8(_ptr(qb), _ptr(kb), _ptr(vb), float(k_scale), float(v_scale), _ptr(sl), _ptr(pt),
                                 _ptr(cuk), 0 if pt is None else pt.shape[1], _ptr(req), n, _ptr(q2k), q2k.shape[2],
                                 float(scale), _ptr(out))
    return out


def pack_metadata(doc_ids):
    """(cu_seqlens int32 [docs+1], token_rows int64 [tokens], max_seqlen) or ValueError."""
    lib = _load()
    ids = _i64(doc_ids)
    if ids.ndim != 2:
        raise ValueError("doc_ids must be [batch, seq]")
    b, s = ids.shape
    n = max(b * s, 1)
    cu = np.zeros(n + 1, dtype=np.int32)
    rows = np.zeros(n, dtype=np.int64)
    nd, nt, mx, bad = (np.zeros(1, dtype=np.int64) for _ in range(4))
    rc = lib.oracle_pack_metadata(_ptr(ids), b, s, _ptr(cu), _ptr(rows), _ptr(nd), _ptr(nt),
                                  _ptr(mx), _ptr(bad))
    if rc:
        err = ValueError(PACK_ERRORS[rc])
        err.code = rc
        err.bad_row = int(bad[0])
        raise err
    return cu[: nd[0] + 1].copy(), rows[: nt[0]].copy(), int(mx[0])


def pack(external, token_rows):
    """Gather external[batch, seq, ...] -> [tokens, ...] (NeMo MSAMicrobatch.pack)."""
    x = np.asarray(external)
    flat = x.reshape((-1,) + x.shape[2:])
    return flat[np.asarray(token_rows)]


def unpack(packed, token_rows, batch, seq):
    """Scatter packed[tokens, ...] -> [batch, seq, ...], zeros elsewhere (NeMo unpack)."""
    p = np.asarray(packed)
    out = np.zeros((batch * seq,) + p.shape[1:], dtype=p.dtype)
    out[np.asarray(token_rows)] = p
    return out.reshape((batch, seq) + p.shape[1:])


def exempt_rows(gap, rel=1e-5):
    """Boolean [G, n]: rows whose k-th / (k+1)-th non-forced scores are a near tie."""
    return np.asarray(gap) < rel


# ---- index producer ------------------------------------------------------------

def index_normalize(x, dtype="bf16"):
    """L2-normalised 128-vectors of a bf16 tensor [..., 128], stored as bf16 bits
    (uint16) or E4M3 bytes (uint8) of the same shape (see the C source for the
    reading of the norm's precision)."""
    lib = _load()
    xb = np.ascontiguousarray(_bits(x))
    if xb.dtype != np.uint16 or xb.shape[-1] != DI:
        raise TypeError("index_normalize takes bf16 [..., 128]")
    n = xb.size // DI
    out = np.zeros(xb.shape, dtype=np.uint16 if dtype == "bf16" else np.uint8)
    lib.oracle_index_normalize(_ptr(xb), n, 0 if dtype == "bf16" else 1, _ptr(out))
    return out


def index_slots_decode(seq_lens, page_table=None, cu_seqlens_k=None):
    """Slot of each request's newest key (position seq_lens[r] - 1): page_table[r][p // 128] * 128 + p % 128
    (paged, the TensorRT-LLM page's index-K cache parallel to the K/V cache) or cu_seqlens_k[r] + p."""
    L = _i64(seq_lens)
    p = L - 1
    if page_table is not None:
        pt = _i64(page_table)
        return pt[np.arange(L.shape[0]), p // BLOCK] * BLOCK + p % BLOCK
    return _i64(cu_seqlens_k)[:-1] + p


def index_slots_prefill(cu_seqlens, page_table):
    """Slot of every compact token: document d, position p = t - cu_seqlens[d], slot
    page_table[d][p // 128] * 128 + p % 128."""
    cu = _i64(cu_seqlens)
    pt = _i64(page_table)
    T = int(cu[-1])
    t = np.arange(T, dtype=np.int64)
    d = np.searchsorted(cu, t, side="right") - 1
    p = t - cu[d]
    return pt[d, p // BLOCK] * BLOCK + p % BLOCK


def index_produce_decode(index_q, index_k, index_k_cache, seq_lens, page_table=None, cu_seqlens_k=None,
                         dtype="bf16"):
    """(index_q_out [B, 4, 128], the index-K cache [slots, 1, 128] with each request's new
    normalised row written at its slot) as raw bits / bytes; the cache passed in is copied."""
    q_out = index_normalize(index_q, dtype)
    k_rows = index_normalize(index_k, dtype)
    cache = np.array(_bits(index_k_cache), copy=True)
    slots = index_slots_decode(seq_lens, page_table, cu_seqlens_k)
    cache[slots] = k_rows
    return q_out, cache


def index_produce_prefill(index_q, index_k, cu_seqlens, dtype="bf16", index_k_cache=None, page_table=None):
    """(index_q_out [T, 4, 128], index_k_out [T, 1, 128], the cache with every token's row at its
    slot, or None) as raw bits / bytes."""
    q_out = index_normalize(index_q, dtype)
    k_out = index_normalize(index_k, dtype)
    cache = None
    if index_k_cache is not None:
        cache = np.array(_bits(index_k_cache), copy=True)
        cache[index_slots_prefill(cu_seqlens, page_table)] = k_out
    return q_out, k_out, cache
