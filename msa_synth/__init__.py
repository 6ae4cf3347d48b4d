"""Seeded synthetic inputs for MiniMax-M3 block-sparse attention workloads.

This module is the one source of inputs for both the CUDA path and the CPU
oracle.  It holds none of the method's arithmetic: it only draws numbers,
normalises index vectors (the pages' index Q/K are "post norm"), casts to the
storage dtype and lays the tensors out.

Recipe (fixed draw order, documented per function):
  * integer structure (context lengths, page permutation, document lengths) is
    drawn on the CPU with numpy PCG64(seed), so it is identical on every device;
  * tensor values are drawn with a torch.Generator on the target device seeded
    with ``seed + 1``: q, k, v ~ N(0, 1) in fp32 then rounded to bf16; index
    q / k ~ N(0, 1), L2-normalised per 128-vector, then bf16 or E4M3
    (round-to-nearest-even; |x| <= 1 never saturates);
  * RoPE is omitted (the workloads fix post-norm, RoPE-free index vectors).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

H, G, D, DI, BLOCK = 64, 4, 128, 128, 128


def _tgen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) + 1)
    return g


def normal_bf16(shape, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def unit_vectors(shape, gen, device, dtype: str = "bf16") -> torch.Tensor:
    """N(0,1) draws normalised to unit L2 norm along the last axis."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    x = x / x.norm(dim=-1, keepdim=True)
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "e4m3":
        return x.to(torch.float8_e4m3fn)
    raise ValueError(dtype)


@dataclass
class DecodeInputs:
    q: torch.Tensor                 # [B, 64, 128] bf16
    index_q: torch.Tensor           # [B, 4, 128] bf16 / e4m3
    k_cache: torch.Tensor           # [num_slots, 4, 128] bf16
    v_cache: torch.Tensor           # [num_slots, 4, 128] bf16
    index_k_cache: torch.Tensor     # [num_slots, 1, 128] bf16 / e4m3
    seq_lens: torch.Tensor          # [B] int32
    page_table: torch.Tensor | None  # [B, max_blocks] int32 (paged) or None
    cu_seqlens_k: torch.Tensor | None  # [B+1] int64 (contiguous) or None
    max_blocks: int
    num_slots: int
    topk: int = 16
    init_blocks: int = 0
    local_blocks: int = 1
    index_dtype: str = "bf16"
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])


def decode_inputs(lens, *, paged: bool, index_dtype: str = "bf16", seed: int = 0,
                  device="cpu", topk: int = 16, init_blocks: int = 0, local_blocks: int = 1,
                  max_blocks: int | None = None) -> DecodeInputs:
    """Decode step over per-request contexts ``lens`` (query at position len-1).

    Draw order: page permutation (numpy, paged only); then on the torch
    generator: q, index_q, index_k_cache, k_cache, v_cache.
    """
    lens = np.asarray(lens, dtype=np.int64)
    B = int(lens.shape[0])
    nbs = (lens + BLOCK - 1) // BLOCK
    mb = int(nbs.max()) if max_blocks is None else int(max_blocks)
    rng = np.random.Generator(np.random.PCG64(seed))
    if paged:
        n_pages = int(nbs.sum())
        perm = rng.permutation(n_pages).astype(np.int32)
        pt = np.zeros((B, mb), dtype=np.int32)
        off = 0
        for r in range(B):
            pt[r, : nbs[r]] = perm[off: off + nbs[r]]
            off += nbs[r]
        num_slots = n_pages * BLOCK
        page_table = torch.from_numpy(pt).to(device)
        cu = None
    else:
        num_slots = int(lens.sum())
        cu_np = np.zeros(B + 1, dtype=np.int64)
        cu_np[1:] = np.cumsum(lens)
        cu = torch.from_numpy(cu_np).to(device)
        page_table = None
    gen = _tgen(seed, device)
    q = normal_bf16((B, H, D), gen, device)
    index_q = unit_vectors((B, G, DI), gen, device, index_dtype)
    index_k = unit_vectors((num_slots, 1, DI), gen, device, index_dtype)
    k_cache = normal_bf16((num_slots, G, D), gen, device)
    v_cache = normal_bf16((num_slots, G, D), gen, device)
    return DecodeInputs(q=q, index_q=index_q, k_cache=k_cache, v_cache=v_cache,
                        index_k_cache=index_k,
                        seq_lens=torch.from_numpy(lens.astype(np.int32)).to(device),
                        page_table=page_table, cu_seqlens_k=cu, max_blocks=mb, num_slots=num_slots,
                        topk=topk, init_blocks=init_blocks, local_blocks=local_blocks,
                        index_dtype=index_dtype)


@dataclass
class PrefillInputs:
    q: torch.Tensor          # [T, 64, 128] bf16
    k: torch.Tensor          # [T, 4, 128] bf16
    v: torch.Tensor          # [T, 4, 128] bf16
    index_q: torch.Tensor    # [T, 4, 128] bf16
    index_k: torch.Tensor    # [T, 1, 128] bf16
    cu_seqlens: torch.Tensor  # [docs+1] int32
    max_seqlen: int
    topk: int = 16
    init_blocks: int = 0
    local_blocks: int = 1
    index_dtype: str = "bf16"
    doc_ids: torch.Tensor | None = None  # [batch, seq] int64 map the tokens were packed from
    token_rows: torch.Tensor | None = None

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_docs(self) -> int:
        return int(self.cu_seqlens.shape[0] - 1)


def prefill_inputs(doc_lens, *, seed: int = 0, device="cpu", topk: int = 16, init_blocks: int = 0,
                   local_blocks: int = 1, index_dtype: str = "bf16") -> PrefillInputs:
    """Packed prefill over documents of lengths ``doc_lens`` (compact order).

    Draw order on the torch generator: q, k, v, index_q, index_k.
    """
    lens = np.asarray(doc_lens, dtype=np.int64)
    T = int(lens.sum())
    cu_np = np.zeros(lens.shape[0] + 1, dtype=np.int32)
    cu_np[1:] = np.cumsum(lens)
    gen = _tgen(seed, device)
    q = normal_bf16((T, H, D), gen, device)
    k = normal_bf16((T, G, D), gen, device)
    v = normal_bf16((T, G, D), gen, device)
    index_q = unit_vectors((T, G, DI), gen, device, index_dtype)
    index_k = unit_vectors((T, 1, DI), gen, device, index_dtype)
    return PrefillInputs(q=q, k=k, v=v, index_q=index_q, index_k=index_k,
                         cu_seqlens=torch.from_numpy(cu_np).to(device), max_seqlen=int(lens.max()),
                         topk=topk, init_blocks=init_blocks, local_blocks=local_blocks,
                         index_dtype=index_dtype)


def packed_doc_map(batch: int = 2, seq: int = 32768, *, min_len: int = 64, max_len: int = 16384,
                   max_pad: int = 1024, seed: int = 0) -> np.ndarray:
    """int64 [batch, seq] document map: per row, trailing padding P ~ U{0..max_pad};
    document lengths floor(exp(U(ln min_len, ln max_len))) drawn until the real
    length seq - P is filled, the last one clipped to fit; ids 1, 2, ... per row.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    ids = np.zeros((batch, seq), dtype=np.int64)
    for r in range(batch):
        pad = int(rng.integers(0, max_pad + 1))
        real = seq - pad
        pos, doc = 0, 1
        while pos < real:
            L = int(math.floor(math.exp(rng.uniform(math.log(min_len), math.log(max_len)))))
            L = max(1, min(L, real - pos))
            ids[r, pos: pos + L] = doc
            pos += L
            doc += 1
    return ids


def doc_lengths_from_map(ids: np.ndarray) -> list[int]:
    """Run lengths of positive ids in row-major order (input bookkeeping only)."""
    out = []
    for row in np.asarray(ids):
        prev, run = 0, 0
        for x in row:
            x = int(x)
            if x != 0 and x == prev:
                run += 1
            else:
                if prev != 0:
                    out.append(run)
                run = 1 if x != 0 else 0
            prev = x
        if prev != 0:
            out.append(run)
    return out


# ---- the named workloads -------------------------------------------------------

WORKLOADS = {
    "decode_b4_ctx8k_contig": "decode, 4 requests x 8192-token contexts, contiguous cache, bf16 index",
    "decode_b64_ctx4k_64k_paged": "decode, 64 requests, contexts U{4096..65536}, paged caches, bf16 index",
    "prefill_1doc_16k": "prefill, one 16384-token document, bf16 index",
    "prefill_packed_2x32k": "packed prefill, 2 rows x 32768 tokens, log-uniform documents, init=1",
    "decode_b16_ctx128k_paged_e4m3": "decode, 16 requests x 131072-token contexts, paged, E4M3 index",
    "prefill_1doc_16k_e4m3": "prefill, one 16384-token document, E4M3 index",
}


def workload(name: str, *, seed: int = 0, device="cpu", scale_down: int = 1, max_requests: int | None = None):
    """Build a named workload.  ``scale_down`` > 1 shrinks the sizes;
    ``max_requests`` keeps the first requests of a decode batch (small
    profiling cases)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    cut = (lambda x: x[:max_requests]) if max_requests else (lambda x: x)
    if name == "decode_b4_ctx8k_contig":
        L = max(8192 // scale_down, 1)
        return decode_inputs(cut([L] * 4), paged=False, seed=seed, device=device)
    if name == "decode_b64_ctx4k_64k_paged":
        lens = rng.integers(4096, 65536 + 1, size=64)
        lens = np.maximum(lens // scale_down, 1)
        return decode_inputs(cut(lens), paged=True, seed=seed, device=device,
                             max_blocks=(65536 // scale_down + BLOCK - 1) // BLOCK)
    if name == "prefill_1doc_16k":
        return prefill_inputs([max(16384 // scale_down, 1)], seed=seed, device=device)
    if name == "prefill_1doc_16k_e4m3":
        return prefill_inputs([max(16384 // scale_down, 1)], seed=seed, device=device, index_dtype="e4m3")
    if name == "prefill_packed_2x32k":
        ids = packed_doc_map(2, 32768 // scale_down, max_len=max(16384 // scale_down, 64),
                             max_pad=1024 // scale_down, seed=seed)
        lens = doc_lengths_from_map(ids)
        p = prefill_inputs(lens, seed=seed, device=device, init_blocks=1)
        p.doc_ids = torch.from_numpy(ids).to(device)
        return p
    if name == "decode_b16_ctx128k_paged_e4m3":
        L = max(131072 // scale_down, 1)
        return decode_inputs(cut([L] * 16), paged=True, index_dtype="e4m3", seed=seed, device=device)
    raise KeyError(name)
