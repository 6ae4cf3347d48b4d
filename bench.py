"""Benchmark of one MiniMax-M3 block-sparse attention step (score + select + attend).

Default workload: a decode step of 64 requests with contexts U{4096..65536}
over paged K/V and index-K caches (bf16), top-16, init 0, local 1.  One step =
msa_select_blocks_decode + msa_sparse_attend_decode over the whole batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  The device-timed value uses CUDA events on the
launching stream around each step, replayed as one CUDA graph of the two calls;
L2 is flushed (256 MiB written, then 256 MiB read) between steps, outside the
timed events.  Under torchrun each rank runs its own
independent batch (weak scaling, no collective on the data path); the time is
the max over ranks.  ``--impl reference`` times the CPU oracle on this host's
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import msa_synth  # noqa: E402

METRIC = "query tokens/s of score+select+attend; HBM GB/s (decode), TFLOP/s (prefill)"
DEFAULT_WORKLOAD = "decode_b64_ctx4k_64k_paged"
SCALE = 1.0 / math.sqrt(128.0)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ---- algorithmic work per step -------------------------------------------------------

def decode_work(d, q2k, mxfp8=False, fp8_kv=False):
    """(bytes_select, bytes_attend).  Select: the index-K of every scored context
    once (contexts with nb <= topk keep every block and read nothing) plus the
    index queries.  Attend: K and V of every attended key once per KV head (2
    bytes per element, or 1 with ``fp8_kv``), plus q and out (bf16, or with
    ``mxfp8`` one E4M3 byte per element and one scale byte per 32)."""
    lens = d.seq_lens.cpu().numpy().astype(np.int64)
    nb = (lens + 127) // 128
    scored = nb > d.topk
    idx_bytes = 128 if d.index_dtype == "e4m3" else 256
    b_sel = int((lens[scored] * idx_bytes).sum()) + d.batch * 4 * idx_bytes
    q = q2k.cpu().numpy()
    keys = 0
    for g in range(4):
        blk = q[g]
        k = np.minimum(128, lens[:, None] - 128 * blk)
        keys += int(np.where(blk >= 0, k, 0).sum())
    out_bytes = d.batch * 64 * 128 * (1 + 1 / 32 if mxfp8 else 2)
    b_att = int(keys * 2 * 128 * (1 if fp8_kv else 2) + d.batch * 64 * 128 * 2 + out_bytes)
    return b_sel, b_att


# DRAM traffic of the dominant kernel(s) per unit of work, from one ncu capture of a
# smaller case of the same workload, scaled by the units of a full launch.  Set to
# None when the kernels change after the capture.
TRAFFIC = {
    # decode_select_kernel<bf16> + scores, first 16 requests: 147.3 MB DRAM / 143.7 MB algorithmic
    "decode_b64_ctx4k_64k_paged": {"kernel": "select", "per": "algorithmic byte", "value": 1.0246,
                                   "capture": "ncu: decode_select_kernel<0>, first 16 requests of "
                                              "decode_b64_ctx4k_64k_paged"},
}
# bw_attend_kernel, 8192-token document: 0.604 GB DRAM / 462848 entries (scaled by entries)
TRAFFIC_BACKWARD = {
    "prefill_1doc_16k": {"per": "entry", "value": 1306.0,
                         "capture": "ncu: bw_attend_kernel, prefill_1doc_16k at half size"},
}

# The other headline workloads, measured in the same run after the bench workload
# and reported in the line's "workloads" object (one GPU only).
EXTRA_WORKLOADS = ["decode_b4_ctx8k_contig", "prefill_1doc_16k", "prefill_packed_2x32k",
                   "decode_b16_ctx128k_paged_e4m3"]


def prefill_entries(q2k):
    """Selected (query, KV head, block) triples: the units of the block-major attention."""
    return int((q2k >= 0).sum().item())


def prefill_work(p, q2k):
    """(flops_select, flops_attend): causal valid index pairs x 4 heads x 2*128;
    selected causal keys x 16 heads x 4*128 (QK^T and PV)."""
    cu = p.cu_seqlens.cpu().numpy().astype(np.int64)
    lens = np.diff(cu)
    f_sel = float(sum(4 * 2 * 128 * n * (n + 1) // 2 for n in lens))
    q = q2k.cpu().numpy()
    T = p.total_tokens
    doc = np.searchsorted(cu, np.arange(T), side="right") - 1
    pos = np.arange(T) - cu[doc]
    keys = 0
    for g in range(4):
        blk = q[g]
        k = np.minimum(128, pos[:, None] - 128 * blk + 1)
        keys += int(np.where(blk >= 0, k, 0).sum())
    return f_sel, float(keys) * 16 * 4 * 128


# ---- clocks --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- the GPU arm -----------------------------------------------------------------------

def _staging(tensors, device):
    """One pinned host buffer holding copies of `tensors` (each at a 256-byte
    offset), a device buffer of the same size, and device views shaped like
    the tensors: the per-step H2D is one copy."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev = torch.empty(total, dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(tensors, offs):
        nb = t.numel() * t.element_size()
        host[o:o + nb].view(t.dtype).view(t.shape).copy_(t.cpu())
        views.append(dev[o:o + nb].view(t.dtype).view(t.shape))
    return host, dev, views


def run_backward(args, device, config):
    """One step = one msa_sparse_attend_prefill_backward call over the workload
    (dq, dk, dv from q, k, v, q2k, the forward's out and log-sum-exp and a
    seeded grad_out, all resident), replayed from a CUDA graph, L2 flushed
    between steps.  Work: five 128-wide GEMM passes per attended key (S, dP,
    dV, dK, dQ) against the forward's two, so 2.5 x the forward's FLOPs."""
    import block_sparse_attention_08_gb300 as msa
    torch.cuda.set_device(device)
    p = msa_synth.workload(args.workload, seed=args.seed, device=device, scale_down=args.scale_down)
    T = p.total_tokens
    q2k = msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen, topk=p.topk,
                                        init_blocks=p.init_blocks, local_blocks=p.local_blocks)
    lse = torch.empty((T, 64), dtype=torch.float32, device=device)
    out = msa.msa_sparse_attend_prefill(p.q, p.k, p.v, q2k, p.cu_seqlens, p.max_seqlen, scale=SCALE, lse=lse)
    gen = torch.Generator(device="cpu").manual_seed(args.seed + 1)
    dout = torch.randn((T, 64, 128), generator=gen).to(torch.bfloat16).to(device)
    dq = torch.empty_like(p.q)
    dk = torch.empty_like(p.k)
    dv = torch.empty_like(p.v)

    def bwd():
        msa.msa_sparse_attend_prefill_backward(p.q, p.k, p.v, q2k, p.cu_seqlens, p.max_seqlen, out, lse, dout,
                                               scale=SCALE, dq=dq, dk=dk, dv=dv)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    for _ in range(args.warmup):
        bwd()
    torch.cuda.synchronize()
    run = bwd
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                bwd()
        stream.wait_stream(cap)
        run = g.replay
        run()
        torch.cuda.synchronize()
    hbm_peak, tf_peak, peak_src = _peaks()
    ms_all = []
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        for i in range(args.steps):
            flush.fill_(i & 255)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run()
            b.record(stream)
            b.synchronize()
            ms_all.append(a.elapsed_time(b))
    ms = sum(ms_all) / len(ms_all)
    _, f_att = prefill_work(p, q2k)
    flop = 2.5 * f_att
    tf = flop / (ms * 1e-3) / 1e12
    tr = TRAFFIC_BACKWARD.get(args.workload) if args.scale_down == 1 else None
    traffic = round(tr["value"] * prefill_entries(q2k)) if tr else None
    config.update({"pass": "attention backward (dq, dk, dv)", "queries_per_step": T,
                   "timing": "eager C-ABI call" if args.no_graph else "CUDA-graph replay of the C-ABI call",
                   "l2": "flushed between steps (256 MiB write, outside the timed events)"})
    return {"metric": "prefill attention backward: query tokens/s; TFLOP/s", "value": round(T / (ms * 1e-3), 1),
            "unit": "query tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": config,
            "roofline": {"bound": "tensor", "kernel": "msa_sparse_attend_prefill_backward (bucketing, "
                         "bw_rowdot_kernel, bw_attend_kernel, bw_to_bf16_kernel)", "achieved": round(tf, 2),
                         "peak": tf_peak, "unit": "TFLOP/s", "frac": round(tf / tf_peak, 4), "traffic": traffic,
                         "traffic_source": tr["capture"] + " (scaled by entries)" if tr else None,
                         "flop": flop, "peak_source": peak_src + " bf16_tflops (burst)"},
            "gpu_launches": 9 * args.steps, "clocks": clk.summary()}


def run_produce(args, device, config):
    """One step = one index-producer call over the workload (C ABI
    msa_index_produce_prefill for a prefill workload: index Q and K of every
    token normalised and stored in the index dtype, the keys also inserted
    into a paged cache; msa_index_produce_decode for a decode workload: each
    request's new index Q and key), replayed from a CUDA graph, L2 flushed
    between steps.  Bytes: the bf16 inputs read once and the outputs written
    once (the HBM roofline of a streaming kernel)."""
    import block_sparse_attention_08_gb300 as msa
    torch.cuda.set_device(device)
    inp = msa_synth.workload(args.workload, seed=args.seed, device=device, scale_down=args.scale_down)
    gen = torch.Generator(device=device).manual_seed(args.seed + 7)
    e4m3 = "e4m3" in args.workload
    esz = 1 if e4m3 else 2
    if args.workload.startswith("prefill"):
        T = inp.total_tokens
        iq = torch.randn((T, 4, 128), generator=gen, device=device).to(torch.bfloat16)
        ik = torch.randn((T, 1, 128), generator=gen, device=device).to(torch.bfloat16)
        dt = torch.float8_e4m3fn if e4m3 else torch.bfloat16
        qo = torch.empty((T, 4, 128), dtype=dt, device=device)
        ko = torch.empty((T, 1, 128), dtype=dt, device=device)
        cu = inp.cu_seqlens
        docs = cu.shape[0] - 1
        nbs = ((cu[1:] - cu[:-1] + 127) // 128).cpu()
        mb = int(nbs.max())
        pages = int(nbs.sum())
        perm = torch.randperm(pages, generator=torch.Generator().manual_seed(args.seed)).to(torch.int32)
        pt = torch.full((docs, mb), -1, dtype=torch.int32)
        o = 0
        for d in range(docs):
            pt[d, : nbs[d]] = perm[o: o + nbs[d]]
            o += int(nbs[d])
        pt = pt.to(device)
        cache = torch.empty((pages * 128, 1, 128), dtype=dt, device=device)

        def call():
            msa.msa_index_produce_prefill(iq, ik, cu, index_dtype="e4m3" if e4m3 else "bf16", index_k_cache=cache,
                                          page_table=pt, q_out=qo, k_out=ko)
        n_q = T
        nbytes = T * 5 * 128 * 2 + T * 5 * 128 * esz + T * 128 * esz
    else:
        d = inp
        B = d.batch
        iq = torch.randn((B, 4, 128), generator=gen, device=device).to(torch.bfloat16)
        ik = torch.randn((B, 1, 128), generator=gen, device=device).to(torch.bfloat16)
        qo = torch.empty((B, 4, 128), dtype=d.index_k_cache.dtype, device=device)

        def call():
            msa.msa_index_produce_decode(iq, ik, d.index_k_cache, d.seq_lens, page_table=d.page_table,
                                         cu_seqlens_k=d.cu_seqlens_k, max_blocks=d.max_blocks, q_out=qo)
        n_q = B
        nbytes = B * 5 * 128 * 2 + B * 5 * 128 * esz
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    run = call
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                call()
        stream.wait_stream(cap)
        run = g.replay
        run()
        torch.cuda.synchronize()
    hbm_peak, _, peak_src = _peaks()
    ms_all = []
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        for i in range(args.steps):
            flush.fill_(i & 255)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run()
            b.record(stream)
            b.synchronize()
            ms_all.append(a.elapsed_time(b))
    ms = sum(ms_all) / len(ms_all)
    gbs = nbytes / (ms * 1e-3) / 1e9
    config.update({"pass": "index producer (L2 norm, storage cast, index-K cache insertion)",
                   "queries_per_step": n_q, "timing": "CUDA-graph replay of the C-ABI call",
                   "l2": "flushed between steps (256 MiB write, outside the timed events)"})
    return {"metric": "index producer: query tokens/s; HBM GB/s", "value": round(n_q / (ms * 1e-3), 1),
            "unit": "query tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "e4m3" if e4m3 else "bf16",
            "data": "synthetic", "config": config,
            "roofline": {"bound": "hbm", "kernel": "index_produce_kernel", "achieved": round(gbs, 1),
                         "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": None,
                         "bytes": nbytes, "peak_source": peak_src + " hbm_gbs (copy, burst)"},
            "gpu_launches": args.steps, "clocks": clk.summary()}


def run_gpu(args, rank, world, device, name=None, steps=None):
    import block_sparse_attention_08_gb300 as msa
    torch.cuda.set_device(device)
    name = name or args.workload
    steps = steps or args.steps
    inp = msa_synth.workload(name, seed=args.seed + rank, device=device, max_requests=args.requests,
                            scale_down=args.scale_down)
    decode = name.startswith("decode")
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    clean = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=device)
    sink = torch.empty((), dtype=torch.float32, device=device)

    def flush_l2(i):
        # write 256 MiB (evicts the step's data from the 129 MB L2), then read
        # another 256 MiB so the L2 holds clean lines: the next step starts with
        # a cold L2 and no pending write-backs
        flush.fill_(i & 255)
        torch.sum(clean, dim=0, out=sink)
    hbm_peak, tf_peak, peak_src = _peaks()

    if decode:
        d = inp
        kw = dict(page_table=d.page_table, cu_seqlens_k=d.cu_seqlens_k, max_blocks=d.max_blocks)
        q2k = torch.empty((4, d.batch, d.topk), dtype=torch.int32, device=device)
        out = torch.empty((d.batch, 64, 128), dtype=torch.bfloat16, device=device)

        def sel():
            msa.msa_select_blocks_decode(d.index_q, d.index_k_cache, d.seq_lens, topk=d.topk,
                                         init_blocks=d.init_blocks, local_blocks=d.local_blocks, q2k=q2k, **kw)

        if args.fp8_kv:
            # the main K / V caches as E4M3 (unit scales): the attention streams half the bytes
            d.k_cache = d.k_cache.to(torch.float8_e4m3fn)
            d.v_cache = d.v_cache.to(torch.float8_e4m3fn)

            def att():
                msa.msa_sparse_attend_decode_fp8kv(d.q, d.k_cache, d.v_cache, q2k, d.seq_lens, scale=SCALE, out=out,
                                                   **kw)
            outs = [out]
        elif args.mxfp8:
            out_q = torch.empty((d.batch, 64 * 128), dtype=torch.uint8, device=device)
            out_sc = torch.empty((d.batch, 64 * 128 // 32), dtype=torch.uint8, device=device)

            def att():
                msa.msa_sparse_attend_decode_mxfp8(d.q, d.k_cache, d.v_cache, q2k, d.seq_lens, scale=SCALE,
                                                   out_q=out_q, out_scale=out_sc, **kw)
            outs = [out_q, out_sc]
        else:
            def att():
                msa.msa_sparse_attend_decode(d.q, d.k_cache, d.v_cache, q2k, d.seq_lens, scale=SCALE, out=out,
                                             **kw)
            outs = [out]
        n_queries = d.batch
    else:
        p = inp
        q2k = torch.empty((4, p.total_tokens, p.topk), dtype=torch.int32, device=device)
        out = torch.empty((p.total_tokens, 64, 128), dtype=torch.bfloat16, device=device)

        def sel():
            msa.msa_select_blocks_prefill(p.index_q, p.index_k, p.cu_seqlens, p.max_seqlen, topk=p.topk,
                                          init_blocks=p.init_blocks, local_blocks=p.local_blocks, q2k=q2k)

        def att():
            msa.msa_sparse_attend_prefill(p.q, p.k, p.v, q2k, p.cu_seqlens, p.max_seqlen, scale=SCALE, out=out)
        outs = [out]
        n_queries = p.total_tokens

    for _ in range(args.warmup):
        sel()
        att()
        flush_l2(1)
    torch.cuda.synchronize()
    work = decode_work(inp, q2k, args.mxfp8, args.fp8_kv) if decode else prefill_work(inp, q2k)
    entries = 0 if decode else prefill_entries(q2k)

    # The timed steps replay a CUDA graph of the step, the two C-ABI calls
    # (captured once, same buffers, as a serving engine replays its decode or
    # prefill step), so host submission cost does not leak into device time.
    # A second pass replays one graph per call, timed call by call, for the
    # per-kernel figures.
    def run_step():
        sel()
        att()
    run_sel, run_att = sel, att
    if not args.no_graph:
        g_sel, g_att, g_step = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g_sel, stream=cap):
                sel()
            with torch.cuda.graph(g_att, stream=cap):
                att()
            with torch.cuda.graph(g_step, stream=cap):
                sel()
                att()
        stream.wait_stream(cap)
        run_sel, run_att, run_step = g_sel.replay, g_att.replay, g_step.replay
        for _ in range(2):
            run_sel()
            run_att()
            run_step()
        torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        for i in range(steps):
            flush_l2(i)
            evs[i][0].record(stream)
            run_step()
            evs[i][1].record(stream)
        for i in range(steps):
            flush_l2(i)
            ev[i][0].record(stream)
            run_sel()
            ev[i][1].record(stream)
            run_att()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_sel = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
    t_att = [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)]
    step_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(steps)]
    ms = sum(step_ms) / steps

    # the same step as eager C-ABI calls (no graph), same L2 flush between steps
    eager_ms = None
    if not args.no_graph:
        ee = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            flush_l2(i)
            ee[i][0].record(stream)
            sel()
            att()
            ee[i][1].record(stream)
        torch.cuda.synchronize()
        eager_ms = sum(ee[i][0].elapsed_time(ee[i][1]) for i in range(steps)) / steps

    # end to end through the public API with host buffers (pinned), per step:
    # H2D of the step's inputs, D2H of the output.  Decode: the new queries,
    # lengths and page table (the K/V and index-K caches are resident state);
    # prefill: every input tensor.  The inputs sit in two pinned staging
    # buffers, one copy each: what the select call reads goes first on the
    # launching stream; what only the attention reads goes on a side stream
    # and overlaps the select call.  The step (copies, the two calls, the D2H
    # of the output) is replayed from a CUDA graph unless --no-graph.
    if decode:
        early = [d.index_q, d.seq_lens, d.page_table if d.page_table is not None else d.cu_seqlens_k]
        late = [d.q]
    else:
        early = [p.index_q, p.index_k, p.cu_seqlens]
        late = [p.q, p.k, p.v]
    h_early, d_early, dv_early = _staging(early, device)
    h_late, d_late, dv_late = _staging(late, device)
    h_outs = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    h2d = sum(x.numel() * x.element_size() for x in early + late)
    d2h = sum(h.numel() * h.element_size() for h in h_outs)
    side = torch.cuda.Stream(device)

    def e2e_step():
        cur = torch.cuda.current_stream()
        side.wait_stream(cur)
        d_early.copy_(h_early, non_blocking=True)
        with torch.cuda.stream(side):
            d_late.copy_(h_late, non_blocking=True)
        if decode:
            diq, dsl, dpt = dv_early
            (dq,) = dv_late
            kw2 = dict(page_table=dpt) if d.page_table is not None else dict(cu_seqlens_k=dpt)
            msa.msa_select_blocks_decode(diq, d.index_k_cache, dsl, topk=d.topk, init_blocks=d.init_blocks,
                                         local_blocks=d.local_blocks, q2k=q2k, max_blocks=d.max_blocks, **kw2)
            cur.wait_stream(side)
            if args.fp8_kv:
                msa.msa_sparse_attend_decode_fp8kv(dq, d.k_cache, d.v_cache, q2k, dsl, scale=SCALE, out=out,
                                                   max_blocks=d.max_blocks, **kw2)
            elif args.mxfp8:
                msa.msa_sparse_attend_decode_mxfp8(dq, d.k_cache, d.v_cache, q2k, dsl, scale=SCALE, out_q=outs[0],
                                                   out_scale=outs[1], max_blocks=d.max_blocks, **kw2)
            else:
                msa.msa_sparse_attend_decode(dq, d.k_cache, d.v_cache, q2k, dsl, scale=SCALE, out=out,
                                             max_blocks=d.max_blocks, **kw2)
        else:
            iq_, ik_, cu_ = dv_early
            q_, k_, v_ = dv_late
            msa.msa_select_blocks_prefill(iq_, ik_, cu_, p.max_seqlen, topk=p.topk, init_blocks=p.init_blocks,
                                          local_blocks=p.local_blocks, q2k=q2k)
            cur.wait_stream(side)
            msa.msa_sparse_attend_prefill(q_, k_, v_, q2k, cu_, p.max_seqlen, scale=SCALE, out=out)
        for h, o in zip(h_outs, outs):
            h.copy_(o, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    run_e2e = e2e_step
    if not args.no_graph:
        g_e2e = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g_e2e, stream=cap):
                e2e_step()
        stream.wait_stream(cap)
        run_e2e = g_e2e.replay
        run_e2e()
        torch.cuda.synchronize()
    e_ms = []
    for i in range(steps):
        flush_l2(i)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run_e2e()
        b.record(stream)
        b.synchronize()
        e_ms.append(a.elapsed_time(b))
    return dict(ms=ms, step_ms=step_ms, eager_ms=eager_ms, sel_ms=sum(t_sel) / len(t_sel), att_ms=sum(t_att) / len(t_att),
                e2e_ms=sum(e_ms) / len(e_ms), n_queries=n_queries, work=work, entries=entries, h2d=h2d, d2h=d2h,
                clocks=clk.summary(), decode=decode, hbm_peak=hbm_peak, tf_peak=tf_peak, peak_src=peak_src,
                inputs=inp, q2k=q2k, steps=steps, name=name)


_CPU_INPUTS: dict = {}


def _host_copy(inp):
    """The same workload object with every tensor moved to host memory."""
    import dataclasses
    return dataclasses.replace(inp, **{f.name: getattr(inp, f.name).cpu() for f in dataclasses.fields(inp)
                                       if isinstance(getattr(inp, f.name), torch.Tensor)})


def cpu_baseline(name, seed, budget_s=15.0, inputs=None, gpu_q2k=None):
    """The oracle, as it stands, on this host's cores over a bounded sample:
    whole requests (decode) or random query tokens (prefill), until the
    budget is spent.  With ``inputs`` (the GPU run's own inputs, on the host)
    and ``gpu_q2k`` (the GPU run's q2k), the oracle's selection of the sampled
    rows is also compared with the GPU's: rows checked, rows that differ, and
    the rows the oracle finds to be near ties (exempt), reported, not hidden."""
    import oracle
    oracle.build()
    if inputs is None:
        key = (name, seed)
        if key not in _CPU_INPUTS:
            _CPU_INPUTS[key] = msa_synth.workload(name, seed=seed, device="cpu")
        inp = _CPU_INPUTS[key]
    else:
        inp = inputs
    cores = os.cpu_count()
    t0 = time.time()
    done = 0
    checked = differ = exempt = 0
    gq = None if gpu_q2k is None else gpu_q2k.cpu().numpy()
    if name.startswith("decode"):
        d = inp
        B = d.batch
        chunk = max(1, min(B, cores))
        while done < B and time.time() - t0 < budget_s:
            req = np.arange(done, min(B, done + chunk), dtype=np.int64)
            q2k, gap = oracle.select_decode(d.index_q, d.index_k_cache, d.seq_lens, page_table=d.page_table,
                                            cu_seqlens_k=d.cu_seqlens_k, requests=req, topk=d.topk,
                                            init=d.init_blocks, local=d.local_blocks)
            if d.k_cache.dtype == torch.float8_e4m3fn:
                oracle.attend_decode_fp8(d.q, d.k_cache, d.v_cache, d.seq_lens, q2k, SCALE, page_table=d.page_table,
                                         cu_seqlens_k=d.cu_seqlens_k, requests=req)
            else:
                oracle.attend_decode(d.q, d.k_cache, d.v_cache, d.seq_lens, q2k, SCALE, page_table=d.page_table,
                                     cu_seqlens_k=d.cu_seqlens_k, requests=req)
            if gq is not None:
                checked += q2k.shape[0] * q2k.shape[1]
                differ += int((gq[:, req] != q2k).any(axis=2).sum())
                exempt += int(oracle.exempt_rows(gap).sum())
            done += len(req)
        sample = f"{done} of {B} requests of {name}, whole select+attend per request"
    else:
        p = inp
        T = p.total_tokens
        perm = np.random.default_rng(seed).permutation(T)
        chunk = max(1, cores)
        while done < T and time.time() - t0 < budget_s:
            tok = np.sort(perm[done: done + chunk]).astype(np.int64)
            q2k, gap = oracle.select_prefill(p.index_q, p.index_k, p.cu_seqlens, tok, topk=p.topk,
                                             init=p.init_blocks, local=p.local_blocks)
            oracle.attend_prefill(p.q, p.k, p.v, p.cu_seqlens, tok, q2k, SCALE)
            if gq is not None:
                checked += q2k.shape[0] * q2k.shape[1]
                differ += int((gq[:, tok] != q2k).any(axis=2).sum())
                exempt += int(oracle.exempt_rows(gap).sum())
            done += len(tok)
        sample = f"{done} random query tokens of {T} of {name}"
    dt = time.time() - t0
    out = {"value": round(done / dt, 3), "unit": "query tokens/s", "cores": cores, "kind": "oracle",
           "sample": sample, "seconds": round(dt, 2)}
    if gq is not None:
        out.update({"q2k_rows_checked": checked, "q2k_rows_differing": differ, "q2k_exempt_rows": exempt,
                    "q2k_note": "(query, KV head) rows of the sample, GPU q2k against the oracle on the GPU "
                                "run's own inputs; exempt = the oracle's k-th and (k+1)-th scores within "
                                "1e-5 relative"})
    return out


def max_over_ranks(values, world):
    """Element-wise max of per-rank timings (host-side gloo collective; the data
    path itself has no collective)."""
    if world <= 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(msa_synth.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager C-ABI calls instead of graph replays")
    ap.add_argument("--scale-down", type=int, default=1,
                    help="divide the workload's lengths by this factor (small profiling cases)")
    ap.add_argument("--requests", type=int, default=None,
                    help="keep only the first N requests of a decode workload (small profiling cases)")
    ap.add_argument("--mxfp8", action="store_true",
                    help="decode: emit the attention output as MXFP8 (E4M3 + E8M0 scales) instead of bf16")
    ap.add_argument("--fp8-kv", action="store_true",
                    help="decode: main K / V caches as E4M3 (msa_sparse_attend_decode_fp8kv, unit scales)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other headline workloads (measured after the bench workload at one GPU)")
    ap.add_argument("--produce", action="store_true",
                    help="time the index producer (norm, storage cast, cache insertion) on the workload's shapes")
    ap.add_argument("--backward", action="store_true",
                    help="time the attention backward of a prefill workload instead of the forward step")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    unit = "query tokens/s"
    config = {"workload": args.workload, "desc": msa_synth.WORKLOADS[args.workload], "seed": args.seed}
    if args.requests:
        config["requests"] = args.requests
    if args.mxfp8 or args.fp8_kv:
        if not args.workload.startswith("decode") or (args.mxfp8 and args.fp8_kv):
            raise SystemExit("--mxfp8 and --fp8-kv apply (one at a time) to the decode attention")
        if args.mxfp8:
            config["output"] = "MXFP8: E4M3 values + one E8M0 scale per 32 elements"
        else:
            config["kv_cache"] = "E4M3 main K / V caches (unit scales)"
    if args.scale_down > 1:
        config["scale_down"] = args.scale_down

    if args.produce:
        if args.impl != "gb300":
            raise SystemExit("--produce times the index producer of this library")
        print(json.dumps(run_produce(args, torch.device("cuda", local), config)))
        return

    if args.backward:
        if args.impl != "gb300" or not args.workload.startswith("prefill"):
            raise SystemExit("--backward times the prefill attention backward of this library")
        print(json.dumps(run_backward(args, torch.device("cuda", local), config)))
        return

    if args.impl == "reference":
        if rank == 0:
            for _ in range(args.warmup):
                cpu_baseline(args.workload, args.seed, budget_s=1.0)
            vals, info = [], None
            for _ in range(args.steps):
                info = cpu_baseline(args.workload, args.seed, budget_s=6.0)
                vals.append(info["value"])
            v = sum(vals) / len(vals)
            info["value"] = v
            inp = _CPU_INPUTS[(args.workload, args.seed)]
            per_step = inp.batch if args.workload.startswith("decode") else inp.total_tokens
            config["queries_per_step"] = per_step
            line = {"impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
                    "steps": args.steps, "warmup": args.warmup,
                    # a whole step of the workload at the sample's rate
                    "ms_per_step": round(per_step / v * 1e3, 4) if v > 0 else None,
                    "higher_is_better": True, "scaling": "weak",
                    "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                    "cpu_baseline": info,
                    "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
            print(json.dumps(line))
        if world > 1:
            torch.distributed.barrier()
        return

    device = torch.device("cuda", local)
    res = run_gpu(args, rank, world, device)
    ms, e2e_ms = max_over_ranks([res["ms"], res["e2e_ms"]], world)
    if rank != 0:
        return
    summ = summarize(res, args, ms, e2e_ms, world)
    config.update({"queries_per_step": res["n_queries"],
                   "timing": ("eager C-ABI calls" if args.no_graph else
                              "CUDA-graph replay of the step (the two C-ABI calls in one graph); per-kernel "
                              "figures from a second pass with one graph per call, timed call by call"),
                   "l2": "flushed between steps (256 MiB write + 256 MiB read, outside the timed events)",
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu"})
    line = {"metric": METRIC, "value": summ["value"], "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "step_ms_percentiles": _percentiles(res["step_ms"]),
            "eager_ms_per_step": round(res["eager_ms"], 4) if res["eager_ms"] is not None else None,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": summ["dtype"], "data": "synthetic", "config": config,
            "roofline": summ["roofline"], "e2e": summ["e2e"],
            "gpu_launches": launches_per_step(res["decode"]) * args.steps, "clocks": res["clocks"]}
    # The other headline workloads, one GPU: each measured the same way (fewer steps), reported with its
    # step time, roofline fraction and end-to-end figure.  They run before the CPU baseline: the oracle's
    # run and its host copies of the inputs slowed the host <-> device copies measured after them by
    # about half (prefill e2e 7.6 against 5.0 ms).
    if world == 1 and not (args.no_workloads or args.mxfp8 or args.fp8_kv) and args.requests is None and \
            args.scale_down == 1:
        extra = {}
        for name in EXTRA_WORKLOADS:
            if name == args.workload:
                continue
            torch.cuda.empty_cache()
            r = run_gpu(args, 0, 1, device, name=name, steps=min(args.steps, 10))
            sm = summarize(r, args, r["ms"], r["e2e_ms"], 1)
            extra[name] = {"desc": msa_synth.WORKLOADS[name], "steps": r["steps"], "warmup": args.warmup,
                           "ms_per_step": round(r["ms"], 4), "value": sm["value"], "unit": unit,
                           "dtype": sm["dtype"], "roofline": sm["roofline"], "e2e": sm["e2e"],
                           "gpu_launches": launches_per_step(r["decode"]) * r["steps"], "clocks": r["clocks"]}
            del r
        line["workloads"] = extra
    if not args.no_cpu_baseline and world == 1:
        inputs, gpu_q2k = _host_copy(res["inputs"]), res["q2k"]
        line["cpu_baseline"] = cpu_baseline(args.workload, args.seed, inputs=inputs, gpu_q2k=gpu_q2k)
        del inputs
    print(json.dumps(line))


def _percentiles(xs):
    """p10 / p50 / p90 of the timed steps (ms), nearest rank."""
    v = sorted(xs)
    pick = lambda q: round(v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))], 4)
    return {"p10": pick(0.1), "p50": pick(0.5), "p90": pick(0.9)}


def launches_per_step(decode):
    """The library's kernels in one step: decode scorer, top-k and attention;
    prefill plan and scorer, then geometry, count, scan, tiles, scatter, the
    tensor-core attention's two phases and the normalisation."""
    return 3 if decode else 10


# Nominal figures of the part, reported beside the measured peaks (the fractions
# against the measured copy and GEMM rates are the ones the roofline uses).
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0

def summarize(res, args, ms, e2e_ms, world):
    """value, dtype, roofline (the dominant call) and e2e of one measured workload."""
    unit = "query tokens/s"
    name = res["name"]
    value = res["n_queries"] * world / (ms * 1e-3)
    e2e = res["n_queries"] * world / (e2e_ms * 1e-3)
    dom = "select" if res["sel_ms"] >= res["att_ms"] else "attend"
    full = args.requests is None and args.scale_down == 1
    if res["decode"]:
        b_sel, b_att = res["work"]
        sel_r = b_sel / (res["sel_ms"] * 1e-3) / 1e9
        att_r = b_att / (res["att_ms"] * 1e-3) / 1e9
        ach = sel_r if dom == "select" else att_r
        tr = TRAFFIC.get(name) if full else None
        traffic = None
        if tr and tr["kernel"] == dom:
            traffic = round(tr["value"] * (b_sel if dom == "select" else b_att))
        roof = {"bound": "hbm",
                "kernel": ("msa_select_blocks_decode (decode_select_kernel + decode_topk_kernel)" if dom == "select"
                           else "msa_sparse_attend_decode (sparse_attend_kernel)" if not args.fp8_kv
                           else "msa_sparse_attend_decode_fp8kv (sparse_attend_kernel<1>)"),
                "achieved": round(ach, 1), "peak": res["hbm_peak"], "unit": "GB/s",
                "frac": round(ach / res["hbm_peak"], 4), "traffic": traffic,
                "traffic_source": tr["capture"] + " (scaled by algorithmic bytes)" if traffic else None,
                "peak_source": res["peak_src"] + " hbm_gbs (copy, burst)",
                "nominal": {"peak": NOMINAL_HBM_GBS, "frac": round(ach / NOMINAL_HBM_GBS, 4),
                            "source": "GB300 HBM3e nominal bandwidth"},
                "per_kernel": {"select": {"ms": round(res["sel_ms"], 4), "bytes": b_sel, "GB/s": round(sel_r, 1)},
                               "attend": {"ms": round(res["att_ms"], 4), "bytes": b_att, "GB/s": round(att_r, 1)},
                               "step_GB/s": round((b_sel + b_att) / (ms * 1e-3) / 1e9, 1),
                               "step_frac": round((b_sel + b_att) / (ms * 1e-3) / 1e9 / res["hbm_peak"], 4)}}
        dtype = ("bf16" if "e4m3" not in name else "e4m3-index/bf16") if not args.fp8_kv else \
            ("bf16-index/e4m3-kv" if "e4m3" not in name else "e4m3-index/e4m3-kv")
    else:
        fp8_index = "e4m3" in name
        f_sel, f_att = res["work"]
        sel_r = f_sel / (res["sel_ms"] * 1e-3) / 1e12
        att_r = f_att / (res["att_ms"] * 1e-3) / 1e12
        ach = sel_r if dom == "select" else att_r
        tr = TRAFFIC.get(name) if full else None
        traffic = None
        if tr and tr["kernel"] == dom:
            traffic = round(tr["value"] * res["entries"])
        roof = {"bound": "tensor",
                "kernel": ("msa_select_blocks_prefill (prefill_plan_kernel + prefill_select_kernel)" if dom == "select"
                           else "msa_sparse_attend_prefill (bucketing, bm_attend_kernel reference and "
                                "accumulate phases, bm_norm_kernel)"),
                "achieved": round(ach, 2), "peak": res["tf_peak"], "unit": "TFLOP/s",
                "frac": round(ach / res["tf_peak"], 4), "traffic": traffic,
                "traffic_source": tr["capture"] + " (scaled by entries)" if traffic else None,
                "peak_source": res["peak_src"] + " bf16_tflops (burst)",
                "nominal": {"peak": NOMINAL_BF16_TFLOPS, "frac": round(ach / NOMINAL_BF16_TFLOPS, 4),
                            "source": "GB300 dense bf16 nominal rate"},
                "per_kernel": {"select": {"ms": round(res["sel_ms"], 4), "flop": f_sel, "TFLOP/s": round(sel_r, 2),
                                          # an E4M3 index runs the scorer's MMAs on the fp8 pipe: its peak is
                                          # the measured bf16 one times the nominal dense ratio (4.5 / 2.25)
                                          "peak_TFLOP/s": round(res["tf_peak"] * (2.0 if fp8_index else 1.0), 1),
                                          "frac": round(sel_r / (res["tf_peak"] * (2.0 if fp8_index else 1.0)), 4)},
                               "attend": {"ms": round(res["att_ms"], 4), "flop": f_att, "TFLOP/s": round(att_r, 2)},
                               "step_TFLOP/s": round((f_sel + f_att) / (ms * 1e-3) / 1e12, 2),
                               "step_frac": round((f_sel + f_att) / (ms * 1e-3) / 1e12 / res["tf_peak"], 4)}}
        dtype = "e4m3-index/bf16" if fp8_index else "bf16"
    e2e_d = {"value": round(e2e, 1), "unit": unit, "h2d_bytes_per_step": res["h2d"],
             "d2h_bytes_per_step": res["d2h"], "ms_per_step": round(e2e_ms, 4),
             "method": ("pinned staging buffers, one H2D copy for the select inputs and one (side stream, "
                        "overlapping the select call) for the attention inputs, the two C-ABI calls, "
                        "D2H of the output; " + ("eager" if args.no_graph else "replayed as one CUDA graph"))}
    return {"value": round(value, 1), "dtype": dtype, "roofline": roof, "e2e": e2e_d}


if __name__ == "__main__":
    main()
