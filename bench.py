#!/usr/bin/env python
"""Benchmark of the block-sparse attention hot path on GB300.

One step = one pass of the prefill path over one batch: block summaries,
router (scores + selection), worklist, sparse attention.  The headline line is
the 128k-token prompt (n=131072, H=64 / H_kv=8, d=128, b=128, top-16 + sink +
diagonal), the largest single-GPU workload; its value is the selected-tile
TFLOP/s of the whole step.  The same line carries, per prefill workload (tiny,
32k prompt, variable-length batch, 128k prompt), the step time, router ms,
stage times, the roofline of the attention kernel (tensor), of the router
(HBM and tensor) and of the summaries kernel (HBM), and the speedup over the
same kernel at density 1; the paged-decode KV GB/s on the 64-request decode
workload; an end-to-end number from host buffers; the float64 oracle timed on
the host cores; and legs run outside the timed loop: router quality
(coverage, token recall against the dense top-t teacher, planted recall), the
backward pass, and the 32k prompt as a chunked prefill over a paged KV cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload long|prompt|varlen|tiny] [--configs tiny,prompt,varlen|none]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

NCORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(NCORES))

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-sparse attn TFLOP/s on selected tiles + router ms; decode KV GB/s"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "dynamic_block_sparse_mean_gb300", "csrc")
L2_BYTES = 129 * 1024 * 1024
WORKLOAD_KEYS = ("tiny", "prompt", "varlen", "long")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="long", choices=list(WORKLOAD_KEYS),
                    help="the headline workload (default: the 128k prompt, the largest)")
    ap.add_argument("--configs", default="tiny,prompt,varlen",
                    help="other prefill workloads timed into the same line ('none': skip)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="cut a fixed-length prefill workload to its first N tokens (small "
                         "cases for profiler captures; the name gets a _firstN suffix)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward leg")
    ap.add_argument("--no-chunked", action="store_true", help="skip the chunked-prefill leg")
    ap.add_argument("--no-quality", action="store_true",
                    help="skip the coverage / planted-recall / density-1 leg")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the paged decode (a diagnostic line, e.g. for profiling)")
    ap.add_argument("--decode-reqs", type=int, default=None,
                    help="run the decode workload on its first N requests (default: all)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- ranks


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int, device=None):
    if world > 1:
        if device is not None and torch.distributed.get_backend() == "nccl":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()


def reduce_max_sum(world: int, ms: float, units: float, device=None):
    """Slowest rank's time and the units all ranks processed."""
    if world == 1:
        return ms, units
    dev = device if (device is not None and torch.distributed.get_backend() == "nccl") else "cpu"
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.sel = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.sel = str(device_index)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons, n = [], None, set(), 0
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            n += 1
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": n}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(kernel: str, workload: str):
    """DRAM read + write bytes per launch of `kernel` on `workload` from the
    committed ncu record (profiles/dram_traffic.json), if the kernel's source file
    is unchanged since the counters were taken (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    for rec in json.load(open(TRAFFIC_FILE)).get("records", []):
        if rec.get("kernel") != kernel or rec.get("workload") != workload:
            continue
        src = os.path.join(CSRC, rec["source"])
        if not os.path.exists(src):
            return None
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        return float(rec["dram_bytes_per_launch"]) if sha == rec.get("source_sha256") else None
    return None


# ---------------------------------------------------------------- workloads


def prefill_workload(name: str, tokens: int | None = None):
    import dataclasses

    from dynamic_block_sparse_mean_gb300 import workloads as W
    table = {"tiny": W.TINY, "prompt": W.PROMPT_32K, "varlen": W.VARLEN_256K, "long": W.LONG_128K}
    w = table[name]
    if tokens is not None and w.seqlen is not None and tokens < w.seqlen:
        w = dataclasses.replace(w, seqlen=tokens, name=f"{w.name}_first{tokens}")
    return w


def to_dev_bf16(a: np.ndarray, device):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def bench_prefill(w, steps, warmup, device, world, sampler):
    import dynamic_block_sparse_mean_gb300 as bsa
    from dynamic_block_sparse_mean_gb300 import accounting, synth

    x = synth.make_prefill(w)
    q, k, v = (to_dev_bf16(a, device) for a in (x.q, x.k, x.v))
    plan = bsa.PrefillPlan(x.cu_seqlens, w.num_heads, w.num_kv_heads, w.head_dim, w.block,
                           bsa.RouteParams(w.mode, w.k_max, w.k_min, w.tau_delta, w.force_sink),
                           device=device)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    # Inputs smaller than twice the L2 would be served from it on repeated steps:
    # then every step is preceded by a write of a buffer larger than the L2.
    flush = (torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
             if in_bytes < 2 * L2_BYTES else None)
    for _ in range(max(3, warmup)):
        plan.run(q, k, v)
    torch.cuda.synchronize(device)
    bsa.check_status(plan.status)

    barrier(world, device)
    torch.cuda.synchronize(device)
    sampler.start()
    if flush is None:
        # The timed loop: whole steps back to back, events only around the loop (an
        # event between two launches would also cut the programmatic dependent launch
        # that lets each kernel's set-up overlap its predecessor).
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for s in range(steps):
            plan.run(q, k, v)
        t1.record()
        torch.cuda.synchronize(device)
        total_ms = t0.elapsed_time(t1)
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for s in range(steps):
            flush.zero_()
            ev[s][0].record()
            plan.run(q, k, v)
            ev[s][1].record()
        torch.cuda.synchronize(device)
        total_ms = sum(a.elapsed_time(b_) for a, b_ in ev)
    clocks = sampler.stop()
    barrier(world, device)
    bsa.check_status(plan.status)
    # Stage breakdown: a second loop with events between the ABI calls.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for s in range(steps):
        e = ev[s]
        if flush is not None:
            flush.zero_()
        e[0].record()
        plan.summaries(k)
        e[1].record()
        plan.select(q)
        e[2].record()
        plan.worklist()
        e[3].record()
        plan.attend(q, k, v)
        e[4].record()
    torch.cuda.synchronize(device)
    bsa.check_status(plan.status)
    stage = lambda a, b_: statistics.mean(ev[s][a].elapsed_time(ev[s][b_]) for s in range(steps))  # noqa: E731
    st = {"summaries": stage(0, 1), "route": stage(1, 2), "worklist": stage(2, 3),
          "attention": stage(3, 4)}
    counts = plan.counts.cpu().numpy()
    J = plan.J.cpu().numpy()
    G = w.num_heads // w.num_kv_heads
    T = int(x.cu_seqlens[-1])
    flops = accounting.attention_tile_flops(counts, G, w.block, w.head_dim)
    eff = accounting.effective_pairs(J, counts, x.cu_seqlens, w.block, G) * 4.0 * w.head_dim
    tiles = counts[counts > 0]
    launches = sum(bsa.PrefillPlan.LAUNCHES.values()) * steps
    l2 = ("inputs larger than L2 (Q+K+V %.0f MB > 129 MB); no flush" % (in_bytes / 1e6)
          if flush is None else
          "L2 flushed before every step (write of %.0f MB); Q+K+V %.1f MB" %
          (flush.numel() * 4 / 1e6, in_bytes / 1e6))
    del flush
    res = dict(x=x, plan=plan, q=q, k=k, v=v, total_ms=total_ms, steps=steps, stages=st, l2=l2,
               flops=flops, eff_flops=eff, clocks=clocks, launches=launches, T=T,
               tiles={"min": int(tiles.min()), "mean": float(tiles.mean()), "max": int(tiles.max()),
                      "total": int(counts.sum())},
               router_flops=accounting.router_flops(x.cu_seqlens, w.block, w.num_heads, w.head_dim),
               attn_bytes=accounting.attention_bytes(w.num_heads, w.num_kv_heads, T, w.head_dim))
    return res


def router_quality(res, w, device):
    """Outside the timed loop: the coverage C_i of eq.(10) of the routed rows
    (the lse of the routed attention against the lse of the same kernel over every
    causal block), the recall of planted (key block, query block) pairs, and the
    density-1 attention time with the same kernel."""
    import dynamic_block_sparse_mean_gb300 as bsa
    from dynamic_block_sparse_mean_gb300 import accounting
    plan, q, k, v, x = res["plan"], res["q"], res["k"], res["v"], res["x"]
    dense = bsa.causal_worklist(plan.shape, device)
    for _ in range(2):
        Od, ld = bsa.attention_fwd(q, k, v, dense, plan.shape, plan.status)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 3
    t0.record()
    for _ in range(reps):
        Od, ld = bsa.attention_fwd(q, k, v, dense, plan.shape, plan.status)
    t1.record()
    torch.cuda.synchronize(device)
    dense_ms = t0.elapsed_time(t1) / reps
    plan.attend(q, k, v)
    C = bsa.coverage(plan.lse, ld, plan.shape)
    torch.cuda.synchronize(device)
    bsa.check_status(plan.status)
    c = C.flatten().float()
    qs = torch.quantile(c[:min(c.numel(), 1 << 24)], torch.tensor([0.001, 0.01, 0.05, 0.5],
                                                                  device=device)).tolist()
    G = w.num_heads // w.num_kv_heads
    info = []
    for i in range(len(x.cu_seqlens) - 1):
        nb = (int(x.cu_seqlens[i + 1] - x.cu_seqlens[i]) + w.block - 1) // w.block
        info.append(nb)
    dense_counts = np.zeros_like(plan.counts.cpu().numpy())
    for i, nb in enumerate(info):
        dense_counts[i, :, :nb] = np.arange(1, nb + 1)
    dense_flops = accounting.attention_tile_flops(dense_counts, G, w.block, w.head_dim)
    out = {"coverage": {"mean": float(c.mean()), "min": float(c.min()), "p0.1": qs[0],
                        "p1": qs[1], "p5": qs[2], "p50": qs[3],
                        "frac_below_0.9": float((c < 0.9).float().mean())},
           "dense_attention_ms": dense_ms,
           "dense_attention_tflops": dense_flops / (dense_ms * 1e-3) / 1e12,
           "density": res["flops"] / dense_flops,
           "speedup_vs_dense": dense_ms / res["stages"]["attention"]}
    if x.planted:
        J = plan.J.cpu().numpy()
        cnt = plan.counts.cpu().numpy()
        hit = sum(1 for (h, j, u) in x.planted if j in set(J[0, h, u, :cnt[0, h, u]].tolist()))
        out["planted_recall"] = hit / len(x.planted)
        out["planted_pairs"] = len(x.planted)
    del Od, ld, C, dense
    out["recall_at_k"] = token_recall_leg(res, w, device)
    return out


def token_recall_leg(res, w, device, t_top=64, max_tiles=20000, sample=2048):
    """Token recall of the routed rows against the dense top-t teacher (the recall@k
    paragraph of 2.1 §1.1), with the physical budget beside it: every query of the
    batch when it has at most max_tiles 64-query tiles, else a seeded sample."""
    import dynamic_block_sparse_mean_gb300 as bsa
    plan, q, k, x = res["plan"], res["q"], res["k"], res["x"]
    sh = plan.shape
    per = bsa.recall_tiles_per_seq(sh)
    cu = np.asarray(x.cu_seqlens, dtype=np.int64)
    lens = np.diff(cu)
    valid = [(i * w.num_heads + hq) * per + c for i in range(len(lens))
             for hq in range(w.num_heads) for c in range((int(lens[i]) + 63) // 64)]
    tiles = None
    if len(valid) > max_tiles:
        pick = np.sort(np.random.default_rng(77).choice(len(valid), size=sample, replace=False))
        tiles = torch.as_tensor(np.asarray(valid, dtype=np.int32)[pick], device=device)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    hits = bsa.token_recall(q, k, plan.J, plan.counts, sh, t_top, tiles=tiles, dev_status=st)
    t1.record()
    torch.cuda.synchronize(device)
    bsa.check_status(st)
    pos = np.concatenate([np.arange(n) for n in lens])
    gsize = np.minimum(t_top, pos + 1)[None, :]
    h = hits.cpu().numpy()
    got = h >= 0
    rec = (h / gsize)[got]
    qs = np.quantile(rec, [0.001, 0.01, 0.05, 0.5])
    return {"t": t_top, "mean": float(rec.mean()), "min": float(rec.min()), "p0.1": float(qs[0]),
            "p1": float(qs[1]), "p5": float(qs[2]), "p50": float(qs[3]),
            "queries": int(got.sum()),
            "sample": "all queries" if tiles is None else
                      f"{sample} random 64-query tiles of {len(valid)} (seed 77)",
            "physical_tiles_per_row_mean": res["tiles"]["mean"],
            "physical_keys_per_query_max": res["tiles"]["mean"] * w.block,
            "kernel_ms": t0.elapsed_time(t1)}


def bench_backward(res, w, device, reps=3):
    """Outside the timed loop: the backward (bsa_attention_bwd) on the forward's
    worklist and lse with a seeded upstream gradient; algorithmic FLOPs are 2.5x the
    forward's tile count (recomputed QK^T, dP = dO V^T, dV, dQ, dK: five b x b x d
    products per tile against the forward's two).  The tensor-core path executes
    seven (its dQ and dK / dV passes each recompute QK^T and dO V^T)."""
    import dynamic_block_sparse_mean_gb300 as bsa
    plan, q, k, v = res["plan"], res["q"], res["k"], res["v"]
    plan.attend(q, k, v)
    g = torch.Generator(device="cpu").manual_seed(1007)
    do = torch.randn(q.shape, generator=g, dtype=torch.float32).to(device=device, dtype=q.dtype)
    s = plan.shape.c()
    import ctypes
    from dynamic_block_sparse_mean_gb300 import _lib
    n = int(_lib.lib().bsa_attention_bwd_workspace_size(ctypes.byref(s)))
    ws = torch.empty(max(256, n), dtype=torch.uint8, device=device)
    dq, dk, dv = bsa.attention_bwd(q, k, v, plan.out, do, plan.lse, plan.wl, plan.shape, ws=ws)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        bsa.attention_bwd(q, k, v, plan.out, do, plan.lse, plan.wl, plan.shape, dq=dq, dk=dk,
                          dv=dv, ws=ws)
    t1.record()
    torch.cuda.synchronize(device)
    bsa.check_status(plan.status)
    ms = t0.elapsed_time(t1) / reps
    flops = 2.5 * res["flops"]
    tf = flops / (ms * 1e-3) / 1e12
    del dq, dk, dv, ws, do
    if w.head_dim == 128:  # the tensor-core path (BF16, head_dim 128)
        peaks, src = measured_peaks()
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        return {"ms": ms, "tflops": tf, "flops_per_call": flops, "path": "tcgen05",
                "executed_flops_per_call": 3.5 * res["flops"],
                "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                             "frac": tf / peak, "peak_source": f"{src} bf16 burst"}}
    # FP32 FFMA peak: 152 SMs x 128 lanes x 2 FLOP x the maximum SM clock
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    peak = sms * 128 * 2 * 2.07e9 / 1e12
    return {"ms": ms, "tflops": tf, "flops_per_call": flops, "path": "simt",
            "roofline": {"bound": "alu", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak,
                         "peak_source": "FP32 FFMA: SMs x 128 lanes x 2 FLOP x 2070 MHz"}}


def bench_chunked(res, w, device, chunk_tokens=8192, reps=3):
    """Outside the timed loop: the same prompt batch as a chunked prefill over a
    paged KV cache whose pages sit in a random physical order.  Each step every
    sequence appends up to chunk_tokens tokens (bsa_chunk_append), routes them
    against the cached page summaries (bsa_route_chunk), and attends the selected
    pages (bsa_build_worklist_chunk, bsa_attention_chunk).  Reports the whole
    prompt's time over all chunks, TFLOP/s on the single-pass tile count, and
    whether the chunked index equals the single-pass one."""
    import dynamic_block_sparse_mean_gb300 as bsa
    if w.block != 64:
        return {"skipped": f"chunks use 64-token pages; this workload's block is {w.block}"}
    x, q, k, v, plan = res["x"], res["q"], res["k"], res["v"], res["plan"]
    cu = np.asarray(x.cu_seqlens, dtype=np.int64)
    lens = np.diff(cu)
    pages = (lens + 63) // 64
    perm = np.random.default_rng(2024).permutation(int(pages.sum()))
    bt = np.full((len(lens), int(pages.max())), -1, dtype=np.int32)
    off = 0
    for i, L in enumerate(pages):
        bt[i, :L] = perm[off:off + L]
        off += int(L)
    cache = bsa.PagedKVCache.allocate(len(perm), w.num_kv_heads, w.head_dim, bt, device=device)
    nsteps = int((lens.max() + chunk_tokens - 1) // chunk_tokens)
    steps = []
    for s in range(nsteps):
        pre = np.minimum(s * chunk_tokens, lens)
        n = np.minimum(chunk_tokens, lens - pre)
        idx = np.concatenate([np.arange(cu[i] + pre[i], cu[i] + pre[i] + n[i])
                              for i in range(len(lens))])
        ti = torch.as_tensor(idx, device=device)
        chunk = bsa.Chunk.make(pre, n, w.num_heads, w.num_kv_heads, w.head_dim, device=device,
                               max_context_blocks=int(pages.max()))
        steps.append((bsa.ChunkPlan(chunk, cache, plan.params, device=device), pre, n,
                      q[:, ti].contiguous(), k[:, ti].contiguous(), v[:, ti].contiguous()))
    for cp, _, _, qc, kc, vc in steps:
        cp.run(qc, kc, vc)
    torch.cuda.synchronize(device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        for cp, _, _, qc, kc, vc in steps:
            cp.run(qc, kc, vc)
    t1.record()
    torch.cuda.synchronize(device)
    for cp, *_ in steps:
        bsa.check_status(cp.status)
    ms = t0.elapsed_time(t1) / reps
    J1, c1 = plan.J.cpu().numpy(), plan.counts.cpu().numpy()
    same = True
    for cp, pre, n, *_ in steps:
        Jc, cc = cp.J.cpu().numpy(), cp.counts.cpu().numpy()
        for i in range(len(lens)):
            nq, r0 = int((n[i] + 63) // 64), int(pre[i] // 64)
            same &= bool(np.array_equal(cc[i, :, :nq], c1[i, :, r0:r0 + nq]) and
                         np.array_equal(Jc[i, :, :nq], J1[i, :, r0:r0 + nq]))
    del steps, cache
    return {"chunk_tokens": chunk_tokens, "chunks": nsteps, "ms": ms,
            "tflops": res["flops"] / (ms * 1e-3) / 1e12,
            "single_pass_ms": res["total_ms"] / res["steps"],
            "index_equals_single_pass": same,
            "launches_per_prompt": nsteps * sum(bsa.ChunkPlan.LAUNCHES.values())}


def bench_e2e(res, w, steps, device):
    """Same metric through the public host-buffer API (bsa.HostPrefill): every step
    uploads Q, K, V from pinned host memory and downloads O into pinned host
    memory; the copies of neighbouring steps overlap the current step's kernels
    (two device slots, one stream per copy direction)."""
    import dynamic_block_sparse_mean_gb300 as bsa
    x = res["x"]
    hq, hk, hv = (torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
                  for a in (x.q, x.k, x.v))
    ho = [torch.empty(hq.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    pipe = bsa.HostPrefill(x.cu_seqlens, w.num_heads, w.num_kv_heads, w.head_dim, w.block,
                           bsa.RouteParams(w.mode, w.k_max, w.k_min, w.tau_delta, w.force_sink),
                           device=device)
    for s in range(3):
        pipe.submit(hq, hk, hv, ho[s % 2])
    pipe.synchronize()
    for st in pipe.status:
        bsa.check_status(st)
    t0 = time.perf_counter()
    for s in range(steps):
        pipe.submit(hq, hk, hv, ho[s % 2])
    pipe.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    for st in pipe.status:
        bsa.check_status(st)
    same = bool(torch.equal(ho[(steps - 1) % 2], res["plan"].out.cpu()))
    bi = sum(t.numel() * 2 for t in (hq, hk, hv))
    bo = ho[0].numel() * 2
    del pipe, ho, hq, hk, hv
    return ms, bi, bo, same


def bench_decode(steps, warmup, device, num_reqs=None):
    import dynamic_block_sparse_mean_gb300 as bsa
    from dynamic_block_sparse_mean_gb300 import accounting, synth
    from dynamic_block_sparse_mean_gb300.workloads import DECODE_64 as w

    R = w.num_reqs if num_reqs is None else min(num_reqs, w.num_reqs)
    dx = synth.make_decode(w, num_reqs=R)
    q = to_dev_bf16(dx.q, device)
    kc = to_dev_bf16(dx.k_cache, device)
    vc = to_dev_bf16(dx.v_cache, device)
    bt = torch.as_tensor(dx.block_table, device=device)
    cl = torch.as_tensor(dx.context_lens, device=device)
    ps = bsa.page_summaries(kc, bt, cl)
    plan = bsa.DecodePlan(R, w.num_heads, w.num_kv_heads, w.head_dim, w.page_size,
                          dx.block_table.shape[1], dx.k_cache.shape[0], w.top_k, device=device)
    for _ in range(max(3, warmup)):
        plan.run(q, kc, vc, ps, bt, cl)
    torch.cuda.synchronize(device)
    bsa.check_status(plan.status)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        plan.run(q, kc, vc, ps, bt, cl)
    t1.record()
    torch.cuda.synchronize(device)
    ms = t0.elapsed_time(t1) / steps
    by = accounting.decode_bytes(dx.context_lens, plan.sel.cpu().numpy(),
                                 plan.sel_counts.cpu().numpy(), w.num_heads, w.num_kv_heads,
                                 w.head_dim, w.page_size)
    del kc, vc
    return ms, by, w, R


# ---------------------------------------------------------------- CPU oracle


def oracle_rows(x, w, rows, cache):
    """The oracle's route + attention for a list of (i, h, r) rows (block
    summaries of the whole batch on first use); returns the selected-tile FLOPs
    processed."""
    import oracle
    from dynamic_block_sparse_mean_gb300 import synth

    class View:  # bf16 bits -> float64, converted slice by slice
        def __init__(self, bits):
            self.bits, self.shape = bits, bits.shape

        def __getitem__(self, idx):
            return synth.bf16_bits_to_f32(np.ascontiguousarray(self.bits[idx])).astype(np.float64)

    Q, K, V = View(x.q), View(x.k), View(x.v)
    G = w.num_heads // w.num_kv_heads
    if "C" not in cache:
        cache["C"] = oracle.block_summaries(K, x.cu_seqlens, w.block)
    C = cache["C"]
    flops = 0.0
    for (i, h, r) in rows:
        g = oracle.route_scores_row(Q, C, x.cu_seqlens, w.block, G, (i, h, r)) if r > 0 else []
        sel = oracle.select_row(g, r, w.mode, w.k_max, w.k_min, w.tau_delta, w.force_sink)
        J = np.full(C.shape[:3] + (len(sel),), -1)
        J[i, h, r] = sel
        cnt = np.zeros(C.shape[:3], dtype=np.int64)
        cnt[i, h, r] = len(sel)
        oracle.attention_row(Q, K, V, x.cu_seqlens, w.block, G, J, cnt, (i, h, r))
        flops += len(sel) * G * 4.0 * w.block * w.block * w.head_dim
    return flops


def cpu_oracle_throughput(x, w, budget_s: float, seed: int = 0, max_rows: int = 4000):
    """Time the oracle on random rows of the workload until budget_s has passed."""
    rng = np.random.default_rng(seed)
    info = [(int(x.cu_seqlens[i]), int(x.cu_seqlens[i + 1] - x.cu_seqlens[i])) for i in range(len(x.cu_seqlens) - 1)]
    C_cache = {}
    flops, n, t0 = 0.0, 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s and n < max_rows:
        i = int(rng.integers(len(info)))
        nb = (info[i][1] + w.block - 1) // w.block
        row = (i, int(rng.integers(w.num_kv_heads)), int(rng.integers(nb)))
        flops += oracle_rows(x, w, [row], C_cache)
        n += 1
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, n, dt


# ---------------------------------------------------------------- arms


def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    from dynamic_block_sparse_mean_gb300 import synth
    w = prefill_workload(args.workload, args.tokens)
    x = synth.make_prefill(w)
    per_step = max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    for s in range(args.warmup):
        cpu_oracle_throughput(x, w, per_step, seed=10_000 + s)
    flops, dt, rows = 0.0, 0.0, 0
    for s in range(args.steps):
        v, n, t = cpu_oracle_throughput(x, w, per_step, seed=s)
        flops += v * 1e12 * t
        dt += t
        rows += n
    value = flops / dt / 1e12
    sample = (f"{rows} random (sequence, KV head, query block) rows of {w.name}: oracle block "
              f"summaries of the touched head, router scores and selection, masked full-row "
              f"attention; about {per_step:.2f} s of rows per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": NCORES, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def decode_entry(args, device, peaks, src):
    d_ms, d_bytes, dw, R = bench_decode(max(20, min(args.steps, 200)), args.warmup, device,
                                        args.decode_reqs)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = d_bytes["total"] / (d_ms * 1e-3) / 1e9
    name = dw.name if R == dw.num_reqs else f"{dw.name}_first{R}"
    return {"workload": name, "value": gbs, "unit": "GB/s", "ms_per_step": d_ms,
            "kv_only_gbs": d_bytes["kv"] / (d_ms * 1e-3) / 1e9, "bytes": d_bytes,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "peak_source": f"{src} copy bandwidth"}}


def stage_rooflines(res, w, peaks, src):
    """Roofline objects of the attention kernel (tensor), the router call (HBM and
    tensor) and the summaries kernel (HBM) from the stage times of one workload."""
    from dynamic_block_sparse_mean_gb300 import accounting
    st = res["stages"]
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    x = res["x"]
    nblocks = int(sum((int(x.cu_seqlens[i + 1] - x.cu_seqlens[i]) + w.block - 1) // w.block
                      for i in range(len(x.cu_seqlens) - 1)))
    Nq = res["plan"].shape.max_blocks
    attn_kernel = f"attn_tc_kernel<{w.head_dim},{w.block}>"
    attn_tf = res["flops"] / (st["attention"] * 1e-3) / 1e12
    attention = {"bound": "tensor", "kernel": attn_kernel, "achieved": attn_tf, "peak": bf16,
                 "unit": "TFLOP/s", "frac": attn_tf / bf16,
                 "peak_source": f"{src} bf16 burst",
                 "traffic": recorded_traffic(attn_kernel, w.name),
                 "algorithmic_flops_per_launch": res["flops"],
                 "compulsory_bytes_per_launch": res["attn_bytes"]}
    rb = accounting.router_bytes(w.num_heads, w.num_kv_heads, res["T"], w.head_dim,
                                 w.num_seqs, Nq, w.k_max)
    r_gbs = rb / (st["route"] * 1e-3) / 1e9
    r_tf = res["router_flops"] / (st["route"] * 1e-3) / 1e12
    router = {"ms": st["route"],
              "hbm": {"bound": "hbm", "kernel": "bsa_route (split + scores + select)",
                      "achieved": r_gbs, "peak": hbm, "unit": "GB/s", "frac": r_gbs / hbm,
                      "peak_source": f"{src} copy bandwidth", "bytes_per_call": rb},
              "tensor": {"bound": "tensor", "kernel": "bsa_route (split + scores + select)",
                         "achieved": r_tf, "peak": bf16, "unit": "TFLOP/s", "frac": r_tf / bf16,
                         "peak_source": f"{src} bf16 burst",
                         "flops_per_call": res["router_flops"],
                         "note": "1x count: 2 d per (query row, history block)"}}
    sb = accounting.summaries_bytes(w.num_kv_heads, res["T"], w.head_dim, nblocks)
    s_gbs = sb / (st["summaries"] * 1e-3) / 1e9
    summaries = {"bound": "hbm", "kernel": "block_summaries_kernel", "achieved": s_gbs,
                 "peak": hbm, "unit": "GB/s", "frac": s_gbs / hbm,
                 "peak_source": f"{src} copy bandwidth", "bytes_per_launch": sb}
    return attention, router, summaries


def prefill_entry(key, args, device, world, rank, local, peaks, src, headline):
    """Time one prefill workload and run its legs; returns (summary dict, res)."""
    w = prefill_workload(key, args.tokens)
    steps = args.steps if headline or key != "tiny" else max(args.steps, 50)
    sampler = ClockSampler(local)
    res = bench_prefill(w, steps, args.warmup, device, world, sampler)
    ms_step = res["total_ms"] / steps
    max_ms, tot_flops = reduce_max_sum(world, ms_step, res["flops"], device)
    attention, router, summaries = stage_rooflines(res, w, peaks, src)
    st = res["stages"]
    out = {"workload": w.name, "value": tot_flops / (max_ms * 1e-3) / 1e12, "unit": UNIT,
           "ms_per_step": max_ms, "steps": steps, "total_tokens": res["T"],
           "l2": res["l2"], "router_ms": st["summaries"] + st["route"], "stages_ms": st,
           "attention_tflops": attention["achieved"],
           "effective_pair_tflops": res["eff_flops"] / (st["attention"] * 1e-3) / 1e12,
           "tiles_per_row": res["tiles"], "roofline": attention, "router": router,
           "summaries": summaries, "clocks": res["clocks"],
           "gpu_launches": res["launches"]}
    if not args.no_quality:
        q = router_quality(res, w, device)
        out["speedup_vs_dense"] = q.pop("speedup_vs_dense")
        out["router_quality"] = q
    if not args.no_backward and w.head_dim == 128 and key in ("prompt", "long"):
        out["backward"] = bench_backward(res, w, device)
    if not args.no_chunked and key == "prompt":
        out["chunked_prefill"] = bench_chunked(res, w, device)
    if headline and not args.no_e2e:
        e_ms, bi, bo, same = bench_e2e(res, w, max(3, min(args.steps, 20)), device)
        out["e2e"] = {"value": res["flops"] * world / (e_ms * 1e-3) / 1e12, "unit": UNIT,
                      "ms_per_step": e_ms, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                      "api": "HostPrefill.submit (copies overlapped with compute)",
                      "output_equals_device_path": same}
    if headline and rank == 0 and world == 1 and not args.no_cpu:
        v, n, dt = cpu_oracle_throughput(res["x"], w, budget_s=12.0)
        out["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": NCORES, "kind": "oracle",
            "sample": f"{n} random rows of {w.name} in {dt:.1f} s (oracle summaries of the "
                      f"touched heads, router scores, selection, masked full-row attention); "
                      f"FLOPs counted as selected physical tiles"}
    return out, res


def free_res(res):
    for key in ("q", "k", "v", "plan", "x"):
        res.pop(key, None)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def run_native(args):
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    barrier(world, device)
    peaks, src = measured_peaks()
    if args.decode_only:  # diagnostic: the decode leg alone, one line
        dec = decode_entry(args, device, peaks, src)
        if rank == 0:
            print(json.dumps({"metric": "decode KV GB/s", "value": dec["value"], "unit": "GB/s",
                              "n_gpus": world, "steps": max(20, min(args.steps, 200)),
                              "warmup": args.warmup, "ms_per_step": dec["ms_per_step"],
                              "higher_is_better": True, "decode": dec}), flush=True)
        return 0
    head, res = prefill_entry(args.workload, args, device, world, rank, local, peaks, src, True)
    w = prefill_workload(args.workload, args.tokens)
    free_res(res)
    configs = {w.name: head}
    others = [] if args.configs == "none" else [c for c in args.configs.split(",") if c]
    for key in others:
        if key == args.workload or key not in WORKLOAD_KEYS:
            continue
        sub, r = prefill_entry(key, args, device, world, rank, local, peaks, src, False)
        free_res(r)
        configs[sub["workload"]] = sub
    dec = None if args.no_decode else decode_entry(args, device, peaks, src)
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "num_seqs": w.num_seqs, "total_tokens": head["total_tokens"],
                   "num_heads": w.num_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "block": w.block, "k_max": w.k_max,
                   "route": "topk" if w.mode == 0 else "threshold", "l2": head["l2"],
                   "parallelism": f"replicas x{world}"},
        "router_ms": head["router_ms"],
        "stages_ms": head["stages_ms"],
        "attention_tflops": head["attention_tflops"],
        "roofline": head["roofline"],
        "router": head["router"],
        "summaries": head["summaries"],
        "speedup_vs_dense": head.get("speedup_vs_dense"),
        "cpu_baseline": head.get("cpu_baseline"),
        "e2e": head.get("e2e"),
        "decode": dec,
        "configs": configs,
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
