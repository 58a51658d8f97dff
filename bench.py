"""Benchmark of the absorbed-MLA decode step on GB300.

One step = the whole hot path on one synthetic decode batch:
  mla_cache_write of the step's new latent rows (one per query token), then
  mla_decode (split-KV plan, tcgen05 decode, LSE combine).
Default workload: DeepSeek-V3-shaped decode, N=128 heads, batch 64, contexts
uniform in [1024, 8192], page 64, bf16 cache in a 40k-page pool.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                       [--workload NAME] [--op decode|q_absorb|v_up_proj|gather]
--op q_absorb / v_up_proj times the per-head projections around the decode
(query absorption q_nope @ W_UK_T, value up-projection o_latent @ W_UV) on
the workload's token and head counts instead of the decode step; --op gather
times the paged context gather (gather_and_maybe_dequant_cache) of every
request's whole context.
Prints one JSON line.  With --gpus N > 1 (under torchrun) every rank runs an
independent replica (the decode of one batch does not shard), value = tokens of
all ranks / max time over ranks.  --impl reference times the fp64 CPU oracle
on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MLA decode tokens/s + HBM GB/s & % roofline (N=128,B=64,ctx 4k,bf16)"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 * 10**6       # GB300 L2


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def source_hash(name: str = "decode.cu") -> str:
    """First 16 hex digits of the sha256 of a kernel source's code: comments
    and blank lines removed, so that only a change of the code itself makes a
    recorded profile stale."""
    import hashlib
    import re
    text = open(os.path.join(ROOT, "mla_latent_kv_15_gb300", "csrc", name)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", l).rstrip() for l in text.splitlines()]
    code = "\n".join(l for l in lines if l.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def profiled_traffic(workload: str, names=None, source: str = "decode.cu"):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if that summary was taken on the current source of the kernel."""
    for name in names or (f"decode_{workload}.md", f"decode_{workload}_bf16.md"):
        path = os.path.join(ROOT, "profiles", name)
        if not os.path.exists(path):
            continue
        sha, traffic = None, None
        for line in open(path):
            if "Kernel code sha256" in line:
                sha = line.strip().split()[-1]
            if line.startswith("traffic_bytes_per_launch:"):
                traffic = int(line.split(":")[1])
        if sha == source_hash(source):
            return traffic
    return None


def max_over_ranks(values, dist, device="cpu"):
    """Element-wise maximum of per-rank timings (the slowest rank sets the
    job's time); identity on one process."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job rate: the units all ranks processed / the max-over-ranks time."""
    return world * units_per_rank / (ms * 1e-3)


HOST_US_PER_STEP = 250.0   # host time budgeted per enqueued step (calls, copies, events)


def host_lead(stream, steps: int = 0, ms: float = 5.0):
    """Keep the GPU busy (a spin kernel of ~`ms`, or HOST_US_PER_STEP per step
    of the `steps` that follow if that is longer, at the maximum clock) while
    the host enqueues the timed launches that follow, so that no timed
    interval includes time the GPU spent waiting for the host to submit work."""
    import torch
    ms = max(ms, steps * HOST_US_PER_STEP / 1000.0)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 2.07e6))


def algorithmic(case):
    """Bytes and FLOPs the decode must move / do at minimum: every visible
    latent row read once per request, queries read, outputs and LSE written;
    2*(576+512) FLOP per (visible key, query row)."""
    N = case.num_heads
    row_bytes = synth.DQK * (2 if case.cache_dtype == "bf16" else 1)
    kv = int(case.seq_lens.clip(min=0).sum()) * row_bytes
    T = case.total_q
    q = T * N * synth.DQK * 2
    out = T * N * synth.LKV * 2 + T * N * 4
    qsl = case.query_start_loc
    vis = 0
    for b in range(case.batch):
        sq = int(qsl[b + 1] - qsl[b])
        for t in range(sq):
            vis += max(int(case.seq_lens[b]) - sq + 1 + t, 0)
    flops = 2 * (synth.DQK + synth.LKV) * N * vis
    write = T * (synth.DQK * 2 + row_bytes)           # new rows read + cache rows written
    return dict(kv=kv, q=q, out=out, decode_bytes=kv + q + out, write_bytes=write, flops=flops)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running;
    the raw samples go to $MLA_CLOCKS_DIR (default: a temporary directory)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        import tempfile
        out_dir = os.environ.get("MLA_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank{device_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.dev), "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def run_gpu(args):
    import torch
    import mla_latent_kv_15_gb300 as mla
    sys.path.insert(0, os.path.join(ROOT, "tests"))

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    mla.load()

    case = synth.workload(args.workload, poison=False, **workload_overrides(args))
    N, T, B = case.num_heads, case.total_q, case.batch
    dev = "cuda"

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    # resident state: the paged cache
    if case.cache_dtype == "bf16":
        cache = bf16(case.pool)
    else:
        cache = torch.zeros(case.pool.shape, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
        flat = case.pool.reshape(-1, synth.DQK)[case.referenced_slots]
        mla.cache_write(bf16(flat[:, :synth.LKV]), bf16(flat[:, synth.LKV:]),
                        torch.from_numpy(case.referenced_slots).to(dev), cache, case.kv_scale)
    # per-step inputs (device copies) and their pinned host twins for the e2e leg
    host = {
        "q_abs": torch.from_numpy(case.q_abs.view(np.int16)).view(torch.bfloat16),
        "q_pe": torch.from_numpy(case.q_pe.view(np.int16)).view(torch.bfloat16),
        "kv_c": torch.from_numpy(case.new_kv_c.view(np.int16)).view(torch.bfloat16),
        "k_pe": torch.from_numpy(case.new_k_pe.view(np.int16)).view(torch.bfloat16),
        "slots": torch.from_numpy(case.slot_mapping),
        "block_table": torch.from_numpy(case.block_table),
        "seq_lens": torch.from_numpy(case.seq_lens),
        "qsl": torch.from_numpy(case.query_start_loc),
    }
    host = {k: v.pin_memory() for k, v in host.items()}
    d = {k: v.to(dev) for k, v in host.items()}
    out = torch.empty((T, N, synth.LKV), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, N), dtype=torch.float32, device=dev)
    ws = torch.empty(mla.decode_workspace_size(B, T, N, args.num_splits), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    fp8q = args.fp8_query
    if fp8q:
        if case.cache_dtype != "fp8":
            raise SystemExit("--fp8-query needs an e4m3-cache workload")
        # a static per-tensor query scale calibrated on this batch (|q| max / 448)
        qmax = max(float(np.abs(synth.bf16_bits_to_f32(case.q_abs)).max()),
                   float(np.abs(synth.bf16_bits_to_f32(case.q_pe)).max()))
        q_scale = float(np.float32(qmax / 448.0))
        q8 = torch.empty((T, N, synth.DQK), dtype=torch.uint8, device=dev)

    def step(inp, o=out, lo=lse):
        if not fp8q:
            # the cache write of the new rows and the decode in one call (the
            # rows are written by extra blocks of the scheduler's launch)
            mla.decode_step(inp["kv_c"], inp["k_pe"], inp["slots"], inp["q_abs"], inp["q_pe"], cache,
                            inp["block_table"], inp["seq_lens"], o, ws, scale=case.scale, query_start_loc=inp["qsl"],
                            lse=lo, num_splits=args.num_splits, kv_scale=case.kv_scale)
            return
        # the cache write, scaled_fp8_quant of q_abs and q_pe into [q_abs | q_pe]
        # rows (both by extra blocks of the scheduler's launch) and the fp8 x
        # fp8 decode in one call
        mla.decode_fp8q_step(inp["kv_c"], inp["k_pe"], inp["slots"], inp["q_abs"], inp["q_pe"], q_scale, q8, cache,
                             inp["block_table"], inp["seq_lens"], o, ws, scale=case.scale,
                             query_start_loc=inp["qsl"], lse=lo, num_splits=args.num_splits,
                             kv_scale=case.kv_scale)

    for _ in range(args.warmup):
        step(d)
    torch.cuda.synchronize()
    status = mla.decode_status(ws)
    if status != 0:
        raise RuntimeError(f"decode reported device error word {status}")

    # ---- timed region: device-resident inputs.  A workload whose step reads
    # more than twice the L2 in cache rows (every decode workload here) runs
    # back to back: the rows one step reads cannot still be in L2 when the
    # next reads them.  A smaller one gets the L2 flushed (a 256 MiB write)
    # before every step.
    # Pass 1 times whole steps (the throughput); pass 2 repeats them with
    # events recorded around the decode kernel (the roofline).  The kernel
    # events sit between launches, so they are kept out of the step timing.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in kev:          # torch creates its events lazily: record once so the handles exist
        a_.record(stream)
        b_.record(stream)
    alg = algorithmic(case)
    do_flush = alg["kv"] < 2 * L2_BYTES
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    with sampler:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        host_lead(stream, args.steps)
        if do_flush:
            # the flush between steps stays outside the timed intervals
            for i in range(args.steps):
                flush.fill_(i & 0xFF)
                ev[i][0].record(stream)
                step(d)
                ev[i][1].record(stream)
        else:
            # one event pair around the K back-to-back steps: an event recorded
            # between two steps would sit between the combine of one and the
            # cache write of the next, which could then no longer launch early
            ev[0][0].record(stream)
            for i in range(args.steps):
                step(d)
            ev[0][1].record(stream)
        torch.cuda.synchronize()
        host_lead(stream, args.steps)
        for i in range(args.steps):
            if do_flush:
                flush.fill_(i & 0xFF)
            mla.set_decode_timing_events(*kev[i])
            step(d)
        mla.set_decode_timing_events(None, None)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    if do_flush:
        ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    else:
        ms = ev[0][0].elapsed_time(ev[0][1]) / args.steps
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    kms = sum(kern_ms) / len(kern_ms)

    # ---- e2e: every step copies its inputs in from pinned host memory and
    # reads its outputs back: the inputs as one packed pinned buffer (one
    # copy), the output and LSE as one packed device buffer (one copy back).
    # Steps run in groups of G back to back: group g+1's inputs travel on a
    # copy stream while group g computes, and group g's outputs travel back
    # on another after it (2G device buffer sets).  The compute stream waits
    # once per group, so within a group every kernel may still launch under
    # the one before it.  A spin kernel ahead of the timed region lets the
    # host enqueue ahead, as for the device-resident timing.  The KV cache
    # (hundreds of MB per step) is larger than L2, so no flush.
    def nbytes(t):
        return t.numel() * t.element_size()

    def layout(tensors):
        offs, off = {}, 0
        for k, t in tensors.items():
            offs[k] = off
            off += (nbytes(t) + 255) // 256 * 256
        return offs, off

    def views(buf, tensors, offs):
        return {k: buf[offs[k]:offs[k] + nbytes(t)].view(t.dtype).view(t.shape) for k, t in tensors.items()}

    G = max(1, min(args.e2e_group, args.steps))
    NB = 2 * G
    in_offs, in_total = layout(host)
    h_in = torch.empty(in_total, dtype=torch.uint8).pin_memory()
    for k, t in host.items():
        h_in[in_offs[k]:in_offs[k] + nbytes(t)].copy_(t.contiguous().view(-1).view(torch.uint8))
    outs_t = {"out": out, "lse": lse}
    out_offs, out_total = layout(outs_t)
    d_in = [torch.empty(in_total, dtype=torch.uint8, device=dev) for _ in range(NB)]
    d_out = [torch.empty(out_total, dtype=torch.uint8, device=dev) for _ in range(NB)]
    h_out = [torch.empty(out_total, dtype=torch.uint8).pin_memory() for _ in range(NB)]
    sets = [views(b, host, in_offs) for b in d_in]
    outs = [(v["out"], v["lse"]) for v in (views(b, outs_t, out_offs) for b in d_out)]
    inp_bytes = sum(nbytes(v) for v in host.values())
    out_bytes = nbytes(out) + nbytes(lse)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    groups = [(g0, min(g0 + G, args.steps)) for g0 in range(0, args.steps, G)]
    in_done = [torch.cuda.Event() for _ in groups]
    comp_done = [torch.cuda.Event() for _ in groups]
    out_done = [torch.cuda.Event() for _ in groups]
    e2e_start, e2e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def copy_in(g):
        # group g's inputs; its buffer sets were last used by group g - 2
        with torch.cuda.stream(s_in):
            if g >= 2:
                s_in.wait_event(comp_done[g - 2])
            for k in range(*groups[g]):
                d_in[k % NB].copy_(h_in, non_blocking=True)
            in_done[g].record(s_in)

    def run_steps(cs, fork):
        # every step's copies and kernels; `cs` is the compute stream, the copy
        # streams start after `fork` (recorded on it) and rejoin it at the end
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        copy_in(0)
        for g, (k0, k1) in enumerate(groups):
            if g + 1 < len(groups):
                copy_in(g + 1)                             # travels while group g computes
            cs.wait_event(in_done[g])
            if g >= 2:
                cs.wait_event(out_done[g - 2])             # its output sets have been read back
            for k in range(k0, k1):
                step(sets[k % NB], *outs[k % NB])
            comp_done[g].record(cs)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[g])
                for k in range(k0, k1):
                    h_out[k % NB].copy_(d_out[k % NB], non_blocking=True)
                out_done[g].record(s_out)
        cs.wait_event(out_done[-1])

    torch.cuda.synchronize()
    host_lead(stream, args.steps)
    e2e_start.record(stream)
    run_steps(stream, e2e_start)
    e2e_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e2e_start.elapsed_time(e2e_end) / args.steps

    ms, kms, e2e_ms = max_over_ranks([ms, kms, e2e_ms], dist, dev)
    if rank != 0:
        return None

    hbm, tflops, src = peaks()
    if fp8q:
        # e4m3 query: one byte per query element; the score FLOPs run on the
        # fp8 tensor peak (2x the measured bf16 one, the nominal ratio), P.V on bf16
        alg["decode_bytes"] -= T * N * synth.DQK
        f_score = alg["flops"] * synth.DQK / (synth.DQK + synth.LKV)
        tflops = alg["flops"] / (f_score / (2 * tflops) + (alg["flops"] - f_score) / tflops)
    achieved = alg["decode_bytes"] / (kms * 1e-3) / 1e9
    achieved_tf = alg["flops"] / (kms * 1e-3) / 1e12
    # the binding roof of the workload: bytes at the HBM peak or FLOPs at the tensor peak
    hbm_bound = alg["decode_bytes"] / (hbm * 1e9) >= alg["flops"] / (tflops * 1e12)
    traffic = profiled_traffic(args.workload, [f"decode_{args.workload}_fp8q.md"] if fp8q else None)
    if hbm_bound:
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(achieved_tf, 1), "peak": tflops, "unit": "TFLOP/s",
                "frac": round(achieved_tf / tflops, 4)}
    roof.update({"traffic": traffic,
                 "peak_source": f"{src} (MEASURED_PEAKS.json {'hbm_gbs' if hbm_bound else 'bf16_tflops'}"
                                + (", score FLOPs at 2x for e4m3 x e4m3)" if fp8q and not hbm_bound else ")"),
                 "algorithmic_bytes_per_launch": alg["decode_bytes"], "algorithmic_flops_per_launch": alg["flops"]})
    tok_s = job_throughput(T, world, ms)
    clocks = sampler.summary()
    res = {
        "metric": METRIC,
        "value": round(tok_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if case.cache_dtype == "bf16" else ("e4m3 q,k / bf16 p,v" if fp8q else "e4m3-cache/bf16"),
        "data": "synthetic",
        "config": {
            "workload": args.workload + ("" if not workload_overrides(args) else
                                         f" (batch {B}, {case.num_blocks} pages)"),
            "num_heads": N, "batch": B, "total_q": T,
            "ctx_sum": int(case.seq_lens.sum()), "page_size": case.page_size, "num_blocks": case.num_blocks,
            "cache_dtype": case.cache_dtype, "query": "e4m3 (scaled_fp8_quant each step)" if fp8q else "bf16",
            "num_splits": args.num_splits, "parallelism": f"replicas{world}",
            "l2": ("flushed (256 MiB write) before every timed step" if do_flush else
                   f"no flush: inputs larger than L2 -- each step reads {alg['kv'] / 1e6:.0f} MB of cache rows "
                   f"({alg['kv'] / L2_BYTES:.1f} x the 129 MB L2)"),
            "timing": ("value: K whole steps, one CUDA event pair around them" if not do_flush else
                       "value: K whole steps, CUDA events around each (the flush outside)")
                      + "; roofline: a second pass of K steps with events around the decode kernel",
        },
        "hbm_gbs": round(achieved, 1),
        "tflops": round(achieved_tf, 1),
        "decode_kernel_ms": round(kms, 5),
        "roofline": roof,
        "e2e": {"value": round(job_throughput(T, world, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": inp_bytes, "d2h_bytes_per_step": out_bytes,
                "copies": f"one packed pinned input buffer and one packed output buffer per step; steps in "
                          f"groups of {G}: group g+1's inputs and group g-1's outputs move on copy streams while "
                          f"group g computes ({NB} device buffer sets)"},
        # per step: plan (with the cache write, and with an e4m3 query its
        # quantisation), decode, combine
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
    return res


def cpu_baseline(case, seconds: float):
    """The fp64 oracle on the host cores over a bounded sample of the workload:
    whole requests (all heads, full contexts) until ~`seconds` of work."""
    import oracle
    cache = oracle.prepare_cache(case)
    N = case.num_heads
    qsl = case.query_start_loc
    done_tokens = 0
    t0 = time.perf_counter()
    cores = 0
    b = 0
    while b < case.batch and (time.perf_counter() - t0) < seconds:
        rows = np.arange(qsl[b] * N, qsl[b + 1] * N, dtype=np.int64)
        _, _, cores = oracle.decode_case(case, cache, rows=rows)
        done_tokens += int(qsl[b + 1] - qsl[b])
        b += 1
    el = time.perf_counter() - t0
    return {"value": round(done_tokens / el, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{b} of {case.batch} requests (all {N} heads, full contexts), {el:.1f} s"}


def run_reference(args):
    """--impl reference: the fp64 oracle as it stands on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    case = synth.workload(args.workload, poison=False, **workload_overrides(args))
    cache = oracle.prepare_cache(case)
    N = case.num_heads
    qsl = case.query_start_loc
    per_step = max(1, args.ref_requests)
    times, cores = [], 0
    b = 0
    for i in range(args.warmup + args.steps):
        reqs = [(b + k) % case.batch for k in range(per_step)]
        b += per_step
        rows = np.concatenate([np.arange(qsl[r] * N, qsl[r + 1] * N, dtype=np.int64) for r in reqs])
        t0 = time.perf_counter()
        _, _, cores = oracle.decode_case(case, cache, rows=rows)
        el = time.perf_counter() - t0
        if i >= args.warmup:
            times.append((el, sum(int(qsl[r + 1] - qsl[r]) for r in reqs)))
    tot = sum(t for t, _ in times)
    toks = sum(n for _, n in times)
    v = toks / tot
    return {
        "metric": METRIC, "impl": "reference", "value": round(v, 3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "num_heads": N, "batch": case.batch,
                   "sample_per_step": f"{per_step} request(s), all heads, full contexts"},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} request(s) per step x {args.steps} steps"},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_proj(args):
    """One per-head projection per step (random bf16 weights of the
    DeepSeek-V3 shapes: P = V = 128, Lkv = 512).  Steps run back to back, as
    the layers of a model do, each on its own weights and activations taken
    round-robin from R sets whose total is more than twice the L2, so every
    step reads cold data; one event pair brackets all K steps."""
    import torch
    import mla_latent_kv_15_gb300 as mla
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    mla.load()
    cfg = synth.WORKLOADS[args.workload]
    N = cfg["num_heads"]
    sq = cfg["sq"]
    T = sum(sq) if isinstance(sq, list) else cfg["batch"] * sq
    P = V = 128
    dev = "cuda"
    w_uk, w_uv = synth.projection_weights(0, N, p=P, v=V)
    if args.op == "q_absorb":
        d_in, d_out, stride = P, synth.LKV, P + synth.ROPE     # q_nope = the first 128 columns of q
        w_host = np.ascontiguousarray(w_uk.transpose(1, 2, 0))   # (N, P, L)
    else:
        d_in, d_out, stride = synth.LKV, V, synth.LKV
        w_host = np.ascontiguousarray(w_uv.transpose(1, 0, 2))   # (N, L, V)
    x_bits = synth.bf16_normal(1, (T, N, stride))

    def t16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    x_h = t16(x_bits).pin_memory()
    y_h = torch.empty((T, N, d_out), dtype=torch.bfloat16).pin_memory()
    set_bytes = (w_host.size + x_bits.size + y_h.numel()) * 2
    R = max(2, -(-L2_FLUSH_BYTES // set_bytes))              # >= 256 MiB (2 x L2) of distinct data
    w0 = t16(w_host).to(dev)
    x0 = x_h.to(dev)
    sets = [(w0, x0, torch.empty(y_h.shape, dtype=torch.bfloat16, device=dev))]
    for _ in range(R - 1):                                   # same values, distinct memory
        sets.append((w0.clone(), x0.clone(), torch.empty_like(sets[0][2])))

    def op(w, xx, yy):
        if args.op == "q_absorb":
            mla.q_absorb(xx[:, :, :P], w, yy)
        else:
            mla.v_up_proj(xx, w, yy)

    stream = torch.cuda.current_stream()
    for i in range(max(args.warmup, R)):
        op(*sets[i % R])
    torch.cuda.synchronize()
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    with sampler:
        host_lead(stream, args.steps)
        t_a.record(stream)
        for i in range(args.steps):
            op(*sets[i % R])
        t_b.record(stream)
        torch.cuda.synchronize()
    ms = t_a.elapsed_time(t_b) / args.steps
    w, x, y = sets[0]
    if mla.proj_status() != 0:
        raise RuntimeError("projection kernel reported a device error")
    # e2e through the public API: x in from pinned host memory, y back
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        x.copy_(x_h, non_blocking=True)
        op(w, x, y)
        y_h.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps

    alg_bytes = T * N * d_in * 2 + N * d_in * d_out * 2 + T * N * d_out * 2
    flops = 2 * T * N * d_in * d_out
    hbm, _, src = peaks()
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    res = {
        "metric": f"{args.op} tokens/s + HBM GB/s & % roofline (N={N}, T={T}, {d_in}->{d_out} per head)",
        "op": args.op, "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload} token/head counts", "num_heads": N, "num_tokens": T,
                   "d_in": d_in, "d_out": d_out, "x_row_stride": stride,
                   "l2": f"no flush: {R} rotating weight/activation sets of {set_bytes} B (>= 2 x L2), "
                         "each step reads data no recent step touched",
                   "timing": f"one CUDA event pair on the launching stream around {args.steps} back-to-back "
                             "launches (programmatic dependent launches)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": (profiled_traffic(args.workload, [f"head_proj_{args.op}_n{N}_t{T}.md"], "proj.cu")
                                 if args.workload.startswith("dsv3_n128_b64") else None),
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": alg_bytes, "algorithmic_flops_per_launch": flops},
        "e2e": {"value": round(T / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": x_h.numel() * 2, "d2h_bytes_per_step": y_h.numel() * 2,
                "copies": "pinned host buffers, copies and launch serialised on one stream"},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
    }
    if not args.no_cpu_baseline:
        from oracle import expanded
        import oracle
        xf = oracle.bf16_to_f64(x_bits[:, :, :d_in])
        t0 = time.perf_counter()
        if args.op == "q_absorb":
            expanded.absorb_query(xf, oracle.bf16_to_f64(w_uk))
        else:
            expanded.up_project(xf, oracle.bf16_to_f64(w_uv))
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(T / el, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                               "sample": f"the whole op ({T} tokens x {N} heads), numpy einsum in fp64, {el:.2f} s"}
    return res


def run_gather(args):
    """--op gather: gather_and_maybe_dequant_cache of every request's whole
    context (cu_seq_lens = cumsum(seq_lens), chunk starts 0) into a dense bf16
    workspace, K launches back to back (the cache rows read and the rows
    written, ~2 x 340 MB, are far larger than L2)."""
    import torch
    import mla_latent_kv_15_gb300 as mla
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    mla.load()
    case = synth.workload(args.workload, poison=False, **workload_overrides(args))
    dev = "cuda"
    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    if case.cache_dtype == "bf16":
        cache = bf16(case.pool)
    else:                                  # quantised on the GPU by the library's cache write
        cache = torch.zeros(case.pool.shape, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
        flat = case.pool.reshape(-1, synth.DQK)[case.referenced_slots]
        mla.cache_write(bf16(flat[:, :synth.LKV]), bf16(flat[:, synth.LKV:]),
                        torch.from_numpy(case.referenced_slots).to(dev), cache, case.kv_scale)
    lens = case.seq_lens.astype(np.int64)
    cu_h = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    rows = int(cu_h[-1])
    bt_h = torch.from_numpy(case.block_table)
    cu, bt = cu_h.to(dev), bt_h.to(dev)
    dst = torch.empty((rows, synth.DQK), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def op(c=cu, b=bt):
        mla.gather_cache(cache, b, c, dst, kv_scale=case.kv_scale, status=status)

    for _ in range(args.warmup):
        op()
    torch.cuda.synchronize()
    t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    with sampler:
        host_lead(stream, args.steps)
        t_a.record(stream)
        for _ in range(args.steps):
            op()
        t_b.record(stream)
        torch.cuda.synchronize()
    ms = t_a.elapsed_time(t_b) / args.steps
    if int(status.item()) != 0:
        raise RuntimeError(f"gather reported device error word {int(status.item())}")
    # e2e: block table and cu_seq_lens in from pinned host memory, the gathered rows back
    cu_p, bt_p = cu_h.pin_memory(), bt_h.pin_memory()
    dst_h = torch.empty(dst.shape, dtype=dst.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_steps = max(1, min(args.steps, 5))
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e_steps):
        cu.copy_(cu_p, non_blocking=True)
        bt.copy_(bt_p, non_blocking=True)
        op()
        dst_h.copy_(dst, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e_steps

    row_bytes = synth.DQK * (2 if case.cache_dtype == "bf16" else 1)
    alg = rows * (row_bytes + synth.DQK * 2) + cu_h.numel() * 4 + bt_h.numel() * 4
    hbm, _, src = peaks()
    achieved = alg / (ms * 1e-3) / 1e9
    res = {
        "metric": f"context gather rows/s + HBM GB/s & % roofline ({case.cache_dtype} cache -> bf16 rows)",
        "op": "gather", "value": round(rows / (ms * 1e-3), 1), "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if case.cache_dtype == "bf16" else "e4m3->bf16",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: every request's whole context", "rows": rows,
                   "batch": case.batch, "page_size": case.page_size,
                   "l2": "no flush: each launch reads and writes ~2 x 340 MB, far more than L2",
                   "timing": f"one CUDA event pair around {args.steps} back-to-back launches"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": profiled_traffic(args.workload, [f"gather_{args.workload}.md"], "gather.cu"),
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)", "algorithmic_bytes_per_launch": alg},
        "e2e": {"value": round(rows / (e2e_ms * 1e-3), 1), "unit": "rows/s",
                "h2d_bytes_per_step": cu_p.numel() * 4 + bt_p.numel() * 4,
                "d2h_bytes_per_step": dst_h.numel() * 2,
                "copies": "pinned host buffers, copies and launch serialised on one stream"},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        host_cache = case.pool if case.cache_dtype == "bf16" else oracle.prepare_cache(case, with_new_rows=False)
        nb = min(case.batch, 16)
        t0 = time.perf_counter()
        oracle.gather_cache(host_cache, case.page_size,
                            oracle.CACHE_BF16 if case.cache_dtype == "bf16" else oracle.CACHE_E4M3, case.kv_scale,
                            case.block_table[:nb], cu_h.numpy()[:nb + 1], None, int(cu_h[nb]))
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(int(cu_h[nb]) / el, 3), "unit": "rows/s", "cores": 1,
                               "kind": "oracle", "sample": f"{nb} of {case.batch} requests' contexts, {el:.2f} s"}
    return res


def run_gather_reference(args):
    """--impl reference --op gather: the oracle's C gather (one thread) of the
    first 16 requests' whole contexts per step."""
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    import oracle
    case = synth.workload(args.workload, poison=False, **workload_overrides(args))
    host_cache = case.pool if case.cache_dtype == "bf16" else oracle.prepare_cache(case, with_new_rows=False)
    nb = min(case.batch, 16)
    cu = np.concatenate([[0], np.cumsum(case.seq_lens.astype(np.int64))]).astype(np.int32)[:nb + 1]
    dt = oracle.CACHE_BF16 if case.cache_dtype == "bf16" else oracle.CACHE_E4M3
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.gather_cache(host_cache, case.page_size, dt, case.kv_scale, case.block_table[:nb], cu, None,
                            int(cu[-1]))
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    v = int(cu[-1]) / (ms * 1e-3)
    return {
        "metric": f"context gather rows/s + HBM GB/s & % roofline ({case.cache_dtype} cache -> bf16 rows)",
        "op": "gather", "impl": "reference", "value": round(v, 3), "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: whole contexts of {nb} requests per step", "rows": int(cu[-1])},
        "cpu_baseline": {"value": round(v, 3), "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{nb} requests' whole contexts per step x {args.steps} steps"},
        "e2e": {"value": round(v, 3), "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_proj_reference(args):
    """--impl reference --op ...: the oracle's fp64 einsum for the projection,
    timed on the host over K steps of the same inputs as the GPU arm."""
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    import oracle
    from oracle import expanded
    cfg = synth.WORKLOADS[args.workload]
    N = cfg["num_heads"]
    sq = cfg["sq"]
    T = sum(sq) if isinstance(sq, list) else cfg["batch"] * sq
    P = V = 128
    w_uk, w_uv = synth.projection_weights(0, N, p=P, v=V)
    if args.op == "q_absorb":
        d_in, d_out = P, synth.LKV
        x = oracle.bf16_to_f64(synth.bf16_normal(1, (T, N, P + synth.ROPE))[:, :, :P])
        w, f = oracle.bf16_to_f64(w_uk), expanded.absorb_query
    else:
        d_in, d_out = synth.LKV, V
        x = oracle.bf16_to_f64(synth.bf16_normal(1, (T, N, synth.LKV)))
        w, f = oracle.bf16_to_f64(w_uv), expanded.up_project
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        f(x, w)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    v = T / (ms * 1e-3)
    return {
        "metric": f"{args.op} tokens/s + HBM GB/s & % roofline (N={N}, T={T}, {d_in}->{d_out} per head)",
        "op": args.op, "impl": "reference", "value": round(v, 3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload} token/head counts", "num_heads": N, "num_tokens": T,
                   "d_in": d_in, "d_out": d_out},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"the whole op per step, numpy einsum in fp64, {args.steps} steps"},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def workload_overrides(args) -> dict:
    """Request-count and page-pool overrides of a named workload (smaller
    cases of the same shapes, e.g. for profiler captures)."""
    over = {}
    if getattr(args, "batch", None):
        over["batch"] = args.batch
        sq = synth.WORKLOADS[args.workload]["sq"]
        if not isinstance(sq, int):
            raise SystemExit("--batch needs a workload with one query count for every request")
    if getattr(args, "num_blocks", None):
        over["num_blocks"] = args.num_blocks
    return over


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv3_n128_b64_ctx1k-8k", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's request count (smaller profiling captures)")
    ap.add_argument("--num-blocks", type=int, default=None,
                    help="override the workload's page pool (with --batch)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-requests", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-group", type=int, default=1,
                    help="end-to-end leg: steps per group between the compute stream's waits for copies")
    ap.add_argument("--fp8-query", action="store_true",
                    help="e4m3 workloads: quantise the query each step and run the fp8 x fp8 decode")
    ap.add_argument("--op", default="decode", choices=["decode", "q_absorb", "v_up_proj", "gather"])
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.op == "gather":
        res = run_gather_reference(args) if args.impl == "reference" else run_gather(args)
    elif args.op != "decode":
        res = run_proj_reference(args) if args.impl == "reference" else run_proj(args)
    else:
        res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
