#!/usr/bin/env python
"""Benchmark of the INT2 rotated paged KV cache decode step on GB300.

One step = the whole hot path for one batch: append one token per request through the
write path (window insert, eviction of the token that leaves the 256-token window,
key rotation, clip, INT2 quantisation, page store), rotate the queries, run the fused
split-K paged GQA decode attention over the INT2 pages plus the BF16 sink / window, and
combine the splits.

Workload (default): a Qwen3-32B-shaped attention layer -- 64 query / 8 KV heads,
head_dim 128, batch 32, 100000 tokens per request, scrambled page tables -- with seeded
synthetic keys / values / queries of the distributions in `synth`.

Printed JSON (rank 0):
  value      decode bytes per step (packed INT2 K+V codes, fp16 scale/min, BF16 sink +
             window K+V, q and out) x ranks / step time, in GB/s; the step time includes
             the write path.
  roofline   the decode attention call (3 launches, the split kernel dominates) against
             the measured HBM copy bandwidth.
  e2e        the same metric with q / k / v in pinned host memory copied in and the
             output copied out every step, host-timed, synchronised per step.
  cpu_baseline  the CPU oracle on a bounded sample of the same workload.

`--impl reference` times the CPU oracle alone on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen3_32b",
                    help="workload: tiny, qwen3_4b, qwen3_8b, qwen3_32b (default), ragged_128k, or all (one line each)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-pairs", type=int, default=max(8, os.cpu_count() or 1),
                    help="(request, KV head) pairs the CPU oracle times for cpu_baseline (about 1 s each, one per host core)")
    ap.add_argument("--ref-pairs", type=int, default=max(3, os.cpu_count() or 1),
                    help="(request, KV head) pairs per step of --impl reference (one per host core)")
    ap.add_argument("--batch", type=int, default=0,
                    help="requests per GPU (0 = the workload's batch); smaller values are for profiling")
    ap.add_argument("--path", default="mma", choices=["mma", "simt"],
                    help="decode kernel: warp-level MMA (default) or the SIMT baseline")
    ap.add_argument("--no-prefill", action="store_true", help="skip the chunked-prefill attention timing")
    ap.add_argument("--no-layers", action="store_true", help="skip the multi-layer append timing")
    ap.add_argument("--unfused", action="store_true",
                    help="run each step as kv_quant_append + oscar_decode_attention instead of oscar_decode_step")
    return ap.parse_args()


# ------------------------------------------------------------------ byte model

def decode_bytes(lens, hkv, hq, q_bytes=4, out_bytes=4):
    """Algorithmic bytes of one decode attention call."""
    tot = 0
    for L in lens:
        n_int2 = max(0, L - 320)
        n_bf16 = min(L, 320)
        tot += hkv * (n_int2 * 2 * (32 + 8) + n_bf16 * 2 * 256)
    return tot + len(lens) * hq * 128 * (q_bytes + out_bytes)


def int2_kernel_bytes(lens, hkv, hq):
    """Algorithmic bytes of one launch of the INT2 attention kernel: every INT2 token's K and V
    codes (32 + 32 B) and fp16 scale/min (8 + 8 B) per KV head, plus the fp32 rotated queries."""
    return sum(hkv * max(0, L - 320) * 80 for L in lens) + len(lens) * hq * 128 * 4


# What each decode path computes in (the line's "dtype" names the tensor-core operand / accumulator
# types of the default path).
PRECISION = {
    "mma": {"kv": "INT2 codes with fp16 scale/min per 64-channel group (exact as MMA operands)",
            "scores": "mma.sync fp16 x fp16 -> fp32; q as fp16 high + low parts (~22 bits) under a "
                      "power-of-two scale per (request, KV head)",
            "pv": "mma.sync fp16 x fp16 -> fp32; P' = p * s_V rounded once to fp16",
            "softmax": "fp32 (packed f32x2), base-2, lazily raised reference max",
            "bf16_part": "bf16 keys x bf16 high + low query parts (~16 bits) -> fp32; P.V fp32",
            "combine": "fp32"},
    "simt": {"kv": "INT2 codes with fp16 scale/min per 64-channel group",
             "scores": "fp32", "pv": "fp32", "softmax": "fp32", "bf16_part": "fp32", "combine": "fp32"},
}
NOMINAL_HBM_GBS = 8000.0   # the GB300 HBM3e figure the workload's target is stated against


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the sources that decide the INT2 attention kernel's memory traffic: the kernel's
    device code and the helpers it shares with the transposed-score kernel, its copy helpers and
    the page layout / parameter structs of internal.h (host-side
    launchers and their declarations are left out), with comments and blank space removed so that
    editing a comment keeps the recorded counters valid."""
    h = hashlib.sha256()
    for name in ("decode_mma.cu", "decode_mma_common.h", "ptx_async.h", "internal.h"):
        text = open(os.path.join(ROOT, "int2_rotated_paged_gb300", "csrc", name)).read()
        if name == "internal.h":
            text = text[:text.index("cudaError_t launch_")]
        if name == "decode_mma.cu":                # the device code, not the host launchers after it
            text = text[:text.index("cudaError_t launch_mma_g")]
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, scale: float):
    """DRAM bytes (read + write) per launch of the INT2 attention kernel, from the committed ncu
    summary: measured on a smaller batch of the same workload and scaled by the INT2 bytes,
    or None when the kernel changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "decode_mma_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("source_sha256_16") != kernel_source_hash() or rec.get("workload") != workload:
            return None
        return rec["dram_bytes_per_launch"] * scale / rec["int2_bytes_per_launch"]
    except Exception:
        return None


# ------------------------------------------------------------------ clocks

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ multi-rank timing

def max_over_ranks(x: float, dist, device) -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle timing

def cpu_oracle_sample(cfg, lens, n_pairs: int, reps: int = 1, ctx_cap: int = 0, threads: int = 1):
    """Time the CPU oracle on (request, KV head) pairs of the workload.  Each rep is one decode
    step of every sampled pair: append one token (window insert and, past 320 tokens, the
    eviction of one token to INT2), then attend.  ctx_cap > 0 keeps only the first ctx_cap
    tokens of each sampled request.  The pairs run on `threads` host threads (the oracle's C
    calls release the interpreter lock).  Returns (bytes per rep, seconds per rep, pairs, context)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    import synth
    oracle.build()
    pairs = [(b % cfg.batch, (3 * b + 1) % cfg.num_kv_heads) for b in range(n_pairs)]
    ctx = [min(lens[b], ctx_cap) if ctx_cap > 0 else lens[b] for b in range(len(lens))]

    def make(bh):
        b, h = bh
        rk = oracle.build_rk(synth.calibration_queries(cfg.seed, h, 4096).numpy())[0]
        oc = oracle.OracleCache(rk)
        oc.append(synth.bf16_bits(synth.keys(cfg.seed, b, h, 0, ctx[b] + reps)),
                  synth.bf16_bits(synth.values(cfg.seed, b, h, 0, ctx[b] + reps)))
        return (b, h, oc)

    g = cfg.group
    times, nbytes = [], []
    with ThreadPoolExecutor(max_workers=threads) as pool:
        caches = list(pool.map(make, pairs))
        for r in range(reps):
            q = synth.queries(cfg.seed, r, cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, dtype=cfg.q_dtype).numpy()
            steps = [(oc, synth.bf16_bits(synth.keys(cfg.seed, b, h, ctx[b] + r, 1)),
                      synth.bf16_bits(synth.values(cfg.seed, b, h, ctx[b] + r, 1)), q[b, h * g:(h + 1) * g])
                     for (b, h, oc) in caches]

            def run(st):
                oc, k1, v1, qb = st
                oc.append(k1, v1)
                oc.attend(qb)

            t0 = time.perf_counter()
            list(pool.map(run, steps))
            times.append(time.perf_counter() - t0)
            nbytes.append(sum(decode_bytes([ctx[b] + r + 1], 1, g) for (b, h, _) in caches))
    return nbytes, times, pairs, ctx


# ------------------------------------------------------------------ main arms

def l2_flush_needed(cfg, lens):
    return decode_bytes(lens, cfg.num_kv_heads, cfg.num_q_heads) < 2 * 129e6


def workload_config(cfg, lens):
    return {"workload": f"{cfg.name}: B{cfg.batch} Hq{cfg.num_q_heads}/Hkv{cfg.num_kv_heads} d128 "
                        f"L{lens[0] if len(set(lens)) == 1 else f'{min(lens)}..{max(lens)}'} INT2 paged decode step "
                        f"(append 1 token + split-K GQA decode), {cfg.table} pages",
            "batch_per_gpu": cfg.batch, "context": lens[0] if len(set(lens)) == 1 else [min(lens), max(lens)],
            "l2": (f"L2 flushed between timed steps (256 MB write, outside the step's events; "
                   f"{decode_bytes(lens, cfg.num_kv_heads, cfg.num_q_heads) / 1e6:.0f} MB per step)"
                   if l2_flush_needed(cfg, lens) else
                   f"inputs larger than L2 (about {decode_bytes(lens, cfg.num_kv_heads, cfg.num_q_heads) / 1e9:.2f} GB "
                   f"per step vs 129 MB)")}


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return
    lens = [int(x) for x in cfg.ctx]
    reps = args.warmup + args.steps
    threads = max(1, min(args.ref_pairs, os.cpu_count() or 1))
    # about 1.2 s per pair per step at 100000 tokens on one core: keep the whole run near two to
    # three minutes
    waves = -(-args.ref_pairs // threads)
    cap = int(min(max(lens), 100000 * 150.0 / (reps * waves * 1.2)))
    nbytes, times, pairs, ctx = cpu_oracle_sample(cfg, lens, args.ref_pairs, reps=reps, ctx_cap=cap, threads=threads)
    per = sum(times[args.warmup:]) / args.steps
    value = sum(nbytes[args.warmup:]) / sum(times[args.warmup:]) / 1e9
    sample = (f"per step: {len(pairs)} of {cfg.batch * cfg.num_kv_heads} (request, KV head) pairs, each "
              f"appending one token and attending over its first {min(ctx[b] for b, _ in pairs)} tokens "
              f"(the oracle's cost is linear in the context)")
    line = {
        "impl": "reference", "metric": "decode_attention_hbm_gbs", "value": value, "unit": "GB/s",
        "n_gpus": world, "world_size": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg, lens),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, cfg, rank, world, dist):
    import numpy as np
    import torch

    import synth
    import int2_rotated_paged_gb300 as K
    from int2_rotated_paged_gb300 import build as kbuild

    kbuild.build()
    K.oscar_set_decode_path({"mma": K.PATH_WARP_MMA, "simt": K.PATH_SIMT}[args.path])
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    seed = cfg.seed + 7919 * rank          # each rank holds its own batch of requests
    B, hq, hkv, g = cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, cfg.group
    lens0 = [int(x) for x in cfg.ctx]
    total_steps = args.warmup + args.steps + (0 if args.no_e2e else args.warmup + args.steps)

    # ---- R_K from 4096 query samples per KV head, on the GPU
    qcal = torch.stack([synth.calibration_queries(seed, h, 4096) for h in range(hkv)]).to(dev).contiguous()
    rk = torch.empty(hkv, 128, 128, device=dev)
    ws = torch.empty(K.oscar_build_rk_workspace_bytes(hkv), dtype=torch.uint8, device=dev)
    K.oscar_build_rk(qcal, 4096, hkv, rk, ws)
    torch.cuda.synchronize()
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    K.oscar_build_rk(qcal, 4096, hkv, rk, ws)      # the same inputs again, timed: same R_K
    c1.record(stream)
    c1.synchronize()
    calib = {"what": f"oscar_build_rk: C_Q (fp64) + cyclic Jacobi (fp64) + H_Had P_br for {hkv} KV heads "
                     f"from 4096 query samples each", "ms": c0.elapsed_time(c1)}
    del ws, qcal

    # ---- cache with scrambled physical pages
    per_seq = max(1, (max(lens0) + total_steps - 320 + 63) // 64 + 1) + 5   # + room for the 256-token prefill chunk
    total_pages = per_seq * B
    order = synth.page_order(seed, total_pages, cfg.table)
    cache = K.Cache(B, hq, hkv, total_pages, per_seq, page_order=order)

    # ---- bulk prefill through the write path (timed as the write-path metric)
    chunk = 16384
    done = [0] * B
    t_append = 0.0
    tok_append = 0
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    while any(done[b] < lens0[b] for b in range(B)):
        n = [min(chunk, lens0[b] - done[b]) for b in range(B)]
        k, v = synth.kv_block(seed, n, done, hkv, device=dev)
        ev0.record(stream)
        cache.append(k, v, n, rk)
        ev1.record(stream)
        ev1.synchronize()
        t_append += ev0.elapsed_time(ev1) * 1e-3
        tok_append += sum(n)
        done = [done[b] + n[b] for b in range(B)]
        del k, v

    # ---- decode inputs of every step, resident on the device
    qs, ks, vs = [], [], []
    for s in range(total_steps):
        qs.append(synth.queries(seed, s, B, hq, hkv, dtype=cfg.q_dtype, device=dev))
        k, v = synth.kv_block(seed, [1] * B, [lens0[b] + s for b in range(B)], hkv, device=dev)
        ks.append(k)
        vs.append(v)
    out = torch.empty(B, hq, 128, device=dev)
    torch.cuda.synchronize()

    ones = [1] * B

    def step_call(k, v, q):
        # one decode step through the public API: the fused call, or its two halves
        if args.unfused:
            cache.append(k, v, ones, rk)
            cache.attend(q, rk, out)
        else:
            cache.step(k, v, q, rk, out)

    def step(s):
        step_call(ks[s], vs[s], qs[s])

    # inputs smaller than twice L2 (129 MB): a 256 MB buffer is rewritten between timed steps
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if l2_flush_needed(cfg, lens0) else None
    for s in range(args.warmup):
        if flush is not None:
            flush.fill_(s & 255)
        step(s)
    clocks = Clocks(dev.index if dev.index is not None else 0)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    lens_at = [cache.length(b) for b in range(B)]
    launches0 = K.oscar_launch_count()
    K.oscar_kernel_timing(cache.handle, args.steps)     # events around the INT2 attention kernel
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    stp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    # byte counts of the timed steps, worked out before the loop so the host stays ahead of the GPU
    bytes_steps = sum(decode_bytes([lens_at[b] + i + 1 for b in range(B)], hkv, hq) for i in range(args.steps))
    kbytes = sum(int2_kernel_bytes([lens_at[b] + i + 1 for b in range(B)], hkv, hq) for i in range(args.steps))
    t0.record(stream)
    for i in range(args.steps):
        s = args.warmup + i
        if flush is not None:
            flush.fill_(i & 255)      # evicts the previous step's pages from L2; outside the step's events
        stp[i][0].record(stream)
        if args.unfused:
            cache.append(ks[s], vs[s], ones, rk)
            dec[i][0].record(stream)
            cache.attend(qs[s], rk, out)
            dec[i][1].record(stream)
        else:
            dec[i][0].record(stream)
            cache.step(ks[s], vs[s], qs[s], rk, out)
            dec[i][1].record(stream)
        stp[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    cache.status()          # raises if a bounded in-kernel wait gave up
    if dist is not None:
        dist.barrier()
    launches = K.oscar_launch_count() - launches0
    kms = K.oscar_kernel_timing_read(cache.handle, args.steps)
    K.oscar_kernel_timing(cache.handle, 0)
    assert len(kms) == args.steps
    k_t = sum(kms) * 1e-3 / args.steps          # seconds per INT2 attention kernel launch
    k_bytes = kbytes / args.steps
    # with inputs larger than L2 the steps run back to back and the two figures agree; with the L2
    # flush between steps only the steps themselves are counted
    elapsed = (sum(a.elapsed_time(b) for a, b in stp) if flush is not None else t0.elapsed_time(t1)) * 1e-3
    dec_t = sum(a.elapsed_time(b) for a, b in dec) * 1e-3 / args.steps
    elapsed = max_over_ranks(elapsed, dist, dev)
    per_step = elapsed / args.steps
    value = bytes_steps * world / elapsed / 1e9
    dec_bytes = bytes_steps / args.steps
    achieved = k_bytes / k_t / 1e9
    peak, peak_kind = peaks()

    # ---- chunked prefill: every request appends a 256-token chunk and its queries attend causally
    # (outside the timed decode steps; the cache grows by the chunk)
    prefill = None
    if args.path == "mma" and not args.no_prefill:
        nq = [256] * B
        lens_p = [cache.length(b) for b in range(B)]
        if all(lens_p[b] + 256 <= (per_seq - 1) * 64 + 320 for b in range(B)):
            kp, vp = synth.kv_block(seed + 1, nq, lens_p, hkv, device=dev)
            qp = torch.randn(sum(nq), hq, 128, device=dev, generator=torch.Generator(device=dev).manual_seed(seed))
            outp = torch.empty_like(qp)
            wsp = torch.empty(K.oscar_prefill_workspace_bytes(cache.handle), dtype=torch.uint8, device=dev)
            cache.append(kp, vp, nq, rk)
            K.oscar_prefill_attention(cache.handle, qp, K.DTYPE_F32, nq, rk, outp, K.DTYPE_F32, wsp)   # warm
            torch.cuda.synchronize()
            p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            p0.record(stream)
            K.oscar_prefill_attention(cache.handle, qp, K.DTYPE_F32, nq, rk, outp, K.DTYPE_F32, wsp)
            p1.record(stream)
            p1.synchronize()
            pms = p0.elapsed_time(p1)
            prefill = {"what": "oscar_prefill_attention: 256 new tokens per request attending causally over the "
                               "mixed cache (INT2 history + BF16 sink / window)", "chunk": 256,
                       "ms": pms, "query_tokens_per_s": sum(nq) / (pms * 1e-3)}
            del kp, vp, qp, outp, wsp

    layers = None
    if not args.no_layers and world == 1:
        layers = time_layer_appends(B, hq, hkv, dev)

    # ---- end to end: pinned host inputs in, output out, synchronised every step
    e2e = None
    if not args.no_e2e:
        base = args.warmup + args.steps
        # each step's q, k and v packed into one pinned host buffer, so one copy brings them in
        nq = qs[0].numel() * qs[0].element_size()
        nk = ks[0].numel() * ks[0].element_size()

        def packed(s):
            buf = torch.empty(nq + 2 * nk, dtype=torch.uint8, pin_memory=True)
            buf[:nq].copy_(qs[base + s].cpu().view(torch.uint8).reshape(-1))
            buf[nq:nq + nk].copy_(ks[base + s].cpu().view(torch.uint8).reshape(-1))
            buf[nq + nk:].copy_(vs[base + s].cpu().view(torch.uint8).reshape(-1))
            return buf
        h_in = [packed(s) for s in range(args.warmup + args.steps)]
        host_out = torch.empty(B, hq, 128, pin_memory=True)
        d_in = torch.empty(nq + 2 * nk, dtype=torch.uint8, device=dev)
        dq = d_in[:nq].view(qs[0].dtype).view(qs[0].shape)
        dk = d_in[nq:nq + nk].view(ks[0].dtype).view(ks[0].shape)
        dv = d_in[nq + nk:].view(vs[0].dtype).view(vs[0].shape)
        e_bytes = 0
        enqueue = 0.0
        enq_steps, wall_steps = [], []       # per timed step: host enqueue, and enqueue to synchronised
        lens_e = [cache.length(b) for b in range(B)]
        # the fused step takes the host buffers itself (oscar_decode_step_host: copies in, step, copy out)
        qd_e = K.DTYPE_BF16 if qs[0].dtype == torch.bfloat16 else K.DTYPE_F32
        staging = None if args.unfused else torch.empty(
            K.oscar_decode_step_host_staging_bytes(cache.handle, qd_e, K.DTYPE_F32), dtype=torch.uint8, device=dev)
        for s in range(args.warmup + args.steps):
            if s == args.warmup:
                if dist is not None:
                    dist.barrier()
                torch.cuda.synchronize()
                w0 = time.perf_counter()
            h0 = time.perf_counter()
            if staging is not None:
                a = h_in[s].data_ptr()
                K.oscar_decode_step_host(cache.handle, a + nq, a + nq + nk, a, qd_e, rk, host_out, K.DTYPE_F32,
                                         staging, cache.workspace, stream)
            else:
                d_in.copy_(h_in[s], non_blocking=True)
                step_call(dk, dv, dq)
                host_out.copy_(out, non_blocking=True)
            if s >= args.warmup:
                enqueue += time.perf_counter() - h0
                enq_steps.append(time.perf_counter() - h0)
            stream.synchronize()
            if s >= args.warmup:
                wall_steps.append(time.perf_counter() - h0)
                e_bytes += decode_bytes([lens_e[b] + s + 1 for b in range(B)], hkv, hq)
        w1 = time.perf_counter()
        welapsed = w1 - w0
        welapsed = max_over_ranks(welapsed, dist, dev)
        h2d = d_in.numel()
        e2e = {"call": ("oscar_decode_step_host on page-locked host q, k, v and output (copies in, fused step, "
                        "copy out)" if staging is not None else
                        "host-to-device copy, kv_quant_append + oscar_decode_attention, device-to-host copy") +
                       ", stream synchronised every step",
               "value": e_bytes * world / welapsed / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": host_out.numel() * host_out.element_size(),
               "ms_per_step": welapsed / args.steps * 1e3,
               "host_enqueue_ms_per_step": enqueue / args.steps * 1e3,
               # spread of the per-step host times, so that a stall of the host shows as such
               "step_ms_median": 1e3 * sorted(wall_steps)[len(wall_steps) // 2] if wall_steps else None,
               "step_ms_max": 1e3 * max(wall_steps) if wall_steps else None,
               "host_enqueue_ms_max": 1e3 * max(enq_steps) if enq_steps else None}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        threads = max(1, min(args.cpu_pairs, os.cpu_count() or 1))
        nb, times, pairs, ctx = cpu_oracle_sample(cfg, lens0, args.cpu_pairs, reps=4, threads=threads)
        cpu = {"value": sum(nb) / sum(times) / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"four decode steps (append 1 token + attend, fp64) of {len(pairs)} of {B * hkv} "
                         f"(request, KV head) pairs at full context on {threads} threads, "
                         f"{sum(times):.1f} s wall ({sum(times) * threads:.0f} thread-s)"}
        if threads > 1:
            # the same oracle on one host thread (one pair, two steps: a smaller sample of the same work)
            nb1, t1, _, _ = cpu_oracle_sample(cfg, lens0, 1, reps=2, threads=1)
            cpu["single_thread"] = {"value": sum(nb1) / sum(t1) / 1e9, "unit": "GB/s", "cores": 1,
                                    "sample": "two decode steps of 1 (request, KV head) pair at full context, "
                                              f"{sum(t1):.1f} s"}
    kname = dict(mma="decode_mma", simt="split_simt")[args.path]
    if args.unfused or args.path != "mma":
        call_what = (f"oscar_decode_attention: prep (q rotation + BF16 sink/window attention) + {kname} + combine"
                     if args.path == "mma" else
                     f"oscar_decode_attention: rotate_q + {kname} (INT2 and BF16 splits) + combine")
        call_what += "; the step adds kv_quant_append before it"
    else:
        call_what = (f"oscar_decode_step (the whole step): prep with the append of one token per request "
                     f"(window insert, leaving key rotated and quantised) + {kname} + combine")
    workload = workload_config(cfg, lens0)
    line = {
        "metric": "decode_attention_hbm_gbs", "value": value, "unit": "GB/s", "n_gpus": world, "world_size": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16-mma/fp32-acc", "data": "synthetic",
        "precision": PRECISION[args.path],
        "config": workload,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind,
                     "nominal": {"peak": NOMINAL_HBM_GBS, "frac": achieved / NOMINAL_HBM_GBS},
                     "traffic": profiled_traffic(workload["workload"], k_bytes),
                     "kernel": kname, "bytes_per_launch": k_bytes, "ms_per_launch": k_t * 1e3,
                     "timing": "CUDA events recorded by the library on the launching stream around each launch",
                     "call": {"what": call_what, "bytes": dec_bytes, "ms": dec_t * 1e3, "gbs": dec_bytes / dec_t / 1e9}},
        "append": {"prefill_tokens_per_s": tok_append / t_append, "prefill_tokens": tok_append,
                   # the two bounds of the bulk write path: FP32 FMA for the serial key rotation
                   # (128 x 128 per token-head) and HBM (512 bytes read + 80 written per token-head)
                   **write_path_fractions(tok_append * hkv / t_append, dev, clk, peak),
                   "step_ms_outside_int2_kernel": (per_step - k_t) * 1e3},
        "calibration": calib,
        "prefill_attention": prefill,
        "append_layers": layers,
        "clocks": clk,
        "gpu_launches": launches,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def write_path_fractions(token_heads_per_s, dev, clk, hbm_peak):
    """Bulk-prefill throughput against its two bounds: the FP32 FMA rate (SMs x 128 FMA per clock x the
    maximum SM clock sampled, else 2070 MHz) that the 16384 FMA of each key rotation need, and HBM
    (592 algorithmic bytes per token-head against the measured copy peak)."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = (clk or {}).get("sm_max_mhz") or 2070.0
    fma_peak = sms * 128 * mhz * 1e6
    fma = token_heads_per_s * ROTATION_FMA_PER_TOKEN_HEAD
    gbs = token_heads_per_s * 592 / 1e9
    return {"fp32_fma_per_s": fma, "fp32_fma_peak": fma_peak, "fp32_fma_frac": fma / fma_peak,
            "fp32_fma_peak_rule": f"{sms} SMs x 128 FP32 FMA per clock x {mhz:.0f} MHz",
            "hbm_gbs": gbs, "hbm_frac": gbs / hbm_peak}


ROTATION_FMA_PER_TOKEN_HEAD = 128 * 128


def time_layer_appends(B, hq, hkv, dev, n_layers=64, L0=512, chunk=16, reps=10):
    """Write path of one step of an n_layers-layer model: every layer's cache appends `chunk` tokens
    per request, as one kv_quant_append_layers call or as one kv_quant_append call per layer.  Host
    wall time per step (enqueue included, synchronised after the timed steps)."""
    import time

    import torch

    import synth
    import int2_rotated_paged_gb300 as K
    per_seq = (L0 + chunk * (reps + 4) - 320 + 63) // 64 + 2
    sets = [[K.Cache(B, hq, hkv, per_seq * B, per_seq) for _ in range(n_layers)] for _ in range(2)]
    rk = torch.linalg.qr(torch.randn(hkv, 128, 128, device=dev))[0].contiguous()
    k0, v0 = synth.kv_block(3, [L0] * B, [0] * B, hkv, device=dev)
    for cs in sets:
        for c in cs:
            c.append(k0, v0, [L0] * B, rk)
    k1, v1 = synth.kv_block(4, [chunk] * B, [L0] * B, hkv, device=dev)
    ws = torch.empty(K.kv_quant_append_layers_workspace_bytes(n_layers), dtype=torch.uint8, device=dev)
    n = [chunk] * B

    def batched():
        K.kv_quant_append_layers(sets[0], [k1] * n_layers, [v1] * n_layers, n, [rk] * n_layers, ws)

    def per_layer():
        for c in sets[1]:
            c.append(k1, v1, n, rk)
    res = {}
    for name, f in (("batched", batched), ("per_layer", per_layer)):
        f()
        f()
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(reps):
            f()
        torch.cuda.synchronize()
        res[name] = (time.perf_counter() - t) / reps * 1e3
    del sets
    torch.cuda.empty_cache()
    return {"what": f"one step's write path of a {n_layers}-layer model: {chunk} new tokens per request into every "
                    "layer's cache (host wall time per step, enqueue included)",
            "layers": n_layers, "tokens_per_request": chunk,
            "one_call_ms": res["batched"], "call_per_layer_ms": res["per_layer"]}


def relaunch_under_torchrun(args) -> int:
    """`bench.py --gpus N` (N > 1) started without torchrun: start N ranks on this node with
    torch.distributed.run (rendezvous on 127.0.0.1) and return their exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.run(cmd).returncode


def main():
    args = parse()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(relaunch_under_torchrun(args))
    import synth
    names = synth.CONFIG_NAMES if args.config == "all" else [args.config]
    cfgs = [synth.config(nm) for nm in names]
    if args.batch:
        cfgs = [synth.scaled(cfg, cfg.ctx, batch=args.batch) for cfg in cfgs]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world != args.gpus:
        sys.exit(f"--gpus {args.gpus} but WORLD_SIZE {world}: launch one rank per GPU")
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group(backend)
        dist = tdist
    try:
        for cfg in cfgs:
            if args.impl == "reference":
                run_reference(args, cfg, rank, world)
            else:
                run_ours(args, cfg, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
