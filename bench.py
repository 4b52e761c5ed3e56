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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen3_32b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-pairs", type=int, default=3, help="(request, KV head) pairs the CPU oracle times")
    ap.add_argument("--batch", type=int, default=0,
                    help="requests per GPU (0 = the workload's batch); smaller values are for profiling")
    ap.add_argument("--path", default="mma", choices=["mma", "tensor", "simt"],
                    help="decode kernel: warp-level MMA (default), tcgen05, or the SIMT baseline")
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


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def profiled_traffic(kernel_src: str):
    """DRAM bytes per decode call from the committed ncu summary, if it still matches the source."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    src = os.path.join(ROOT, "int2_rotated_paged_gb300", "csrc", kernel_src)
    try:
        with open(path) as f:
            rec = json.load(f)
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return rec["bytes_per_call"] if rec.get("source_sha256_16") == h else None
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
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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


# ------------------------------------------------------------------ CPU oracle timing

def cpu_oracle_sample(cfg, lens, n_pairs: int, reps: int = 1):
    """Time the CPU oracle's decode attention on (request, KV head) pairs of the workload."""
    import numpy as np
    import oracle
    import synth
    oracle.build()
    pairs = [(b % cfg.batch, (3 * b + 1) % cfg.num_kv_heads) for b in range(n_pairs)]
    caches = []
    for (b, h) in pairs:
        rk = oracle.build_rk(synth.calibration_queries(cfg.seed, h, 4096).numpy())[0]
        oc = oracle.OracleCache(rk)
        oc.append(synth.bf16_bits(synth.keys(cfg.seed, b, h, 0, lens[b])),
                  synth.bf16_bits(synth.values(cfg.seed, b, h, 0, lens[b])))
        caches.append((b, h, oc))
    q = synth.queries(cfg.seed, 0, cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, dtype=cfg.q_dtype).numpy()
    g = cfg.group
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        for (b, h, oc) in caches:
            oc.attend(q[b, h * g:(h + 1) * g])
        times.append(time.perf_counter() - t0)
    nbytes = sum(decode_bytes([lens[b]], 1, g) for (b, h, _) in caches)
    return nbytes, times, pairs


# ------------------------------------------------------------------ main arms

def run_reference(args, cfg, rank, world):
    if rank != 0:
        return
    lens = [int(x) for x in cfg.ctx]
    nbytes, times, pairs = cpu_oracle_sample(cfg, lens, args.cpu_pairs, reps=args.warmup + args.steps)
    t = times[args.warmup:]
    per = sum(t) / len(t)
    value = nbytes / per / 1e9
    line = {
        "impl": "reference", "metric": "decode_attention_hbm_gbs", "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: B{cfg.batch} Hq{cfg.num_q_heads}/Hkv{cfg.num_kv_heads} "
                               f"d128 L{lens[0]} INT2 paged decode", "sample": f"{len(pairs)} (request, KV head) pairs"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{len(pairs)} of {cfg.batch * cfg.num_kv_heads} (request, KV head) pairs, full context"},
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
    K.oscar_set_decode_path({"mma": K.PATH_WARP_MMA, "tensor": K.PATH_TENSOR, "simt": K.PATH_SIMT}[args.path])
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
    del ws, qcal

    # ---- cache with scrambled physical pages
    per_seq = max(1, (max(lens0) + total_steps - 320 + 63) // 64 + 1)
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

    def step(s):
        cache.append(ks[s], vs[s], [1] * B, rk)
        cache.attend(qs[s], rk, out)

    for s in range(args.warmup):
        step(s)
    clocks = Clocks(dev.index if dev.index is not None else 0)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    lens_at = [cache.length(b) for b in range(B)]
    launches0 = K.oscar_launch_count()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    bytes_steps = 0
    t0.record(stream)
    for i in range(args.steps):
        s = args.warmup + i
        cache.append(ks[s], vs[s], [1] * B, rk)
        bytes_steps += decode_bytes([lens_at[b] + i + 1 for b in range(B)], hkv, hq)
        dec[i][0].record(stream)
        cache.attend(qs[s], rk, out)
        dec[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    cache.status()          # raises if a bounded in-kernel wait gave up
    if dist is not None:
        dist.barrier()
    launches = K.oscar_launch_count() - launches0
    elapsed = t0.elapsed_time(t1) * 1e-3
    dec_t = sum(a.elapsed_time(b) for a, b in dec) * 1e-3 / args.steps
    if dist is not None:
        tt = torch.tensor([elapsed], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        elapsed = float(tt.item())
    per_step = elapsed / args.steps
    value = bytes_steps * world / elapsed / 1e9
    dec_bytes = bytes_steps / args.steps
    achieved = dec_bytes / dec_t / 1e9
    peak, peak_kind = peaks()

    # ---- end to end: pinned host inputs in, output out, synchronised every step
    e2e = None
    if not args.no_e2e:
        base = args.warmup + args.steps
        hq_in = [qs[base + s].cpu().pin_memory() for s in range(args.warmup + args.steps)]
        hk_in = [ks[base + s].cpu().pin_memory() for s in range(args.warmup + args.steps)]
        hv_in = [vs[base + s].cpu().pin_memory() for s in range(args.warmup + args.steps)]
        host_out = torch.empty(B, hq, 128, pin_memory=True)
        dq = torch.empty_like(qs[0])
        dk = torch.empty_like(ks[0])
        dv = torch.empty_like(vs[0])
        e_bytes = 0
        lens_e = [cache.length(b) for b in range(B)]
        for s in range(args.warmup + args.steps):
            if s == args.warmup:
                if dist is not None:
                    dist.barrier()
                torch.cuda.synchronize()
                w0 = time.perf_counter()
            dq.copy_(hq_in[s], non_blocking=True)
            dk.copy_(hk_in[s], non_blocking=True)
            dv.copy_(hv_in[s], non_blocking=True)
            cache.append(dk, dv, [1] * B, rk)
            cache.attend(dq, rk, out)
            host_out.copy_(out, non_blocking=True)
            stream.synchronize()
            if s >= args.warmup:
                e_bytes += decode_bytes([lens_e[b] + s + 1 for b in range(B)], hkv, hq)
        w1 = time.perf_counter()
        welapsed = w1 - w0
        if dist is not None:
            tt = torch.tensor([welapsed], dtype=torch.float64, device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            welapsed = float(tt.item())
        h2d = dq.numel() * dq.element_size() + dk.numel() * dk.element_size() + dv.numel() * dv.element_size()
        e2e = {"value": e_bytes * world / welapsed / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": host_out.numel() * host_out.element_size(),
               "ms_per_step": welapsed / args.steps * 1e3}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        nb, times, pairs = cpu_oracle_sample(cfg, lens0, args.cpu_pairs)
        cpu = {"value": nb / times[0] / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"decode attention of {len(pairs)} of {B * hkv} (request, KV head) pairs at "
                         f"{lens0[0]} tokens, fp64, single thread"}
    line = {
        "metric": "decode_attention_hbm_gbs", "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int2+fp32", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: B{B} Hq{hq}/Hkv{hkv} d128 L{lens0[0]} INT2 paged decode step "
                               f"(append 1 token + split-K GQA decode), {cfg.table} pages",
                   "batch_per_gpu": B, "context": lens0[0], "l2": "inputs larger than L2 (about 2.1 GB per step vs 129 MB)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "kernel": f"oscar_decode_attention, {args.path} path (rotate_q + bf16 split + "
                               f"{dict(mma='decode_mma', tensor='decode_tc', simt='split_simt')[args.path]} + combine)",
                     "traffic": profiled_traffic("decode.cu"), "bytes_per_call": dec_bytes,
                     "ms_per_call": dec_t * 1e3},
        "append": {"prefill_tokens_per_s": tok_append / t_append, "prefill_tokens": tok_append,
                   "step_ms_excl_decode": (per_step - dec_t) * 1e3},
        "clocks": clk,
        "gpu_launches": launches,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    import synth
    cfg = synth.config(args.config)
    if args.batch:
        cfg = synth.scaled(cfg, cfg.ctx, batch=args.batch)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
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
        if args.impl == "reference":
            run_reference(args, cfg, rank, world)
        else:
            run_ours(args, cfg, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
