"""CSA2 sparse-decode benchmark.

One step = one decode token per sequence through a CSA2 layer group: write
the new token's FP4 main-KV entry, then every layer of the workload's schedule
(Full: indexer sweep + top-K (+ HSI pool) + sparse readout; Reindex: pool
sweep + top-K + readout; Reuse: readout), on seeded synthetic inputs resident
in HBM.  The step is captured once in a CUDA graph and replayed; each step is
timed with CUDA events on the launching stream and L2 is flushed (a 512 MB
write) between steps, outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config group_decode_32x64k|hsi_reindex_16x256k|decoder20_4x1m] [--impl ours|reference]

N > 1 (torchrun): replicas -- every rank runs the same per-GPU workload on its
own GPU; value = total tokens of all ranks / max-over-ranks time.
--impl reference times the oracle (plain fp64 CPU implementation) on the host
cores, on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 sparse-decode tokens/s at 64K/1M ctx; achieved HBM GB/s vs ~8 TB/s"
ATTN_BYTES = 512 * 288 + (128 * 512 + 128 * 4) + 64 * 512 * 2 + 64 * 512 * 4 + 512 * 4   # per (seq, layer)
SWEEP_FIXED = 32 * 128 * 2 + 32 * 4        # q_idx + w per sequence
REINDEX_BYTES = 16384 * 256 + 18560         # per (seq, layer)
KVW_BYTES = 1024 + 288 + 16                 # new entry per sequence


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="group_decode_32x64k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling runs)")
    return ap.parse_args()


def algorithmic_bytes(cfg, hsi):
    B, N = cfg.batch, cfg.n_ctx
    total = B * KVW_BYTES
    for m in cfg.schedule:
        total += B * ATTN_BYTES
        if m == "full":
            total += B * (256 * N + SWEEP_FIXED + 512 * 4)
        elif m == "reindex":
            total += B * REINDEX_BYTES
    return total


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, path):
        self.path = path
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self, device_index):
        if not self.proc or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9 or not f[0].isdigit() or int(f[0]) != device_index:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class Workload:
    """Device-resident inputs of one decode step and its launch sequence."""

    def __init__(self, cfg, device):
        import torch

        import synth
        import sparse_attention_fp4_csa2_gb300 as c2
        self.c2, self.cfg, self.dev = c2, cfg, device
        B, N = cfg.batch, cfg.n_ctx
        self.B, self.N = B, N
        self.hsi = 1 if cfg.hsi else 0
        self.params = c2.Params.make(hsi=self.hsi)
        seed = cfg.layer_seeds[0]
        # context: latents -> FP4 main KV with this library's writer; indexer K bf16
        self.kv = torch.empty(B, N, 288, dtype=torch.uint8, device=device)
        chunk = max(1, (1 << 22) // N)       # sequences per writer call (bounded temporary)
        for b0 in range(0, B, chunk):
            nb = min(chunk, B - b0)
            lat = synth.context_latent(seed * 977 + b0, nb, N, device=device)
            pos = torch.arange(N, dtype=torch.int64, device=device).repeat(nb)
            slot = torch.arange(b0 * N, (b0 + nb) * N, dtype=torch.int64, device=device)
            c2.kv_quant_write(lat.reshape(nb * N, 512), None, 1, pos, slot, self.kv.view(B * N, 288))
            del lat
        self.k_idx = synth.indexer_keys(seed, B, N, device=device)
        if cfg.planted_blocks:
            li0 = synth.layer_inputs(cfg.layer_seeds[0], B, device=device)
            synth.plant_blocks(self.k_idx, li0.q_idx, li0.w, N, cfg.planted_blocks, seed)
        self.layers = [synth.layer_inputs(s, B, device=device) for s in cfg.layer_seeds]
        self.new_latent = synth.normal((B, 512), seed + 7, 0, device)
        self.new_pos = torch.full((B,), N - 1, dtype=torch.int64, device=device)
        self.new_slot = torch.arange(B, dtype=torch.int64, device=device) * N + (N - 1)
        self.n_vis = torch.full((B,), N, dtype=torch.int32, device=device)
        self.topk = torch.zeros(B, 512, dtype=torch.int32, device=device)
        self.pool = torch.zeros(B, 2048, dtype=torch.int32, device=device)
        self.out = torch.empty(len(cfg.schedule), B, 64, 512, device=device)
        self.lse = torch.empty(len(cfg.schedule), B, 64, device=device)
        self.ws = c2.workspace(c2.OP_DECODE, B, N, self.params, device=device)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    def step(self, sweep_events=None):
        """Enqueue one decode step; with sweep_events, the Full layer's indexer
        sweep launch is bracketed by those events."""
        c2, L = self.c2, self.layers
        launches = 0
        c2.kv_quant_write(self.new_latent, None, 1, self.new_pos, self.new_slot, self.kv.view(-1, 288))
        launches += c2.last_launch_count()
        for i, mode in enumerate(self.cfg.schedule):
            li = L[i]
            idx_args = {} if mode == "reuse" else dict(q_idx=li.q_idx, w=li.w, k_idx=self.k_idx)
            if sweep_events and mode == "full":
                c2.set_profile_events(c2.KERNEL_INDEXER_SWEEP, *sweep_events)
            c2.sparse_decode(mode, self.params, li.q, self.kv, self.n_vis, self.N, li.swa, li.swa_scale,
                             li.swa_len, self.topk, self.out[i], self.ws, pool_blocks=self.pool,
                             lse=self.lse[i], **idx_args)
            if sweep_events and mode == "full":
                c2.set_profile_events(c2.KERNEL_INDEXER_SWEEP, None, None)
            launches += c2.last_launch_count()
        return launches

    def host_io(self):
        """Pinned host copies of every per-step input and output (for e2e)."""
        import torch
        ins = [self.new_latent] + [t for li in self.layers for t in (li.q, li.swa, li.swa_scale)]
        ins += [t for li, m in zip(self.layers, self.cfg.schedule) if m != "reuse" for t in (li.q_idx, li.w)]
        hin = [(t.cpu().pin_memory(), t) for t in ins]
        hout = [(torch.empty(t.shape, dtype=t.dtype).pin_memory(), t) for t in (self.out, self.lse)]
        return hin, hout


def run_ours(args, rank, world, local_rank):
    import torch

    import synth
    import sparse_attention_fp4_csa2_gb300 as c2
    from sparse_attention_fp4_csa2_gb300 import build as b
    b.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = synth.CONFIGS[args.config]
    if args.batch:
        import dataclasses
        cfg = dataclasses.replace(cfg, batch=args.batch, name=f"{cfg.name}[batch={args.batch}]")
    wl = Workload(cfg, dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush2 = torch.ones(128 << 20, dtype=torch.float32, device=dev)

    # eager warm-up (also counts our launches per step), then capture the step
    with torch.cuda.stream(stream):
        launches = wl.step()
    stream.synchronize()
    assert c2.get_device_status(stream) == 0
    sweep_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    attn_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for ev in sweep_ev + attn_ev:
        ev.record(stream)          # marks the events recorded; the graph re-records them every replay
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        wl.step(sweep_events=sweep_ev)

    def flush_l2():
        # write a buffer larger than L2, then read another one so the written
        # lines are evicted (written back) before the timed region starts
        flush.zero_()
        flush2.sum()

    for _ in range(max(3, args.warmup)):
        with torch.cuda.stream(stream):
            flush_l2()
            g.replay()
    stream.synchronize()

    def timed(n, with_io=None):
        tot, sweep = 0.0, []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(n):
            with torch.cuda.stream(stream):
                flush_l2()
                e0.record(stream)
                if with_io:
                    for h, d in with_io[0]:
                        d.copy_(h, non_blocking=True)
                g.replay()
                if with_io:
                    for h, d in with_io[1]:
                        h.copy_(d, non_blocking=True)
                e1.record(stream)
            stream.synchronize()
            tot += e0.elapsed_time(e1)
            sweep.append(sweep_ev[0].elapsed_time(sweep_ev[1]))
        return tot, sweep

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(os.path.join(ROOT, "gpurun_out", f"clocks_r{rank}.csv") if os.path.isdir(
            os.path.join(ROOT, "gpurun_out")) else f"/tmp/csa2_clocks_r{rank}.csv") as clk:
        total_ms, sweep_ms = timed(args.steps)
    torch.cuda.synchronize()
    t = torch.tensor([total_ms], device=dev)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.barrier()
    total_ms = float(t.item())

    # end to end: per-step inputs copied from pinned host memory, outputs read back
    hin, hout = wl.host_io()
    e2e_steps = max(3, min(args.steps, 10))
    e2e_ms, _ = timed(e2e_steps, with_io=(hin, hout))
    h2d = sum(h.numel() * h.element_size() for h, _ in hin)
    d2h = sum(h.numel() * h.element_size() for h, _ in hout)
    assert c2.get_device_status(stream) == 0

    B = cfg.batch
    ms = total_ms / args.steps
    tokens_per_s = world * B / (ms / 1e3)
    hbm, kind = peaks()
    sweep_avg = statistics.mean(sweep_ms) if sweep_ms and "full" in cfg.schedule else None
    roof = None
    if sweep_avg:
        alg = B * (256 * cfg.n_ctx + SWEEP_FIXED)
        ach = alg / (sweep_avg / 1e3) / 1e9
        roof = {"kernel": "indexer_sweep_kernel", "bound": "hbm", "achieved": round(ach, 1),
                "peak": hbm, "peak_kind": kind, "unit": "GB/s", "frac": round(ach / hbm, 4),
                "traffic": None, "launch_ms": round(sweep_avg, 4), "alg_bytes_per_launch": alg}
    step_bytes = algorithmic_bytes(cfg, wl.hsi)
    line = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "batch": B, "context": cfg.n_ctx, "layers": "+".join(cfg.schedule),
                   "hsi": bool(wl.hsi), "l2": "flushed between steps (512 MB write, then 512 MB read), outside the timed events",
                   "storage": "FP4 E2M1+E4M3/16 main KV, bf16 indexer K, E4M3 SWA",
                   "step_alg_bytes": step_bytes,
                   "step_hbm_gbs": round(step_bytes / (ms / 1e3) / 1e9, 1)},
        "roofline": roof,
        "e2e": {"value": round(world * B / (e2e_ms / e2e_steps / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(local_rank),
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args, cfg, seconds=args.cpu_seconds)
        print(json.dumps(line), flush=True)


def cpu_baseline(args, cfg, seconds=12.0):
    """The oracle, as it stands, on the host cores: whole decode steps of
    single sequences of the same workload until ~`seconds` elapse."""
    import numpy as np
    import torch

    import oracle
    import synth
    oracle.build()
    B, N = cfg.batch, cfg.n_ctx
    seed = cfg.layer_seeds[0]
    layers = [synth.layer_inputs(s, 1) for s in cfg.layer_seeds]
    done, t_total, b = 0, 0.0, 0
    while b < B and (t_total < seconds or done == 0):
        k = synth.indexer_keys(seed * 31 + b, 1, N)[0]
        lat = synth.context_latent(seed * 37 + b, 1, N)[0]
        t0 = time.perf_counter()
        sel = pool = None
        for i, mode in enumerate(cfg.schedule):
            li = layers[i]
            if mode == "full":
                s = oracle.index_scores(li.q_idx[0], li.w[0], k)
                sel = oracle.topk(s, 512)
                if cfg.hsi:
                    pool = oracle.hsi_pool(s, N, 8, 2048)
            elif mode == "reindex":
                sel = oracle.reindex_topk(li.q_idx[0], li.w[0], k, pool, N, 512)
            valid = sel[sel >= 0]
            rows = oracle.kv_entries(lat[valid], None, 1, valid)
            oracle.sparse_attn(li.q[0], rows, np.arange(len(valid)), li.swa[0], li.swa_scale[0], 128)
        t_total += time.perf_counter() - t0
        done += 1
        b += 1
    return {"value": round(done / t_total, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"{done} of {B} sequences, one full step each ({cfg.name}); "
                                        f"FP4 entries of the selected rows written inside the timed region"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import synth
    cfg = synth.CONFIGS[args.config]
    per_step = []
    for _ in range(args.steps):
        r = cpu_baseline(args, cfg, seconds=max(1.0, args.cpu_seconds / max(1, args.steps)))
        per_step.append(r)
    v = statistics.mean(r["value"] for r in per_step)
    line = {"metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(cfg.batch / v * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "batch": cfg.batch, "context": cfg.n_ctx,
                       "layers": "+".join(cfg.schedule)},
            "impl": "reference",
            "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": per_step[0]["cores"],
                             "kind": "oracle", "sample": per_step[0]["sample"]},
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
