"""Benchmark: KV tokens scored + compacted per second per layer, with the HBM / tensor roofline.

One step = one pass of the prefill compression hot path over one synthetic layer: window
scores (two passes over K on tensor cores) -> per-KV-head top-k with the observation window
protected -> gather-compaction of the kept K/V rows.  Default workload: the SnapKV prefill of
a Llama-3-8B-shaped layer (batch 1, 32 query / 8 KV heads, head_dim 128, 32768 tokens,
window 64, keep 4096 per KV head, bf16, 1% heavy-hitter keys).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (torchrun): every rank compresses its own replica (independent layers, weak scaling,
no collective on the data path); the timed region is bracketed by barriers and the max over
ranks is reported.
"""
from __future__ import annotations

import argparse
import json
import math
import multiprocessing as mp
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import WORKLOADS, SNAPKV_32K, prefill_inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_gpu{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------------
# CPU baseline: the oracle, timed in a spawned child (no CUDA in that process)
# ----------------------------------------------------------------------------------------


def _oracle_sample(config: str, budget_s: float, threads: int, q):
    os.environ.setdefault("OPENBLAS_NUM_THREADS", str(threads))
    os.environ.setdefault("OMP_NUM_THREADS", str(threads))
    import oracle as O
    wl = WORKLOADS[config]
    inp = prefill_inputs(wl)
    G = wl.G
    t0 = time.perf_counter()
    heads = 0
    # sample: one KV head (its G query heads, the whole sequence) per iteration
    while True:
        kv = heads % wl.KVH
        qg = inp["q"][:, kv * G:(kv + 1) * G]
        Kg = inp["K"][:, kv:kv + 1]
        Vg = inp["V"][:, kv:kv + 1]
        O.compress_prefill(qg, Kg, Vg, wl.scale, wl.k, protect_tail=wl.protect_tail, reduce="gqa")
        heads += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    tokens = wl.B * wl.S * heads / wl.KVH  # a layer's tokens are scored once all KV heads are done
    q.put({"value": tokens / dt, "seconds": dt, "kv_heads": heads})


def cpu_baseline(config: str, budget_s: float = 10.0):
    threads = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_oracle_sample, args=(config, budget_s, threads, q))
    p.start()
    res = q.get(timeout=budget_s * 20 + 600)
    p.join()
    wl = WORKLOADS[config]
    return {"value": res["value"], "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{res['kv_heads']} KV-head groups of the {wl.name} layer (oracle compress_prefill, "
                      f"float64 numpy, {res['seconds']:.1f} s), scaled to a full layer of {wl.KVH} KV heads"}


# ----------------------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ----------------------------------------------------------------------------------------


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = WORKLOADS[args.config]
    threads = os.cpu_count() or 1
    import oracle as O
    inp = prefill_inputs(wl)
    G = wl.G

    def step(i):
        kv = i % wl.KVH
        O.compress_prefill(inp["q"][:, kv * G:(kv + 1) * G], inp["K"][:, kv:kv + 1], inp["V"][:, kv:kv + 1],
                           wl.scale, wl.k, protect_tail=wl.protect_tail, reduce="gqa")

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = wl.B * wl.S * args.steps / wl.KVH / dt
    line = {"impl": "reference", "metric": "kv_tokens_scored_compacted_per_s_per_layer", "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "sample": "one KV head per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: one of {wl.KVH} KV-head groups of {wl.name}, scaled to a layer"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import attention_score_kv_window_gb300 as kvc

    kvc.load_library()
    wl = WORKLOADS[args.config]
    peaks = _peaks()

    inp = prefill_inputs(wl, seed=wl.seed + rank)

    def to_dev(u16):
        return torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16).to(dev)

    q0, K0, V0 = to_dev(inp["q"]), to_dev(inp["K"]), to_dev(inp["V"])
    in_bytes = (q0.numel() + K0.numel() + V0.numel()) * 2
    R = max(2, math.ceil(3 * L2_BYTES / in_bytes))
    reps = [(q0, K0, V0)] + [(q0.clone(), K0.clone(), V0.clone()) for _ in range(R - 1)]
    B, KVH, S, D = K0.shape
    k = min(wl.k, S)
    outs = [(torch.empty((B, KVH, S), dtype=torch.float32, device=dev),
             torch.empty((B, KVH, k), dtype=torch.int32, device=dev),
             torch.empty((B, KVH, k, D), dtype=torch.bfloat16, device=dev),
             torch.empty((B, KVH, k, D), dtype=torch.bfloat16, device=dev)) for _ in range(R)]
    ws_bytes = kvc.load_library().kvc_workspace_size(2, kvc.kv_desc(K0, wl.H), wl.w, k)
    ws = torch.empty(int(ws_bytes), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(i, ev=None):
        q, K, V = reps[i % R]
        sc, idx, Ko, Vo = outs[i % R]
        if ev is not None:
            ev[0].record(stream)
        kvc.kvc_window_scores(q, K, wl.scale, causal=True, reduce=wl.reduce, scores=sc, ws=ws)
        if ev is not None:
            ev[1].record(stream)
        kvc.kvc_topk_select(sc, k, protect_tail=wl.protect_tail, idx=idx)
        if ev is not None:
            ev[2].record(stream)
        kvc.kvc_compact_kv(K, V, idx, H=wl.H, K_out=Ko, V_out=Vo)
        if ev is not None:
            ev[3].record(stream)

    launches_per_step = 3 + (1 if wl.reduce == "all_heads" else 0) + 1 + 1

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert kvc.kvc_get_device_status() == kvc.KVC_OK

    sampler = ClockSampler(local) if not args.no_clocks else None
    if sampler:
        sampler.start()
        # keep the GPU busy for a moment so the sampler sees the loaded clock
        t_end = time.time() + 0.5
        i = 0
        while time.time() < t_end:
            step(i)
            i += 1
        torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        step(i, evs[i])
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = start.elapsed_time(stop)
    clocks = sampler.stop() if sampler else None
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    assert kvc.kvc_get_device_status() == kvc.KVC_OK

    t_scores = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    t_topk = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    t_compact = float(np.mean([e[2].elapsed_time(e[3]) for e in evs]))

    tokens_per_step = B * S
    value = tokens_per_step * args.steps * world / (ms / 1e3)

    # roofline of the dominant call: window scores (two passes over K on the tensor cores)
    G = wl.H // wl.KVH
    flops = 2 * 2.0 * B * wl.H * wl.w * S * D  # two passes of q_win K^T (the pass structure the method fixes)
    achieved_tflops = flops / (t_scores / 1e3) / 1e12
    roof = {"kernel": "kvc_window_scores (pass 1 + merge + pass 2)", "bound": "tensor",
            "achieved": achieved_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved_tflops / peaks["bf16_tflops"], "traffic": None,
            "peak_source": f"{peaks['source']} bf16 burst",
            "algorithmic_flops_per_launch": flops,
            "algorithmic_bytes_per_launch": B * KVH * S * D * 2 + B * wl.H * wl.w * D * 2 + B * KVH * S * 4}
    sc_bytes = roof["algorithmic_bytes_per_launch"]
    compact_bytes = 4 * B * KVH * k * D * 2 + B * KVH * k * 4
    kernels = {
        "window_scores_ms": t_scores,
        "window_scores_hbm_gbs": sc_bytes / (t_scores / 1e3) / 1e9,
        "topk_ms": t_topk,
        "compact_ms": t_compact,
        "compact_hbm_gbs": compact_bytes / (t_compact / 1e3) / 1e9,
    }

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    hq = torch.from_numpy(inp["q"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hK = torch.from_numpy(inp["K"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hV = torch.from_numpy(inp["V"].view(np.int16)).view(torch.bfloat16).pin_memory()
    h_idx = torch.empty((B, KVH, k), dtype=torch.int32).pin_memory()
    h_Ko = torch.empty((B, KVH, k, D), dtype=torch.bfloat16).pin_memory()
    h_Vo = torch.empty((B, KVH, k, D), dtype=torch.bfloat16).pin_memory()
    dq, dK, dV = reps[0]
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step(i):
        dq.copy_(hq, non_blocking=True)
        dK.copy_(hK, non_blocking=True)
        dV.copy_(hV, non_blocking=True)
        sc, idx, Ko, Vo = outs[0]
        kvc.kvc_compress_prefill(dq, dK, dV, wl.scale, k, protect_tail=wl.protect_tail, reduce=wl.reduce,
                                 out=(sc, idx, Ko, Vo), ws=ws)
        h_idx.copy_(idx, non_blocking=True)
        h_Ko.copy_(Ko, non_blocking=True)
        h_Vo.copy_(Vo, non_blocking=True)

    e2e_step(0)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if world > 1:
        t = torch.tensor([e2e_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e = {"value": tokens_per_step * e2e_steps * world / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": int((hq.numel() + hK.numel() + hV.numel()) * 2),
           "d2h_bytes_per_step": int(h_idx.numel() * 4 + (h_Ko.numel() + h_Vo.numel()) * 2)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.config, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": "kv_tokens_scored_compacted_per_s_per_layer", "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": wl.name, "B": B, "H": wl.H, "KVH": KVH, "D": D, "S": S, "w": wl.w, "k": k,
                       "l2": f"inputs rotate over {R} replicas ({R * in_bytes / 2**20:.0f} MiB > L2)"},
            "roofline": roof, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=SNAPKV_32K.name,
                    choices=[n for n, w in sorted(WORKLOADS.items()) if w.steps == 0])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
