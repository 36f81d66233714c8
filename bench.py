"""Benchmark: KV tokens scored + compacted per second per layer, with the HBM / tensor roofline.

One step = one pass of the prefill compression hot path over one synthetic batch: window
scores -> per-KV-head top-k (the observation window protected for SnapKV) -> gather-compaction
of the kept K/V rows.  Default workload: TOVA prefill (8 query / 2 KV heads, head_dim 64, 512
tokens, the last query's attention averaged over all heads, keep 256 per KV head, bf16), run as
8192 independent instances per step (one layer of 256 requests x 32 layers, or any other set
of independent prefills of this shape); on this shape the library runs the whole path as one
fused kernel.  Other workloads: ``--config``.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]
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
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import WORKLOADS, TOVA_PREFILL, prefill_inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
# independent instances stacked into one step when --instances is not given: TOVA prefill of a
# 512-token layer is far too small to measure alone, so the step runs 8192 of them
DEFAULT_INSTANCES = {TOVA_PREFILL.name: 8192}


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
        # the raw samples go to KVC_CLOCKS_DIR when set (kept for inspection), else a temp dir
        out_dir = os.environ.get("KVC_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"kvc_clocks_gpu{gpu_index}.csv")

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


def _oracle_unit(wl, inp, i):
    """One unit of oracle work on a prefill workload and the tokens it covers.  All-heads
    scoring (TOVA) needs every head of an instance: one whole instance per unit.  Group
    scoring (SnapKV, ThinK): one KV head and its query group per unit, a 1/KVH share of a
    layer's tokens."""
    import oracle as O
    if wl.reduce == "all_heads":
        O.compress_prefill(inp["q"], inp["K"], inp["V"], wl.scale, wl.k, protect_tail=wl.protect_tail,
                           reduce="all_heads")
        return wl.B * wl.S
    G = wl.G
    kv = i % wl.KVH
    O.compress_prefill(inp["q"][:, kv * G:(kv + 1) * G], inp["K"][:, kv:kv + 1], inp["V"][:, kv:kv + 1],
                       wl.scale, wl.k, protect_tail=wl.protect_tail, reduce="gqa")
    return wl.B * wl.S / wl.KVH


def _oracle_worker(config: str, budget_s: float, worker: int, q):
    """One process of the oracle sample: whole units until the time budget is used.  Each
    worker takes its own instance seed (instances are independent units of work)."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"  # before numpy loads its BLAS in this fresh process
    wl = WORKLOADS[config]
    inp = prefill_inputs(wl, seed=wl.seed + worker)
    t0 = time.perf_counter()
    tokens, units = 0.0, 0
    while True:
        tokens += _oracle_unit(wl, inp, units)
        units += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    q.put({"tokens": tokens, "seconds": time.perf_counter() - t0, "units": units})


def _oracle_run(config: str, budget_s: float, workers: int) -> dict:
    """``workers`` spawned processes (no CUDA in them) run the oracle at the same time, each
    on its own units; the rate is the tokens of all of them over the longest one's time."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_oracle_worker, args=(config, budget_s, w, q)) for w in range(workers)]
    for p_ in ps:
        p_.start()
    res = [q.get(timeout=budget_s * 20 + 900) for _ in ps]
    for p_ in ps:
        p_.join()
    dt = max(r["seconds"] for r in res)
    return {"value": sum(r["tokens"] for r in res) / dt, "seconds": dt, "units": sum(r["units"] for r in res)}


def cpu_baseline(config: str, budget_s: float = 10.0):
    """The oracle (float64 numpy, single-threaded per process) on the host's cores: one process
    per core, each on its own independent units, and one process alone for the one-core rate."""
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    res = _oracle_run(config, budget_s / 4, cores)
    one = _oracle_run(config, budget_s, 1)
    wl = WORKLOADS[config]
    unit = "whole instances (B 1)" if wl.reduce == "all_heads" else f"KV-head groups (one of {wl.KVH} per layer)"
    return {"value": res["value"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "single_thread_value": one["value"], "cpu": _cpu_model(),
            "sample": f"{res['units']} {unit} of {wl.name} (oracle compress_prefill, float64 numpy) in "
                      f"{res['seconds']:.1f} s, {cores} processes of one thread each, one per core; "
                      f"rate scaled to tokens"}


def _cpu_model() -> str:
    """The host CPU's model name as the kernel reports it; on Arm the core's part number
    (0xd4f: Neoverse V2, Grace's core), else the architecture name."""
    import platform
    part = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model"):
                    return line.split(":", 1)[1].strip()
                if key == "cpu part" and part is None:
                    part = line.split(":", 1)[1].strip()
    except OSError:
        pass
    if part is not None:
        return f"{platform.machine()} " + ({"0xd4f": "Neoverse V2"}.get(part.lower(), f"cpu part {part}"))
    return platform.machine()


# ----------------------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ----------------------------------------------------------------------------------------


def _reference_case(wl):
    """The oracle's version of one workload step on a sample: (step(i), tokens a step of the
    sample covers, description).  Samples are one KV head (prefill) or one batch row
    (decode); rates scale to the whole workload by tokens."""
    import oracle as O
    from synth import decode_step_inputs, normal_bf16
    G = wl.G
    name = wl.name
    if name.startswith("tova_decode"):
        n = wl.k + 1
        Kc = normal_bf16((1, wl.KVH, n, wl.D), wl.seed, 901)
        Vc = normal_bf16((1, wl.KVH, n, wl.D), wl.seed, 902)
        st = {"K": Kc, "V": Vc, "free": np.full((1, wl.KVH), wl.k, np.int32)}

        def step(i):
            x = decode_step_inputs(wl.with_(B=1), i)
            _, ev, st["K"], st["V"] = O.tova_decode_step(st["K"], st["V"], x["q"], x["k"], x["v"], st["free"],
                                                         wl.scale)
            st["free"] = ev.astype(np.int32)
        return step, n, "one batch row per step (oracle tova_decode_step)"
    if name.startswith("scissorhands"):
        cap = wl.S
        K = normal_bf16((1, wl.KVH, cap, wl.D), wl.seed, 903)
        sh = O.Scissorhands(1, wl.KVH, cap, history=wl.history)
        sh.prefill(wl.prefill_live)
        st = {"K": K, "queue": None, "pos": wl.m, "n": 0}

        def step(i):
            x = decode_step_inputs(wl.with_(B=1), i)
            rep = None
            if wl.policy == "queue" and sh.live.all():
                if st["pos"] == wl.m:
                    st["queue"], st["pos"] = sh.refill_queue(wl.m), 0
                rep = st["queue"][..., st["pos"]]
                st["pos"] += 1
            slot = sh.insert(replace=rep)
            st["K"], _ = O.write_slots(st["K"], st["K"], x["k"], x["k"], slot)
            if st["n"] % wl.record_every == 0:
                sh.record(O.scissorhands_probs(x["q"], st["K"], wl.scale, sh.live))
            st["n"] += 1
            if wl.policy != "queue" and not (~sh.live).any():
                sh.evict(wl.m)
        return step, cap, f"one batch row per step (oracle Scissorhands, {wl.policy} eviction)"
    if "decode_b16_s8192" in name:
        q = normal_bf16((1, wl.H, wl.D), wl.seed, 904)
        Kf = normal_bf16((1, wl.KVH, wl.S, wl.D), wl.seed, 905)
        V = normal_bf16((1, wl.KVH, wl.S, wl.D), wl.seed, 906)
        C = wl.C
        if C < wl.D:
            ch = np.sort(np.stack([np.random.Generator(np.random.PCG64([wl.seed, 907, kv])).permutation(wl.D)[:C]
                                   for kv in range(wl.KVH)])[None], axis=-1).astype(np.int32)
            Kp = np.take_along_axis(Kf, ch[:, :, None, :].astype(np.int64), axis=-1)

            def step(i):
                O.decode_attention_pruned(q, ch, Kp, V, wl.scale)
        else:
            def step(i):
                O.decode_attention(q, Kf, V, wl.scale)
        return step, wl.S, "one batch row per step (oracle decode attention)"
    inp = prefill_inputs(wl)
    if wl.reduce == "all_heads":  # all-heads scoring needs a whole instance
        def step(i):
            _oracle_unit(wl, inp, i)
        return step, wl.B * wl.S, "one whole instance (B 1) per step (oracle compress_prefill)"

    def step(i):
        _oracle_unit(wl, inp, i)
    return step, wl.B * wl.S / wl.KVH, f"one of {wl.KVH} KV-head groups per step (oracle compress_prefill)"


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = WORKLOADS[args.config]
    threads = 1  # the oracle as it stands: one process, single-threaded numpy loops
    step, tokens, sample = _reference_case(wl)
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = tokens * args.steps / dt
    line = {"impl": "reference", "metric": "kv_tokens_scored_compacted_per_s_per_layer", "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "sample": sample,
                       "instances": args.instances if args.instances is not None
                       else DEFAULT_INSTANCES.get(wl.name, 1)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{sample}, of {wl.name}, scaled by tokens"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------
# our arm: one case per workload; a step is one pass of that workload's hot path
# ----------------------------------------------------------------------------------------


def rank_seed(base_seed: int, rank: int) -> int:
    """Every rank compresses its own layer (independent units, weak scaling): its own seed."""
    return base_seed + rank


def max_over_ranks(ms: float, world: int, dist, device) -> float:
    """The job's time is the slowest rank's (no data-path collective: only this reduction)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, steps: int, world: int, ms: float) -> float:
    """Whole-job rate: units all ranks processed / the max-over-ranks time."""
    return units_per_rank_step * steps * world / (ms / 1e3)


def _source_sha(paths):
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel_key, sources):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    source of the kernel (else None: the counters no longer describe this code)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel_key)
    if not rec or rec.get("source_sha") != _source_sha(sources):
        return None
    return rec.get("dram_bytes_per_launch")


CSRC = "attention_score_kv_window_gb300/csrc/"
SCORE_SOURCES = [CSRC + f for f in ("kvc_scores.cu", "kvc_scores_tc.cu", "kvc_internal.cuh")]
DECODE_SOURCES = [CSRC + f for f in ("kvc_decode.cu", "kvc_decode.cuh")]
PREFILL_SOURCES = [CSRC + f for f in ("kvc_prefill.cu", "kvc_internal.cuh")]
STREAM_SOURCES = [CSRC + f for f in ("kvc_scores.cu", "kvc_scores_stream.cu", "kvc_internal.cuh")]


def _sha256_arrays(arrays) -> str:
    """SHA-256 of the input bytes (numpy arrays, or torch tensors copied to the host), in order:
    the oracle and the GPU path consume these same bytes."""
    import hashlib
    h = hashlib.sha256()
    for a in arrays:
        if not isinstance(a, np.ndarray):
            a = a.detach().cpu().contiguous().view(-1).view(__import__("torch").uint8).numpy()
        h.update(np.ascontiguousarray(a).view(np.uint8).reshape(-1).data)
    return h.hexdigest()


class Call:
    """One library call of a step.  ``roofline=True`` names the call whose roofline the line
    reports (else the call with the largest share of the instrumented step)."""

    def __init__(self, label, fn, nbytes, flops=0.0, bound="hbm", sources=None, kernel_key=None, roofline=False):
        self.label, self.fn, self.nbytes, self.flops, self.bound = label, fn, nbytes, flops, bound
        self.sources, self.kernel_key, self.roofline = sources, kernel_key, roofline
        self.one_pass_flops = None  # tensor-bound scoring: the flops of one pass over K
        self.times = []


class PrefillCase:
    """Prefill compression of one layer (TOVA or SnapKV; ThinK adds channel score + prune)."""

    def __init__(self, wl, dev, rank, instances):
        import torch
        import attention_score_kv_window_gb300 as kvc
        self.kvc, self.torch = kvc, torch
        if instances > 1:
            wl = wl.with_(B=instances)
        self.wl = wl
        inp = prefill_inputs(wl, seed=rank_seed(wl.seed, rank))
        self.host = inp
        self.inputs_sha256 = _sha256_arrays([inp["q"], inp["K"], inp["V"]])

        def to_dev(u16):
            return torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16).to(dev)

        q0, K0, V0 = to_dev(inp["q"]), to_dev(inp["K"]), to_dev(inp["V"])
        self.in_bytes = (q0.numel() + K0.numel() + V0.numel()) * 2
        self.R = R = max(2, math.ceil(3 * L2_BYTES / self.in_bytes))
        self.reps = [(q0, K0, V0)] + [(q0.clone(), K0.clone(), V0.clone()) for _ in range(R - 1)]
        B, KVH, S, D = K0.shape
        self.B, self.KVH, self.S, self.D = B, KVH, S, D
        k = self.k = min(wl.k, S)
        f32, i32, bf = torch.float32, torch.int32, torch.bfloat16
        self.outs = [(torch.empty((B, KVH, S), dtype=f32, device=dev), torch.empty((B, KVH, k), dtype=i32, device=dev),
                      torch.empty((B, KVH, k, D), dtype=bf, device=dev), torch.empty((B, KVH, k, D), dtype=bf, device=dev))
                     for _ in range(R)]
        lib = kvc.load_library()
        ws_bytes = int(lib.kvc_workspace_size(2, kvc.kv_desc(K0, wl.H), wl.w, k))
        # shapes the library runs as one fused kernel need no workspace
        self.fused = ws_bytes == 0 and not wl.C
        self.ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.tokens_per_step = B * S
        G = wl.H // wl.KVH
        # the step's algorithmic bytes: K read once, the kept V rows read, the kept K and V rows
        # written, the window queries and the indices
        self.step_bytes = B * KVH * D * 2 * (S + 3 * k) + B * wl.H * wl.w * D * 2 + B * KVH * k * 4
        sc_bytes = B * KVH * S * D * 2 + B * wl.H * wl.w * D * 2 + B * KVH * S * 4
        sc_flops = 2 * 2.0 * B * wl.H * wl.w * S * D  # both passes of q_win K^T (the two-pass softmax)
        big_w = wl.w * G > 32
        if self.fused:
            self.calls = [Call("compress_prefill", self._compress, self.step_bytes, 2.0 * B * wl.H * wl.w * S * D,
                               "hbm", PREFILL_SOURCES, f"compress_prefill/{wl.name}/B{B}", roofline=True)]
        else:
            self.calls = [
                Call("window_scores", self._scores, sc_bytes, sc_flops, "tensor" if big_w else "hbm", SCORE_SOURCES,
                     f"window_scores/{wl.name}/B{B}"),
                Call("topk_compact", self._topk_compact, B * KVH * S * 4 + 4 * B * KVH * k * D * 2 + B * KVH * k * 4),
            ]
            self.calls[0].one_pass_flops = sc_flops / 2
        if wl.C:
            # ThinK: the compaction also sums the kept keys' squares per channel (the key half of
            # the channel score comes from the same read of the kept K rows); then the prune
            C = wl.C
            self.cs = torch.empty((B, KVH, D), dtype=f32, device=dev)
            self.ch = torch.empty((B, KVH, C), dtype=i32, device=dev)
            self.Kp = torch.empty((B, KVH, k, C), dtype=bf, device=dev)
            self.cws = torch.empty(int(lib.kvc_workspace_size(10, kvc.kv_desc(K0, wl.H), 0, k)), dtype=torch.uint8,
                                   device=dev)
            assert not self.fused
            tc = self.calls[1]
            self.calls[1] = Call("topk_compact_channels", self._topk_compact_ch,
                                 tc.nbytes + B * wl.H * wl.w * D * 2 + B * KVH * D * 4)
            self.calls += [Call("channel_prune", self._cprune, B * KVH * k * D * 2 + B * KVH * k * C * 2)]
        if wl.extra.get("values"):  # value channels too: score over the compressed cache, then prune
            C = wl.C
            self.vcs = torch.empty((B, KVH, D), dtype=f32, device=dev)
            self.vch = torch.empty((B, KVH, C), dtype=i32, device=dev)
            self.Vp = torch.empty((B, KVH, k, C), dtype=bf, device=dev)
            self.vws = torch.empty(int(lib.kvc_workspace_size(8, kvc.kv_desc(self.outs[0][2], wl.H), wl.w, 0)),
                                   dtype=torch.uint8, device=dev)
            vflops = 2 * 2.0 * B * wl.H * wl.w * k * D
            self.calls += [Call("value_channel_score", self._vscore, 2 * B * KVH * k * D * 2 + B * wl.H * wl.w * D * 2,
                                vflops, "tensor"),
                           Call("value_channel_prune", self._vprune, B * KVH * k * D * 2 + B * KVH * k * C * 2)]

    def _compress(self, i):
        q, K, V = self.reps[i % self.R]
        _, idx, Ko, Vo = self.outs[i % self.R]
        self.kvc.kvc_compress_prefill(q, K, V, self.wl.scale, self.k, protect_tail=self.wl.protect_tail,
                                      reduce=self.wl.reduce, out=(None, idx, Ko, Vo))

    def _scores(self, i):
        q, K, V = self.reps[i % self.R]
        self.kvc.kvc_window_scores(q, K, self.wl.scale, causal=True, reduce=self.wl.reduce,
                                   scores=self.outs[i % self.R][0], ws=self.ws)

    def _topk_compact(self, i):
        q, K, V = self.reps[i % self.R]
        sc, idx, Ko, Vo = self.outs[i % self.R]
        self.kvc.kvc_topk_compact(sc, K, V, self.k, protect_tail=self.wl.protect_tail, H=self.wl.H, idx=idx,
                                  K_out=Ko, V_out=Vo)

    def _topk_compact_ch(self, i):
        q, K, V = self.reps[i % self.R]
        sc, idx, Ko, Vo = self.outs[i % self.R]
        self.kvc.kvc_topk_compact_channels(sc, K, V, self.k, q, protect_tail=self.wl.protect_tail, idx=idx, K_out=Ko,
                                           V_out=Vo, cs=self.cs, ws=self.cws)

    def _cprune(self, i):
        self.kvc.kvc_channel_prune(self.cs, self.outs[i % self.R][2], self.wl.C, ch_idx=self.ch, K_out=self.Kp,
                                   H=self.wl.H)

    def _vscore(self, i):
        q, _, _ = self.reps[i % self.R]
        _, _, Ko, Vo = self.outs[i % self.R]
        self.kvc.kvc_value_channel_score(q, Ko, Vo, self.wl.scale, cs=self.vcs, ws=self.vws)

    def _vprune(self, i):
        self.kvc.kvc_channel_prune(self.vcs, self.outs[i % self.R][3], self.wl.C, ch_idx=self.vch, K_out=self.Vp,
                                   H=self.wl.H)

    def config(self):
        wl = self.wl
        c = {"workload": wl.name, "B": self.B, "H": wl.H, "KVH": self.KVH, "D": self.D, "S": self.S, "w": wl.w,
             "k": self.k, "C": wl.C or None, "value_channels_pruned": bool(wl.extra.get("values")),
             "l2": f"inputs rotate over {self.R} replicas ({self.R * self.in_bytes / 2**20:.0f} MiB > L2)",
             "inputs_sha256": self.inputs_sha256, "path": "one fused kernel" if self.fused else "library calls"}
        if self.B > 1 and WORKLOADS[wl.name].B == 1:
            c["instances"] = self.B
            c["instances_note"] = (f"the {wl.name} layer (batch 1) stacked as {self.B} independent instances "
                                   f"in one call: a single instance is too small to load the GPU (its latency "
                                   f"is reported as single_instance)")
        return c

    def single_instance(self, steps):
        """Latency of one instance of the workload (batch 1) through the same call: ``steps``
        calls captured in a CUDA graph and replayed, CUDA events around the replay."""
        torch, kvc, wl = self.torch, self.kvc, self.wl
        q, K, V = (t[:1] for t in self.reps[0])
        _, idx, Ko, Vo = (None if t is None else t[:1] for t in self.outs[0])
        sc = self.outs[0][0][:1]
        ws = self.ws

        def call():
            kvc.kvc_compress_prefill(q, K, V, wl.scale, self.k, protect_tail=wl.protect_tail, reduce=wl.reduce,
                                     out=(None if self.fused else sc, idx, Ko, Vo), ws=None if self.fused else ws)
        for _ in range(3):
            call()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for _ in range(steps):
                    call()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        nbytes = self.step_bytes / self.B
        return {"ms": ms, "tokens_per_s": self.S / (ms / 1e3), "alg_bytes": nbytes,
                "gbs": nbytes / (ms / 1e3) / 1e9}

    def e2e(self, steps, stream, world, dist, dev):
        """Same step through kvc_compress_prefill with pinned host inputs and outputs.  Steps are
        pipelined over two device buffer sets: step i+1's host->device copies (the four
        quarters of K each on its own copy stream, q with the last) overlap step i's compute and
        its device->host read-back (another stream).  V stays in page-locked host memory: the
        compaction kernel reads the kept rows over the host link (kvc_host_device_pointer), so
        only those cross it.  Every step moves its inputs and results."""
        torch, kvc, wl = self.torch, self.kvc, self.wl
        inp = self.host
        hq = torch.from_numpy(inp["q"].view(np.int16)).view(torch.bfloat16).pin_memory()
        hK = torch.from_numpy(inp["K"].view(np.int16)).view(torch.bfloat16).pin_memory()
        hV = torch.from_numpy(inp["V"].view(np.int16)).view(torch.bfloat16).pin_memory()
        B, KVH, k, D = self.B, self.KVH, self.k, self.D
        h_out = [(torch.empty((B, KVH, k), dtype=torch.int32).pin_memory(),
                  torch.empty((B, KVH, k, D), dtype=torch.bfloat16).pin_memory(),
                  torch.empty((B, KVH, k, D), dtype=torch.bfloat16).pin_memory()) for _ in range(2)]
        ws2 = torch.empty_like(self.ws)
        bufs = [(self.reps[0], self.outs[0], self.ws), (self.reps[1], self.outs[1], ws2)]
        s_up = [torch.cuda.Stream() for _ in range(4)]
        s_out = torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_ready = [[ev() for _ in range(4)] for _ in range(2)]   # inputs of a buffer set uploaded
        fK = hK.view(-1)
        qn = fK.numel() // 4

        def pieces(dq, dK, dV):  # contiguous quarters of the flattened K
            gK = dK.view(-1)
            return (((gK[:qn], fK[:qn]),), ((gK[qn:2 * qn], fK[qn:2 * qn]),),
                    ((gK[2 * qn:3 * qn], fK[2 * qn:3 * qn]),), ((gK[3 * qn:], fK[3 * qn:]), (dq, hq)))
        comp_done = [ev() for _ in range(2)]          # compute on a buffer set finished
        out_done = [ev() for _ in range(2)]           # results of a buffer set read back
        used = [False, False]

        def e2e_step(i):
            x = i % 2
            (dq, dK, dV), (sc, idx, Ko, Vo), ws = bufs[x]
            hi, hKo, hVo = h_out[x]
            # upload into set x once its previous compute has consumed it
            for st_, ev_, pairs in zip(s_up, in_ready[x], pieces(dq, dK, dV)):
                if used[x]:
                    st_.wait_event(comp_done[x])
                with torch.cuda.stream(st_):
                    for d_, h_ in pairs:
                        d_.copy_(h_, non_blocking=True)
                ev_.record(st_)
            for ev_ in in_ready[x]:
                stream.wait_event(ev_)
            if used[x]:
                stream.wait_event(out_done[x])  # its previous results were read back
            kvc.kvc_compress_prefill(dq, dK, hV, wl.scale, k, protect_tail=wl.protect_tail, reduce=wl.reduce,
                                     out=(None if self.fused else sc, idx, Ko, Vo), ws=None if self.fused else ws)
            comp_done[x].record(stream)
            s_out.wait_event(comp_done[x])
            with torch.cuda.stream(s_out):
                hi.copy_(idx, non_blocking=True)
                hKo.copy_(Ko, non_blocking=True)
                hVo.copy_(Vo, non_blocking=True)
            out_done[x].record(s_out)
            used[x] = True

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st_ in s_up + [s_out]:
            st_.wait_event(e0)
        for i in range(steps):
            e2e_step(i)
        for x in range(2):
            stream.wait_event(out_done[x])
        e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), world, dist, dev)
        return {"value": self.tokens_per_step * steps * world / (ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int((hq.numel() + hK.numel()) * 2 + B * KVH * k * D * 2),
                "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in h_out[0])),
                "pipeline": "two buffer sets; K uploads (four streams), compute and read-back on separate "
                            "streams; V read in place from page-locked host memory, kept rows only"}


class TovaDecodeCase:
    """TOVA generation: a cache of budget+1 slots; each step writes the new token into the free
    slot, scores every slot with the new query (mean over all heads), evicts the minimum."""

    def __init__(self, wl, dev, rank, instances):
        import torch
        import attention_score_kv_window_gb300 as kvc
        self.kvc, self.torch, self.wl = kvc, torch, wl
        B, H, KVH, D, S0, budget = wl.B, wl.H, wl.KVH, wl.D, wl.S, wl.k
        n = budget + 1
        self.cache_bytes = B * KVH * n * D * 2
        self.R = R = max(2, math.ceil(3 * L2_BYTES / self.cache_bytes))
        g = torch.Generator(device=dev)
        g.manual_seed(rank_seed(wl.seed, rank))
        bf = torch.bfloat16
        self.caches = []
        for r in range(R):
            Kf = torch.randn((B, KVH, S0 + 1, D), generator=g, device=dev).to(bf)
            Vf = torch.randn((B, KVH, S0 + 1, D), generator=g, device=dev).to(bf)
            q0 = torch.randn((B, H, 1, D), generator=g, device=dev).to(bf)
            sc = kvc.kvc_window_scores(q0, Kf, wl.scale, causal=False, reduce="all_heads")
            idx = kvc.kvc_topk_select(sc, budget)
            Kk, Vk = kvc.kvc_compact_kv(Kf, Vf, idx, H=H)
            Kc = torch.zeros((B, KVH, n, D), dtype=bf, device=dev)
            Vc = torch.zeros_like(Kc)
            Kc[:, :, :budget] = Kk
            Vc[:, :, :budget] = Vk
            del Kk, Vk
            free = torch.full((B, KVH), budget, dtype=torch.int32, device=dev)
            self.caches.append((Kc, Vc, free, torch.empty((B, KVH, n), dtype=torch.float32, device=dev)))
            del Kf, Vf
        self.nq = 64
        self.q = torch.randn((self.nq, B, H, D), generator=g, device=dev).to(bf)
        self.kn = torch.randn((self.nq, B, KVH, D), generator=g, device=dev).to(bf)
        self.vn = torch.randn((self.nq, B, KVH, D), generator=g, device=dev).to(bf)
        Kc0 = self.caches[0][0]
        self.ws = torch.empty(int(kvc.load_library().kvc_workspace_size(3, kvc.kv_desc(Kc0, H), 1, 0)),
                              dtype=torch.uint8, device=dev)
        self.B, self.KVH, self.S, self.D = B, KVH, n, D
        self.tokens_per_step = B * n
        self.inputs_sha256 = _sha256_arrays([self.caches[0][0], self.caches[0][1], self.q, self.kn, self.vn])
        nbytes = B * KVH * n * D * 2 + 2 * B * KVH * D * 2 + 2 * B * KVH * n * 4 + B * H * D * 2
        self.calls = [Call("tova_decode_step", self._step, nbytes, 2.0 * B * H * n * D, "hbm", STREAM_SOURCES,
                           f"tova_decode/{wl.name}")]

    def _step(self, i):
        Kc, Vc, free, sc = self.caches[i % self.R]
        j = i % self.nq
        self.kvc.kvc_tova_decode_step(self.q[j], self.kn[j], self.vn[j], Kc, Vc, self.wl.scale, free, scores=sc,
                                      ws=self.ws)

    def config(self):
        wl = self.wl
        return {"workload": wl.name, "B": wl.B, "H": wl.H, "KVH": wl.KVH, "D": wl.D, "slots": self.S,
                "l2": f"steps rotate over {self.R} caches ({self.R * self.cache_bytes / 2**20:.0f} MiB > L2)",
                "inputs_sha256": self.inputs_sha256, "inputs": "drawn on the device (torch.Generator, seeded)"}

    def e2e(self, *a):
        return None


class ScissorhandsCase:
    """Scissorhands decode: insert, score the new query over the live slots, record the low-
    attention flags into the 400-step history.  Policies: bulk eviction of m slots per head
    when the cache is full; or an eviction queue refilled every m steps once the cache is full,
    each step's token replacing the next queued one.  With record_every = M > 1 only every
    M-th step scores and records; the other steps only insert."""

    def __init__(self, wl, dev, rank, instances):
        import torch
        import attention_score_kv_window_gb300 as kvc
        self.kvc, self.torch, self.wl = kvc, torch, wl
        B, H, KVH, D, cap = wl.B, wl.H, wl.KVH, wl.D, wl.S
        self.cache_bytes = B * KVH * cap * D * 2
        self.R = R = max(2, math.ceil(3 * L2_BYTES / self.cache_bytes))
        g = torch.Generator(device=dev)
        g.manual_seed(rank_seed(wl.seed, rank))
        bf = torch.bfloat16
        self.reps = []
        for r in range(R):
            K = torch.randn((B, KVH, cap, D), generator=g, device=dev).to(bf)
            V = torch.randn((B, KVH, cap, D), generator=g, device=dev).to(bf)
            st = kvc.ScissorhandsState(B, KVH, cap, history=wl.history, device=dev)
            kvc.kvc_scissorhands_init(st, wl.prefill_live)
            self.reps.append({"K": K, "V": V, "st": st,
                              "probs": torch.empty((B, KVH, cap), dtype=torch.float32, device=dev),
                              "ev": torch.empty((B, KVH, wl.m), dtype=torch.int32, device=dev),
                              "steps": 0, "pos": wl.m})
        self.nq = 64
        self.q = torch.randn((self.nq, B, H, D), generator=g, device=dev).to(bf)
        self.kn = torch.randn((self.nq, B, KVH, D), generator=g, device=dev).to(bf)
        self.vn = torch.randn((self.nq, B, KVH, D), generator=g, device=dev).to(bf)
        self.ws = torch.empty(int(kvc.load_library().kvc_workspace_size(4, kvc.kv_desc(self.reps[0]["K"], H), 1, 0)),
                              dtype=torch.uint8, device=dev)
        self.B, self.H, self.KVH, self.S, self.D = B, H, KVH, cap, D
        self.tokens_per_step = B * cap
        self.inputs_sha256 = _sha256_arrays([self.reps[0]["K"], self.reps[0]["V"], self.q, self.kn, self.vn])
        rows, slots = B * KVH, B * KVH * cap
        state = 2 * slots * 4 + slots * 4 + 2 * slots * 2 + 2 * slots // 8  # probs, insert steps, counts, flags
        new_rows = 2 * rows * D * 2
        upd = slots * D * 2 + new_rows + state + B * H * D * 2
        rank_bytes = slots * (2 + 4 + 0.125) + rows * wl.m * 4
        # the roofline is the update's (score + record over the whole cache); under sparse
        # recording the insert-only steps are tiny, launch-bound kernels
        self.calls = [Call("scissorhands_update", self._update, upd, 2.0 * B * H * cap * D, "hbm", STREAM_SOURCES,
                           f"scissorhands/{wl.name}", roofline=True)]
        if wl.record_every > 1:
            self.calls.append(Call("scissorhands_insert", self._insert, 2 * new_rows + slots // 8 + rows * 12))
        if wl.policy == "queue":
            self.calls.insert(0, Call("scissorhands_refill_queue", self._refill, rank_bytes))
        else:
            self.calls.append(Call("scissorhands_evict", self._evict, rank_bytes))

    def _queue_args(self, rep):
        if self.wl.policy != "queue" or rep["st"].n_free > 0:
            return {}
        return {"queue": rep["ev"], "pos": rep["pos"]}

    def _refill(self, i):
        rep = self.reps[i % self.R]
        if rep["st"].n_free > 0 or rep["pos"] < self.wl.m:
            return False
        self.kvc.kvc_scissorhands_refill_queue(rep["st"], self.wl.m, queue=rep["ev"])
        rep["pos"] = 0

    def _advance(self, rep, qa):
        rep["steps"] += 1
        if qa:
            rep["pos"] += 1

    def _update(self, i):
        rep = self.reps[i % self.R]
        rep["record"] = rep["steps"] % self.wl.record_every == 0  # this step scores and records
        if not rep["record"]:
            return False
        j = i % self.nq
        qa = self._queue_args(rep)
        self.kvc.kvc_scissorhands_update(rep["st"], self.q[j], self.kn[j], self.vn[j], rep["K"], rep["V"],
                                         self.wl.scale, probs=rep["probs"], ws=self.ws, **qa)
        self._advance(rep, qa)

    def _insert(self, i):
        rep = self.reps[i % self.R]
        if rep["record"]:
            return False
        j = i % self.nq
        qa = self._queue_args(rep)
        self.kvc.kvc_scissorhands_insert(rep["st"], self.kn[j], self.vn[j], rep["K"], rep["V"], self.H, **qa)
        self._advance(rep, qa)

    def _evict(self, i):
        rep = self.reps[i % self.R]
        if rep["st"].n_free > 0:
            return False
        self.kvc.kvc_scissorhands_evict(rep["st"], self.wl.m, evicted=rep["ev"])

    def config(self):
        wl = self.wl
        return {"workload": wl.name, "B": wl.B, "H": wl.H, "KVH": wl.KVH, "D": wl.D, "cap": wl.S,
                "history": wl.history, "m": wl.m, "policy": wl.policy, "record_every": wl.record_every,
                "l2": f"steps rotate over {self.R} caches ({self.R * self.cache_bytes / 2**20:.0f} MiB > L2)",
                "inputs_sha256": self.inputs_sha256, "inputs": "drawn on the device (torch.Generator, seeded)"}

    def e2e(self, *a):
        return None


class DecodeCase:
    """Decoding over a compressed cache: one new query per head attends the kept tokens; the
    keys keep C of the D channels ("Add ThinK_Press" option 3c: the query is pruned to them)
    or all of them (plain attention)."""

    def __init__(self, wl, dev, rank, instances):
        import torch
        import attention_score_kv_window_gb300 as kvc
        self.kvc, self.torch, self.wl = kvc, torch, wl
        B, H, KVH, D, S, C = wl.B, wl.H, wl.KVH, wl.D, wl.S, wl.C
        self.cache_bytes = B * KVH * S * (C + D) * 2
        self.R = R = max(2, math.ceil(3 * L2_BYTES / self.cache_bytes))
        g = torch.Generator(device=dev)
        g.manual_seed(rank_seed(wl.seed, rank))
        bf = torch.bfloat16
        self.reps = []
        for r in range(R):
            K = torch.randn((B, KVH, S, C), generator=g, device=dev).to(bf)
            V = torch.randn((B, KVH, S, D), generator=g, device=dev).to(bf)
            ch = None
            if C < D:  # a kept-channel list per (b, kvh): C distinct channels, ascending
                ch = torch.sort(torch.rand((B, KVH, D), generator=g, device=dev).argsort(-1)[..., :C], -1)[0]
                ch = ch.to(torch.int32).contiguous()
            self.reps.append((K, V, ch))
        self.nq = 64
        self.q = torch.randn((self.nq, B, H, D), generator=g, device=dev).to(bf)
        self.out = torch.empty((B, H, D), dtype=torch.float32, device=dev)
        vd = kvc.kv_desc(self.reps[0][1], H)
        self.ws = torch.empty(int(kvc.load_library().kvc_workspace_size(7, vd, 0, 0)), dtype=torch.uint8, device=dev)
        self.tokens_per_step = B * S
        r0 = self.reps[0]
        self.inputs_sha256 = _sha256_arrays([t for t in r0 if t is not None] + [self.q])
        nbytes = self.cache_bytes + B * H * D * 2 + B * H * D * 4 + (B * KVH * C * 4 if C < D else 0)
        self.calls = [Call("decode_attention", self._step, nbytes, 2.0 * B * H * S * (C + D), "hbm", DECODE_SOURCES,
                           f"decode_attention/{wl.name}")]

    def _step(self, i):
        K, V, ch = self.reps[i % self.R]
        self.kvc.kvc_decode_attention(self.q[i % self.nq], K, V, self.wl.scale, ch=ch, out=self.out, ws=self.ws)

    def config(self):
        wl = self.wl
        return {"workload": wl.name, "B": wl.B, "H": wl.H, "KVH": wl.KVH, "D": wl.D, "kept_tokens": wl.S,
                "key_channels": wl.C, "l2": f"steps rotate over {self.R} caches "
                                            f"({self.R * self.cache_bytes / 2**20:.0f} MiB > L2)",
                "inputs_sha256": self.inputs_sha256, "inputs": "drawn on the device (torch.Generator, seeded)"}

    def e2e(self, *a):
        return None


def make_case(wl, dev, rank, instances):
    if wl.name.startswith("tova_decode"):
        return TovaDecodeCase(wl, dev, rank, instances)
    if wl.name.startswith("scissorhands"):
        return ScissorhandsCase(wl, dev, rank, instances)
    if "decode_b16_s8192" in wl.name:
        return DecodeCase(wl, dev, rank, instances)
    return PrefillCase(wl, dev, rank, instances)


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
    instances = args.instances if args.instances is not None else DEFAULT_INSTANCES.get(wl.name, 1)
    case = make_case(wl, dev, rank, instances)
    stream = torch.cuda.current_stream()
    calls = case.calls

    # a call's fn returns False when it had nothing to do this step (e.g. eviction while
    # slots are free); its time is averaged over the steps where it ran
    ran = [[True] * len(calls) for _ in range(args.steps)]

    def step(i, ev=None, r=None):
        for c, call in enumerate(calls):
            if ev is not None:
                ev[c].record(stream)
            did = call.fn(i) is not False
            if r is not None:
                r[c] = did
        if ev is not None:
            ev[len(calls)].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert kvc.kvc_get_device_status() == kvc.KVC_OK

    sampler = ClockSampler(local) if not args.no_clocks else None
    base = args.warmup
    if sampler:
        sampler.start()
        # keep the GPU busy for a moment so the sampler sees the loaded clock
        t_end = time.time() + 0.5
        while time.time() < t_end:
            step(base)
            base += 1
        torch.cuda.synchronize()

    # The K timed steps are captured into one CUDA graph and replayed once: the GPU then runs
    # them back to back, without host-side gaps from the Python binding, and consecutive
    # kernels may overlap launch and tail (programmatic dependent launch).  The step time
    # comes from that replay.  A second graph of the same K steps with a timing event before
    # every call gives the per-kernel durations (events between kernels serialise them, so
    # the per-kernel sum can exceed the step time).  Falls back to direct launches where
    # events cannot be captured.
    use_graph = not args.no_graph
    try:
        mk = (lambda: torch.cuda.Event(enable_timing=True, external=True)) if use_graph else \
            (lambda: torch.cuda.Event(enable_timing=True))
        mk()
    except TypeError:
        use_graph = False
        mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    evs = [[mk() for _ in range(len(calls) + 1)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph = graph_timed = None
    launches0 = kvc.kvc_launch_count()
    if use_graph:
        graph, graph_timed = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for i in range(args.steps):
                    for call in calls:
                        call.fn(base + i)
            launches = kvc.kvc_launch_count() - launches0
            with torch.cuda.graph(graph_timed, stream=cap):
                cs = torch.cuda.current_stream()
                for i in range(args.steps):
                    for c, call in enumerate(calls):
                        evs[i][c].record(cs)
                        ran[i][c] = call.fn(base + i) is not False
                    evs[i][len(calls)].record(cs)
        stream.wait_stream(cap)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    host0 = time.perf_counter()
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        launches0 = kvc.kvc_launch_count()
        for i in range(args.steps):
            step(base + i)
        launches = kvc.kvc_launch_count() - launches0
    stop.record(stream)
    host_ms = (time.perf_counter() - host0) * 1e3
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(start.elapsed_time(stop), world, dist, dev)
    # per-kernel durations: the instrumented replay of the same steps
    if graph_timed is not None:
        graph_timed.replay()
    else:
        for i in range(args.steps):
            step(base + i, evs[i], ran[i])
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    assert kvc.kvc_get_device_status() == kvc.KVC_OK

    kernels = {}
    for c, call in enumerate(calls):
        ts = [e[c].elapsed_time(e[c + 1]) for e, r in zip(evs, ran) if r[c]]
        if not ts:
            continue
        t = float(np.mean(ts))
        kernels[call.label] = {"ms": t, "calls": len(ts), "alg_bytes": call.nbytes,
                               "gbs": call.nbytes / (t / 1e3) / 1e9, "share": t * len(ts)}
        if call.flops:
            kernels[call.label]["tflops"] = call.flops / (t / 1e3) / 1e12
    total = sum(k["share"] for k in kernels.values())
    for k in kernels.values():
        k["share"] = k["share"] / total
    # the dominant call takes the largest share of the step (unless the case names one); its
    # roofline is per launch
    ran_calls = [c for c in calls if c.label in kernels]
    named = [c for c in ran_calls if c.roofline]
    dom = named[0] if named else max(ran_calls, key=lambda c: kernels[c.label]["share"])
    t_dom = kernels[dom.label]["ms"]
    if dom.bound == "tensor":
        achieved = dom.flops / (t_dom / 1e3) / 1e12
        roof = {"kernel": f"kvc_{dom.label}", "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "peak_source": f"{peaks['source']} bf16 burst (of measured)" if peaks["source"] == "measured"
                else "fallback bf16"}
    else:
        achieved = dom.nbytes / (t_dom / 1e3) / 1e9
        roof = {"kernel": f"kvc_{dom.label}", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "peak_source": f"{peaks['source']} HBM copy"}
    roof["traffic"] = _traffic(dom.kernel_key, dom.sources) if dom.kernel_key else None
    roof["algorithmic_bytes_per_launch"] = dom.nbytes
    if dom.bound == "tensor":
        # both passes of the two-pass softmax over K (the probabilities never reach memory);
        # the frac of the one-pass minimum is given beside it
        roof["executed_flops_per_launch"] = dom.flops
        if dom.one_pass_flops:
            roof["one_pass_flops_per_launch"] = dom.one_pass_flops
            roof["one_pass_frac"] = dom.one_pass_flops / (t_dom / 1e3) / 1e12 / peaks["bf16_tflops"]
    else:
        roof["flops_per_launch"] = dom.flops

    # the whole step against the HBM roofline: its algorithmic bytes over the replayed step time
    step_bytes = getattr(case, "step_bytes", None)
    if step_bytes is None:
        step_bytes = sum(c.nbytes * kernels[c.label]["calls"] / args.steps for c in ran_calls)
    step_gbs = step_bytes / (ms / args.steps / 1e3) / 1e9
    step_roof = {"bound": "hbm", "bytes_per_step": step_bytes, "ms_per_step": ms / args.steps,
                 "achieved": step_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": step_gbs / peaks["hbm_gbs"],
                 "basis": "algorithmic bytes of the whole step / the step time of the CUDA-graph replay"}
    single = case.single_instance(50) if isinstance(case, PrefillCase) and case.B > 1 and \
        WORKLOADS[case.wl.name].B == 1 else None
    if single is not None:
        single["frac"] = single["gbs"] / peaks["hbm_gbs"]

    value = job_throughput(case.tokens_per_step, args.steps, world, ms)
    e2e = case.e2e(max(3, min(args.steps, 20)), stream, world, dist, dev) if not args.no_e2e else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and isinstance(case, PrefillCase):
        cpu = cpu_baseline(args.config, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": "kv_tokens_scored_compacted_per_s_per_layer", "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": case.config(), "roofline": roof, "step_roofline": step_roof,
            "single_instance": single, "kernels": kernels,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches), "clocks": clocks,
            "timing": {"cuda_graph": graph is not None, "host_enqueue_ms": host_ms,
                       "kernels": "separate replay with an event before every call"},
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
    ap.add_argument("--config", default=TOVA_PREFILL.name, choices=sorted(WORKLOADS))
    ap.add_argument("--instances", type=int, default=None,
                    help="independent prefill instances batched into one step (default: 8192 for TOVA "
                         "prefill, 1 otherwise)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the timed steps directly (no CUDA graph)")
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
