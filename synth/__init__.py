"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module only draws random numbers and stores them as bf16 bit patterns.  It holds none
of the method's arithmetic (no softmax, no scores, no selection): both the oracle and the
GPU path receive the same bytes from here and compute everything else on their own.

Random source: numpy's PCG64 bit generator, seeded with a list ``[seed, tag...]`` so that
every tensor (and every decode step) has its own independent substream.  bf16 values are
produced by round-to-nearest-even from float32 draws.

The workloads follow the shapes of the pages' examples:

* TOVA prefill (kvpress PR "Add TOVA press", the last-query head-mean score),
* SnapKV prefill with a 64-query observation window (cold-compress PR #11, SnapKV paragraph),
* TOVA decode eviction,
* Scissorhands decode with a 400-step history (cold-compress PR #11), with bulk eviction,
  with the PR's eviction queue, or with flags recorded only every 8th step,
* ThinK key-channel pruning after SnapKV (kvpress PR "Add ThinK_Press"), and decoding over
  the pruned cache it leaves (the thread's options 3b/3c).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
import numpy as np

# ----------------------------------------------------------------------------------------
# bf16 storage helpers (data format only)
# ----------------------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _rng(*tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(t) for t in tag]))


def normal_bf16(shape, *tag: int) -> np.ndarray:
    """bf16 bits of N(0,1) draws from the substream ``tag``."""
    n = int(np.prod(shape)) if len(shape) else 1
    z = _rng(*tag).standard_normal(n, dtype=np.float32).reshape(shape)
    return f32_to_bf16_bits(z)


# stream tags (second element of the PCG64 seed list)
TAG_Q, TAG_K, TAG_V, TAG_HH, TAG_CHS, TAG_STEP, TAG_SCORES, TAG_LIVE, TAG_PROBS = range(1, 10)


# ----------------------------------------------------------------------------------------
# workload descriptions
# ----------------------------------------------------------------------------------------


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    KVH: int
    D: int
    S: int                 # cached tokens (prefill length, or decode capacity)
    w: int                 # observation window (1 for TOVA / decode)
    k: int                 # kept tokens per KV head (budget)
    reduce: str            # "all_heads" (TOVA) or "gqa" (SnapKV, Scissorhands, ThinK)
    protect_tail: int = 0  # SnapKV keeps the window itself
    causal: bool = True
    heavy_hitters: float = 0.0    # fraction of prefix keys shifted toward the window query mean
    channel_scales: bool = False  # per-(kvh, channel) LogNormal(0,1) key scales
    steps: int = 0                # decode steps
    history: int = 0              # Scissorhands history window
    m: int = 0                    # Scissorhands drop amount / eviction period
    prefill_live: int = 0         # Scissorhands: live tokens at the start of decode
    policy: str = "bulk"          # Scissorhands: "bulk" eviction every m steps, or an eviction "queue"
    record_every: int = 1         # Scissorhands: record the flags every M-th step (1: every step)
    C: int = 0                    # ThinK kept key channels
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.H // self.KVH

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


TOVA_PREFILL = Workload("tova_prefill_s512", B=1, H=8, KVH=2, D=64, S=512, w=1, k=256,
                        reduce="all_heads")
SNAPKV_32K = Workload("snapkv_prefill_s32768", B=1, H=32, KVH=8, D=128, S=32768, w=64, k=4096,
                      reduce="gqa", protect_tail=64, heavy_hitters=0.01)
TOVA_DECODE = Workload("tova_decode_b16_c8192_budget2048", B=16, H=32, KVH=8, D=128, S=8192, w=1,
                       k=2048, reduce="all_heads", causal=False, steps=256)
SCISSORHANDS = Workload("scissorhands_decode_b8_cap4096", B=8, H=32, KVH=8, D=128, S=4096, w=1,
                        k=4096, reduce="gqa", causal=False, steps=1024, history=400, m=64,
                        prefill_live=4032)
SCISSORHANDS_QUEUE = SCISSORHANDS.with_(name="scissorhands_queue_decode_b8_cap4096", policy="queue")
SCISSORHANDS_SPARSE = SCISSORHANDS.with_(name="scissorhands_sparse8_decode_b8_cap4096", record_every=8)
THINK_128K = Workload("think_snapkv_prefill_s131072", B=1, H=32, KVH=8, D=128, S=131072, w=64,
                      k=8192, reduce="gqa", protect_tail=64, channel_scales=True, C=64)

# keys and values pruned to 64 channels (value scores over the compressed cache)
THINK_KV_128K = THINK_128K.with_(name="think_kv_snapkv_prefill_s131072", extra={"values": True})
# decoding over the cache ThinK + SnapKV leave (8192 kept tokens, 64 of 128 key channels),
# for a decode batch of 16 such caches; the _full variant attends unpruned keys
THINK_DECODE = Workload("think_decode_b16_s8192_c64", B=16, H=32, KVH=8, D=128, S=8192, w=1, k=8192,
                        reduce="gqa", causal=False, C=64)
FULL_DECODE = THINK_DECODE.with_(name="decode_b16_s8192_full", C=128)
WORKLOADS = {wl.name: wl for wl in (TOVA_PREFILL, SNAPKV_32K, TOVA_DECODE, SCISSORHANDS, SCISSORHANDS_QUEUE,
                                    SCISSORHANDS_SPARSE, THINK_128K, THINK_KV_128K, THINK_DECODE, FULL_DECODE)}


# ----------------------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------------------


def prefill_inputs(wl: Workload, seed: int | None = None) -> dict:
    """q_win [B,H,w,D], K and V [B,KVH,S,D] as bf16 bit patterns (uint16).

    * heavy hitters: a seeded ``heavy_hitters`` fraction of the prefix positions of every
      (b, kvh) get ``k_j <- bf16(k_j + 3 * qbar)``, where ``qbar`` is the float32 mean of that
      KV head's window queries over the window rows and the group's query heads;
    * channel scales: ``K[b,kvh,j,d] = bf16(z * s[kvh,d])`` with ``s ~ LogNormal(0, 1)``
      drawn once per (kvh, d) and ``z ~ N(0, 1)``.
    """
    seed = wl.seed if seed is None else seed
    B, H, KVH, D, S, w = wl.B, wl.H, wl.KVH, wl.D, wl.S, wl.w
    q = normal_bf16((B, H, w, D), seed, TAG_Q)
    if wl.channel_scales:
        z = _rng(seed, TAG_K).standard_normal(B * KVH * S * D, dtype=np.float32)
        z = z.reshape(B, KVH, S, D)
        s = _rng(seed, TAG_CHS).lognormal(0.0, 1.0, size=(KVH, D)).astype(np.float32)
        K = f32_to_bf16_bits(z * s[None, :, None, :])
        del z
    else:
        K = normal_bf16((B, KVH, S, D), seed, TAG_K)
    V = normal_bf16((B, KVH, S, D), seed, TAG_V)
    if wl.heavy_hitters > 0.0 and S > w:
        G = H // KVH
        qf = bf16_bits_to_f32(q).reshape(B, KVH, G * w, D)
        qbar = qf.mean(axis=2, dtype=np.float32)  # [B, KVH, D]
        n_hh = max(1, int(round(wl.heavy_hitters * (S - w))))
        g = _rng(seed, TAG_HH)
        for b in range(B):
            for kv in range(KVH):
                pos = g.choice(S - w, size=n_hh, replace=False)
                rows = bf16_bits_to_f32(K[b, kv, pos]) + np.float32(3.0) * qbar[b, kv]
                K[b, kv, pos] = f32_to_bf16_bits(rows.astype(np.float32))
    return {"q": q, "K": K, "V": V}


def decode_step_inputs(wl: Workload, step: int, seed: int | None = None) -> dict:
    """One decode step: new query [B,H,D], new key/value rows [B,KVH,D] (bf16 bits)."""
    seed = wl.seed if seed is None else seed
    return {
        "q": normal_bf16((wl.B, wl.H, wl.D), seed, TAG_STEP, step, 0),
        "k": normal_bf16((wl.B, wl.KVH, wl.D), seed, TAG_STEP, step, 1),
        "v": normal_bf16((wl.B, wl.KVH, wl.D), seed, TAG_STEP, step, 2),
    }


def random_scores(shape, seed: int, tie_levels: int = 0) -> np.ndarray:
    """Non-negative float32 scores for selection tests.  ``tie_levels > 0`` draws from only
    that many distinct values, so that many exact ties occur."""
    g = _rng(seed, TAG_SCORES)
    if tie_levels > 0:
        lv = g.random(tie_levels, dtype=np.float32)
        return lv[g.integers(0, tie_levels, size=shape)]
    return g.random(shape, dtype=np.float32)


def random_live_mask(shape, seed: int, p_live: float = 0.7) -> np.ndarray:
    """Boolean liveness pattern for decode caches (``shape`` = [B, KVH, S])."""
    return _rng(seed, TAG_LIVE).random(shape) < p_live


def pack_live_bits(live: np.ndarray) -> np.ndarray:
    """Pack a boolean [..., S] mask into little-endian uint32 words [..., ceil(S/32)]
    (bit j%32 of word j//32 is slot j)."""
    live = np.asarray(live, dtype=bool)
    S = live.shape[-1]
    n_w = (S + 31) // 32
    pad = np.zeros(live.shape[:-1] + (n_w * 32,), dtype=bool)
    pad[..., :S] = live
    bits = pad.reshape(live.shape[:-1] + (n_w, 32)).astype(np.uint64)
    words = (bits << np.arange(32, dtype=np.uint64)).sum(axis=-1)
    return words.astype(np.uint32)


def unpack_live_bits(words: np.ndarray, S: int) -> np.ndarray:
    words = np.asarray(words, dtype=np.uint32).astype(np.uint64)
    bits = (words[..., None] >> np.arange(32, dtype=np.uint64)) & 1
    return bits.reshape(words.shape[:-1] + (-1,))[..., :S].astype(bool)
