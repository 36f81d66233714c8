"""Repeat-run determinism: every C-ABI call, run ten times on the same inputs (and, for the
decode steps, from the same starting state), gives bit-identical outputs.

Each kernel path is covered: the tensor-core window scores with split key ranges, the
streaming decode-row scores (one-kernel TOVA step with its cluster head-mean), the small-row
fallback, the single-CTA and cluster top-k, the fused one-CTA prefill, the Scissorhands
update/evict/queue, the channel scores and prune, and decode attention over many key ranges.
No kernel uses floating-point atomics or arrival-order reductions, so any difference between
runs is a bug (a race or an uninitialised read), not rounding.
"""
import numpy as np
import pytest
import torch

import attention_score_kv_window_gb300 as kvc
from synth import Workload, prefill_inputs, decode_step_inputs, random_scores, normal_bf16
from tests.helpers import dev_bf16, dev_i32

pytestmark = pytest.mark.gpu

RUNS = 10


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kvc.load_library()
    yield
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


def _same(runs):
    """All runs equal the first, tensor by tensor, bit for bit."""
    first = runs[0]
    for r in runs[1:]:
        for a, b in zip(first, r):
            if a is None:
                assert b is None
                continue
            assert a.dtype == b.dtype and a.shape == b.shape
            if a.is_floating_point():
                assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                                   b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))
            else:
                assert torch.equal(a, b)


def _wl(B, H, KVH, D, S, w, seed, **kw):
    return Workload("t", B=B, H=H, KVH=KVH, D=D, S=S, w=w, k=1, reduce="gqa", seed=seed, **kw)


@pytest.mark.parametrize("B,H,KVH,D,S,w,causal,reduce", [
    (1, 32, 8, 128, 32768, 64, True, "gqa"),       # tensor-core scores, split key ranges
    (2, 16, 4, 64, 5000, 40, True, "all_heads"),   # tensor-core, D = 64, all-heads mean
    (16, 32, 8, 128, 8193, 1, False, "all_heads"),  # streaming decode rows
    (3, 8, 8, 64, 777, 5, True, "all_heads"),      # small-row kernel
])
def test_window_scores_repeatable(B, H, KVH, D, S, w, causal, reduce):
    inp = prefill_inputs(_wl(B, H, KVH, D, S, w, seed=S))
    q, K = dev_bf16(inp["q"]), dev_bf16(inp["K"])
    _same([(kvc.kvc_window_scores(q, K, 0.09, causal=causal, reduce=reduce),) for _ in range(RUNS)])


@pytest.mark.parametrize("B,KVH,S,k,protect,largest", [
    (2, 8, 4096, 1024, 64, True),      # one CTA per row
    (1, 2, 131072, 8192, 64, True),    # cluster rows
    (2, 2, 9000, 3000, 0, False),      # cluster rows, evict (smallest)
])
def test_topk_select_repeatable(B, KVH, S, k, protect, largest):
    # few distinct values, so that many keys tie at the threshold: the tie-break must be stable too
    scd = torch.from_numpy(random_scores((B, KVH, S), S + k, tie_levels=50)).cuda()
    _same([(kvc.kvc_topk_select(scd, k, protect_tail=protect, largest=largest),) for _ in range(RUNS)])


@pytest.mark.parametrize("B,H,KVH,D,S,w,k,protect,reduce", [
    (256, 8, 2, 64, 512, 1, 256, 0, "all_heads"),      # fused one-CTA prefill (TOVA at prefill)
    (1, 32, 8, 128, 32768, 64, 4096, 64, "gqa"),       # SnapKV layer: scores, cluster select, gather
])
def test_compress_prefill_repeatable(B, H, KVH, D, S, w, k, protect, reduce):
    inp = prefill_inputs(_wl(B, H, KVH, D, S, w, seed=7 + S))
    q, K, V = dev_bf16(inp["q"]), dev_bf16(inp["K"]), dev_bf16(inp["V"])
    scale = 1.0 / np.sqrt(D)
    _same([kvc.kvc_compress_prefill(q, K, V, scale, k, protect_tail=protect, reduce=reduce) for _ in range(RUNS)])


def test_tova_decode_step_repeatable():
    """Three decode steps from the same cache state, ten times: scores, evicted slots and the
    cache contents agree bit for bit (one-kernel step with the cluster head-mean)."""
    B, H, KVH, D, budget = 16, 32, 8, 128, 2048
    wl = Workload("t", B=B, H=H, KVH=KVH, D=D, S=budget + 1, w=1, k=budget, reduce="all_heads", causal=False,
                  seed=61)
    pre = prefill_inputs(wl)
    K0, V0 = dev_bf16(pre["K"]), dev_bf16(pre["V"])
    steps = [decode_step_inputs(wl, t) for t in range(3)]
    scale = 1.0 / np.sqrt(D)
    runs = []
    for _ in range(RUNS):
        K, V = K0.clone(), V0.clone()
        free = dev_i32(np.full((B, KVH), budget, np.int32))
        out = []
        for s in steps:
            sc = kvc.kvc_tova_decode_step(dev_bf16(s["q"]), dev_bf16(s["k"]), dev_bf16(s["v"]), K, V, scale, free)
            out += [sc, free.clone()]
        runs.append(out + [K, V])
    _same(runs)


@pytest.mark.parametrize("policy", ["bulk", "queue"])
def test_scissorhands_repeatable(policy):
    """Decode steps with history recording and eviction, ten times from the same state."""
    B, H, KVH, D, cap, hist, m = 8, 32, 8, 128, 4096, 400, 32
    wl = Workload("t", B=B, H=H, KVH=KVH, D=D, S=cap, w=1, k=cap, reduce="gqa", causal=False, seed=71)
    pre = prefill_inputs(wl)
    K0, V0 = dev_bf16(pre["K"]), dev_bf16(pre["V"])
    steps = [decode_step_inputs(wl, t) for t in range(m + 4)]
    scale = 1.0 / np.sqrt(D)
    runs = []
    for _ in range(RUNS):
        st = kvc.ScissorhandsState(B, KVH, cap, history=hist)
        kvc.kvc_scissorhands_init(st, cap - m)
        K, V = K0.clone(), V0.clone()
        out, queue, pos = [], None, m
        for i, s in enumerate(steps):
            qa = {}
            if policy == "queue" and i >= m:
                if pos == m:
                    queue = kvc.kvc_scissorhands_refill_queue(st, m)
                    out.append(queue.clone())
                    pos = 0
                qa, pos = {"queue": queue, "pos": pos}, pos + 1
            out.append(kvc.kvc_scissorhands_update(st, dev_bf16(s["q"]), dev_bf16(s["k"]), dev_bf16(s["v"]), K, V,
                                                   scale, **qa))
            if policy == "bulk" and (i + 1) % m == 0:
                out.append(kvc.kvc_scissorhands_evict(st, m))
        runs.append(out + [K, V, st.hist.clone(), st.low_count.clone(), st.insert_step.clone(), st.live.clone(),
                           st.slot.clone()])
    _same(runs)


def test_compress_prefill_channels_repeatable():
    """Compaction with the kept keys' channel sums (per-CTA partials in a fixed order)."""
    B, H, KVH, D, S, w, k = 1, 32, 8, 128, 32768, 64, 4096
    inp = prefill_inputs(_wl(B, H, KVH, D, S, w, seed=91))
    q, K, V = dev_bf16(inp["q"]), dev_bf16(inp["K"]), dev_bf16(inp["V"])
    _same([kvc.kvc_compress_prefill_channels(q, K, V, 0.088, k, protect_tail=w) for _ in range(RUNS)])


def test_channel_paths_repeatable():
    """Channel scores (query rows by kept keys), channel prune, value-channel scores."""
    B, H, KVH, D, S, w, k, C = 2, 32, 8, 128, 4096, 64, 1024, 64
    inp = prefill_inputs(_wl(B, H, KVH, D, S, w, seed=81))
    q, K, V = dev_bf16(inp["q"]), dev_bf16(inp["K"]), dev_bf16(inp["V"])
    idx = dev_i32(np.sort(np.random.default_rng(8).permutation(S)[:k]).astype(np.int32)[None, None]
                  .repeat(B, 0).repeat(KVH, 1))
    scale = 1.0 / np.sqrt(D)
    runs = []
    for _ in range(RUNS):
        cs = kvc.kvc_channel_score(q, K, idx=idx)
        ch, Kp = kvc.kvc_channel_prune(cs, K, C)
        vs = kvc.kvc_value_channel_score(q, K[:, :, :k].contiguous(), V[:, :, :k].contiguous(), scale)
        runs.append((cs, ch, Kp, vs))
    _same(runs)


@pytest.mark.parametrize("C,S", [(64, 8192), (128, 40000)])
def test_decode_attention_repeatable(C, S):
    """Decode attention over the channel-pruned (C < D) or full cache, many key ranges merged."""
    B, H, KVH, D = 16 if S <= 8192 else 2, 32, 8, 128
    q = normal_bf16((B, H, D), S, 1)
    K = normal_bf16((B, KVH, S, D), S, 2)
    V = normal_bf16((B, KVH, S, D), S, 3)
    qd, Vd = dev_bf16(q), dev_bf16(V)
    scale = 1.0 / np.sqrt(D)
    if C < D:
        cs = torch.from_numpy(random_scores((B, KVH, D), S + 1)).cuda()
        ch, Kp = kvc.kvc_channel_prune(cs, dev_bf16(K), C)
        call = lambda: (kvc.kvc_decode_attention(qd, Kp, Vd, scale, ch=ch),)
    else:
        Kd = dev_bf16(K)
        call = lambda: (kvc.kvc_decode_attention(qd, Kd, Vd, scale),)
    _same([call() for _ in range(RUNS)])
