"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Sizes span several key tiles (64 keys) and split ranges, with ragged tails; tolerances are
the ones stated for this method: fp32 scores within 1e-3 relative, compaction bit-exact,
kept sets identical except oracle near-ties (within 1e-3 of the k-th score).
"""
import numpy as np
import pytest
import torch

import oracle as O
import attention_score_kv_window_gb300 as kvc
from synth import (Workload, prefill_inputs, decode_step_inputs, random_scores, random_live_mask,
                   pack_live_bits, normal_bf16)
from tests.helpers import (dev_bf16, host_bits, dev_i32, dev_u32, assert_scores_close,
                           assert_selection_matches)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kvc.load_library()
    yield
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


def _wl(B, H, KVH, D, S, w, seed=0, **kw):
    return Workload("t", B=B, H=H, KVH=KVH, D=D, S=S, w=w, k=1, reduce="gqa", seed=seed, **kw)


# ----------------------------------------------------------------------------------------
# window scores
# ----------------------------------------------------------------------------------------

SCORE_CASES = [
    # B, H, KVH, D, S, w, causal, reduce
    (1, 8, 2, 64, 512, 1, True, "all_heads"),
    (1, 8, 2, 64, 1, 1, True, "gqa"),
    (2, 4, 4, 64, 7, 7, True, "gqa"),
    (1, 8, 1, 128, 63, 63, True, "gqa"),
    (1, 4, 1, 128, 65, 64, True, "gqa"),
    (1, 16, 2, 128, 129, 64, True, "gqa"),
    (2, 8, 2, 128, 1000, 64, True, "gqa"),
    (1, 32, 8, 128, 1000, 64, True, "gqa"),
    (3, 8, 8, 64, 777, 5, True, "all_heads"),
    (2, 32, 8, 128, 2049, 1, False, "all_heads"),
    (1, 4, 1, 64, 300, 128, True, "gqa"),     # R = 512 rows: two pass-1 row groups
    (1, 12, 4, 128, 333, 48, True, "gqa"),    # R = 144: odd m-tile count
    (1, 8, 8, 64, 4000, 40, True, "gqa"),     # R = 40
    (4, 8, 2, 128, 4096, 1, False, "gqa"),
    (1, 8, 2, 64, 3000, 32, True, "gqa"),     # R = 128: tensor-core path, one query half
    (2, 32, 8, 128, 5000, 64, False, "all_heads"),
    (40, 16, 4, 64, 256, 16, True, "gqa"),    # 160 (b, kvh) > one CTA per SM: two launches
]


@pytest.mark.parametrize("B,H,KVH,D,S,w,causal,reduce", SCORE_CASES)
def test_window_scores_parity(B, H, KVH, D, S, w, causal, reduce):
    inp = prefill_inputs(_wl(B, H, KVH, D, S, w, seed=S + w))
    scale = 1.0 / np.sqrt(D)
    got = kvc.kvc_window_scores(dev_bf16(inp["q"]), dev_bf16(inp["K"]), scale, causal=causal, reduce=reduce)
    ref = O.window_scores(inp["q"], inp["K"], scale, causal=causal, reduce=reduce)
    assert_scores_close(got.cpu().numpy(), ref)
    # sum over keys equals the window length (each window row's softmax sums to one)
    np.testing.assert_allclose(got.double().sum(-1).cpu().numpy(), w, rtol=1e-4)


def test_window_scores_shared_workspace_any_content():
    """One workspace, filled with random bytes first, serves several shapes in turn (different
    key-range counts per KV head, so the bookkeeping words land on different offsets)."""
    g = torch.Generator(device="cuda").manual_seed(11)
    ws = torch.randint(0, 256, (64 << 20,), dtype=torch.uint8, device="cuda", generator=g)
    shapes = [(1, 32, 8, 128, 32768, 64), (2, 8, 2, 128, 1000, 64), (1, 32, 8, 128, 5000, 64),
              (1, 8, 8, 64, 4000, 40), (1, 32, 8, 128, 32768, 64)]
    for i, (B, H, KVH, D, S, w) in enumerate(shapes):
        inp = prefill_inputs(_wl(B, H, KVH, D, S, w, seed=100 + i))
        scale = 1.0 / np.sqrt(D)
        q, K = dev_bf16(inp["q"]), dev_bf16(inp["K"])
        for _ in range(2):
            got = kvc.kvc_window_scores(q, K, scale, causal=True, reduce="gqa", ws=ws)
        ref = O.window_scores(inp["q"], inp["K"], scale, causal=True, reduce="gqa")
        assert_scores_close(got.cpu().numpy(), ref)
        assert kvc.kvc_get_device_status() == kvc.KVC_OK


@pytest.mark.parametrize("S,p_live", [(256, 0.7), (4096, 0.5), (100, 0.05), (64, 0.0)])
def test_window_scores_live_mask(S, p_live):
    B, H, KVH, D = 2, 8, 2, 128
    inp = prefill_inputs(_wl(B, H, KVH, D, S, 1, seed=7))
    live = random_live_mask((B, KVH, S), 3, p_live)
    got = kvc.kvc_window_scores(dev_bf16(inp["q"]), dev_bf16(inp["K"]), 0.1, causal=False,
                                live_mask=dev_u32(pack_live_bits(live)), reduce="gqa")
    ref = O.window_scores(inp["q"], inp["K"], 0.1, causal=False, live=live, reduce="gqa")
    assert_scores_close(got.cpu().numpy(), ref)
    assert np.all(got.cpu().numpy()[~live] == 0)


def test_window_scores_strided_cache():
    """K as a view with padded slots (stride_s > D, stride_h > S*D)."""
    B, H, KVH, D, S = 2, 8, 2, 128, 300
    inp = prefill_inputs(_wl(B, H, KVH, D, S, 16, seed=9))
    big = torch.zeros((B, KVH, S + 37, D + 64), dtype=torch.bfloat16, device="cuda")
    big[:, :, :S, :D] = dev_bf16(inp["K"])
    Kv = big[:, :, :S, :D]
    got = kvc.kvc_window_scores(dev_bf16(inp["q"]), Kv, 0.09, causal=True, reduce="gqa")
    ref = O.window_scores(inp["q"], inp["K"], 0.09, causal=True, reduce="gqa")
    assert_scores_close(got.cpu().numpy(), ref)


def test_window_scores_uniform_and_deterministic():
    B, H, KVH, D, S = 1, 8, 2, 64, 999
    q = np.zeros((B, H, 1, D), np.uint16)
    K = normal_bf16((B, KVH, S, D), 5, 2)
    a = kvc.kvc_window_scores(dev_bf16(q), dev_bf16(K), 0.125, causal=True, reduce="all_heads")
    np.testing.assert_allclose(a.cpu().numpy(), 1.0 / S, rtol=1e-5)
    inp = prefill_inputs(_wl(1, 32, 8, 128, 5000, 64, seed=4))
    runs = [kvc.kvc_window_scores(dev_bf16(inp["q"]), dev_bf16(inp["K"]), 0.088, reduce="gqa") for _ in range(3)]
    for r in runs[1:]:
        assert torch.equal(r, runs[0])


# ----------------------------------------------------------------------------------------
# selection
# ----------------------------------------------------------------------------------------

TOPK_CASES = [
    # B, KVH, S, k, protect, ties, largest, live_p
    (1, 2, 512, 256, 0, 0, True, None),
    (2, 3, 1000, 100, 64, 0, True, None),
    (2, 3, 1000, 100, 64, 7, True, None),
    (1, 8, 32768, 4096, 64, 0, True, None),
    (1, 2, 50000, 999, 0, 50, True, None),      # 8-CTA cluster, 50 tie levels
    # cluster rows (S > 4096): evict with ties and dead slots, fewer eligible than k, the
    # longest row, protected tails with ties and dead slots, k = S - 1
    (2, 2, 9000, 3000, 0, 2, False, 0.8),
    (1, 3, 20000, 19000, 100, 0, True, 0.9),
    (1, 2, 131072, 8192, 64, 0, True, None),
    (2, 1, 40000, 5000, 32, 3, True, 0.7),
    (1, 1, 327680, 1000, 0, 0, False, None),
    # long rows (8-CTA clusters of 8-25K keys each): live masks, ties, k close to S
    (2, 1, 100000, 5000, 32, 3, True, 0.7),
    (1, 2, 70000, 69000, 0, 0, True, None),
    (1, 1, 200000, 100, 0, 50, False, 0.5),
    (1, 2, 6000, 5999, 0, 0, True, None),
    (4, 2, 2049, 1, 0, 0, False, None),
    (4, 2, 2049, 1, 0, 3, False, None),
    (2, 2, 4096, 64, 0, 5, True, 0.9),
    (2, 2, 300, 290, 0, 0, True, 0.5),         # fewer eligible than k -> -1 padding
    (1, 1, 7, 7, 7, 0, True, None),
    (1, 1, 33, 40, 0, 0, True, None),          # k > S
    (3, 1, 129, 65, 1, 2, True, None),
    (2, 2, 777, 13, 0, 1, False, 0.6),
    (3, 2, 5000, 1, 0, 0, True, 0.5),          # k = 1 (one CTA per row), keep, live mask
    (2, 3, 70000, 1, 0, 4, False, None),       # k = 1, evict, long rows with ties
    (1, 2, 100, 1, 0, 0, True, 0.0),           # k = 1, nothing live -> -1
    # one warp per row (S <= 1024): 4, 8, 16 and 32 keys per lane
    (64, 4, 512, 256, 0, 3, True, None),       # many rows, heavy ties
    (8, 2, 1024, 1000, 20, 0, True, None),
    (8, 2, 1024, 517, 0, 9, False, 0.7),       # evict with ties and dead slots
    (5, 3, 200, 100, 32, 4, True, 0.8),
    (3, 3, 128, 2, 0, 2, False, None),
    (2, 2, 300, 299, 0, 0, True, None),
    (1, 1, 1, 1, 0, 0, True, None),
]


@pytest.mark.parametrize("B,KVH,S,k,protect,ties,largest,live_p", TOPK_CASES)
def test_topk_parity_exact(B, KVH, S, k, protect, ties, largest, live_p):
    sc = random_scores((B, KVH, S), 100 + S + k, tie_levels=ties)
    live = None if live_p is None else random_live_mask((B, KVH, S), 11, live_p)
    got = kvc.kvc_topk_select(torch.from_numpy(sc).cuda(), k, protect_tail=protect,
                              live_mask=None if live is None else dev_u32(pack_live_bits(live)), largest=largest)
    ref = O.topk_select(sc, k, protect_tail=protect, live=live, largest=largest)
    np.testing.assert_array_equal(got.cpu().numpy(), ref)


def test_topk_all_equal_scores():
    sc = np.full((2, 2, 5000), 0.25, np.float32)
    got = kvc.kvc_topk_select(torch.from_numpy(sc).cuda(), 123)
    np.testing.assert_array_equal(got.cpu().numpy(), O.topk_select(sc, 123))
    got = kvc.kvc_topk_select(torch.from_numpy(sc).cuda(), 9, largest=False)
    np.testing.assert_array_equal(got.cpu().numpy(), O.topk_select(sc, 9, largest=False))


# ----------------------------------------------------------------------------------------
# compaction
# ----------------------------------------------------------------------------------------


@pytest.mark.parametrize("D", [64, 128])
def test_compact_bit_exact(D):
    B, KVH, S, k = 2, 3, 517, 200
    K = normal_bf16((B, KVH, S, D), 21, 1)
    V = normal_bf16((B, KVH, S, D), 21, 2)
    idx = O.topk_select(random_scores((B, KVH, S), 4), k)
    idx[0, 1, -5:] = -1
    big = torch.zeros((B, KVH, S + 3, D), dtype=torch.bfloat16, device="cuda")
    big[:, :, :S] = dev_bf16(K)
    bigv = torch.zeros_like(big)
    bigv[:, :, :S] = dev_bf16(V)
    Ko, Vo = kvc.kvc_compact_kv(big[:, :, :S], bigv[:, :, :S], dev_i32(idx))
    Kr, Vr = O.compact_kv(K, V, idx)
    np.testing.assert_array_equal(host_bits(Ko), Kr)
    np.testing.assert_array_equal(host_bits(Vo), Vr)


TOPK_COMPACT_CASES = [
    # B, KVH, S, k, protect, D, ties, largest, live_p, with_v, strided
    (1, 8, 32768, 4096, 64, 128, 0, True, None, True, False),   # SnapKV layer, full size
    (2, 3, 10000, 777, 0, 64, 5, True, None, True, True),       # heavy ties, strided cache
    (1, 2, 5000, 6000, 0, 128, 0, True, None, True, False),     # k > S: -1 padding, zero rows
    (2, 2, 3000, 100, 0, 64, 0, True, None, True, False),       # short rows: two launches
    (1, 4, 20000, 1500, 0, 128, 0, False, None, False, False),  # evict order, keys only
    (1, 2, 12000, 500, 0, 128, 0, True, 0.5, True, False),      # live mask
    (1, 2, 12000, 9000, 0, 64, 0, True, 0.5, True, False),      # fewer live than k
]


@pytest.mark.parametrize("B,KVH,S,k,protect,D,ties,largest,live_p,with_v,strided", TOPK_COMPACT_CASES)
def test_topk_compact_exact(B, KVH, S, k, protect, D, ties, largest, live_p, with_v, strided):
    """Selection and gather in one call: indices equal the oracle's on the same fp32 scores,
    gathered rows bit-exact, zero rows where the index is -1."""
    sc = random_scores((B, KVH, S), 300 + S + k, tie_levels=ties)
    live = None if live_p is None else random_live_mask((B, KVH, S), 12, live_p)
    K = normal_bf16((B, KVH, S, D), 31, 1)
    V = normal_bf16((B, KVH, S, D), 31, 2)
    if strided:
        big = torch.zeros((B, KVH, S + 5, D), dtype=torch.bfloat16, device="cuda")
        big[:, :, :S] = dev_bf16(K)
        bigv = torch.zeros_like(big)
        bigv[:, :, :S] = dev_bf16(V)
        Kd, Vd = big[:, :, :S], bigv[:, :, :S]
    else:
        Kd, Vd = dev_bf16(K), dev_bf16(V)
    idx, Ko, Vo = kvc.kvc_topk_compact(torch.from_numpy(sc).cuda(), Kd, Vd if with_v else None, k,
                                       protect_tail=protect, largest=largest,
                                       live_mask=None if live is None else dev_u32(pack_live_bits(live)))
    ref = O.topk_select(sc, k, protect_tail=protect, live=live, largest=largest)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)
    Kr, Vr = O.compact_kv(K, V, ref)
    np.testing.assert_array_equal(host_bits(Ko), Kr)
    if with_v:
        np.testing.assert_array_equal(host_bits(Vo), Vr)
    else:
        assert Vo is None
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


def test_compaction_reads_v_from_page_locked_host_memory():
    """V may stay in page-locked host memory: the compaction kernel reads the kept rows over
    the host link; results are bit-identical to a device V."""
    B, H, KVH, D, S, k = 2, 8, 2, 128, 3000, 700
    sc = random_scores((B, KVH, S), 71, tie_levels=0)
    K = normal_bf16((B, KVH, S, D), 71, 2)
    V = normal_bf16((B, KVH, S, D), 71, 3)
    hV = torch.from_numpy(V.view(np.int16)).view(torch.bfloat16).pin_memory()
    idx, Ko, Vo = kvc.kvc_topk_compact(torch.from_numpy(sc).cuda(), dev_bf16(K), hV, k, protect_tail=64, H=H)
    ref_idx = O.topk_select(sc, k, protect_tail=64)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    rK, rV = O.compact_kv(K, V, ref_idx)
    np.testing.assert_array_equal(host_bits(Ko), rK)
    np.testing.assert_array_equal(host_bits(Vo), rV)
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


def test_compact_out_of_range_index_reports_bounds():
    K = dev_bf16(normal_bf16((1, 1, 10, 64), 1, 1))
    idx = dev_i32(np.array([[[0, 10, 3]]]))
    kvc.kvc_compact_kv(K, None, idx)
    assert kvc.kvc_get_device_status() == kvc.KVC_ERR_DEVICE_BOUNDS
    assert kvc.kvc_get_device_status() == kvc.KVC_OK  # cleared on read


# ----------------------------------------------------------------------------------------
# fused prefill compression (TOVA / SnapKV)
# ----------------------------------------------------------------------------------------

PREFILL_CASES = [
    # B, H, KVH, D, S, w, k, protect, reduce, hh
    (1, 8, 2, 64, 512, 1, 256, 0, "all_heads", 0.0),
    (1, 32, 8, 128, 2000, 64, 512, 64, "gqa", 0.01),
    (2, 16, 4, 128, 1500, 64, 200, 64, "gqa", 0.01),
    (1, 8, 2, 64, 100, 16, 128, 16, "gqa", 0.0),   # k > S: keep all
    # short rows: the fused one-kernel path (G*w <= 16, the key block in shared memory)
    (3, 8, 2, 64, 500, 1, 256, 0, "all_heads", 0.0),     # ragged S, 2-CTA clusters
    (2, 8, 8, 64, 1000, 2, 300, 2, "gqa", 0.0),          # G 1, 16 key tiles per warp
    (2, 16, 4, 128, 300, 4, 100, 4, "gqa", 0.01),        # 16 query rows, 128 channels
    (2, 32, 8, 128, 64, 1, 16, 0, "all_heads", 0.0),     # 8-CTA clusters, one key tile per warp
    (1, 8, 2, 64, 40, 2, 64, 2, "all_heads", 0.0),       # k > S: all kept, -1 padded, zero rows
    (1, 4, 4, 64, 1024, 16, 512, 16, "gqa", 0.01),       # w 16, window protected
    (4, 16, 8, 64, 777, 2, 513, 0, "gqa", 0.0),          # k not a multiple of 64
    # all-heads rows scored head by head in one CTA: 4 heads of 128 channels, 8 heads of 64
    # channels over 16 key tiles per warp, 3 heads with every token kept
    (2, 16, 4, 128, 512, 2, 200, 2, "all_heads", 0.01),
    (1, 16, 8, 64, 1000, 1, 300, 1, "all_heads", 0.0),
    (3, 12, 3, 64, 333, 4, 333, 4, "all_heads", 0.0),
]


@pytest.mark.parametrize("B,H,KVH,D,S,w,k,protect,reduce,hh", PREFILL_CASES)
def test_compress_prefill_parity(B, H, KVH, D, S, w, k, protect, reduce, hh):
    wl = _wl(B, H, KVH, D, S, w, seed=31, heavy_hitters=hh)
    inp = prefill_inputs(wl)
    scale = 1.0 / np.sqrt(D)
    sc, idx, Ko, Vo = kvc.kvc_compress_prefill(dev_bf16(inp["q"]), dev_bf16(inp["K"]), dev_bf16(inp["V"]), scale, k,
                                               protect_tail=protect, reduce=reduce)
    ref = O.window_scores(inp["q"], inp["K"], scale, causal=True, reduce=reduce)
    assert_scores_close(sc.cpu().numpy(), ref)
    gi = idx.cpu().numpy()
    assert_selection_matches(gi, ref, k, protect_tail=protect)
    if protect:
        for b in range(B):
            for kv in range(KVH):
                assert set(range(S - protect, S)) <= set(gi[b, kv].tolist())
    # compaction is exact given the chosen indices
    Kr, Vr = O.compact_kv(inp["K"], inp["V"], gi)
    np.testing.assert_array_equal(host_bits(Ko), Kr)
    np.testing.assert_array_equal(host_bits(Vo), Vr)


def test_compress_prefill_fused_options():
    """The short-row kernel: scores left unwritten give the same selection and compaction bit
    for bit; a strided cache (a view of a longer one) and V in page-locked host memory give
    the oracle's rows."""
    B, H, KVH, D, S, w, k = 2, 8, 2, 64, 512, 1, 256
    wl = _wl(B, H, KVH, D, S, w, seed=57)
    inp = prefill_inputs(wl)
    scale = 1.0 / np.sqrt(D)
    q, K, V = dev_bf16(inp["q"]), dev_bf16(inp["K"]), dev_bf16(inp["V"])
    sc, idx, Ko, Vo = kvc.kvc_compress_prefill(q, K, V, scale, k, reduce="all_heads")
    none, idx2, Ko2, Vo2 = kvc.kvc_compress_prefill(q, K, V, scale, k, reduce="all_heads", keep_scores=False)
    assert none is None
    assert torch.equal(idx, idx2) and torch.equal(Ko, Ko2) and torch.equal(Vo, Vo2)
    # a strided cache: rows 0..S-1 of a longer buffer
    bigK = torch.zeros((B, KVH, S + 37, D), dtype=torch.bfloat16, device="cuda")
    bigV = torch.zeros_like(bigK)
    bigK[:, :, :S] = K
    bigV[:, :, :S] = V
    sc3, idx3, Ko3, Vo3 = kvc.kvc_compress_prefill(q, bigK[:, :, :S], bigV[:, :, :S], scale, k, reduce="all_heads")
    assert torch.equal(sc, sc3) and torch.equal(idx, idx3) and torch.equal(Ko, Ko3) and torch.equal(Vo, Vo3)
    # V read over the host link
    hV = torch.from_numpy(inp["V"].view(np.int16)).view(torch.bfloat16).pin_memory()
    _, idx4, Ko4, Vo4 = kvc.kvc_compress_prefill(q, K, hV, scale, k, reduce="all_heads", keep_scores=False)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx4) and torch.equal(Ko, Ko4) and torch.equal(Vo, Vo4)
    ref = O.window_scores(inp["q"], inp["K"], scale, causal=True, reduce="all_heads")
    assert_scores_close(sc.cpu().numpy(), ref)
    gi = idx.cpu().numpy()
    assert_selection_matches(gi, ref, k)
    Kr, Vr = O.compact_kv(inp["K"], inp["V"], gi)
    np.testing.assert_array_equal(host_bits(Ko), Kr)
    np.testing.assert_array_equal(host_bits(Vo), Vr)


def test_tova_prefill_8192_instances_sampled():
    """TOVA prefill (8 query / 2 KV heads, 64 channels, 512 tokens, keep 256) stacked as 8192
    independent instances in one call: the benchmark's launch configuration.  All instances
    on the GPU; a seeded sample of 16 by the oracle (scores, kept set, compacted rows); every
    instance's scores sum to 1 and are identical for both KV heads (mean over all heads)."""
    from synth import TOVA_PREFILL
    wl = TOVA_PREFILL.with_(B=8192)
    inp = prefill_inputs(wl)
    q, K, V = dev_bf16(inp["q"]), dev_bf16(inp["K"]), dev_bf16(inp["V"])
    sc, idx, Ko, Vo = kvc.kvc_compress_prefill(q, K, V, wl.scale, wl.k, reduce="all_heads")
    g_sc = sc.cpu().numpy()
    np.testing.assert_allclose(g_sc.astype(np.float64).sum(-1), 1.0, rtol=1e-4)
    assert np.array_equal(g_sc[:, 0], g_sc[:, 1])
    g_idx = idx.cpu().numpy()
    assert np.array_equal(g_idx[:, 0], g_idx[:, 1])
    hK, hV = host_bits(Ko), host_bits(Vo)
    sample = np.random.Generator(np.random.PCG64([2024])).choice(wl.B, size=16, replace=False)
    for b in sample:
        sl = slice(int(b), int(b) + 1)
        ref = O.window_scores(inp["q"][sl], inp["K"][sl], wl.scale, causal=True, reduce="all_heads")
        assert_scores_close(g_sc[sl], ref, what=f"instance {b} scores")
        assert_selection_matches(g_idx[sl], ref, wl.k)
        rK, rV = O.compact_kv(inp["K"][sl], inp["V"][sl], g_idx[sl])
        np.testing.assert_array_equal(hK[sl], rK)
        np.testing.assert_array_equal(hV[sl], rV)


def test_snapkv_32k_layer_sampled_kv_head():
    """The SnapKV 32K layer (32 query / 8 KV heads, 128 channels, window 64, keep 4096, 1 %
    heavy hitters) at full size through kvc_compress_prefill, the chain the benchmark times:
    every KV head on the GPU, one by the oracle (scores, kept set with the window, compacted
    rows); every row's scores sum to the window length."""
    from synth import SNAPKV_32K
    wl = SNAPKV_32K
    inp = prefill_inputs(wl)
    G, scale = wl.G, wl.scale
    q, K, V = dev_bf16(inp["q"]), dev_bf16(inp["K"]), dev_bf16(inp["V"])
    sc, idx, Ko, Vo = kvc.kvc_compress_prefill(q, K, V, scale, wl.k, protect_tail=wl.protect_tail, reduce="gqa")
    np.testing.assert_allclose(sc.double().sum(-1).cpu().numpy(), wl.w, rtol=1e-4)
    kv = 5
    qh, Kh, Vh = inp["q"][:, kv * G:(kv + 1) * G], inp["K"][:, kv:kv + 1], inp["V"][:, kv:kv + 1]
    ref = O.window_scores(qh, Kh, scale, causal=True, reduce="gqa")
    assert_scores_close(sc.cpu().numpy()[:, kv:kv + 1], ref)
    g_idx = idx.cpu().numpy()[:, kv:kv + 1]
    assert_selection_matches(g_idx, ref, wl.k, protect_tail=wl.protect_tail)
    assert set(range(wl.S - wl.w, wl.S)) <= set(g_idx[0, 0].tolist())
    rK, rV = O.compact_kv(Kh, Vh, g_idx)
    np.testing.assert_array_equal(host_bits(Ko)[:, kv:kv + 1], rK)
    np.testing.assert_array_equal(host_bits(Vo)[:, kv:kv + 1], rV)


# ----------------------------------------------------------------------------------------
# TOVA decode (teacher-forced)
# ----------------------------------------------------------------------------------------


@pytest.mark.parametrize("B,H,KVH,D,S,budget,steps", [
    (2, 8, 2, 128, 700, 256, 8), (2, 16, 4, 64, 3000, 2048, 4),
    # B x KVH above half the SM count: one CTA per (b, kvh) and the step is one kernel (head
    # clusters of KVH CTAs average over the heads and evict); the first is the benchmark's shape
    (16, 32, 8, 128, 2100, 2048, 3), (40, 8, 2, 128, 1100, 1000, 3), (20, 16, 4, 64, 900, 777, 3),
])
def test_tova_decode_steps_teacher_forced(B, H, KVH, D, S, budget, steps):
    wl = Workload("t", B=B, H=H, KVH=KVH, D=D, S=S, w=1, k=budget, reduce="all_heads", causal=False, seed=41)
    pre = prefill_inputs(wl)
    scale = 1.0 / np.sqrt(D)
    st0 = decode_step_inputs(wl, 0)
    # first step: append, score, keep the budget
    sc0, idx0, Kc, Vc = O.tova_first_step(pre["K"], pre["V"], st0["q"], st0["k"], st0["v"], scale, budget)
    Kf = np.concatenate([pre["K"], st0["k"][:, :, None]], axis=2)
    Vf = np.concatenate([pre["V"], st0["v"][:, :, None]], axis=2)
    q0 = dev_bf16(st0["q"])[:, :, None, :]
    g_sc0 = kvc.kvc_window_scores(q0, dev_bf16(Kf), scale, causal=False, reduce="all_heads")
    assert_scores_close(g_sc0.cpu().numpy(), sc0)
    g_idx0 = kvc.kvc_topk_select(g_sc0, budget)
    assert_selection_matches(g_idx0.cpu().numpy(), sc0, budget)
    # later steps on a (budget+1)-slot cache, fed the same state on both sides
    Kd = torch.zeros((B, KVH, budget + 1, D), dtype=torch.bfloat16, device="cuda")
    Vd = torch.zeros_like(Kd)
    Kd[:] = dev_bf16(Kc)
    Vd[:] = dev_bf16(Vc)
    free = np.full((B, KVH), budget, np.int32)
    near = 0
    for t in range(1, steps + 1):
        st = decode_step_inputs(wl, t)
        fs = dev_i32(free)
        qd, kd, vd = dev_bf16(st["q"]), dev_bf16(st["k"]), dev_bf16(st["v"])
        n0 = kvc.kvc_launch_count()
        g_sc = kvc.kvc_tova_decode_step(qd, kd, vd, Kd, Vd, scale, fs)
        if 2 * B * KVH > torch.cuda.get_device_properties(0).multi_processor_count:
            assert kvc.kvc_launch_count() - n0 == 1  # the one-kernel step
        r_sc, r_ev, Kc, Vc = O.tova_decode_step(Kc, Vc, st["q"], st["k"], st["v"], free, scale)
        np.testing.assert_array_equal(host_bits(Kd), Kc)
        np.testing.assert_array_equal(host_bits(Vd), Vc)
        assert_scores_close(g_sc.cpu().numpy(), r_sc)
        g_ev = fs.cpu().numpy()
        assert np.all(g_ev == g_ev[:, :1])
        for b in range(B):
            if g_ev[b, 0] != r_ev[b, 0]:
                a, c = r_sc[b, 0, g_ev[b, 0]], r_sc[b, 0, r_ev[b, 0]]
                assert abs(a - c) <= 1e-3 * abs(c)
                near += 1
        free = r_ev.astype(np.int32)  # teacher forcing: continue from the oracle's choice
    assert near <= max(2, B * steps // 8)


def test_think_128k_layer_sampled_kv_head():
    """The ThinK + SnapKV 128K layer at full size, in the launch configuration the benchmark
    times: every KV head on the GPU, one KV head by the oracle (scores, kept set, compacted
    rows, channel scores); every row's scores sum to the window length."""
    from synth import THINK_128K
    wl = THINK_128K
    inp = prefill_inputs(wl)
    G, scale = wl.G, wl.scale
    q, K, V = dev_bf16(inp["q"]), dev_bf16(inp["K"]), dev_bf16(inp["V"])
    sc, idx, Ko, Vo, cs = kvc.kvc_compress_prefill_channels(q, K, V, scale, wl.k, protect_tail=wl.protect_tail,
                                                            reduce="gqa")
    cs = cs.cpu().numpy()
    np.testing.assert_allclose(sc.double().sum(-1).cpu().numpy(), wl.w, rtol=1e-4)
    kv = 3
    qh, Kh, Vh = inp["q"][:, kv * G:(kv + 1) * G], inp["K"][:, kv:kv + 1], inp["V"][:, kv:kv + 1]
    ref = O.window_scores(qh, Kh, scale, causal=True, reduce="gqa")
    g_sc = sc.cpu().numpy()[:, kv:kv + 1]
    assert_scores_close(g_sc, ref)
    g_idx = idx.cpu().numpy()[:, kv:kv + 1]
    assert_selection_matches(g_idx, ref, wl.k, protect_tail=wl.protect_tail)
    rK, rV = O.compact_kv(Kh, Vh, g_idx)  # the gather, given the GPU's kept set
    np.testing.assert_array_equal(host_bits(Ko)[:, kv:kv + 1], rK)
    np.testing.assert_array_equal(host_bits(Vo)[:, kv:kv + 1], rV)
    assert_scores_close(cs[:, kv:kv + 1], O.channel_score(qh, Kh, kept=g_idx), what="channel score")


def test_tova_decode_full_size_properties():
    """B 16, 2049 slots (the benchmark's decode shape): each row's scores are a mean of softmax
    rows (sum 1), identical for every KV head of a batch row, and the evicted slot is their
    argmin (lowest score; ties: highest slot); the new rows land in the freed slots."""
    B, H, KVH, D, n = 16, 32, 8, 128, 2049
    g = torch.Generator(device="cuda").manual_seed(5)
    K = torch.randn((B, KVH, n, D), generator=g, device="cuda").to(torch.bfloat16)
    V = torch.randn((B, KVH, n, D), generator=g, device="cuda").to(torch.bfloat16)
    free = torch.full((B, KVH), n - 1, dtype=torch.int32, device="cuda")
    for step in range(3):
        q = torch.randn((B, H, D), generator=g, device="cuda").to(torch.bfloat16)
        kn = torch.randn((B, KVH, D), generator=g, device="cuda").to(torch.bfloat16)
        vn = torch.randn((B, KVH, D), generator=g, device="cuda").to(torch.bfloat16)
        slot = free.clone()
        sc = kvc.kvc_tova_decode_step(q, kn, vn, K, V, 1.0 / np.sqrt(D), free).cpu().numpy()
        s = slot.cpu().numpy()
        for b in range(B):
            for h in range(KVH):
                assert torch.equal(K[b, h, s[b, h]], kn[b, h]) and torch.equal(V[b, h, s[b, h]], vn[b, h])
        np.testing.assert_allclose(sc.astype(np.float64).sum(-1), 1.0, rtol=1e-4)
        assert np.all(sc == sc[:, :1])
        ev = free.cpu().numpy()
        for b in range(B):
            row = sc[b, 0]
            exp = max(range(n), key=lambda j: (-row[j], j))
            assert np.all(ev[b] == exp)


# ----------------------------------------------------------------------------------------
# Scissorhands
# ----------------------------------------------------------------------------------------


def _sh_host(state):
    live = np.unpackbits(state.live.cpu().numpy().view(np.uint8), bitorder="little").reshape(
        state.live.shape[0], state.live.shape[1], -1).astype(bool)
    return (live, state.low_count.cpu().numpy().view(np.uint16).astype(np.int64),
            state.insert_step.cpu().numpy().astype(np.int64))


def test_scissorhands_update_from_probs_and_evict_exact():
    """Given the same float32 probabilities, flags, counts and evictions are exact
    (no insertions here: the live set only shrinks by eviction)."""
    B, KVH, cap, hist, m = 2, 3, 256, 9, 8
    st = kvc.ScissorhandsState(B, KVH, cap, history=hist)
    kvc.kvc_scissorhands_init(st, cap)
    ref = O.Scissorhands(B, KVH, cap, history=hist)
    ref.prefill(cap)
    g = np.random.Generator(np.random.PCG64([77]))
    for step in range(40):
        keys = ref.live.sum(-1, keepdims=True)
        p = np.where(ref.live, g.random((B, KVH, cap)) * 2.0 / keys, 0.0).astype(np.float32)
        if step % 5 == 0:  # values exactly at the threshold are not low (strict <)
            p[..., :4] = (np.float32(1) / keys.astype(np.float32))[..., 0:1]
        kvc.kvc_scissorhands_update_from_probs(st, torch.from_numpy(p).cuda())
        ref.record(p)
        live, low, ins = _sh_host(st)
        np.testing.assert_array_equal(live, ref.live)
        np.testing.assert_array_equal(np.where(live, low, 0), np.where(ref.live, ref.low, 0))
        if (step + 1) % m == 0:
            ev = kvc.kvc_scissorhands_evict(st, m)
            np.testing.assert_array_equal(ev.cpu().numpy(), ref.evict(m))
    assert st.t == 40
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


def test_scissorhands_threshold_counts_live_keys_hand_built():
    """cold-compress PR 11 (``keys = attn.shape[1]``, flags written to ``[:keys]``): the
    threshold is 1/(live keys), not 1/capacity.  5 of 32 slots live (slots 0..4); the flags,
    bit plane and counts expected are written out here, not taken from the oracle."""
    cap = 32
    st = kvc.ScissorhandsState(1, 1, cap, history=4)
    kvc.kvc_scissorhands_init(st, 5)
    fifth = np.float32(1) / np.float32(5)
    p = np.zeros((1, 1, cap), np.float32)
    p[0, 0, :5] = [fifth, np.nextafter(fifth, np.float32(0)), np.float32(0.0625),
                   np.nextafter(fifth, np.float32(1)), np.float32(0.5)]
    p[0, 0, 5:] = np.float32(1e-9)  # dead slots: never flagged
    kvc.kvc_scissorhands_update_from_probs(st, torch.from_numpy(p).cuda())
    plane0 = st.hist[0, 0, 0, 0].item() & 0xffffffff
    assert plane0 == 0b00110, bin(plane0)  # slots 1 and 2 are low
    low = st.low_count.cpu().numpy().view(np.uint16)[0, 0]
    np.testing.assert_array_equal(low[:5], [0, 1, 1, 0, 0])
    assert st.t == 1
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


SH_SHAPES = {"g4": (2, 8, 2, 128, 512, 400, 32), "g16_d64": (1, 16, 1, 64, 256, 5, 16),
             # 64 (b, kvh) rows of 8192 slots: two CTAs per row of 4096 slots each, so the output
             # pass runs more iterations than it loads the history state for ahead of the stream
             "long": (8, 8, 8, 128, 8192, 400, 8)}


@pytest.mark.parametrize("policy,shape", [("bulk", "g4"), ("queue", "g4"), ("sparse", "g4"), ("bulk", "g16_d64"),
                                          ("queue", "g16_d64"), ("bulk", "long"), ("queue", "long")])
def test_scissorhands_full_update_teacher_forced(policy, shape):
    """Full decode steps through the library.  bulk: evict m every m steps; queue: once full,
    refill an eviction queue every m steps and replace one queued token per step; sparse:
    insert every step, score and record only every M-th step (bulk eviction).  g16_d64: 16
    query rows per KV head (both accumulator halves), 64-channel rows, a short history."""
    B, H, KVH, D, cap, hist, m = SH_SHAPES[shape]
    M = 3 if policy == "sparse" else 1
    wl = Workload("t", B=B, H=H, KVH=KVH, D=D, S=cap, w=1, k=cap, reduce="gqa", causal=False, seed=51)
    pre = prefill_inputs(wl)
    scale = 1.0 / np.sqrt(D)
    st = kvc.ScissorhandsState(B, KVH, cap, history=hist)
    kvc.kvc_scissorhands_init(st, cap - m)
    Kd, Vd = dev_bf16(pre["K"]), dev_bf16(pre["V"])
    ref = O.Scissorhands(B, KVH, cap, history=hist)
    ref.prefill(cap - m)
    Kr, Vr = pre["K"].copy(), pre["V"].copy()
    queue, rq, pos, refills = None, None, m, 0
    for step in range((3 if policy == "queue" else 2) * m):
        s = decode_step_inputs(wl, step)
        rep = None
        if policy == "queue" and ref.live.all():
            if pos == m:
                queue = kvc.kvc_scissorhands_refill_queue(st, m)
                rq = ref.refill_queue(m)
                np.testing.assert_array_equal(queue.cpu().numpy(), rq)
                pos, refills = 0, refills + 1
            rep, pos = pos, pos + 1
        qa = {} if rep is None else {"queue": queue, "pos": rep}
        record = step % M == 0
        if record:
            probs = kvc.kvc_scissorhands_update(st, dev_bf16(s["q"]), dev_bf16(s["k"]), dev_bf16(s["v"]), Kd, Vd,
                                                scale, **qa)
        else:
            kvc.kvc_scissorhands_insert(st, dev_bf16(s["k"]), dev_bf16(s["v"]), Kd, Vd, H, **qa)
        slot = ref.insert(replace=None if rep is None else rq[..., rep])
        np.testing.assert_array_equal(st.slot.cpu().numpy(), slot)
        Kr, Vr = O.write_slots(Kr, Vr, s["k"], s["v"], slot)
        if record:
            p_ref = O.scissorhands_probs(s["q"], Kr, scale, ref.live)
            gp = probs.cpu().numpy()
            assert_scores_close(gp, p_ref)
            # flags: identical except where p is within 1e-3/keys of the threshold
            keys = ref.live.sum(-1, keepdims=True)
            near = np.abs(p_ref - 1.0 / keys) <= 1e-3 / keys
            bits_ref = O.low_attention_bits(p_ref, ref.live)
            bits_gpu = O.low_attention_bits(gp, ref.live)
            assert np.all((bits_ref == bits_gpu) | near)
            ref.record(gp)  # teacher forcing on the GPU's probabilities: counts must then be exact
        assert st.t == ref.t
        live, low, ins = _sh_host(st)
        np.testing.assert_array_equal(live, ref.live)
        np.testing.assert_array_equal(np.where(live, low, 0), np.where(ref.live, ref.low, 0))
        np.testing.assert_array_equal(np.where(live, ins, 0), np.where(ref.live, ref.insert_step, 0))
        if policy != "queue" and (step + 1) % m == 0:
            ev = kvc.kvc_scissorhands_evict(st, m)
            np.testing.assert_array_equal(ev.cpu().numpy(), ref.evict(m))
    np.testing.assert_array_equal(host_bits(Kd), Kr)
    np.testing.assert_array_equal(host_bits(Vd), Vr)
    if policy == "queue":
        assert refills == 2 and st.n_free == 0
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


def test_scissorhands_resume_from_saved_state():
    """Checkpoint / resume: the state is plain caller-owned tensors plus two host counters, so
    copying them out and back in continues the run exactly (same flags, counts, evictions)."""
    B, KVH, cap, hist, m = 2, 2, 128, 7, 8
    g = np.random.Generator(np.random.PCG64([61]))
    probs = [g.random((B, KVH, cap)).astype(np.float32) * np.float32(2.0 / cap) for _ in range(24)]
    st = kvc.ScissorhandsState(B, KVH, cap, history=hist)
    kvc.kvc_scissorhands_init(st, cap)

    def run(state, steps):
        evs = []
        for i in steps:
            kvc.kvc_scissorhands_update_from_probs(state, torch.from_numpy(probs[i]).cuda())
            if (i + 1) % m == 0:
                evs.append(kvc.kvc_scissorhands_evict(state, m).cpu().numpy())
        return evs

    run(st, range(12))
    saved = {n: getattr(st, n).clone() for n in ("hist", "low_count", "insert_step", "live", "slot")}
    t, n_free = st.c.t, st.c.n_free
    ev_a = run(st, range(12, 24))
    after = {n: getattr(st, n).clone() for n in saved}
    st2 = kvc.ScissorhandsState(B, KVH, cap, history=hist)
    for n, v in saved.items():
        getattr(st2, n).copy_(v)
    st2.c.t, st2.c.n_free = t, n_free
    ev_b = run(st2, range(12, 24))
    assert len(ev_a) == len(ev_b) == 2
    for a, b in zip(ev_a, ev_b):
        np.testing.assert_array_equal(a, b)
    for n in saved:
        assert torch.equal(after[n], getattr(st2, n)), n
    assert (st.t, st.n_free) == (st2.t, st2.n_free)


def test_scissorhands_refill_queue_exact_with_ties():
    """Refills on states with many equal fractions (short history, few distinct counts):
    the queue lists the oracle's order exactly, -1 padded when fewer slots are live."""
    B, KVH, cap, hist = 2, 3, 320, 3
    st = kvc.ScissorhandsState(B, KVH, cap, history=hist)
    kvc.kvc_scissorhands_init(st, cap)
    ref = O.Scissorhands(B, KVH, cap, history=hist)
    ref.prefill(cap)
    g = np.random.Generator(np.random.PCG64([83]))
    for step in range(12):
        keys = ref.live.sum(-1, keepdims=True)
        p = np.where(ref.live, g.random((B, KVH, cap)) * 2.0 / keys, 0.0).astype(np.float32)
        kvc.kvc_scissorhands_update_from_probs(st, torch.from_numpy(p).cuda())
        ref.record(p)
        for m in (1, 7, 64, 300):
            np.testing.assert_array_equal(kvc.kvc_scissorhands_refill_queue(st, m).cpu().numpy(),
                                          ref.refill_queue(m))
        if step % 4 == 3:  # shrink the live set so that some queues need padding
            np.testing.assert_array_equal(kvc.kvc_scissorhands_evict(st, 100).cpu().numpy(), ref.evict(100))
    assert ref.live.sum(-1).min() < 300
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


# ----------------------------------------------------------------------------------------
# ThinK
# ----------------------------------------------------------------------------------------


@pytest.mark.parametrize("D,use_idx", [(128, False), (128, True), (64, True)])
def test_channel_score_parity(D, use_idx):
    B, H, KVH, S, w, k = 1, 32, 8, 3000, 64, 700
    wl = _wl(B, H, KVH, D, S, w, seed=61, channel_scales=True)
    inp = prefill_inputs(wl)
    idx = O.topk_select(random_scores((B, KVH, S), 62), k) if use_idx else None
    cs = kvc.kvc_channel_score(dev_bf16(inp["q"]), dev_bf16(inp["K"]), idx=None if idx is None else dev_i32(idx))
    ref = O.channel_score(inp["q"], inp["K"], kept=idx)
    assert_scores_close(cs.cpu().numpy(), ref)


@pytest.mark.parametrize("B,H,KVH,D,S,w,k,protect,reduce", [
    (1, 32, 8, 128, 3000, 64, 700, 64, "gqa"),    # several chunks per KV head, ragged last chunk
    (2, 8, 2, 64, 2500, 32, 1000, 32, "gqa"),
    (2, 16, 4, 128, 2049, 1, 512, 0, "all_heads"),
    (1, 4, 1, 64, 300, 16, 290, 16, "gqa"),      # fewer eligible tokens than k: -1 rows add nothing
])
def test_compress_prefill_channels_parity(B, H, KVH, D, S, w, k, protect, reduce):
    """The compaction that also sums the kept keys' squares: the same kept set and compacted
    rows as kvc_compress_prefill (bit for bit), and ThinK's channel scores of the kept keys
    against the oracle's closed form on the GPU's kept set."""
    wl = _wl(B, H, KVH, D, S, w, seed=S + k, channel_scales=True)
    inp = prefill_inputs(wl)
    q, K, V = dev_bf16(inp["q"]), dev_bf16(inp["K"]), dev_bf16(inp["V"])
    scale = 1.0 / np.sqrt(D)
    sc, idx, Ko, Vo = kvc.kvc_compress_prefill(q, K, V, scale, k, protect_tail=protect, reduce=reduce)
    sc2, idx2, Ko2, Vo2, cs = kvc.kvc_compress_prefill_channels(q, K, V, scale, k, protect_tail=protect, reduce=reduce)
    assert torch.equal(sc.view(torch.int32), sc2.view(torch.int32))
    assert torch.equal(idx, idx2)
    assert torch.equal(Ko, Ko2) and torch.equal(Vo, Vo2)
    g_idx = idx2.cpu().numpy()
    assert_scores_close(cs.cpu().numpy(), O.channel_score(inp["q"], inp["K"], kept=g_idx), what="channel score")
    # the separate call over the compacted keys agrees to fp32 rounding (other summation order)
    cs_sep = kvc.kvc_channel_score(q, Ko2).cpu().numpy()
    np.testing.assert_allclose(cs.cpu().numpy(), cs_sep, rtol=1e-5, atol=1e-6 * float(np.abs(cs_sep).max()))
    # scores not kept: room for them comes from the workspace
    none, idx3, Ko3, Vo3, cs3 = kvc.kvc_compress_prefill_channels(q, K, V, scale, k, protect_tail=protect, reduce=reduce,
                                                                  keep_scores=False)
    assert none is None and torch.equal(idx3, idx2) and torch.equal(Ko3, Ko2)
    assert torch.equal(cs3.view(torch.int32), cs.view(torch.int32))


@pytest.mark.parametrize("B,KVH,S,D,C", [
    (2, 4, 1000, 128, 64),    # one 64-row pass per CTA, ragged last pass
    (1, 8, 40000, 64, 32),    # several passes per CTA (the next pass's loads in flight), D = 64
    (2, 4, 20011, 128, 8),    # ~2 passes per CTA, ragged tail, few channels kept
    (1, 2, 777, 128, 120),    # nearly all channels kept
])
@pytest.mark.parametrize("zero_mode", [False, True])
def test_channel_prune_parity(zero_mode, B, KVH, S, D, C):
    cs = random_scores((B, KVH, D), 71 + S, tie_levels=40).astype(np.float32)
    K = normal_bf16((B, KVH, S, D), 72 + S, 1)
    ch, Ko = kvc.kvc_channel_prune(torch.from_numpy(cs).cuda(), dev_bf16(K), C, zero_mode=zero_mode)
    r_ch, r_K = O.channel_prune(cs, K, C, zero_mode=zero_mode)
    np.testing.assert_array_equal(ch.cpu().numpy(), r_ch)
    np.testing.assert_array_equal(host_bits(Ko), r_K)


def test_channel_prune_in_place_zero():
    B, KVH, S, D, C = 1, 2, 300, 64, 20
    cs = random_scores((B, KVH, D), 73).astype(np.float32)
    K = normal_bf16((B, KVH, S, D), 74, 1)
    Kd = dev_bf16(K)
    kvc.kvc_channel_prune(torch.from_numpy(cs).cuda(), Kd, C, zero_mode=True, K_out=Kd)
    np.testing.assert_array_equal(host_bits(Kd), O.channel_prune(cs, K, C, zero_mode=True)[1])


# ----------------------------------------------------------------------------------------
# host validation through the ABI on a live device
# ----------------------------------------------------------------------------------------


VALUE_SCORE_CASES = [
    # B, H, KVH, D, kept tokens, w: the three scoring paths (G*w = 256, 16, 512)
    (1, 32, 8, 128, 2000, 64),
    (2, 8, 2, 64, 333, 4),
    (1, 8, 1, 128, 700, 64),
    (1, 32, 8, 128, 8192, 64),  # the ThinK 128K layer's compressed cache (the bench's launch shape)
]


@pytest.mark.parametrize("B,H,KVH,D,k,w", VALUE_SCORE_CASES)
def test_value_channel_score_parity(B, H, KVH, D, k, w):
    seed = k + w
    q = normal_bf16((B, H, w, D), seed, 1)
    Kc = normal_bf16((B, KVH, k, D), seed, 2)
    Vc = normal_bf16((B, KVH, k, D), seed, 3)
    scale = 1.0 / np.sqrt(D)
    got = kvc.kvc_value_channel_score(dev_bf16(q), dev_bf16(Kc), dev_bf16(Vc), scale).cpu().numpy()
    assert_scores_close(got, O.value_channel_score(q, Kc, Vc, scale), what="value channel score")
    # the same scoring kernels with p (not p^2) still give the window scores
    sc = kvc.kvc_window_scores(dev_bf16(q), dev_bf16(Kc), scale, causal=True, reduce="gqa").cpu().numpy()
    assert_scores_close(sc, O.window_scores(q, Kc, scale, causal=True, reduce="gqa"))


# ----------------------------------------------------------------------------------------
# Decoding over the channel-pruned cache (ThinK options 3b / 3c)
# ----------------------------------------------------------------------------------------


def _assert_attention_close(got, ref, V):
    """fp32 attention outputs against the float64 oracle: |g - r| <= 1e-3 |r| + 1e-4 max|V|
    (outputs are convex combinations of value rows; the absolute term covers cancellation)."""
    vmax = float(np.abs(O.as_f64(V)).max())
    assert_scores_close(got, ref, rtol=1e-3, atol=1e-4 * vmax, what="attention")


DECODE_CASES = [
    # B, H, KVH, D, C (kept key channels; C == D: plain attention), S, live fraction
    (2, 32, 8, 128, 128, 1000, None),   # ragged last tile
    (2, 32, 8, 128, 64, 3000, None),    # option 3c: pruned query against pruned keys
    (1, 4, 4, 64, 64, 777, 0.6),        # one head per KV head, dead slots
    (1, 16, 2, 128, 128, 500, None),    # 8 heads per KV head: two head groups per range
    (1, 6, 2, 128, 64, 129, 0.9),       # 3 heads per KV head (padded group)
    (3, 8, 4, 64, 64, 5, None),         # a single partial tile
    (1, 8, 2, 128, 64, 64, None),       # exactly one tile
    (1, 8, 2, 128, 64, 40000, 0.5),     # many key ranges
    (16, 32, 8, 128, 64, 4096, None),   # 128 (b, kvh) rows
    (16, 32, 8, 128, 128, 4100, 0.5),   # 128 rows, ragged, dead slots
    (2, 32, 8, 128, 64, 40000, 0.5),    # 16 rows over all SMs: up to 11 pieces per row
]


@pytest.mark.parametrize("B,H,KVH,D,C,S,p_live", DECODE_CASES)
def test_decode_attention_parity(B, H, KVH, D, C, S, p_live):
    seed = B * 1000 + S
    q = normal_bf16((B, H, D), seed, 1)
    K = normal_bf16((B, KVH, S, D), seed, 2)
    V = normal_bf16((B, KVH, S, D), seed, 3)
    scale = 1.0 / np.sqrt(D)
    live = None
    if p_live is not None:
        live = random_live_mask((B, KVH, S), seed, p_live)
        live[0, 0, :] = False  # a KV head with no live slot: zeros
    if C < D:
        cs = random_scores((B, KVH, D), seed + 1)
        ch, Kp = O.channel_prune(cs, K, C)
        ref = O.decode_attention_pruned(q, ch, Kp, V, scale, live)
        got = kvc.kvc_decode_attention(dev_bf16(q), dev_bf16(Kp), dev_bf16(V), scale, ch=dev_i32(ch),
                                       live_mask=None if live is None else dev_u32(pack_live_bits(live)))
    else:
        ref = O.decode_attention(q, K, V, scale, live)
        got = kvc.kvc_decode_attention(dev_bf16(q), dev_bf16(K), dev_bf16(V), scale,
                                       live_mask=None if live is None else dev_u32(pack_live_bits(live)))
    _assert_attention_close(got.cpu().numpy(), ref, V)
    if live is not None:
        assert np.all(got[0, :H // KVH].cpu().numpy() == 0)
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


def test_zero_add_back_bit_exact_and_3b_equals_3c():
    B, H, KVH, D, C, S = 2, 16, 4, 128, 64, 700
    q = normal_bf16((B, H, D), 95, 1)
    K = normal_bf16((B, KVH, S, D), 95, 2)
    V = normal_bf16((B, KVH, S, D), 95, 3)
    cs = O.channel_score(normal_bf16((B, H, 8, D), 95, 4), K)
    ch, Kp = O.channel_prune(cs, K, C)
    Kz = kvc.kvc_zero_add_back(dev_bf16(Kp), dev_i32(ch), D)
    np.testing.assert_array_equal(host_bits(Kz), O.zero_add_back(Kp, ch, D))
    scale = 1.0 / np.sqrt(D)
    o3b = kvc.kvc_decode_attention(dev_bf16(q), Kz, dev_bf16(V), scale).cpu().numpy()
    o3c = kvc.kvc_decode_attention(dev_bf16(q), dev_bf16(Kp), dev_bf16(V), scale, ch=dev_i32(ch)).cpu().numpy()
    ref = O.decode_attention_pruned(q, ch, Kp, V, scale)
    _assert_attention_close(o3b, ref, V)
    _assert_attention_close(o3c, ref, V)


def test_decode_attention_bad_channel_reports_bounds():
    B, H, KVH, D, C, S = 1, 4, 2, 128, 64, 100
    q = dev_bf16(normal_bf16((B, H, D), 96, 1))
    Kp = dev_bf16(normal_bf16((B, KVH, S, C), 96, 2))
    V = dev_bf16(normal_bf16((B, KVH, S, D), 96, 3))
    ch = np.tile(np.arange(C, dtype=np.int32), (B, KVH, 1))
    ch[0, 1, 5] = 500  # outside [0, D): counted as a zero query channel, reported
    kvc.kvc_decode_attention(q, Kp, V, 0.1, ch=dev_i32(ch))
    assert kvc.kvc_get_device_status() == kvc.KVC_ERR_DEVICE_BOUNDS
    assert kvc.kvc_get_device_status() == kvc.KVC_OK  # read-and-clear


def test_invalid_arguments_raise_and_enqueue_nothing():
    K = dev_bf16(normal_bf16((1, 2, 64, 64), 1, 1))
    q = dev_bf16(normal_bf16((1, 6, 1, 64), 1, 2))  # H=6 not a multiple of... 6 % 2 == 0 -> ok
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_window_scores(q, K, 0.1, reduce="gqa", ws=torch.empty(1, dtype=torch.uint8, device="cuda"))
    assert e.value.status == kvc.KVC_ERR_WORKSPACE
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_topk_select(torch.zeros((1, 2, 64), device="cuda"), 4, protect_tail=8)
    assert e.value.status == kvc.KVC_ERR_INVALID_ARG
    with pytest.raises(kvc.KvcError):
        # V_out is a dense view into V's own storage: the library refuses the overlap
        kvc.kvc_compact_kv(K, K, dev_i32(np.zeros((1, 2, 4))), K_out=K[:, :, :4].contiguous(),
                           V_out=K.view(-1)[:512].view(1, 2, 4, 64))
    with pytest.raises(ValueError):
        kvc.kvc_compact_kv(K, K, dev_i32(np.zeros((1, 2, 4))), K_out=K[:, :, :4])  # not dense
    assert kvc.kvc_get_device_status() == kvc.KVC_OK
