"""Pins of the CPU oracle to facts the pages and the mathematics fix (no GPU needed).

Every check here is independent of the oracle's own code: closed forms, invariants,
brute-force loops written separately in this file, or sizes printed on the pages.
"""
import copy
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from synth import f32_to_bf16_bits, bf16_bits_to_f32, normal_bf16, random_scores

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


# ----------------------------------------------------------------------------------------
# window softmax / scores
# ----------------------------------------------------------------------------------------


def _full_causal_attention_loops(Qf, Kf, scale):
    """Independent brute force: the full S x S causal softmax of one head, pure Python."""
    S = len(Qf)
    P = [[0.0] * S for _ in range(S)]
    for i in range(S):
        logits = [scale * sum(Qf[i][d] * Kf[j][d] for d in range(len(Qf[i]))) for j in range(i + 1)]
        mx = max(logits)
        ex = [math.exp(x - mx) for x in logits]
        tot = sum(ex)
        for j in range(i + 1):
            P[i][j] = ex[j] / tot
    return P


@pytest.mark.parametrize("w", [1, 3, 12])
def test_window_rows_are_last_rows_of_full_causal_matrix(w):
    """'Add TOVA press': attn_weights = full_attn_weights[:, :, -window_size:, :]."""
    B, H, KVH, D, S = 1, 4, 2, 8, 12
    G = H // KVH
    Qfull = bf16_bits_to_f32(normal_bf16((B, H, S, D), 11, 1)).astype(np.float64)
    K = normal_bf16((B, KVH, S, D), 11, 2)
    Kf = bf16_bits_to_f32(K).astype(np.float64)
    scale = 1 / math.sqrt(D)
    q_win = f32_to_bf16_bits(Qfull[:, :, S - w:, :].astype(np.float32))
    p = O.window_softmax(q_win, K, scale, causal=True)
    for h in range(H):
        P = _full_causal_attention_loops(Qfull[0, h].tolist(), Kf[0, h // G].tolist(), scale)
        for i in range(w):
            np.testing.assert_allclose(p[0, h, i], P[S - w + i], rtol=1e-12, atol=1e-15)


def test_tova_score_is_head_mean_of_last_row():
    """'Add TOVA press' (hassidm): torch.mean(attn_weights[:,:,-1:,:], dim=1), repeated
    over KV heads."""
    B, H, KVH, D, S = 1, 8, 2, 8, 10
    G = H // KVH
    Qfull = bf16_bits_to_f32(normal_bf16((B, H, S, D), 12, 1)).astype(np.float64)
    K = normal_bf16((B, KVH, S, D), 12, 2)
    Kf = bf16_bits_to_f32(K).astype(np.float64)
    scale = 1 / math.sqrt(D)
    q_win = f32_to_bf16_bits(Qfull[:, :, S - 1:, :].astype(np.float32))
    sc = O.window_scores(q_win, K, scale, causal=True, reduce="all_heads")
    assert sc.shape == (B, KVH, S)
    last = np.zeros(S)
    for h in range(H):
        last += np.array(_full_causal_attention_loops(Qfull[0, h].tolist(), Kf[0, h // G].tolist(), scale)[S - 1])
    last /= H
    for kv in range(KVH):
        np.testing.assert_allclose(sc[0, kv], last, rtol=1e-12, atol=1e-15)


def test_closed_form_logits_three_keys():
    """One head, q = e_0, keys with first coordinate 0, 1, 2 and scale 1: p_j = e^j / (1 + e + e^2)."""
    q = np.zeros((1, 1, 1, 4), np.float32)
    q[..., 0] = 1.0
    K = np.zeros((1, 1, 3, 4), np.float32)
    K[0, 0, :, 0] = [0.0, 1.0, 2.0]
    p = O.window_softmax(_bf16(q), _bf16(K), 1.0, causal=False)
    z = 1 + math.e + math.e ** 2
    np.testing.assert_allclose(p[0, 0, 0], [1 / z, math.e / z, math.e ** 2 / z], rtol=1e-14)


def test_rows_sum_to_one_and_scores_sum_to_w():
    B, H, KVH, D, S, w = 2, 8, 2, 16, 40, 5
    q = normal_bf16((B, H, w, D), 13, 1)
    K = normal_bf16((B, KVH, S, D), 13, 2)
    p = O.window_softmax(q, K, 0.25)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-13)
    for red in ("gqa", "all_heads"):
        sc = O.window_scores(q, K, 0.25, reduce=red)
        np.testing.assert_allclose(sc.sum(-1), w, rtol=1e-13)
    # all-heads = mean over KV heads of the per-group result
    g = O.window_scores(q, K, 0.25, reduce="gqa")
    a = O.window_scores(q, K, 0.25, reduce="all_heads")
    np.testing.assert_allclose(a[:, 0], g.mean(axis=1), rtol=1e-13)


def test_causal_mask_in_window():
    """Window row i (absolute position S-w+i) gives zero probability to later keys."""
    B, H, KVH, D, S, w = 1, 2, 1, 8, 9, 4
    p = O.window_softmax(normal_bf16((B, H, w, D), 14, 1), normal_bf16((B, KVH, S, D), 14, 2), 0.3)
    for i in range(w):
        assert np.all(p[0, :, i, S - w + i + 1:] == 0)
        assert np.all(p[0, :, i, :S - w + i + 1] > 0)


def test_uniform_attention_gives_one_over_keys():
    B, H, KVH, D, S = 1, 4, 2, 8, 37
    q = np.zeros((B, H, 1, D), np.uint16)
    sc = O.window_scores(q, normal_bf16((B, KVH, S, D), 15, 2), 0.3, causal=False, reduce="all_heads")
    np.testing.assert_allclose(sc, 1.0 / S, rtol=1e-15)


def test_live_mask_excludes_dead_slots_and_empty_rows_are_zero():
    B, H, KVH, D, S = 1, 4, 2, 8, 20
    q = normal_bf16((B, H, 1, D), 16, 1)
    K = normal_bf16((B, KVH, S, D), 16, 2)
    live = np.ones((B, KVH, S), bool)
    live[0, 0, ::3] = False
    live[0, 1, :] = False
    sc = O.window_scores(q, K, 0.3, causal=False, live=live, reduce="gqa")
    assert np.all(sc[0, 0, ::3] == 0)
    np.testing.assert_allclose(sc[0, 0].sum(), 1.0, rtol=1e-13)
    assert np.all(sc[0, 1] == 0)
    # a dead slot's key has no effect on the others
    K2 = K.copy()
    K2[0, 0, 0] = normal_bf16((D,), 99, 9)
    sc2 = O.window_scores(q, K2, 0.3, causal=False, live=live, reduce="gqa")
    np.testing.assert_array_equal(sc, sc2)


# ----------------------------------------------------------------------------------------
# selection
# ----------------------------------------------------------------------------------------


def _topk_brute(row, k, protect, live, largest):
    S = len(row)
    idx = [j for j in range(S) if live is None or live[j]]
    forced = [j for j in idx if protect and j >= S - protect]
    cand = [j for j in idx if not (protect and j >= S - protect)]
    if largest:
        cand.sort(key=lambda j: (-float(row[j]), j))
    else:
        cand.sort(key=lambda j: (float(row[j]), -j))
    keep = sorted(forced[:k] + cand[:max(0, k - len(forced))])
    return keep + [-1] * (k - len(keep))


@pytest.mark.parametrize("S,k,protect,ties,largest,use_live", [
    (50, 10, 0, 0, True, False), (50, 10, 0, 3, True, False), (64, 20, 8, 4, True, False),
    (33, 33, 0, 0, True, False), (10, 16, 0, 0, True, False), (40, 1, 0, 2, False, False),
    (40, 5, 0, 0, False, True), (40, 30, 0, 2, True, True), (7, 7, 7, 0, True, False),
])
def test_topk_matches_brute_force_sort(S, k, protect, ties, largest, use_live):
    sc = random_scores((2, 3, S), 17 + S + k, tie_levels=ties)
    live = (random_scores((2, 3, S), 5) < 0.6) if use_live else None
    got = O.topk_select(sc, k, protect_tail=protect, live=live, largest=largest)
    for b in range(2):
        for kv in range(3):
            exp = _topk_brute(sc[b, kv], k, protect, None if live is None else live[b, kv], largest)
            assert got[b, kv].tolist() == exp


def test_snapkv_keeps_the_window():
    """cold-compress PR 11: SnapKV keeps every token in the observation window."""
    S, w, k = 100, 16, 30
    sc = random_scores((1, 2, S), 18)
    sc[..., S - w:] = 0.0  # even the lowest-scoring window tokens are kept
    idx = O.topk_select(sc, k, protect_tail=w)
    for kv in range(2):
        assert set(range(S - w, S)) <= set(idx[0, kv].tolist())
        assert np.all(np.diff(idx[0, kv]) > 0)


def test_compact_is_a_row_gather():
    K = normal_bf16((1, 2, 9, 4), 19, 1)
    V = normal_bf16((1, 2, 9, 4), 19, 2)
    idx = np.array([[[0, 3, 8, -1], [1, 2, 5, 6]]], np.int32)
    Kc, Vc = O.compact_kv(K, V, idx)
    np.testing.assert_array_equal(Kc[0, 0, 1], K[0, 0, 3])
    np.testing.assert_array_equal(Vc[0, 1, 3], V[0, 1, 6])
    assert np.all(Kc[0, 0, 3] == 0)


def test_write_slots_replaces_one_row_per_head():
    B, KVH, S, D = 2, 3, 9, 4
    K = normal_bf16((B, KVH, S, D), 23, 1)
    V = normal_bf16((B, KVH, S, D), 23, 2)
    kn = normal_bf16((B, KVH, D), 23, 3)
    vn = normal_bf16((B, KVH, D), 23, 4)
    slot = np.array([[0, 8, 4], [3, 3, 7]], np.int32)
    K2, V2 = O.write_slots(K, V, kn, vn, slot)
    for b in range(B):
        for kv in range(KVH):
            for j in range(S):
                want_k = kn[b, kv] if j == slot[b, kv] else K[b, kv, j]
                want_v = vn[b, kv] if j == slot[b, kv] else V[b, kv, j]
                assert K2[b, kv, j].tolist() == want_k.tolist() and V2[b, kv, j].tolist() == want_v.tolist()
    np.testing.assert_array_equal(K, normal_bf16((B, KVH, S, D), 23, 1))  # inputs are not modified in place


# ----------------------------------------------------------------------------------------
# ThinK
# ----------------------------------------------------------------------------------------


def test_think_closed_form_equals_bruteforce():
    """'Add ThinK_Press': sum_{i,j}(q_id k_jd)^2 = (sum_i q_id^2)(sum_j k_jd^2)."""
    B, H, KVH, D, S, w = 2, 8, 2, 16, 30, 6
    q = normal_bf16((B, H, w, D), 20, 1)
    K = normal_bf16((B, KVH, S, D), 20, 2)
    a = O.channel_score(q, K)
    b = O.channel_score_bruteforce(q, K)
    np.testing.assert_allclose(a, b, rtol=1e-12)
    kept = O.topk_select(random_scores((B, KVH, S), 3), 11)
    np.testing.assert_allclose(O.channel_score(q, K, kept), O.channel_score_bruteforce(q, K, kept), rtol=1e-12)


def test_think_score_by_loops():
    """Direct loop over the definition for one channel (no vectorisation)."""
    q = bf16_bits_to_f32(normal_bf16((1, 2, 3, 4), 21, 1)).astype(np.float64)
    K = bf16_bits_to_f32(normal_bf16((1, 1, 5, 4), 21, 2)).astype(np.float64)
    cs = O.channel_score(f32_to_bf16_bits(q.astype(np.float32)), f32_to_bf16_bits(K.astype(np.float32)))
    for d in range(4):
        tot = 0.0
        for h in range(2):
            for i in range(3):
                for j in range(5):
                    tot += (q[0, h, i, d] * K[0, 0, j, d]) ** 2
        assert abs(cs[0, 0, d] - tot / 2) <= 1e-12 * tot


def test_think_prune_compact_and_zero():
    cs = random_scores((1, 2, 16), 22, tie_levels=5).astype(np.float64)
    K = normal_bf16((1, 2, 7, 16), 22, 2)
    ch, Kp = O.channel_prune(cs, K, 8)
    ch0, Kz = O.channel_prune(cs, K, 8, zero_mode=True)
    np.testing.assert_array_equal(ch, ch0)
    for kv in range(2):
        exp = sorted(sorted(range(16), key=lambda d: (-cs[0, kv, d], d))[:8])
        assert ch[0, kv].tolist() == exp
        np.testing.assert_array_equal(Kp[0, kv], K[0, kv][:, exp])
        rest = [d for d in range(16) if d not in exp]
        assert np.all(Kz[0, kv][:, rest] == 0)
        np.testing.assert_array_equal(Kz[0, kv][:, exp], K[0, kv][:, exp])


def test_value_channel_score_by_loops():
    """The value score against a pure-Python sum over (head, window row, token) with its own
    causal softmax over the compressed cache."""
    B, H, KVH, w, k, D = 1, 4, 2, 3, 6, 4
    q = bf16_bits_to_f32(normal_bf16((B, H, w, D), 97, 1)).astype(np.float64)
    Kc = bf16_bits_to_f32(normal_bf16((B, KVH, k, D), 97, 2)).astype(np.float64)
    Vc = bf16_bits_to_f32(normal_bf16((B, KVH, k, D), 97, 3)).astype(np.float64)
    scale, G = 0.5, H // KVH
    exp = np.zeros((B, KVH, D))
    for kv in range(KVH):
        for h in range(kv * G, (kv + 1) * G):
            for i in range(w):
                vis = list(range(k - w + i + 1))  # window row i sits at index k - w + i
                lg = [scale * sum(q[0, h, i, d] * Kc[0, kv, j, d] for d in range(D)) for j in vis]
                mx = max(lg)
                ex = [math.exp(x - mx) for x in lg]
                tot = sum(ex)
                for n, j in enumerate(vis):
                    for d in range(D):
                        exp[0, kv, d] += (ex[n] / tot * Vc[0, kv, j, d]) ** 2 / G
    got = O.value_channel_score(_bf16(q), _bf16(Kc), _bf16(Vc), scale)
    np.testing.assert_allclose(got, exp, rtol=1e-12)


def test_value_channel_score_factorises_and_uniform_case():
    """sum_i sum_j (p_ij v_jd)^2 = sum_j (sum_i p_ij^2) v_jd^2; with a zero query every
    visible token gets 1/n_i, so the weights have a closed form."""
    B, H, KVH, w, k, D = 2, 8, 2, 5, 40, 16
    q = normal_bf16((B, H, w, D), 98, 1)
    Kc = normal_bf16((B, KVH, k, D), 98, 2)
    Vc = normal_bf16((B, KVH, k, D), 98, 3)
    G = H // KVH
    p = O.window_softmax(q, Kc, 0.3)
    wj = np.stack([(p[:, kv * G:(kv + 1) * G] ** 2).sum(axis=(1, 2)) / G for kv in range(KVH)], axis=1)
    V2 = bf16_bits_to_f32(Vc).astype(np.float64) ** 2
    np.testing.assert_allclose(O.value_channel_score(q, Kc, Vc, 0.3), np.einsum("bkj,bkjd->bkd", wj, V2),
                               rtol=1e-12)
    # zero query: row i sees n_i = k - w + i + 1 tokens, each with p = 1/n_i
    w0 = np.zeros(k)
    for i in range(w):
        n = k - w + i + 1
        w0[:n] += 1.0 / n ** 2
    np.testing.assert_allclose(O.value_channel_score(np.zeros_like(q), Kc, Vc, 0.3),
                               np.einsum("j,bkjd->bkd", w0, V2), rtol=1e-12)


def _decode_attention_loops(q, K, V, scale, live=None):
    """Independent brute force: one new query per head, pure Python loops."""
    B, H, D = len(q), len(q[0]), len(q[0][0])
    KVH, S, Dv = len(K[0]), len(K[0][0]), len(V[0][0][0])
    G = H // KVH
    out = [[[0.0] * Dv for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            kv = h // G
            js = [j for j in range(S) if live is None or live[b][kv][j]]
            if not js:
                continue
            lg = [scale * sum(q[b][h][d] * K[b][kv][j][d] for d in range(D)) for j in js]
            mx = max(lg)
            ex = [math.exp(x - mx) for x in lg]
            tot = sum(ex)
            for n, j in enumerate(js):
                for d in range(Dv):
                    out[b][h][d] += ex[n] / tot * V[b][kv][j][d]
    return out


def test_decode_attention_by_loops():
    B, H, KVH, D, S = 2, 4, 2, 6, 7
    q = bf16_bits_to_f32(normal_bf16((B, H, D), 90, 1)).astype(np.float64)
    K = bf16_bits_to_f32(normal_bf16((B, KVH, S, D), 90, 2)).astype(np.float64)
    V = bf16_bits_to_f32(normal_bf16((B, KVH, S, D), 90, 3)).astype(np.float64)
    live = np.random.Generator(np.random.PCG64([90])).random((B, KVH, S)) < 0.6
    live[1, 1] = False  # a head group with no live slot attends nothing
    for lv in (None, live):
        got = O.decode_attention(_bf16(q), _bf16(K), _bf16(V), 0.4, lv)
        exp = _decode_attention_loops(q.tolist(), K.tolist(), V.tolist(), 0.4, None if lv is None else lv.tolist())
        np.testing.assert_allclose(got, np.array(exp), rtol=1e-12, atol=1e-14)
    assert np.all(O.decode_attention(_bf16(q), _bf16(K), _bf16(V), 0.4, live)[1, 2:] == 0)


def test_decode_attention_closed_forms():
    B, H, KVH, D, S = 1, 4, 2, 8, 9
    K = normal_bf16((B, KVH, S, D), 91, 2)
    V = normal_bf16((B, KVH, S, D), 91, 3)
    Vf = bf16_bits_to_f32(V).astype(np.float64)
    # a zero query attends uniformly: the mean of the value rows
    out = O.decode_attention(np.zeros((B, H, D), np.uint16), K, V, 0.3)
    np.testing.assert_allclose(out[0, 0], Vf[0, 0].mean(0), rtol=1e-13)
    np.testing.assert_allclose(out[0, 3], Vf[0, 1].mean(0), rtol=1e-13)
    # one key aligned with a large query takes all the weight
    Kd = np.zeros((B, KVH, S, D), np.float32)
    Kd[:, :, 4, 0] = 1.0
    q = np.zeros((B, H, D), np.float32)
    q[..., 0] = 64.0
    out = O.decode_attention(_bf16(q), _bf16(Kd), V, 1.0)
    np.testing.assert_allclose(out[0, 1], Vf[0, 0, 4], rtol=1e-12)
    np.testing.assert_allclose(out[0, 2], Vf[0, 1, 4], rtol=1e-12)


def test_pruned_query_equals_zero_filled_keys():
    """Options 3b and 3c give the attention of option 3a: pruning the query to the kept
    channels (3c) equals attending the zero-filled keys (3b = 3a's cache)."""
    B, H, KVH, D, S, C = 2, 8, 2, 16, 11, 8
    q = normal_bf16((B, H, D), 92, 1)
    K = normal_bf16((B, KVH, S, D), 92, 2)
    V = normal_bf16((B, KVH, S, D), 92, 3)
    cs = O.channel_score(normal_bf16((B, H, 4, D), 92, 4), K)
    ch, Kp = O.channel_prune(cs, K, C)
    _, Kz = O.channel_prune(cs, K, C, zero_mode=True)
    np.testing.assert_array_equal(O.zero_add_back(Kp, ch, D), Kz)
    live = np.random.Generator(np.random.PCG64([92])).random((B, KVH, S)) < 0.7
    for lv in (None, live):
        np.testing.assert_allclose(O.decode_attention_pruned(q, ch, Kp, V, 0.25, lv),
                                   O.decode_attention(q, Kz, V, 0.25, lv), rtol=1e-12, atol=1e-15)
    # keeping every channel is plain attention
    full = np.broadcast_to(np.arange(D, dtype=np.int32), (B, KVH, D))
    np.testing.assert_array_equal(O.decode_attention_pruned(q, full, K, V, 0.25), O.decode_attention(q, K, V, 0.25))


def test_page_shapes_and_memory_ratio():
    g = json.load(open(os.path.join(GOLDEN, "page_shapes.json")))
    # TOVA walk-through: scores [batch, num_kv_heads, seq_len]
    B, H, KVH, D, S = 2, 8, 4, 8, 6
    sc = O.window_scores(normal_bf16((B, H, 1, D), 23, 1), normal_bf16((B, KVH, S, D), 23, 2), 0.3,
                         reduce="all_heads")
    assert len(g["tova_walkthrough"]["scores_after_repeat"]) == sc.ndim and sc.shape == (B, KVH, S)
    assert np.all(sc == sc[:, :1])
    # ThinK: channel_attn per head is [head_dim, window, seq]; 32 heads of it vs a 32-layer,
    # 8-KV-head key cache is 8x larger
    r = g["think_memory_ratio"]
    head_dim, seq = 128, 1000
    channel_attn = r["num_heads"] * head_dim * r["window_size"] * seq
    key_cache = r["num_layers"] * r["num_key_value_heads"] * head_dim * seq
    assert channel_attn // key_cache == r["ratio"]
    cs = O.channel_score(normal_bf16((1, 4, 3, 8), 24, 1), normal_bf16((1, 2, 5, 8), 24, 2))
    assert cs.shape == (1, 2, 8)  # (bsz, kv heads, head_dim)


# ----------------------------------------------------------------------------------------
# Scissorhands
# ----------------------------------------------------------------------------------------


def test_low_flag_threshold_is_strict_float32():
    """cold-compress PR 11: attn_is_low = attn < 1/keys (strict; below uniform)."""
    keys = 3
    thr = np.float32(1) / np.float32(keys)
    live = np.ones((1, 1, keys), bool)
    p = np.array([[[thr, np.nextafter(thr, np.float32(0)), np.nextafter(thr, np.float32(1))]]], np.float32)
    assert O.low_attention_bits(p, live).tolist() == [[[False, True, False]]]


def test_low_flag_threshold_counts_live_keys_not_capacity():
    """cold-compress PR 11, review of ``cache.py``: ``keys = attn.shape[1]`` is the width of
    the attention row, and the step's flags are written to ``attn_history[:, :, :keys, ...]``,
    the slots the query attended.  Uniform attention over those keys is 1/keys, so with
    5 live slots out of 32 the threshold is float32(1/5), not 1/32.  Expected flags written
    out by hand: exactly 1/5 is not low; one ulp below 1/5 is low although it is 6x above
    1/32; dead slots are never flagged whatever their probability."""
    cap = 32
    live = np.zeros((1, 1, cap), bool)
    live[0, 0, [1, 4, 9, 20, 31]] = True
    fifth = np.float32(1) / np.float32(5)
    p = np.zeros((1, 1, cap), np.float32)
    p[0, 0, 1] = fifth                                   # uniform: not low
    p[0, 0, 4] = np.nextafter(fifth, np.float32(0))     # below uniform, far above 1/cap: low
    p[0, 0, 9] = np.float32(0.0625)                      # 1/16 < 1/5: low
    p[0, 0, 20] = np.nextafter(fifth, np.float32(1))    # above uniform: not low
    p[0, 0, 31] = np.float32(0.5)                        # not low
    p[0, 0, 0] = np.float32(0.0)                         # dead slots: never low
    p[0, 0, 2] = np.float32(1e-9)
    expected = np.zeros((1, 1, cap), bool)
    expected[0, 0, 4] = True
    expected[0, 0, 9] = True
    np.testing.assert_array_equal(O.low_attention_bits(p, live), expected)


def test_uniform_attention_sets_no_flag_and_dominant_key_flags_the_rest():
    B, H, KVH, D, cap = 1, 4, 2, 8, 64
    live = np.zeros((B, KVH, cap), bool)
    live[..., :37] = True
    K = normal_bf16((B, KVH, cap, D), 25, 2)
    p0 = O.scissorhands_probs(np.zeros((B, H, D), np.uint16), K, 0.3, live)
    assert not O.low_attention_bits(p0, live).any()
    # one key aligned with a large query dominates every head
    Kd = bf16_bits_to_f32(K).copy()
    Kd[:, :, 5] = 8.0
    q = np.full((B, H, D), 8.0, np.float32)
    p1 = O.scissorhands_probs(_bf16(q), _bf16(Kd), 1.0, live)
    bits = O.low_attention_bits(p1, live)
    assert not bits[:, :, 5].any()
    exp = live.copy()
    exp[:, :, 5] = False
    np.testing.assert_array_equal(bits, exp)


class _FullLog:
    """Independent brute force: keep every step's flags and the slot's occupant, count over
    the last min(400, age) observations of the current occupant, evict by exact Fractions."""

    def __init__(self, shape, history):
        self.history = history
        self.log = []  # list of (bits, occupant id) per step
        self.occ = np.full(shape, -1, np.int64)
        self.born = np.zeros(shape, np.int64)
        self.next_id = 0
        self.t = 0

    def insert_at(self, mask):
        n = int(mask.sum())
        self.occ[mask] = np.arange(self.next_id, self.next_id + n)
        self.born[mask] = self.t
        self.next_id += n

    def record(self, bits):
        self.log.append((bits.copy(), self.occ.copy()))
        self.t += 1

    def counts(self):
        c = np.zeros(self.occ.shape, np.int64)
        for s in range(max(0, self.t - self.history), self.t):
            bits, occ = self.log[s]
            c += bits & (occ == self.occ) & (self.occ >= 0)
        return c

    def nobs(self):
        return np.minimum(self.history, self.t - self.born)

    def queue_order(self, b, kv, live, m):
        """The m most evictable live slots, most evictable first.  A token with no
        observation yet (sparse recording) has no low flag: fraction 0."""
        c, n = self.counts(), self.nobs()
        cand = [s for s in range(live.shape[-1]) if live[b, kv, s]]
        cand.sort(key=lambda s: (-Fraction(int(c[b, kv, s]), max(1, int(n[b, kv, s]))), s))
        return cand[:m]

    def evict_order(self, b, kv, live, m):
        return sorted(self.queue_order(b, kv, live, m))


def test_circular_history_matches_full_log_and_exact_eviction():
    B, KVH, cap, hist, m = 2, 2, 32, 7, 4
    sh = O.Scissorhands(B, KVH, cap, history=hist)
    sh.prefill(cap - m)
    ref = _FullLog((B, KVH, cap), hist)
    ref.insert_at(sh.live.copy())
    g = np.random.Generator(np.random.PCG64([26]))
    for step in range(60):
        before = sh.live.copy()
        sh.insert()
        ref.insert_at(sh.live & ~before)
        keys = sh.live.sum(-1, keepdims=True)
        p = np.where(sh.live, g.random((B, KVH, cap)) * 2.0 / keys, 0.0)
        ref.record(O.low_attention_bits(p, sh.live))
        sh.record(p)
        np.testing.assert_array_equal(np.where(sh.live, sh.low, 0), np.where(sh.live, ref.counts(), 0))
        np.testing.assert_array_equal(np.where(sh.live, sh.n_obs(), 0), np.where(sh.live, ref.nobs(), 0))
        if (step + 1) % m == 0:
            live_before = sh.live.copy()
            exp = [[ref.evict_order(b, kv, live_before, m) for kv in range(KVH)] for b in range(B)]
            ev = sh.evict(m)
            assert ev.tolist() == exp
            ref.occ[~sh.live] = -1


def test_eviction_queue_matches_full_log():
    """Queue variant: once the cache is full, every m steps the queue is refilled with the
    m most evictable tokens (most evictable first), and each step's new token replaces the
    next queued one.  The queue holds the same tokens bulk eviction would take."""
    B, KVH, cap, hist, m = 2, 2, 32, 7, 4
    sh = O.Scissorhands(B, KVH, cap, history=hist)
    sh.prefill(cap - 3)
    ref = _FullLog((B, KVH, cap), hist)
    ref.insert_at(sh.live.copy())
    g = np.random.Generator(np.random.PCG64([29]))
    queue, pos, refills = None, m, 0
    for step in range(70):
        if sh.live.all():
            if pos == m:
                exp = [[ref.queue_order(b, kv, sh.live, m) for kv in range(KVH)] for b in range(B)]
                bulk = copy.deepcopy(sh).evict(m)
                queue, pos = sh.refill_queue(m), 0
                refills += 1
                assert queue.tolist() == exp
                np.testing.assert_array_equal(np.sort(queue, axis=-1), bulk)
                assert sh.live.all()  # the queue evicts nothing by itself
            slot = sh.insert(replace=queue[..., pos])
            np.testing.assert_array_equal(slot, queue[..., pos])
            pos += 1
            hit = np.zeros(sh.live.shape, bool)
            np.put_along_axis(hit, slot[..., None].astype(np.int64), True, axis=-1)
            ref.insert_at(hit)
        else:
            before = sh.live.copy()
            sh.insert()
            ref.insert_at(sh.live & ~before)
        keys = sh.live.sum(-1, keepdims=True)
        p = np.where(sh.live, g.random((B, KVH, cap)) * 2.0 / keys, 0.0)
        ref.record(O.low_attention_bits(p, sh.live))
        sh.record(p)
        np.testing.assert_array_equal(np.where(sh.live, sh.low, 0), np.where(sh.live, ref.counts(), 0))
        np.testing.assert_array_equal(np.where(sh.live, sh.n_obs(), 0), np.where(sh.live, ref.nobs(), 0))
    assert refills >= 10


def test_sparse_recording_matches_full_log():
    """Sparse recording: every step inserts, only every M-th step records; counts and
    n_obs are over recordings, and bulk eviction still ranks by exact fractions (tokens
    not yet observed rank as fraction 0)."""
    B, KVH, cap, hist, m, M = 2, 2, 32, 5, 4, 3
    sh = O.Scissorhands(B, KVH, cap, history=hist)
    sh.prefill(cap - m)
    ref = _FullLog((B, KVH, cap), hist)
    ref.insert_at(sh.live.copy())
    g = np.random.Generator(np.random.PCG64([31]))
    unobserved = 0
    for step in range(80):
        before = sh.live.copy()
        sh.insert()
        ref.insert_at(sh.live & ~before)
        if step % M == 0:
            keys = sh.live.sum(-1, keepdims=True)
            p = np.where(sh.live, g.random((B, KVH, cap)) * 2.0 / keys, 0.0)
            ref.record(O.low_attention_bits(p, sh.live))
            sh.record(p)
        assert sh.t == ref.t == step // M + 1
        np.testing.assert_array_equal(np.where(sh.live, sh.low, 0), np.where(sh.live, ref.counts(), 0))
        np.testing.assert_array_equal(np.where(sh.live, sh.n_obs(), 0), np.where(sh.live, ref.nobs(), 0))
        if (step + 1) % m == 0:
            unobserved += int((sh.live & (sh.n_obs() == 0)).sum())
            live_before = sh.live.copy()
            exp = [[ref.evict_order(b, kv, live_before, m) for kv in range(KVH)] for b in range(B)]
            assert sh.evict(m).tolist() == exp
            ref.occ[~sh.live] = -1
    assert unobserved > 0  # the n_obs = 0 reading was exercised


def test_unobserved_token_ranks_as_fraction_zero():
    """A token inserted after the last recording has no observation: its fraction reads as
    0, tied with observed tokens that were never low, so ties go by slot."""
    sh = O.Scissorhands(1, 1, 32, history=5)
    sh.prefill(28)
    sh.record(np.full((1, 1, 32), 1.0))  # nothing below 1/keys: every fraction is 0
    assert sh.evict(4).tolist() == [[[0, 1, 2, 3]]]
    for _ in range(4):
        sh.insert()  # slots 0..3, not yet observed
    assert (sh.n_obs()[0, 0, :4] == 0).all() and (sh.n_obs()[0, 0, 4:28] == 1).all()
    assert sh.refill_queue(6).tolist() == [[[0, 1, 2, 3, 4, 5]]]
    assert sh.evict(6).tolist() == [[[0, 1, 2, 3, 4, 5]]]


# ----------------------------------------------------------------------------------------
# TOVA decode
# ----------------------------------------------------------------------------------------


def test_tova_decode_keeps_budget_and_evicts_argmin():
    B, H, KVH, D, S, budget = 2, 4, 2, 8, 20, 8
    K = normal_bf16((B, KVH, S, D), 27, 1)
    V = normal_bf16((B, KVH, S, D), 27, 2)
    st = {t: {n: normal_bf16(sh, 27, 10 + t, i) for i, (n, sh) in
              enumerate((("q", (B, H, D)), ("k", (B, KVH, D)), ("v", (B, KVH, D))))} for t in range(3)}
    sc, idx, Kc, Vc = O.tova_first_step(K, V, st[0]["q"], st[0]["k"], st[0]["v"], 0.3, budget)
    assert Kc.shape == (B, KVH, budget + 1, D)
    for b in range(B):
        assert np.all(idx[b] == idx[b, 0])  # head-mean score: same tokens for every KV head
        order = sorted(range(S + 1), key=lambda j: (-sc[b, 0, j], j))[:budget]
        assert idx[b, 0].tolist() == sorted(order)
    free = np.full((B, KVH), budget, np.int32)
    sc2, ev, Kc2, Vc2 = O.tova_decode_step(Kc, Vc, st[1]["q"], st[1]["k"], st[1]["v"], free, 0.3)
    for b in range(B):
        np.testing.assert_array_equal(Kc2[b, :, budget], st[1]["k"][b])
        j = min(range(budget + 1), key=lambda s: (sc2[b, 0, s], -s))
        assert np.all(ev[b] == j)


def test_tova_new_token_is_a_candidate():
    """A new token with the lowest score is evicted at once (its slot is free again)."""
    B, H, KVH, D, n = 1, 2, 1, 4, 5
    Kc = np.zeros((B, KVH, n, D), np.float32)
    Kc[0, 0, :, 0] = 1.0
    q = np.zeros((B, H, D), np.float32)
    q[..., 0] = 4.0
    knew = np.zeros((B, KVH, D), np.float32)
    knew[..., 0] = -1.0
    free = np.array([[2]], np.int32)
    sc, ev, _, _ = O.tova_decode_step(_bf16(Kc), _bf16(Kc), _bf16(q), _bf16(knew), _bf16(knew), free, 1.0)
    assert ev.tolist() == [[2]]
