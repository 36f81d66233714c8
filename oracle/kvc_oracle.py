"""CPU oracle: attention-score-driven KV-cache compression, written from the pages' definitions.

TEST INFRASTRUCTURE.  Plain numpy, float64 arithmetic (bf16 inputs are widened exactly).
Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline arm import it;
the CUDA library never does, and nothing here imports the library.  It is deliberately
slow and unblocked: each function follows one definition so that it can be checked by eye.

Sources (page titles and sections of the web pages this method is taken from):

* "Add TOVA press" (kvpress pull request 12), SimJeg's shape walk-through: only the last
  ``window_size`` rows of the attention matrix are formed (``full_attn_weights[:, :, -w:, :]``);
  the TOVA score is ``attn_weights.mean(1)`` (mean over query heads) repeated over KV heads;
  hassidm's first comment: TOVA uses the last token's attention row averaged over heads.
* "Implement Scissorhands KV-cache compression & SnapKV prompt compression" (cold-compress
  pull request 11): review comments on ``cache.py`` (``attn_is_low = attn < 1/keys`` with
  ``keys = attn.shape[1]``; the history column ``counter % history_window_size`` is
  overwritten each step; attention is mean-pooled over each KV head's grouped queries before
  the callback) and the PR description (history window 400; per attention head, evict the
  tokens with the highest fraction of low-attention observations, in bulk every m steps;
  SnapKV keeps the whole observation window and compresses the prefix by the window's
  attention, only when the prompt is longer than the cache).
* "Add ThinK_Press" (kvpress pull request 18): SimJeg's first comment defines the channel
  score as ``sum_{i,j} (q_id * k_jd)^2`` over the 64 window queries and all keys;
  yuhuixu1993's reply gives the factorised form ``query_norm * key_norm``; SimJeg's option
  list (3a zero the pruned channels, 3b a smaller key cache with the zeros added back for
  decoding, 3c a smaller key cache and an attention that prunes the query too, as the
  author's reply proposes); the thread settles on pruning tokens first, then channels.

Readings where the pages are silent or garbled are listed in the repository's design notes;
the ones that decide a number are repeated beside the code below.
"""
from __future__ import annotations

from fractions import Fraction
from functools import lru_cache

import numpy as np

__all__ = [
    "as_f64", "visible_mask", "window_softmax", "window_scores", "topk_select", "compact_kv",
    "write_slots", "channel_score", "channel_score_bruteforce", "channel_prune",
    "compress_prefill", "value_channel_score", "zero_add_back", "decode_attention", "decode_attention_pruned",
    "tova_first_step", "tova_decode_step", "Scissorhands",
    "scissorhands_probs", "low_attention_bits", "fraction_rank_table",
]


# ----------------------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------------------


def as_f64(x: np.ndarray) -> np.ndarray:
    """Exact float64 view of an input: uint16 arrays are bf16 bit patterns."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def visible_mask(S: int, w: int, causal: bool, live_row: np.ndarray | None) -> np.ndarray:
    """[w, S] boolean: which keys window row ``i`` may attend.

    The window rows are the last ``w`` rows of the causal attention matrix ("Add TOVA
    press", SimJeg: ``attn_weights = full_attn_weights[:, :, -window_size:, :]``), so row i
    sits at absolute position ``S - w + i`` and sees keys ``j <= S - w + i``.  Decode
    queries (``causal=False``) see every live slot.  ``live_row`` ([S] bool) removes dead
    slots of a decode cache."""
    vis = np.ones((w, S), dtype=bool)
    if causal:
        j = np.arange(S)[None, :]
        i = np.arange(w)[:, None]
        vis &= j <= (S - w + i)
    if live_row is not None:
        vis &= np.asarray(live_row, dtype=bool)[None, :]
    return vis


def _group_probs(qg: np.ndarray, Kb: np.ndarray, scale: float, vis: np.ndarray) -> np.ndarray:
    """Softmax probabilities of one KV head's query group.

    qg [G, w, D], Kb [S, D] (float64), vis [w, S] → p [G, w, S]:
    ``s_ij = scale * q_i . k_j``; ``m_i = max_j s_ij``; ``l_i = sum_j exp(s_ij - m_i)``;
    ``p_ij = exp(s_ij - m_i) / l_i`` over the visible keys, 0 elsewhere.  A row with no
    visible key gets all-zero probabilities."""
    s = scale * np.einsum("gid,jd->gij", qg, Kb)
    s = np.where(vis[None], s, -np.inf)
    m = s.max(axis=2, keepdims=True)
    has = np.isfinite(m)
    e = np.where(vis[None], np.exp(s - np.where(has, m, 0.0)), 0.0)
    l = e.sum(axis=2, keepdims=True)
    return np.where(has, e / np.where(l > 0, l, 1.0), 0.0)


# ----------------------------------------------------------------------------------------
# step 1: window attention and token scores
# ----------------------------------------------------------------------------------------


def window_softmax(q, K, scale: float, causal: bool = True, live=None) -> np.ndarray:
    """Window attention probabilities p [B, H, w, S] (small inputs only).

    q [B, H, w, D] are the last ``w`` query rows, K [B, KVH, S, D]; query head h reads KV head
    ``h // (H // KVH)`` (grouped-query attention).  ``live`` is an optional [B, KVH, S] bool."""
    q = as_f64(q)
    K = as_f64(K)
    B, H, w, D = q.shape
    KVH, S = K.shape[1], K.shape[2]
    G = H // KVH
    p = np.zeros((B, H, w, S))
    for b in range(B):
        for kv in range(KVH):
            vis = visible_mask(S, w, causal, None if live is None else live[b, kv])
            p[b, kv * G:(kv + 1) * G] = _group_probs(q[b, kv * G:(kv + 1) * G], K[b, kv], scale, vis)
    return p


def window_scores(q, K, scale: float, causal: bool = True, live=None,
                  reduce: str = "gqa") -> np.ndarray:
    """Token scores [B, KVH, S] from the window attention.

    * ``reduce="gqa"``: ``score[b,kvh,j] = sum_i mean_{h in group(kvh)} p[b,h,i,j]`` — the
      attention is mean-pooled over each KV head's grouped queries (cold-compress PR 11,
      review comment on the attention callback) and summed over the window rows (SnapKV's
      observation window votes for prefix tokens).
    * ``reduce="all_heads"``: ``score[b,:,j] = sum_i mean_h p[b,h,i,j]``, the same vector
      for every KV head ("Add TOVA press": ``attn_weights.mean(1)`` then
      ``repeat(1, num_key_value_heads, 1)``).
    """
    q = as_f64(q)
    K = as_f64(K)
    B, H, w, D = q.shape
    KVH, S = K.shape[1], K.shape[2]
    G = H // KVH
    out = np.zeros((B, KVH, S))
    for b in range(B):
        for kv in range(KVH):
            vis = visible_mask(S, w, causal, None if live is None else live[b, kv])
            p = _group_probs(q[b, kv * G:(kv + 1) * G], K[b, kv], scale, vis)
            out[b, kv] = p.sum(axis=1).mean(axis=0)
        if reduce == "all_heads":
            # mean over all H heads = mean over KV heads of the per-group means (equal groups)
            out[b, :] = out[b].mean(axis=0)[None, :]
        elif reduce != "gqa":
            raise ValueError(reduce)
    return out


# ----------------------------------------------------------------------------------------
# step 2: selection
# ----------------------------------------------------------------------------------------


def _ranked(idx: np.ndarray, sc: np.ndarray, largest: bool) -> np.ndarray:
    """Candidates ``idx`` ordered from first-chosen to last-chosen.

    Ranking: token a outranks b iff ``score_a > score_b``, or the scores are equal and
    ``a < b``.  Keeping takes the top of this order; evicting takes its bottom (lowest score
    first; among equal scores the highest index first)."""
    if largest:
        order = np.lexsort((idx, -sc))
    else:
        order = np.lexsort((-idx, sc))
    return idx[order]


def topk_select(scores, k: int, protect_tail: int = 0, live=None, largest: bool = True) -> np.ndarray:
    """Per (b, kvh): indices of the ``k`` chosen tokens, ascending, int32 [B, KVH, k].

    ``largest=True`` keeps the k highest-ranked eligible tokens; ``largest=False`` picks the
    k lowest-ranked (eviction).  ``protect_tail=w`` forces the last w positions in (SnapKV
    keeps the whole observation window and selects only among the prefix), so ``k - w`` are
    chosen from ``[0, S - w)``.  Only live tokens are eligible.  When fewer than k tokens
    are eligible, all of them are returned and the tail is padded with -1 (with ``k >= S``
    this is SnapKV's "no overflow, nothing to compress" case)."""
    sc = np.asarray(scores)
    B, KVH, S = sc.shape
    if protect_tail and not largest:
        raise ValueError("protect_tail applies to keeping, not evicting")
    out = np.full((B, KVH, k), -1, dtype=np.int32)
    for b in range(B):
        for kv in range(KVH):
            elig = np.ones(S, dtype=bool) if live is None else np.asarray(live[b, kv], dtype=bool).copy()
            forced = np.zeros(S, dtype=bool)
            if protect_tail:
                forced[S - protect_tail:] = True
                forced &= elig
                elig[S - protect_tail:] = False
            n_forced = int(forced.sum())
            cand = np.nonzero(elig)[0]
            need = max(0, k - n_forced)
            chosen = _ranked(cand, sc[b, kv, cand].astype(np.float64), largest)[:need]
            keep = np.sort(np.concatenate([np.nonzero(forced)[0][:k], chosen]))
            out[b, kv, :keep.size] = keep
    return out


# ----------------------------------------------------------------------------------------
# step 3: gather-compaction
# ----------------------------------------------------------------------------------------


def compact_kv(K, V, idx):
    """``Kc[b,kvh,t] = K[b,kvh,idx[b,kvh,t]]`` (same for V); rows with index -1 are zero."""
    K = np.asarray(K)
    V = np.asarray(V)
    idx = np.asarray(idx)
    B, KVH, k = idx.shape
    Kc = np.zeros((B, KVH, k) + K.shape[3:], dtype=K.dtype)
    Vc = np.zeros((B, KVH, k) + V.shape[3:], dtype=V.dtype)
    for b in range(B):
        for kv in range(KVH):
            for t in range(k):
                j = int(idx[b, kv, t])
                if j >= 0:
                    Kc[b, kv, t] = K[b, kv, j]
                    Vc[b, kv, t] = V[b, kv, j]
    return Kc, Vc


def write_slots(K, V, k_new, v_new, slot):
    """Copies of K, V with ``K[b,kvh,slot[b,kvh]] = k_new[b,kvh]`` (same for V)."""
    K = np.array(K, copy=True)
    V = np.array(V, copy=True)
    B, KVH = slot.shape
    for b in range(B):
        for kv in range(KVH):
            K[b, kv, int(slot[b, kv])] = k_new[b, kv]
            V[b, kv, int(slot[b, kv])] = v_new[b, kv]
    return K, V


def compress_prefill(q, K, V, scale, k, protect_tail=0, reduce="gqa", causal=True):
    """Prefill compression: window scores → top-k (window protected) → gather."""
    sc = window_scores(q, K, scale, causal=causal, reduce=reduce)
    idx = topk_select(sc, k, protect_tail=protect_tail)
    Kc, Vc = compact_kv(K, V, idx)
    return sc, idx, Kc, Vc


# ----------------------------------------------------------------------------------------
# ThinK key-channel score and pruning
# ----------------------------------------------------------------------------------------


def channel_score(q, K, kept=None) -> np.ndarray:
    """Closed-form ThinK channel score [B, KVH, D].

    ``cs[b,kvh,d] = (mean_{h in group} sum_i q_{h,i,d}^2) * sum_{j} k_{j,d}^2`` — the
    factorised ``query_norm * key_norm`` of "Add ThinK_Press" (yuhuixu1993's reply), with the
    sums taken over the token axes (window rows i, key rows j) as the brute-force definition
    requires; queries are the raw (unscaled) window queries; per KV head the query factor is
    the mean over the group's query heads.  ``kept`` ([B, KVH, k] indices, -1 ignored)
    restricts the key sum to the tokens kept by a preceding sequence compression."""
    q = as_f64(q)
    K = as_f64(K)
    B, H, w, D = q.shape
    KVH = K.shape[1]
    G = H // KVH
    cs = np.zeros((B, KVH, D))
    for b in range(B):
        for kv in range(KVH):
            qn = (q[b, kv * G:(kv + 1) * G] ** 2).sum(axis=1).mean(axis=0)  # [D]
            rows = K[b, kv]
            if kept is not None:
                ids = np.asarray(kept[b, kv])
                rows = rows[ids[ids >= 0]]
            kn = (rows ** 2).sum(axis=0)  # [D]
            cs[b, kv] = qn * kn
    return cs


def channel_score_bruteforce(q, K, kept=None) -> np.ndarray:
    """ThinK's defining form: ``sum_i sum_j (q_{i,d} * k_{j,d})^2`` built from the explicit
    per-channel outer products ``[D, w, S]`` ("Add ThinK_Press", SimJeg's ``channel_attn``),
    averaged over each KV head's query group.  Memory is D*w*S per head: tiny inputs only."""
    q = as_f64(q)
    K = as_f64(K)
    B, H, w, D = q.shape
    KVH = K.shape[1]
    G = H // KVH
    cs = np.zeros((B, KVH, D))
    for b in range(B):
        for kv in range(KVH):
            rows = K[b, kv]
            if kept is not None:
                ids = np.asarray(kept[b, kv])
                rows = rows[ids[ids >= 0]]
            acc = np.zeros(D)
            for h in range(kv * G, (kv + 1) * G):
                channel_attn = q[b, h].T[:, :, None] * rows.T[:, None, :]  # [D, w, S]
                acc += (channel_attn ** 2).sum(axis=(1, 2))
            cs[b, kv] = acc / G
    return cs


def channel_prune(cs, K, C: int, zero_mode: bool = False):
    """Keep the ``C`` highest-scoring key channels per (b, kvh) (same ranking rule as
    tokens: higher score first, lower channel index on ties); channel list ascending.

    Compact mode returns ``K[..., ch]`` ([B, KVH, S, C], the smaller cache of options 3b/3c);
    zero mode returns K with the other channels set to zero (option 3a)."""
    cs = np.asarray(cs, dtype=np.float64)
    B, KVH, D = cs.shape
    ch = np.zeros((B, KVH, C), dtype=np.int32)
    K = np.asarray(K)
    out = np.zeros(K.shape[:3] + (C,), dtype=K.dtype) if not zero_mode else np.zeros_like(K)
    for b in range(B):
        for kv in range(KVH):
            sel = np.sort(_ranked(np.arange(D), cs[b, kv], True)[:C])
            ch[b, kv] = sel
            if zero_mode:
                out[b, kv][:, sel] = K[b, kv][:, sel]
            else:
                out[b, kv] = K[b, kv][:, sel]
    return ch, out


def value_channel_score(q, Kc, Vc, scale: float, causal: bool = True) -> np.ndarray:
    """ThinK value-channel score [B, KVH, D] ("Add ThinK_Press" names value pruning without
    defining it; this is the key score's definition carried over to values).

    The key score sums, over window rows i and kept tokens j, the squared contribution
    ``(q_id k_jd)^2`` of channel d to the logit s_ij.  Channel d of value row j contributes
    ``p_ij v_jd`` to output channel d of row i, so the value score is
    ``cs_v[b,kvh,d] = mean_{h in group} sum_i sum_j (p_hij v_jd)^2``, where ``p`` is the window's
    attention over the compressed cache ``Kc`` (tokens first, then channels): the window rows
    are the last w tokens of ``Kc`` (SnapKV keeps them), so the causal rule of the compressed
    cache is the ordinary one on its own indices."""
    q = np.asarray(q)
    Vc = as_f64(Vc)
    B, H, w, D = q.shape
    KVH = Vc.shape[1]
    G = H // KVH
    p = window_softmax(q, Kc, scale, causal=causal)  # [B, H, w, k]
    cs = np.zeros((B, KVH, Vc.shape[-1]))
    for b in range(B):
        for kv in range(KVH):
            for h in range(kv * G, (kv + 1) * G):
                # sum_i sum_j (p_hij v_jd)^2, one (i, j) pair at a time
                for i in range(w):
                    cs[b, kv] += ((p[b, h, i][:, None] * Vc[b, kv]) ** 2).sum(axis=0)
            cs[b, kv] /= G
    return cs


# ----------------------------------------------------------------------------------------
# Decoding over the channel-pruned cache ("Add ThinK_Press" options 3b and 3c)
# ----------------------------------------------------------------------------------------


def zero_add_back(Kp, ch, D: int):
    """Option 3b: the full-width key cache rebuilt from the pruned one, the dropped channels
    filled with zeros: ``K[b, kvh, j, ch[b, kvh, c]] = Kp[b, kvh, j, c]``, every other channel 0.
    Values are moved, not converted (bf16 bit patterns stay bit patterns)."""
    Kp = np.asarray(Kp)
    ch = np.asarray(ch)
    B, KVH, S, C = Kp.shape
    K = np.zeros((B, KVH, S, D), dtype=Kp.dtype)
    for b in range(B):
        for kv in range(KVH):
            for c in range(C):
                K[b, kv, :, ch[b, kv, c]] = Kp[b, kv, :, c]
    return K


def decode_attention(q, K, V, scale: float, live=None) -> np.ndarray:
    """Attention of one new query per head over a cache: query head h reads KV head
    ``h // G``; logits ``s_j = scale * q[b,h,:] . K[b,kvh,j,:]`` over the live slots j,
    ``p = softmax(s)``, output ``sum_j p_j V[b,kvh,j,:]``.  float64 [B, H, Dv]; a head with no
    live slot gets zeros."""
    q, K, V = as_f64(q), as_f64(K), as_f64(V)
    B, H, _ = q.shape
    KVH, S = K.shape[1], K.shape[2]
    G = H // KVH
    out = np.zeros((B, H, V.shape[-1]))
    for b in range(B):
        for h in range(H):
            kv = h // G
            vis = np.ones(S, bool) if live is None else np.asarray(live, bool)[b, kv]
            if not vis.any():
                continue
            s = scale * (K[b, kv][vis] @ q[b, h])
            e = np.exp(s - s.max())
            out[b, h] = (e / e.sum()) @ V[b, kv][vis]
    return out


def decode_attention_pruned(q, ch, Kp, V, scale: float, live=None) -> np.ndarray:
    """Option 3c: the query is pruned to the key channels the cache kept,
    ``q'[b,h,c] = q[b,h,ch[b,kvh,c]]``, and attends the pruned keys directly.  The logits equal
    those of the full query against the zero-filled keys, so the scale stays that of the full
    head (``1/sqrt(D)``); values keep all channels."""
    q = np.asarray(q)
    ch = np.asarray(ch)
    B, H, _ = q.shape
    G = H // ch.shape[1]
    qp = np.stack([np.stack([q[b, h, ch[b, h // G]] for h in range(H)]) for b in range(B)])
    return decode_attention(qp, Kp, V, scale, live)


# ----------------------------------------------------------------------------------------
# TOVA decode: one eviction per generated token
# ----------------------------------------------------------------------------------------


def tova_first_step(K, V, q_new, k_new, v_new, scale, budget):
    """First decode step after a prefill cache of S tokens: the new token is appended
    (position S), scored together with the cache by the new query's head-mean attention,
    and the cache is cut to the ``budget`` highest-ranked tokens (ascending original order).

    Returns (scores [B,KVH,S+1], kept idx [B,KVH,budget], Kc, Vc) with Kc/Vc holding
    ``budget + 1`` slots; the last slot is free for the next token."""
    K = np.asarray(K)
    V = np.asarray(V)
    B, KVH, S, D = K.shape
    Kf = np.concatenate([K, np.asarray(k_new)[:, :, None, :]], axis=2)
    Vf = np.concatenate([V, np.asarray(v_new)[:, :, None, :]], axis=2)
    sc = window_scores(np.asarray(q_new)[:, :, None, :], Kf, scale, causal=False, reduce="all_heads")
    idx = topk_select(sc, budget)
    Kc, Vc = compact_kv(Kf, Vf, idx)
    Kc = np.concatenate([Kc, np.zeros((B, KVH, 1, D), dtype=Kc.dtype)], axis=2)
    Vc = np.concatenate([Vc, np.zeros((B, KVH, 1, D), dtype=Vc.dtype)], axis=2)
    return sc, idx, Kc, Vc


def tova_decode_step(Kc, Vc, q_new, k_new, v_new, free_slot, scale):
    """Later TOVA steps: the cache holds budget+1 slots, one of them free.  Write the new
    token into the free slot, score every slot with the new query (mean over all heads,
    shared by all KV heads), and evict the lowest-ranked slot, which becomes the next free
    slot.  Returns (scores, evicted [B, KVH], Kc', Vc')."""
    Kc, Vc = write_slots(Kc, Vc, k_new, v_new, np.asarray(free_slot))
    sc = window_scores(np.asarray(q_new)[:, :, None, :], Kc, scale, causal=False, reduce="all_heads")
    ev = topk_select(sc, 1, largest=False)[:, :, 0]
    return sc, ev, Kc, Vc


# ----------------------------------------------------------------------------------------
# Scissorhands: circular low-attention history and bulk eviction
# ----------------------------------------------------------------------------------------


def scissorhands_probs(q_new, K, scale, live) -> np.ndarray:
    """GQA-mean attention probability [B, KVH, S] of the new query over the live slots."""
    q = np.asarray(q_new)
    return window_scores(q[:, :, None, :], K, scale, causal=False, live=live, reduce="gqa")


def low_attention_bits(p, live) -> np.ndarray:
    """``attn < 1/keys`` with ``keys`` = number of live keys attended (cold-compress PR 11,
    ``keys = attn.shape[1]``).  The comparison is made in float32 — the attention tensor's
    precision against the scalar rounded to it — so p is rounded to float32 and the threshold
    is ``float32(1) / float32(keys)``.  Dead slots get 0."""
    live = np.asarray(live, dtype=bool)
    keys = live.sum(axis=-1, keepdims=True).astype(np.float32)
    thr = np.float32(1.0) / np.maximum(keys, np.float32(1.0))
    p32 = np.asarray(p).astype(np.float32)
    return (p32 < thr) & live


@lru_cache(maxsize=8)
def fraction_rank_table(history: int) -> np.ndarray:
    """rank[c, n] for 0 <= c <= n <= history, n >= 1: the position of the rational c/n in
    the sorted set of all such rationals (equal rationals share a rank).  Lets the eviction
    order low-attention fractions exactly."""
    fr = sorted({Fraction(c, n) for n in range(1, history + 1) for c in range(0, n + 1)})
    pos = {f: i for i, f in enumerate(fr)}
    rank = np.full((history + 1, history + 1), -1, dtype=np.int64)
    for n in range(1, history + 1):
        for c in range(0, n + 1):
            rank[c, n] = pos[Fraction(c, n)]
    return rank


class Scissorhands:
    """Scissorhands state for a [B, KVH, cap] slot cache.

    * ``hist[history, B, KVH, cap]``: bit plane ``t % history`` holds step t's
      low-attention flags (the circular queue overwrites the stalest column);
    * ``low[b,kvh,s]``: number of low flags of the slot's current token over its last
      ``n_obs = min(history, t - insert_step + 1)`` observations;
    * ``insert_step``: step at which the slot's token entered (prefill tokens: 0).

    ``t`` counts recordings.  Dense recording calls ``insert`` then ``record`` every decode
    step.  Sparse recording (suggested in the PR's review thread: look at the attention only
    every M steps and update numerator and denominator from that step alone) calls ``record``
    only every M-th step; ``insert_step`` then holds the index of the token's first
    recording, so ``n_obs`` counts observations, not steps.
    """

    def __init__(self, B: int, KVH: int, cap: int, history: int = 400):
        self.B, self.KVH, self.cap, self.history = B, KVH, cap, history
        self.live = np.zeros((B, KVH, cap), dtype=bool)
        self.insert_step = np.zeros((B, KVH, cap), dtype=np.int64)
        self.hist = np.zeros((history, B, KVH, cap), dtype=bool)
        self.low = np.zeros((B, KVH, cap), dtype=np.int64)
        self.t = 0  # index of the next update step

    def prefill(self, n_live: int):
        self.live[..., :n_live] = True
        self.insert_step[..., :n_live] = 0

    def insert(self, replace=None) -> np.ndarray:
        """Place the new token in one slot of every (b, kvh); returns the slots [B, KVH].

        ``replace is None``: the lowest free slot.  Otherwise ``replace[b, kvh]`` names a live
        slot whose token is evicted and overwritten by the new one (the eviction-queue
        variant: one eviction per step, so no slot is ever left empty).  Either way the slot
        starts afresh: ``insert_step = t`` (the index of the next recording) and no low
        flags; the flags its previous token left in the history are ignored by ``record``."""
        slot = np.zeros((self.B, self.KVH), dtype=np.int32)
        for b in range(self.B):
            for kv in range(self.KVH):
                if replace is None:
                    free = np.nonzero(~self.live[b, kv])[0]
                    if free.size == 0:
                        raise RuntimeError("no free slot")
                    s = int(free[0])
                else:
                    s = int(replace[b, kv])
                    if not (0 <= s < self.cap and self.live[b, kv, s]):
                        raise RuntimeError("queued slot is not live")
                slot[b, kv] = s
                self.live[b, kv, s] = True
                self.insert_step[b, kv, s] = self.t
                self.low[b, kv, s] = 0
        return slot

    def record(self, p) -> np.ndarray:
        """Record step t's flags (from GQA-mean probabilities p [B, KVH, cap])."""
        bits = low_attention_bits(p, self.live)
        plane = self.t % self.history
        # the overwritten flag belongs to the current token only if it was recorded after
        # the token's insertion, i.e. the token is at least ``history`` steps old
        old_valid = (self.t - self.insert_step) >= self.history
        old = self.hist[plane] & old_valid & self.live
        self.low += bits.astype(np.int64) - old.astype(np.int64)
        self.hist[plane] = bits
        self.t += 1
        return bits

    def n_obs(self) -> np.ndarray:
        return np.minimum(self.history, (self.t - 1) - self.insert_step + 1)

    def _eviction_order(self, b: int, kv: int) -> np.ndarray:
        """Live slots of (b, kvh), most evictable first: highest fraction ``low / n_obs``
        (compared exactly), ties to the lower slot.  A token inserted after the last
        recording (possible only when recording is sparse) has no observation and no low
        flag: its fraction reads as 0, like a token never found below uniform attention."""
        rank = fraction_rank_table(self.history)
        nobs = np.maximum(self.n_obs()[b, kv], 1)
        cand = np.nonzero(self.live[b, kv])[0]
        r = rank[self.low[b, kv, cand], nobs[cand]].astype(np.float64)
        return _ranked(cand, r, True)

    def evict(self, m: int) -> np.ndarray:
        """Bulk eviction: per (b, kvh), evict the ``m`` most evictable live tokens.  Returns
        the evicted slots ascending [B, KVH, m] (-1 padded); their slots become free."""
        out = np.full((self.B, self.KVH, m), -1, dtype=np.int32)
        for b in range(self.B):
            for kv in range(self.KVH):
                ev = np.sort(self._eviction_order(b, kv)[:m])
                out[b, kv, :ev.size] = ev
                self.live[b, kv, ev] = False
        return out

    def refill_queue(self, m: int) -> np.ndarray:
        """Eviction-queue variant (the PR description's change to Scissorhands): per
        (b, kvh), the ``m`` tokens bulk eviction would take, listed most evictable first,
        [B, KVH, m] (-1 padded).  Nothing is evicted here: the tokens stay live (and keep
        being recorded) until a step replaces them, one per step in queue order."""
        out = np.full((self.B, self.KVH, m), -1, dtype=np.int32)
        for b in range(self.B):
            for kv in range(self.KVH):
                q = self._eviction_order(b, kv)[:m]
                out[b, kv, :q.size] = q
        return out
