"""CPU-side checks of the C ABI: the library builds, loads, exports every declared symbol,
and rejects bad arguments on the host before anything is launched (no GPU needed)."""
import ctypes
import os
import re

import pytest

import attention_score_kv_window_gb300 as kvc
from attention_score_kv_window_gb300 import _binding as bnd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvc.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(bnd.LIB_PATH):
        from attention_score_kv_window_gb300.build import build_library
        build_library()
    return kvc.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kvc_window_scores", "kvc_topk_select", "kvc_compact_kv", "kvc_scissorhands_update",
                 "kvc_scissorhands_evict", "kvc_channel_score", "kvc_channel_prune"):
        assert must in names


def test_header_is_plain_c(tmp_path):
    """include/kvc.h compiles as C99 and as C++ (no torch or CUDA headers needed)."""
    import shutil
    import subprocess
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    for compiler, std, ext in (("gcc", "-std=c99", "c"), ("g++", "-std=c++17", "cpp")):
        if shutil.which(compiler) is None:
            pytest.skip(f"{compiler} not available")
        src = tmp_path / f"use.{ext}"
        src.write_text('#include "kvc.h"\nint use(void) { return (int)kvc_version(); }\n')
        r = subprocess.run([compiler, std, "-Wall", "-Werror", "-pedantic", "-fsyntax-only", "-I", inc, str(src)],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in bnd.exported_symbols(), f"binding lacks {name}"


def test_status_strings(lib):
    assert kvc.kvc_status_string(0) == "ok"
    assert "workspace" in kvc.kvc_status_string(kvc.KVC_ERR_WORKSPACE)
    assert kvc.kvc_version() >= 10000


def _desc(B=1, H=8, KVH=2, D=64, S=128):
    return bnd.KvDesc(B, H, KVH, D, S, KVH * S * D, S * D, D)


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced (validation fails first)


def test_host_validation_without_gpu(lib):
    d = _desc()
    # head_dim not supported
    bad = _desc(D=96)
    assert lib.kvc_window_scores(FAKE, FAKE, ctypes.byref(bad), 1, 0.1, 1, None, 0, FAKE, FAKE, 1 << 30, None) \
        == kvc.KVC_ERR_UNSUPPORTED
    # H not a multiple of KVH
    bad = _desc(H=7)
    assert lib.kvc_window_scores(FAKE, FAKE, ctypes.byref(bad), 1, 0.1, 1, None, 0, FAKE, FAKE, 1 << 30, None) \
        == kvc.KVC_ERR_INVALID_ARG
    # window longer than the sequence
    assert lib.kvc_window_scores(FAKE, FAKE, ctypes.byref(d), 129, 0.1, 1, None, 0, FAKE, FAKE, 1 << 30, None) \
        == kvc.KVC_ERR_INVALID_ARG
    # null and misaligned pointers
    assert lib.kvc_window_scores(None, FAKE, ctypes.byref(d), 1, 0.1, 1, None, 0, FAKE, FAKE, 1 << 30, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_window_scores(FAKE + 2, FAKE, ctypes.byref(d), 1, 0.1, 1, None, 0, FAKE, FAKE, 1 << 30, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert "aligned" in kvc.load_library().kvc_last_error_message().decode()
    # empty cache, and a row longer than the selection supports
    empty = _desc(S=0)
    assert lib.kvc_window_scores(FAKE, FAKE, ctypes.byref(empty), 1, 0.1, 1, None, 0, FAKE, FAKE, 1 << 30, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_topk_select(FAKE, 1, 1, 0, 4, 0, None, 1, FAKE, None, 0, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_topk_select(FAKE, 1, 1, 8 * 40960 + 1, 4, 0, None, 1, FAKE, None, 0, None) \
        == kvc.KVC_ERR_UNSUPPORTED
    # protect_tail larger than k, and with evict order
    assert lib.kvc_topk_select(FAKE, 1, 2, 128, 4, 8, None, 1, FAKE, None, 0, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_topk_select(FAKE, 1, 2, 128, 4, 2, None, 0, FAKE, None, 0, None) == kvc.KVC_ERR_INVALID_ARG
    # compaction outputs overlapping the inputs
    assert lib.kvc_compact_kv(FAKE, None, ctypes.byref(d), FAKE, 4, FAKE + 256, None, None) \
        == kvc.KVC_ERR_INVALID_ARG
    # fused selection + gather: idx overlapping the scores, and protect_tail in evict order
    big = FAKE * 64
    assert lib.kvc_topk_compact(big, FAKE, None, ctypes.byref(d), 4, 0, None, 1, big, FAKE * 128, None, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_topk_compact(big, FAKE, None, ctypes.byref(d), 4, 2, None, 0, FAKE * 256, FAKE * 128, None,
                                None) == kvc.KVC_ERR_INVALID_ARG
    # compaction with the key-channel sums: no channel_scores, a misaligned one, one that
    # overlaps the indices, and a workspace too small
    cws = lib.kvc_workspace_size(bnd.KVC_OP_TOPK_COMPACT_CHANNELS, ctypes.byref(d), 0, 4)
    assert cws > 0
    assert lib.kvc_topk_compact_channels(big, FAKE, None, ctypes.byref(d), 4, 0, None, 1, FAKE * 256, FAKE * 128,
                                         None, FAKE * 512, 1, None, FAKE * 1024, cws, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_topk_compact_channels(big, FAKE, None, ctypes.byref(d), 4, 0, None, 1, FAKE * 256, FAKE * 128,
                                         None, FAKE * 512, 1, FAKE * 768 + 4, FAKE * 1024, cws, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_topk_compact_channels(big, FAKE, None, ctypes.byref(d), 4, 0, None, 1, FAKE * 256, FAKE * 128,
                                         None, FAKE * 512, 1, FAKE * 256, FAKE * 1024, cws, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_topk_compact_channels(big, FAKE, None, ctypes.byref(d), 4, 0, None, 1, FAKE * 256, FAKE * 128,
                                         None, FAKE * 512, 1, FAKE * 768, FAKE * 1024, cws - 16, None) \
        == kvc.KVC_ERR_WORKSPACE
    wide = _desc(B=40000, H=8, KVH=2)
    assert lib.kvc_topk_compact_channels(big, FAKE, None, ctypes.byref(wide), 4, 0, None, 1, FAKE * 256, FAKE * 128,
                                         None, FAKE * 512, 1, FAKE * 768, FAKE * 1024, 1 << 40, None) \
        == kvc.KVC_ERR_UNSUPPORTED
    assert lib.kvc_compress_prefill_channels(FAKE * 512, FAKE, None, ctypes.byref(d), 1, 0.1, 1, 4, 0, None,
                                             FAKE * 256, FAKE * 128, None, None, FAKE * 1024, 1 << 30, None) \
        == kvc.KVC_ERR_INVALID_ARG
    # channel prune: compact mode needs C % 8 == 0; the channel list may not overlap the scores,
    # the keys or the pruned keys
    assert lib.kvc_channel_prune(FAKE, FAKE, ctypes.byref(d), 12, 0, FAKE, FAKE * 64, None) \
        == kvc.KVC_ERR_UNSUPPORTED
    assert lib.kvc_channel_prune(FAKE * 512, FAKE, ctypes.byref(d), 16, 0, FAKE * 512 + 64, FAKE * 64, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_channel_prune(FAKE * 512, FAKE, ctypes.byref(d), 16, 0, FAKE + 256, FAKE * 64, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_channel_prune(FAKE * 512, FAKE, ctypes.byref(d), 16, 0, FAKE * 64 + 256, FAKE * 64, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert "ch_idx overlaps" in kvc.load_library().kvc_last_error_message().decode()
    # value-channel scores: cs may not overlap the workspace or the caches
    vws = lib.kvc_workspace_size(bnd.KVC_OP_VALUE_CHANNEL_SCORE, ctypes.byref(d), 4, 0)
    assert vws > 0
    assert lib.kvc_value_channel_score(FAKE * 512, 4, FAKE, FAKE * 64, ctypes.byref(d), ctypes.c_float(0.1),
                                       FAKE * 1024 + 256, FAKE * 1024, vws, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_value_channel_score(FAKE * 512, 4, FAKE, FAKE * 64, ctypes.byref(d), ctypes.c_float(0.1),
                                       FAKE * 64 + 512, FAKE * 1024, vws, None) == kvc.KVC_ERR_INVALID_ARG
    assert "cs overlaps" in kvc.load_library().kvc_last_error_message().decode()
    # Scissorhands: capacity must be a multiple of 32; no free slot -> refused
    st = bnd.ShState(1, 2, 40, 400, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0)
    assert lib.kvc_scissorhands_init(ctypes.byref(st), 0, None) == kvc.KVC_ERR_INVALID_ARG
    st = bnd.ShState(1, 2, 128, 400, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0)
    assert lib.kvc_scissorhands_update(ctypes.byref(st), FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(d), 0.1, FAKE,
                                       FAKE, 1 << 30, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_scissorhands_evict(ctypes.byref(st), 8, FAKE, None) == kvc.KVC_ERR_INVALID_ARG  # t == 0
    # eviction queue: nothing recorded yet; m above the sort limit; position outside the queue
    assert lib.kvc_scissorhands_refill_queue(ctypes.byref(st), 8, FAKE, None) == kvc.KVC_ERR_INVALID_ARG
    st1 = bnd.ShState(1, 2, 4096, 400, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0)
    assert lib.kvc_scissorhands_refill_queue(ctypes.byref(st1), 4096, FAKE, None) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_scissorhands_update_queued(ctypes.byref(st), FAKE, 8, 8, FAKE, FAKE, FAKE, FAKE, FAKE,
                                              ctypes.byref(d), 0.1, FAKE, FAKE, 1 << 30, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_scissorhands_update_queued(ctypes.byref(st), None, 8, 0, FAKE, FAKE, FAKE, FAKE, FAKE,
                                              ctypes.byref(d), 0.1, FAKE, FAKE, 1 << 30, None) \
        == kvc.KVC_ERR_INVALID_ARG
    # insertion without a queue needs a free slot (n_free == 0 here)
    assert lib.kvc_scissorhands_insert(ctypes.byref(st), None, 0, 0, FAKE, FAKE, FAKE, FAKE, ctypes.byref(d),
                                       None) == kvc.KVC_ERR_INVALID_ARG
    assert "free slot" in kvc.load_library().kvc_last_error_message().decode()
    # decoding attention: K keeps 64 of 128 channels but no channel list; K and V disagree on S
    kd, vd = _desc(D=64, S=128), _desc(D=128, S=128)
    assert lib.kvc_decode_attention(FAKE, None, FAKE, ctypes.byref(kd), FAKE, ctypes.byref(vd), None, 0.1, FAKE,
                                    FAKE, 1 << 30, None) == kvc.KVC_ERR_INVALID_ARG
    vd2 = _desc(D=128, S=64)
    assert lib.kvc_decode_attention(FAKE, FAKE, FAKE, ctypes.byref(kd), FAKE, ctypes.byref(vd2), None, 0.1, FAKE,
                                    FAKE, 1 << 30, None) == kvc.KVC_ERR_INVALID_ARG
    # keys wider than the values, and strided (non-dense) rows are refused
    assert lib.kvc_decode_attention(FAKE, FAKE, FAKE, ctypes.byref(vd), FAKE, ctypes.byref(kd), None, 0.1, FAKE,
                                    FAKE, 1 << 30, None) == kvc.KVC_ERR_UNSUPPORTED
    strided = bnd.KvDesc(1, 8, 2, 128, 128, 2 * 128 * 256, 128 * 256, 256)
    assert lib.kvc_decode_attention(FAKE, None, FAKE, ctypes.byref(strided), FAKE, ctypes.byref(vd), None, 0.1,
                                    FAKE, FAKE, 1 << 30, None) == kvc.KVC_ERR_UNSUPPORTED
    # zero add-back: output overlapping the pruned input
    assert lib.kvc_zero_add_back(FAKE, ctypes.byref(kd), FAKE * 2, FAKE + 64, ctypes.byref(vd), None) \
        == kvc.KVC_ERR_INVALID_ARG
    # outputs that share bytes with an input or the workspace: the scores with K, q or the
    # workspace; the channel scores with their workspace; decoding's output with V
    M = FAKE * 256  # q at M, K at 2M, the workspace at 4M, outputs elsewhere unless overlapped
    wsz = lib.kvc_workspace_size(bnd.KVC_OP_WINDOW_SCORES, ctypes.byref(d), 4, 0)
    for out in (2 * M + 1024, M + 16, 4 * M + 32):
        assert lib.kvc_window_scores(M, 2 * M, ctypes.byref(d), 4, 0.1, 1, None, 0, out, 4 * M, wsz, None) \
            == kvc.KVC_ERR_INVALID_ARG
        assert "scores overlaps" in kvc.load_library().kvc_last_error_message().decode()
    assert lib.kvc_window_scores_noalloc(M, 2 * M, ctypes.byref(d), 4, 0.1, 1, None, 0, 2 * M + 1024, None) \
        == kvc.KVC_ERR_INVALID_ARG
    csz = lib.kvc_workspace_size(bnd.KVC_OP_CHANNEL_SCORE, ctypes.byref(d), 4, 0)
    assert lib.kvc_channel_score(M, 4, 2 * M, ctypes.byref(d), None, 0, 4 * M + 64, 4 * M, csz, None) \
        == kvc.KVC_ERR_INVALID_ARG
    assert "cs overlaps" in kvc.load_library().kvc_last_error_message().decode()
    assert lib.kvc_decode_attention(M, None, 2 * M, ctypes.byref(vd), 3 * M, ctypes.byref(vd), None, 0.1,
                                    3 * M + 4096, 4 * M, 1 << 30, None) == kvc.KVC_ERR_INVALID_ARG
    assert "out overlaps" in kvc.load_library().kvc_last_error_message().decode()


def test_workspace_size_rules(lib):
    d = _desc(S=4096, H=32, KVH=8, D=128)
    assert lib.kvc_workspace_size(bnd.KVC_OP_TOPK_SELECT, ctypes.byref(d), 1, 1) == 0
    assert lib.kvc_workspace_size(bnd.KVC_OP_WINDOW_SCORES, ctypes.byref(d), 64, 0) > 0
    assert lib.kvc_workspace_size(bnd.KVC_OP_WINDOW_SCORES, ctypes.byref(d), 5000, 0) == ctypes.c_size_t(-1).value
    # the channel-summing compaction: room for the key and query partials; the fused prefill
    # entry adds the window-score scratch and the scores
    ch = lib.kvc_workspace_size(bnd.KVC_OP_TOPK_COMPACT_CHANNELS, ctypes.byref(d), 0, 512)
    assert ch > 0 and ch % (2 * 8 * 128 * 4) == 0
    assert lib.kvc_workspace_size(bnd.KVC_OP_TOPK_COMPACT_CHANNELS, ctypes.byref(d), 0, 0) == ctypes.c_size_t(-1).value
    assert lib.kvc_workspace_size(bnd.KVC_OP_COMPRESS_PREFILL_CHANNELS, ctypes.byref(d), 64, 512) >= \
        ch + lib.kvc_workspace_size(bnd.KVC_OP_WINDOW_SCORES, ctypes.byref(d), 64, 0)
