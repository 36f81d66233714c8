"""Attention-score-driven KV-cache compression for GB300 (sm_103a).

The compute lives in ``_lib/libkvc.so`` (hand-written CUDA, C ABI declared in
``include/kvc.h``); this package is its thin Python binding.  Importing it does not touch
the GPU; the first call loads the library and raises if it has not been built.
"""
from ._binding import (  # noqa: F401
    KvcError, KvDesc, ShState, ScissorhandsState, LIB_PATH, exported_symbols, load_library, kv_desc,
    host_device_pointer,
    kvc_window_scores, kvc_window_scores_noalloc, kvc_topk_select, kvc_compact_kv, kvc_topk_compact, kvc_topk_compact_channels,
    kvc_compress_prefill, kvc_compress_prefill_channels, kvc_write_slots,
    kvc_tova_decode_step, kvc_scissorhands_init, kvc_scissorhands_update,
    kvc_scissorhands_update_from_probs, kvc_scissorhands_evict, kvc_scissorhands_refill_queue,
    kvc_scissorhands_insert, kvc_channel_score, kvc_channel_prune, kvc_decode_attention, kvc_zero_add_back,
    kvc_value_channel_score,
    kvc_get_device_status, kvc_status_string, kvc_version, kvc_launch_count, kvc_debug_inject_timeout,
    KVC_OK, KVC_ERR_INVALID_ARG, KVC_ERR_UNSUPPORTED, KVC_ERR_CUDA, KVC_ERR_TIMEOUT,
    KVC_ERR_DEVICE_BOUNDS, KVC_ERR_WORKSPACE,
)
