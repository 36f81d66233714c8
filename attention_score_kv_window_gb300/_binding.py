"""ctypes binding of libkvc (argument marshalling only; every step runs in the CUDA library).

Each ``kvc_*`` function here takes torch tensors that live on the current CUDA device,
checks dtypes and shapes, passes raw device pointers and the current torch stream to the C
function of the same name, and raises :class:`KvcError` on a non-OK status.  Outputs and
scratch buffers the caller does not pass are allocated with torch (device memory only).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libkvc.so")

KVC_OK, KVC_ERR_INVALID_ARG, KVC_ERR_UNSUPPORTED, KVC_ERR_CUDA, KVC_ERR_TIMEOUT, \
    KVC_ERR_DEVICE_BOUNDS, KVC_ERR_WORKSPACE = range(7)
KVC_REDUCE_GQA_GROUP, KVC_REDUCE_ALL_HEADS = 0, 1
(KVC_OP_WINDOW_SCORES, KVC_OP_TOPK_SELECT, KVC_OP_COMPRESS_PREFILL, KVC_OP_TOVA_DECODE_STEP,
 KVC_OP_SCISSORHANDS_UPDATE, KVC_OP_SCISSORHANDS_EVICT, KVC_OP_CHANNEL_SCORE, KVC_OP_DECODE_ATTENTION,
 KVC_OP_VALUE_CHANNEL_SCORE, KVC_OP_COMPRESS_PREFILL_CHANNELS, KVC_OP_TOPK_COMPACT_CHANNELS) = range(11)

REDUCE = {"gqa": KVC_REDUCE_GQA_GROUP, "all_heads": KVC_REDUCE_ALL_HEADS}


class KvcError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"kvc status {status}: {msg}")
        self.status = status


class KvDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("KVH", ctypes.c_int32), ("D", ctypes.c_int32),
                ("S", ctypes.c_int64), ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64),
                ("stride_s", ctypes.c_int64)]


class ShState(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("KVH", ctypes.c_int32), ("cap", ctypes.c_int32),
                ("history", ctypes.c_int32), ("hist", ctypes.c_void_p), ("low_count", ctypes.c_void_p),
                ("insert_step", ctypes.c_void_p), ("live", ctypes.c_void_p), ("slot", ctypes.c_void_p),
                ("t", ctypes.c_int64), ("n_free", ctypes.c_int32)]


_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_DESC = ctypes.POINTER(KvDesc)
_SH = ctypes.POINTER(ShState)

_SIGNATURES = {
    "kvc_workspace_size": (_SZ, [_I32, _DESC, _I32, _I32]),
    "kvc_window_scores": (_I32, [_P, _P, _DESC, _I32, _F, _I32, _P, _I32, _P, _P, _SZ, _P]),
    "kvc_window_scores_noalloc": (_I32, [_P, _P, _DESC, _I32, _F, _I32, _P, _I32, _P, _P]),
    "kvc_topk_select": (_I32, [_P, _I32, _I32, _I64, _I32, _I32, _P, _I32, _P, _P, _SZ, _P]),
    "kvc_compact_kv": (_I32, [_P, _P, _DESC, _P, _I32, _P, _P, _P]),
    "kvc_topk_compact": (_I32, [_P, _P, _P, _DESC, _I32, _I32, _P, _I32, _P, _P, _P, _P]),
    "kvc_topk_compact_channels": (_I32, [_P, _P, _P, _DESC, _I32, _I32, _P, _I32, _P, _P, _P, _P, _I32, _P, _P, _SZ,
                                         _P]),
    "kvc_compress_prefill": (_I32, [_P, _P, _P, _DESC, _I32, _F, _I32, _I32, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "kvc_compress_prefill_channels": (_I32, [_P, _P, _P, _DESC, _I32, _F, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                             _SZ, _P]),
    "kvc_write_slots": (_I32, [_P, _P, _P, _P, _P, _DESC, _P]),
    "kvc_tova_decode_step": (_I32, [_P, _P, _P, _P, _P, _DESC, _F, _P, _P, _P, _SZ, _P]),
    "kvc_scissorhands_init": (_I32, [_SH, _I32, _P]),
    "kvc_scissorhands_update_from_probs": (_I32, [_SH, _P, _P]),
    "kvc_scissorhands_update": (_I32, [_SH, _P, _P, _P, _P, _P, _DESC, _F, _P, _P, _SZ, _P]),
    "kvc_scissorhands_evict": (_I32, [_SH, _I32, _P, _P]),
    "kvc_scissorhands_refill_queue": (_I32, [_SH, _I32, _P, _P]),
    "kvc_scissorhands_update_queued": (_I32, [_SH, _P, _I32, _I32, _P, _P, _P, _P, _P, _DESC, _F, _P, _P, _SZ,
                                              _P]),
    "kvc_scissorhands_insert": (_I32, [_SH, _P, _I32, _I32, _P, _P, _P, _P, _DESC, _P]),
    "kvc_channel_score": (_I32, [_P, _I32, _P, _DESC, _P, _I32, _P, _P, _SZ, _P]),
    "kvc_channel_prune": (_I32, [_P, _P, _DESC, _I32, _I32, _P, _P, _P]),
    "kvc_decode_attention": (_I32, [_P, _P, _P, _DESC, _P, _DESC, _P, _F, _P, _P, _SZ, _P]),
    "kvc_zero_add_back": (_I32, [_P, _DESC, _P, _P, _DESC, _P]),
    "kvc_value_channel_score": (_I32, [_P, _I32, _P, _P, _DESC, _F, _P, _P, _SZ, _P]),
    "kvc_host_device_pointer": (_I32, [_P, ctypes.POINTER(ctypes.c_void_p)]),
    "kvc_get_device_status": (_I32, [_P]),
    "kvc_status_string": (ctypes.c_char_p, [_I32]),
    "kvc_last_error_message": (ctypes.c_char_p, []),
    "kvc_version": (_I32, []),
    "kvc_launch_count": (_I64, []),
    "kvc_debug_inject_timeout": (_I32, [_I32]),
}


def exported_symbols() -> list[str]:
    return list(_SIGNATURES)


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvc.so (raises if it has not been built: there is no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libkvc.so not found at {path}; build it with "
                           "`python -m attention_score_kv_window_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != KVC_OK:
        msg = _lib.kvc_last_error_message().decode(errors="replace")
        raise KvcError(status, msg)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    return t.data_ptr()


def host_device_pointer(t) -> int:
    """Device address of a page-locked host tensor (kvc_host_device_pointer)."""
    out = ctypes.c_void_p()
    _check(load_library().kvc_host_device_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(out)))
    return out.value


def _vptr(V) -> int | None:
    """V of the compaction calls: a CUDA tensor, or a page-locked host tensor whose kept rows
    the compaction kernel reads over the host link."""
    if V is not None and not V.is_cuda:
        if not V.is_pinned():
            raise ValueError("V must be on a CUDA device or in page-locked host memory")
        return host_device_pointer(V)
    return _ptr(V)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _bf16(t, name):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    return t


def _dense(t, shape, name):
    """Outputs the library writes densely must be contiguous tensors of exactly this shape."""
    if tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor of shape {tuple(shape)}")


def kv_desc(K: torch.Tensor, H: int) -> KvDesc:
    """Descriptor of a [B, KVH, S, D] bf16 cache (any strides with a unit innermost stride)."""
    if K.dim() != 4 or K.stride(3) != 1:
        raise ValueError("K must be [B, KVH, S, D] with unit stride in D")
    B, KVH, S, D = K.shape
    return KvDesc(B, H, KVH, D, S, K.stride(0), K.stride(1), K.stride(2))


def _ws(op: int, desc: KvDesc, w: int, k: int, ws, device):
    need = load_library().kvc_workspace_size(op, ctypes.byref(desc), w, k)
    if need == ctypes.c_size_t(-1).value:
        _check(KVC_ERR_INVALID_ARG)
    if ws is None and need > 0:
        ws = torch.empty(int(need), dtype=torch.uint8, device=device)
    return ws, (0 if ws is None else ws.numel() * ws.element_size())


# ----------------------------------------------------------------------------------------
# calls
# ----------------------------------------------------------------------------------------


def kvc_window_scores(q_win, K, scale, causal=True, live_mask=None, reduce="gqa", scores=None,
                      ws=None, stream=None):
    """scores [B,KVH,S] float32 from the window queries q_win [B,H,w,D] and cache K."""
    lib = load_library()
    _bf16(q_win, "q_win"), _bf16(K, "K")
    B, H, w, D = q_win.shape
    desc = kv_desc(K, H)
    if scores is None:
        scores = torch.empty((B, K.shape[1], K.shape[2]), dtype=torch.float32, device=K.device)
    ws, nbytes = _ws(KVC_OP_WINDOW_SCORES, desc, w, 0, ws, K.device)
    _check(lib.kvc_window_scores(_ptr(q_win.contiguous()), _ptr(K), ctypes.byref(desc), w, float(scale),
                                 int(bool(causal)), _ptr(live_mask), REDUCE[reduce], _ptr(scores),
                                 _ptr(ws), nbytes, _stream(stream)))
    return scores


def kvc_window_scores_noalloc(q_win, K, scale, causal=True, live_mask=None, reduce="gqa", scores=None,
                              stream=None):
    """kvc_window_scores with the library's fixed device scratch instead of a workspace.

    For callers that may not allocate device memory during the call (their memory is
    planned by a host runtime).  ``scores`` should be preallocated by such callers; calls
    sharing a device must not overlap on the GPU (they share the scratch array)."""
    lib = load_library()
    _bf16(q_win, "q_win"), _bf16(K, "K")
    B, H, w, D = q_win.shape
    desc = kv_desc(K, H)
    if scores is None:
        scores = torch.empty((B, K.shape[1], K.shape[2]), dtype=torch.float32, device=K.device)
    _check(lib.kvc_window_scores_noalloc(_ptr(q_win.contiguous()), _ptr(K), ctypes.byref(desc), w, float(scale),
                                         int(bool(causal)), _ptr(live_mask), REDUCE[reduce], _ptr(scores),
                                         _stream(stream)))
    return scores


def kvc_topk_select(scores, k, protect_tail=0, live_mask=None, largest=True, idx=None, stream=None):
    lib = load_library()
    if scores.dtype != torch.float32:
        raise TypeError("scores must be float32")
    B, KVH, S = scores.shape
    if idx is None:
        idx = torch.empty((B, KVH, k), dtype=torch.int32, device=scores.device)
    _check(lib.kvc_topk_select(_ptr(scores.contiguous()), B, KVH, S, int(k), int(protect_tail),
                               _ptr(live_mask), int(bool(largest)), _ptr(idx), None, 0, _stream(stream)))
    return idx


def kvc_compact_kv(K, V, idx, H=None, K_out=None, V_out=None, stream=None):
    lib = load_library()
    B, KVH, S, D = K.shape
    k = idx.shape[-1]
    desc = kv_desc(K, H or KVH)
    if V is not None and (V.shape != K.shape or V.stride() != K.stride()):
        raise ValueError("V must have K's shape and strides")
    if K_out is None:
        K_out = torch.empty((B, KVH, k, D), dtype=K.dtype, device=K.device)
    if V is not None and V_out is None:
        V_out = torch.empty((B, KVH, k, D), dtype=V.dtype, device=K.device)
    _dense(K_out, (B, KVH, k, D), "K_out")
    if V_out is not None:
        _dense(V_out, (B, KVH, k, D), "V_out")
    _check(lib.kvc_compact_kv(_ptr(K), _vptr(V), ctypes.byref(desc), _ptr(idx.contiguous()), k, _ptr(K_out),
                              _ptr(V_out), _stream(stream)))
    return K_out, V_out


def kvc_topk_compact(scores, K, V, k, protect_tail=0, live_mask=None, largest=True, H=None, idx=None,
                     K_out=None, V_out=None, stream=None):
    """Top-k of each scores row and the gather of the chosen K/V rows; returns (idx, K_out, V_out)."""
    lib = load_library()
    if scores.dtype != torch.float32:
        raise TypeError("scores must be float32")
    B, KVH, S, D = K.shape
    desc = kv_desc(K, H or KVH)
    if V is not None and (V.shape != K.shape or V.stride() != K.stride()):
        raise ValueError("V must have K's shape and strides")
    if idx is None:
        idx = torch.empty((B, KVH, k), dtype=torch.int32, device=K.device)
    if K_out is None:
        K_out = torch.empty((B, KVH, k, D), dtype=K.dtype, device=K.device)
    if V is not None and V_out is None:
        V_out = torch.empty((B, KVH, k, D), dtype=V.dtype, device=K.device)
    _dense(K_out, (B, KVH, k, D), "K_out")
    if V_out is not None:
        _dense(V_out, (B, KVH, k, D), "V_out")
    _check(lib.kvc_topk_compact(_ptr(scores.contiguous()), _ptr(K), _vptr(V), ctypes.byref(desc), int(k),
                                int(protect_tail), _ptr(live_mask), int(bool(largest)), _ptr(idx), _ptr(K_out),
                                _ptr(V_out), _stream(stream)))
    return idx, K_out, V_out


def kvc_topk_compact_channels(scores, K, V, k, q_win, protect_tail=0, live_mask=None, largest=True, idx=None,
                              K_out=None, V_out=None, cs=None, ws=None, stream=None):
    """kvc_topk_compact plus ThinK's key-channel scores of the kept keys (summed by the
    compaction; ``q_win`` [B,H,w,D] the window queries).  Returns (idx, K_out, V_out, cs)."""
    lib = load_library()
    if scores.dtype != torch.float32:
        raise TypeError("scores must be float32")
    B, KVH, S, D = K.shape
    H, w = q_win.shape[1], q_win.shape[2]
    desc = kv_desc(K, H)
    if V is not None and (V.shape != K.shape or V.stride() != K.stride()):
        raise ValueError("V must have K's shape and strides")
    if idx is None:
        idx = torch.empty((B, KVH, k), dtype=torch.int32, device=K.device)
    if K_out is None:
        K_out = torch.empty((B, KVH, k, D), dtype=K.dtype, device=K.device)
    if V is not None and V_out is None:
        V_out = torch.empty((B, KVH, k, D), dtype=V.dtype, device=K.device)
    _dense(K_out, (B, KVH, k, D), "K_out")
    if V_out is not None:
        _dense(V_out, (B, KVH, k, D), "V_out")
    if cs is None:
        cs = torch.empty((B, KVH, D), dtype=torch.float32, device=K.device)
    ws, nbytes = _ws(KVC_OP_TOPK_COMPACT_CHANNELS, desc, 0, k, ws, K.device)
    _check(lib.kvc_topk_compact_channels(_ptr(scores.contiguous()), _ptr(K), _vptr(V), ctypes.byref(desc), int(k),
                                         int(protect_tail), _ptr(live_mask), int(bool(largest)), _ptr(idx),
                                         _ptr(K_out), _ptr(V_out), _ptr(q_win.contiguous()), int(w), _ptr(cs),
                                         _ptr(ws), nbytes, _stream(stream)))
    return idx, K_out, V_out, cs


def kvc_compress_prefill(q_win, K, V, scale, k, protect_tail=0, reduce="gqa", out=None, ws=None,
                         stream=None, keep_scores=True):
    """Returns (scores, idx, K_out, V_out).  ``keep_scores=False`` (or ``out`` with scores
    None) leaves the scores unwritten: the call then returns None in their place."""
    lib = load_library()
    B, H, w, D = q_win.shape
    _, KVH, S, _ = K.shape
    desc = kv_desc(K, H)
    if V.shape != K.shape or V.stride() != K.stride():
        raise ValueError("V must have K's shape and strides")
    if out is None:
        dev = K.device
        out = (torch.empty((B, KVH, S), dtype=torch.float32, device=dev) if keep_scores else None,
               torch.empty((B, KVH, k), dtype=torch.int32, device=dev),
               torch.empty((B, KVH, k, D), dtype=K.dtype, device=dev),
               torch.empty((B, KVH, k, D), dtype=V.dtype, device=dev))
    scores, idx, K_out, V_out = out
    ws, nbytes = _ws(KVC_OP_COMPRESS_PREFILL, desc, w, k, ws, K.device)
    _check(lib.kvc_compress_prefill(_ptr(q_win.contiguous()), _ptr(K), _vptr(V), ctypes.byref(desc), w,
                                    float(scale), REDUCE[reduce], int(k), int(protect_tail), _ptr(scores),
                                    _ptr(idx), _ptr(K_out), _ptr(V_out), _ptr(ws), nbytes, _stream(stream)))
    return scores, idx, K_out, V_out


def kvc_compress_prefill_channels(q_win, K, V, scale, k, protect_tail=0, reduce="gqa", out=None, cs=None, ws=None,
                                  stream=None, keep_scores=True):
    """kvc_compress_prefill plus ThinK's key-channel scores of the kept keys, summed by the
    compaction.  Returns (scores, idx, K_out, V_out, cs) with cs [B,KVH,D] float32."""
    lib = load_library()
    B, H, w, D = q_win.shape
    _, KVH, S, _ = K.shape
    desc = kv_desc(K, H)
    if V is not None and (V.shape != K.shape or V.stride() != K.stride()):
        raise ValueError("V must have K's shape and strides")
    dev = K.device
    if out is None:
        out = (torch.empty((B, KVH, S), dtype=torch.float32, device=dev) if keep_scores else None,
               torch.empty((B, KVH, k), dtype=torch.int32, device=dev),
               torch.empty((B, KVH, k, D), dtype=K.dtype, device=dev),
               torch.empty((B, KVH, k, D), dtype=K.dtype, device=dev) if V is not None else None)
    scores, idx, K_out, V_out = out
    if cs is None:
        cs = torch.empty((B, KVH, D), dtype=torch.float32, device=dev)
    ws, nbytes = _ws(KVC_OP_COMPRESS_PREFILL_CHANNELS, desc, w, k, ws, dev)
    _check(lib.kvc_compress_prefill_channels(_ptr(q_win.contiguous()), _ptr(K), _vptr(V), ctypes.byref(desc), w,
                                             float(scale), REDUCE[reduce], int(k), int(protect_tail), _ptr(scores),
                                             _ptr(idx), _ptr(K_out), _ptr(V_out), _ptr(cs), _ptr(ws), nbytes,
                                             _stream(stream)))
    return scores, idx, K_out, V_out, cs


def kvc_write_slots(k_new, v_new, slot, K, V, H=None, stream=None):
    lib = load_library()
    desc = kv_desc(K, H or K.shape[1])
    _check(lib.kvc_write_slots(_ptr(k_new.contiguous()), _ptr(None if v_new is None else v_new.contiguous()),
                               _ptr(slot.contiguous()), _ptr(K), _ptr(V), ctypes.byref(desc), _stream(stream)))


def kvc_tova_decode_step(q_new, k_new, v_new, K, V, scale, free_slot, scores=None, ws=None, stream=None):
    """One TOVA step; ``free_slot`` [B,KVH] int32 is updated in place to the evicted slot."""
    lib = load_library()
    B, H, D = q_new.shape
    desc = kv_desc(K, H)
    if scores is None:
        scores = torch.empty((B, K.shape[1], K.shape[2]), dtype=torch.float32, device=K.device)
    ws, nbytes = _ws(KVC_OP_TOVA_DECODE_STEP, desc, 1, 0, ws, K.device)
    _check(lib.kvc_tova_decode_step(_ptr(q_new.contiguous()), _ptr(k_new.contiguous()), _ptr(v_new.contiguous()),
                                    _ptr(K), _ptr(V), ctypes.byref(desc), float(scale), _ptr(free_slot),
                                    _ptr(scores), _ptr(ws), nbytes, _stream(stream)))
    return scores


class ScissorhandsState:
    """Device buffers of the Scissorhands history for a [B, KVH, cap] slot cache."""

    def __init__(self, B, KVH, cap, history=400, device="cuda"):
        self.hist = torch.zeros((history, B, KVH, cap // 32), dtype=torch.int32, device=device)
        self.low_count = torch.zeros((B, KVH, cap), dtype=torch.int16, device=device)
        self.insert_step = torch.zeros((B, KVH, cap), dtype=torch.int32, device=device)
        self.live = torch.zeros((B, KVH, cap // 32), dtype=torch.int32, device=device)
        self.slot = torch.zeros((B, KVH), dtype=torch.int32, device=device)
        self.c = ShState(B, KVH, cap, history, self.hist.data_ptr(), self.low_count.data_ptr(),
                         self.insert_step.data_ptr(), self.live.data_ptr(), self.slot.data_ptr(), 0, 0)

    @property
    def t(self) -> int:
        return self.c.t

    @property
    def n_free(self) -> int:
        return self.c.n_free


def kvc_scissorhands_init(state: ScissorhandsState, n_live: int, stream=None):
    _check(load_library().kvc_scissorhands_init(ctypes.byref(state.c), int(n_live), _stream(stream)))


def kvc_scissorhands_update_from_probs(state: ScissorhandsState, p, stream=None):
    _check(load_library().kvc_scissorhands_update_from_probs(ctypes.byref(state.c), _ptr(p.contiguous()),
                                                             _stream(stream)))


def kvc_scissorhands_update(state: ScissorhandsState, q_new, k_new, v_new, K, V, scale, probs=None,
                            ws=None, stream=None, queue=None, pos=0):
    """One decode step: insert (the lowest free slot, or with ``queue`` [B,KVH,m] over slot
    ``queue[..., pos]``), score the new query over the live slots, record the flags."""
    lib = load_library()
    B, H, D = q_new.shape
    desc = kv_desc(K, H)
    if probs is None:
        probs = torch.empty((B, K.shape[1], K.shape[2]), dtype=torch.float32, device=K.device)
    ws, nbytes = _ws(KVC_OP_SCISSORHANDS_UPDATE, desc, 1, 0, ws, K.device)
    vp = None if v_new is None else _ptr(v_new.contiguous())
    if queue is None:
        _check(lib.kvc_scissorhands_update(ctypes.byref(state.c), _ptr(q_new.contiguous()), _ptr(k_new.contiguous()),
                                           vp, _ptr(K), _ptr(V), ctypes.byref(desc), float(scale), _ptr(probs),
                                           _ptr(ws), nbytes, _stream(stream)))
    else:
        _check(lib.kvc_scissorhands_update_queued(ctypes.byref(state.c), _ptr(queue.contiguous()), queue.shape[-1],
                                                  int(pos), _ptr(q_new.contiguous()), _ptr(k_new.contiguous()), vp,
                                                  _ptr(K), _ptr(V), ctypes.byref(desc), float(scale), _ptr(probs),
                                                  _ptr(ws), nbytes, _stream(stream)))
    return probs


def kvc_scissorhands_insert(state: ScissorhandsState, k_new, v_new, K, V, H, queue=None, pos=0, stream=None):
    """Insert without recording (sparse recording's unobserved steps); ``queue`` as in
    kvc_scissorhands_update.  ``H`` is the number of query heads of the cache's layer."""
    desc = kv_desc(K, H)
    vp = None if v_new is None else _ptr(v_new.contiguous())
    qp, m = (None, 0) if queue is None else (_ptr(queue.contiguous()), queue.shape[-1])
    _check(load_library().kvc_scissorhands_insert(ctypes.byref(state.c), qp, m, int(pos), _ptr(k_new.contiguous()),
                                                  vp, _ptr(K), _ptr(V), ctypes.byref(desc), _stream(stream)))


def kvc_scissorhands_refill_queue(state: ScissorhandsState, m: int, queue=None, stream=None):
    """Eviction queue [B,KVH,m] int32: the m most evictable live slots, most evictable first."""
    if queue is None:
        queue = torch.empty((state.c.B, state.c.KVH, m), dtype=torch.int32, device=state.hist.device)
    _check(load_library().kvc_scissorhands_refill_queue(ctypes.byref(state.c), int(m), _ptr(queue),
                                                        _stream(stream)))
    return queue


def kvc_scissorhands_evict(state: ScissorhandsState, m: int, evicted=None, stream=None):
    if evicted is None:
        evicted = torch.empty((state.c.B, state.c.KVH, m), dtype=torch.int32, device=state.hist.device)
    _check(load_library().kvc_scissorhands_evict(ctypes.byref(state.c), int(m), _ptr(evicted), _stream(stream)))
    return evicted


def kvc_channel_score(q_win, K, idx=None, cs=None, ws=None, stream=None):
    lib = load_library()
    B, H, w, D = q_win.shape
    desc = kv_desc(K, H)
    k = 0 if idx is None else idx.shape[-1]
    if cs is None:
        cs = torch.empty((B, K.shape[1], D), dtype=torch.float32, device=K.device)
    ws, nbytes = _ws(KVC_OP_CHANNEL_SCORE, desc, w, k, ws, K.device)
    _check(lib.kvc_channel_score(_ptr(q_win.contiguous()), w, _ptr(K), ctypes.byref(desc),
                                 _ptr(None if idx is None else idx.contiguous()), k, _ptr(cs), _ptr(ws), nbytes,
                                 _stream(stream)))
    return cs


def kvc_channel_prune(cs, K, C, zero_mode=False, ch_idx=None, K_out=None, H=None, stream=None):
    lib = load_library()
    B, KVH, S, D = K.shape
    desc = kv_desc(K, H or KVH)
    if ch_idx is None:
        ch_idx = torch.empty((B, KVH, C), dtype=torch.int32, device=K.device)
    if K_out is None:
        K_out = torch.empty((B, KVH, S, D if zero_mode else C), dtype=K.dtype, device=K.device)
    _check(lib.kvc_channel_prune(_ptr(cs.contiguous()), _ptr(K), ctypes.byref(desc), int(C), int(bool(zero_mode)),
                                 _ptr(ch_idx), _ptr(K_out), _stream(stream)))
    return ch_idx, K_out


def kvc_decode_attention(q, K, V, scale, ch=None, live_mask=None, out=None, ws=None, stream=None):
    """One new query per head ``q`` [B,H,D] over the cache ``K`` [B,KVH,S,Ck] / ``V``
    [B,KVH,S,D]; ``ch`` [B,KVH,Ck] lists the key channels K kept (None: Ck == D).
    Returns ``out`` [B,H,D] float32."""
    lib = load_library()
    B, H, D = q.shape
    kd, vd = kv_desc(K, H), kv_desc(V, H)
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float32, device=q.device)
    ws, nbytes = _ws(KVC_OP_DECODE_ATTENTION, vd, 0, 0, ws, q.device)
    _check(lib.kvc_decode_attention(_ptr(q.contiguous()), _ptr(None if ch is None else ch.contiguous()), _ptr(K),
                                    ctypes.byref(kd), _ptr(V), ctypes.byref(vd),
                                    _ptr(None if live_mask is None else live_mask.contiguous()), float(scale),
                                    _ptr(out), _ptr(ws), nbytes, _stream(stream)))
    return out


def kvc_value_channel_score(q_win, Kc, Vc, scale, cs=None, ws=None, stream=None):
    """ThinK value-channel score [B,KVH,D] over the compressed cache ``Kc``/``Vc`` whose last
    w tokens are the window rows of ``q_win`` [B,H,w,D]."""
    lib = load_library()
    B, H, w, D = q_win.shape
    desc = kv_desc(Kc, H)
    if tuple(Vc.stride()) != tuple(Kc.stride()) or Vc.shape != Kc.shape:
        raise ValueError("Kc and Vc must have the same shape and strides")
    if cs is None:
        cs = torch.empty((B, Kc.shape[1], D), dtype=torch.float32, device=Kc.device)
    ws, nbytes = _ws(KVC_OP_VALUE_CHANNEL_SCORE, desc, w, 0, ws, Kc.device)
    _check(lib.kvc_value_channel_score(_ptr(q_win.contiguous()), w, _ptr(Kc), _ptr(Vc), ctypes.byref(desc),
                                       float(scale), _ptr(cs), _ptr(ws), nbytes, _stream(stream)))
    return cs


def kvc_zero_add_back(Kp, ch, D, H=None, K_out=None, stream=None):
    """Option 3b: the [B,KVH,S,D] key cache rebuilt from the pruned ``Kp`` [B,KVH,S,C]."""
    B, KVH, S, C = Kp.shape
    if K_out is None:
        K_out = torch.empty((B, KVH, S, D), dtype=Kp.dtype, device=Kp.device)
    pd, od = kv_desc(Kp, H or KVH), kv_desc(K_out, H or KVH)
    _check(load_library().kvc_zero_add_back(_ptr(Kp), ctypes.byref(pd), _ptr(ch.contiguous()), _ptr(K_out),
                                             ctypes.byref(od), _stream(stream)))
    return K_out


def kvc_get_device_status(stream=None) -> int:
    return int(load_library().kvc_get_device_status(_stream(stream)))


def kvc_status_string(s: int) -> str:
    return load_library().kvc_status_string(int(s)).decode()


def kvc_version() -> int:
    return int(load_library().kvc_version())


def kvc_debug_inject_timeout(armed: bool = True) -> None:
    """Test hook: the next fused tensor-core scoring launch waits at most 1 ms and leaves out
    one CTA's key-range arrival, so it times out (see include/kvc.h); False disarms it."""
    _check(load_library().kvc_debug_inject_timeout(int(bool(armed))))


def kvc_launch_count() -> int:
    """Kernels the library has enqueued since it was loaded (diagnostic counter)."""
    return int(load_library().kvc_launch_count())
