"""Failure detection on the GPU without a GPU fault: a bounded device wait is made to run out
and must come back as a status, with the context still usable.

The fused tensor-core scoring launch has CTAs that wait for the other key ranges of their
(b, kvh).  The test hook makes the next such launch wait at most 1 ms and leaves out one CTA's
arrival; the launch must return, kvc_get_device_status must report KVC_ERR_TIMEOUT, and the
next ordinary call must match the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import attention_score_kv_window_gb300 as kvc
from synth import Workload, prefill_inputs
from tests.helpers import dev_bf16, assert_scores_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kvc.load_library()
    yield
    kvc.kvc_debug_inject_timeout(False)


def test_bounded_wait_times_out_and_the_device_stays_usable():
    # 32 query / 8 KV heads, window 64 (256 query rows per KV head: the tensor-core kernel),
    # 5000 keys: 19 key ranges per KV head, 152 CTAs, all resident (the fused launch)
    wl = Workload("t", B=1, H=32, KVH=8, D=128, S=5000, w=64, k=1, reduce="gqa", seed=61)
    inp = prefill_inputs(wl)
    q, K = dev_bf16(inp["q"]), dev_bf16(inp["K"])
    ref = O.window_scores(inp["q"], inp["K"], wl.scale, causal=True, reduce="gqa")
    assert kvc.kvc_get_device_status() == kvc.KVC_OK
    kvc.kvc_debug_inject_timeout(True)
    try:
        kvc.kvc_window_scores(q, K, wl.scale, causal=True, reduce="gqa")
        assert kvc.kvc_get_device_status() == kvc.KVC_ERR_TIMEOUT
    finally:
        kvc.kvc_debug_inject_timeout(False)
    assert kvc.kvc_get_device_status() == kvc.KVC_OK  # read and cleared
    for _ in range(2):
        got = kvc.kvc_window_scores(q, K, wl.scale, causal=True, reduce="gqa")
        assert_scores_close(got.cpu().numpy(), ref)
    assert kvc.kvc_get_device_status() == kvc.KVC_OK
