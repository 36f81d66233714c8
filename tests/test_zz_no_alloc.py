"""kvc_window_scores_noalloc: the window-score call for callers that cannot allocate device
memory (their runtime plans every buffer and hands them only inputs and outputs).  Its
scratch is a fixed device array inside the library; the results must match the
workspace-taking kvc_window_scores.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import attention_score_kv_window_gb300 as kvc
from synth import Workload, prefill_inputs
from tests.helpers import dev_bf16, assert_scores_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kvc.load_library()


CASES = [
    # B, H, KVH, D, S, w, causal, reduce
    (1, 32, 8, 128, 32768, 64, True, "gqa"),      # SnapKV prefill layer
    (2, 32, 8, 128, 2049, 1, False, "all_heads"),  # TOVA decode scores
]


@pytest.mark.parametrize("B,H,KVH,D,S,w,causal,reduce", CASES)
def test_noalloc_matches_workspace_call_twice(B, H, KVH, D, S, w, causal, reduce):
    wl = Workload("t", B=B, H=H, KVH=KVH, D=D, S=S, w=w, k=1, reduce=reduce, seed=S)
    inp = prefill_inputs(wl)
    q, K = dev_bf16(inp["q"]), dev_bf16(inp["K"])
    ref = kvc.kvc_window_scores(q, K, wl.scale, causal=causal, reduce=reduce).cpu().numpy()
    out = torch.empty((B, KVH, S), dtype=torch.float32, device="cuda")
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        out.fill_(-1.0)
        kvc.kvc_window_scores_noalloc(q, K, wl.scale, causal=causal, reduce=reduce, scores=out)
        torch.cuda.synchronize()
        assert_scores_close(out.cpu().numpy(), ref)
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


def test_noalloc_alternating_shapes_share_the_array():
    """Calls of different shapes in turn (A, B, A): each call finds the array as the other
    shape left it (the fused tensor-core launch's bookkeeping words at other offsets) and
    must still match the workspace call."""
    runs = []
    for B, H, KVH, D, S, w, causal, reduce in CASES:
        wl = Workload("t", B=B, H=H, KVH=KVH, D=D, S=S, w=w, k=1, reduce=reduce, seed=S + 1)
        inp = prefill_inputs(wl)
        q, K = dev_bf16(inp["q"]), dev_bf16(inp["K"])
        ref = kvc.kvc_window_scores(q, K, wl.scale, causal=causal, reduce=reduce).cpu().numpy()
        runs.append((q, K, wl.scale, causal, reduce, ref))
    for i in (0, 1, 0, 1):
        q, K, scale, causal, reduce, ref = runs[i]
        out = torch.full(ref.shape, -1.0, dtype=torch.float32, device="cuda")
        kvc.kvc_window_scores_noalloc(q, K, scale, causal=causal, reduce=reduce, scores=out)
        torch.cuda.synchronize()
        assert_scores_close(out.cpu().numpy(), ref)
    assert kvc.kvc_get_device_status() == kvc.KVC_OK


def test_noalloc_rejects_shapes_beyond_the_fixed_scratch():
    # 64 batch rows x 8 KV heads x 32768 slots of all-heads partial scores need 64 MiB > 4 MiB
    # (one batch row broadcast with stride 0: the check is on the host, nothing is read)
    K = torch.zeros((1, 8, 32768, 128), dtype=torch.bfloat16, device="cuda").expand(64, 8, 32768, 128)
    q = torch.zeros((64, 32, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_window_scores_noalloc(q, K, 0.1, causal=False, reduce="all_heads")
    assert e.value.status == kvc.KVC_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
