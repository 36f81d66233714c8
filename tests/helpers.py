"""Test helpers: moving synthetic bf16 bit patterns to the GPU and comparing with the oracle."""
import numpy as np
import torch

import oracle as O

# fp32 scores against the float64 oracle: |g - r| <= RTOL*|r| + ATOL
RTOL = 1e-3
ATOL = 1e-30


def dev_bf16(u16: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def dev_i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def dev_u32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).to(device)


def assert_scores_close(got: np.ndarray, ref: np.ndarray, rtol=RTOL, atol=ATOL, what="scores"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = err > rtol * np.abs(ref) + atol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"got {got[tuple(i)]!r} ref {ref[tuple(i)]!r}")


def assert_selection_matches(got_idx, ref_scores, k, protect_tail=0, live=None, largest=True, rtol=RTOL):
    """Kept sets identical except items whose oracle score is within rtol of the k-th
    chosen score (near-ties may legitimately fall either way in fp32)."""
    got_idx = np.asarray(got_idx)
    ref_idx = O.topk_select(ref_scores, k, protect_tail=protect_tail, live=live, largest=largest)
    B, KVH, S = ref_scores.shape
    for b in range(B):
        for kv in range(KVH):
            g = got_idx[b, kv]
            r = ref_idx[b, kv]
            assert np.all(np.diff(g[g >= 0]) > 0), "indices must be ascending"
            assert (g >= 0).sum() == (r >= 0).sum()
            gs, rs = set(g[g >= 0].tolist()), set(r[r >= 0].tolist())
            diff = gs ^ rs
            if not diff:
                continue
            chosen = [j for j in rs if not (protect_tail and j >= S - protect_tail)]
            sc = ref_scores[b, kv]
            kth = min(sc[j] for j in chosen) if largest else max(sc[j] for j in chosen)
            for j in diff:
                assert abs(sc[j] - kth) <= rtol * abs(kth) + ATOL, \
                    f"(b={b},kvh={kv}) index {j} score {sc[j]} vs k-th {kth}"
