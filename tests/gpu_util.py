"""Shared helpers for the GPU parity tests (comparison rules and torch plumbing)."""
import numpy as np

# Per-value tolerance for logits, checkpoints and KV rows of the whole model:
# |got - want| <= ATOL + RTOL * |want|.
ATOL = 2e-3
RTOL = 2e-3
# Greedy ids must agree wherever the oracle's top-2 margin exceeds this.
MARGIN = 1e-2


def violation(got, want, atol=ATOL, rtol=RTOL) -> float:
    """Largest amount by which |got - want| exceeds atol + rtol |want| (<= 0 passes)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    if not np.all(np.isfinite(got)):
        return float("inf")
    return float((np.abs(got - want) - (atol + rtol * np.abs(want))).max())


def top2_margin(logits) -> float:
    part = np.partition(np.asarray(logits, np.float64), -2)
    return float(part[-1] - part[-2])


def dev(arr):
    import torch
    a = np.ascontiguousarray(arr)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to("cuda")


def host(t, dtype=None):
    import torch
    torch.cuda.synchronize()
    a = t.cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a
