"""Helpers shared by the GPU parity tests: host<->device conversion, margins, tolerances."""
import numpy as np

from structured_slot_reads_gb300 import inputs

# tolerances (stated once, used by every parity test)
TOL_LOGPROB = 2e-3     # absolute, nats: lse, entropy, max logit, label logprobs, slot entropy
TOL_REL = 1e-2         # relative: attention outputs and expected embeddings


def dev_bf16(x, device="cuda"):
    """bf16-valued float32 numpy array -> torch bf16 tensor on the device (bit exact)."""
    import torch
    bits = inputs.bf16_bits(np.ascontiguousarray(x, dtype=np.float32))
    return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16)


def dev(x, dtype=None, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def host(t):
    import torch
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def assert_rel(x, y, tol=TOL_REL, what=""):
    """Row-wise relative error and elementwise bound (|x-y| <= tol * (|y| + rms(row)))."""
    x = np.asarray(x, np.float64).reshape(-1, np.shape(y)[-1])
    y = np.asarray(y, np.float64).reshape(-1, np.shape(y)[-1])
    rms = np.sqrt(np.mean(y * y, axis=1, keepdims=True)) + 1e-30
    rowerr = np.linalg.norm(x - y, axis=1) / (np.linalg.norm(y, axis=1) + 1e-30)
    assert rowerr.max() <= tol, f"{what}: worst row relative error {rowerr.max():.3e}"
    bound = tol * (np.abs(y) + rms)
    bad = np.abs(x - y) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond bound, worst {np.max(np.abs(x - y) - bound):.3e}"


def assert_abs(x, y, tol=TOL_LOGPROB, what=""):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    err = np.abs(x - y)
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    assert err.max() <= tol, f"{what}: max abs error {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"


def top2_gap(z):
    """Gap between the largest and second largest entries of each row."""
    part = np.partition(z, -2, axis=1)
    return part[:, -1] - part[:, -2]
