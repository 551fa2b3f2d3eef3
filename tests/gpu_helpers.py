"""Shared helpers of the GPU parity tests.

Inputs come from the seeded generators in ``workloads``; expected values come
from the CPU oracle only.  Tolerances are the ones the target states for
floating-point outputs: relative Frobenius error <= 1e-3 and max elementwise
error <= 1e-2 x output RMS.  Integer work (codes, scales, ids, permutation)
is compared bit for bit.
"""
import numpy as np
import pytest
import torch

REL_FROB_TOL = 1e-3
MAX_ERR_RMS_TOL = 1e-2


def cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_mixture_experts_top_gb300 import binding
    binding.load()
    binding.nvfp4_device_check()
    return torch.device("cuda:0")


def errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = got - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(diff) / nref if nref > 0 else np.linalg.norm(diff)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    mx = np.abs(diff).max() / rms if rms > 0 else np.abs(diff).max()
    return rel, mx


def assert_close(got, ref, what=""):
    assert np.isfinite(np.asarray(got)).all(), what + ": non-finite output"
    rel, mx = errors(got, ref)
    assert rel <= REL_FROB_TOL and mx <= MAX_ERR_RMS_TOL, "%s: rel_frob=%.3e max/rms=%.3e" % (what, rel, mx)
    return rel, mx


def to_dev(a, device, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def upload_weights(w, E, N, K, device):
    """(codes, linear scales, S) numpy -> GPU tuple (codes, packed scales, S)."""
    from nvfp4_mixture_experts_top_gb300 import binding as B
    codes = to_dev(w[0], device)
    scales = to_dev(w[1], device)
    S = to_dev(w[2], device)
    packed = B.nvfp4_pack_weight_scales(scales, E, N, K)
    return codes, packed, S


def nvfp4_ambiguous(v, S, rel=1e-5):
    """Per element of v [rows, cols] (fp32 values about to be quantised with
    decode scale S): True where the element's E2M1 decision or its block's
    E4M3 scale decision lies within `rel` (relative) of a rounding midpoint,
    so that a last-bits difference in v may legitimately change the code.
    Uses torch's E4M3 decode for the scale grid."""
    v = np.asarray(v, np.float64)
    rows, cols = v.shape
    blk = np.abs(v).reshape(rows, cols // 16, 16).max(-1)
    b = blk / 6.0 / np.float64(S)
    grid = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = (grid[1:] + grid[:-1]) / 2
    idx = np.clip(np.searchsorted(mids, b), 1, len(mids) - 1)
    near_scale = np.minimum(np.abs(b - mids[idx - 1]), np.abs(b - mids[np.minimum(idx, len(mids) - 1)]))
    amb_scale = near_scale <= rel * np.maximum(b, 1e-30)
    # element decision with the scale the block actually gets
    sc = grid[np.clip(np.searchsorted(mids, b), 0, len(grid) - 1)]
    d = np.repeat(sc * np.float64(S), 16, axis=1)
    q = np.abs(v) / np.where(d > 0, d, 1.0)
    e2 = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    near_el = np.min(np.abs(q[..., None] - e2), axis=-1) <= rel * np.maximum(q, 1e-30)
    return near_el | np.repeat(amb_scale, 16, axis=1)


def unpack_codes(codes):
    c = np.asarray(codes)
    return np.stack([c & 15, c >> 4], -1).reshape(c.shape[0], -1)
