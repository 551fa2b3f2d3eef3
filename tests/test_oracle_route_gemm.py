"""Pins of the oracle's router, permutation, grouped GEMM, SwiGLU, combine and
full layer (CPU only).  Each pin is something the oracle cannot satisfy by
construction: a library routine, a closed form, an invariant, brute force,
or a second independent restatement.
"""
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

from conftest import read_golden
from nvfp4_mixture_experts_top_gb300 import workloads as wl

E2M1 = [float(v) for _, v in read_golden("e2m1_values.txt")]


def e4m3_np(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def dequant_np(codes, scales, K):
    """Independent dequantiser: golden E2M1 list + torch's E4M3 decode."""
    lo = codes & 15
    hi = codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], K)
    v = np.array(E2M1)[c]
    s = np.repeat(e4m3_np(scales), 16, axis=-1)
    return v * s


# ---------------------------------------------------------------- router

def test_route_weights_sum_to_one_and_order(orc):
    rng = np.random.default_rng(0)
    logits = rng.normal(0, 1, (64, 32)).astype(np.float32)
    ids, w = orc.route(logits, 6)
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-12)
    sel = np.take_along_axis(logits, ids, 1)
    assert np.all(np.diff(sel, axis=1) <= 0)
    assert np.all(w[:, :-1] >= w[:, 1:])


def test_route_vs_stable_argsort_and_softmax(orc):
    rng = np.random.default_rng(1)
    logits = rng.normal(0, 1, (40, 16)).astype(np.float32)
    logits[:, 3] = logits[:, 7]                     # exact ties
    logits[5, :] = 0.25                             # a fully tied row
    k = 5
    ids, w = orc.route(logits, k)
    ref = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref)
    assert list(ids[5]) == [0, 1, 2, 3, 4]
    sm = scipy.special.softmax(np.take_along_axis(logits, ref, 1).astype(np.float64), axis=1)
    assert np.allclose(w, sm, rtol=1e-13, atol=0)


def test_route_zipf_workload_is_ragged(orc):
    cfg = wl.small_variant(wl.CONFIGS["decode_b512"], H=256, I=128)
    logits = wl.router_logits(cfg).numpy()
    ids, _ = orc.route(logits, cfg.k)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    assert counts[0] > 8 * np.median(counts)  # expert 0 is the most popular


# ---------------------------------------------------------------- permute

def test_permute_invariants_and_stable_sort(orc):
    rng = np.random.default_rng(2)
    T, E, k = 37, 12, 4
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    offsets, perm, inv = orc.permute(ids, E)
    R = T * k
    assert offsets[0] == 0 and offsets[E] == R and np.all(np.diff(offsets) >= 0)
    assert np.array_equal(np.diff(offsets), np.bincount(ids.ravel(), minlength=E))
    assert sorted(inv.tolist()) == list(range(R))          # bijection
    order = np.argsort(ids.ravel(), kind="stable")          # pairs sorted by expert, stable
    assert np.array_equal(perm, order // k)
    assert np.array_equal(inv[order], np.arange(R))
    for t in range(T):
        for j in range(k):
            r = inv[t * k + j]
            assert perm[r] == t and offsets[ids[t, j]] <= r < offsets[ids[t, j] + 1]


# ---------------------------------------------------------------- GEMM

def _rand_nvfp4(rng, shape_rows, K, scale_lo=0x30, scale_hi=0x48):
    codes = rng.integers(0, 256, (*shape_rows, K // 2)).astype(np.uint8)
    scales = rng.integers(scale_lo, scale_hi, (*shape_rows, K // 16)).astype(np.uint8)
    return codes, scales


def test_gemm_brute_force_2x16x16(orc):
    """M=2 rows, N=16 outputs, K=16 (one block): exact rational sums from the
    golden E2M1 list and torch's E4M3 decode."""
    rng = np.random.default_rng(3)
    ac, as_ = _rand_nvfp4(rng, (2,), 16)
    wc, ws = _rand_nvfp4(rng, (1, 16), 16)
    S_a, S_w = np.float32(0.375), np.float32(1.25)
    offsets = np.array([0, 2], np.int32)
    out = orc.grouped_gemm_w4a4(ac, as_, S_a, wc, ws, np.array([S_w]), offsets)
    sa = e4m3_np(as_)
    sw = e4m3_np(ws)
    for r in range(2):
        for n in range(16):
            acc = Fraction(0)
            for c in range(16):
                a = E2M1[(ac[r, c // 2] >> (4 * (c % 2))) & 15] * sa[r, 0]
                w = E2M1[(wc[0, n, c // 2] >> (4 * (c % 2))) & 15] * sw[0, n, 0]
                acc += Fraction(a) * Fraction(w)
            want = acc * Fraction(float(S_a)) * Fraction(float(S_w))
            assert abs(Fraction(out[r, n]) - want) <= abs(want) * Fraction(1, 2 ** 50)


def test_gemm_grouped_vs_numpy_matmul(orc):
    rng = np.random.default_rng(4)
    E, N, K = 5, 32, 64
    counts = np.array([3, 0, 1, 7, 2])
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offsets[-1])
    ac, as_ = _rand_nvfp4(rng, (R,), K)
    wc, ws = _rand_nvfp4(rng, (E, N), K)
    w_S = rng.uniform(0.5, 2, E).astype(np.float32)
    S_a = np.float32(0.01)
    out = orc.grouped_gemm_w4a4(ac, as_, S_a, wc, ws, w_S, offsets)
    A = dequant_np(ac, as_, K)
    W = dequant_np(wc, ws, K)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        ref = (A[r0:r1] @ W[e].T) * np.float64(S_a) * np.float64(w_S[e])
        assert np.allclose(out[r0:r1], ref, rtol=1e-12, atol=1e-300)


def test_gemm_one_hot_rows_pick_weight_columns(orc):
    rng = np.random.default_rng(5)
    E, N, K = 2, 16, 64
    wc, ws = _rand_nvfp4(rng, (E, N), K)
    w_S = np.array([1.0, 0.5], np.float32)
    offsets = np.array([0, 2, 4], np.int32)
    ac = np.zeros((4, K // 2), np.uint8)
    as_ = np.full((4, K // 16), 0x38, np.uint8)     # scale 1.0
    cols = [0, 17, 40, 63]
    for r, c in enumerate(cols):
        ac[r, c // 2] = 2 << (4 * (c % 2))              # value 1.0 at column c
    out = orc.grouped_gemm_w4a4(ac, as_, 1.0, wc, ws, w_S, offsets)
    W = dequant_np(wc, ws, K)
    for r, c in enumerate(cols):
        e = 0 if r < 2 else 1
        assert np.array_equal(out[r], W[e][:, c] * w_S[e])


def test_gemm_w4a16_vs_numpy(orc):
    rng = np.random.default_rng(6)
    E, N, K = 3, 16, 64
    offsets = np.array([0, 2, 2, 5], np.int32)
    a = torch.randn(5, K, dtype=torch.float32).to(torch.bfloat16).float().numpy()
    wc, ws = _rand_nvfp4(rng, (E, N), K)
    w_S = np.array([1.0, 2.0, 0.25], np.float32)
    out = orc.grouped_gemm_w4a16(a, wc, ws, w_S, offsets)
    W = dequant_np(wc, ws, K)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        assert np.allclose(out[r0:r1], a[r0:r1].astype(np.float64) @ W[e].T * w_S[e], rtol=1e-12)


# ---------------------------------------------------------------- SwiGLU, combine

def test_swiglu_closed_forms_and_library(orc):
    g = np.array([0.0, 30.0, -3.0, 3.0, 1.5, -60.0], np.float32)
    u = np.ones_like(g)
    G = np.concatenate([g, u])[None, :]
    h = orc.swiglu(G)[0]
    assert h[0] == 0.0                                   # silu(0) = 0
    assert abs(h[1] - 30.0) < 1e-11                      # silu(x) -> x
    assert abs(h[2] - (h[3] - 3.0)) < 1e-15              # silu(-x) = silu(x) - x
    assert abs(h[5]) < 1e-24
    rng = np.random.default_rng(7)
    G = rng.normal(0, 2, (9, 64)).astype(np.float32)
    h = orc.swiglu(G)
    gg, uu = G[:, :32].astype(np.float64), G[:, 32:].astype(np.float64)
    assert np.allclose(h, gg * scipy.special.expit(gg) * uu, rtol=1e-14, atol=1e-300)


def test_combine_gather_and_linearity(orc):
    rng = np.random.default_rng(8)
    T, k, H = 6, 1, 8
    Y = rng.normal(0, 1, (T * k, H)).astype(np.float32)
    inv = rng.permutation(T * k).astype(np.int32)
    out = orc.combine(Y, inv, np.ones((T, k)))
    assert np.array_equal(out, Y[inv].astype(np.float64))
    k = 3
    Y1 = rng.normal(0, 1, (T * k, H)).astype(np.float32)
    Y2 = rng.normal(0, 1, (T * k, H)).astype(np.float32)
    inv = rng.permutation(T * k).astype(np.int32)
    w = rng.uniform(0, 1, (T, k))
    a = orc.combine(Y1, inv, w) + orc.combine(Y2, inv, w)
    Ysum = (Y1.astype(np.float64) + Y2.astype(np.float64))
    # Y1+Y2 is not exactly representable in fp32; compare against fp64 sum
    ref = np.stack([sum(w[t, j] * Ysum[inv[t * k + j]] for j in range(k)) for t in range(T)])
    assert np.allclose(a, ref, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- full layer

def _layer_inputs(cfg, seed=0):
    x = wl.activations_bf16(cfg.T, cfg.H, seed).float().numpy()
    logits = wl.router_logits(cfg, seed).numpy()
    w13 = np.stack([wl.expert_weight_fp32("w13", e, 2 * cfg.I, cfg.H, seed).numpy() for e in range(cfg.E)])
    w2 = np.stack([wl.expert_weight_fp32("w2", e, cfg.H, cfg.I, seed).numpy() for e in range(cfg.E)])
    return x, logits, w13, w2


@pytest.mark.parametrize("mode", ["w4a4", "w4a16"])
@pytest.mark.parametrize("cfgname", ["tiny", "c16_lite"])
def test_layer_vs_naive_restatement(orc, mode, cfgname):
    if cfgname == "tiny":
        cfg = wl.CONFIGS["tiny"]
    else:
        cfg = wl.small_variant(wl.CONFIGS["decode_c16"], H=256, I=128, E=32)
    x, logits, w13f, w2f = _layer_inputs(cfg)
    w13 = orc.quantize_experts(w13f)
    w2 = orc.quantize_experts(w2f)
    out, mids = orc.moe_layer(mode, x, logits, cfg.k, w13, w2, cfg.S_h, intermediates=True)
    ref = orc.moe_layer_naive(mode, x, logits, cfg.k, w13, w2, cfg.S_h)
    assert np.isfinite(out).all() and np.abs(out).max() > 0
    assert np.allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())
    # intermediates are consistent with the stage functions
    ids, w = orc.route(logits, cfg.k)
    assert np.array_equal(ids, mids["ids"])
    offs, perm, inv = orc.permute(ids, cfg.E)
    assert np.array_equal(offs, mids["offsets"]) and np.array_equal(inv, mids["inv"])


def _numpy_moe(x, logits, k, w13, w2, I):
    """fp64 MoE from numpy primitives: stable arg-sort top-k, scipy softmax
    and expit, dense matmuls.  w13 [E, 2I, H], w2 [E, H, I] as fp64."""
    T = x.shape[0]
    ref = np.zeros((T, w2.shape[1]))
    sel = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
    ww = scipy.special.softmax(np.take_along_axis(logits, sel, 1).astype(np.float64), axis=1)
    for t in range(T):
        for j in range(k):
            e = sel[t, j]
            gu = w13[e] @ x[t].astype(np.float64)
            h = gu[:I] * scipy.special.expit(gu[:I]) * gu[I:]
            ref[t] += ww[t, j] * (w2[e] @ h)
    return ref


def test_layer_w4a16_vs_numpy_on_dequantised_weights(orc):
    """W4A16 layer against an fp64 numpy MoE over the independently
    dequantised weights: only the storage roundings (G, h fp32, h bf16, Y)
    separate them, so the gap is at the bf16 level (2^-9 per element)."""
    cfg = wl.CONFIGS["tiny"]
    x, logits, w13f, w2f = _layer_inputs(cfg)
    w13 = orc.quantize_experts(w13f)
    w2 = orc.quantize_experts(w2f)
    out = orc.moe_layer("w4a16", x, logits, cfg.k, w13, w2, cfg.S_h)
    W13 = dequant_np(w13[0], w13[1], cfg.H) * w13[2][:, None, None].astype(np.float64)
    W2 = dequant_np(w2[0], w2[1], cfg.I) * w2[2][:, None, None].astype(np.float64)
    ref = _numpy_moe(x, logits, cfg.k, W13, W2, cfg.I)
    rel = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    assert rel < 3e-3, rel
    # and the NVFP4 weights stay close to the unquantised layer (~10% noise per
    # quantised matrix), so nothing is grossly wrong with the encoding itself
    ref32 = _numpy_moe(x, logits, cfg.k, w13f.astype(np.float64), w2f.astype(np.float64), cfg.I)
    assert np.linalg.norm(out - ref32) / np.linalg.norm(ref32) < 0.25


def test_layer_token_subset_with_batch_scale(orc):
    """Rows of the layer are independent once the activation scale is fixed:
    running a subset of tokens (with the full batch's scale and the logits of
    only the experts they use) reproduces those rows of the full layer."""
    cfg = wl.small_variant(wl.CONFIGS["decode_c16"], H=256, I=128, E=32)
    x, logits, w13f, w2f = _layer_inputs(cfg)
    w13 = orc.quantize_experts(w13f)
    w2 = orc.quantize_experts(w2f)
    full = orc.moe_layer("w4a4", x, logits, cfg.k, w13, w2, cfg.S_h)
    S_x = orc.tensor_scale(x)
    assert np.array_equal(full, orc.moe_layer("w4a4", x, logits, cfg.k, w13, w2, cfg.S_h, S_x=S_x))
    toks = [3, 11]
    ids, _ = orc.route(logits[toks], cfg.k)
    used = np.unique(ids)
    sub = orc.moe_layer("w4a4", x[toks], logits[toks][:, used], cfg.k,
                        tuple(a[used] for a in w13), tuple(a[used] for a in w2), cfg.S_h, S_x=S_x)
    assert np.array_equal(sub, full[toks])


def test_router_logits_vs_numpy_and_one_hot(orc):
    """The oracle's router-logits loop against numpy's fp64 matmul (an
    independent implementation), and one-hot activations that must pick out
    router-weight columns exactly."""
    T, H, E = 9, 320, 40
    x = wl.activations_bf16(T, H, seed=3).float().numpy()
    w = wl.router_weight_bf16(E, H, seed=3).float().numpy()
    got = orc.router_logits(x, w)
    ref = (x.astype(np.float64) @ w.astype(np.float64).T).astype(np.float32)
    # both sum in fp64 and round once to fp32; only the fp64 summation order
    # differs, which can move a rare result by one fp32 ulp
    assert np.allclose(got, ref, rtol=2e-7, atol=1e-9) and (got == ref).mean() > 0.99
    assert 0.5 < got.std() < 2.0     # logits of the expected scale
    oh = np.zeros((3, H), np.float32)
    oh[0, 0] = oh[1, 77] = oh[2, H - 1] = 1.0
    assert np.array_equal(orc.router_logits(oh, w), w[:, [0, 77, H - 1]].T)
