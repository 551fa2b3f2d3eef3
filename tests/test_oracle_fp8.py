"""Pins of the oracle's W4A8 arithmetic (CPU only): FP8 E4M3 activations
with one fp32 per-tensor scale ("Native FP4 Is Slower Than Emulated FP4",
section 1: NVFP4 as FP4 weights with FP8 activations) against NVFP4
weights.  Each pin is independent of the oracle: torch's float8_e4m3fn
conversion, exact round trips, closed forms, exact rational brute force,
one-hot rows, and a second restatement of the layer."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from test_oracle_route_gemm import E2M1, _layer_inputs, dequant_np, e4m3_np
from nvfp4_mixture_experts_top_gb300 import workloads as wl


def _torch_e4m3(q):
    """torch's fp32 -> float8_e4m3fn conversion (round to nearest even) as codes."""
    return torch.from_numpy(np.asarray(q, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_fp8_encode_vs_torch_with_sign():
    from oracle import oracle as orc
    grid = e4m3_np(np.arange(0, 0x7F, dtype=np.uint8))       # finite non-negative E4M3 values
    mids = (grid[1:] + grid[:-1]) / 2
    vals = [np.float32(v) for v in np.concatenate([grid, mids])]
    vals += [np.nextafter(v, np.float32(np.inf)) for v in vals] + [np.nextafter(v, np.float32(0)) for v in vals]
    vals += list(np.random.default_rng(5).uniform(0, 447, 2000).astype(np.float32))
    vals += list(np.float32(2.0) ** np.arange(-14, 8, dtype=np.float32))
    q = np.array([v for v in vals if v < 448], np.float32)
    for sign in (1, -1):
        got = np.array([orc.fp8_encode(sign * v) for v in q], np.uint8)
        assert np.array_equal(got, _torch_e4m3(sign * q))
    # saturation (torch has no saturating cast): 448 and beyond -> 0x7E
    assert orc.fp8_encode(448.0) == 0x7E and orc.fp8_encode(1e9) == 0x7E and orc.fp8_encode(-500.0) == 0xFE
    # the sign is kept when the magnitude rounds to zero
    assert orc.fp8_encode(-1e-9) == 0x80 and orc.fp8_encode(1e-9) == 0x00


def test_fp8_round_trip_of_representable_values(orc):
    """x = (every finite E4M3 value, both signs) * 2^-3 with amax = 448 * 2^-3:
    the dynamic scale is exactly 2^-3 and every code comes back unchanged."""
    codes = np.concatenate([np.arange(0, 0x7F), np.arange(0x80, 0xFF)]).astype(np.uint8)
    x = (e4m3_np(codes) * 2.0 ** -3).astype(np.float32)[None, :]
    got, S = orc.fp8_quantize(x)
    assert S == np.float32(2.0 ** -3)
    assert np.array_equal(got[0], codes)  # -0.0 keeps its sign bit (0x80)


def test_fp8_dynamic_scale_amax_and_error_bound(orc):
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((37, 96)) * 3).astype(np.float32)
    codes, S = orc.fp8_quantize(x)
    assert S == np.float32(np.abs(x).max()) / np.float32(448.0)
    i = np.unravel_index(np.abs(x).argmax(), x.shape)
    assert codes[i] & 0x7F == 0x7E and (codes[i] >> 7) == (x[i] < 0)
    # decoded error: at most half a step of E4M3 (2^-4 relative for normals,
    # 2^-10 * S absolute in the subnormal range)
    dec = e4m3_np(codes) * float(S)
    err = np.abs(dec - x)
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * float(S)) * (1 + 1e-6))
    # a static scale is taken as given
    c2, S2 = orc.fp8_quantize(x, S=0.5)
    assert S2 == np.float32(0.5) and np.array_equal(c2, _torch_e4m3(np.clip(x / np.float32(0.5), -448, 448)))


def test_fp8_zero_tensor(orc):
    codes, S = orc.fp8_quantize(np.zeros((3, 32), np.float32))
    assert S == 0 and not codes.any()


def test_gemm_w4a8_brute_force_2x16x16(orc):
    """Exact rational sums from torch's E4M3 decode (activations and weight
    block scales) and the golden E2M1 list."""
    rng = np.random.default_rng(7)
    a = rng.integers(0, 256, (2, 16)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x38                       # no NaN codes
    wc = rng.integers(0, 256, (1, 16, 8)).astype(np.uint8)
    ws = rng.integers(0x30, 0x48, (1, 16, 1)).astype(np.uint8)
    S_a, S_w = np.float32(0.375), np.float32(1.25)
    out = orc.grouped_gemm_w4a8(a, S_a, wc, ws, np.array([S_w]), np.array([0, 2], np.int32))
    av = e4m3_np(a)
    sw = e4m3_np(ws)
    for r in range(2):
        for n in range(16):
            acc = Fraction(0)
            for c in range(16):
                w = E2M1[(wc[0, n, c // 2] >> (4 * (c % 2))) & 15] * sw[0, n, 0]
                acc += Fraction(av[r, c]) * Fraction(w)
            want = acc * Fraction(float(S_a)) * Fraction(float(S_w))
            assert abs(Fraction(out[r, n]) - want) <= abs(want) * Fraction(1, 2 ** 50)


def test_gemm_w4a8_one_hot_and_grouped_vs_numpy(orc):
    rng = np.random.default_rng(8)
    E, N, K = 3, 32, 64
    wc = rng.integers(0, 256, (E, N, K // 2)).astype(np.uint8)
    ws = rng.integers(0x30, 0x48, (E, N, K // 16)).astype(np.uint8)
    wS = np.array([0.5, 1.0, 2.0], np.float32)
    # one-hot rows (code 0x38 = 1.0) pick out decoded weight columns exactly
    cols = [0, 17, 63]
    a = np.zeros((3, K), np.uint8)
    for r, c in enumerate(cols):
        a[r, c] = 0x38
    offs = np.array([0, 1, 1, 3], np.int32)
    out = orc.grouped_gemm_w4a8(a, np.float32(0.25), wc, ws, wS, offs)
    W = dequant_np(wc, ws, K)
    for r, (c, e) in enumerate(zip(cols, [0, 2, 2])):
        assert np.array_equal(out[r], 0.25 * wS[e] * W[e][:, c])
    # random rows against numpy's fp64 matmul on independently decoded values
    a = rng.integers(0, 256, (9, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0
    offs = np.array([0, 4, 4, 9], np.int32)
    out = orc.grouped_gemm_w4a8(a, np.float32(0.75), wc, ws, wS, offs)
    ref = np.zeros_like(out)
    for e in range(E):
        ref[offs[e]:offs[e + 1]] = 0.75 * wS[e] * (e4m3_np(a[offs[e]:offs[e + 1]]) @ W[e].T)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("cfgname", ["tiny", "c16_lite"])
def test_layer_w4a8_vs_naive_restatement(orc, cfgname):
    cfg = (wl.CONFIGS["tiny"] if cfgname == "tiny"
           else wl.small_variant(wl.CONFIGS["decode_c16"], H=256, I=128, E=32))
    x, logits, w13f, w2f = _layer_inputs(cfg)
    w13 = orc.quantize_experts(w13f)
    w2 = orc.quantize_experts(w2f)
    out, mids = orc.moe_layer("w4a8", x, logits, cfg.k, w13, w2, cfg.S_h8, intermediates=True)
    ref = orc.moe_layer_naive("w4a8", x, logits, cfg.k, w13, w2, cfg.S_h8)
    assert np.isfinite(out).all() and np.abs(out).max() > 0
    assert np.allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())
    # the layer's own intermediates: x's dynamic FP8 scale, h's FP8 codes
    assert mids["S_x"] == np.float32(np.abs(x).max()) / np.float32(448.0)
    hq, _ = orc.fp8_quantize(mids["h32"], S=cfg.S_h8)
    assert np.array_equal(mids["hq_codes"], hq)


def test_layer_w4a8_vs_numpy_with_torch_fp8(orc):
    """The W4A8 layer against an fp64 numpy MoE whose FP8 roundings are
    torch's float8_e4m3fn casts and whose weights are independently
    dequantised: only the fp32 storage of G, h and Y separates the two."""
    import scipy.special
    cfg = wl.CONFIGS["tiny"]
    x, logits, w13f, w2f = _layer_inputs(cfg)
    w13 = orc.quantize_experts(w13f)
    w2 = orc.quantize_experts(w2f)
    out = orc.moe_layer("w4a8", x, logits, cfg.k, w13, w2, cfg.S_h8)
    W13 = dequant_np(w13[0], w13[1], cfg.H) * w13[2][:, None, None].astype(np.float64)
    W2 = dequant_np(w2[0], w2[1], cfg.I) * w2[2][:, None, None].astype(np.float64)
    S_x = np.float32(np.abs(x).max()) / np.float32(448.0)
    xq = e4m3_np(_torch_e4m3(x / S_x)) * float(S_x)
    S_h = np.float32(cfg.S_h8)
    sel = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :cfg.k]
    ww = scipy.special.softmax(np.take_along_axis(logits, sel, 1).astype(np.float64), axis=1)
    ref = np.zeros((cfg.T, cfg.H))
    for t in range(cfg.T):
        for j in range(cfg.k):
            e = sel[t, j]
            gu = W13[e] @ xq[t]
            h = (gu[:cfg.I] * scipy.special.expit(gu[:cfg.I]) * gu[cfg.I:]).astype(np.float32)
            hq = e4m3_np(_torch_e4m3(np.clip(h / S_h, -448, 448))) * float(S_h)
            ref[t] += ww[t, j] * (W2[e] @ hq)
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < 1e-3
