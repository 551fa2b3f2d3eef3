"""Pins of the oracle's MXFP4 path (CPU only): the UE8M0 scale table, the
OCP MX conversion of 32-element blocks, the MXFP4 grouped GEMM and the
MXFP4 layer.

* UE8M0 decode against hand-listed spot values (tests/golden) and against
  torch's float8_e8m0fnu conversion, an independent implementation.
* Exact round trip: a block built from E2M1 values times 2^E whose largest
  magnitude is 4 or 6 has shared exponent E, so it must re-encode to the
  same scale code and element codes, for every E the fp32 range allows.
* Closed forms: saturation of [6, 8) * 2^E to 6, ties to the even code,
  kept sign of zero, the all-zero block, the clamp at the smallest scale.
* The quantisation error stays within half an E2M1 step times 2^E.
* GEMM against a pure-Python brute force from the format tables, and
  one-hot rows that must pick out weight columns exactly.
* The layer: structured restatement against the naive per-token one.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden
from nvfp4_mixture_experts_top_gb300 import workloads as wl

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_ue8m0_spot_values(orc):
    for code, val in read_golden("ue8m0_spot_values.txt"):
        assert orc.ue8m0_value(int(code, 16)) == float(val)
    assert math.isnan(orc.ue8m0_value(0xFF))


def test_ue8m0_all_codes_vs_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float32).numpy()
    for c in range(255):
        assert orc.ue8m0_value(c) == float(ref[c]), c
    assert math.isnan(ref[255])


@pytest.mark.parametrize("E", list(range(-127, -118)) + [-40, -3, -1, 0, 1, 2, 7, 30] + list(range(118, 126)))
def test_mx_block_exact_round_trip(orc, E):
    rng = np.random.default_rng(E + 1000)
    codes = rng.integers(0, 16, 32).astype(np.uint8)
    codes[rng.integers(0, 32)] = rng.choice([6, 7, 14, 15])  # largest magnitude 4 or 6
    vals = np.array([math.ldexp(E2M1[c], E) for c in codes], np.float64)
    x = vals.astype(np.float32)
    assert np.array_equal(x.astype(np.float64), vals)  # representable
    sc, ec = orc.mx_quantize_block(x)
    assert sc == E + 127
    assert np.array_equal(ec, codes)


def test_mx_saturation_ties_signs(orc):
    # amax = 7 (floor(log2 7) = 2, so E = 0): 7 saturates to 6
    x = np.zeros(32, np.float32)
    x[:10] = [7.0, -7.5, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.1]
    sc, ec = orc.mx_quantize_block(x)
    assert sc == 127
    #         7->6  -7.5->-6  .25->0  .75->1  1.25->1  1.75->2  2.5->2  3.5->4  5->4  -0.1->-0
    assert list(ec[:10]) == [7, 15, 0, 2, 2, 4, 4, 6, 6, 8]
    assert not ec[10:].any()
    # a block of 8 * 2^-3: E = floor(log2 1) - 2 = -3, q = 8 saturates
    x = np.full(32, 1.0, np.float32)
    sc, ec = orc.mx_quantize_block(x)
    assert sc == 127 - 2 and (ec == 6).all()  # 1.0 / 2^-2 = 4 -> code 6
    x = np.full(32, 1.9, np.float32)
    sc, ec = orc.mx_quantize_block(x)
    assert sc == 127 - 2 and (ec == 7).all()  # 1.9 / 2^-2 = 7.6 -> 6


def test_mx_zero_and_tiny_blocks(orc):
    sc, ec = orc.mx_quantize_block(np.zeros(32, np.float32))
    assert sc == 0 and not ec.any()
    neg0 = np.full(32, -0.0, np.float32)
    sc, ec = orc.mx_quantize_block(neg0)
    assert sc == 0 and (ec == 8).all()
    # smallest subnormal: floor(log2) = -149, E clamps to -127, q = 2^-22 -> 0
    tiny = np.zeros(32, np.float32)
    tiny[3] = np.float32(2.0 ** -149)
    sc, ec = orc.mx_quantize_block(tiny)
    assert sc == 0 and not ec.any()
    # 2^-126 (E clamps to -127): q = 2 -> code 4
    t2 = np.zeros(32, np.float32)
    t2[0] = np.float32(2.0 ** -126)
    sc, ec = orc.mx_quantize_block(t2)
    assert sc == 0 and ec[0] == 4


def test_mx_error_bound_random(orc):
    x = (np.random.default_rng(3).standard_normal((64, 256)) * np.exp2(np.random.default_rng(4).integers(-20, 20, (64, 1)))).astype(np.float32)
    codes, scales = orc.mx_quantize(x)
    dq = orc.mx_dequantize(codes, scales, 256)
    E = scales.astype(np.int64).repeat(32, axis=1) - 127
    q = np.abs(x.astype(np.float64)) / np.exp2(E)
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    bound = np.where(q <= 6, step / 2, q - 6) * np.exp2(E)
    assert np.all(np.abs(dq - x) <= bound * (1 + 1e-12))
    # the shared exponent puts every block's amax in [4, 8) * 2^E
    amax = np.abs(x).reshape(64, 8, 32).max(-1).astype(np.float64)
    e = scales.astype(np.int64) - 127
    assert np.all((amax >= 4 * np.exp2(e)) & (amax < 8 * np.exp2(e)))


def _brute_dec(codes, scales, r, c):
    byte = int(codes[r, c // 2])
    code = (byte >> 4) if c & 1 else (byte & 15)
    return Fraction(E2M1[code]) * Fraction(2) ** (int(scales[r, c // 32]) - 127)


def test_mx_gemm_brute_force(orc):
    rng = np.random.default_rng(7)
    K, N = 64, 3
    counts = [2, 0, 1]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offs[-1])
    ac = rng.integers(0, 256, (R, K // 2)).astype(np.uint8)
    as_ = rng.integers(120, 135, (R, K // 32)).astype(np.uint8)
    wc = rng.integers(0, 256, (3, N, K // 2)).astype(np.uint8)
    ws = rng.integers(118, 134, (3, N, K // 32)).astype(np.uint8)
    out = orc.grouped_gemm_mx(ac, as_, wc, ws, offs)
    for e in range(3):
        for r in range(offs[e], offs[e + 1]):
            for n in range(N):
                want = sum(_brute_dec(ac, as_, r, c) * _brute_dec(wc[e], ws[e], n, c) for c in range(K))
                assert abs(Fraction(out[r, n]) - want) <= abs(want) * Fraction(1, 2 ** 50)


def test_mx_gemm_one_hot_rows(orc):
    rng = np.random.default_rng(8)
    E, N, K = 2, 8, 64
    W = rng.standard_normal((E, N, K)).astype(np.float32)
    wq = orc.mx_quantize_experts(W)
    Wd = np.stack([orc.mx_dequantize(wq[0][e], wq[1][e], K) for e in range(E)])
    rows = [(0, 5), (0, 0), (1, 63)]
    a = np.zeros((3, K), np.float32)
    for i, (_, c) in enumerate(rows):
        a[i, c] = 1.0
    ac, as_ = orc.mx_quantize(a)
    offs = np.array([0, 2, 3], np.int32)
    out = orc.grouped_gemm_mx(ac, as_, wq[0], wq[1], offs)
    for i, (e, c) in enumerate(rows):
        assert np.array_equal(out[i], Wd[e][:, c])


@pytest.mark.parametrize("cfgname", ["tiny"])
def test_mx_layer_vs_naive_restatement(orc, cfgname):
    cfg = wl.CONFIGS[cfgname]
    x = wl.activations_bf16(cfg.T, cfg.H).float().numpy()
    logits = wl.router_logits(cfg).numpy()
    w13 = orc.mx_quantize_experts(np.stack([wl.expert_weight_fp32("w13", e, 2 * cfg.I, cfg.H).numpy()
                                            for e in range(cfg.E)]))
    w2 = orc.mx_quantize_experts(np.stack([wl.expert_weight_fp32("w2", e, cfg.H, cfg.I).numpy()
                                           for e in range(cfg.E)]))
    out, mids = orc.moe_layer("mxw4a4", x, logits, cfg.k, w13, w2, 0.0, intermediates=True)
    ref = orc.moe_layer_naive("mxw4a4", x, logits, cfg.k, w13, w2, 0.0)
    assert np.isfinite(out).all() and np.abs(out).max() > 0
    assert np.allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())
    assert mids["hq_scales"].shape == (cfg.T * cfg.k, cfg.I // 32)
    # the requantised h decodes to within the MXFP4 error bound of h32
    hq = orc.mx_dequantize(mids["hq_codes"], mids["hq_scales"], cfg.I)
    h = mids["h32"].astype(np.float64)
    E = mids["hq_scales"].astype(np.int64).repeat(32, axis=1) - 127
    assert np.all(np.abs(hq - h) <= 2.0 * np.exp2(E))
    # against the unquantised layer on the dequantised weights: MXFP4 noise only
    ref32 = orc.moe_layer("w4a16", x, logits, cfg.k, _as_nvfp4_free(orc, w13, cfg, 2 * cfg.I, cfg.H),
                          _as_nvfp4_free(orc, w2, cfg, cfg.H, cfg.I), 0.0)
    assert np.linalg.norm(out - ref32) / np.linalg.norm(ref32) < 0.25


def _as_nvfp4_free(orc, wq, cfg, N, K):
    """MXFP4 weights re-expressed exactly as NVFP4 with per-tensor scale 1 is
    not generally possible (2^E exceeds E4M3's range); instead quantise the
    dequantised weights with NVFP4 so the W4A16 restatement sees nearly the
    same weights.  Only used for a loose sanity bound."""
    W = np.stack([orc.mx_dequantize(wq[0][e], wq[1][e], K) for e in range(cfg.E)]).astype(np.float32)
    return orc.quantize_experts(W)
