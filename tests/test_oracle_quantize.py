"""Pins of the oracle's NVFP4 quantiser (CPU only).

* Exact round trip: with S = 1, a block {6s, e2m1_i * s} for every finite
  E4M3 scale s re-encodes to s's code and the original element codes
  (6s/6 and e2m1*s/s are exact in fp32).
* Dynamic scaling: the block holding the tensor amax gets the largest scale
  code 0x7E (448) and its largest element code +-6.
* Degenerate cases: S == 0, an all-zero block, negative zero.
* Nibble order: element 2i in the low nibble, checked on a hand-built row.
* Error bound: every element decodes within half the E2M1 gap at its
  magnitude (times the block's decode scale), or saturates at 6*d.
"""
import numpy as np
import torch

from conftest import read_golden


def _e2m1_vals():
    return [float(v) for _, v in read_golden("e2m1_values.txt")]


def _e4m3_finite_pos():
    out = []
    for c in range(1, 0x7F):
        out.append((c, float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item())))
    return out


def test_round_trip_every_scale(orc):
    vals = _e2m1_vals()
    rng = np.random.default_rng(3)
    for sc, s in _e4m3_finite_pos():
        codes = rng.integers(0, 16, 16)
        codes[rng.integers(0, 16)] = 7 if rng.random() < 0.5 else 15  # the block amax is 6s
        xb = np.array([vals[c] * s for c in codes], np.float32)
        got_sc, got_codes = orc.quantize_block(xb, 1.0)
        assert got_sc == sc
        # -0 and +0 decode equal; compare values, then the sign convention
        for c, g in zip(codes, got_codes):
            assert vals[int(g)] == vals[int(c)]


def test_dynamic_scale_max_block(orc):
    rng = np.random.default_rng(4)
    x = rng.normal(0, 1, (8, 64)).astype(np.float32)
    x[3, 17] = 9.5  # unique tensor amax
    codes, scales, S = orc.quantize(x)
    assert S == np.float32(np.float32(9.5) / np.float32(2688.0))
    assert scales[3, 1] == 0x7E
    byte = codes[3, 17 // 2]
    assert (byte >> 4) == 7  # element 17 is odd -> high nibble; +6
    x[3, 17] = -9.5
    codes, scales, S = orc.quantize(x)
    assert (codes[3, 8] >> 4) == 15


def test_zero_scale_and_zero_block(orc):
    x = np.zeros((2, 32), np.float32)
    codes, scales, S = orc.quantize(x)
    assert S == 0 and not codes.any() and not scales.any()
    x = np.random.default_rng(5).normal(0, 1, (2, 32)).astype(np.float32)
    codes, scales, _ = orc.quantize(x, S=0.0)
    assert not codes.any() and not scales.any()
    x[1, 16:] = 0.0
    codes, scales, _ = orc.quantize(x)
    assert scales[1, 1] == 0 and not codes[1, 8:].any()


def test_negative_zero_sign_kept(orc):
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 6.0
    x[0, 1] = -0.01   # rounds to -0
    x[0, 2] = -0.0
    codes, scales, _ = orc.quantize(x, S=1.0)
    assert scales[0, 0] == 0x38           # (6/6)/1 = 1.0
    assert codes[0, 0] == (7 | (8 << 4))  # element0 = +6, element1 = -0
    assert (codes[0, 1] & 15) == 8        # element2 = -0


def test_nibble_order_hand_built(orc):
    # with S = 1 and amax 6 the block scale is 1.0 and the codes are the values
    vals = [0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0, 0.0, 6.0]
    x = np.array([vals], np.float32)
    codes, scales, _ = orc.quantize(x, S=1.0)
    want_codes = [1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15, 0, 7]
    want_bytes = [want_codes[2 * i] | (want_codes[2 * i + 1] << 4) for i in range(8)]
    assert list(codes[0]) == want_bytes
    assert scales[0, 0] == 0x38


def test_dequant_error_bound(orc):
    rng = np.random.default_rng(6)
    x = (rng.normal(0, 1, (64, 256)) * np.exp(rng.normal(0, 2, (64, 1)))).astype(np.float32)
    codes, scales, S = orc.quantize(x)
    xd = orc.dequantize(codes, scales, S, 256)
    sv = scales.astype(np.int64)
    d = np.array([[orc.e4m3_value(int(c)) for c in row] for row in sv]) * np.float64(S)
    d = np.repeat(d, 16, axis=1)
    # half the gap between neighbouring E2M1 magnitudes, as a function of |q|
    q = np.abs(x.astype(np.float64)) / np.where(d > 0, d, 1)
    half_gap = np.where(q < 2.0, 0.25, np.where(q < 4.0, 0.5, 1.0))
    err = np.abs(x - xd)
    sat = np.maximum(np.abs(x) - 6 * d, 0)
    assert np.all(err <= half_gap * d * (1 + 1e-6) + sat + 1e-30)
    # where the block scale is a normal E4M3 number (relative step 2^-3, so
    # RNE error <= 2^-4), every block's q stays within 6 * (1 + 2^-4)
    normal = np.repeat(sv >= 0x08, 16, axis=1)
    assert normal.any() and (~normal).any()
    assert np.all(q[normal] <= 6.0 / (1 - 2 ** -4) + 1e-6)


def test_quantize_matches_blockwise(orc):
    rng = np.random.default_rng(7)
    x = rng.normal(0, 1, (5, 48)).astype(np.float32)
    codes, scales, S = orc.quantize(x)
    for r in range(5):
        for b in range(3):
            sc, ec = orc.quantize_block(x[r, 16 * b:16 * b + 16], S)
            assert scales[r, b] == sc
            packed = [ec[2 * i] | (ec[2 * i + 1] << 4) for i in range(8)]
            assert list(codes[r, 8 * b:8 * b + 8]) == packed
