"""Pins of the oracle's number formats against fixed facts and library
routines (CPU only).

* E2M1 values against the hand-listed table in tests/golden.
* E4M3 decode of all 256 codes against torch's float8_e4m3fn conversion
  (an independent implementation) and against hand-listed spot values.
* E4M3 round-to-nearest-even encoding against torch's fp32 -> e4m3fn cast
  on a dense sweep that includes every midpoint; saturation by construction.
* E2M1 encoding against hand-worked tie cases and a brute-force nearest
  search over the golden value list.
* bf16 rounding against torch's fp32 -> bf16 cast.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden


def test_e2m1_table_matches_golden(orc):
    rows = read_golden("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        v = orc.e2m1_value(int(code))
        assert v == float(val)
        assert math.copysign(1.0, v) == math.copysign(1.0, float(val))


def test_e4m3_decode_all_codes_vs_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    for c in range(256):
        v = orc.e4m3_value(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(v) and math.isnan(ref[c])
        else:
            assert v == ref[c], (hex(c), v, ref[c])


def test_e4m3_spot_values(orc):
    for code, val in read_golden("e4m3_spot_values.txt"):
        assert orc.e4m3_value(int(code, 16)) == float(val)


def _e4m3_sweep():
    # every finite non-negative e4m3 value, every midpoint between neighbours,
    # one fp32 ulp either side of each midpoint, and a random fill
    vals = [np.float64(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item())
            for c in range(0x7F)]
    pts = set()
    for a, b in zip(vals[:-1], vals[1:]):
        m = np.float32((a + b) / 2)
        pts.update([np.float32(a), m, np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(1e9))])
    rng = np.random.default_rng(0)
    pts.update(np.float32(v) for v in rng.uniform(0, 448, 4000))
    pts.update(np.float32(v) for v in np.exp2(rng.uniform(-12, 8.8, 4000)))
    return sorted(p for p in pts if p <= 448)


def test_e4m3_encode_rne_vs_torch(orc):
    pts = _e4m3_sweep()
    ref = torch.tensor(np.array(pts, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(p) for p in pts])
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(pts[i], got[i], ref[i]) for i in bad[:10]]


def test_e4m3_encode_saturates(orc):
    for v in [448.0, 448.0001, 463.9, 464.0, 500.0, 1e6, 3.0e38, float("inf")]:
        assert orc.e4m3_encode(v) == 0x7E
    assert orc.e4m3_encode(0.0) == 0
    # below half the smallest subnormal rounds to zero; exactly half ties to 0
    assert orc.e4m3_encode(2.0 ** -10) == 0
    assert orc.e4m3_encode(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 1


def test_e2m1_encode_hand_cases(orc):
    for q, code in read_golden("e2m1_rounding.txt"):
        assert orc.e2m1_encode(float(q)) == int(code), q


def test_e2m1_encode_brute_force(orc):
    table = [float(v) for _, v in read_golden("e2m1_values.txt")][:8]
    rng = np.random.default_rng(1)
    qs = np.concatenate([rng.uniform(-8, 8, 5000), rng.normal(0, 0.3, 2000)]).astype(np.float32)
    for q in qs:
        a = abs(float(q))
        if a >= 6.0:
            want = 7
        else:
            d = [abs(a - t) for t in table]
            m = min(d)
            cands = [c for c in range(8) if d[c] == m]
            want = [c for c in cands if c % 2 == 0][0] if len(cands) > 1 else cands[0]
        want |= 8 if math.copysign(1.0, float(q)) < 0 else 0
        assert orc.e2m1_encode(float(q)) == want, q


def test_round_bf16_vs_torch(orc):
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-3, 1000), rng.normal(0, 1e4, 1000)])
    v = v.astype(np.float32)
    # exact ties: bf16 value + half an ulp
    base = torch.tensor(v[:500]).to(torch.bfloat16).float().numpy()
    ties = (base.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    v = np.concatenate([v, ties])
    ref = torch.tensor(v).to(torch.bfloat16).float().numpy()
    got = np.array([orc.round_bf16(x) for x in v], np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
