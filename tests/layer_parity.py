"""Full-size layer parity against the oracle, shared by the NVFP4 (W4A4,
W4A16) and MXFP4 layer tests.

The GPU side runs the layer at full size through the staged entry points (so
its intermediates are visible) and through moe_layer_forward (which must be
bitwise the same).  The oracle runs the requested tokens -- by default every
token of the batch -- with the experts they use, quantised by the oracle from
the same seeded fp32 weights (and checked bit-exact against the GPU's
quantisation of them), and with the whole batch's activation scale.

Checks
* routing ids, offsets restricted to the sample, and the permutation through
  inv: bit for bit (routing of the GPU logits equals the oracle's routing);
* every requantised h code (W4A4 NVFP4 with the static S_h; MXFP4 with its
  per-block shared exponent; W4A8 FP8 with its static scale): equal to the
  oracle's, except where the oracle's own fp32 h lies within FLIP_WINDOW
  (relative) of that decision's rounding boundary, or within the measured
  difference between the GPU's pre-rounding h (from its fp32 G) and the
  oracle's -- G is accumulated in fp32 on the tensor cores and in fp64 by
  the oracle, so h can differ in its last bits;
* the output as a whole: relative Frobenius error <= 1e-3;
* every token without an h-code difference: relative Frobenius error <= 1e-3
  and max error <= 1e-2 x that token's output RMS;
* every token with an h-code difference: the same max-error bound, widened by
  exactly what the differing codes can move the output: for output column n,
    sum_j w[t, j] * sum_c |dec_gpu(h[r_j, c]) - dec_oracle(h[r_j, c])|
                  * |W2_e(j)[n, c]|
  (the down GEMM is linear in h, so this is the exact first-order effect of
  the differing codes; dec(.) decodes an h code with its block scale).

Each check prints its figures (worst relative Frobenius error, worst
max/RMS, flipped tokens and their observed excess over the plain bound, the
distribution of |h_gpu - h_oracle| / |h| measured from the GPU's fp32 G, and
the largest boundary distance a flip actually needed), so the log shows how
much margin every tolerance has.
"""
import numpy as np
import torch

from gpu_helpers import MAX_ERR_RMS_TOL, REL_FROB_TOL, errors, unpack_codes
from nvfp4_mixture_experts_top_gb300 import workloads as wl

# Where a requantised h code may differ: the oracle's fp32 h lies within
# this relative distance of the decision's rounding boundary.  Measured on
# GB300 over every token of decode_c16, wide and decode_b512 (NVFP4 and
# MXFP4 requantisation): |h_gpu - h_oracle| / |h| from the GPU's fp32 G is at
# most 5.4e-7, and the largest boundary distance any differing code needed was
# 2.7e-7, so 1e-5 leaves an 18x margin.  The W4A8 mode's G comes from F16
# MMAs whose accumulation differs more from fp64 (p99 5e-6 relative in h),
# so there a code may also differ where the measured pre-rounding difference
# of that element reaches the boundary.
FLIP_WINDOW = 1e-5

# E4M3 decode table from torch's own float8 type (independent of both sides)
_E4M3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
_E2_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])

# oracle-quantised expert weights of the most recent (format, workload)
_CACHE = {"key": None, "w": {}}


def oracle_expert_weights(orc, fmt, cfg, experts, seed=0, device="cpu"):
    """Oracle quantisation of experts' w13 and w2 (fp32 weights from their
    seeds, generated on `device` like the GPU side's).  fmt: 'nvfp4' or 'mx'.
    Returns (w13, w2), each (codes [n, N, K/2], scales, S [n] or None)."""
    key = (fmt, cfg.name, cfg.H, cfg.I, seed)
    if _CACHE["key"] != key:
        _CACHE["key"], _CACHE["w"] = key, {}
    cache = _CACHE["w"]
    out = []
    for which, N, K in (("w13", 2 * cfg.I, cfg.H), ("w2", cfg.H, cfg.I)):
        cs, ss, Ss = [], [], []
        for e in experts:
            k2 = (which, int(e))
            if k2 not in cache:
                wf = wl.expert_weight_fp32(which, int(e), N, K, seed, device).cpu().numpy()
                if fmt == "nvfp4":
                    c, s, S = orc.quantize(wf)
                else:
                    (c, s), S = orc.mx_quantize(wf), None
                cache[k2] = (c, s, S)
            c, s, S = cache[k2]
            cs.append(c)
            ss.append(s)
            Ss.append(S)
        out.append((np.stack(cs), np.stack(ss), None if fmt == "mx" else np.array(Ss, np.float32)))
    return out[0], out[1]


def nvfp4_boundary_distance(v, S):
    """Relative distance of every element of v [rows, cols] (fp32 values
    about to be NVFP4-quantised with decode scale S) to the nearer of its two
    decisions' rounding boundaries: its E2M1 element midpoint, and its
    block's E4M3 scale midpoint."""
    v = np.asarray(v, np.float64)
    rows, cols = v.shape
    b = np.abs(v).reshape(rows, cols // 16, 16).max(-1) / 6.0 / np.float64(S)
    grid = _E4M3[:0x7F]
    mids = (grid[1:] + grid[:-1]) / 2
    idx = np.clip(np.searchsorted(mids, b), 1, len(mids) - 1)
    d_scale = np.minimum(np.abs(b - mids[idx - 1]), np.abs(b - mids[idx])) / np.maximum(b, 1e-30)
    sc = grid[np.clip(np.searchsorted(mids, b), 0, len(grid) - 1)]
    q = np.abs(v) / np.where(np.repeat(sc, 16, 1) > 0, np.repeat(sc * np.float64(S), 16, 1), 1.0)
    d_el = np.min(np.abs(q[..., None] - _E2_MIDS), axis=-1) / np.maximum(q, 1e-30)
    return np.minimum(d_el, np.repeat(d_scale, 16, axis=1))


def mx_boundary_distance(v):
    """The same for MXFP4: the element midpoint at the block's shared
    exponent, and the block amax's distance to a power of two (where the
    shared exponent changes)."""
    v = np.asarray(v, np.float64)
    rows, cols = v.shape
    amax = np.abs(v).reshape(rows, cols // 32, 32).max(-1)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(amax > 0, amax, 1.0))
    d_scale = np.abs(amax - np.exp2(np.round(lg))) / np.maximum(amax, 1e-300)
    E = np.clip(np.floor(lg) - 2, -127, 127)
    q = np.abs(v) / np.repeat(np.exp2(E), 32, axis=1)
    d_el = np.min(np.abs(q[..., None] - _E2_MIDS), axis=-1) / np.maximum(q, 1e-30)
    return np.minimum(d_el, np.repeat(d_scale, 32, axis=1))


def fp8_boundary_distance(v, S):
    """Relative distance of every element of v (fp32 values about to be
    FP8-quantised with decode scale S) to the nearest E4M3 rounding midpoint."""
    q = np.abs(np.asarray(v, np.float64)) / np.float64(S)
    grid = _E4M3[:0x7F]
    mids = (grid[1:] + grid[:-1]) / 2
    idx = np.clip(np.searchsorted(mids, q), 1, len(mids) - 1)
    d = np.minimum(np.abs(q - mids[idx - 1]), np.abs(q - mids[idx]))
    return d / np.maximum(q, 1e-30)


def _decode_h(codes, scales, fmt, S_h):
    """Decoded h [rows, I] (fp64) from packed codes and linear block scales
    (FP8: one E4M3 code per element, no block scales)."""
    if fmt == "fp8":
        return _E4M3[codes] * np.float64(S_h)
    c = unpack_codes(codes)
    v = _E2M1[c]
    if fmt == "nvfp4":
        return v * np.repeat(_E4M3[scales], 16, axis=1) * np.float64(S_h)
    return v * np.repeat(np.exp2(scales.astype(np.float64) - 127.0), 32, axis=1)


def _w2_columns(w2, i, cols, fmt):
    """|W2_i[:, cols]| decoded in fp64 (with the per-tensor scale)."""
    codes, scales, S = w2
    byte = codes[i][:, cols // 2]
    nib = np.where(cols % 2 == 1, byte >> 4, byte & 15)
    v = np.abs(_E2M1[nib])
    if fmt == "nvfp4":
        return v * _E4M3[scales[i][:, cols // 16]] * np.float64(S[i])
    return v * np.exp2(scales[i][:, cols // 32].astype(np.float64) - 127.0)


def _silu_mul_f32(G, I):
    g = G[:, :I].astype(np.float32)
    u = G[:, I:].astype(np.float32)
    with np.errstate(over="ignore"):
        return (g / (np.float32(1) + np.exp(-g))) * u


def check_layer(orc, cfg, mode, d, x, logits, gpu_w, tokens=None, seed=0, device="cpu"):
    """Compare the GPU layer (staged outputs `d`: rt, G, out and hc/hs or hb)
    with the oracle on `tokens` (default: all).  gpu_w: ((codes13, lin13),
    (codes2, lin2)) on the GPU, to check the weights are the oracle's.
    Returns a dict of the figures it printed."""
    fmt = "mx" if mode == "mxw4a4" else "nvfp4"           # the weights' format
    hfmt = {"w4a4": "nvfp4", "mxw4a4": "mx", "w4a8": "fp8"}.get(mode)  # requantised h
    T, k, I, H = cfg.T, cfg.k, cfg.I, cfg.H
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    x_np = x.float().cpu().numpy()
    lg_np = logits.cpu().numpy()
    ids_o, _ = orc.route(lg_np[tokens], k)
    used = np.unique(ids_o)
    w13, w2 = oracle_expert_weights(orc, fmt, cfg, used, seed, device)
    # the GPU quantised the same weights: identical codes and scales
    (c13, l13), (c2, l2) = gpu_w
    idx = torch.as_tensor(used, device=c13.device, dtype=torch.long)
    assert np.array_equal(c13.index_select(0, idx).cpu().numpy(), w13[0])
    assert np.array_equal(l13.index_select(0, idx).cpu().numpy()[..., : w13[1].shape[-1]], w13[1])
    assert np.array_equal(c2.index_select(0, idx).cpu().numpy(), w2[0])
    assert np.array_equal(l2.index_select(0, idx).cpu().numpy()[..., : w2[1].shape[-1]], w2[1])
    S_x = {"w4a4": orc.tensor_scale, "w4a8": orc.fp8_tensor_scale}[mode](x_np) if mode in ("w4a4", "w4a8") else None
    if S_x is not None:
        assert float(d["S_x"].item()) == float(S_x)
    S_h = {"w4a4": cfg.S_h, "w4a8": cfg.S_h8}.get(mode, 0.0)
    ref, mids = orc.moe_layer(mode, x_np[tokens], lg_np[tokens][:, used], k, w13, w2, S_h,
                              intermediates=True, S_x=S_x)
    # routing: the GPU's ids (global expert numbers) are the oracle's
    ids_g = d["rt"]["ids"].cpu().numpy()[tokens]
    assert np.array_equal(ids_g, used[mids["ids"]])
    got = d["out"].cpu().numpy()[tokens].astype(np.float64)
    inv_g = d["rt"]["inv"].cpu().numpy().reshape(T, k)
    inv_o = mids["inv"].reshape(len(tokens), k)
    w_tok = mids["w"].reshape(len(tokens), k)
    figs = {"config": cfg.name, "mode": mode, "tokens": int(len(tokens))}
    flipped = {}
    if hfmt is not None:
        hc_g = d["hc"].cpu().numpy()
        rows_g = inv_g[tokens].ravel()
        rows_o = inv_o.ravel()
        h32 = mids["h32"][rows_o]
        dist_fn = {"nvfp4": lambda v: nvfp4_boundary_distance(v, S_h), "mx": mx_boundary_distance,
                   "fp8": lambda v: fp8_boundary_distance(v, S_h)}[hfmt]
        d_o = np.concatenate([dist_fn(h32[r:r + 256]) for r in range(0, len(rows_o), 256)])
        if hfmt == "fp8":
            hs_g = hs_o = None
            diff = hc_g[rows_g] != mids["hq_codes"][rows_o]
        else:
            hs_g = d["hs"].cpu().numpy()[:, : (I // 16 if hfmt == "nvfp4" else I // 32)]
            hs_o = mids["hq_scales"]
            cg = unpack_codes(hc_g[rows_g])
            co = unpack_codes(mids["hq_codes"][rows_o])
            diff = (cg != co) | np.repeat(hs_g[rows_g] != hs_o[rows_o], 16 if hfmt == "nvfp4" else 32, 1)
        # pre-rounding difference of h, from the GPU's own fp32 G (the host's
        # fp32 SwiGLU of it; the GPU's own expf may differ by an ulp or two)
        h_g = _silu_mul_f32(d["G"].cpu().numpy()[rows_g], I).astype(np.float64)
        h_o = mids["h32"][rows_o].astype(np.float64)
        relh = np.abs(h_g - h_o) / np.maximum(np.abs(h_o), 1e-30)
        big = np.abs(h_o) > 1e-6 * np.abs(h_o).max()
        q = np.quantile(relh[big], [0.5, 0.99, 0.9999, 1.0])
        figs["h_rel_diff_quantiles"] = {"p50": q[0], "p99": q[1], "p99.99": q[2], "max": q[3]}
        figs["h_elements"] = int(diff.size)
        figs["h_code_flips"] = int(diff.sum())
        figs["flip_max_boundary_distance"] = float(d_o[diff].max()) if diff.any() else 0.0
        # a code may differ where the oracle's h lies within FLIP_WINDOW of the
        # boundary, or within the measured pre-rounding difference at that
        # element (which the boundary then lies between, up to ulp slack)
        legit = (d_o <= FLIP_WINDOW) | (d_o <= 2.0 * relh + 1e-6)
        figs["flips_beyond_window"] = int((diff & (d_o > FLIP_WINDOW)).sum())
        assert not (diff & ~legit).any(), \
            "h code differs where the oracle's h is %.3e (relative) from a boundary and the GPU's pre-rounding h " \
            "only %.3e away" % (d_o[diff & ~legit].max(), relh[diff & ~legit].max())
        if diff.any():
            dec_g = _decode_h(hc_g[rows_g], None if hs_g is None else hs_g[rows_g], hfmt, S_h)
            dec_o = _decode_h(mids["hq_codes"][rows_o], None if hs_o is None else hs_o[rows_o], hfmt, S_h)
            dh = np.abs(dec_g - dec_o) * diff
            dh = dh.reshape(len(tokens), k, I)
            for i in np.nonzero(dh.reshape(len(tokens), -1).any(1))[0]:
                bound = np.zeros(H)
                for j in range(k):
                    cols = np.nonzero(dh[i, j])[0]
                    if cols.size:
                        e_local = mids["ids"][i, j]
                        bound += w_tok[i, j] * (_w2_columns(w2, e_local, cols, fmt) @ dh[i, j, cols])
                flipped[int(i)] = bound
    rel_all, _ = errors(got, ref)
    assert rel_all <= REL_FROB_TOL, rel_all
    worst_rel, worst_mx, worst_flip_excess = 0.0, 0.0, 0.0
    for i in range(len(tokens)):
        rel, mx = errors(got[i], ref[i])
        assert np.isfinite(got[i]).all()
        rms = np.sqrt(np.mean(ref[i] ** 2))
        if i in flipped:
            excess = np.abs(got[i] - ref[i]) - flipped[i]
            assert (excess <= MAX_ERR_RMS_TOL * rms).all(), \
                "token %d: error %.3e x RMS beyond the flip bound" % (tokens[i], excess.max() / rms)
            worst_flip_excess = max(worst_flip_excess, float(excess.max() / rms))
            continue
        assert rel <= REL_FROB_TOL and mx <= MAX_ERR_RMS_TOL, \
            "token %d: rel_frob=%.3e max/rms=%.3e" % (tokens[i], rel, mx)
        worst_rel, worst_mx = max(worst_rel, rel), max(worst_mx, mx)
    figs.update(rel_frob_all=rel_all, worst_token_rel_frob=worst_rel, worst_token_max_over_rms=worst_mx,
                flipped_tokens=len(flipped), worst_flipped_excess_over_rms=worst_flip_excess)
    print("LAYER-PARITY", figs)
    return figs
