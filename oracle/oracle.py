"""ctypes binding of the C oracle (``nvfp4moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the checker the CUDA path is compared against.
Arrays are numpy; every function returns fresh numpy arrays.  The math lives
in the C file; this module only marshals arguments.
"""
import ctypes as C

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = C.CDLL(path)
        _declare(_lib)
    return _lib


_P = C.c_void_p
_I64 = C.c_int64


def _declare(L):
    L.orc_e2m1_value.restype = C.c_double
    L.orc_e2m1_value.argtypes = [C.c_int]
    L.orc_e4m3_value.restype = C.c_double
    L.orc_e4m3_value.argtypes = [C.c_int]
    L.orc_e4m3_encode.restype = C.c_int
    L.orc_e4m3_encode.argtypes = [C.c_float]
    L.orc_e2m1_encode.restype = C.c_int
    L.orc_e2m1_encode.argtypes = [C.c_float]
    L.orc_round_bf16.restype = C.c_float
    L.orc_round_bf16.argtypes = [C.c_float]
    L.orc_tensor_scale.restype = C.c_float
    L.orc_tensor_scale.argtypes = [_P, _I64, _I64, _I64]
    L.orc_quantize_block.restype = None
    L.orc_quantize_block.argtypes = [_P, C.c_float, _P, _P]
    L.orc_quantize.restype = None
    L.orc_quantize.argtypes = [_P, _I64, _I64, _I64, C.c_int, _P, _P, _P]
    L.orc_dequantize.restype = None
    L.orc_dequantize.argtypes = [_P, _P, C.c_float, _I64, _I64, _P]
    L.orc_route.restype = None
    L.orc_route.argtypes = [_P, C.c_int, C.c_int, C.c_int, _P, _P]
    L.orc_permute.restype = None
    L.orc_permute.argtypes = [_P, C.c_int, C.c_int, C.c_int, _P, _P, _P]
    L.orc_grouped_gemm_w4a4.restype = None
    L.orc_grouped_gemm_w4a4.argtypes = [_P, _P, C.c_float, _P, _P, _P, _P, C.c_int, C.c_int, C.c_int, _P]
    L.orc_grouped_gemm_w4a16.restype = None
    L.orc_grouped_gemm_w4a16.argtypes = [_P, _P, _P, _P, _P, C.c_int, C.c_int, C.c_int, _P]
    L.orc_swiglu.restype = None
    L.orc_swiglu.argtypes = [_P, _I64, _I64, _P]
    L.orc_combine.restype = None
    L.orc_combine.argtypes = [_P, _P, _P, C.c_int, C.c_int, _I64, _P]
    layer_args = [C.c_int, _P, _P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                  _P, _P, _P, _P, _P, _P, C.c_float, _P, _P]
    L.orc_moe_layer.restype = None
    L.orc_moe_layer.argtypes = layer_args + [_P] * 9
    L.orc_moe_layer_naive.restype = None
    L.orc_moe_layer_naive.argtypes = layer_args
    L.orc_num_threads.restype = C.c_int
    L.orc_num_threads.argtypes = []
    L.orc_ue8m0_value.restype = C.c_double
    L.orc_ue8m0_value.argtypes = [C.c_int]
    L.orc_mx_quantize_block.restype = None
    L.orc_mx_quantize_block.argtypes = [_P, _P, _P]
    L.orc_mx_quantize.restype = None
    L.orc_mx_quantize.argtypes = [_P, _I64, _I64, _I64, _P, _P]
    L.orc_mx_dequantize.restype = None
    L.orc_mx_dequantize.argtypes = [_P, _P, _I64, _I64, _P]
    L.orc_router_logits.restype = None
    L.orc_router_logits.argtypes = [_P, _P, C.c_int, C.c_int, C.c_int, _P]
    L.orc_fp8_encode.restype = C.c_int
    L.orc_fp8_encode.argtypes = [C.c_float]
    L.orc_fp8_tensor_scale.restype = C.c_float
    L.orc_fp8_tensor_scale.argtypes = [_P, _I64, _I64, _I64]
    L.orc_fp8_quantize.restype = None
    L.orc_fp8_quantize.argtypes = [_P, _I64, _I64, _I64, C.c_int, _P, _P]
    L.orc_grouped_gemm_w4a8.restype = None
    L.orc_grouped_gemm_w4a8.argtypes = [_P, C.c_float, _P, _P, _P, _P, C.c_int, C.c_int, C.c_int, _P]
    L.orc_grouped_gemm_mx.restype = None
    L.orc_grouped_gemm_mx.argtypes = [_P, _P, _P, _P, _P, C.c_int, C.c_int, C.c_int, _P]


def _c(a, dtype):
    """Contiguous array of the given dtype (copy only if needed)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


# --------------------------------------------------------------------------
# scalar format helpers
# --------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def e4m3_encode(b: float) -> int:
    return lib().orc_e4m3_encode(float(np.float32(b)))


def e2m1_encode(q: float) -> int:
    return lib().orc_e2m1_encode(float(np.float32(q)))


def round_bf16(v: float) -> float:
    return float(lib().orc_round_bf16(float(np.float32(v))))


def ue8m0_value(code: int) -> float:
    return lib().orc_ue8m0_value(int(code))


def num_threads() -> int:
    return lib().orc_num_threads()


# --------------------------------------------------------------------------
# array functions
# --------------------------------------------------------------------------

def tensor_scale(x) -> np.float32:
    x = _c(x, np.float32)
    rows, cols = x.shape
    return np.float32(lib().orc_tensor_scale(_p(x), rows, cols, cols))


def quantize(x, S=None):
    """NVFP4-quantise x [rows, cols]. S=None: dynamic (S = amax/2688).
    Returns (codes uint8 [rows, cols/2], scales uint8 [rows, cols/16], S)."""
    x = _c(x, np.float32)
    rows, cols = x.shape
    assert cols % 16 == 0
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 16), np.uint8)
    s = np.zeros(1, np.float32)
    if S is not None:
        s[0] = np.float32(S)
    lib().orc_quantize(_p(x), rows, cols, cols, 0 if S is not None else 1, _p(s), _p(codes), _p(scales))
    return codes, scales, np.float32(s[0])


def quantize_block(xb, S):
    xb = _c(xb, np.float32)
    assert xb.shape == (16,)
    sc = np.zeros(1, np.uint8)
    ec = np.zeros(16, np.uint8)
    lib().orc_quantize_block(_p(xb), float(np.float32(S)), _p(sc), _p(ec))
    return int(sc[0]), ec


def dequantize(codes, scales, S, cols):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows = codes.shape[0]
    out = np.zeros((rows, cols), np.float64)
    lib().orc_dequantize(_p(codes), _p(scales), float(np.float32(S)), rows, cols, _p(out))
    return out


def fp8_encode(q: float) -> int:
    return lib().orc_fp8_encode(float(np.float32(q)))


def fp8_tensor_scale(x) -> np.float32:
    x = _c(x, np.float32)
    rows, cols = x.shape
    return np.float32(lib().orc_fp8_tensor_scale(_p(x), rows, cols, cols))


def fp8_quantize(x, S=None):
    """FP8 (E4M3) quantisation of x [rows, cols] with one per-tensor decode
    scale.  S=None: dynamic (S = amax/448).  Returns (codes uint8 [rows,
    cols], S)."""
    x = _c(x, np.float32)
    rows, cols = x.shape
    codes = np.zeros((rows, cols), np.uint8)
    s = np.zeros(1, np.float32)
    if S is not None:
        s[0] = np.float32(S)
    lib().orc_fp8_quantize(_p(x), rows, cols, cols, 0 if S is not None else 1, _p(s), _p(codes))
    return codes, np.float32(s[0])


def mx_quantize(x):
    """MXFP4-quantise x [rows, cols] (cols a multiple of 32).  Returns
    (codes uint8 [rows, cols/2], scales uint8 [rows, cols/32])."""
    x = _c(x, np.float32)
    rows, cols = x.shape
    assert cols % 32 == 0
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 32), np.uint8)
    lib().orc_mx_quantize(_p(x), rows, cols, cols, _p(codes), _p(scales))
    return codes, scales


def mx_quantize_block(xb):
    xb = _c(xb, np.float32)
    assert xb.shape == (32,)
    sc = np.zeros(1, np.uint8)
    ec = np.zeros(32, np.uint8)
    lib().orc_mx_quantize_block(_p(xb), _p(sc), _p(ec))
    return int(sc[0]), ec


def mx_dequantize(codes, scales, cols):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows = codes.shape[0]
    out = np.zeros((rows, cols), np.float64)
    lib().orc_mx_dequantize(_p(codes), _p(scales), rows, cols, _p(out))
    return out


def mx_quantize_experts(w):
    """MXFP4-quantise a stack of expert weight matrices w [E, N, K].  Returns
    (codes [E, N, K/2], scales [E, N, K/32], None) -- the format has no
    per-tensor scale."""
    w = np.asarray(w, np.float32)
    E, N, K = w.shape
    codes = np.zeros((E, N, K // 2), np.uint8)
    scales = np.zeros((E, N, K // 32), np.uint8)
    for e in range(E):
        codes[e], scales[e] = mx_quantize(w[e])
    return codes, scales, None


def router_logits(x, w):
    """logits [T, E] (fp32) = x [T, H] . w [E, H]^T, summed in fp64."""
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    T, H = x.shape
    E = w.shape[0]
    out = np.zeros((T, E), np.float32)
    lib().orc_router_logits(_p(x), _p(w), T, H, E, _p(out))
    return out


def route(logits, k):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    lib().orc_route(_p(logits), T, E, k, _p(ids), _p(w))
    return ids, w


def permute(ids, E):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    inv = np.zeros(T * k, np.int32)
    lib().orc_permute(_p(ids), T, E, k, _p(offsets), _p(perm), _p(inv))
    return offsets, perm, inv


def grouped_gemm_w4a4(a_codes, a_scales, S_a, w_codes, w_scales, w_S, offsets):
    a_codes = _c(a_codes, np.uint8)
    a_scales = _c(a_scales, np.uint8)
    w_codes = _c(w_codes, np.uint8)
    w_scales = _c(w_scales, np.uint8)
    w_S = _c(w_S, np.float32)
    offsets = _c(offsets, np.int32)
    E, N, Kh = w_codes.shape
    K = 2 * Kh
    R = int(offsets[E])
    out = np.zeros((R, N), np.float64)
    lib().orc_grouped_gemm_w4a4(_p(a_codes), _p(a_scales), float(np.float32(S_a)), _p(w_codes), _p(w_scales),
                                _p(w_S), _p(offsets), E, N, K, _p(out))
    return out


def grouped_gemm_w4a16(a, w_codes, w_scales, w_S, offsets):
    a = _c(a, np.float32)
    w_codes = _c(w_codes, np.uint8)
    w_scales = _c(w_scales, np.uint8)
    w_S = _c(w_S, np.float32)
    offsets = _c(offsets, np.int32)
    E, N, Kh = w_codes.shape
    K = 2 * Kh
    R = int(offsets[E])
    out = np.zeros((R, N), np.float64)
    lib().orc_grouped_gemm_w4a16(_p(a), _p(w_codes), _p(w_scales), _p(w_S), _p(offsets), E, N, K, _p(out))
    return out


def grouped_gemm_w4a8(a_codes, S_a, w_codes, w_scales, w_S, offsets):
    """FP8 activations [R, K] x NVFP4 weights, fp64 [R, N]."""
    a_codes = _c(a_codes, np.uint8)
    w_codes = _c(w_codes, np.uint8)
    w_scales = _c(w_scales, np.uint8)
    w_S = _c(w_S, np.float32)
    offsets = _c(offsets, np.int32)
    E, N = w_codes.shape[0], w_codes.shape[1]
    K = a_codes.shape[1]
    out = np.zeros((int(offsets[-1]), N), np.float64)
    lib().orc_grouped_gemm_w4a8(_p(a_codes), float(np.float32(S_a)), _p(w_codes), _p(w_scales), _p(w_S),
                                _p(offsets), E, N, K, _p(out))
    return out


def grouped_gemm_mx(a_codes, a_scales, w_codes, w_scales, offsets):
    a_codes = _c(a_codes, np.uint8)
    a_scales = _c(a_scales, np.uint8)
    w_codes = _c(w_codes, np.uint8)
    w_scales = _c(w_scales, np.uint8)
    offsets = _c(offsets, np.int32)
    E, N, Kh = w_codes.shape
    K = 2 * Kh
    R = int(offsets[E])
    out = np.zeros((R, N), np.float64)
    lib().orc_grouped_gemm_mx(_p(a_codes), _p(a_scales), _p(w_codes), _p(w_scales), _p(offsets), E, N, K, _p(out))
    return out


def swiglu(G):
    G = _c(G, np.float32)
    R, I2 = G.shape
    h = np.zeros((R, I2 // 2), np.float64)
    lib().orc_swiglu(_p(G), R, I2 // 2, _p(h))
    return h


def combine(Y, inv, w):
    Y = _c(Y, np.float32)
    w = _c(w, np.float64)
    inv = _c(inv, np.int32)
    T, k = w.shape
    H = Y.shape[1]
    out = np.zeros((T, H), np.float64)
    lib().orc_combine(_p(Y), _p(inv), _p(w), T, k, H, _p(out))
    return out


_MODES = {"w4a4": 0, "w4a16": 1, "mxw4a4": 2, "w4a8": 3}


def _weights(w13, w2):
    """Contiguous (codes, scales, S) of both projections; a missing S (MXFP4)
    becomes ones, which the oracle does not read in that mode."""
    def one(w):
        c = _c(w[0], np.uint8)
        S = np.ones(c.shape[0], np.float32) if w[2] is None else _c(w[2], np.float32)
        return c, _c(w[1], np.uint8), S
    return one(w13) + one(w2)


def _sx(S_x):
    return None if S_x is None else np.array([S_x], np.float32)


def moe_layer(mode, x, logits, k, w13, w2, S_h, intermediates=False, S_x=None):
    """Full layer.  mode: 'w4a4' | 'w4a16' | 'mxw4a4' | 'w4a8'.  w13 / w2:
    (codes, scales, S[E]); for 'mxw4a4' the scales are UE8M0 per 32 and S is
    None.  'w4a8': S_h is the static FP8 decode scale of h, and hq_codes are
    FP8 codes [R, I].
    S_x: None = dynamic activation scale of x; else the given scale (for a
    sample of rows of a larger batch).  Returns out fp64 [T, H] (and a dict
    of intermediates if asked)."""
    x = _c(x, np.float32)
    logits = _c(logits, np.float32)
    T, H = x.shape
    E = logits.shape[1]
    c13, s13, S13, c2, s2, S2 = _weights(w13, w2)
    I = c2.shape[2] * 2
    R = T * k
    out = np.zeros((T, H), np.float64)
    m = _MODES[mode]
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(R, np.int32)
    inv = np.zeros(R, np.int32)
    S_x_out = np.zeros(1, np.float32)
    hq_c = np.zeros((R, I if m == 3 else I // 2), np.uint8)
    hq_s = np.zeros((R, I // (32 if m == 2 else 16)), np.uint8)
    h32 = np.zeros((R, I), np.float32)
    sx = _sx(S_x)
    lib().orc_moe_layer(m, _p(x), _p(logits), T, H, I, E, k, _p(c13), _p(s13), _p(S13), _p(c2), _p(s2), _p(S2),
                        float(np.float32(S_h)), _p(sx), _p(out), _p(ids), _p(w), _p(offsets), _p(perm), _p(inv), _p(S_x_out),
                        _p(hq_c), _p(hq_s), _p(h32))
    if not intermediates:
        return out
    return out, dict(ids=ids, w=w, offsets=offsets, perm=perm, inv=inv, S_x=np.float32(S_x_out[0]),
                     hq_codes=hq_c, hq_scales=hq_s, h32=h32)


def moe_layer_naive(mode, x, logits, k, w13, w2, S_h, S_x=None):
    x = _c(x, np.float32)
    logits = _c(logits, np.float32)
    T, H = x.shape
    E = logits.shape[1]
    c13, s13, S13, c2, s2, S2 = _weights(w13, w2)
    I = c2.shape[2] * 2
    out = np.zeros((T, H), np.float64)
    m = _MODES[mode]
    sx = _sx(S_x)
    lib().orc_moe_layer_naive(m, _p(x), _p(logits), T, H, I, E, k, _p(c13), _p(s13), _p(S13), _p(c2), _p(s2),
                              _p(S2), float(np.float32(S_h)), _p(sx), _p(out))
    return out


def quantize_experts(w):
    """Quantise a stack of expert weight matrices w [E, N, K] one expert at a
    time, each with its own dynamic per-tensor scale.  Returns (codes
    [E, N, K/2], scales [E, N, K/16], S [E])."""
    w = np.asarray(w, np.float32)
    E, N, K = w.shape
    codes = np.zeros((E, N, K // 2), np.uint8)
    scales = np.zeros((E, N, K // 16), np.uint8)
    S = np.zeros(E, np.float32)
    for e in range(E):
        codes[e], scales[e], S[e] = quantize(w[e])
    return codes, scales, S
