"""Thin Python binding of ``libnvfp4moe.so`` (the C ABI in include/nvfp4moe.h).

Each function has the name of its C entry point, takes torch tensors that
already live on the GPU, passes their data pointers and the current CUDA
stream, and raises ``Nvfp4Error`` if the library returns a status other than
NVFP4_OK.  Every computation runs in the library's kernels; this module only
marshals arguments and allocates outputs with torch.  There is no fallback:
if the library cannot be loaded, importing the functions raises.
"""
import ctypes as C
import os

import torch

from . import build as _build

NVFP4_OK = 0
NVFP4_DT_BF16, NVFP4_DT_F32 = 0, 1
NVFP4_SCALE_STATIC, NVFP4_SCALE_DYNAMIC = 0, 1
MOE_W4A4, MOE_W4A16, MOE_MXW4A4, MOE_W4A8, MOE_W4A16F = 0, 1, 2, 3, 4
MOE_ACT_NONE, MOE_ACT_NVFP4, MOE_ACT_BF16 = 0, 1, 2
STATUS_NAMES = {0: "NVFP4_OK", 1: "NVFP4_E_INVAL", 2: "NVFP4_E_SHAPE", 3: "NVFP4_E_ALIGN", 4: "NVFP4_E_WORKSPACE",
                5: "NVFP4_E_ARCH", 6: "NVFP4_E_CUDA", 7: "NVFP4_E_DEVICE_TIMEOUT", 8: "NVFP4_E_BAD_ROUTING"}

# every symbol the header declares, in declaration order
EXPORTS = ("nvfp4_status_string", "nvfp4_device_check", "nvfp4_quantize_workspace_bytes", "nvfp4_quantize",
           "nvfp4_pack_weight_scales", "moe_align_permute_workspace_bytes", "moe_align_permute",
           "moe_grouped_gemm_nvfp4", "moe_swiglu_requant", "moe_combine", "moe_layer_workspace_bytes",
           "moe_layer_forward", "moe_align_permute_noalloc", "moe_route_quantize_nvfp4", "mxfp4_scale_pitch",
           "mxfp4_quantize", "mxfp4_pack_weight_scales", "moe_route_quantize_mxfp4",
           "moe_router_logits_workspace_bytes", "moe_router_logits", "moe_layer_host_workspace_bytes",
           "moe_layer_forward_host", "fp8_quantize", "moe_route_quantize_fp8", "moe_router_route_workspace_bytes",
           "moe_router_route", "moe_gather_f16", "moe_swiglu_f16", "moe_route_quantize_fp8_f16",
           "moe_swiglu_fp8_f16")


class Nvfp4Error(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s" % (fn, STATUS_NAMES.get(status, status)))


_lib = None

_P, _I, _I64, _SZ = C.c_void_p, C.c_int, C.c_int64, C.c_size_t


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load the library (building it in-tree first if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError("libnvfp4moe.so is not built (%s); run __graft_entry__.build()" % path)
    L = C.CDLL(path)
    L.nvfp4_status_string.restype = C.c_char_p
    L.nvfp4_status_string.argtypes = [_I]
    L.nvfp4_device_check.restype = _I
    L.nvfp4_device_check.argtypes = []
    L.nvfp4_quantize_workspace_bytes.restype = _SZ
    L.nvfp4_quantize_workspace_bytes.argtypes = [_I64, _I64]
    L.nvfp4_quantize.restype = _I
    L.nvfp4_quantize.argtypes = [_P, _I, _I64, _I64, _I64, _P, _I, _P, _P, _P, _SZ, _P]
    L.nvfp4_pack_weight_scales.restype = _I
    L.nvfp4_pack_weight_scales.argtypes = [_P, _I, _I, _I, _P, _P]
    L.moe_align_permute_workspace_bytes.restype = _SZ
    L.moe_align_permute_workspace_bytes.argtypes = [_I, _I, _I]
    L.moe_align_permute.restype = _I
    L.moe_align_permute.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _I64, _P, _P, _P, _P, _SZ, _P]
    L.moe_grouped_gemm_nvfp4.restype = _I
    L.moe_grouped_gemm_nvfp4.argtypes = [_I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P]
    L.moe_swiglu_requant.restype = _I
    L.moe_swiglu_requant.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P]
    L.moe_combine.restype = _I
    L.moe_combine.argtypes = [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P]
    L.moe_layer_workspace_bytes.restype = _SZ
    L.moe_layer_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I]
    L.moe_layer_forward.restype = _I
    L.moe_layer_forward.argtypes = [_I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_layer_host_workspace_bytes.restype = _SZ
    L.moe_layer_host_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I]
    L.moe_layer_forward_host.restype = _I
    L.moe_layer_forward_host.argtypes = [_I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                         _P]
    L.moe_route_quantize_nvfp4.restype = _I
    L.moe_route_quantize_nvfp4.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_align_permute_noalloc.restype = _I
    L.moe_align_permute_noalloc.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _I64, _P, _P, _P, _P]
    L.moe_router_logits_workspace_bytes.restype = _SZ
    L.moe_router_logits_workspace_bytes.argtypes = [_I, _I, _I]
    L.moe_router_logits.restype = _I
    L.moe_router_logits.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P, _SZ, _P]
    L.mxfp4_scale_pitch.restype = _I64
    L.mxfp4_scale_pitch.argtypes = [_I64]
    L.mxfp4_quantize.restype = _I
    L.mxfp4_quantize.argtypes = [_P, _I, _I64, _I64, _I64, _P, _P, _P]
    L.mxfp4_pack_weight_scales.restype = _I
    L.mxfp4_pack_weight_scales.argtypes = [_P, _I, _I, _I, _P, _P]
    L.moe_route_quantize_mxfp4.restype = _I
    L.moe_route_quantize_mxfp4.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_router_route_workspace_bytes.restype = _SZ
    L.moe_router_route_workspace_bytes.argtypes = [_I, _I, _I, _I]
    L.moe_router_route.restype = _I
    L.moe_router_route.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_gather_f16.restype = _I
    L.moe_gather_f16.argtypes = [_P, _I, _I, _P, _I, _P, _P, _P]
    L.moe_swiglu_f16.restype = _I
    L.moe_swiglu_f16.argtypes = [_P, _I, _I, _P, _P, _P]
    L.moe_route_quantize_fp8_f16.restype = _I
    L.moe_route_quantize_fp8_f16.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.moe_swiglu_fp8_f16.restype = _I
    L.moe_swiglu_fp8_f16.argtypes = [_P, _I, _I, _P, _P, _P, _P]
    L.fp8_quantize.restype = _I
    L.fp8_quantize.argtypes = [_P, _I, _I64, _I64, _I64, _P, _I, _P, _P, _SZ, _P]
    L.moe_route_quantize_fp8.restype = _I
    L.moe_route_quantize_fp8.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return C.c_void_p(t.data_ptr())


def _hptr(t):
    if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
        raise ValueError("expected a contiguous page-locked (pinned) CPU tensor")
    return C.c_void_p(t.data_ptr())


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn, status):
    if status != NVFP4_OK:
        raise Nvfp4Error(fn, status)


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


# ---------------------------------------------------------------------------
# entry points (names as in the C ABI)
# ---------------------------------------------------------------------------

def nvfp4_device_check():
    _check("nvfp4_device_check", load().nvfp4_device_check())


def nvfp4_quantize(x, S=None, codes=None, scales=None, workspace=None):
    """Quantise x [rows, cols] (bf16 or fp32, CUDA) to NVFP4.  S=None ->
    dynamic scale (returned as a 1-element fp32 tensor); otherwise S is a
    1-element fp32 CUDA tensor read as the static decode scale."""
    L = load()
    rows, cols = x.shape
    dev = x.device
    dt = NVFP4_DT_BF16 if x.dtype == torch.bfloat16 else NVFP4_DT_F32
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("x must be bf16 or fp32")
    dynamic = S is None
    if dynamic:
        S = torch.zeros(4, dtype=torch.float32, device=dev)
    if codes is None:
        codes = _empty((rows, cols // 2), torch.uint8, dev)
    if scales is None:
        scales = _empty((rows, cols // 16), torch.uint8, dev)
    if dynamic and workspace is None:
        workspace = _empty(int(L.nvfp4_quantize_workspace_bytes(rows, cols)), torch.uint8, dev)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("nvfp4_quantize", L.nvfp4_quantize(_ptr(x), dt, rows, cols, x.stride(0), _ptr(S),
                                              NVFP4_SCALE_DYNAMIC if dynamic else NVFP4_SCALE_STATIC, _ptr(codes),
                                              _ptr(scales), _ptr(workspace), ws_bytes, _stream()))
    return codes, scales, S[:1]


def nvfp4_pack_weight_scales(scales_linear, E, N, K, out=None):
    L = load()
    if out is None:
        out = _empty(E * N * (K // 16), torch.uint8, scales_linear.device)
    _check("nvfp4_pack_weight_scales",
           L.nvfp4_pack_weight_scales(_ptr(scales_linear), E, N, K, _ptr(out), _stream()))
    return out


def mxfp4_scale_pitch(cols):
    return int(load().mxfp4_scale_pitch(cols))


def mxfp4_quantize(x, codes=None, scales=None):
    """Quantise x [rows, cols] (bf16 or fp32, CUDA) to MXFP4.  Returns (codes
    [rows, cols/2], scales [rows, mxfp4_scale_pitch(cols)])."""
    L = load()
    rows, cols = x.shape
    dev = x.device
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("x must be bf16 or fp32")
    dt = NVFP4_DT_BF16 if x.dtype == torch.bfloat16 else NVFP4_DT_F32
    if codes is None:
        codes = _empty((rows, cols // 2), torch.uint8, dev)
    if scales is None:
        scales = _empty((rows, mxfp4_scale_pitch(cols)), torch.uint8, dev)
    _check("mxfp4_quantize", L.mxfp4_quantize(_ptr(x), dt, rows, cols, x.stride(0), _ptr(codes), _ptr(scales),
                                              _stream()))
    return codes, scales


def mxfp4_pack_weight_scales(scales_linear, E, N, K, out=None):
    L = load()
    if out is None:
        out = _empty(E * N * (K // 32), torch.uint8, scales_linear.device)
    _check("mxfp4_pack_weight_scales",
           L.mxfp4_pack_weight_scales(_ptr(scales_linear), E, N, K, _ptr(out), _stream()))
    return out


def moe_router_logits(x, w_router, out=None, workspace=None, dev_status=None):
    """logits [T, E] fp32 = x [T, H] bf16 . w_router [E, H] bf16 ^T."""
    L = load()
    T, H = x.shape
    E = w_router.shape[0]
    if out is None:
        out = _empty((T, E), torch.float32, x.device)
    if workspace is None:
        workspace = _empty(int(L.moe_router_logits_workspace_bytes(T, H, E)), torch.uint8, x.device)
    _check("moe_router_logits", L.moe_router_logits(_ptr(x), _ptr(w_router), T, H, E, _ptr(out), _ptr(dev_status),
                                                    _ptr(workspace), workspace.numel(), _stream()))
    return out


def moe_router_route(x, w_router, k, want_logits=True, dev_status=None, workspace=None):
    """Router logits + top-k + permutation of x [T, H] bf16 with w_router
    [E, H] bf16.  Returns dict(ids, w, offsets, perm, inv[, logits])."""
    L = load()
    T, H = x.shape
    E = w_router.shape[0]
    dev = x.device
    R = T * k
    out = dict(ids=_empty((T, k), torch.int32, dev), w=_empty((T, k), torch.float32, dev),
               offsets=_empty((E + 1,), torch.int32, dev), perm=_empty((max(R, 1),), torch.int32, dev),
               inv=_empty((max(R, 1),), torch.int32, dev))
    if want_logits:
        out["logits"] = _empty((T, E), torch.float32, dev)
    if workspace is None:
        workspace = _empty(max(int(L.moe_router_route_workspace_bytes(T, H, E, k)), 256), torch.uint8, dev)
    _check("moe_router_route",
           L.moe_router_route(_ptr(x), _ptr(w_router), T, H, E, k, _ptr(out.get("logits")), _ptr(out["ids"]),
                              _ptr(out["w"]), _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["inv"]),
                              _ptr(dev_status), _ptr(workspace), workspace.numel(), _stream()))
    out["perm"], out["inv"] = out["perm"][:R], out["inv"][:R]
    return out


def moe_align_permute(logits, k, act=None, act_kind=MOE_ACT_NONE, dev_status=None):
    """Route + permute.  act: None, (codes, scales) for NVFP4 rows, or a bf16
    [T, H] tensor.  Returns dict(ids, w, offsets, perm, inv[, act_codes,
    act_scales | act_bf16])."""
    L = load()
    T, E = logits.shape
    dev = logits.device
    R = T * k
    ids = _empty((T, k), torch.int32, dev)
    w = _empty((T, k), torch.float32, dev)
    offsets = _empty((E + 1,), torch.int32, dev)
    perm = _empty((max(R, 1),), torch.int32, dev)
    inv = _empty((max(R, 1),), torch.int32, dev)
    ws = _empty(max(int(L.moe_align_permute_workspace_bytes(T, E, k)), 256), torch.uint8, dev)
    out = dict(ids=ids, w=w, offsets=offsets, perm=perm[:R], inv=inv[:R])
    a_in = a_in_sc = a_out = a_out_sc = None
    cols = 0
    if act_kind == MOE_ACT_NVFP4:
        a_in, a_in_sc = act
        cols = a_in.shape[1] * 2
        a_out = _empty((max(R, 1), cols // 2), torch.uint8, dev)
        a_out_sc = _empty((max(R, 1), cols // 16), torch.uint8, dev)
        out["act_codes"], out["act_scales"] = a_out[:R], a_out_sc[:R]
    elif act_kind == MOE_ACT_BF16:
        a_in = act
        cols = a_in.shape[1]
        a_out = _empty((max(R, 1), cols), torch.bfloat16, dev)
        out["act_bf16"] = a_out[:R]
    _check("moe_align_permute",
           L.moe_align_permute(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _ptr(offsets), _ptr(perm), _ptr(inv),
                               act_kind, _ptr(a_in), _ptr(a_in_sc), cols, _ptr(a_out), _ptr(a_out_sc),
                               _ptr(dev_status), _ptr(ws), ws.numel(), _stream()))
    return out


def moe_route_quantize_nvfp4(x, logits, k, dev_status=None):
    """Routing + NVFP4 quantisation of x [T, H] bf16 written in permuted order.
    Returns dict(ids, w, offsets, perm, inv, S_x, act_codes, act_scales)."""
    L = load()
    T, H = x.shape
    E = logits.shape[1]
    dev = x.device
    R = T * k
    out = dict(ids=_empty((T, k), torch.int32, dev), w=_empty((T, k), torch.float32, dev),
               offsets=_empty((E + 1,), torch.int32, dev), perm=_empty((max(R, 1),), torch.int32, dev),
               inv=_empty((max(R, 1),), torch.int32, dev), S_x=torch.zeros(4, dtype=torch.float32, device=dev),
               act_codes=_empty((max(R, 1), H // 2), torch.uint8, dev),
               act_scales=_empty((max(R, 1), H // 16), torch.uint8, dev))
    ws = _empty(max(int(L.moe_align_permute_workspace_bytes(T, E, k)), 256), torch.uint8, dev)
    _check("moe_route_quantize_nvfp4",
           L.moe_route_quantize_nvfp4(_ptr(x), _ptr(logits), T, H, E, k, _ptr(out["ids"]), _ptr(out["w"]),
                                      _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["inv"]), _ptr(out["S_x"]),
                                      _ptr(out["act_codes"]), _ptr(out["act_scales"]), _ptr(dev_status), _ptr(ws),
                                      ws.numel(), _stream()))
    for key in ("perm", "inv", "act_codes", "act_scales"):
        out[key] = out[key][:R]
    out["S_x"] = out["S_x"][:1]
    return out


def moe_route_quantize_mxfp4(x, logits, k, dev_status=None):
    """Routing + MXFP4 quantisation of x [T, H] bf16 written in permuted order.
    Returns dict(ids, w, offsets, perm, inv, act_codes, act_scales)."""
    L = load()
    T, H = x.shape
    E = logits.shape[1]
    dev = x.device
    R = T * k
    out = dict(ids=_empty((T, k), torch.int32, dev), w=_empty((T, k), torch.float32, dev),
               offsets=_empty((E + 1,), torch.int32, dev), perm=_empty((max(R, 1),), torch.int32, dev),
               inv=_empty((max(R, 1),), torch.int32, dev),
               act_codes=_empty((max(R, 1), H // 2), torch.uint8, dev),
               act_scales=_empty((max(R, 1), mxfp4_scale_pitch(H)), torch.uint8, dev))
    ws = _empty(max(int(L.moe_align_permute_workspace_bytes(T, E, k)), 256), torch.uint8, dev)
    _check("moe_route_quantize_mxfp4",
           L.moe_route_quantize_mxfp4(_ptr(x), _ptr(logits), T, H, E, k, _ptr(out["ids"]), _ptr(out["w"]),
                                      _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["inv"]),
                                      _ptr(out["act_codes"]), _ptr(out["act_scales"]), _ptr(dev_status), _ptr(ws),
                                      ws.numel(), _stream()))
    for key in ("perm", "inv", "act_codes", "act_scales"):
        out[key] = out[key][:R]
    return out


def fp8_quantize(x, S=None, codes=None, workspace=None):
    """FP8 (E4M3) codes of x [rows, cols] (bf16 or fp32) with one per-tensor
    decode scale.  S=None: dynamic (written to a new device scalar).
    Returns (codes uint8 [rows, cols], S)."""
    L = load()
    rows, cols = x.shape
    dev = x.device
    dt = NVFP4_DT_BF16 if x.dtype == torch.bfloat16 else NVFP4_DT_F32
    dynamic = S is None
    if S is None:
        S = torch.zeros(4, dtype=torch.float32, device=dev)
    if codes is None:
        codes = _empty((rows, cols), torch.uint8, dev)
    if workspace is None and dynamic:
        workspace = _empty(int(L.nvfp4_quantize_workspace_bytes(rows, cols)), torch.uint8, dev)
    _check("fp8_quantize", L.fp8_quantize(_ptr(x), dt, rows, cols, x.stride(0), _ptr(S),
                                          NVFP4_SCALE_DYNAMIC if dynamic else NVFP4_SCALE_STATIC, _ptr(codes),
                                          _ptr(workspace), 0 if workspace is None else workspace.numel(), _stream()))
    return codes, S[:1]


def moe_route_quantize_fp8(x, logits, k, dev_status=None):
    """Routing + FP8 quantisation of x [T, H] bf16 written in permuted order.
    Returns dict(ids, w, offsets, perm, inv, S_x, act_codes)."""
    L = load()
    T, H = x.shape
    E = logits.shape[1]
    dev = x.device
    R = T * k
    out = dict(ids=_empty((T, k), torch.int32, dev), w=_empty((T, k), torch.float32, dev),
               offsets=_empty((E + 1,), torch.int32, dev), perm=_empty((max(R, 1),), torch.int32, dev),
               inv=_empty((max(R, 1),), torch.int32, dev), S_x=torch.zeros(4, dtype=torch.float32, device=dev),
               act_codes=_empty((max(R, 1), H), torch.uint8, dev))
    ws = _empty(max(int(L.moe_align_permute_workspace_bytes(T, E, k)), 256), torch.uint8, dev)
    _check("moe_route_quantize_fp8",
           L.moe_route_quantize_fp8(_ptr(x), _ptr(logits), T, H, E, k, _ptr(out["ids"]), _ptr(out["w"]),
                                    _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["inv"]), _ptr(out["S_x"]),
                                    _ptr(out["act_codes"]), _ptr(dev_status), _ptr(ws), ws.numel(), _stream()))
    for key in ("perm", "inv", "act_codes"):
        out[key] = out[key][:R]
    out["S_x"] = out["S_x"][:1]
    return out


def moe_grouped_gemm_nvfp4(mode, a, a_scales, a_S, w_codes, w_scales_packed, w_S, offsets, N, K, out=None,
                           dev_status=None):
    L = load()
    E = offsets.numel() - 1
    R = a.shape[0]
    if out is None:
        out = _empty((max(R, 1), N), torch.float32, a.device)[:R]
    _check("moe_grouped_gemm_nvfp4",
           L.moe_grouped_gemm_nvfp4(mode, _ptr(a), _ptr(a_scales), _ptr(a_S), _ptr(w_codes), _ptr(w_scales_packed),
                                    _ptr(w_S), _ptr(offsets), E, N, K, R, _ptr(out), _ptr(dev_status), _stream()))
    return out


def moe_swiglu_requant(G, mode, S_h=None):
    L = load()
    R, I2 = G.shape
    I = I2 // 2
    dev = G.device
    if mode == MOE_W4A8:
        hc = _empty((max(R, 1), I), torch.uint8, dev)
        _check("moe_swiglu_requant",
               L.moe_swiglu_requant(_ptr(G), R, I, mode, _ptr(S_h), _ptr(hc), None, None, _stream()))
        return hc[:R]
    if mode in (MOE_W4A4, MOE_MXW4A4):
        hc = _empty((max(R, 1), I // 2), torch.uint8, dev)
        hs = _empty((max(R, 1), I // 16 if mode == MOE_W4A4 else mxfp4_scale_pitch(I)), torch.uint8, dev)
        _check("moe_swiglu_requant",
               L.moe_swiglu_requant(_ptr(G), R, I, mode, _ptr(S_h), _ptr(hc), _ptr(hs), None, _stream()))
        return hc[:R], hs[:R]
    hb = _empty((max(R, 1), I), torch.bfloat16, dev)
    _check("moe_swiglu_requant", L.moe_swiglu_requant(_ptr(G), R, I, mode, None, None, None, _ptr(hb), _stream()))
    return hb[:R]


def moe_gather_f16(x, perm=None, R=None):
    """bf16 rows x[perm[r]] (or x[r]) carried as F16: returns (a_f16 [R, H]
    float16 holding x * 2^e_r, a_rs [R] fp32 = 2^-e_r)."""
    L = load()
    T, H = x.shape
    R = (perm.numel() if perm is not None else T) if R is None else R
    a = _empty((max(R, 1), H), torch.float16, x.device)
    rs = _empty((max(R, 1),), torch.float32, x.device)
    _check("moe_gather_f16", L.moe_gather_f16(_ptr(x), T, H, _ptr(perm), R, _ptr(a), _ptr(rs), _stream()))
    return a[:R], rs[:R]


def moe_swiglu_f16(G):
    """The W4A16 SwiGLU (h rounded to bf16) carried as F16 rows: returns
    (h_f16 [R, I] float16 = h * 2^e_r, h_rs [R] fp32 = 2^-e_r)."""
    L = load()
    R, I2 = G.shape
    I = I2 // 2
    h = _empty((max(R, 1), I), torch.float16, G.device)
    rs = _empty((max(R, 1),), torch.float32, G.device)
    _check("moe_swiglu_f16", L.moe_swiglu_f16(_ptr(G), R, I, _ptr(h), _ptr(rs), _stream()))
    return h[:R], rs[:R]


def moe_route_quantize_fp8_f16(x, logits, k, dev_status=None):
    """moe_route_quantize_fp8 with the codes as their f16 values: returns
    dict(ids, w, offsets, perm, inv, S_x, act_f16 [T*k, H] float16, act_rs [T*k])."""
    L = load()
    T, H = x.shape
    E = logits.shape[1]
    dev = x.device
    R = T * k
    out = dict(ids=_empty((max(T, 1), k), torch.int32, dev), w=_empty((max(T, 1), k), torch.float32, dev),
               offsets=_empty((E + 1,), torch.int32, dev), perm=_empty((max(R, 1),), torch.int32, dev),
               inv=_empty((max(R, 1),), torch.int32, dev), S_x=_empty((4,), torch.float32, dev),
               act_f16=_empty((max(R, 1), H), torch.float16, dev), act_rs=_empty((max(R, 1),), torch.float32, dev))
    ws = _empty((max(int(L.moe_align_permute_workspace_bytes(T, E, k)), 256),), torch.uint8, dev)
    _check("moe_route_quantize_fp8_f16",
           L.moe_route_quantize_fp8_f16(_ptr(x), _ptr(logits), T, H, E, k, _ptr(out["ids"]), _ptr(out["w"]),
                                        _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(out["inv"]), _ptr(out["S_x"]),
                                        _ptr(out["act_f16"]), _ptr(out["act_rs"]), _ptr(dev_status), _ptr(ws),
                                        ws.numel(), _stream()))
    for key in ("ids", "w"):
        out[key] = out[key][:T]
    for key in ("perm", "inv", "act_f16", "act_rs"):
        out[key] = out[key][:R]
    out["S_x"] = out["S_x"][:1]
    return out


def moe_swiglu_fp8_f16(G, S_h):
    """The W4A8 SwiGLU's FP8 codes as their f16 values: returns (h_f16 [R, I]
    float16, h_rs [R] fp32 = S_h)."""
    L = load()
    R, I2 = G.shape
    I = I2 // 2
    h = _empty((max(R, 1), I), torch.float16, G.device)
    rs = _empty((max(R, 1),), torch.float32, G.device)
    _check("moe_swiglu_fp8_f16", L.moe_swiglu_fp8_f16(_ptr(G), R, I, _ptr(S_h), _ptr(h), _ptr(rs), _stream()))
    return h[:R], rs[:R]


def moe_combine(Y, inv, topk_w, out_dtype=torch.float32, dev_status=None):
    L = load()
    T, k = topk_w.shape
    H = Y.shape[1]
    out = _empty((T, H), out_dtype, Y.device)
    dt = NVFP4_DT_F32 if out_dtype == torch.float32 else NVFP4_DT_BF16
    _check("moe_combine", L.moe_combine(_ptr(Y), _ptr(inv), _ptr(topk_w), T, k, H, dt, _ptr(out), _ptr(dev_status),
                                        _stream()))
    return out


def moe_layer_workspace_bytes(mode, T, H, I, E, k):
    return int(load().moe_layer_workspace_bytes(mode, T, H, I, E, k))


def moe_layer_forward(mode, x, logits, k, w13, w2, S_h, out=None, workspace=None, dev_status=None):
    """Whole layer.  w13 / w2: (codes, packed scales, S[E]) on the GPU (S is
    None for MOE_MXW4A4)."""
    L = load()
    T, H = x.shape
    E = logits.shape[1]
    I = w2[0].shape[2] * 2
    dev = x.device
    if out is None:
        out = _empty((T, H), torch.float32, dev)
    if workspace is None:
        workspace = _empty(moe_layer_workspace_bytes(mode, T, H, I, E, k), torch.uint8, dev)
    _check("moe_layer_forward",
           L.moe_layer_forward(mode, _ptr(x), _ptr(logits), T, H, I, E, k, _ptr(w13[0]), _ptr(w13[1]), _ptr(w13[2]),
                               _ptr(w2[0]), _ptr(w2[1]), _ptr(w2[2]), _ptr(S_h), _ptr(out), _ptr(dev_status),
                               _ptr(workspace), workspace.numel(), _stream()))
    return out


def moe_layer_host_workspace_bytes(mode, T, H, I, E, k):
    return int(load().moe_layer_host_workspace_bytes(mode, T, H, I, E, k))


def moe_layer_forward_host(mode, x_host, logits_host, k, w13, w2, S_h, out_host=None, workspace=None,
                           dev_status=None):
    """Whole layer from and to page-locked host memory: x_host bf16 [T, H]
    and logits_host fp32 [T, E] pinned CPU tensors; returns out_host, a
    pinned fp32 [T, H] CPU tensor the device writes (valid once the current
    stream has reached this point).  w13 / w2 as for moe_layer_forward."""
    for t in (x_host, logits_host) + (() if out_host is None else (out_host,)):
        _hptr(t)  # rejects device, pageable or strided tensors before any work
    L = load()
    T, H = x_host.shape
    E = logits_host.shape[1]
    I = w2[0].shape[2] * 2
    dev = w13[0].device
    if out_host is None:
        out_host = torch.empty((T, H), dtype=torch.float32).pin_memory()
    if workspace is None:
        workspace = _empty(moe_layer_host_workspace_bytes(mode, T, H, I, E, k), torch.uint8, dev)
    _check("moe_layer_forward_host",
           L.moe_layer_forward_host(mode, _hptr(x_host), _hptr(logits_host), T, H, I, E, k, _ptr(w13[0]),
                                    _ptr(w13[1]), _ptr(w13[2]), _ptr(w2[0]), _ptr(w2[1]), _ptr(w2[2]), _ptr(S_h),
                                    _hptr(out_host), _ptr(dev_status), _ptr(workspace), workspace.numel(),
                                    _stream()))
    return out_host


class MoELayerGraph:
    """moe_layer_forward_host for fixed shapes and weights, replayed as one
    CUDA graph: x and logits are read from pinned host buffers and the output
    is written to a pinned host buffer by the layer's own kernels, so the
    graph is one chain of kernels.  A decode step of many small kernels is
    dominated by launch overhead otherwise (the CUDA-graph lesson of "Native
    FP4 Is Slower Than Emulated FP4", section 3).

    Usage: g = MoELayerGraph(mode, T, H, E, k, w13, w2, S_h); write the step's
    inputs into g.x_host / g.logits_host (or pass them to run()); g.run()
    returns g.out_host, valid until the next run()."""

    def __init__(self, mode, T, H, E, k, w13, w2, S_h, device=None):
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        I = w2[0].shape[2] * 2
        self.x_host = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        self.logits_host = torch.empty(T, E, dtype=torch.float32).pin_memory()
        self.out_host = torch.empty(T, H, dtype=torch.float32).pin_memory()
        self._ws = torch.empty(moe_layer_host_workspace_bytes(mode, T, H, I, E, k), dtype=torch.uint8, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        args = (mode, k, w13, w2, S_h)

        def body():
            moe_layer_forward_host(args[0], self.x_host, self.logits_host, args[1], args[2], args[3], args[4],
                                   out_host=self.out_host, workspace=self._ws, dev_status=self.dev_status)

        self.x_host.zero_()
        self.logits_host.zero_()
        self._stream = torch.cuda.Stream(device=dev)
        self._stream.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(self._stream):
            body()  # eager run first: one-time library setup happens outside the capture
            self._stream.synchronize()
            self._graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self._graph, stream=self._stream):
                body()
        self._stream.synchronize()

    def run(self, x_host=None, logits_host=None):
        if x_host is not None:
            self.x_host.copy_(x_host)
        if logits_host is not None:
            self.logits_host.copy_(logits_host)
        with torch.cuda.stream(self._stream):
            self._graph.replay()  # launches on the current stream
        self._stream.synchronize()
        return self.out_host
