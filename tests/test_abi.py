"""The C-ABI library builds for sm_103a, loads, and exports every function
that include/nvfp4moe.h declares (CPU only: no compute call is made)."""
import ctypes
import os
import re

from conftest import ROOT


def _declared():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([a-z][a-z0-9_]+)\s*\(", text, re.M)
    return names


def test_header_declares_the_path():
    names = set(_declared())
    for n in ("nvfp4_quantize", "moe_align_permute", "moe_grouped_gemm_nvfp4", "moe_swiglu_requant", "moe_combine"):
        assert n in names


def test_library_exports_every_declared_symbol():
    from nvfp4_mixture_experts_top_gb300 import binding, build
    path = build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(binding.EXPORTS) == set(_declared())


def test_status_strings_without_gpu():
    from nvfp4_mixture_experts_top_gb300 import binding
    L = binding.load()
    for s in range(9):
        assert L.nvfp4_status_string(s).startswith(b"NVFP4_")
    assert L.moe_layer_workspace_bytes(0, 16, 4096, 2048, 256, 8) > 16 * 8 * 2 * 2048 * 4


def test_host_validation_without_gpu():
    """Argument errors are caught on the host, before any device call."""
    from nvfp4_mixture_experts_top_gb300 import binding
    L = binding.load()
    # cols not a multiple of 16 -> E_SHAPE; null scale pointer -> E_INVAL
    assert L.nvfp4_quantize(None, 0, 4, 24, 24, ctypes.c_void_p(16), 0, None, None, None, 0, None) == 2
    assert L.nvfp4_quantize(None, 0, 4, 32, 32, None, 0, None, None, None, 0, None) == 1
    # misaligned pointer -> E_ALIGN
    assert L.nvfp4_quantize(ctypes.c_void_p(8), 0, 4, 32, 32, ctypes.c_void_p(16), 0, ctypes.c_void_p(16),
                            ctypes.c_void_p(16), None, 0, None) == 3
    # grouped GEMM with N % 128 != 0 -> E_SHAPE; bad mode -> E_INVAL
    assert L.moe_grouped_gemm_nvfp4(0, None, None, None, None, None, None, None, 4, 100, 256, 8, None, None,
                                    None) == 2
    assert L.moe_grouped_gemm_nvfp4(7, None, None, None, None, None, None, None, 4, 128, 256, 8, None, None,
                                    None) == 1
    # routing with k > 32 -> E_SHAPE
    assert L.moe_align_permute(None, 4, 64, 33, None, None, ctypes.c_void_p(16), None, None, 0, None, None, 0,
                               None, None, None, None, 0, None) == 2


def test_mxfp4_host_side_without_gpu():
    """The MXFP4 scale pitch (a host computation) and the MXFP4 argument
    checks, which run before any device call."""
    from nvfp4_mixture_experts_top_gb300 import binding
    L = binding.load()
    # cols/32 rounded up to a multiple of 16 bytes, at least 128
    assert [L.mxfp4_scale_pitch(c) for c in (32, 256, 2048, 4096, 4608, 6144, 8192)] == [128, 128, 128, 128, 144,
                                                                                         192, 256]
    # cols not a multiple of 32 -> E_SHAPE; null outputs -> E_INVAL; bad dtype -> E_INVAL
    assert L.mxfp4_quantize(None, 0, 4, 48, 48, None, None, None) == 2
    assert L.mxfp4_quantize(None, 0, 4, 64, 64, None, None, None) == 1
    assert L.mxfp4_quantize(None, 5, 4, 64, 64, None, None, None) == 1
    # MXFP4 grouped GEMM needs activation scales but no per-tensor scales
    assert L.moe_grouped_gemm_nvfp4(2, ctypes.c_void_p(16), None, None, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                    None, ctypes.c_void_p(16), 4, 128, 256, 8, ctypes.c_void_p(16), None,
                                    None) == 1
    # MXFP4 weight-scale packing shape rule
    assert L.mxfp4_pack_weight_scales(None, 2, 100, 256, None, None) == 2
    # SwiGLU/requant in MXFP4 needs I % 32 == 0
    assert L.moe_swiglu_requant(ctypes.c_void_p(16), 4, 48, 2, None, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                None, None) == 2
    assert L.moe_layer_workspace_bytes(2, 16, 4096, 2048, 256, 8) > 16 * 8 * 2 * 2048 * 4


def test_host_layer_entry_rejects_device_or_pageable_buffers_without_gpu():
    """moe_layer_forward_host takes page-locked CPU tensors only; the binding
    refuses others before doing any work."""
    import pytest
    import torch
    from nvfp4_mixture_experts_top_gb300 import binding
    x = torch.zeros(2, 256, dtype=torch.bfloat16)  # pageable
    lg = torch.zeros(2, 8, dtype=torch.float32)
    with pytest.raises(ValueError):
        binding.moe_layer_forward_host(binding.MOE_W4A4, x, lg, 2, None, None, None)
    L = binding.load()
    assert L.moe_layer_host_workspace_bytes(0, 16, 4096, 2048, 256, 8) == (
        L.moe_layer_workspace_bytes(0, 16, 4096, 2048, 256, 8) + 16 * 4096 * 2 + 16 * 256 * 4)
    assert L.moe_layer_host_workspace_bytes(0, -1, 4096, 2048, 256, 8) == 0


def test_layer_entries_validate_on_the_host_without_gpu():
    """moe_layer_forward and moe_layer_forward_host reject bad arguments on the
    host, before any device call: status codes, not launches."""
    from nvfp4_mixture_experts_top_gb300 import binding
    L = binding.load()
    P = ctypes.c_void_p
    ok = P(4096)  # an aligned non-null stand-in; never dereferenced on these paths
    ws = L.moe_layer_host_workspace_bytes(0, 16, 4096, 2048, 256, 8)

    def host(mode=0, x=ok, lg=ok, T=16, H=4096, I=2048, E=256, k=8, out=ok, work=ok, nbytes=ws):
        return L.moe_layer_forward_host(mode, x, lg, T, H, I, E, k, ok, ok, ok, ok, ok, ok, ok, out, None, work,
                                        nbytes, None)

    assert host(mode=7) == 1                    # bad mode
    assert host(H=100) == 2                     # H % 256 != 0
    assert host(k=33) == 2                      # k > 32
    assert host(E=2048) == 2                    # E > 1024
    assert host(T=0, x=None, lg=None, out=None) == 0  # nothing to do
    assert host(x=None) == 1                    # null input
    assert host(out=None) == 1                  # null output
    assert host(nbytes=ws - 1) == 4             # workspace too small
    assert host(work=None) == 4
    assert host(x=P(4096 + 8)) == 3             # misaligned x
    assert host(lg=P(4096 + 2)) == 3            # logits need 4-byte alignment
    # the device-memory layer entry: the same shape checks
    assert L.moe_layer_forward(0, ok, ok, 16, 4000, 2048, 256, 8, ok, ok, ok, ok, ok, ok, ok, ok, None, ok,
                               L.moe_layer_workspace_bytes(0, 16, 4000, 2048, 256, 8), None) == 2
    assert L.moe_layer_forward(0, ok, ok, 16, 4096, 2048, 256, 8, ok, ok, ok, ok, ok, ok, ok, ok, None, ok,
                               L.moe_layer_workspace_bytes(0, 16, 4096, 2048, 256, 8) - 1, None) == 4


def test_carrier_entries_validate_on_the_host_without_gpu():
    """The F16-carrier entry points and GEMM mode MOE_W4A16F reject bad
    arguments on the host: shapes, missing pointers and misalignment."""
    from nvfp4_mixture_experts_top_gb300 import binding
    L = binding.load()
    p16, p8 = ctypes.c_void_p(16), ctypes.c_void_p(8)
    # W4A16F needs its row multipliers (a_S) -> E_INVAL
    assert L.moe_grouped_gemm_nvfp4(binding.MOE_W4A16F, p16, None, None, p16, p16, p16, p16, 4, 128, 256, 8, p16,
                                    None, None) == 1
    # moe_gather_f16: H % 8 != 0 -> E_SHAPE; no row-multiplier output -> E_INVAL; misaligned rows -> E_ALIGN;
    # no permutation and more output rows than tokens -> E_INVAL; nothing to do -> OK
    assert L.moe_gather_f16(p16, 4, 12, None, 4, p16, p16, None) == 2
    assert L.moe_gather_f16(p16, 4, 16, None, 4, p16, None, None) == 1
    assert L.moe_gather_f16(p8, 4, 16, None, 4, p16, p16, None) == 3
    assert L.moe_gather_f16(p16, 4, 16, None, 8, p16, p16, None) == 1
    assert L.moe_gather_f16(None, 0, 16, None, 0, None, None, None) == 0
    # moe_swiglu_f16 / moe_swiglu_fp8_f16: I % 16 != 0 -> E_SHAPE; missing S_h -> E_INVAL
    assert L.moe_swiglu_f16(p16, 4, 24, p16, p16, None) == 2
    assert L.moe_swiglu_f16(p16, 4, 32, p16, None, None) == 1
    assert L.moe_swiglu_fp8_f16(p16, 4, 32, None, p16, p16, None) == 1
    assert L.moe_swiglu_fp8_f16(p16, 4, 24, p16, p16, p16, None) == 2
    # moe_route_quantize_fp8_f16: H % 256 != 0 -> E_SHAPE; no carrier output -> E_INVAL
    assert L.moe_route_quantize_fp8_f16(p16, p16, 4, 200, 64, 8, p16, p16, p16, p16, p16, p16, p16, p16, None, p16,
                                        1 << 20, None) == 2
    assert L.moe_route_quantize_fp8_f16(p16, p16, 4, 256, 64, 8, p16, p16, p16, p16, p16, p16, None, p16, None, p16,
                                        1 << 20, None) == 1


def test_combine_rejects_more_than_32_slots_without_gpu():
    """k > 32 (more slots than routing produces) is refused on the host."""
    from nvfp4_mixture_experts_top_gb300 import binding
    L = binding.load()
    p16 = ctypes.c_void_p(16)
    assert L.moe_combine(p16, p16, p16, 4, 33, 64, 1, p16, None, None) == 2


def test_early_gemms_only_inside_the_layer_chain():
    """The grouped GEMMs' early mode reads the routing and issues weight
    copies before the grid-dependency wait.  That is safe only where the
    routing was written by a kernel that completed before the GEMM's
    predecessor passed its own wait: inside moe_layer_forward's chain.  So
    every internal GEMM call that passes early = true must sit in that
    function, and the public entry point must pass false (source check)."""
    src = open(os.path.join(ROOT, "nvfp4_mixture_experts_top_gb300", "csrc", "api.cu")).read()
    lines = src.splitlines()
    owner = None
    early_calls, public_false = [], False
    for i, line in enumerate(lines):
        m = re.match(r"^(?:static\s+)?int\s+(\w+)\(", line)
        if m:
            owner = m.group(1)
        if re.search(r"\bgrouped_gemm\(", line) and not line.lstrip().startswith("static"):
            call = " ".join(lines[i:i + 4])
            call = call[: call.index(";") + 1]
            flag = call.rstrip(");").rsplit(",", 1)[1].strip()
            if flag == "true":
                early_calls.append(owner)
            elif owner == "moe_grouped_gemm_nvfp4" and flag == "false":
                public_false = True
    assert early_calls and set(early_calls) == {"moe_layer_forward"}, early_calls
    assert public_false
    # no other file launches a GEMM in early mode
    csrc = os.path.join(ROOT, "nvfp4_mixture_experts_top_gb300", "csrc")
    for fn in os.listdir(csrc):
        if fn.endswith(".cu") and fn not in ("api.cu", "gemm_w4a4.cu"):
            assert not re.search(r"\bearly\b", open(os.path.join(csrc, fn)).read()), fn
