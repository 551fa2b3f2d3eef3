"""Named workloads and their seeded synthetic inputs.

This module holds the input recipe only -- shapes, distributions and seeds --
and none of the method's arithmetic (no quantisation, routing, GEMM or
combine).  The CUDA path, the tests and the CPU oracle all draw their inputs
from here, so both sides of every parity check see the same numbers.

Shapes stand in for the workloads the reference pages describe:
  * ``tiny``        -- a correctness case small enough for the oracle in
                       seconds (T=8, hidden 256, intermediate 512, 8 experts,
                       top-2).
  * ``decode_c16``  -- decode at 16 concurrent requests ("The Benchmark That
                       Confirmed the Ceiling", section "Why This Message Was
                       Written": C=16 decode), 256 experts top-8.
  * ``decode_b512`` -- 512 concurrent decode tokens over 256 experts, top-8,
                       ~16 tokens per expert on average ("The 2x Gap",
                       section "The Investigation So Far"), with a Zipf(1.1)
                       expert-popularity bias so per-expert M is ragged.
  * ``wide``        -- 512 routed experts, 22 active per token ("Native FP4
                       Is Slower Than Emulated FP4", section 1).
  * ``gemm_sweep``  -- one expert, N=2048, K=6144, M in {1,16,64,512,4096}
                       ("The 2x Gap", section "The Pivot": M=512, N=2048,
                       K=6144).

Inputs: activations N(0,1) rounded to bf16; weights N(0, 0.02) in fp32 (the
caller quantises them); router logits N(0,1) fp32, plus ln(p_e) with
p_e proportional to (e+1)^-1.1 for the Zipf-biased workload.
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int          # tokens
    H: int          # hidden size (K of gate_up, N of down)
    I: int          # expert intermediate size
    E: int          # experts
    k: int          # experts per token
    routing: str    # "uniform" | "zipf"
    modes: tuple = ("w4a4",)
    zipf_s: float = 1.1

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def S_h(self) -> float:
        """Static decode scale of the requantised SwiGLU output h.

        A gate/up pre-activation is a dot product of H unit-variance inputs
        with N(0, 0.02) weights, so its variance is s2 = 0.02^2 * H; h is a
        product of two of them, and 16*s2 covers |h| up to the product of two
        4-sigma values.  The scale maps that bound to the largest NVFP4 value
        6 * 448 = 2688."""
        s2 = 0.02 * 0.02 * self.H
        return float(np.float32(16.0 * s2 / 2688.0))

    @property
    def S_h8(self) -> float:
        """Static decode scale of h requantised to FP8 E4M3 (the W4A8 mode):
        the same bound 16 * 0.02^2 * H mapped to E4M3's largest value 448."""
        s2 = 0.02 * 0.02 * self.H
        return float(np.float32(16.0 * s2 / 448.0))


CONFIGS = {
    "tiny": MoEConfig("tiny", T=8, H=256, I=512, E=8, k=2, routing="uniform"),
    "decode_c16": MoEConfig("decode_c16", T=16, H=4096, I=2048, E=256, k=8, routing="uniform",
                            modes=("w4a4", "w4a16")),
    "decode_b512": MoEConfig("decode_b512", T=512, H=6144, I=2048, E=256, k=8, routing="zipf"),
    "wide": MoEConfig("wide", T=64, H=4096, I=2048, E=512, k=22, routing="uniform",
                      modes=("w4a4", "w4a16")),
}

GEMM_SWEEP = dict(N=2048, K=6144, Ms=(1, 16, 64, 512, 4096))

WEIGHT_STD = 0.02


def _seed(*parts) -> int:
    """Deterministic 63-bit seed from a tuple of small integers / strings."""
    h = 1469598103934665603
    for p in parts:
        for b in str(p).encode():
            h = ((h ^ b) * 1099511628211) & ((1 << 64) - 1)
        h = ((h ^ 0xFF) * 1099511628211) & ((1 << 64) - 1)
    return h & ((1 << 63) - 1)


def _gen(device, *parts):
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def activations_bf16(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """x [T, H] ~ N(0, 1), rounded to bf16."""
    g = _gen(device, "x", seed, T, H)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def router_logits(cfg: MoEConfig, seed: int = 0, device="cpu") -> torch.Tensor:
    """Router logits [T, E] fp32: N(0,1), plus the Zipf popularity bias
    ln(p_e), p_e ~ (e+1)^-s (expert 0 most popular), for routing='zipf'."""
    g = _gen(device, "logits", seed, cfg.T, cfg.E)
    z = torch.randn(cfg.T, cfg.E, generator=g, device=device, dtype=torch.float32)
    if cfg.routing == "zipf":
        r = np.arange(1, cfg.E + 1, dtype=np.float64)
        p = r ** (-cfg.zipf_s)
        p /= p.sum()
        bias = torch.from_numpy(np.log(p).astype(np.float32)).to(device)
        z = z + bias[None, :]
    elif cfg.routing != "uniform":
        raise ValueError(cfg.routing)
    return z.contiguous()


def router_weight_bf16(E: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Router weight [E, H] ~ N(0, 1/H) rounded to bf16, so that the logits of
    N(0, 1) activations are about N(0, 1) (the scale of router_logits)."""
    g = _gen(device, "router", seed, E, H)
    w = torch.randn(E, H, generator=g, device=device, dtype=torch.float32) / float(np.sqrt(H))
    return w.to(torch.bfloat16)


def expert_weight_fp32(which: str, e: int, N: int, K: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """One expert's weight matrix [N, K] ~ N(0, 0.02) in fp32.  which is
    'w13' (gate rows 0..I-1 then up rows I..2I-1, K = hidden) or 'w2'
    (down, N = hidden, K = intermediate).  Seeded per (which, expert), so any
    subset of experts can be regenerated on its own."""
    g = _gen(device, which, seed, e, N, K)
    return torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * WEIGHT_STD


def gemm_operands_fp32(M: int, N: int, K: int, seed: int = 0, device="cpu"):
    """Single-expert GEMM operands: A [M, K] ~ N(0,1), W [N, K] ~ N(0, 0.02)."""
    ga = _gen(device, "gemmA", seed, M, K)
    gw = _gen(device, "gemmW", seed, N, K)
    a = torch.randn(M, K, generator=ga, device=device, dtype=torch.float32)
    w = torch.randn(N, K, generator=gw, device=device, dtype=torch.float32) * WEIGHT_STD
    return a, w


def random_fp32(shape, seed: int, scale: float = 1.0, device="cpu", tag="rand") -> torch.Tensor:
    """Generic N(0, scale^2) fp32 tensor for stage tests."""
    g = _gen(device, tag, seed, *shape)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * scale


def small_variant(cfg: MoEConfig, **over) -> MoEConfig:
    """A copy of a config with some fields replaced (for oracle-sized tests)."""
    d = dict(name=cfg.name + "_small", T=cfg.T, H=cfg.H, I=cfg.I, E=cfg.E, k=cfg.k, routing=cfg.routing,
             modes=cfg.modes, zipf_s=cfg.zipf_s)
    d.update(over)
    return MoEConfig(**d)
