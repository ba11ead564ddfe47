"""Seeded synthetic inputs for the DeepSeekMoE layer (shapes and distributions only).

This module is shared by the CUDA path's tests/bench and by the CPU oracle's tests.
It draws random numbers and nothing else: no routing, no expert arithmetic, no
quantisation.  Every tensor comes from a ``torch.Generator`` seeded from
``(config seed, tensor id[, expert id])`` so that any one expert's weights can be
regenerated or copied on its own.

Workloads (T tokens, d model width, E routed experts, S shared experts, k top-k,
I expert intermediate size) follow the layer described on the pages:
  * "DeepSeek-V3 详解" (yudonglee.me), section 2.2: 256 routed + 1 shared, top-8.
  * "DeepSeek-V3 技术报告要点" (deepseek.csdn.net), section 3 table: hidden 7168,
    moe_intermediate_size 2048.
Distributions: x ~ N(0, 1); router weight ~ N(0, sigma_r); expert weights
~ N(0, 1/sqrt(fan_in)) (the second argument of N is a standard deviation);
bias b = 0 or U(-0.05, 0.05); the skewed decode workload adds per-expert logit
offsets o_i = A * r_i^(-1.1) for a seeded permutation r of 1..E (Zipf, s = 1.1).
The backward pass takes an upstream gradient dout ~ N(0, 1) of the output's shape.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    E: int
    S: int
    k: int
    I: int
    router_std: float | None  # None -> 1/sqrt(d)
    bias_uniform: float = 0.0  # b ~ U(-a, a); 0 -> b = 0
    zipf_amp: float = 0.0  # logit offsets A * r^-1.1; 0 -> none
    fp8: bool = False
    pow2: bool = False  # FP8 with power-of-two block scales
    n_group: int = 0  # group-limited routing: groups of experts (0 = none)
    topk_group: int = 0  # groups kept per token
    seed: int = 0
    gamma: float = 0.001

    @property
    def rows_routed(self) -> int:
        return self.T * self.k

    @property
    def rows_total(self) -> int:
        return self.T * self.k + self.S * self.T

    def expert_flops(self) -> float:
        """Algorithmic expert-GEMM FLOPs: 2 * T * (k + S) * 3 * d * I."""
        return 2.0 * self.T * (self.k + self.S) * 3.0 * self.d * self.I

    def with_(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS: dict[str, MoEConfig] = {
    # T=256, d=256, 16 routed + 1 shared, top-2, I=128, router N(0, 0.02), b = 0
    "tiny": MoEConfig("tiny", 256, 256, 16, 1, 2, 128, 0.02),
    # T=4096, d=2048, 64 routed + 2 shared, top-6, I=1408, b ~ U(-0.05, 0.05)
    "mid": MoEConfig("mid", 4096, 2048, 64, 2, 6, 1408, None, bias_uniform=0.05),
    # V3-shaped layer: T=8192, d=7168, 256 + 1, top-8, I=2048, router N(0, 0.006)
    "v3": MoEConfig("v3", 8192, 7168, 256, 1, 8, 2048, 0.006),
    # V3-shaped FP8 path: T=16384
    "v3fp8": MoEConfig("v3fp8", 16384, 7168, 256, 1, 8, 2048, 0.006, fp8=True),
    # the same with power-of-two block scales (applied by the block-scaled tensor-core MMA)
    "v3fp8p2": MoEConfig("v3fp8p2", 16384, 7168, 256, 1, 8, 2048, 0.006, fp8=True, pow2=True),
    # V3 shape with group-limited routing: 8 groups of 32 experts, 4 groups per token
    "v3grp": MoEConfig("v3grp", 8192, 7168, 256, 1, 8, 2048, 0.006, n_group=8, topk_group=4),
    # skewed-load decode regime: T=256 with Zipf(1.1) logit offsets, amplitude 2.0
    "skew": MoEConfig("skew", 256, 7168, 256, 1, 8, 2048, 0.006, zipf_amp=2.0),
}

# tensor ids mixed into the seeds
_ID_X, _ID_WR, _ID_B, _ID_OFF, _ID_WGU, _ID_WD = 1, 2, 3, 4, 5, 6
_ID_DOUT = 9


def _gen(device, *parts: int) -> torch.Generator:
    seed = 0
    for p in parts:
        seed = (seed * 1_000_003 + int(p) + 1) % (2**62)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_x(cfg: MoEConfig, device="cpu", T: int | None = None) -> torch.Tensor:
    """x ~ N(0,1) as bf16 [T, d] (row-major)."""
    T = cfg.T if T is None else T
    g = _gen(device, cfg.seed, _ID_X, T)
    return torch.randn(T, cfg.d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_dout(cfg: MoEConfig, device="cpu", T: int | None = None) -> torch.Tensor:
    """Upstream gradient of the layer output, N(0,1) as bf16 [T, d]."""
    T = cfg.T if T is None else T
    g = _gen(device, cfg.seed, _ID_DOUT, T)
    return torch.randn(T, cfg.d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_router(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """Router weight bf16 [E, d] ~ N(0, sigma_r)."""
    std = cfg.router_std if cfg.router_std is not None else 1.0 / math.sqrt(cfg.d)
    g = _gen(device, cfg.seed, _ID_WR)
    w = torch.randn(cfg.E, cfg.d, generator=g, device=device, dtype=torch.float32) * std
    return w.to(torch.bfloat16)


def make_bias(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """Selection bias fp32 [E]: zero, or U(-a, a)."""
    if cfg.bias_uniform == 0.0:
        return torch.zeros(cfg.E, dtype=torch.float32, device=device)
    g = _gen(device, cfg.seed, _ID_B)
    u = torch.rand(cfg.E, generator=g, device=device, dtype=torch.float32)
    return (u * 2.0 - 1.0) * cfg.bias_uniform


def make_logit_offset(cfg: MoEConfig, device="cpu") -> torch.Tensor | None:
    """Zipf(s=1.1) per-expert logit offsets o_i = A * r_i^-1.1, r a seeded permutation of 1..E."""
    if cfg.zipf_amp == 0.0:
        return None
    g = _gen("cpu", cfg.seed, _ID_OFF)
    r = torch.randperm(cfg.E, generator=g).to(torch.float64) + 1.0
    o = cfg.zipf_amp * r.pow(-1.1)
    return o.to(torch.float32).to(device)


def make_expert(cfg: MoEConfig, e: int, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """Weights of expert e (0..E-1 routed, E..E+S-1 shared), bf16.

    Returns (w_gate_up [2I, d] with gate rows first then up rows, w_down [d, I]).
    """
    g1 = _gen(device, cfg.seed, _ID_WGU, e)
    wgu = torch.randn(2 * cfg.I, cfg.d, generator=g1, device=device, dtype=torch.float32)
    wgu = (wgu * (1.0 / math.sqrt(cfg.d))).to(torch.bfloat16)
    g2 = _gen(device, cfg.seed, _ID_WD, e)
    wd = torch.randn(cfg.d, cfg.I, generator=g2, device=device, dtype=torch.float32)
    wd = (wd * (1.0 / math.sqrt(cfg.I))).to(torch.bfloat16)
    return wgu, wd


def make_experts(cfg: MoEConfig, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """All E+S experts: w_gate_up bf16 [E+S, 2I, d], w_down bf16 [E+S, d, I]."""
    n = cfg.E + cfg.S
    wgu = torch.empty(n, 2 * cfg.I, cfg.d, dtype=torch.bfloat16, device=device)
    wd = torch.empty(n, cfg.d, cfg.I, dtype=torch.bfloat16, device=device)
    for e in range(n):
        a, b = make_expert(cfg, e, device)
        wgu[e].copy_(a)
        wd[e].copy_(b)
    return wgu, wd


_ID_WGU8, _ID_WD8 = 7, 8


def make_expert_fp8(cfg: MoEConfig, e: int, device="cpu", pow2: bool = False):
    """FP8 weights of expert e drawn directly (not quantised from bf16): E4M3 codes of
    N(0, 64) values (torch's float8_e4m3fn cast) and per-128x128-block scales around
    1/(64 sqrt(fan_in)), so that code * scale ~ N(0, 1/sqrt(fan_in)); pow2: scales drawn
    from the two powers of two 2^-(p + b), p = round(log2(64 sqrt(fan_in))), b in {0, 1}.
    Returns (wgu_q [2I, d], wgu_scale [2I/128, d/128], wd_q [d, I], wd_scale [d/128, I/128])."""
    out = []
    for tid, (n, k) in ((_ID_WGU8, (2 * cfg.I, cfg.d)), (_ID_WD8, (cfg.d, cfg.I))):
        g = _gen(device, cfg.seed, tid, e)
        q = (torch.randn(n, k, generator=g, device=device) * 64.0).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        u = torch.rand(n // 128, k // 128, generator=g, device=device)
        if pow2:
            p = round(math.log2(64.0 * math.sqrt(k)))
            sc = torch.exp2(-(p + (u < 0.5).to(torch.float32)))
        else:
            sc = (0.5 + u) / (64.0 * math.sqrt(k))
        out += [q, sc.to(torch.float32)]
    return tuple(out)


def make_experts_fp8(cfg: MoEConfig, device="cpu", pow2: bool = False):
    """All E+S experts in FP8: (wgu_q [E+S, 2I, d], wgu_scale, wd_q [E+S, d, I], wd_scale)."""
    n = cfg.E + cfg.S
    wgu = torch.empty(n, 2 * cfg.I, cfg.d, dtype=torch.float8_e4m3fn, device=device)
    gs = torch.empty(n, 2 * cfg.I // 128, cfg.d // 128, dtype=torch.float32, device=device)
    wd = torch.empty(n, cfg.d, cfg.I, dtype=torch.float8_e4m3fn, device=device)
    ds = torch.empty(n, cfg.d // 128, cfg.I // 128, dtype=torch.float32, device=device)
    for e in range(n):
        a, b, c, d_ = make_expert_fp8(cfg, e, device, pow2)
        wgu[e].copy_(a)
        gs[e].copy_(b)
        wd[e].copy_(c)
        ds[e].copy_(d_)
    return wgu, gs, wd, ds


def make_all(cfg: MoEConfig, device="cpu") -> dict:
    wgu, wd = make_experts(cfg, device)
    return dict(
        x=make_x(cfg, device),
        w_router=make_router(cfg, device),
        bias=make_bias(cfg, device),
        logit_offset=make_logit_offset(cfg, device),
        w_gate_up=wgu,
        w_down=wd,
    )
