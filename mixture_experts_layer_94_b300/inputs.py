"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random tensors of the right shapes, distributions and
dtypes. It holds none of the layer's arithmetic (no routing, scoring or FFN), so
the CUDA path and the oracle can both take their inputs from it.

Recipe (every tensor is drawn in this fixed order from its own seeded stream):
  * hidden   ~ N(0, 1), [T, d]; fp32 for the tiny workload, else rounded to bf16
  * w_router ~ N(0, 1/d) * router_scale, fp32 [d, N]
  * router_bias (the router's bias term): a Zipf(s) popularity tilt
    -s * ln(rank_e) with rank a seeded permutation of 1..N, else none
  * sel_bias (selection-only): N(0, variance v), else none
  * per routed expert e: W_gate[e], W_up[e] ~ N(0, 1/d) [F, d];
    W_down[e] ~ N(0, 1/F) [d, F]; drawn in fp32, rounded once to bf16
  * per shared expert s: the same with Fs in place of F
  * FP8 expert weights (expert_dtype "fp8"): the same fp32 draws, then per
    matrix row a scale amax(|row|) / 448 (fp32) and E4M3 codes of row / scale
    (torch's round-to-nearest-even cast, clamped to +-448, so no NaN code)
  * MXFP4 expert weights (expert_dtype "mxfp4"): the same fp32 draws, then per
    32 consecutive elements of a row the OCP microscaling recipe: shared
    exponent X = floor(log2(amax)) - 2 (E8M0 code X + 127), elements rounded
    to the nearest E2M1 value of v / 2^X (ties to the even code, saturating at
    6), packed two per byte with the even element in the low nibble
Router-side tensors (hidden, w_router, biases) always come from a CPU
generator, so routing is identical whatever device holds the experts. Expert
weights come from a generator on `device` seeded per expert: large workloads
draw them on the GPU (the CPU and CUDA generators give different, equally
distributed values).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    N: int
    K: int
    F: int
    S: int = 0
    Fs: int = 0
    score: str = "softmax"          # "softmax" | "sigmoid"
    renormalize: int = 1
    hidden_dtype: str = "bf16"      # "f32" | "bf16"
    router_scale: float = 1.0
    sel_bias_var: Optional[float] = None
    zipf: Optional[float] = None
    n_groups: int = 0        # group-limited routing (0: off)
    topk_groups: int = 0
    capacity_factor: float = 0.0  # expert capacity ceil(c T K / N) (0: dropless)
    routing: str = "token"   # "token" (tokens pick K experts) | "expert" (experts pick C tokens)
    expert_dtype: str = "bf16"  # "bf16" | "fp8" (E4M3 codes + fp32 row scales) | "mxfp4" (E2M1 + E8M0 per 32)

    def with_(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)

    @property
    def score_fn(self) -> int:
        return 0 if self.score == "softmax" else 1


# Scale of w_router that makes the token-mean of the largest full-softmax
# probability 0.40 on the Mixtral-shaped workload ("top-1 share about 0.4").
# Found by bisection with the oracle router on this module's seed-0 inputs:
# tests/golden/make_mixtral_router_scale.py writes it to
# tests/golden/mixtral_router_scale.json, and a test checks the two agree.
MIXTRAL_ROUTER_SCALE = 1.1661

TINY = MoEConfig("tiny", T=64, d=128, N=8, K=2, F=256, score="softmax", hidden_dtype="f32")
MIXTRAL = MoEConfig("mixtral", T=4096, d=4096, N=8, K=2, F=14336,
                    router_scale=MIXTRAL_ROUTER_SCALE)
DSV3 = MoEConfig("dsv3", T=8192, d=7168, N=256, K=8, F=2048, S=1, Fs=2048, score="sigmoid",
                 sel_bias_var=0.1, zipf=1.1)
# The DeepSeek-shaped layer with node-limited routing: 8 groups of 32 experts,
# a token may pick from 4 of them.
DSV3_GROUPED = DSV3.with_(name="dsv3_grouped", n_groups=8, topk_groups=4)
# The Mixtral-shaped layer with expert capacity factor 1.0 (C = 1024 copies).
MIXTRAL_CAPACITY = MIXTRAL.with_(name="mixtral_capacity", capacity_factor=1.0)
# The Mixtral-shaped layer with expert-choice routing: every expert takes
# C = T*K/N = 1024 tokens.
MIXTRAL_EC = MIXTRAL.with_(name="mixtral_ec", routing="expert")
GPTOSS = MoEConfig("gptoss", T=2048, d=2880, N=128, K=4, F=2880)
QWEN_DECODE = MoEConfig("qwen_decode", T=1, d=4096, N=128, K=8, F=1536)
# The same layers with FP8 E4M3 expert weights.
MIXTRAL_FP8 = MIXTRAL.with_(name="mixtral_fp8", expert_dtype="fp8")
QWEN_DECODE_FP8 = QWEN_DECODE.with_(name="qwen_decode_fp8", expert_dtype="fp8")
# MXFP4 expert weights: the format gpt-oss ships its experts in.
GPTOSS_MXFP4 = GPTOSS.with_(name="gptoss_mxfp4", expert_dtype="mxfp4")
QWEN_DECODE_MXFP4 = QWEN_DECODE.with_(name="qwen_decode_mxfp4", expert_dtype="mxfp4")
DECODE_BATCHES = (1, 8, 32, 128, 512)

CONFIGS = {c.name: c for c in (TINY, MIXTRAL, MIXTRAL_CAPACITY, MIXTRAL_EC, DSV3, DSV3_GROUPED, GPTOSS,
                               QWEN_DECODE, MIXTRAL_FP8, QWEN_DECODE_FP8, GPTOSS_MXFP4, QWEN_DECODE_MXFP4)}


def _seed(seed: int, *parts) -> int:
    """Derive a stream seed from the base seed and a label (stable across runs)."""
    h = 1469598103934665603
    for p in (seed,) + parts:
        for ch in str(p).encode():
            h = ((h ^ ch) * 1099511628211) & ((1 << 63) - 1)
        h = ((h ^ 0x2F) * 1099511628211) & ((1 << 63) - 1)
    return h


def make_router_inputs(cfg: MoEConfig, seed: int = 0) -> dict:
    """hidden, w_router, router_bias, sel_bias on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed(seed, "hidden"))
    hidden = torch.randn(cfg.T, cfg.d, generator=g, dtype=torch.float32)
    if cfg.hidden_dtype == "bf16":
        hidden = hidden.to(torch.bfloat16)
    g.manual_seed(_seed(seed, "w_router"))
    w_router = torch.randn(cfg.d, cfg.N, generator=g, dtype=torch.float32)
    w_router.mul_(cfg.router_scale / math.sqrt(cfg.d))
    router_bias = None
    if cfg.zipf is not None:
        g.manual_seed(_seed(seed, "zipf"))
        rank = torch.randperm(cfg.N, generator=g).to(torch.float64) + 1.0
        router_bias = (-cfg.zipf * torch.log(rank)).to(torch.float32)
    sel_bias = None
    if cfg.sel_bias_var is not None:
        g.manual_seed(_seed(seed, "sel_bias"))
        sel_bias = torch.randn(cfg.N, generator=g, dtype=torch.float32)
        sel_bias.mul_(math.sqrt(cfg.sel_bias_var))
    return dict(hidden=hidden, w_router=w_router, router_bias=router_bias, sel_bias=sel_bias)


def _draw_bf16(out: torch.Tensor, gen: torch.Generator, std: float) -> None:
    tmp = torch.randn(out.shape, generator=gen, dtype=torch.float32, device=out.device)
    tmp.mul_(std)
    out.copy_(tmp)


E4M3_MAX = 448.0


def _draw_fp8(codes: torch.Tensor, scale: torch.Tensor, gen: torch.Generator, std: float) -> None:
    tmp = torch.randn(codes.shape, generator=gen, dtype=torch.float32, device=codes.device)
    tmp.mul_(std)
    s = tmp.abs().amax(dim=1).clamp_min(1e-30) / E4M3_MAX
    scale.copy_(s)
    tmp.div_(s[:, None]).clamp_(-E4M3_MAX, E4M3_MAX)
    codes.copy_(tmp.to(torch.float8_e4m3fn).view(torch.uint8))


# E2M1 magnitudes by code (OCP microscaling FP4).
E2M1_VALUES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _draw_mxfp4(codes: torch.Tensor, bscale: torch.Tensor, gen: torch.Generator, std: float) -> None:
    rows, half = codes.shape
    tmp = torch.randn((rows, 2 * half), generator=gen, dtype=torch.float32, device=codes.device)
    tmp.mul_(std)
    blk = tmp.view(rows, -1, 32)
    amax = blk.abs().amax(dim=2).clamp_min(1e-30)
    x = torch.floor(torch.log2(amax)) - 2  # the block's shared exponent
    bscale.copy_((x + 127).clamp(0, 254).to(torch.uint8))
    v = (blk / torch.exp2(x)[..., None]).abs().clamp_max(6.0)
    grid = torch.tensor(E2M1_VALUES, dtype=torch.float32, device=codes.device)
    dist = (v[..., None] - grid).abs()
    # nearest E2M1 value; an exact tie goes to the even code (mantissa bit 0)
    dist = dist + torch.tensor([0.0, 1e-30] * 4, device=codes.device) * (dist > 0)
    mag = dist.argmin(dim=-1).to(torch.uint8)
    sign = (blk < 0).to(torch.uint8) * 8
    c4 = (mag | sign).view(rows, -1)
    codes.copy_(c4[:, 0::2] | (c4[:, 1::2] << 4))


def make_expert_weights_mxfp4(cfg: MoEConfig, seed: int = 0, device="cpu") -> dict:
    """Stacked MXFP4 expert weights on `device`: packed E2M1 codes (uint8)
    w_gate, w_up [N, F, d/2], w_down [N, d, F/2] with E8M0 block scales
    w_gate_scale, w_up_scale [N, F, d/32], w_down_scale [N, d, F/32]; shared
    experts likewise. Draws the same normal values as make_expert_weights."""
    device = torch.device(device)
    u8 = torch.uint8
    out = {}
    g = torch.Generator(device=device)

    def stack(kind, n, f):
        gate = torch.empty(n, f, cfg.d // 2, dtype=u8, device=device)
        up = torch.empty_like(gate)
        down = torch.empty(n, cfg.d, f // 2, dtype=u8, device=device)
        sg = torch.empty(n, f, cfg.d // 32, dtype=u8, device=device)
        su = torch.empty_like(sg)
        sd = torch.empty(n, cfg.d, f // 32, dtype=u8, device=device)
        for e in range(n):
            g.manual_seed(_seed(seed, kind, e))
            _draw_mxfp4(gate[e], sg[e], g, 1.0 / math.sqrt(cfg.d))
            _draw_mxfp4(up[e], su[e], g, 1.0 / math.sqrt(cfg.d))
            _draw_mxfp4(down[e], sd[e], g, 1.0 / math.sqrt(f))
        return gate, up, down, sg, su, sd

    (out["w_gate"], out["w_up"], out["w_down"], out["w_gate_scale"], out["w_up_scale"],
     out["w_down_scale"]) = stack("routed", cfg.N, cfg.F)
    for k in ("ws_gate", "ws_up", "ws_down", "ws_gate_scale", "ws_up_scale", "ws_down_scale"):
        out[k] = None
    if cfg.S > 0:
        (out["ws_gate"], out["ws_up"], out["ws_down"], out["ws_gate_scale"], out["ws_up_scale"],
         out["ws_down_scale"]) = stack("shared", cfg.S, cfg.Fs)
    return out


def make_expert_weights_fp8(cfg: MoEConfig, seed: int = 0, device="cpu") -> dict:
    """Stacked FP8 E4M3 expert weights on `device`: codes (uint8) w_gate, w_up
    [N, F, d], w_down [N, d, F] with fp32 row scales w_gate_scale, w_up_scale
    [N, F], w_down_scale [N, d]; shared experts likewise (ws_*, None when
    S == 0). Draws the same normal values as make_expert_weights."""
    device = torch.device(device)
    u8, f32 = torch.uint8, torch.float32
    out = {}
    g = torch.Generator(device=device)

    def stack(kind, n, f):
        gate = torch.empty(n, f, cfg.d, dtype=u8, device=device)
        up = torch.empty_like(gate)
        down = torch.empty(n, cfg.d, f, dtype=u8, device=device)
        sg = torch.empty(n, f, dtype=f32, device=device)
        su = torch.empty_like(sg)
        sd = torch.empty(n, cfg.d, dtype=f32, device=device)
        for e in range(n):
            g.manual_seed(_seed(seed, kind, e))
            _draw_fp8(gate[e], sg[e], g, 1.0 / math.sqrt(cfg.d))
            _draw_fp8(up[e], su[e], g, 1.0 / math.sqrt(cfg.d))
            _draw_fp8(down[e], sd[e], g, 1.0 / math.sqrt(f))
        return gate, up, down, sg, su, sd

    (out["w_gate"], out["w_up"], out["w_down"], out["w_gate_scale"], out["w_up_scale"],
     out["w_down_scale"]) = stack("routed", cfg.N, cfg.F)
    for k in ("ws_gate", "ws_up", "ws_down", "ws_gate_scale", "ws_up_scale", "ws_down_scale"):
        out[k] = None
    if cfg.S > 0:
        (out["ws_gate"], out["ws_up"], out["ws_down"], out["ws_gate_scale"], out["ws_up_scale"],
         out["ws_down_scale"]) = stack("shared", cfg.S, cfg.Fs)
    return out


def make_expert_weights(cfg: MoEConfig, seed: int = 0, device="cpu") -> dict:
    """Stacked bf16 expert weights on `device`:
    w_gate, w_up [N, F, d]; w_down [N, d, F]; ws_gate, ws_up [S, Fs, d];
    ws_down [S, d, Fs] (None when S == 0). FP8 configs: make_expert_weights_fp8."""
    if cfg.expert_dtype == "fp8":
        return make_expert_weights_fp8(cfg, seed, device)
    if cfg.expert_dtype == "mxfp4":
        return make_expert_weights_mxfp4(cfg, seed, device)
    device = torch.device(device)
    bf = torch.bfloat16
    w_gate = torch.empty(cfg.N, cfg.F, cfg.d, dtype=bf, device=device)
    w_up = torch.empty_like(w_gate)
    w_down = torch.empty(cfg.N, cfg.d, cfg.F, dtype=bf, device=device)
    g = torch.Generator(device=device)
    for e in range(cfg.N):
        g.manual_seed(_seed(seed, "routed", e))
        _draw_bf16(w_gate[e], g, 1.0 / math.sqrt(cfg.d))
        _draw_bf16(w_up[e], g, 1.0 / math.sqrt(cfg.d))
        _draw_bf16(w_down[e], g, 1.0 / math.sqrt(cfg.F))
    ws_gate = ws_up = ws_down = None
    if cfg.S > 0:
        ws_gate = torch.empty(cfg.S, cfg.Fs, cfg.d, dtype=bf, device=device)
        ws_up = torch.empty_like(ws_gate)
        ws_down = torch.empty(cfg.S, cfg.d, cfg.Fs, dtype=bf, device=device)
        for s in range(cfg.S):
            g.manual_seed(_seed(seed, "shared", s))
            _draw_bf16(ws_gate[s], g, 1.0 / math.sqrt(cfg.d))
            _draw_bf16(ws_up[s], g, 1.0 / math.sqrt(cfg.d))
            _draw_bf16(ws_down[s], g, 1.0 / math.sqrt(cfg.Fs))
    return dict(w_gate=w_gate, w_up=w_up, w_down=w_down, ws_gate=ws_gate, ws_up=ws_up,
                ws_down=ws_down)


def make_inputs(cfg: MoEConfig, seed: int = 0, device="cpu") -> dict:
    """Router-side inputs (CPU) plus expert weights on `device`."""
    out = make_router_inputs(cfg, seed)
    out.update(make_expert_weights(cfg, seed, device))
    return out
