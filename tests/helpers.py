"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same inputs, and apply the acceptance bar.

Acceptance (fixed for this layer):
  * expert indices, per-expert counts and the permutation bit-exact; tokens
    whose oracle top-K margin is below 1e-5 are counted and reported apart;
  * gate weights within 1e-5 absolute (fp32 router);
  * layer outputs (bf16, fp32 accumulation): max|gpu - ref| <= 2e-2 * max|ref|
    and sum|gpu - ref| / sum|ref| <= 5e-3.
"""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_layer_94_b300 import inputs
from oracle import oracle

MARGIN_TIE = 1e-5
W_ATOL = 1e-5
MAX_REL = 2e-2
L1_REL = 5e-3


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def hidden_f32(ins) -> np.ndarray:
    return ins["hidden"].float().cpu().numpy()


def np32(t):
    return None if t is None else t.detach().cpu().float().numpy()


def oracle_router(cfg, ins, rows=None):
    x = hidden_f32(ins)
    if rows is not None:
        x = x[rows]
    return oracle.router(x, np32(ins["w_router"]), K=cfg.K, score_fn=cfg.score_fn,
                         renormalize=cfg.renormalize, router_bias=np32(ins.get("router_bias")),
                         sel_bias=np32(ins.get("sel_bias")), n_groups=cfg.n_groups,
                         topk_groups=cfg.topk_groups)


def capacity_keep(cfg, topk_idx):
    """uint8 [T][K]: 1 where a copy survives its expert's capacity, computed by
    the oracle's capacity-limited permutation of the given routing."""
    inv = oracle.permute(np.asarray(topk_idx, np.int32), cfg.N, capacity_factor=cfg.capacity_factor)["inv_row"]
    return (inv >= 0).reshape(-1, cfg.K).astype(np.uint8)


def u8(t) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def _oracle_layer_rows_fp8(cfg, ins, rows, used, keep):
    mx = cfg.expert_dtype == "mxfp4"
    sconv = u8 if mx else np32  # E8M0 block scales (MXFP4) or fp32 row scales (FP8)
    q = {k: [None] * cfg.N for k in ("w_gate", "w_up", "w_down")}
    sc = {k: [None] * cfg.N for k in ("w_gate_scale", "w_up_scale", "w_down_scale")}
    for e in used:
        for k in q:
            q[k][e] = u8(ins[k][e])
        for k in sc:
            sc[k][e] = sconv(ins[k][e])
    sh = {}
    if cfg.S > 0:
        sk = "bs" if mx else "ss"
        sh = dict(qs_gate=[u8(ins["ws_gate"][s]) for s in range(cfg.S)],
                  qs_up=[u8(ins["ws_up"][s]) for s in range(cfg.S)],
                  qs_down=[u8(ins["ws_down"][s]) for s in range(cfg.S)])
        sh[sk + "_gate"] = [sconv(ins["ws_gate_scale"][s]) for s in range(cfg.S)]
        sh[sk + "_up"] = [sconv(ins["ws_up_scale"][s]) for s in range(cfg.S)]
        sh[sk + "_down"] = [sconv(ins["ws_down_scale"][s]) for s in range(cfg.S)]
    fn = oracle.layer_mxfp4 if mx else oracle.layer_fp8
    return fn(hidden_f32(ins)[rows], np32(ins["w_router"]), q["w_gate"], sc["w_gate_scale"],
                            q["w_up"], sc["w_up_scale"], q["w_down"], sc["w_down_scale"], K=cfg.K,
                            score_fn=cfg.score_fn, renormalize=cfg.renormalize,
                            router_bias=np32(ins.get("router_bias")), sel_bias=np32(ins.get("sel_bias")),
                            n_groups=cfg.n_groups, topk_groups=cfg.topk_groups, keep=keep, **sh)


def oracle_layer_rows(cfg, ins, rows, keep=None):
    """Oracle layer output for the given token rows. Only the experts those
    tokens pick are copied to the host. keep: uint8 [len(rows)][K] capacity
    mask, or None (dropless). FP8 configs use the oracle's FP8 layer."""
    rows = np.asarray(rows, dtype=np.int64)
    r = oracle_router(cfg, ins, rows)
    used = sorted(set(r["idx"].reshape(-1).tolist()))
    if cfg.expert_dtype in ("fp8", "mxfp4"):
        return _oracle_layer_rows_fp8(cfg, ins, rows, used, keep)
    wg = [None] * cfg.N
    wu = [None] * cfg.N
    wd = [None] * cfg.N
    for e in used:
        wg[e] = bf16_bits(ins["w_gate"][e])
        wu[e] = bf16_bits(ins["w_up"][e])
        wd[e] = bf16_bits(ins["w_down"][e])
    sh = {}
    if cfg.S > 0:
        sh = dict(ws_gate=[bf16_bits(ins["ws_gate"][s]) for s in range(cfg.S)],
                  ws_up=[bf16_bits(ins["ws_up"][s]) for s in range(cfg.S)],
                  ws_down=[bf16_bits(ins["ws_down"][s]) for s in range(cfg.S)])
    return oracle.layer(hidden_f32(ins)[rows], np32(ins["w_router"]), wg, wu, wd, K=cfg.K,
                        score_fn=cfg.score_fn, renormalize=cfg.renormalize,
                        router_bias=np32(ins.get("router_bias")), sel_bias=np32(ins.get("sel_bias")),
                        n_groups=cfg.n_groups, topk_groups=cfg.topk_groups, keep=keep, **sh)


def output_errors(gpu: np.ndarray, ref: np.ndarray) -> dict:
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = np.abs(gpu - ref)
    mref = float(np.abs(ref).max()) if ref.size else 0.0
    sref = float(np.abs(ref).sum()) if ref.size else 0.0
    return dict(max_rel=float(diff.max()) / mref if ref.size and mref > 0 else float(diff.max(initial=0)),
                l1_rel=float(diff.sum()) / sref if sref > 0 else float(diff.sum()))


def assert_output_close(gpu, ref, what=""):
    e = output_errors(gpu, ref)
    assert e["max_rel"] <= MAX_REL and e["l1_rel"] <= L1_REL, f"{what}: {e}"
    return e


def compare_router(gpu_idx: np.ndarray, gpu_w: np.ndarray, ref: dict):
    """Bit-exact indices on tokens with margin >= 1e-5 (near ties reported),
    weights within 1e-5 wherever the indices agree. Returns the near-tie report."""
    near = ref["margin"] < MARGIN_TIE
    same = np.all(gpu_idx == ref["idx"], axis=1)
    bad = ~same & ~near
    assert not bad.any(), f"index mismatch on {int(bad.sum())} tokens with margin >= 1e-5: {np.nonzero(bad)[0][:10]}"
    dw = np.abs(gpu_w.astype(np.float64) - ref["w"])[same]
    assert dw.size == 0 or dw.max() <= W_ATOL, f"gate weight error {dw.max()}"
    return dict(near_ties=int(near.sum()), near_tie_flips=int((~same & near).sum()),
                flipped_tokens=np.nonzero(~same)[0])


def make_case(cfg, seed=0, device="cuda", expert_device=None):
    """Seeded inputs; router-side tensors on the CPU and a device copy of all."""
    ins = inputs.make_inputs(cfg, seed=seed, device=expert_device or "cpu")
    dev = {k: (None if v is None else v.to(device).contiguous()) for k, v in ins.items()}
    return ins, dev


def assert_same_but_summation_order(a, b, name):
    """Two runs of the same GEMMs: the down GEMM adds a token's K expert rows
    into fp32 with atomics, in no fixed order, so the bf16 outputs may differ
    by the rounding of that order: one bf16 ulp, or, where the K terms nearly
    cancel, the fp32 rounding of the terms themselves (bounded here by
    2^-16 of the largest output), in few elements."""
    a, b = a.float().cpu().numpy(), b.float().cpu().numpy()
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(a), np.abs(b)))[1] - 8)
    diff = np.abs(a - b)
    bound = ulp + np.ldexp(float(np.abs(a).max()), -16)
    assert (diff <= bound).all(), (name, float((diff - bound).max()))
    assert (diff > 0).mean() < 0.02, (name, float((diff > 0).mean()))
