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


def _group_sets(cfg, keys_row, tol):
    """Every set of topk_groups expert groups that is a top-topk_groups choice
    of the group scores up to `tol` (each kept score >= each dropped score -
    tol). A group's score is the sum of its two largest keys (its one key for
    groups of one); groups are consecutive expert indices. Without a group
    limit: the one set of all experts."""
    import itertools

    N = keys_row.shape[0]
    if cfg is None or cfg.n_groups <= 1 or cfg.topk_groups >= cfg.n_groups:
        return [np.arange(N)]
    gs = N // cfg.n_groups
    kg = np.sort(keys_row.astype(np.float64).reshape(cfg.n_groups, gs), axis=1)[:, ::-1]
    score = kg[:, 0] + (kg[:, 1] if gs > 1 else 0.0)
    thr = np.sort(score)[::-1][cfg.topk_groups - 1]
    cand = [g for g in range(cfg.n_groups) if score[g] >= thr - tol]
    sets = []
    for G in itertools.combinations(cand, cfg.topk_groups):
        rest = [g for g in range(cfg.n_groups) if g not in G]
        if not rest or min(score[list(G)]) >= max(score[rest]) - tol:
            sets.append(np.concatenate([np.arange(g * gs, (g + 1) * gs) for g in G]))
    return sets


def topk_is_valid(cfg, chosen, keys_row, tol=MARGIN_TIE):
    """True when `chosen` (slot order) is a correct top-K of the oracle's fp32
    selection keys up to `tol`, the case where several answers are correct:
    distinct in-range experts, slots in descending key order, and inside some
    valid choice of groups every chosen key >= every unchosen key - tol."""
    N = keys_row.shape[0]
    chosen = np.asarray(chosen)
    if len(set(chosen.tolist())) != len(chosen) or chosen.min() < 0 or chosen.max() >= N:
        return False
    k = keys_row.astype(np.float64)
    if np.any(k[chosen[1:]] > k[chosen[:-1]] + tol):
        return False
    for allowed in _group_sets(cfg, keys_row, tol):
        if not np.isin(chosen, allowed).all():
            continue
        others = np.setdiff1d(allowed, chosen)
        if others.size == 0 or k[chosen].min() >= k[others].max() - tol:
            return True
    return False


def weights_for_choice(cfg, chosen, ref, t):
    """The gate weights the router's formula gives token t on the expert set
    `chosen`, from the oracle's logits and scores: softmax over the chosen
    logits, or the chosen sigmoid scores over their sum; without
    renormalisation the full-softmax probability or the raw score."""
    chosen = np.asarray(chosen)
    score_fn = 0 if cfg is None else cfg.score_fn
    renorm = 1 if cfg is None else cfg.renormalize
    if not renorm:
        return ref["probs"][t, chosen]
    if score_fn == 0:
        l = ref["logits"][t, chosen]
        e = np.exp(l - l.max())
        return e / e.sum()
    s = ref["probs"][t, chosen]
    return s / s.sum()


def compare_router(gpu_idx: np.ndarray, gpu_w: np.ndarray, ref: dict, cfg=None):
    """Bit-exact indices on tokens with margin >= 1e-5; weights within 1e-5
    where the indices agree. A token whose indices differ must be a near tie
    (margin < 1e-5), its GPU choice a valid top-K under the oracle's fp32
    keys (topk_is_valid), and its GPU weights the router formula's on the
    GPU's choice within 1e-5. `ref` is oracle.router's output (keys, logits
    and probs are needed for the differing tokens). Returns the near-tie
    report with the formula weights of the differing tokens."""
    near = ref["margin"] < MARGIN_TIE
    same = np.all(gpu_idx == ref["idx"], axis=1)
    bad = ~same & ~near
    assert not bad.any(), f"index mismatch on {int(bad.sum())} tokens with margin >= 1e-5: {np.nonzero(bad)[0][:10]}"
    dw = np.abs(gpu_w.astype(np.float64) - ref["w"])[same]
    assert dw.size == 0 or dw.max() <= W_ATOL, f"gate weight error {dw.max()}"
    flipped = np.nonzero(~same)[0]
    w_flip = np.zeros((flipped.size, gpu_idx.shape[1]))
    for i, t in enumerate(flipped):
        assert topk_is_valid(cfg, gpu_idx[t], ref["keys"][t]), \
            f"token {t}: GPU choice {gpu_idx[t]} is not a top-K of the keys (oracle {ref['idx'][t]})"
        w_flip[i] = weights_for_choice(cfg, gpu_idx[t], ref, t)
        err = np.abs(gpu_w[t].astype(np.float64) - w_flip[i]).max()
        assert err <= W_ATOL, f"token {t}: gate weights on the GPU's choice off by {err}"
    return dict(near_ties=int(near.sum()), near_tie_flips=int(flipped.size),
                flipped_tokens=flipped, flipped_w=w_flip)


def oracle_rows_routed(cfg, ins, rows, idx, w):
    """Oracle layer outputs for `rows` under a given routing (idx [n][M], -1 =
    no contribution; w fp64 [n][M]), in the workload's expert format. Only
    the experts the routing names are copied to the host."""
    rows = np.asarray(rows, dtype=np.int64)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    used = sorted(set(idx[idx >= 0].reshape(-1).tolist()))
    x = hidden_f32(ins)[rows]
    fmt = cfg.expert_dtype
    if fmt in ("fp8", "mxfp4"):
        sconv = u8 if fmt == "mxfp4" else np32
        q = {k: [None] * cfg.N for k in ("w_gate", "w_up", "w_down")}
        sc = {k: [None] * cfg.N for k in ("w_gate_scale", "w_up_scale", "w_down_scale")}
        for e in used:
            for k in q:
                q[k][e] = u8(ins[k][e])
            for k in sc:
                sc[k][e] = sconv(ins[k][e])
        sh = {}
        if cfg.S > 0:
            sk = "bs" if fmt == "mxfp4" else "ss"
            for k, a in (("ws_gate", "gate"), ("ws_up", "up"), ("ws_down", "down")):
                sh["qs_" + a] = [u8(ins[k][s]) for s in range(cfg.S)]
                sh[f"{sk}_{a}"] = [sconv(ins[k + "_scale"][s]) for s in range(cfg.S)]
        fn = oracle.layer_routed_mxfp4 if fmt == "mxfp4" else oracle.layer_routed_fp8
        if not used:  # the oracle needs one expert's matrices to size F
            used = [0]
            for k in q:
                q[k][0] = u8(ins[k][0])
            for k in sc:
                sc[k][0] = sconv(ins[k][0])
        return fn(x, idx, w, q["w_gate"], sc["w_gate_scale"], q["w_up"], sc["w_up_scale"], q["w_down"],
                  sc["w_down_scale"], **sh)
    wts = {k: [None] * cfg.N for k in ("w_gate", "w_up", "w_down")}
    for e in (used or [0]):
        for k in wts:
            wts[k][e] = bf16_bits(ins[k][e])
    sh = {}
    if cfg.S > 0:
        sh = {k: [bf16_bits(ins[k][s]) for s in range(cfg.S)] for k in ("ws_gate", "ws_up", "ws_down")}
    return oracle.layer_routed(x, idx, w, wts["w_gate"], wts["w_up"], wts["w_down"], **sh)


def reference_outputs(cfg, ins, rows, ref_out, gpu_idx, rep, keep_all=None):
    """The oracle output for `rows` with every near-tie token the GPU routed
    differently recomputed under the GPU's own (validated) routing and the
    formula weights on it. ref_out: the oracle layer's output for `rows`;
    gpu_idx: the GPU's routing of the whole batch; keep_all: the capacity
    mask of the whole batch or None. Returns (outputs, number recomputed)."""
    rows = np.asarray(rows, dtype=np.int64)
    flipped = rep["flipped_tokens"]
    pos = {int(t): i for i, t in enumerate(flipped)}
    sel = [j for j, r in enumerate(rows.tolist()) if r in pos]
    out = np.array(ref_out, dtype=np.float64, copy=True)
    if not sel:
        return out, 0
    toks = rows[sel]
    idx = gpu_idx[toks].astype(np.int32).copy()
    if keep_all is not None:
        idx[keep_all[toks] == 0] = -1
    w = np.stack([rep["flipped_w"][pos[int(t)]] for t in toks])
    out[sel] = oracle_rows_routed(cfg, ins, toks, idx, w)
    return out, len(sel)


def segment_ends(idx, N, keep=None):
    """Tokens at the first and the last packed row of every expert: rows of an
    expert are in token order, so these are the smallest and largest tokens
    that kept a copy at it (the last row sits in the expert's last, usually
    ragged, tile)."""
    ends = set()
    for e in range(N):
        sel = idx == e
        if keep is not None:
            sel &= keep > 0
        toks = np.nonzero(sel.any(axis=1))[0]
        if toks.size:
            ends |= {int(toks[0]), int(toks[-1])}
    return ends


def compare_expert_choice(cfg, ins, C, row_token, row_w, offsets, name=""):
    """Expert-choice selection against the oracle: bit-exact tokens for every
    expert whose C-th / (C+1)-th score gap is >= 1e-5. An expert below that
    gap whose tokens differ must hold a valid top-C of the oracle's fp32
    scores (every picked score >= every unpicked one - 1e-5, tokens distinct
    and ascending). Every expert's weights are the oracle's scores of its
    tokens within 1e-5. Returns the number of near-tie experts."""
    ref = oracle.expert_choice(hidden_f32(ins), np32(ins["w_router"]), C, score_fn=cfg.score_fn,
                               router_bias=np32(ins.get("router_bias")))
    assert offsets.tolist() == [e * C for e in range(cfg.N + 1)]
    scores = oracle_router(cfg.with_(K=1), ins)["probs"]  # full softmax or sigmoid, fp64 [T][N]
    s32 = scores.astype(np.float32).astype(np.float64)
    exact = ref["margin"] >= MARGIN_TIE
    differ = 0
    for e in range(cfg.N):
        toks = row_token[e]
        if not np.array_equal(toks, ref["row_token"][e]):
            assert not exact[e], f"expert {e}: tokens differ at a score gap >= 1e-5"
            assert np.all(np.diff(toks) > 0) and toks.min() >= 0 and toks.max() < cfg.T, e
            rest = np.setdiff1d(np.arange(cfg.T), toks)
            assert rest.size == 0 or s32[toks, e].min() >= s32[rest, e].max() - MARGIN_TIE, e
            differ += 1
        assert np.abs(row_w[e].astype(np.float64) - scores[toks, e]).max() <= W_ATOL, e
    print(f"{name}: experts with a near tie at the capacity boundary {int((~exact).sum())} of {cfg.N}, "
          f"selection differs (checked) {differ}")
    return int((~exact).sum())


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
