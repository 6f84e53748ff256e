"""Pins of the oracle (CPU only).

Each test ties the oracle to something other than itself: a worked example
printed on the pages, a library routine (numpy / scipy / torch), a closed form,
an invariant the pages state, or brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import oracle
from mixture_experts_layer_94_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(a):
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _identity_router(logits):
    """hidden = logits and W_router = I, so the router's logits are the given values."""
    logits = np.asarray(logits, dtype=np.float32)[None, :]
    return logits, np.eye(logits.shape[1], dtype=np.float32)


# ---------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------

def test_p5_worked_example_top2_softmax_over_pair():
    """"Mixture of Experts Explained", 'The router, with real numbers'."""
    g = _golden("p5_router_example.json")
    pr = g["printed"]
    x, W = _identity_router(g["logits"])
    r = oracle.router(x, W, K=2, score_fn=oracle.SOFTMAX, renormalize=1)
    assert (r["idx"][0] + 1).tolist() == pr["top2_experts_1based"]
    l1, l2 = r["logits"][0, r["idx"][0]]
    assert round(math.exp(l1), 1) == pr["exp_winner1"]
    assert round(math.exp(l2), 1) == pr["exp_winner2"]
    assert abs(math.exp(l1) + math.exp(l2) - pr["exp_sum"]) < 0.05
    assert round(r["w"][0, 0], 3) == pr["gate_winner1"]
    assert round(r["w"][0, 1], 3) == pr["gate_winner2"]
    # The page's "about" values for the full 8-way softmax of the winners.
    p = r["probs"][0, r["idx"][0]]
    assert abs(p[0] - pr["full_softmax_winner1_about"]) < 0.005
    assert abs(p[1] - pr["full_softmax_winner2_about"]) < 0.005
    assert abs(p.sum() - pr["full_softmax_pair_sum_about"]) < 0.005
    # Without renormalisation the weights are those full-softmax values.
    r0 = oracle.router(x, W, K=2, score_fn=oracle.SOFTMAX, renormalize=0)
    np.testing.assert_allclose(r0["w"][0], p, rtol=0, atol=1e-15)


def test_p2_worked_example_router_and_mix():
    """"AI Infrastructure series Part 12", 'How does the router decide? A worked
    example': full softmax, keep two, renormalise, mix the two expert vectors."""
    g = _golden("p2_router_example.json")
    pr = g["printed"]
    x, W = _identity_router(g["reconstructed_logits"])
    assert abs(np.exp(np.asarray(g["reconstructed_logits"])).sum() - pr["exp_sum"]) < 0.005
    r = oracle.router(x, W, K=2, score_fn=oracle.SOFTMAX, renormalize=1)
    assert (r["idx"][0] + 1).tolist() == pr["winners_1based"]
    p = r["probs"][0, r["idx"][0]]
    assert round(p[0], 3) == pr["prob_winner1"]
    assert round(p[1], 3) == pr["prob_winner2"]
    assert round(p.sum(), 3) == pr["prob_pair_sum"]
    assert round(r["w"][0, 0], 2) == pr["weight_winner1"]
    assert round(r["w"][0, 1], 2) == pr["weight_winner2"]
    y = np.array([pr["expert_out_winner1_prefix"], pr["expert_out_winner2_prefix"]])
    out = oracle.combine(r["w"][0], y)
    np.testing.assert_allclose(out, g["output_prefix_from_printed_weights"], atol=0.006)
    # And exactly the printed-weight arithmetic when fed the printed weights.
    out_printed = oracle.combine([pr["weight_winner1"], pr["weight_winner2"]], y)
    np.testing.assert_allclose(out_printed, g["output_prefix_from_printed_weights"], atol=5e-4)


# ---------------------------------------------------------------------------
# Router: library routines, equivalences the pages state, brute force
# ---------------------------------------------------------------------------

def _rand_router_case(rng, T, d, N, dup_cols=0):
    x = rng.standard_normal((T, d)).astype(np.float32)
    W = (rng.standard_normal((d, N)) / math.sqrt(d)).astype(np.float32)
    for _ in range(dup_cols):  # exact ties: two experts with identical router columns
        a, b = rng.choice(N, size=2, replace=False)
        W[:, b] = W[:, a]
    return x, W


def test_logits_match_library_matmul_with_router_bias():
    rng = np.random.default_rng(1)
    x, W = _rand_router_case(rng, 200, 96, 16)
    b = rng.standard_normal(16).astype(np.float32)
    r = oracle.router(x, W, K=3, router_bias=b)
    ref = (x.astype(np.float64) @ W.astype(np.float64) + b).astype(np.float32)
    ulp = np.spacing(np.abs(ref)).astype(np.float64)
    assert np.all(np.abs(r["logits"] - ref) <= ulp)


def test_softmax_over_topk_equals_full_softmax_renormalised():
    """"Chapter 19", §19.3.2: softmax over the selected logits equals softmax
    over all logits, then Top-K, then renormalisation ("AI Infrastructure
    series Part 12": Mixtral's top-two softmax gives the same weights)."""
    rng = np.random.default_rng(2)
    x, W = _rand_router_case(rng, 10000, 32, 8)
    r = oracle.router(x, W, K=2, score_fn=oracle.SOFTMAX, renormalize=1)
    full = scipy.special.softmax(r["logits"], axis=1)           # library softmax
    np.testing.assert_allclose(r["probs"], full, rtol=1e-12, atol=1e-15)
    chosen = np.take_along_axis(full, r["idx"].astype(np.int64), axis=1)
    ren = chosen / chosen.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(r["w"], ren, rtol=0, atol=1e-12)


@pytest.mark.parametrize("score_fn", [oracle.SOFTMAX, oracle.SIGMOID])
def test_weights_sum_to_one(score_fn):
    """"Mixture of Experts for LLM Inference", 'Opening the router': the survivors
    are renormalised so the budget adds back to 1."""
    rng = np.random.default_rng(3)
    x, W = _rand_router_case(rng, 3000, 40, 32)
    sb = rng.standard_normal(32).astype(np.float32) * 0.3 if score_fn == oracle.SIGMOID else None
    for K in (1, 2, 8, 32):
        r = oracle.router(x, W, K=K, score_fn=score_fn, sel_bias=sb)
        np.testing.assert_allclose(r["w"].sum(axis=1), 1.0, rtol=0, atol=1e-12)
        assert np.all(r["w"] >= 0)


def test_sigmoid_selection_bias_hand_case():
    """DeepSeek-V3 style ("Chapter 19", §19.3.4; "AI Infrastructure series Part
    12", worked example): sigmoid scores, a bias that shifts selection only,
    chosen scores normalised to sum to 1."""
    logits = [2.0, 1.0, 0.5, -1.0]
    sel = np.array([0.0, 0.0, 0.5, 0.0], np.float32)
    x, W = _identity_router(logits)
    s = scipy.special.expit(np.asarray(logits, np.float64))     # library sigmoid
    r = oracle.router(x, W, K=2, score_fn=oracle.SIGMOID, sel_bias=sel)
    # keys: s + b = [0.881, 0.731, 1.122, 0.269]: the bias moves expert 2 to the top
    assert r["idx"][0].tolist() == [2, 0]
    np.testing.assert_allclose(r["w"][0], [s[2] / (s[2] + s[0]), s[0] / (s[2] + s[0])],
                               rtol=0, atol=1e-12)
    # without the bias the selection is the two largest logits
    r0 = oracle.router(x, W, K=2, score_fn=oracle.SIGMOID)
    assert r0["idx"][0].tolist() == [0, 1]
    np.testing.assert_allclose(r0["w"][0], [s[0] / (s[0] + s[1]), s[1] / (s[0] + s[1])],
                               rtol=0, atol=1e-12)
    # no renormalisation -> the raw sigmoid scores of the chosen experts
    r1 = oracle.router(x, W, K=2, score_fn=oracle.SIGMOID, sel_bias=sel, renormalize=0)
    np.testing.assert_allclose(r1["w"][0], [s[2], s[0]], rtol=0, atol=1e-12)


def test_sigmoid_zero_bias_selects_top_logits():
    rng = np.random.default_rng(4)
    x, W = _rand_router_case(rng, 2000, 64, 64)
    r = oracle.router(x, W, K=8, score_fn=oracle.SIGMOID)
    ref = np.argsort(-r["logits"], axis=1, kind="stable")[:, :8]
    ok = r["margin"] > 0
    assert ok.mean() > 0.99
    assert np.array_equal(r["idx"][ok], ref[ok])


@pytest.mark.parametrize("score_fn", [oracle.SOFTMAX, oracle.SIGMOID])
def test_topk_equals_brute_force_sort_with_ties(score_fn):
    """Top-K equals a full stable sort by (key descending, expert ascending),
    including exact ties made by duplicated router columns."""
    rng = np.random.default_rng(5)
    for N in (1, 2, 3, 5, 8):
        x, W = _rand_router_case(rng, 300, 12, N, dup_cols=1 if N >= 2 else 0)
        sb = (rng.standard_normal(N) * 0.2).astype(np.float32) if score_fn else None
        if sb is not None and N >= 2:
            sb[1] = sb[0]  # keep some ties alive through the bias
        lg = (x.astype(np.float64) @ W.astype(np.float64)).astype(np.float32)
        if score_fn == oracle.SOFTMAX:
            keys = lg
        else:
            keys = (scipy.special.expit(lg.astype(np.float64)) + sb.astype(np.float64)).astype(np.float32)
        for K in range(1, N + 1):
            r = oracle.router(x, W, K=K, score_fn=score_fn, sel_bias=sb)
            assert np.all(np.abs(r["keys"].astype(np.float64) - keys) <=
                          np.spacing(np.abs(keys)).astype(np.float64))
            ks = r["keys"]
            for t in range(x.shape[0]):
                order = sorted(range(N), key=lambda e: (-float(ks[t, e]), e))
                assert r["idx"][t].tolist() == order[:K]


def test_margin_definition_hand_case():
    x, W = _identity_router([3.0, 2.0, 2.5, 0.0])
    r = oracle.router(x, W, K=2)
    assert r["idx"][0].tolist() == [0, 2]
    assert r["margin"][0] == pytest.approx(0.5)          # gaps 0.5 (3->2.5) and 0.5 (2.5->2)
    x, W = _identity_router([3.0, 3.0, 1.0])
    r = oracle.router(x, W, K=1)
    assert r["idx"][0].tolist() == [0] and r["margin"][0] == 0.0
    x, W = _identity_router([1.0, 4.0, 2.0])
    r = oracle.router(x, W, K=3)                           # K == N: all consecutive gaps
    assert r["idx"][0].tolist() == [1, 2, 0] and r["margin"][0] == pytest.approx(1.0)


# ---------------------------------------------------------------------------
# Route and pack: invariants and a library stable sort
# ---------------------------------------------------------------------------

def _random_topk(rng, T, N, K, skew=False):
    idx = np.empty((T, K), np.int32)
    p = None
    if skew:
        p = 1.0 / np.arange(1, N + 1) ** 1.5
        p /= p.sum()
    for t in range(T):
        idx[t] = rng.choice(N, size=K, replace=False, p=p)
    return idx


@pytest.mark.parametrize("T,N,K,skew", [(0, 4, 2, False), (1, 8, 8, False), (37, 8, 2, False),
                                        (500, 64, 6, True), (300, 256, 8, True)])
def test_permute_invariants_and_stable_sort(T, N, K, skew):
    rng = np.random.default_rng(6)
    idx = _random_topk(rng, T, N, K, skew)
    p = oracle.permute(idx, N)
    flat = idx.reshape(-1)
    assert np.array_equal(p["counts"], np.bincount(flat, minlength=N))
    assert np.array_equal(p["offsets"], np.concatenate([[0], np.cumsum(p["counts"])]))
    assert p["counts"].sum() == T * K
    assert np.array_equal(p["perm_src"], np.argsort(flat, kind="stable").astype(np.int32))
    assert np.array_equal(p["inv_row"][p["perm_src"]], np.arange(T * K))
    for e in range(N):  # each expert's segment: that expert only, tokens ascending
        seg = p["perm_src"][p["offsets"][e]:p["offsets"][e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg // K) > 0)


def test_permute_rejects_out_of_range_index():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 9]], np.int32), 8)


# ---------------------------------------------------------------------------
# Expert FFN, combine and the whole layer: closed forms and library routines
# ---------------------------------------------------------------------------

def test_silu_closed_form():
    assert oracle.silu(0.0) == 0.0
    for z in (-20.0, -3.0, -0.5, 0.7, 1.0, 4.0, 30.0):
        assert oracle.silu(z) == pytest.approx(z * scipy.special.expit(z), rel=1e-14, abs=1e-300)
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)


def _torch_swiglu(x, wg, wu, wd):
    """Dense SwiGLU FFN from torch library routines, fp64."""
    x = torch.as_tensor(x, dtype=torch.float64)
    g = torch.as_tensor(_bf16_to_f64(wg)) @ x
    u = torch.as_tensor(_bf16_to_f64(wu)) @ x
    return (torch.as_tensor(_bf16_to_f64(wd)) @ (torch.nn.functional.silu(g) * u)).numpy()


def test_expert_ffn_matches_torch():
    rng = np.random.default_rng(7)
    d, F = 24, 40
    x = rng.standard_normal(d)
    wg = _bf16_bits(rng.standard_normal((F, d)) / math.sqrt(d))
    wu = _bf16_bits(rng.standard_normal((F, d)) / math.sqrt(d))
    wd = _bf16_bits(rng.standard_normal((d, F)) / math.sqrt(F))
    y = oracle.expert_ffn(x, wg, wu, wd)
    np.testing.assert_allclose(y, _torch_swiglu(x, wg, wu, wd), rtol=1e-12, atol=1e-14)


def _rand_experts(rng, n, d, F):
    return ([_bf16_bits(rng.standard_normal((F, d)) / math.sqrt(d)) for _ in range(n)],
            [_bf16_bits(rng.standard_normal((F, d)) / math.sqrt(d)) for _ in range(n)],
            [_bf16_bits(rng.standard_normal((d, F)) / math.sqrt(F)) for _ in range(n)])


def test_K_equals_N_is_dense_softmax_mixture():
    """K = N with renormalisation: every expert runs and the weights are the full
    softmax, so the layer is the textbook dense mixture sum_e softmax(l)_e E_e(x)."""
    rng = np.random.default_rng(8)
    T, d, N, F = 6, 16, 4, 20
    x, W = _rand_router_case(rng, T, d, N)
    wg, wu, wd = _rand_experts(rng, N, d, F)
    r = oracle.layer(x, W, wg, wu, wd, K=N)
    lg = torch.as_tensor((x.astype(np.float64) @ W.astype(np.float64)).astype(np.float32),
                         dtype=torch.float64)
    p = torch.softmax(lg, dim=1).numpy()
    ref = np.stack([sum(p[t, e] * _torch_swiglu(x[t].astype(np.float64), wg[e], wu[e], wd[e])
                        for e in range(N)) for t in range(T)])
    np.testing.assert_allclose(r["out"], ref, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("score_fn", [oracle.SOFTMAX, oracle.SIGMOID])
def test_single_expert_is_dense_ffn(score_fn):
    """N = K = 1: the router always picks the one expert with weight 1 and the
    layer is a dense SwiGLU FFN."""
    rng = np.random.default_rng(9)
    T, d, F = 5, 32, 48
    x, W = _rand_router_case(rng, T, d, 1)
    wg, wu, wd = _rand_experts(rng, 1, d, F)
    r = oracle.layer(x, W, wg, wu, wd, K=1, score_fn=score_fn)
    assert np.all(r["idx"] == 0) and np.all(r["w"] == 1.0)
    ref = np.stack([_torch_swiglu(x[t].astype(np.float64), wg[0], wu[0], wd[0]) for t in range(T)])
    np.testing.assert_allclose(r["out"], ref, rtol=1e-10, atol=1e-13)


def test_shared_expert_alone_when_routed_outputs_vanish():
    """"Mixture of Experts for LLM Inference", 'Shared experts': the shared expert
    runs for every token outside the router; with the routed experts' W_down all
    zero the layer output is exactly the shared FFN."""
    rng = np.random.default_rng(10)
    T, d, N, K, F, Fs = 7, 16, 6, 2, 24, 40
    x, W = _rand_router_case(rng, T, d, N)
    wg, wu, _ = _rand_experts(rng, N, d, F)
    wd = [np.zeros((d, F), np.uint16) for _ in range(N)]
    sg, su, sd = _rand_experts(rng, 1, d, Fs)
    r = oracle.layer(x, W, wg, wu, wd, K=K, score_fn=oracle.SIGMOID, ws_gate=sg, ws_up=su,
                     ws_down=sd)
    ref = np.stack([_torch_swiglu(x[t].astype(np.float64), sg[0], su[0], sd[0]) for t in range(T)])
    np.testing.assert_allclose(r["out"], ref, rtol=1e-10, atol=1e-13)
    # two shared experts add up
    sg2, su2, sd2 = _rand_experts(rng, 1, d, Fs)
    r2 = oracle.layer(x, W, wg, wu, wd, K=K, ws_gate=sg + sg2, ws_up=su + su2, ws_down=sd + sd2)
    ref2 = ref + np.stack([_torch_swiglu(x[t].astype(np.float64), sg2[0], su2[0], sd2[0])
                           for t in range(T)])
    np.testing.assert_allclose(r2["out"], ref2, rtol=1e-10, atol=1e-13)


def test_layer_matches_independent_numpy_on_tiny_workload():
    """Cross-check (not a pin): an independent numpy fp64 statement of the whole
    layer on the tiny workload agrees with the C oracle."""
    cfg = inputs.TINY
    ins = inputs.make_inputs(cfg, seed=0)
    x = ins["hidden"].numpy().astype(np.float32)
    W = ins["w_router"].numpy()
    bits = {k: ins[k].view(torch.int16).numpy().view(np.uint16) for k in ("w_gate", "w_up", "w_down")}
    r = oracle.layer(x, W, list(bits["w_gate"]), list(bits["w_up"]), list(bits["w_down"]), K=cfg.K)
    lg = (x.astype(np.float64) @ W.astype(np.float64)).astype(np.float32).astype(np.float64)
    idx = np.argsort(-lg, axis=1, kind="stable")[:, :cfg.K]
    assert np.array_equal(idx, r["idx"])
    sel = np.take_along_axis(lg, idx, axis=1)
    w = np.exp(sel - sel[:, :1])
    w /= w.sum(axis=1, keepdims=True)
    wg, wu, wd = (_bf16_to_f64(bits[k]) for k in ("w_gate", "w_up", "w_down"))
    out = np.zeros((cfg.T, cfg.d))
    for t in range(cfg.T):
        for k in range(cfg.K):
            e = idx[t, k]
            g = wg[e] @ x[t].astype(np.float64)
            u = wu[e] @ x[t].astype(np.float64)
            out[t] += w[t, k] * (wd[e] @ (g / (1 + np.exp(-g)) * u))
    np.testing.assert_allclose(r["out"], out, rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------------------
# Generator sanity and stored constants
# ---------------------------------------------------------------------------

def test_union_of_touched_experts_follows_independent_routing_formula():
    """"AI Infrastructure series Part 12", 'What happens when many users share the
    GPU?' and "Mixture of Experts Explained", 'Why batching erodes the advantage':
    with independent routing, B tokens picking k of N touch N(1-(1-k/N)^B)
    distinct experts on average. A sanity check of the decode workload's
    Gaussian router, not of the oracle."""
    cfg = inputs.QWEN_DECODE
    for T in (8, 32):
        counts = []
        for seed in range(6):
            ri = inputs.make_router_inputs(cfg.with_(T=T), seed=seed)
            r = oracle.router(ri["hidden"].float().numpy(), ri["w_router"].numpy(), K=cfg.K)
            counts.append(len(np.unique(r["idx"])))
        p = 1 - (1 - cfg.K / cfg.N) ** T
        mean, sd = cfg.N * p, math.sqrt(cfg.N * p * (1 - p))
        assert all(abs(c - mean) <= 4 * sd for c in counts), (T, counts, mean, sd)


def test_mixtral_router_scale_constant_matches_fixture():
    g = _golden("mixtral_router_scale.json")
    assert g["router_scale"] == inputs.MIXTRAL_ROUTER_SCALE
    assert abs(g["top1_share_at_scale"] - 0.40) < 0.002


# ---------------------------------------------------------------------------
# Group-limited (node-limited) routing
# ---------------------------------------------------------------------------

def test_group_limited_routing_hand_case():
    """"Mixture of Experts for LLM Inference", 'Three tricks that tame the
    all-to-alls' (node-limited routing caps how many nodes a token may visit):
    8 experts in 4 groups of 2; a group's score is the sum of its two largest
    keys."""
    x, W = _identity_router([5.0, 0.0, 4.9, 4.8, 1.0, 1.0, 0.5, 0.2])
    # group scores: g0 5.0, g1 9.7, g2 2.0, g3 0.7
    assert oracle.router(x, W, K=2)["idx"][0].tolist() == [0, 2]
    r1 = oracle.router(x, W, K=2, n_groups=4, topk_groups=1)
    assert r1["idx"][0].tolist() == [2, 3]
    # margin: group-score gaps (9.7 -> 5.0) and key gaps among the allowed picks (4.9 -> 4.8)
    assert r1["margin"][0] == pytest.approx(0.1, abs=1e-6)
    r2 = oracle.router(x, W, K=2, n_groups=4, topk_groups=2)
    assert r2["idx"][0].tolist() == [0, 2]
    # weights: softmax over the chosen logits, as without groups
    e = np.exp(np.array([4.9, 4.8]) - 4.9)
    np.testing.assert_allclose(r1["w"][0], e / e.sum(), atol=1e-7)


@pytest.mark.parametrize("score_fn", [oracle.SOFTMAX, oracle.SIGMOID])
def test_group_limit_reduces_to_plain_topk_when_all_groups_kept(score_fn):
    rng = np.random.default_rng(11)
    x, W = _rand_router_case(rng, 500, 24, 16)
    sb = (rng.standard_normal(16) * 0.3).astype(np.float32) if score_fn else None
    ref = oracle.router(x, W, K=4, score_fn=score_fn, sel_bias=sb)
    for ng in (1, 4):
        r = oracle.router(x, W, K=4, score_fn=score_fn, sel_bias=sb, n_groups=ng, topk_groups=ng)
        assert np.array_equal(r["idx"], ref["idx"])
        np.testing.assert_array_equal(r["w"], ref["w"])


@pytest.mark.parametrize("N,G,M,K", [(16, 4, 2, 4), (12, 6, 3, 5), (256, 8, 4, 8)])
def test_group_limited_routing_against_library_sorts(N, G, M, K):
    """Chosen experts lie in at most M groups, the kept groups are the M best by
    (sum of the two largest keys, lower index first), and the chosen experts are
    the stable top-K of the keys restricted to those groups."""
    rng = np.random.default_rng(N + G)
    x, W = _rand_router_case(rng, 300, 32, N)
    sb = (rng.standard_normal(N) * 0.3).astype(np.float32)
    r = oracle.router(x, W, K=K, score_fn=oracle.SIGMOID, sel_bias=sb, n_groups=G, topk_groups=M)
    keys = r["keys"].astype(np.float64)
    gs = N // G
    for t in range(x.shape[0]):
        groups_used = set((r["idx"][t] // gs).tolist())
        assert len(groups_used) <= M
        gk = np.sort(keys[t].reshape(G, gs), axis=1)[:, ::-1]
        gscore = gk[:, 0] + (gk[:, 1] if gs > 1 else 0.0)
        kept = np.lexsort((np.arange(G), -gscore))[:M]
        allowed = np.zeros(N, bool)
        for g in kept:
            allowed[g * gs:(g + 1) * gs] = True
        cand = np.nonzero(allowed)[0]
        order = cand[np.lexsort((cand, -keys[t][cand]))]
        assert r["idx"][t].tolist() == order[:K].tolist()


# ---------------------------------------------------------------------------
# Capacity-limited routing
# ---------------------------------------------------------------------------

def test_capacity_formula():
    """"Chapter 19", §19.6.1: C = ceil(c T K / N)."""
    assert oracle.capacity(1.0, 4096, 2, 8) == 1024
    assert oracle.capacity(1.25, 100, 3, 7) == math.ceil(1.25 * 100 * 3 / 7)
    assert oracle.capacity(0.0, 100, 3, 7) == -1


def test_capacity_hand_case_drops_the_later_tokens():
    """Four tokens all pick expert 0: with c = 1 (C = ceil(4 * 1 / 2) = 2) the
    first two keep their copy, the last two pass on the residual alone
    ("Mixture of Experts Explained", 'Routing collapses unless you stop it')."""
    idx = np.array([[0], [0], [0], [0]], np.int32)
    p = oracle.permute(idx, 2, capacity_factor=1.0)
    assert p["counts"].tolist() == [4, 0]
    assert p["offsets"].tolist() == [0, 2, 2]
    assert p["perm_src"][:2].tolist() == [0, 1]
    assert p["inv_row"].tolist() == [0, 1, -1, -1]


@pytest.mark.parametrize("c", [0.5, 1.0, 1.25])
def test_capacity_permute_against_library_sort(c):
    rng = np.random.default_rng(12)
    idx = _random_topk(rng, 400, 16, 3, skew=True)
    cap = oracle.capacity(c, 400, 3, 16)
    p = oracle.permute(idx, 16, capacity_factor=c)
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")           # library stable sort
    counts = np.bincount(flat, minlength=16)
    kept = np.minimum(counts, cap)
    assert np.array_equal(p["counts"], counts)
    assert np.array_equal(p["offsets"], np.concatenate([[0], np.cumsum(kept)]))
    start = np.concatenate([[0], np.cumsum(counts)])
    expect = np.concatenate([order[start[e]:start[e] + kept[e]] for e in range(16)])
    assert np.array_equal(p["perm_src"][:kept.sum()], expect)
    inv = np.full(flat.size, -1)
    inv[expect] = np.arange(expect.size)
    assert np.array_equal(p["inv_row"], inv)
    # a huge factor is dropless
    q = oracle.permute(idx, 16, capacity_factor=1e6)
    assert np.array_equal(q["perm_src"], oracle.permute(idx, 16)["perm_src"])


def test_layer_keep_mask_drops_whole_copies():
    """A dropped copy contributes nothing and the kept weights are not
    renormalised: out = sum over kept k of w_k E_k(x)."""
    rng = np.random.default_rng(13)
    T, d, N, K, F = 6, 16, 4, 2, 20
    x, W = _rand_router_case(rng, T, d, N)
    wg, wu, wd = _rand_experts(rng, N, d, F)
    keep = np.ones((T, K), np.uint8)
    keep[1, 0] = keep[3, 1] = keep[4, :] = 0
    r = oracle.layer(x, W, wg, wu, wd, K=K, keep=keep)
    full = oracle.layer(x, W, wg, wu, wd, K=K)
    assert np.array_equal(r["w"], full["w"])
    for t in range(T):
        ref = sum(full["w"][t, k] * _torch_swiglu(x[t].astype(np.float64), wg[r["idx"][t, k]],
                                                  wu[r["idx"][t, k]], wd[r["idx"][t, k]])
                  for k in range(K) if keep[t, k]) if keep[t].any() else np.zeros(d)
        np.testing.assert_allclose(r["out"][t], ref, rtol=1e-10, atol=1e-13)


# ---------------------------------------------------------------------------
# Expert-choice routing
# ---------------------------------------------------------------------------

def test_expert_choice_hand_case():
    """"Mixture of Experts for LLM Inference", 'Token choice vs expert choice':
    each expert picks its own top tokens up to a fixed capacity; a token nobody
    picks is skipped for that layer."""
    logits = np.array([[2.0, 0.0], [0.0, 2.0], [1.0, 1.0], [3.0, 0.0]], np.float32)
    W = np.eye(2, dtype=np.float32)
    # softmax scores: expert 0 column [0.881, 0.119, 0.5, 0.953]; expert 1 [0.119, 0.881, 0.5, 0.047]
    r = oracle.expert_choice(logits, W, C=2)
    assert r["row_token"].tolist() == [[0, 3], [1, 2]]
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(r["row_w"], [[p[0, 0], p[3, 0]], [p[1, 1], p[2, 1]]], atol=1e-7)
    r1 = oracle.expert_choice(logits, W, C=1)
    assert r1["row_token"].tolist() == [[3], [1]]  # tokens 0 and 2 are picked by nobody
    idx, w = oracle.routing_from_expert_choice(r1["row_token"], r1["row_w"], 4)
    assert idx[0].tolist() == [-1] and idx[2].tolist() == [-1]


@pytest.mark.parametrize("score_fn", [oracle.SOFTMAX, oracle.SIGMOID])
def test_expert_choice_against_library_sort(score_fn):
    """Balanced by construction (every expert takes exactly C tokens) and each
    expert's tokens are its C best scores (stable: lower token first)."""
    rng = np.random.default_rng(14)
    T, d, N = 300, 24, 8
    x, W = _rand_router_case(rng, T, d, N)
    C = oracle.expert_choice_capacity(1.0, T, 2, N)
    assert C == math.ceil(T * 2 / N)
    r = oracle.expert_choice(x, W, C, score_fn=score_fn)
    lg = (x.astype(np.float64) @ W.astype(np.float64)).astype(np.float32).astype(np.float64)
    S = scipy.special.softmax(lg, axis=1) if score_fn == oracle.SOFTMAX else scipy.special.expit(lg)
    S32 = S.astype(np.float32)
    for e in range(N):
        assert r["row_token"].shape[1] == C
        if r["margin"][e] < 1e-6:
            continue
        pick = np.lexsort((np.arange(T), -S32[:, e].astype(np.float64)))[:C]
        assert r["row_token"][e].tolist() == sorted(pick.tolist())
        np.testing.assert_allclose(r["row_w"][e], S[r["row_token"][e], e], atol=1e-7)


def test_expert_choice_with_every_token_is_the_dense_mixture():
    """C = T: every expert takes every token, so the layer is
    sum_e softmax(l)_e E_e(x): the token-choice layer with K = N."""
    rng = np.random.default_rng(15)
    T, d, N, F = 9, 16, 4, 24
    x, W = _rand_router_case(rng, T, d, N)
    wg, wu, wd = _rand_experts(rng, N, d, F)
    r = oracle.expert_choice(x, W, C=T)
    idx, w = oracle.routing_from_expert_choice(r["row_token"], r["row_w"], T)
    out = oracle.layer_routed(x, idx, w, wg, wu, wd)
    dense = oracle.layer(x, W, wg, wu, wd, K=N)["out"]
    np.testing.assert_allclose(out, dense, rtol=1e-9, atol=1e-12)


def test_layer_routed_matches_token_choice_layer():
    """layer_routed under the router's own top-K routing is the token-choice layer."""
    rng = np.random.default_rng(16)
    T, d, N, K, F = 7, 16, 6, 2, 20
    x, W = _rand_router_case(rng, T, d, N)
    wg, wu, wd = _rand_experts(rng, N, d, F)
    ref = oracle.layer(x, W, wg, wu, wd, K=K)
    out = oracle.layer_routed(x, ref["idx"], ref["w"], wg, wu, wd)
    np.testing.assert_allclose(out, ref["out"], rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- FP8 E4M3 experts


def test_e4m3_decode_closed_form_points():
    # OCP 8-bit floating point, E4M3: bias 7, no infinities, S.1111.111 is NaN.
    assert oracle.e4m3_value(0x00) == 0.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9            # smallest subnormal: 1/8 * 2^-6
    assert oracle.e4m3_value(0x07) == 7 * 2.0 ** -9        # largest subnormal
    assert oracle.e4m3_value(0x08) == 2.0 ** -6            # smallest normal
    assert oracle.e4m3_value(0x38) == 1.0                  # exponent 7 = bias
    assert oracle.e4m3_value(0x3C) == 1.5
    assert oracle.e4m3_value(0x7E) == 448.0                # largest finite
    assert math.isnan(oracle.e4m3_value(0x7F))
    assert math.isnan(oracle.e4m3_value(0xFF))
    z = oracle.e4m3_value(0x80)
    assert z == 0.0 and math.copysign(1.0, z) < 0
    assert oracle.e4m3_value(0xFE) == -448.0


def test_e4m3_decode_matches_torch_float8_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decode_is_monotone_and_sign_symmetric():
    pos = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    assert np.all(np.diff(pos) > 0)
    neg = np.array([oracle.e4m3_value(c | 0x80) for c in range(0x7F)])
    assert np.array_equal(neg, -pos)


def _fp8_case(rng, F, d, pow2_scales):
    """E4M3 codes (no NaN) and row scales, plus the same weights as bf16 bits
    (exact when the scales are powers of two: a code has at most 4 significant
    bits, bf16 holds 8)."""
    def mat(rows, cols):
        q = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] ^= 0x01  # NaN -> the largest finite code of that sign
        if pow2_scales:
            s = np.ldexp(1.0, rng.integers(-12, -4, size=rows)).astype(np.float32)
        else:
            s = rng.uniform(1e-4, 3e-3, size=rows).astype(np.float32)
        vals = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        w = vals * s.astype(np.float64)[:, None]
        return q, s, w
    qg, sg, wg = mat(F, d)
    qu, su, wu = mat(F, d)
    qd, sd, wd = mat(d, F)
    return (qg, sg, qu, su, qd, sd), (wg, wu, wd)


def test_expert_ffn_fp8_equals_bf16_expert_on_exact_weights():
    rng = np.random.default_rng(11)
    F, d = 24, 40
    (qg, sg, qu, su, qd, sd), (wg, wu, wd) = _fp8_case(rng, F, d, pow2_scales=True)
    bits = [_bf16_bits(m) for m in (wg, wu, wd)]
    for m, b in zip((wg, wu, wd), bits):
        assert np.array_equal(_bf16_to_f64(b), m)  # the weights are exact in bf16
    x = rng.standard_normal(d)
    h8, y8 = oracle.expert_ffn_fp8(x, qg, sg, qu, su, qd, sd, return_h=True)
    h16, y16 = oracle.expert_ffn(x, *bits, return_h=True)
    assert np.array_equal(h8, h16)
    assert np.array_equal(y8, y16)


def test_expert_ffn_fp8_row_scales_factor_out():
    # A per-row scale multiplies that row's dot product: u_f (hence h_f, since
    # h = SiLU(g) * u) scales with s_up[f], and y_i with s_down[i].
    rng = np.random.default_rng(12)
    F, d = 16, 32
    (qg, sg, qu, su, qd, sd), _ = _fp8_case(rng, F, d, pow2_scales=False)
    x = rng.standard_normal(d)
    ones_u, ones_d = np.ones(F, np.float32), np.ones(d, np.float32)
    h, y = oracle.expert_ffn_fp8(x, qg, sg, qu, su, qd, sd, return_h=True)
    h1, _ = oracle.expert_ffn_fp8(x, qg, sg, qu, ones_u, qd, sd, return_h=True)
    np.testing.assert_allclose(h, h1 * su.astype(np.float64), rtol=1e-13, atol=0)
    _, y1 = oracle.expert_ffn_fp8(x, qg, sg, qu, su, qd, ones_d, return_h=True)
    np.testing.assert_allclose(y, y1 * sd.astype(np.float64), rtol=1e-13, atol=1e-300)


def test_layer_fp8_equals_bf16_layer_on_exact_weights():
    rng = np.random.default_rng(13)
    T, d, N, K, F, Fs = 9, 32, 4, 2, 16, 24
    hidden = rng.standard_normal((T, d)).astype(np.float32)
    w_router = rng.standard_normal((d, N)).astype(np.float32)
    routed = [_fp8_case(rng, F, d, True) for _ in range(N)]
    shared = [_fp8_case(rng, Fs, d, True)]
    q = lambda cases, j: [c[0][j] for c in cases]  # noqa: E731
    b = lambda cases, j: [_bf16_bits(c[1][j]) for c in cases]  # noqa: E731
    got = oracle.layer_fp8(hidden, w_router, q(routed, 0), q(routed, 1), q(routed, 2), q(routed, 3),
                           q(routed, 4), q(routed, 5), K=K, score_fn=oracle.SIGMOID,
                           qs_gate=q(shared, 0), ss_gate=q(shared, 1), qs_up=q(shared, 2),
                           ss_up=q(shared, 3), qs_down=q(shared, 4), ss_down=q(shared, 5))
    ref = oracle.layer(hidden, w_router, b(routed, 0), b(routed, 1), b(routed, 2), K=K,
                       score_fn=oracle.SIGMOID, ws_gate=b(shared, 0), ws_up=b(shared, 1),
                       ws_down=b(shared, 2))
    assert np.array_equal(got["idx"], ref["idx"])
    assert np.array_equal(got["w"], ref["w"])
    assert np.array_equal(got["out"], ref["out"])


def test_fp8_input_codes_decode_to_the_drawn_weights():
    # The generator's codes times their row scale reproduce the normal draw to
    # E4M3 precision (relative step 2^-3 for normal codes), and never hit NaN.
    cfg = inputs.TINY.with_(expert_dtype="fp8")
    w = inputs.make_expert_weights(cfg, seed=3)
    q = w["w_gate"][0].numpy()
    assert not np.any((q & 0x7F) == 0x7F)
    s = w["w_gate_scale"][0].numpy().astype(np.float64)
    vals = np.vectorize(oracle.e4m3_value)(q) * s[:, None]
    assert np.allclose(np.abs(vals).max(axis=1), 448.0 * s, rtol=0, atol=0)
    std = vals.std()
    assert abs(std - 1.0 / math.sqrt(cfg.d)) < 0.1 / math.sqrt(cfg.d)


def test_layer_routed_fp8_equals_bf16_on_exact_weights():
    rng = np.random.default_rng(14)
    T, d, N, M, F, Fs = 7, 32, 3, 3, 16, 16
    hidden = rng.standard_normal((T, d)).astype(np.float32)
    idx = rng.integers(-1, N, size=(T, M)).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(T, M))
    routed = [_fp8_case(rng, F, d, True) for _ in range(N)]
    shared = [_fp8_case(rng, Fs, d, True)]
    q = lambda cases, j: [c[0][j] for c in cases]  # noqa: E731
    b = lambda cases, j: [_bf16_bits(c[1][j]) for c in cases]  # noqa: E731
    got = oracle.layer_routed_fp8(hidden, idx, w, q(routed, 0), q(routed, 1), q(routed, 2), q(routed, 3),
                                  q(routed, 4), q(routed, 5), qs_gate=q(shared, 0), ss_gate=q(shared, 1),
                                  qs_up=q(shared, 2), ss_up=q(shared, 3), qs_down=q(shared, 4),
                                  ss_down=q(shared, 5))
    ref = oracle.layer_routed(hidden, idx, w, b(routed, 0), b(routed, 1), b(routed, 2), ws_gate=b(shared, 0),
                              ws_up=b(shared, 1), ws_down=b(shared, 2))
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- MXFP4 experts

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP MX: FP4 E2M1 magnitudes, codes 0..7


def test_e2m1_and_e8m0_decode():
    for c in range(16):
        v = oracle.e2m1_value(c)
        mag = E2M1_TABLE[c & 7]
        assert v == (-mag if c & 8 else mag)
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert oracle.e8m0_value(120) == 2.0 ** -7
    assert math.isnan(oracle.e8m0_value(255))


def _mxfp4_case(rng, rows, cols, e_lo=118, e_hi=126):
    """Weights built as E2M1 values x per-block powers of two, then packed by
    the OCP layout (element 2i in the low nibble); returns (codes, scales, w)."""
    mags = rng.integers(0, 8, size=(rows, cols))
    signs = rng.integers(0, 2, size=(rows, cols))
    exps = rng.integers(e_lo, e_hi + 1, size=(rows, cols // 32)).astype(np.uint8)
    w = (np.array(E2M1_TABLE)[mags] * np.where(signs == 1, -1.0, 1.0) *
         np.ldexp(1.0, np.repeat(exps.astype(np.int64) - 127, 32, axis=1)))
    codes4 = (mags | (signs << 3)).astype(np.uint8)
    packed = (codes4[:, 0::2] | (codes4[:, 1::2] << 4)).astype(np.uint8)
    return packed, exps, w


def test_expert_ffn_mxfp4_equals_bf16_expert_on_exact_weights():
    # E2M1 values times powers of two have at most two significant bits:
    # exact in bf16, so the MXFP4 expert must equal the bf16 expert bit for bit.
    rng = np.random.default_rng(21)
    F, d = 64, 96
    qg, bg, wg = _mxfp4_case(rng, F, d)
    qu, bu, wu = _mxfp4_case(rng, F, d)
    qd, bd, wd = _mxfp4_case(rng, d, F)
    bits = [_bf16_bits(m) for m in (wg, wu, wd)]
    for m, b in zip((wg, wu, wd), bits):
        assert np.array_equal(_bf16_to_f64(b), m)
    x = rng.standard_normal(d)
    h4, y4 = oracle.expert_ffn_mxfp4(x, qg, bg, qu, bu, qd, bd, return_h=True)
    h16, y16 = oracle.expert_ffn(x, *bits, return_h=True)
    assert np.array_equal(h4, h16) and np.array_equal(y4, y16)


def test_layer_mxfp4_equals_bf16_layer_on_exact_weights():
    rng = np.random.default_rng(22)
    T, d, N, K, F, Fs = 7, 64, 4, 2, 32, 64
    hidden = rng.standard_normal((T, d)).astype(np.float32)
    w_router = rng.standard_normal((d, N)).astype(np.float32)
    routed = [(_mxfp4_case(rng, F, d), _mxfp4_case(rng, F, d), _mxfp4_case(rng, d, F)) for _ in range(N)]
    shared = [(_mxfp4_case(rng, Fs, d), _mxfp4_case(rng, Fs, d), _mxfp4_case(rng, d, Fs))]
    q = lambda cases, m, j: [c[m][j] for c in cases]  # noqa: E731
    b = lambda cases, m: [_bf16_bits(c[m][2]) for c in cases]  # noqa: E731
    got = oracle.layer_mxfp4(hidden, w_router, q(routed, 0, 0), q(routed, 0, 1), q(routed, 1, 0),
                             q(routed, 1, 1), q(routed, 2, 0), q(routed, 2, 1), K=K, qs_gate=q(shared, 0, 0),
                             bs_gate=q(shared, 0, 1), qs_up=q(shared, 1, 0), bs_up=q(shared, 1, 1),
                             qs_down=q(shared, 2, 0), bs_down=q(shared, 2, 1))
    ref = oracle.layer(hidden, w_router, b(routed, 0), b(routed, 1), b(routed, 2), K=K, ws_gate=b(shared, 0),
                       ws_up=b(shared, 1), ws_down=b(shared, 2))
    assert np.array_equal(got["idx"], ref["idx"])
    assert np.array_equal(got["out"], ref["out"])


def test_layer_routed_mxfp4_equals_bf16_on_exact_weights():
    """The MXFP4 routed layer (a given routing, slots with index -1 skipped)
    equals the bf16 routed layer bit for bit on weights exact in both formats,
    and equals the MXFP4 token-choice layer under that layer's own routing."""
    rng = np.random.default_rng(23)
    T, d, N, M, F, Fs = 7, 64, 4, 3, 32, 64
    hidden = rng.standard_normal((T, d)).astype(np.float32)
    idx = rng.integers(-1, N, size=(T, M)).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(T, M))
    routed = [(_mxfp4_case(rng, F, d), _mxfp4_case(rng, F, d), _mxfp4_case(rng, d, F)) for _ in range(N)]
    shared = [(_mxfp4_case(rng, Fs, d), _mxfp4_case(rng, Fs, d), _mxfp4_case(rng, d, Fs))]
    q = lambda cases, m, j: [c[m][j] for c in cases]  # noqa: E731
    b = lambda cases, m: [_bf16_bits(c[m][2]) for c in cases]  # noqa: E731
    mx = dict(qs_gate=q(shared, 0, 0), bs_gate=q(shared, 0, 1), qs_up=q(shared, 1, 0), bs_up=q(shared, 1, 1),
              qs_down=q(shared, 2, 0), bs_down=q(shared, 2, 1))
    got = oracle.layer_routed_mxfp4(hidden, idx, w, q(routed, 0, 0), q(routed, 0, 1), q(routed, 1, 0),
                                    q(routed, 1, 1), q(routed, 2, 0), q(routed, 2, 1), **mx)
    ref = oracle.layer_routed(hidden, idx, w, b(routed, 0), b(routed, 1), b(routed, 2), ws_gate=b(shared, 0),
                              ws_up=b(shared, 1), ws_down=b(shared, 2))
    assert np.array_equal(got, ref)
    w_router = rng.standard_normal((d, N)).astype(np.float32)
    tc = oracle.layer_mxfp4(hidden, w_router, q(routed, 0, 0), q(routed, 0, 1), q(routed, 1, 0), q(routed, 1, 1),
                            q(routed, 2, 0), q(routed, 2, 1), K=2, **mx)
    again = oracle.layer_routed_mxfp4(hidden, tc["idx"], tc["w"], q(routed, 0, 0), q(routed, 0, 1),
                                      q(routed, 1, 0), q(routed, 1, 1), q(routed, 2, 0), q(routed, 2, 1), **mx)
    np.testing.assert_allclose(again, tc["out"], rtol=1e-12, atol=1e-14)
