"""The GPU acceptance checks themselves, on the CPU: where several top-K
answers are correct (near ties), a routing that differs from the oracle's must
still be a top-K of the oracle's keys with the router formula's weights, and
its outputs are compared under that routing. Mistakes are planted in a copy of
the oracle's own routing (standing in for a GPU result); each must fail."""
import numpy as np
import pytest

from mixture_experts_layer_94_b300 import inputs
from oracle import oracle
from tests import helpers as H


def _tie_case(score="softmax", n_groups=0, topk_groups=0, N=8, K=3, T=300, seed=3):
    """A router whose columns come in equal pairs (0=4, 1=5, 2=6, 3=7): every
    key is tied with its partner's, so with an odd K the K-th pick has an
    unchosen partner of equal key: a second correct answer."""
    cfg = inputs.MoEConfig("ties", T=T, d=32, N=N, K=K, F=32, score=score, n_groups=n_groups,
                           topk_groups=topk_groups)
    ins = inputs.make_router_inputs(cfg, seed=seed)
    W = ins["w_router"].clone()
    half = N // 2
    W[:, half:] = W[:, :half]
    ins["w_router"] = W
    return cfg, ins, H.oracle_router(cfg, ins)


def _swap_partner(cfg, ref, t):
    """The oracle's choice for token t with one expert replaced by its tied
    partner (e <-> e +- N/2), when the partner is not chosen; else None."""
    half = cfg.N // 2
    idx = ref["idx"][t].copy()
    for k, e in enumerate(idx):
        p = (e + half) % cfg.N
        if p not in idx:
            idx[k] = p
            return idx
    return None


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
def test_a_tied_alternative_is_accepted_and_checked(score):
    cfg, ins, ref = _tie_case(score)
    gpu_idx, gpu_w = ref["idx"].copy(), ref["w"].astype(np.float32)
    changed = []
    for t in range(cfg.T):
        alt = _swap_partner(cfg, ref, t)
        if alt is not None and ref["margin"][t] < H.MARGIN_TIE:
            # the partner has the same key, so slot order and weights stay the oracle's formula
            order = np.argsort(-ref["keys"][t][alt].astype(np.float64), kind="stable")
            gpu_idx[t] = alt[order]
            gpu_w[t] = H.weights_for_choice(cfg, gpu_idx[t], ref, t)
            changed.append(t)
    assert len(changed) > 20
    rep = H.compare_router(gpu_idx, gpu_w, ref, cfg)
    assert set(rep["flipped_tokens"].tolist()) == set(changed)


def test_an_invalid_choice_on_a_near_tie_token_fails():
    cfg, ins, ref = _tie_case()
    t = int(np.nonzero(ref["margin"] < H.MARGIN_TIE)[0][0])
    gpu_idx, gpu_w = ref["idx"].copy(), ref["w"].astype(np.float32)
    keys = ref["keys"][t].astype(np.float64)
    worst = int(np.argmin(keys))  # far below the chosen keys
    assert worst not in gpu_idx[t]
    gpu_idx[t, -1] = worst
    with pytest.raises(AssertionError, match="not a top-K"):
        H.compare_router(gpu_idx, gpu_w, ref, cfg)


def test_wrong_weights_on_a_flipped_token_fail():
    cfg, ins, ref = _tie_case()
    gpu_idx, gpu_w = ref["idx"].copy(), ref["w"].astype(np.float32)
    for t in range(cfg.T):
        alt = _swap_partner(cfg, ref, t)
        if alt is not None and ref["margin"][t] < H.MARGIN_TIE:
            gpu_idx[t] = alt
            gpu_w[t] = H.weights_for_choice(cfg, alt, ref, t)[::-1] + 0.01  # planted: weights off
            break
    with pytest.raises(AssertionError, match="gate weights"):
        H.compare_router(gpu_idx, gpu_w, ref, cfg)


def test_a_flip_at_a_clear_margin_fails():
    cfg = inputs.MoEConfig("clear", T=200, d=32, N=8, K=2, F=32)
    ins = inputs.make_router_inputs(cfg, seed=4)
    ref = H.oracle_router(cfg, ins)
    t = int(np.argmax(ref["margin"]))
    assert ref["margin"][t] >= 1e-3
    gpu_idx = ref["idx"].copy()
    gpu_idx[t] = gpu_idx[t][::-1]
    with pytest.raises(AssertionError, match="index mismatch"):
        H.compare_router(gpu_idx, ref["w"].astype(np.float32), ref, cfg)


def test_slot_order_against_the_keys_is_checked():
    cfg, ins, ref = _tie_case()
    t = next(t for t in range(cfg.T) if ref["margin"][t] < H.MARGIN_TIE and
             ref["keys"][t][ref["idx"][t][0]] > ref["keys"][t][ref["idx"][t][2]] + 1e-3)
    bad = ref["idx"][t][::-1].copy()  # the smallest chosen key first
    assert not H.topk_is_valid(cfg, bad, ref["keys"][t])
    assert H.topk_is_valid(cfg, ref["idx"][t], ref["keys"][t])


def test_group_limited_validity():
    """With a group limit, an alternative must lie in a valid choice of
    groups: a tied partner from a group outside the kept ones is invalid."""
    cfg, ins, ref = _tie_case("sigmoid", n_groups=4, topk_groups=2, N=16, K=3)
    for t in range(cfg.T):
        assert H.topk_is_valid(cfg, ref["idx"][t], ref["keys"][t])
    gs = cfg.N // cfg.n_groups
    kg = np.sort(ref["keys"].astype(np.float64).reshape(cfg.T, cfg.n_groups, gs), axis=2)[:, :, ::-1]
    score = kg[:, :, 0] + kg[:, :, 1]
    hits = 0
    for t in range(cfg.T):
        order = np.argsort(-score[t], kind="stable")
        if score[t][order[1]] - score[t][order[2]] < 1e-3:
            continue
        dropped = order[-1]
        e = dropped * gs + int(np.argmax(ref["keys"][t][dropped * gs:(dropped + 1) * gs]))
        alt = ref["idx"][t].copy()
        alt[-1] = e
        assert not H.topk_is_valid(cfg, alt, ref["keys"][t])
        hits += 1
    assert hits > 10


def test_outputs_of_a_flipped_token_use_the_gpus_routing():
    """reference_outputs recomputes exactly the flipped tokens, under the
    GPU's routing and formula weights; a GPU output computed under the
    oracle's routing for such a token would fail the comparison."""
    cfg, ins, ref = _tie_case(T=40)
    full = inputs.make_inputs(cfg, seed=3)
    full["w_router"] = ins["w_router"]
    gpu_idx, gpu_w = ref["idx"].copy(), ref["w"].astype(np.float32)
    t = next(t for t in range(cfg.T) if _swap_partner(cfg, ref, t) is not None and ref["margin"][t] < H.MARGIN_TIE)
    alt = _swap_partner(cfg, ref, t)
    gpu_idx[t] = alt[np.argsort(-ref["keys"][t][alt].astype(np.float64), kind="stable")]
    gpu_w[t] = H.weights_for_choice(cfg, gpu_idx[t], ref, t)
    rep = H.compare_router(gpu_idx, gpu_w, ref, cfg)
    rows = np.arange(cfg.T)
    lay = H.oracle_layer_rows(cfg, full, rows)
    got, n = H.reference_outputs(cfg, full, rows, lay["out"], gpu_idx, rep)
    assert n == 1
    under_gpu = H.oracle_rows_routed(cfg, full, [t], gpu_idx[t:t + 1], rep["flipped_w"][:1])
    np.testing.assert_array_equal(got[t], under_gpu[0])
    others = np.arange(cfg.T) != t
    np.testing.assert_array_equal(got[others], lay["out"][others])
    # the tied partner's expert differs, so the two references differ at t
    assert H.output_errors(lay["out"][t:t + 1], got[t:t + 1])["max_rel"] > 2e-2


def test_expert_choice_near_tie_validity():
    """An expert's alternative token set at an exact tie of its C-th score is
    accepted; a set holding a clearly lower score is rejected, and so are
    weights that are not the oracle's scores of the set."""
    cfg = inputs.MoEConfig("ec", T=64, d=32, N=4, K=1, F=32, routing="expert")
    ins = inputs.make_router_inputs(cfg, seed=5)
    C = oracle.expert_choice_capacity(0.0, cfg.T, cfg.K, cfg.N)
    ref0 = oracle.expert_choice(H.hidden_f32(ins), H.np32(ins["w_router"]), C, score_fn=cfg.score_fn)
    s0 = H.oracle_router(cfg, ins)["probs"]
    e = 0
    picked = ref0["row_token"][e]
    last = picked[np.argmin(s0[picked, e])]            # expert 0's C-th pick
    u = int(max(set(range(cfg.T)) - set(picked.tolist())))  # an unpicked token after it
    assert u > last
    ins["hidden"][u] = ins["hidden"][last]              # now u ties with the C-th pick
    ref = oracle.expert_choice(H.hidden_f32(ins), H.np32(ins["w_router"]), C, score_fn=cfg.score_fn)
    scores = H.oracle_router(cfg, ins)["probs"]
    assert ref["margin"][e] < H.MARGIN_TIE and u not in ref["row_token"][e]
    offsets = np.arange(cfg.N + 1) * C
    rt, rw = ref["row_token"].copy(), ref["row_w"].astype(np.float32)
    H.compare_expert_choice(cfg, ins, C, rt, rw, offsets)
    alt = np.sort(np.array([u if x == last else x for x in rt[e]]))
    rt[e], rw[e] = alt, scores[alt, e]
    H.compare_expert_choice(cfg, ins, C, rt, rw, offsets)  # the other correct answer
    bad_w = rw.copy()
    bad_w[e, 0] += 1e-3
    with pytest.raises(AssertionError):
        H.compare_expert_choice(cfg, ins, C, rt, bad_w, offsets)
    low = int(np.argmin(scores[:, e]))
    bad = rt.copy()
    bad[e] = np.sort(np.array([low if x == u else x for x in rt[e]]))
    bw = rw.copy()
    bw[e] = scores[bad[e], e]
    with pytest.raises(AssertionError):
        H.compare_expert_choice(cfg, ins, C, bad, bw, offsets)
