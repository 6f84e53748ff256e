"""GPU parity: every C-ABI entry point and the whole layer against the oracle.

Run on a B300 with libmoe.so built. Inputs are the seeded synthetic workloads;
the oracle sees exactly the tensors the GPU sees.
"""
import math

import numpy as np
import pytest
import torch

from mixture_experts_layer_94_b300 import inputs
from oracle import oracle
from tests import helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from mixture_experts_layer_94_b300 import binding as B


def _dev(t):
    return None if t is None else t.cuda().contiguous()


# Small and mid-size workloads the full oracle finishes in seconds. They span
# several 128-row tiles, ragged row / column / K tails, empty experts, shared
# experts, both score functions and both hidden dtypes.
MID = {
    "tiny": inputs.TINY,
    "ragged_softmax": inputs.MoEConfig("ragged_softmax", T=300, d=264, N=16, K=4, F=392),
    "dsv3_like": inputs.MoEConfig("dsv3_like", T=333, d=256, N=64, K=6, F=200, S=1, Fs=136,
                                  score="sigmoid", sel_bias_var=0.1, zipf=1.1),
    "gptoss_like": inputs.MoEConfig("gptoss_like", T=200, d=320, N=32, K=4, F=320),
    "two_shared_f32": inputs.MoEConfig("two_shared_f32", T=130, d=128, N=8, K=2, F=128, S=2, Fs=64,
                                       hidden_dtype="f32"),
    "no_renorm_sigmoid": inputs.MoEConfig("no_renorm_sigmoid", T=97, d=192, N=12, K=3, F=96,
                                          score="sigmoid", renormalize=0),
    "no_renorm_softmax": inputs.MoEConfig("no_renorm_softmax", T=64, d=64, N=8, K=2, F=64,
                                          renormalize=0),
    "K_equals_N": inputs.MoEConfig("K_equals_N", T=70, d=128, N=4, K=4, F=136),
    "N_K_1": inputs.MoEConfig("N_K_1", T=129, d=128, N=1, K=1, F=256),
    "T1": inputs.MoEConfig("T1", T=1, d=256, N=16, K=4, F=128),
    "d72_tail": inputs.MoEConfig("d72_tail", T=150, d=72, N=6, K=2, F=40),
    # gate/up groups whose rows outweigh their 2F weight rows run their tiles n
    # fastest: 4 experts of about 1500 rows (6 pair row blocks x 3 column
    # blocks, a half tile at each group's end) and a shared expert of 3000 rows
    "n_fastest_pairs": inputs.MoEConfig("n_fastest_pairs", T=3000, d=320, N=4, K=2, F=384, S=1, Fs=256),
    # the tensor-core router on both sides of the shared-tile limit (N <= 80):
    # 80 experts with the three parts in one tile, 40 token blocks and a ragged
    # d (not a whole number of 64-wide k-blocks); 96 experts with a tile per part
    "router_merged_N80": inputs.MoEConfig("router_merged_N80", T=5000, d=1000, N=80, K=4, F=64),
    "router_parts_N96": inputs.MoEConfig("router_parts_N96", T=300, d=512, N=96, K=6, F=64, score="sigmoid",
                                         sel_bias_var=0.1),
    # router d-split paths (few token tiles): large N and small non-power-of-two N
    "decode_like_T3": inputs.MoEConfig("decode_like_T3", T=3, d=1024, N=128, K=8, F=64),
    "small_n_split_T5": inputs.MoEConfig("small_n_split_T5", T=5, d=2048, N=6, K=2, F=64,
                                         hidden_dtype="f32"),
    # batches of at most 8 tokens with N > 32 (split-d logits, one warp per token in the top-K)
    "fused_topk_grouped_T4": inputs.MoEConfig("fused_topk_grouped_T4", T=4, d=512, N=64, K=6, F=64, S=1, Fs=64,
                                              score="sigmoid", sel_bias_var=0.1, n_groups=8, topk_groups=3),
    "fused_topk_f32_T7": inputs.MoEConfig("fused_topk_f32_T7", T=7, d=384, N=256, K=8, F=64, hidden_dtype="f32",
                                          renormalize=0),
    "fused_topk_T8_N96": inputs.MoEConfig("fused_topk_T8_N96", T=8, d=256, N=96, K=4, F=64),
    # decode-sized batches (T <= 4): expert FFNs on the CUDA cores; ragged d (17
    # 16-byte units per row), a capacity limit, two shared experts, fp32 hidden
    "small_capacity_shared_f32": inputs.MoEConfig("small_capacity_shared_f32", T=4, d=136, N=8, K=3, F=72, S=2,
                                                  Fs=40, hidden_dtype="f32", score="sigmoid",
                                                  capacity_factor=0.5),
    "small_T2_ragged": inputs.MoEConfig("small_T2_ragged", T=2, d=200, N=32, K=4, F=104),
    # more one-kernel decode shapes: a single expert, K = N (a dense mixture),
    # no renormalisation, an FFN much wider than d with a wider shared expert,
    # 256 experts under a group limit, a d long enough for several router
    # loads per thread
    "decode_N1_K1_T2": inputs.MoEConfig("decode_N1_K1_T2", T=2, d=128, N=1, K=1, F=256),
    "decode_K_equals_N_T3": inputs.MoEConfig("decode_K_equals_N_T3", T=3, d=128, N=4, K=4, F=136),
    "decode_no_renorm_sigmoid_T4": inputs.MoEConfig("decode_no_renorm_sigmoid_T4", T=4, d=192, N=12, K=3, F=96,
                                                    score="sigmoid", renormalize=0),
    "decode_wide_ffn_T2": inputs.MoEConfig("decode_wide_ffn_T2", T=2, d=128, N=8, K=2, F=1000, S=1, Fs=1200),
    "decode_256_grouped_T4": inputs.MoEConfig("decode_256_grouped_T4", T=4, d=512, N=256, K=8, F=128, S=1,
                                              Fs=128, score="sigmoid", sel_bias_var=0.1, zipf=1.1, n_groups=8,
                                              topk_groups=4),
    "decode_long_d_T1": inputs.MoEConfig("decode_long_d_T1", T=1, d=16384, N=4, K=2, F=64, hidden_dtype="f32"),
    # T*K >= 8192 copies: the token-major row copy (ragged d; fp32 hidden with a shared
    # expert and a capacity limit)
    "scatter_copy_ragged": inputs.MoEConfig("scatter_copy_ragged", T=2100, d=264, N=16, K=4, F=136),
    "scatter_copy_f32_shared_capacity": inputs.MoEConfig("scatter_copy_f32_shared_capacity", T=1100, d=136, N=8,
                                                         K=8, F=72, S=1, Fs=64, hidden_dtype="f32",
                                                         capacity_factor=0.8),
    # group-limited routing: 8 groups of 8 experts, 3 groups per token
    "grouped_routing": inputs.MoEConfig("grouped_routing", T=333, d=256, N=64, K=6, F=200, S=1, Fs=136,
                                        score="sigmoid", sel_bias_var=0.1, zipf=1.1, n_groups=8,
                                        topk_groups=3),
    "grouped_softmax_f32": inputs.MoEConfig("grouped_softmax_f32", T=100, d=64, N=32, K=4, F=64,
                                            hidden_dtype="f32", n_groups=16, topk_groups=2),
    # capacity-limited routing: copies beyond ceil(c T K / N) per expert are dropped
    "capacity_ragged": inputs.MoEConfig("capacity_ragged", T=300, d=264, N=16, K=4, F=392,
                                        capacity_factor=0.75),
    "capacity_small_f32": inputs.MoEConfig("capacity_small_f32", T=40, d=128, N=8, K=2, F=64,
                                           hidden_dtype="f32", capacity_factor=0.6),
    # mean expert group >= 256 rows: 256-row tiles on 2-CTA clusters
    "pair_ragged": inputs.MoEConfig("pair_ragged", T=700, d=264, N=4, K=2, F=392),
    "pair_shared_sigmoid": inputs.MoEConfig("pair_shared_sigmoid", T=520, d=192, N=2, K=1, F=136, S=1,
                                            Fs=72, score="sigmoid", sel_bias_var=0.1),
}


def _run_layer(cfg, dev, T=None):
    layer = B.MoELayer(cfg, dev, T=T)
    T = cfg.T if T is None else T
    topk_idx = torch.empty(T, cfg.K, dtype=torch.int32, device="cuda")
    topk_w = torch.empty(T, cfg.K, dtype=torch.float32, device="cuda")
    counts = torch.empty(cfg.N, dtype=torch.int32, device="cuda")
    out = layer.forward(dev["hidden"], topk_idx=topk_idx, topk_w=topk_w, counts=counts)
    torch.cuda.synchronize()
    assert layer.status(T) == 0
    return out, topk_idx.cpu().numpy(), topk_w.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("name", list(MID))
def test_layer_matches_oracle(name):
    cfg = MID[name]
    ins, dev = H.make_case(cfg)
    out, idx, w, counts = _run_layer(cfg, dev)
    cap_keep = H.capacity_keep(cfg, idx) if cfg.capacity_factor > 0 else None
    ref = H.oracle_layer_rows(cfg, ins, np.arange(cfg.T), keep=cap_keep)
    rep = H.compare_router(idx, w, H.oracle_router(cfg, ins), cfg)
    assert np.array_equal(counts, np.bincount(idx.reshape(-1), minlength=cfg.N))
    if cap_keep is not None:
        assert cap_keep.min() == 0  # the case does drop copies
    ref_out, _ = H.reference_outputs(cfg, ins, np.arange(cfg.T), ref["out"], idx, rep, cap_keep)
    H.assert_output_close(out.float().cpu().numpy(), ref_out, name)
    print(f"{name}: near ties {rep['near_ties']}, routed differently (checked) {rep['near_tie_flips']}")


def test_layer_empty_batch():
    cfg = inputs.TINY.with_(T=0)
    _, dev = H.make_case(inputs.TINY)
    layer = B.MoELayer(cfg, dev)
    counts = torch.full((cfg.N,), -1, dtype=torch.int32, device="cuda")
    out = layer.forward(dev["hidden"][:0], counts=counts)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.d) and torch.all(counts == 0)


def test_layer_one_expert_takes_every_token():
    """A router bias that sends every token to expert 5 first: one group holds
    all T rows (many row tiles), the others get the second choices."""
    cfg = inputs.MoEConfig("hot", T=640, d=128, N=8, K=2, F=256)
    ins, dev = H.make_case(cfg)
    rb = torch.zeros(cfg.N)
    rb[5] = 50.0
    ins["router_bias"] = rb
    dev["router_bias"] = rb.cuda()
    out, idx, w, counts = _run_layer(cfg, dev)
    assert np.all(idx[:, 0] == 5) and counts[5] == cfg.T
    ref = H.oracle_layer_rows(cfg, ins, np.arange(cfg.T))
    rep = H.compare_router(idx, w, H.oracle_router(cfg, ins), cfg)
    ref_out, _ = H.reference_outputs(cfg, ins, np.arange(cfg.T), ref["out"], idx, rep)
    H.assert_output_close(out.float().cpu().numpy(), ref_out, "hot expert")


def test_layer_is_repeatable():
    cfg = MID["ragged_softmax"]
    _, dev = H.make_case(cfg)
    a = _run_layer(cfg, dev)[0]
    b = _run_layer(cfg, dev)[0]
    # fp32 scatter-add order may differ in the last bit of the fp32 sum; bf16 outputs agree to 1 ulp
    diff = (a.float() - b.float()).abs()
    assert float(diff.max()) <= float(a.float().abs().max()) * 2 ** -7


# --------------------------------------------------------------------------- router
ROUTER_CASES = ["tiny", "ragged_softmax", "dsv3_like", "no_renorm_sigmoid", "no_renorm_softmax",
                "K_equals_N", "N_K_1", "T1", "decode_like_T3", "small_n_split_T5", "grouped_routing",
                "grouped_softmax_f32", "router_merged_N80", "router_parts_N96"]


@pytest.mark.parametrize("name", ROUTER_CASES)
def test_router_matches_oracle(name):
    cfg = MID[name]
    ins = inputs.make_router_inputs(cfg, seed=1)
    p = B.problem(cfg)
    idx = torch.empty(cfg.T, cfg.K, dtype=torch.int32, device="cuda")
    w = torch.empty(cfg.T, cfg.K, dtype=torch.float32, device="cuda")
    logits = torch.empty(cfg.T, cfg.N, dtype=torch.float32, device="cuda")
    B.router_topk(p, _dev(ins["hidden"]), _dev(ins["w_router"]), idx, w,
                  router_bias=_dev(ins["router_bias"]), sel_bias=_dev(ins["sel_bias"]), logits=logits)
    torch.cuda.synchronize()
    ref = H.oracle_router(cfg, ins)
    rep = H.compare_router(idx.cpu().numpy(), w.cpu().numpy(), ref, cfg)
    print(f"{name}: near ties {rep['near_ties']}, routed differently (checked) {rep['near_tie_flips']}")
    lg = logits.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref["logits"]) <= 1e-5 * (1 + np.abs(ref["logits"])))


def test_router_exact_ties_break_to_lower_index():
    """Duplicated router columns give exactly equal logits on both sides."""
    cfg = inputs.MoEConfig("ties", T=200, d=64, N=8, K=3, F=8)
    ins = inputs.make_router_inputs(cfg, seed=2)
    W = ins["w_router"].clone()
    W[:, 6] = W[:, 1]
    W[:, 3] = W[:, 0]
    idx = torch.empty(cfg.T, cfg.K, dtype=torch.int32, device="cuda")
    w = torch.empty(cfg.T, cfg.K, dtype=torch.float32, device="cuda")
    B.router_topk(B.problem(cfg), _dev(ins["hidden"]), _dev(W), idx, w)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    for t in range(cfg.T):
        for a, b in ((1, 6), (0, 3)):
            if a in gi[t] and b in gi[t]:
                assert list(gi[t]).index(a) < list(gi[t]).index(b)


# --------------------------------------------------------------------------- permute
# T*K >= 8192 copies take the token-major copy (each hidden row read once, stored K times)
PERMUTE_CASES = [(1, 8, 2, False), (37, 8, 2, False), (500, 64, 6, True), (1000, 256, 8, True),
                 (4096, 8, 2, False), (33, 1, 1, False), (2100, 64, 4, True), (1100, 16, 8, True)]


@pytest.mark.parametrize("T,N,K,skew", PERMUTE_CASES)
@pytest.mark.parametrize("hidden_dtype,capacity_factor", [("bf16", 0.0), ("f32", 0.0), ("bf16", 0.8)])
def test_permute_bit_exact(T, N, K, skew, hidden_dtype, capacity_factor):
    rng = np.random.default_rng(T + N)
    p_e = None
    if skew:
        p_e = 1.0 / np.arange(1, N + 1) ** 1.5
        p_e /= p_e.sum()
    idx = np.stack([rng.choice(N, size=K, replace=False, p=p_e) for _ in range(T)]).astype(np.int32)
    d = 136
    cfg = inputs.MoEConfig("perm", T=T, d=d, N=N, K=K, F=8, hidden_dtype=hidden_dtype,
                           capacity_factor=capacity_factor)
    hidden = inputs.make_router_inputs(cfg, seed=3)["hidden"]
    p = B.problem(cfg)
    ws = B.new_workspace(p, B.CALL_PERMUTE)
    counts = torch.empty(N, dtype=torch.int32, device="cuda")
    offsets = torch.empty(N + 1, dtype=torch.int32, device="cuda")
    perm_src = torch.empty(T * K, dtype=torch.int32, device="cuda")
    inv_row = torch.empty(T * K, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(T * K, d, dtype=torch.bfloat16, device="cuda")
    B.permute(p, _dev(torch.from_numpy(idx)), _dev(hidden), counts, offsets, perm_src, inv_row, x_perm, ws)
    torch.cuda.synchronize()
    assert B.get_device_status(ws) == 0
    ref = oracle.permute(idx, N, capacity_factor=capacity_factor)
    placed = int(ref["offsets"][-1])
    got = dict(counts=counts, offsets=offsets, perm_src=perm_src, inv_row=inv_row)
    for k in ("counts", "offsets", "inv_row"):
        assert np.array_equal(got[k].cpu().numpy(), ref[k]), k
    assert np.array_equal(perm_src.cpu().numpy()[:placed], ref["perm_src"][:placed])
    expect = hidden.to(torch.bfloat16)[torch.from_numpy(ref["perm_src"][:placed] // K).long()]
    assert torch.equal(x_perm.cpu()[:placed].view(torch.int16), expect.view(torch.int16))


def test_permute_reports_out_of_range_index():
    cfg = inputs.MoEConfig("bad", T=40, d=64, N=8, K=2, F=8)
    idx = np.tile(np.array([[0, 1]], np.int32), (cfg.T, 1))
    idx[17, 1] = 9
    p = B.problem(cfg)
    ws = B.new_workspace(p, B.CALL_PERMUTE)
    hidden = torch.zeros(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    t = lambda *s, dt=torch.int32: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    B.permute(p, _dev(torch.from_numpy(idx)), hidden, t(cfg.N), t(cfg.N + 1), t(cfg.T * 2),
              t(cfg.T * 2), t(cfg.T * 2, cfg.d, dt=torch.bfloat16), ws)
    assert B.get_device_status(ws) == -6  # MOE_ERR_DEVICE_BOUNDS
    assert B.get_device_status(ws) == 0   # read-and-clear


def test_permute_out_of_range_index_token_major_copy():
    # 8200 copies: the token-major copy; the bad copy has no row (inv_row -1),
    # every placed row still holds its token's hidden row
    cfg = inputs.MoEConfig("bad_large", T=4100, d=64, N=8, K=2, F=8)
    idx = np.stack([np.arange(cfg.T) % 8, (np.arange(cfg.T) + 3) % 8], axis=1).astype(np.int32)
    idx[1234, 0] = -2
    p = B.problem(cfg)
    ws = B.new_workspace(p, B.CALL_PERMUTE)
    hidden = inputs.make_router_inputs(cfg, seed=5)["hidden"]
    t = lambda *s, dt=torch.int32: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    offsets, perm_src, inv_row = t(cfg.N + 1), t(cfg.T * 2), t(cfg.T * 2)
    x_perm = t(cfg.T * 2, cfg.d, dt=torch.bfloat16)
    B.permute(p, _dev(torch.from_numpy(idx)), _dev(hidden), t(cfg.N), offsets, perm_src, inv_row, x_perm, ws)
    assert B.get_device_status(ws) == -6  # MOE_ERR_DEVICE_BOUNDS
    assert inv_row.cpu().numpy()[1234 * 2] == -1
    placed = int(offsets.cpu().numpy()[-1])
    assert placed == cfg.T * 2 - 1
    src = perm_src.cpu().numpy()[:placed]
    expect = hidden.to(torch.bfloat16)[torch.from_numpy(src // 2).long()]
    assert torch.equal(x_perm.cpu()[:placed].view(torch.int16), expect.view(torch.int16))


# --------------------------------------------------------------------------- grouped SwiGLU
SWIGLU_CASES = [(128, 256, 8, 2, 64), (320, 200, 5, 2, 300), (72, 40, 3, 1, 130), (256, 512, 16, 4, 700),
                # pair tiles (mean group >= 256 rows), ragged rows / columns / K, an empty expert
                (128, 256, 2, 1, 600), (320, 200, 3, 2, 500)]


@pytest.mark.parametrize("d,F,N,K,T", SWIGLU_CASES)
def test_grouped_swiglu_matches_oracle(d, F, N, K, T):
    cfg = inputs.MoEConfig("gs", T=T, d=d, N=N, K=K, F=F)
    ins = inputs.make_inputs(cfg, seed=4)
    rng = np.random.default_rng(d + F)
    p_e = np.linspace(3.0, 0.0, N) ** 2 + 1e-9  # skewed, last expert (nearly) empty
    p_e[-1] = 0.0
    p_e /= p_e.sum()
    K_eff = min(K, int((p_e > 0).sum()))
    cfg = cfg.with_(K=K_eff)
    idx = np.stack([rng.choice(N, size=K_eff, replace=False, p=p_e) for _ in range(T)]).astype(np.int32)
    perm = oracle.permute(idx, N)
    hid = ins["hidden"]
    x_perm = hid[torch.from_numpy(perm["perm_src"] // K_eff).long()].to(torch.bfloat16).contiguous()
    p = B.problem(cfg)
    ws = B.new_workspace(p, B.CALL_GROUPED_SWIGLU)
    h = torch.empty(T * K_eff, F, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(T * K_eff, d, dtype=torch.bfloat16, device="cuda")
    B.grouped_swiglu(p, x_perm.cuda(), torch.from_numpy(perm["offsets"]).cuda(), _dev(ins["w_gate"]),
                     _dev(ins["w_up"]), _dev(ins["w_down"]), h, y, ws)
    torch.cuda.synchronize()
    assert B.get_device_status(ws) == 0
    hg, yg = h.float().cpu().numpy(), y.float().cpu().numpy()
    href = np.empty((T * K_eff, F))
    yref = np.empty((T * K_eff, d))
    xp = x_perm.float().numpy().astype(np.float64)
    for e in range(N):
        wg, wu, wd = (H.bf16_bits(ins[k][e]) for k in ("w_gate", "w_up", "w_down"))
        for r in range(perm["offsets"][e], perm["offsets"][e + 1]):
            href[r], yref[r] = oracle.expert_ffn(xp[r], wg, wu, wd, return_h=True)
    H.assert_output_close(hg, href, "h_perm")
    H.assert_output_close(yg, yref, "y_perm")


# --------------------------------------------------------------------------- combine
@pytest.mark.parametrize("T,K,d,shared,dropped", [(1, 1, 8, False, 0), (77, 2, 136, True, 0),
                                                  (300, 8, 512, False, 0), (64, 4, 64, True, 40)])
def test_combine_matches_oracle(T, K, d, shared, dropped):
    g = torch.Generator().manual_seed(T * K)
    y = torch.randn(T * K, d, generator=g).to(torch.bfloat16)
    perm = torch.randperm(T * K, generator=g).to(torch.int32)          # inv_row: a bijection
    if dropped:  # copies dropped by capacity: inv_row -1, they contribute nothing
        perm[torch.randperm(T * K, generator=g)[:dropped]] = -1
    w = torch.rand(T, K, generator=g)
    w = (w / w.sum(1, keepdim=True)).float()
    sh = torch.randn(T, d, generator=g).to(torch.bfloat16) if shared else None
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    p = B.problem(None, T=T, d_model=d, n_experts=max(K, 2), top_k=K, ffn=8, n_shared=0, shared_ffn=0,
                  score_fn=0, renormalize=1, hidden_dtype=1)
    B.combine(p, y.cuda(), perm.cuda(), w.cuda(), out, shared_out=_dev(sh))
    torch.cuda.synchronize()
    yf = y.double().numpy()
    rows = perm.long().numpy().reshape(T, K)
    wk = w.double().numpy() * (rows >= 0)
    ref = np.stack([oracle.combine(wk[t], yf[np.maximum(rows[t], 0)],
                                   None if sh is None else sh[t].double().numpy()) for t in range(T)])
    got = out.double().cpu().numpy()
    # one bf16 rounding of an fp32 sum: at most half an ulp of bf16 plus fp32 noise
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


# --------------------------------------------------------------------------- step-wise == fused
def test_stepwise_path_matches_fused_layer():
    cfg = MID["ragged_softmax"]
    ins, dev = H.make_case(cfg)
    fused, idx_f, w_f, _ = _run_layer(cfg, dev)
    p = B.problem(cfg)
    T, K, N, d, F = cfg.T, cfg.K, cfg.N, cfg.d, cfg.F
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    w = torch.empty(T, K, dtype=torch.float32, device="cuda")
    B.router_topk(p, dev["hidden"], dev["w_router"], idx, w)
    e = lambda *s, dt=torch.int32: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    counts, offsets, perm_src, inv_row = e(N), e(N + 1), e(T * K), e(T * K)
    x_perm = e(T * K, d, dt=torch.bfloat16)
    ws = B.new_workspace(p, B.CALL_LAYER_FORWARD)
    B.permute(p, idx, dev["hidden"], counts, offsets, perm_src, inv_row, x_perm, ws)
    h, y = e(T * K, F, dt=torch.bfloat16), e(T * K, d, dt=torch.bfloat16)
    B.grouped_swiglu(p, x_perm, offsets, dev["w_gate"], dev["w_up"], dev["w_down"], h, y, ws)
    out = e(T, d, dt=torch.bfloat16)
    B.combine(p, y, inv_row, w, out)
    torch.cuda.synchronize()
    assert B.get_device_status(ws) == 0
    assert np.array_equal(idx.cpu().numpy(), idx_f) and np.array_equal(w.cpu().numpy(), w_f)
    H.assert_output_close(out.float().cpu().numpy(), fused.float().cpu().numpy(), "stepwise vs fused")


# --------------------------------------------------------------------------- full-size workloads
def _sample_rows(T, n, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, T - 1} | set(rng.choice(T, size=min(T, n), replace=False).tolist())
    return np.array(sorted(rows))


FULL = [("mixtral", inputs.MIXTRAL, 64), ("gptoss", inputs.GPTOSS, 64), ("dsv3", inputs.DSV3, 64),
        ("dsv3_grouped", inputs.DSV3_GROUPED, 64), ("mixtral_capacity", inputs.MIXTRAL_CAPACITY, 64)] + [
    (f"qwen_decode_T{T}", inputs.QWEN_DECODE.with_(T=T), 64) for T in inputs.DECODE_BATCHES] + [
    # the one-kernel decode path at 2 and 4 tokens
    (f"qwen_decode_T{T}_one_kernel", inputs.QWEN_DECODE.with_(T=T), 4) for T in (2, 4)]


@pytest.mark.parametrize("name,cfg,n_sample", FULL, ids=[f[0] for f in FULL])
def test_full_size_workload(name, cfg, n_sample):
    """The full-size workloads through moe_layer_forward (the launch configuration
    the benchmark times): router and counts on every token; outputs on sampled
    tokens the oracle computes one by one: random ones, the first and last
    row of every expert, and every token the GPU routed differently at a
    near tie (checked under the GPU's routing)."""
    ins = inputs.make_inputs(cfg, seed=0, device="cuda")
    dev = {k: (None if v is None else v.cuda().contiguous()) for k, v in ins.items()}
    out, idx, w, counts = _run_layer(cfg, dev)
    ref_r = H.oracle_router(cfg, ins)
    rep = H.compare_router(idx, w, ref_r, cfg)
    if cfg.n_groups > 1:  # every token's experts lie in at most topk_groups groups
        gs = cfg.N // cfg.n_groups
        assert max(len(set((row // gs).tolist())) for row in idx) <= cfg.topk_groups
    # counts: the GPU's own histogram, and the oracle's up to the near-tie flips
    assert np.array_equal(counts, np.bincount(idx.reshape(-1), minlength=cfg.N))
    ref_counts = np.bincount(ref_r["idx"].reshape(-1), minlength=cfg.N)
    fl = rep["flipped_tokens"]
    delta = np.bincount(idx[fl].reshape(-1), minlength=cfg.N) - np.bincount(ref_r["idx"][fl].reshape(-1), minlength=cfg.N)
    assert np.array_equal(counts - ref_counts, delta)
    keep_all = H.capacity_keep(cfg, idx) if cfg.capacity_factor > 0 else None
    rows = set(_sample_rows(cfg.T, n_sample).tolist()) | H.segment_ends(idx, cfg.N, keep_all) | set(fl.tolist())
    keep = None
    if keep_all is not None:
        # sample dropped copies too: the last tokens of the most loaded expert
        hot = int(np.argmax(counts))
        rows |= set(np.nonzero((idx == hot).any(axis=1))[0][-4:].tolist())
        assert keep_all.min() == 0
    rows = np.array(sorted(rows))
    if keep_all is not None:
        keep = keep_all[rows]
    ref = H.oracle_layer_rows(cfg, ins, rows, keep=keep)
    ref_out, n_re = H.reference_outputs(cfg, ins, rows, ref["out"], idx, rep, keep_all)
    e = H.assert_output_close(out.float().cpu().numpy()[rows], ref_out, name)
    print(f"{name}: near ties {rep['near_ties']} (routed differently, checked under the GPU's routing: "
          f"{rep['near_tie_flips']}), rows compared {rows.size}, errors {e}, "
          f"touched experts {int((counts > 0).sum())}")


# --------------------------------------------------------------------------- expert choice
EC_CASES = {
    "ec_softmax": inputs.MoEConfig("ec_softmax", T=300, d=264, N=8, K=2, F=392, routing="expert"),
    "ec_sigmoid_f32_half": inputs.MoEConfig("ec_sigmoid_f32_half", T=200, d=128, N=16, K=3, F=136,
                                            score="sigmoid", hidden_dtype="f32", capacity_factor=0.5,
                                            routing="expert"),
    "ec_small_T6": inputs.MoEConfig("ec_small_T6", T=6, d=256, N=64, K=2, F=64, routing="expert"),
    "ec_every_token": inputs.MoEConfig("ec_every_token", T=77, d=64, N=4, K=4, F=64, routing="expert"),
    "ec_shared_pairs": inputs.MoEConfig("ec_shared_pairs", T=600, d=192, N=2, K=1, F=136, S=1, Fs=72,
                                        routing="expert"),
}


def _ec_select_gpu(cfg, dev):
    C = B.expert_choice_capacity(cfg)
    row_token = torch.empty(cfg.N, C, dtype=torch.int32, device="cuda")
    row_w = torch.empty(cfg.N, C, dtype=torch.float32, device="cuda")
    offsets = torch.empty(cfg.N + 1, dtype=torch.int32, device="cuda")
    B.expert_choice_select(B.problem(cfg), dev["hidden"], dev["w_router"], row_token, row_w, offsets,
                           router_bias=dev.get("router_bias"))
    torch.cuda.synchronize()
    return C, row_token.cpu().numpy(), row_w.cpu().numpy(), offsets.cpu().numpy()


@pytest.mark.parametrize("name", list(EC_CASES))
def test_expert_choice_matches_oracle(name):
    cfg = EC_CASES[name]
    ins, dev = H.make_case(cfg)
    C, row_token, row_w, offsets = _ec_select_gpu(cfg, dev)
    H.compare_expert_choice(cfg, ins, C, row_token, row_w, offsets, name)
    # the layer under that (verified) selection
    out, _, _, counts = None, None, None, None
    layer = B.MoELayer(cfg, dev)
    counts = torch.empty(cfg.N, dtype=torch.int32, device="cuda")
    out = layer.forward(dev["hidden"], counts=counts)
    torch.cuda.synchronize()
    assert layer.status(cfg.T) == 0
    assert torch.all(counts == C)
    idx, w = oracle.routing_from_expert_choice(row_token, row_w.astype(np.float64), cfg.T)
    bits = {k: [H.bf16_bits(m) for m in ins[k]] for k in ("w_gate", "w_up", "w_down")}
    sh = {}
    if cfg.S:
        sh = {k: [H.bf16_bits(m) for m in ins[k]] for k in ("ws_gate", "ws_up", "ws_down")}
    ref = oracle.layer_routed(H.hidden_f32(ins), idx, w, bits["w_gate"], bits["w_up"], bits["w_down"], **sh)
    H.assert_output_close(out.float().cpu().numpy(), ref, name)


def test_expert_choice_full_size_mixtral():
    """The Mixtral-shaped layer with expert-choice routing (C = 1024 tokens per
    expert): selection bit-exact, outputs on sampled tokens."""
    cfg = inputs.MIXTRAL_EC
    ins = inputs.make_inputs(cfg, seed=0, device="cuda")
    dev = {k: (None if v is None else v.cuda().contiguous()) for k, v in ins.items()}
    C, row_token, row_w, offsets = _ec_select_gpu(cfg, dev)
    H.compare_expert_choice(cfg, ins, C, row_token, row_w, offsets, "mixtral_ec")
    layer = B.MoELayer(cfg, dev)
    out = layer.forward(dev["hidden"])
    torch.cuda.synchronize()
    assert layer.status(cfg.T) == 0
    idx, w = oracle.routing_from_expert_choice(row_token, row_w.astype(np.float64), cfg.T)
    rows = _sample_rows(cfg.T, 12)
    picked_by = (idx >= 0).sum(axis=1)
    rows = np.array(sorted(set(rows.tolist()) | {int(np.argmax(picked_by)), int(np.argmin(picked_by))}))
    bits = {k: [H.bf16_bits(m) for m in ins[k]] for k in ("w_gate", "w_up", "w_down")}
    ref = oracle.layer_routed(H.hidden_f32(ins)[rows], idx[rows], w[rows], bits["w_gate"], bits["w_up"],
                              bits["w_down"])
    H.assert_output_close(out.float().cpu().numpy()[rows], ref, "mixtral_ec")
