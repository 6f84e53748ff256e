"""GPU parity of the MXFP4 expert path against the oracle's MXFP4 layer.

The expert matrices are E2M1 codes (two per byte) with one E8M0 scale per
32 elements of a row; the oracle decodes them exactly in fp64. The GPU
rewrites each block as E4M3 codes relative to its row's reference exponent
(exact for the synthetic weights, whose block exponents span a few binades)
and runs the 8-bit tensor-core GEMMs on two-term E4M3 activations. The
acceptance bar is the layer's: router bit-exact (near ties reported apart),
outputs max|gpu - ref| <= 2e-2 max|ref| and mean relative L1 <= 5e-3.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_94_b300 import inputs
from oracle import oracle
from tests import helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from mixture_experts_layer_94_b300 import binding as B


def _cfg(name, **kw):
    return inputs.MoEConfig(name, expert_dtype="mxfp4", **kw)


MID = {
    "mx_tiny_f32": _cfg("mx_tiny_f32", T=64, d=128, N=8, K=2, F=256, hidden_dtype="f32"),
    "mx_shared_sigmoid": _cfg("mx_shared_sigmoid", T=333, d=256, N=64, K=6, F=224, S=1, Fs=160,
                              score="sigmoid", sel_bias_var=0.1, zipf=1.1),
    "mx_ragged": _cfg("mx_ragged", T=300, d=288, N=16, K=4, F=416),
    "mx_multi_tile": _cfg("mx_multi_tile", T=700, d=416, N=4, K=2, F=160),
    "mx_decode_T3": _cfg("mx_decode_T3", T=3, d=1024, N=128, K=8, F=64),
    "mx_gptoss_like": _cfg("mx_gptoss_like", T=200, d=320, N=32, K=4, F=320),
    "mx_capacity": _cfg("mx_capacity", T=300, d=288, N=16, K=4, F=416, capacity_factor=0.8),
    # a small batch with few GEMM tiles and a shared expert
    "mx_small_shared": _cfg("mx_small_shared", T=2, d=2048, N=64, K=4, F=288, S=1, Fs=256),
    # a small batch with a capacity limit (two tokens on three experts always
    # share one), a shared expert, fp32 hidden
    "mx_small_capacity_shared_f32": _cfg("mx_small_capacity_shared_f32", T=2, d=96, N=3, K=2, F=160, S=1, Fs=64,
                                         hidden_dtype="f32", capacity_factor=0.5),
    # T*K >= 8192 copies: the token-major split, with a shared expert
    "mx_token_major_shared": _cfg("mx_token_major_shared", T=1100, d=288, N=8, K=8, F=160, S=1, Fs=128),
}


def _run_layer(cfg, dev):
    layer = B.MoELayer(cfg, dev)
    idx = torch.empty(cfg.T, cfg.K, dtype=torch.int32, device="cuda")
    w = torch.empty(cfg.T, cfg.K, dtype=torch.float32, device="cuda")
    counts = torch.empty(cfg.N, dtype=torch.int32, device="cuda")
    out = layer.forward(dev["hidden"], topk_idx=idx, topk_w=w, counts=counts)
    torch.cuda.synchronize()
    assert layer.status(cfg.T) == 0
    return out, idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("name", list(MID))
def test_mxfp4_layer_matches_oracle(name):
    cfg = MID[name]
    ins, dev = H.make_case(cfg)
    out, idx, w, counts = _run_layer(cfg, dev)
    keep_cap = H.capacity_keep(cfg, idx) if cfg.capacity_factor > 0 else None
    ref = H.oracle_layer_rows(cfg, ins, np.arange(cfg.T), keep=keep_cap)
    rep = H.compare_router(idx, w, H.oracle_router(cfg, ins), cfg)
    assert np.array_equal(counts, np.bincount(idx.reshape(-1), minlength=cfg.N))
    ref_out, _ = H.reference_outputs(cfg, ins, np.arange(cfg.T), ref["out"], idx, rep, keep_cap)
    e = H.assert_output_close(out.float().cpu().numpy(), ref_out, name)
    print(f"{name}: {e}; near ties {rep['near_ties']}, routed differently (checked) {rep['near_tie_flips']}")


SWIGLU_CASES = [(128, 256, 8, 2, 64), (288, 416, 5, 2, 300), (256, 512, 16, 4, 700)]


@pytest.mark.parametrize("d,F,N,K,T", SWIGLU_CASES)
def test_grouped_swiglu_mxfp4_matches_oracle(d, F, N, K, T):
    cfg = _cfg("gs4", T=T, d=d, N=N, K=K, F=F)
    ins = inputs.make_inputs(cfg, seed=6)
    rng = np.random.default_rng(d + F + 1)
    p_e = np.linspace(3.0, 0.0, N) ** 2 + 1e-9
    p_e[-1] = 0.0
    p_e /= p_e.sum()
    K_eff = min(K, int((p_e > 0).sum()))
    cfg = cfg.with_(K=K_eff)
    idx = np.stack([rng.choice(N, size=K_eff, replace=False, p=p_e) for _ in range(T)]).astype(np.int32)
    perm = oracle.permute(idx, N)
    x_perm = ins["hidden"][torch.from_numpy(perm["perm_src"] // K_eff).long()].to(torch.float16).contiguous()
    p = B.problem(cfg)
    ws = B.new_workspace(p, B.CALL_GROUPED_SWIGLU)
    h = torch.empty(T * K_eff, F, dtype=torch.float16, device="cuda")
    y = torch.empty(T * K_eff, d, dtype=torch.bfloat16, device="cuda")
    d_ = lambda k: ins[k].cuda().contiguous()  # noqa: E731
    B.grouped_swiglu_mxfp4(p, x_perm.cuda(), torch.from_numpy(perm["offsets"]).cuda(), d_("w_gate"),
                           d_("w_gate_scale"), d_("w_up"), d_("w_up_scale"), d_("w_down"), d_("w_down_scale"), h,
                           y, ws)
    torch.cuda.synchronize()
    assert B.get_device_status(ws) == 0
    hg, yg = h.float().cpu().numpy(), y.float().cpu().numpy()
    href = np.empty((T * K_eff, F))
    yref = np.empty((T * K_eff, d))
    xp = x_perm.float().numpy().astype(np.float64)
    for e in range(N):
        q = [H.u8(ins[k][e]) for k in ("w_gate", "w_up", "w_down")]
        s = [H.u8(ins[k][e]) for k in ("w_gate_scale", "w_up_scale", "w_down_scale")]
        for r in range(perm["offsets"][e], perm["offsets"][e + 1]):
            href[r], yref[r] = oracle.expert_ffn_mxfp4(xp[r], q[0], s[0], q[1], s[1], q[2], s[2], return_h=True)
    H.assert_output_close(hg, href, "h_perm")
    H.assert_output_close(yg, yref, "y_perm")


def test_mxfp4_wide_exponent_span_rounds_small_blocks_only():
    """A row whose block exponents span more than 14 binades: the blocks far
    below the row's largest round to the E4M3 grid (no longer exact), which
    moves the outputs by far less than the tolerance."""
    cfg = _cfg("mx_span", T=64, d=128, N=4, K=2, F=64)
    ins = inputs.make_inputs(cfg, seed=7)
    for k in ("w_gate_scale", "w_up_scale", "w_down_scale"):
        ins[k][:, :, 0] = (ins[k][:, :, 0].int() - 20).clamp_min(1).to(torch.uint8)  # first block 2^-20 smaller
    dev = {k: (None if v is None else v.cuda().contiguous()) for k, v in ins.items()}
    out, idx, w, _ = _run_layer(cfg, dev)
    ref = H.oracle_layer_rows(cfg, ins, np.arange(cfg.T))
    rep = H.compare_router(idx, w, H.oracle_router(cfg, ins), cfg)
    ref_out, _ = H.reference_outputs(cfg, ins, np.arange(cfg.T), ref["out"], idx, rep)
    H.assert_output_close(out.float().cpu().numpy(), ref_out, "wide span")


def _sample_rows(T, n, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, T - 1} | set(rng.choice(T, size=min(T, n), replace=False).tolist())
    return np.array(sorted(rows))


FULL = [("gptoss_mxfp4", inputs.GPTOSS_MXFP4, 64)] + [
    (f"qwen_decode_mxfp4_T{T}", inputs.QWEN_DECODE_MXFP4.with_(T=T), 64) for T in (1, 32, 512)]


@pytest.mark.parametrize("name,cfg,n_sample", FULL, ids=[f[0] for f in FULL])
def test_mxfp4_full_size_workload(name, cfg, n_sample):
    ins = inputs.make_inputs(cfg, seed=0, device="cuda")
    dev = {k: (None if v is None else v.cuda().contiguous()) for k, v in ins.items()}
    out, idx, w, counts = _run_layer(cfg, dev)
    # the per-call preparation (only the experts in use) gives the same result
    per_call = B.MoELayer(cfg, dev, mx_prepare=False).forward(dev["hidden"])
    torch.cuda.synchronize()
    H.assert_same_but_summation_order(out, per_call, name)
    rep = H.compare_router(idx, w, H.oracle_router(cfg, ins), cfg)
    assert np.array_equal(counts, np.bincount(idx.reshape(-1), minlength=cfg.N))
    rows = np.array(sorted(set(_sample_rows(cfg.T, n_sample).tolist()) | H.segment_ends(idx, cfg.N) |
                           set(rep["flipped_tokens"].tolist())))
    ref = H.oracle_layer_rows(cfg, ins, rows)
    ref_out, _ = H.reference_outputs(cfg, ins, rows, ref["out"], idx, rep)
    e = H.assert_output_close(out.float().cpu().numpy()[rows], ref_out, name)
    print(f"{name}: errors {e}; rows compared {rows.size}; near ties {rep['near_ties']}, "
          f"routed differently (checked) {rep['near_tie_flips']}")


def _prep_reference(bscale, nblk):
    """The preparation of one weight matrix from its E8M0 block scales [rows][nblk]
    (uint8), as the header defines it: E_R = clamp(max of the row's non-NaN
    exponents - 6, 1, 254), the fp32 scale 2^(E_R - 127), and index
    clamp(E_b - E_R, -15, 6) + 15 per block, four per word (block 4kb + c in
    byte c, 0 past the row's end), K-step-major [kb][rows]."""
    rows = bscale.shape[0]
    e = bscale.astype(np.int64)
    m = np.where(e == 255, 0, e).max(axis=1)
    e_row = np.clip(m - 6, 1, 254)
    rs = np.ldexp(1.0, e_row - 127).astype(np.float32)
    kb = -(-nblk // 4)
    idx = np.zeros((rows, 4 * kb), np.int64)
    idx[:, :nblk] = np.clip(e - e_row[:, None], -15, 6) + 15
    words = (idx.reshape(rows, kb, 4) << (8 * np.arange(4))).sum(axis=2).astype(np.uint32)
    return rs, words.T.copy()


def _prep_arrays(buf, cfg):
    """Splits a prepared buffer into its arrays (header order, 256-byte aligned)."""
    N, S, d, F, Fs = cfg.N, cfg.S, cfg.d, cfg.F, cfg.Fs
    kb = lambda k: -(-k // 128)  # noqa: E731
    shapes = [("rs", N * F), ("rs", N * F), ("rs", N * d), ("ki", (kb(d), N * F)), ("ki", (kb(d), N * F)),
              ("ki", (kb(F), N * d))]
    if S:
        shapes += [("rs", S * Fs), ("rs", S * Fs), ("rs", S * d), ("ki", (kb(d), S * Fs)),
                   ("ki", (kb(d), S * Fs)), ("ki", (kb(Fs), S * d))]
    out, off = [], 0
    for kind, shp in shapes:
        n = int(np.prod(shp))
        a = buf[off:off + 4 * n].view(np.float32 if kind == "rs" else np.uint32).reshape(shp)
        out.append(a)
        off = (off + 4 * n + 255) // 256 * 256
    return out


@pytest.mark.parametrize("d,F,Fs", [(288, 160, 96), (256, 128, 512)])
def test_mxfp4_prepare_matches_its_definition(d, F, Fs):
    # block scales with NaN blocks, blocks far below the row's largest (the
    # index clamps at -15) and a row of all-zero exponents (E_R clamps at 1);
    # rows of 9, 5, 3 blocks (byte-wise staging) and of 8, 4, 16 (word-wise)
    cfg = _cfg("prep", T=4, d=d, N=4, K=2, F=F, S=1, Fs=Fs)
    ins = inputs.make_inputs(cfg, seed=3)
    rng = np.random.default_rng(11)
    for k in ("w_gate_scale", "w_up_scale", "w_down_scale", "ws_gate_scale", "ws_up_scale", "ws_down_scale"):
        s = rng.integers(100, 140, size=tuple(ins[k].shape)).astype(np.uint8)
        flat = s.reshape(-1, s.shape[-1])
        flat[1, 0] = 255
        flat[2, :] = 255
        flat[2, 1] = 120
        flat[3, -1] = 2
        flat[4, :] = 0
        ins[k] = torch.from_numpy(s)
    dev = {k: (None if v is None else v.cuda().contiguous()) for k, v in ins.items()}
    layer = B.MoELayer(cfg, dev)
    torch.cuda.synchronize()
    got = _prep_arrays(layer.mx_prep.cpu().numpy(), cfg)
    mats = [("w_gate_scale", cfg.d), ("w_up_scale", cfg.d), ("w_down_scale", cfg.F),
            ("ws_gate_scale", cfg.d), ("ws_up_scale", cfg.d), ("ws_down_scale", cfg.Fs)]
    refs = [_prep_reference(ins[k].numpy().reshape(-1, K // 32), K // 32) for k, K in mats]
    for i, (rs, ki) in enumerate(refs):
        j = i if i < 3 else i + 3
        assert np.array_equal(got[j], rs), mats[i][0]
        assert np.array_equal(got[j + 3], ki), mats[i][0]


@pytest.mark.parametrize("name", ["mx_shared_sigmoid", "mx_decode_T3", "mx_ragged", "mx_capacity"])
def test_mxfp4_prepared_and_per_call_agree(name):
    cfg = MID[name]
    ins, dev = H.make_case(cfg)
    prepared = B.MoELayer(cfg, dev)
    per_call = B.MoELayer(cfg, dev, mx_prepare=False)
    assert prepared.mx_prep is not None and per_call.mx_prep is None
    a = prepared.forward(dev["hidden"])
    b = per_call.forward(dev["hidden"])
    torch.cuda.synchronize()
    assert prepared.status(cfg.T) == 0 and per_call.status(cfg.T) == 0
    H.assert_same_but_summation_order(a, b, name)
