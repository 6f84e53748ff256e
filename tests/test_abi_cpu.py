"""The C-ABI library on the CPU: it loads, exports every symbol include/moe.h
declares, and its host-only functions (status strings, problem validation,
workspace sizing) behave as documented. No CUDA call is made here."""
import ctypes
import subprocess

import pytest

from mixture_experts_layer_94_b300 import binding as B
from mixture_experts_layer_94_b300 import inputs


def test_header_declares_the_abi():
    names = B.header_functions()
    for n in ("moe_router_topk", "moe_permute", "moe_grouped_swiglu", "moe_combine",
              "moe_layer_forward", "moe_workspace_bytes", "moe_get_device_status",
              "moe_status_string", "moe_problem_check"):
        assert n in names


def test_library_exports_every_header_symbol():
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in B.header_functions():
        assert hasattr(lib, n), n
    syms = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                          text=True, check=True).stdout
    exported = {line.split()[-1] for line in syms.splitlines() if " T " in line}
    assert set(B.header_functions()) <= exported


def test_status_strings():
    for s, key in ((0, "MOE_OK"), (-1, "INVALID_ARG"), (-2, "UNSUPPORTED"), (-3, "WORKSPACE"),
                   (-4, "CUDA"), (-5, "TIMEOUT"), (-6, "DEVICE_BOUNDS"), (-7, "RANGE"), (7, "UNKNOWN")):
        assert key in B.status_string(s)


@pytest.mark.parametrize("cfg", list(inputs.CONFIGS.values()), ids=list(inputs.CONFIGS))
def test_workload_problems_are_valid(cfg):
    p = B.problem(cfg)
    assert B.problem_check(p) == 0
    for call in (B.CALL_PERMUTE, B.CALL_GROUPED_SWIGLU, B.CALL_LAYER_FORWARD, B.CALL_ROUTER):
        n = B.workspace_bytes(p, call)
        assert n > 0 and n % 256 == 0
    assert B.workspace_bytes(p, B.CALL_LAYER_FORWARD) > B.workspace_bytes(p, B.CALL_PERMUTE)


@pytest.mark.parametrize("field,value,status", [
    ("T", -1, -1), ("d_model", 0, -1), ("d_model", 12, -1), ("n_experts", 0, -1),
    ("top_k", 0, -1), ("top_k", 9, -1), ("ffn", 100, -1), ("n_shared", -1, -1),
    ("score_fn", 2, -1), ("renormalize", 3, -1), ("hidden_dtype", 5, -1),
    ("n_experts", 257, -2), ("n_shared", 9, -2),
])
def test_problem_check_rejects(field, value, status):
    cfg = inputs.TINY.with_(Fs=64)
    p = B.problem(cfg, **{field: value})
    assert B.problem_check(p) == status
    assert B.workspace_bytes(p, B.CALL_LAYER_FORWARD) == 0


def test_problem_check_shared_width_and_topk_cap():
    p = B.problem(inputs.TINY, n_shared=1, shared_ffn=0)
    assert B.problem_check(p) == -1
    p = B.problem(inputs.TINY, n_experts=64, top_k=33)
    assert B.problem_check(p) == -2
    assert B.lib.moe_problem_check(None) == -1


def test_workspace_grows_with_tokens():
    a = B.workspace_bytes(B.problem(inputs.MIXTRAL, T=1), B.CALL_LAYER_FORWARD)
    b = B.workspace_bytes(B.problem(inputs.MIXTRAL, T=4096), B.CALL_LAYER_FORWARD)
    assert b > a
    # the fused layer needs x_perm, h and the fp32 accumulator at least
    m = inputs.MIXTRAL
    assert b >= m.T * m.K * (m.d + m.F) * 2 + m.T * m.d * 4


def test_layer_kernel_count():
    assert B.layer_forward_kernel_count(B.problem(inputs.MIXTRAL)) == 10
    assert B.layer_forward_kernel_count(B.problem(inputs.MIXTRAL, T=1024)) == 8
    assert B.layer_forward_kernel_count(B.problem(inputs.TINY)) == 7
    assert B.layer_forward_kernel_count(B.problem(inputs.MIXTRAL, T=0)) == 1
    assert B.layer_forward_kernel_count(B.problem(inputs.MIXTRAL, top_k=0)) == 0


def test_decode_sized_batches_run_as_one_kernel():
    # token choice with T <= 4 and bf16 or FP8 experts runs the whole layer as
    # one kernel; larger batches, MXFP4 experts and expert choice keep the
    # router, route-and-pack and grouped GEMM kernels
    q = inputs.QWEN_DECODE
    for T, want in ((1, True), (2, True), (4, True), (5, False), (8, False), (0, False)):
        assert B.layer_small_batch(B.problem(q, T=T)) == want, T
    for T, want in ((1, True), (4, True), (5, False)):
        assert B.layer_small_batch(B.problem(inputs.QWEN_DECODE_FP8, T=T)) == want, T
    assert not B.layer_small_batch(B.problem(inputs.QWEN_DECODE_MXFP4, T=1))
    assert not B.layer_small_batch(B.problem(inputs.MIXTRAL_EC, T=2))
    # the staged token rows and h rows must fit the kernel's shared memory
    assert B.layer_small_batch(B.problem(q, T=1, d_model=16384))
    assert not B.layer_small_batch(B.problem(q, T=4, d_model=16384, top_k=32, ffn=4096))
    with pytest.raises(ValueError):
        B.layer_small_batch(B.problem(q, top_k=0))
    for cfg in (q, inputs.QWEN_DECODE_FP8, q.with_(S=1, Fs=512, hidden_dtype="f32")):
        assert B.layer_forward_kernel_count(B.problem(cfg, T=1)) == 1, cfg.name
    # the GEMM path: router, routing, gather + activation split, gate/up, split of h, down, finalise
    assert B.layer_forward_kernel_count(B.problem(inputs.QWEN_DECODE_FP8, T=5)) == 8
    assert B.layer_forward_kernel_count(B.problem(inputs.QWEN_DECODE_MXFP4, T=1)) == 11


def test_one_kernel_decision_agrees_with_the_launch_count():
    # over random valid problems: the one-kernel path is token choice, T <= 4,
    # bf16 or FP8 experts, and launches exactly one kernel
    import numpy as np

    rng = np.random.default_rng(0)
    seen = set()
    for _ in range(300):
        fmt = ["bf16", "fp8", "mxfp4"][rng.integers(3)]
        N = int(rng.integers(1, 257))
        K = int(rng.integers(1, min(N, 32) + 1))
        unit = 32 if fmt == "mxfp4" else 16 if fmt == "fp8" else 8
        S = int(rng.integers(0, 3))
        cfg = inputs.MoEConfig("rand", T=int(rng.integers(0, 9)), d=unit * int(rng.integers(1, 200)), N=N, K=K,
                               F=unit * int(rng.integers(1, 100)), S=S, Fs=unit * int(rng.integers(1, 50)) if S else 0,
                               hidden_dtype=["bf16", "f32"][rng.integers(2)], expert_dtype=fmt,
                               routing="expert" if rng.random() < 0.2 else "token")
        p = B.problem(cfg)
        if B.problem_check(p) != B.MOE_OK:
            continue
        one = B.layer_small_batch(p)
        seen.add(one)
        if one:
            assert cfg.routing == "token" and 1 <= cfg.T <= 4 and fmt != "mxfp4"
            assert B.layer_forward_kernel_count(p) == 1
        else:
            assert cfg.T == 0 or B.layer_forward_kernel_count(p) > 1
    assert seen == {True, False}


def _fake_prepared():
    w = B.Weights()
    w.mx_prep = 256  # only its nullness is read by the host-side count
    return w


def test_kernel_count_without_per_call_mxfp4_preparation():
    # a prepared buffer removes the preparation of gate, up and down (and of
    # the shared experts' three matrices)
    for cfg, n in ((inputs.GPTOSS_MXFP4, 3), (inputs.GPTOSS_MXFP4.with_(S=1, Fs=256), 6)):
        p = B.problem(cfg)
        assert B.layer_forward_kernel_count(p) - B.layer_forward_kernel_count(p, _fake_prepared()) == n
    p = B.problem(inputs.MIXTRAL_FP8)
    assert B.layer_forward_kernel_count(p) == B.layer_forward_kernel_count(p, _fake_prepared())


def test_mxfp4_prep_bytes_covers_every_array():
    for cfg in (inputs.GPTOSS_MXFP4, inputs.QWEN_DECODE_MXFP4, inputs.GPTOSS_MXFP4.with_(S=2, Fs=320)):
        N, S, d, F, Fs = cfg.N, cfg.S, cfg.d, cfg.F, cfg.Fs
        kb = lambda k: -(-k // 128)  # noqa: E731  (K steps of 128 elements)
        arrays = [N * F * 4, N * F * 4, N * d * 4, N * F * kb(d) * 4, N * F * kb(d) * 4, N * d * kb(F) * 4]
        if S:
            arrays += [S * Fs * 4, S * Fs * 4, S * d * 4, S * Fs * kb(d) * 4, S * Fs * kb(d) * 4,
                       S * d * kb(Fs) * 4]
        got = B.mxfp4_prep_bytes(B.problem(cfg))
        assert sum(arrays) <= got < sum(arrays) + 256 * len(arrays)
        assert got == B.mxfp4_prep_bytes(B.problem(cfg, T=1))  # weights only, not the batch
    assert B.mxfp4_prep_bytes(B.problem(inputs.MIXTRAL_FP8)) == 0
    assert B.mxfp4_prep_bytes(B.problem(inputs.MIXTRAL)) == 0


def test_mxfp4_prepare_validates_before_any_cuda_call():
    w = B.Weights()
    w.w_gate_scale = w.w_up_scale = w.w_down_scale = 4096
    P = B.lib.moe_mxfp4_prepare
    p = B.problem(inputs.GPTOSS_MXFP4)
    need = B.mxfp4_prep_bytes(p)
    assert P(ctypes.byref(B.problem(inputs.MIXTRAL_FP8)), ctypes.byref(w), 256, need, None) == B.MOE_ERR_INVALID_ARG
    assert P(ctypes.byref(p), None, 256, need, None) == B.MOE_ERR_INVALID_ARG
    assert P(ctypes.byref(p), ctypes.byref(w), None, need, None) == B.MOE_ERR_INVALID_ARG
    assert P(ctypes.byref(p), ctypes.byref(w), 256 + 16, need, None) == B.MOE_ERR_WORKSPACE
    assert P(ctypes.byref(p), ctypes.byref(w), 256, need - 1, None) == B.MOE_ERR_WORKSPACE
    w.w_up_scale = None
    assert P(ctypes.byref(p), ctypes.byref(w), 256, need, None) == B.MOE_ERR_INVALID_ARG
    ps = B.problem(inputs.GPTOSS_MXFP4.with_(S=1, Fs=256))  # shared experts need their scales too
    w.w_up_scale = 4096
    assert P(ctypes.byref(ps), ctypes.byref(w), 256, B.mxfp4_prep_bytes(ps), None) == B.MOE_ERR_INVALID_ARG


def test_mxfp4_rejects_rows_wider_than_the_preparation_stages():
    assert B.problem_check(B.problem(inputs.GPTOSS_MXFP4.with_(d=32768))) == 0
    assert B.problem_check(B.problem(inputs.GPTOSS_MXFP4.with_(d=32800))) == B.MOE_ERR_UNSUPPORTED
    assert B.problem_check(B.problem(inputs.GPTOSS_MXFP4.with_(F=32800))) == B.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("cfg", list(inputs.CONFIGS.values()), ids=list(inputs.CONFIGS))
def test_workspace_sizing_for_empty_and_single_token_batches(cfg):
    for T in (0, 1, 3):
        p = B.problem(cfg, T=T)
        assert B.problem_check(p) == 0
        for call in (B.CALL_PERMUTE, B.CALL_GROUPED_SWIGLU, B.CALL_LAYER_FORWARD, B.CALL_ROUTER):
            assert B.workspace_bytes(p, call) >= 256


@pytest.mark.parametrize("kw,status", [
    (dict(n_groups=3), -1),                      # 8 experts do not split into 3 groups
    (dict(n_groups=4, topk_groups=0), -1),
    (dict(n_groups=4, topk_groups=5), -1),
    (dict(n_groups=4, topk_groups=1, top_k=3), -1),  # K > experts in the kept groups
    (dict(n_groups=4, topk_groups=1), 0),
    (dict(n_groups=-1), -1),
])
def test_problem_check_group_limited_routing(kw, status):
    assert B.problem_check(B.problem(inputs.TINY, **kw)) == status


def test_problem_check_capacity_factor():
    assert B.problem_check(B.problem(inputs.TINY, capacity_factor=0.6)) == 0
    assert B.problem_check(B.problem(inputs.TINY, capacity_factor=-1.0)) == -1
    assert B.problem_check(B.problem(inputs.TINY, capacity_factor=float("nan"))) == -1


def test_problem_check_fp8_experts():
    fp8 = inputs.TINY.with_(expert_dtype="fp8")
    assert B.problem_check(B.problem(fp8)) == 0
    assert B.problem_check(B.problem(fp8, expert_dtype=3)) == -1
    assert B.problem_check(B.problem(fp8, d_model=136)) == -1   # FP8 code rows: 16-byte multiples
    assert B.problem_check(B.problem(fp8, ffn=264)) == -1
    assert B.problem_check(B.problem(fp8, n_shared=1, shared_ffn=72)) == -1
    assert B.problem_check(B.problem(fp8, n_shared=1, shared_ffn=80)) == 0
    assert B.problem_check(B.problem(inputs.TINY, d_model=136)) == 0  # bf16 experts: multiples of 8


def test_fp8_workspace_holds_an_fp16_copy_for_shared_experts():
    base = inputs.TINY.with_(hidden_dtype="bf16", S=1, Fs=64)
    n16 = B.workspace_bytes(B.problem(base), B.CALL_LAYER_FORWARD)
    n8 = B.workspace_bytes(B.problem(base.with_(expert_dtype="fp8")), B.CALL_LAYER_FORWARD)
    assert n8 >= n16 + base.T * base.d * 2


def test_grouped_swiglu_entry_points_check_the_expert_format():
    """Host-side checks only: each grouped-SwiGLU entry point refuses the other
    format before touching the device."""
    p8 = B.problem(inputs.TINY.with_(expert_dtype="fp8"))
    assert B.lib.moe_grouped_swiglu(p8, *([None] * 8), 0, None) == -1
    p16 = B.problem(inputs.TINY)
    assert B.lib.moe_grouped_swiglu_fp8(p16, *([None] * 11), 0, None) == -1


def test_problem_check_mxfp4_experts():
    mx = inputs.TINY.with_(expert_dtype="mxfp4")
    assert B.problem_check(B.problem(mx)) == 0
    assert B.problem_check(B.problem(mx, d_model=144)) == -1     # 32-element scale blocks
    assert B.problem_check(B.problem(mx, ffn=272)) == -1
    assert B.problem_check(B.problem(mx, n_shared=1, shared_ffn=80)) == -1
    assert B.problem_check(B.problem(mx, n_shared=1, shared_ffn=96)) == 0
    p = B.problem(mx)
    assert B.lib.moe_grouped_swiglu_mxfp4(p, *([None] * 11), 0, None) == -1  # null pointers
    assert B.lib.moe_grouped_swiglu_fp8(p, *([None] * 11), 0, None) == -1   # the other format
    assert B.workspace_bytes(p, B.CALL_LAYER_FORWARD) > B.workspace_bytes(
        B.problem(inputs.TINY.with_(expert_dtype="fp8")), B.CALL_LAYER_FORWARD)  # + row reference scales


@pytest.mark.parametrize("T,K,N,c", [(4096, 2, 8, 0.0), (40, 2, 8, 0.6), (7, 4, 4, 0.0), (6, 2, 64, 0.0),
                                     (200, 3, 16, 0.5), (10, 8, 8, 3.0), (0, 2, 8, 0.0), (1, 1, 1, 0.0)])
def test_expert_choice_capacity_is_the_oracles(T, K, N, c):
    """The library's C (which sizes the binding's buffers) against the oracle's
    capacity formula, min(ceil(c T K / N), T) with c = 1 when unset."""
    from oracle import oracle

    cfg = inputs.MoEConfig("ec", T=T, d=64, N=N, K=K, F=64, capacity_factor=c, routing="expert")
    assert B.expert_choice_capacity(cfg) == oracle.expert_choice_capacity(c, T, K, N)
    assert B.lib.moe_expert_choice_capacity(ctypes.byref(B.problem(cfg, top_k=N + 1))) == -1
