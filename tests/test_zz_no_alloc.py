"""moe_permute_static: route and pack for callers that cannot allocate device
memory (its scratch is a fixed array inside the library instead of a caller
workspace). Called through the C ABI and checked, bit for bit, against
moe_permute with a workspace, on two calls in a row: the second call runs on
the scratch the first one left behind.

This file is collected last so that a stop-at-first-failure run has run every
other test before it; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_94_b300 import inputs

pytestmark = pytest.mark.gpu

MAX_CHUNK_COUNTS = 65536  # MOE_PERMUTE_STATIC_MAX_CHUNK_COUNTS in include/moe.h


def _binding():
    from mixture_experts_layer_94_b300 import binding as B

    fn = B.lib.moe_permute_static
    fn.argtypes = [ctypes.POINTER(B.Problem)] + [ctypes.c_void_p] * 8
    fn.restype = ctypes.c_int32
    return B


def _case(T, N, K, d, seed, expert_dtype="bf16"):
    rng = np.random.default_rng(seed)
    p_e = 1.0 / np.arange(1, N + 1) ** 1.2
    p_e /= p_e.sum()
    idx = np.stack([rng.choice(N, size=K, replace=False, p=p_e) for _ in range(T)]).astype(np.int32)
    cfg = inputs.MoEConfig("noalloc", T=T, d=d, N=N, K=K, F=16, expert_dtype=expert_dtype)
    hidden = inputs.make_router_inputs(cfg, seed=seed)["hidden"].cuda()
    return cfg, torch.from_numpy(idx).cuda(), hidden


def _outputs(cfg):
    T, N, K, d = cfg.T, cfg.N, cfg.K, cfg.d
    e = lambda *s, dt=torch.int32: torch.full(s, -7, dtype=dt, device="cuda")  # noqa: E731
    return dict(counts=e(N), offsets=e(N + 1), perm_src=e(T * K), inv_row=e(T * K),
                x_perm=torch.zeros(T * K, d, dtype=torch.bfloat16, device="cuda"))


def _run_static(B, cfg, idx, hidden):
    o = _outputs(cfg)
    p = B.problem(cfg)
    st = B.lib.moe_permute_static(ctypes.byref(p), idx.data_ptr(), hidden.data_ptr(),
                                  o["counts"].data_ptr(), o["offsets"].data_ptr(),
                                  o["perm_src"].data_ptr(), o["inv_row"].data_ptr(),
                                  o["x_perm"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, B.status_string(st)
    return o


def _run_workspace(B, cfg, idx, hidden):
    o = _outputs(cfg)
    p = B.problem(cfg)
    ws = B.new_workspace(p, B.CALL_PERMUTE)
    B.permute(p, idx, hidden, o["counts"], o["offsets"], o["perm_src"], o["inv_row"], o["x_perm"], ws)
    torch.cuda.synchronize()
    assert B.get_device_status(ws) == 0
    return o


def test_static_scratch_permute_matches_workspace_permute_on_two_calls():
    B = _binding()
    # First a problem that fills the whole array (256 experts x 256 chunks),
    # then a smaller one that finds the first call's counts still there.
    # The third call is an FP8-expert problem: its packed rows are fp16.
    for T, N, K, d, seed, dt in ((8192, 256, 8, 64, 11, "bf16"), (300, 64, 6, 136, 12, "bf16"),
                                 (200, 16, 4, 144, 14, "fp8")):
        cfg, idx, hidden = _case(T, N, K, d, seed, dt)
        got = _run_static(B, cfg, idx, hidden)
        torch.cuda.synchronize()
        ref = _run_workspace(B, cfg, idx, hidden)
        for k in ("counts", "offsets", "perm_src", "inv_row"):
            assert torch.equal(got[k], ref[k]), k
        assert torch.equal(got["x_perm"].view(torch.int16), ref["x_perm"].view(torch.int16))
        assert int(got["offsets"][-1]) == T * K


def test_static_scratch_rejects_problems_beyond_its_limit():
    B = _binding()
    cfg, idx, hidden = _case(64, 8, 2, 8, 13)
    big = B.problem(cfg, T=32 * (MAX_CHUNK_COUNTS // 8) + 1)  # 8 * chunks = limit + 8
    o = _outputs(cfg)
    st = B.lib.moe_permute_static(ctypes.byref(big), idx.data_ptr(), hidden.data_ptr(),
                                  o["counts"].data_ptr(), o["offsets"].data_ptr(),
                                  o["perm_src"].data_ptr(), o["inv_row"].data_ptr(),
                                  o["x_perm"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == -2  # MOE_ERR_UNSUPPORTED, nothing enqueued
    torch.cuda.synchronize()
    assert torch.all(o["counts"] == -7)
