"""moe_permute_static: route and pack for callers that cannot allocate device
memory (its scratch is a fixed array inside the library instead of a caller
workspace). Called through the C ABI and checked bit for bit against the
oracle's permutation and against moe_permute with a workspace, on calls in a
row: each later call runs on the scratch the previous one left behind.

This file is collected last so that a stop-at-first-failure run has run every
other test before it; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_94_b300 import inputs
from oracle import oracle

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
    cfg = inputs.MoEConfig("noalloc", T=T, d=d, N=N, K=K, F=32, expert_dtype=expert_dtype)
    hidden = inputs.make_router_inputs(cfg, seed=seed)["hidden"].cuda()
    return cfg, idx, hidden


def _outputs(cfg):
    T, N, K, d = cfg.T, cfg.N, cfg.K, cfg.d
    e = lambda *s, dt=torch.int32: torch.full(s, -7, dtype=dt, device="cuda")  # noqa: E731
    return dict(counts=e(N), offsets=e(N + 1), perm_src=e(T * K), inv_row=e(T * K),
                x_perm=torch.zeros(T * K, d, dtype=torch.int16, device="cuda"))


def _run_static(B, cfg, idx, hidden):
    o = _outputs(cfg)
    p = B.problem(cfg)
    idx_d = torch.from_numpy(idx).cuda()
    st = B.lib.moe_permute_static(ctypes.byref(p), idx_d.data_ptr(), hidden.data_ptr(),
                                  o["counts"].data_ptr(), o["offsets"].data_ptr(),
                                  o["perm_src"].data_ptr(), o["inv_row"].data_ptr(),
                                  o["x_perm"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, B.status_string(st)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in o.items()}


def _run_workspace(B, cfg, idx, hidden):
    o = _outputs(cfg)
    p = B.problem(cfg)
    ws = B.new_workspace(p, B.CALL_PERMUTE)
    B.permute(p, torch.from_numpy(idx).cuda(), hidden, o["counts"], o["offsets"], o["perm_src"],
              o["inv_row"], o["x_perm"], ws)
    torch.cuda.synchronize()
    st = B.get_device_status(ws)
    return {k: v.cpu() for k, v in o.items()}, st


def _packed_rows(cfg, hidden, src_tokens):
    """The rows moe_permute stores: bf16 for bf16 experts, fp16 for FP8 and
    MXFP4 experts (exact for these N(0,1) hidden values), as int16 bits."""
    act = torch.bfloat16 if cfg.expert_dtype == "bf16" else torch.float16
    return hidden.cpu().to(act)[torch.from_numpy(src_tokens).long()].view(torch.int16)


def _check_against_oracle(cfg, idx, hidden, got):
    ref = oracle.permute(idx, cfg.N)
    for k in ("counts", "offsets", "perm_src", "inv_row"):
        assert np.array_equal(got[k].numpy(), ref[k]), k
    expect = _packed_rows(cfg, hidden, ref["perm_src"] // cfg.K)
    assert torch.equal(got["x_perm"], expect)


def test_static_scratch_permute_matches_oracle_and_workspace_permute_on_calls_in_a_row():
    B = _binding()
    # First a problem that fills the whole array (256 experts x 256 chunks),
    # then smaller ones that find the previous call's counts still there.
    # The FP8- and MXFP4-expert problems pack fp16 rows.
    for T, N, K, d, seed, dt in ((8192, 256, 8, 64, 11, "bf16"), (300, 64, 6, 136, 12, "bf16"),
                                 (200, 16, 4, 144, 14, "fp8"), (333, 32, 4, 160, 15, "mxfp4"),
                                 (97, 8, 2, 64, 16, "mxfp4")):
        cfg, idx, hidden = _case(T, N, K, d, seed, dt)
        got = _run_static(B, cfg, idx, hidden)
        _check_against_oracle(cfg, idx, hidden, got)
        ref, st = _run_workspace(B, cfg, idx, hidden)
        assert st == 0
        for k in ("counts", "offsets", "perm_src", "inv_row", "x_perm"):
            assert torch.equal(got[k], ref[k]), (dt, k)
        assert int(got["offsets"][-1]) == T * K


def test_static_scratch_skips_an_out_of_range_index():
    """An expert index outside [0, N) is skipped: offsets[N] < T*K, its copy
    has inv_row -1, and every placed row is the oracle's. The oracle sees the
    bad copy as an extra expert N, which sorts after every real one, so its
    first offsets[N] rows are the placed rows."""
    B = _binding()
    for T, N, K, d, bad, val in ((500, 16, 4, 72, (123, 2), 16), (4100, 8, 2, 64, (1234, 0), -3)):
        cfg, idx, hidden = _case(T, N, K, d, T)
        idx[bad] = val
        got = _run_static(B, cfg, idx, hidden)
        placed = int(got["offsets"][-1])
        assert placed == T * K - 1
        flat = bad[0] * K + bad[1]
        assert int(got["inv_row"][flat]) == -1
        virt = idx.copy()
        virt[bad] = N
        ref = oracle.permute(virt, N + 1)
        assert np.array_equal(got["counts"].numpy(), ref["counts"][:N])
        assert np.array_equal(got["offsets"].numpy(), ref["offsets"][:N + 1])
        assert np.array_equal(got["perm_src"].numpy()[:placed], ref["perm_src"][:placed])
        inv = ref["inv_row"].copy()
        inv[flat] = -1
        assert np.array_equal(got["inv_row"].numpy(), inv)
        expect = _packed_rows(cfg, hidden, ref["perm_src"][:placed] // K)
        assert torch.equal(got["x_perm"][:placed], expect)
        # moe_permute on the same input agrees and reports the bad index
        ws_out, st = _run_workspace(B, cfg, idx, hidden)
        assert st == -6  # MOE_ERR_DEVICE_BOUNDS
        for k in ("counts", "offsets", "inv_row"):
            assert torch.equal(got[k], ws_out[k]), k
        assert torch.equal(got["x_perm"][:placed], ws_out["x_perm"][:placed])


def test_static_scratch_rejects_problems_beyond_its_limit():
    B = _binding()
    cfg, idx, hidden = _case(64, 8, 2, 8, 13)
    big = B.problem(cfg, T=32 * (MAX_CHUNK_COUNTS // 8) + 1)  # 8 * chunks = limit + 8
    o = _outputs(cfg)
    idx_d = torch.from_numpy(idx).cuda()
    st = B.lib.moe_permute_static(ctypes.byref(big), idx_d.data_ptr(), hidden.data_ptr(),
                                  o["counts"].data_ptr(), o["offsets"].data_ptr(),
                                  o["perm_src"].data_ptr(), o["inv_row"].data_ptr(),
                                  o["x_perm"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == -2  # MOE_ERR_UNSUPPORTED, nothing enqueued
    torch.cuda.synchronize()
    assert torch.all(o["counts"] == -7)
