"""Python view of the MoE layer ORACLE (oracle/moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the CUDA library or its binding. The
arithmetic lives in moe_oracle.c (plain C, fp64, fp32 router decision); this
module only marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/liboracle.so with gcc + OpenMP."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.moe_oracle_router.argtypes = [i64, i32, i32, i32, i32, i32, i32, i32] + [P] * 10
        lib.moe_oracle_router.restype = ctypes.c_int
        lib.moe_oracle_permute.argtypes = [i64, i32, i32, P, P, P, P, P]
        lib.moe_oracle_permute.restype = ctypes.c_int
        lib.moe_oracle_permute_cap.argtypes = [i64, i32, i32, i64, P, P, P, P, P]
        lib.moe_oracle_permute_cap.restype = ctypes.c_int
        lib.moe_oracle_capacity.argtypes = [ctypes.c_double, i64, i32, i32]
        lib.moe_oracle_capacity.restype = i64
        lib.moe_oracle_expert_ffn.argtypes = [i32, i32, P, P, P, P, P, P]
        lib.moe_oracle_expert_ffn.restype = None
        lib.moe_oracle_combine.argtypes = [i32, i32, P, P, P, P]
        lib.moe_oracle_combine.restype = None
        lib.moe_oracle_layer.argtypes = [i64] + [i32] * 10 + [P] * 15
        lib.moe_oracle_layer.restype = ctypes.c_int
        lib.moe_oracle_expert_choice.argtypes = [i64, i32, i32, i32, i64, P, P, P, P, P, P]
        lib.moe_oracle_expert_choice.restype = ctypes.c_int
        lib.moe_oracle_layer_routed.argtypes = [i64] + [i32] * 6 + [P] * 10
        lib.moe_oracle_layer_routed.restype = ctypes.c_int
        lib.moe_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.moe_oracle_e4m3_to_double.restype = ctypes.c_double
        lib.moe_oracle_expert_ffn_fp8.argtypes = [i32, i32] + [P] * 9
        lib.moe_oracle_expert_ffn_fp8.restype = None
        lib.moe_oracle_layer_fp8.argtypes = [i64] + [i32] * 10 + [P] * 21
        lib.moe_oracle_layer_fp8.restype = ctypes.c_int
        lib.moe_oracle_layer_routed_fp8.argtypes = [i64] + [i32] * 6 + [P] * 16
        lib.moe_oracle_layer_routed_fp8.restype = ctypes.c_int
        lib.moe_oracle_layer_routed_mxfp4.argtypes = [i64] + [i32] * 6 + [P] * 16
        lib.moe_oracle_layer_routed_mxfp4.restype = ctypes.c_int
        lib.moe_oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
        lib.moe_oracle_e2m1_to_double.restype = ctypes.c_double
        lib.moe_oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
        lib.moe_oracle_e8m0_to_double.restype = ctypes.c_double
        lib.moe_oracle_expert_ffn_mxfp4.argtypes = [i32, i32] + [P] * 9
        lib.moe_oracle_expert_ffn_mxfp4.restype = None
        lib.moe_oracle_layer_mxfp4.argtypes = [i64] + [i32] * 10 + [P] * 21
        lib.moe_oracle_layer_mxfp4.restype = ctypes.c_int
        lib.moe_oracle_silu.argtypes = [ctypes.c_double]
        lib.moe_oracle_silu.restype = ctypes.c_double
        lib.moe_oracle_num_threads.argtypes = []
        lib.moe_oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _bf16_bits(a):
    """Accept a uint16 array of bf16 bit patterns (or a torch bf16 tensor)."""
    if a is None:
        return None
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch

        return np.ascontiguousarray(a.contiguous().view(torch.int16).numpy().view(np.uint16))
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("expert weights must be bf16 bit patterns (uint16)")
    return a


SOFTMAX, SIGMOID = 0, 1


def num_threads() -> int:
    return int(_load().moe_oracle_num_threads())


def silu(z: float) -> float:
    return float(_load().moe_oracle_silu(float(z)))


def router(hidden, w_router, K, score_fn=SOFTMAX, renormalize=1, router_bias=None,
           sel_bias=None, n_groups=0, topk_groups=0):
    """Router over the rows of `hidden` (fp32 [T][d]). Returns a dict with
    logits (fp64 [T][N]), probs (fp64 [T][N]: full softmax or sigmoid scores),
    keys (fp32 [T][N]), idx (int32 [T][K]), w (fp64 [T][K]), margin (fp64 [T])."""
    lib = _load()
    x = _f32(hidden)
    W = _f32(w_router)
    T, d = x.shape
    d2, N = W.shape
    assert d == d2
    rb, sb = _f32(router_bias), _f32(sel_bias)
    logits = np.empty((T, N), np.float64)
    probs = np.empty((T, N), np.float64)
    keys = np.empty((T, N), np.float32)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    margin = np.empty((T,), np.float64)
    rc = lib.moe_oracle_router(T, d, N, K, score_fn, renormalize, n_groups, topk_groups, _ptr(x),
                               _ptr(W), _ptr(rb),
                               _ptr(sb), _ptr(logits), _ptr(probs), _ptr(keys), _ptr(idx),
                               _ptr(w), _ptr(margin))
    if rc != 0:
        raise ValueError(f"moe_oracle_router failed ({rc})")
    return dict(logits=logits, probs=probs, keys=keys, idx=idx, w=w, margin=margin)


def capacity(capacity_factor, T, K, N):
    """C = ceil(c T K / N), or -1 for no cap (c <= 0)."""
    return int(_load().moe_oracle_capacity(float(capacity_factor), T, K, N))


def permute(topk_idx, N, capacity_factor=0.0):
    """Counting sort of the token copies by expert. Returns counts, offsets,
    perm_src, inv_row (int32). With capacity_factor > 0 only the first
    ceil(c T K / N) copies of each expert (token order) are placed: offsets
    count kept copies, perm_src lists them, inv_row is -1 for dropped ones."""
    lib = _load()
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, K = idx.shape
    counts = np.empty((N,), np.int32)
    offsets = np.empty((N + 1,), np.int32)
    perm_src = np.full((T * K,), -1, np.int32)
    inv_row = np.empty((T * K,), np.int32)
    if capacity_factor > 0:
        cap = capacity(capacity_factor, T, K, N)
        rc = lib.moe_oracle_permute_cap(T, K, N, cap, _ptr(idx), _ptr(counts), _ptr(offsets),
                                        _ptr(perm_src), _ptr(inv_row))
        if rc != 0:
            raise ValueError(f"moe_oracle_permute_cap failed ({rc})")
        return dict(counts=counts, offsets=offsets, perm_src=perm_src, inv_row=inv_row)
    rc = lib.moe_oracle_permute(T, K, N, _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(perm_src),
                                _ptr(inv_row))
    if rc != 0:
        raise ValueError(f"moe_oracle_permute failed ({rc})")
    return dict(counts=counts, offsets=offsets, perm_src=perm_src, inv_row=inv_row)


def expert_ffn(x, w_gate, w_up, w_down, return_h=False):
    """One SwiGLU expert on one token: x fp64 [d], weights bf16 bit patterns.
    Returns y (fp64 [d]), or (h, y) with the fp64 hidden activation h [F]."""
    lib = _load()
    x = _f64(x)
    wg, wu, wd = _bf16_bits(w_gate), _bf16_bits(w_up), _bf16_bits(w_down)
    F, d = wg.shape
    assert x.shape == (d,) and wu.shape == (F, d) and wd.shape == (d, F)
    h = np.empty((F,), np.float64)
    y = np.empty((d,), np.float64)
    lib.moe_oracle_expert_ffn(d, F, _ptr(x), _ptr(wg), _ptr(wu), _ptr(wd), _ptr(h), _ptr(y))
    return (h, y) if return_h else y


def e4m3_value(code: int) -> float:
    """The value of one FP8 E4M3 code (0..255) as the oracle decodes it."""
    return float(_load().moe_oracle_e4m3_to_double(int(code)))


def _u8(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError("fp8 expert weights must be E4M3 codes (uint8)")
    return a


def expert_ffn_fp8(x, q_gate, s_gate, q_up, s_up, q_down, s_down, return_h=False):
    """One SwiGLU expert with FP8 E4M3 weights: codes uint8 ([F][d], [F][d],
    [d][F]) and fp32 per-row scales ([F], [F], [d]). Returns y (or (h, y))."""
    lib = _load()
    x = _f64(x)
    qg, qu, qd = _u8(q_gate), _u8(q_up), _u8(q_down)
    sg, su, sd = _f32(s_gate), _f32(s_up), _f32(s_down)
    F, d = qg.shape
    assert x.shape == (d,) and qu.shape == (F, d) and qd.shape == (d, F)
    assert sg.shape == (F,) and su.shape == (F,) and sd.shape == (d,)
    h = np.empty((F,), np.float64)
    y = np.empty((d,), np.float64)
    lib.moe_oracle_expert_ffn_fp8(d, F, _ptr(x), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su), _ptr(qd),
                                  _ptr(sd), _ptr(h), _ptr(y))
    return (h, y) if return_h else y


def combine(w, y, shared=None):
    """out = sum_k w[k] * y[k] (+ shared)."""
    lib = _load()
    w = _f64(w)
    y = _f64(y)
    K, d = y.shape
    sh = _f64(shared)
    out = np.empty((d,), np.float64)
    lib.moe_oracle_combine(K, d, _ptr(w), _ptr(y), _ptr(sh), _ptr(out))
    return out


def _ptr_array(mats, n):
    arr = (ctypes.c_void_p * n)()
    keep = []
    for i in range(n):
        m = mats[i] if mats is not None and i < len(mats) else None
        if m is None:
            arr[i] = None
        else:
            b = _bf16_bits(m)
            keep.append(b)
            arr[i] = b.ctypes.data
    return arr, keep


def layer(hidden, w_router, w_gate, w_up, w_down, K, score_fn=SOFTMAX, renormalize=1,
          router_bias=None, sel_bias=None, ws_gate=None, ws_up=None, ws_down=None, n_groups=0,
          topk_groups=0, keep=None):
    """The whole layer for the rows of `hidden` (fp32 [n][d]).

    w_gate / w_up / w_down: sequences of N per-expert bf16 matrices (uint16 bit
    patterns or torch bf16), an entry may be None if no token picks it.
    ws_*: sequences of S shared-expert matrices or None.
    keep: uint8 [n][K] or None; 0 marks a copy dropped by its expert's capacity.
    Returns dict(idx, w, margin, out) with out fp64 [n][d].
    """
    lib = _load()
    x = _f32(hidden)
    W = _f32(w_router)
    n, d = x.shape
    N = W.shape[1]
    F = next(_bf16_bits(m).shape[0] for m in w_gate if m is not None)
    S = 0 if ws_gate is None else len(ws_gate)
    Fs = _bf16_bits(ws_gate[0]).shape[0] if S else 0
    g_arr, k1 = _ptr_array(w_gate, N)
    u_arr, k2 = _ptr_array(w_up, N)
    d_arr, k3 = _ptr_array(w_down, N)
    sg_arr, k4 = _ptr_array(ws_gate, max(S, 1))
    su_arr, k5 = _ptr_array(ws_up, max(S, 1))
    sd_arr, k6 = _ptr_array(ws_down, max(S, 1))
    rb, sb = _f32(router_bias), _f32(sel_bias)
    keep_a = None if keep is None else np.ascontiguousarray(keep, dtype=np.uint8)
    idx = np.empty((n, K), np.int32)
    w = np.empty((n, K), np.float64)
    margin = np.empty((n,), np.float64)
    out = np.empty((n, d), np.float64)
    rc = lib.moe_oracle_layer(n, d, N, K, F, S, Fs, score_fn, renormalize, n_groups, topk_groups,
                              _ptr(x), _ptr(W),
                              _ptr(rb), _ptr(sb), ctypes.cast(g_arr, ctypes.c_void_p),
                              ctypes.cast(u_arr, ctypes.c_void_p),
                              ctypes.cast(d_arr, ctypes.c_void_p),
                              ctypes.cast(sg_arr, ctypes.c_void_p) if S else None,
                              ctypes.cast(su_arr, ctypes.c_void_p) if S else None,
                              ctypes.cast(sd_arr, ctypes.c_void_p) if S else None,
                              _ptr(keep_a), _ptr(idx), _ptr(w), _ptr(margin), _ptr(out))
    del k1, k2, k3, k4, k5, k6
    if rc != 0:
        raise ValueError(f"moe_oracle_layer failed ({rc})")
    return dict(idx=idx, w=w, margin=margin, out=out)


def _raw_ptr_array(mats, n, conv):
    arr = (ctypes.c_void_p * n)()
    keep = []
    for i in range(n):
        m = mats[i] if mats is not None and i < len(mats) else None
        if m is None:
            arr[i] = None
        else:
            b = conv(m)
            keep.append(b)
            arr[i] = b.ctypes.data
    return arr, keep


def layer_fp8(hidden, w_router, q_gate, s_gate, q_up, s_up, q_down, s_down, K, score_fn=SOFTMAX,
              renormalize=1, router_bias=None, sel_bias=None, qs_gate=None, ss_gate=None, qs_up=None,
              ss_up=None, qs_down=None, ss_down=None, n_groups=0, topk_groups=0, keep=None):
    """The whole layer with FP8 E4M3 expert weights (per-expert uint8 codes
    and fp32 per-row scales; routed: q_*/s_*, shared: qs_*/ss_*). Otherwise
    as layer(). Returns dict(idx, w, margin, out)."""
    lib = _load()
    x = _f32(hidden)
    W = _f32(w_router)
    n, d = x.shape
    N = W.shape[1]
    F = next(_u8(m).shape[0] for m in q_gate if m is not None)
    S = 0 if qs_gate is None else len(qs_gate)
    Fs = _u8(qs_gate[0]).shape[0] if S else 0
    arrays = []
    keepalive = []
    for mats, cnt, conv in ((q_gate, N, _u8), (q_up, N, _u8), (q_down, N, _u8), (s_gate, N, _f32),
                            (s_up, N, _f32), (s_down, N, _f32), (qs_gate, S, _u8), (qs_up, S, _u8),
                            (qs_down, S, _u8), (ss_gate, S, _f32), (ss_up, S, _f32),
                            (ss_down, S, _f32)):
        if cnt == 0:
            arrays.append(None)
            continue
        arr, k = _raw_ptr_array(mats, cnt, conv)
        keepalive.append((arr, k))
        arrays.append(ctypes.cast(arr, ctypes.c_void_p))
    rb, sb = _f32(router_bias), _f32(sel_bias)
    keep_a = None if keep is None else np.ascontiguousarray(keep, dtype=np.uint8)
    idx = np.empty((n, K), np.int32)
    w = np.empty((n, K), np.float64)
    margin = np.empty((n,), np.float64)
    out = np.empty((n, d), np.float64)
    rc = lib.moe_oracle_layer_fp8(n, d, N, K, F, S, Fs, score_fn, renormalize, n_groups, topk_groups,
                                  _ptr(x), _ptr(W), _ptr(rb), _ptr(sb), *arrays, _ptr(keep_a),
                                  _ptr(idx), _ptr(w), _ptr(margin), _ptr(out))
    del keepalive
    if rc != 0:
        raise ValueError(f"moe_oracle_layer_fp8 failed ({rc})")
    return dict(idx=idx, w=w, margin=margin, out=out)


def expert_choice_capacity(capacity_factor, T, K, N):
    """Tokens each expert takes under expert-choice routing: ceil(c T K / N)
    (c = 1 when not given), at most T."""
    c = capacity(capacity_factor if capacity_factor > 0 else 1.0, T, K, N)
    return min(c, T)


def expert_choice(hidden, w_router, C, score_fn=SOFTMAX, router_bias=None):
    """Expert-choice selection over the rows of `hidden`: each expert's C
    tokens (ascending), their scores and the per-expert selection margin.
    Returns dict(row_token int32 [N][C], row_w fp64 [N][C], margin fp64 [N])."""
    lib = _load()
    x = _f32(hidden)
    W = _f32(w_router)
    T, d = x.shape
    N = W.shape[1]
    rb = _f32(router_bias)
    row_token = np.empty((N, C), np.int32)
    row_w = np.empty((N, C), np.float64)
    margin = np.empty((N,), np.float64)
    rc = lib.moe_oracle_expert_choice(T, d, N, score_fn, C, _ptr(x), _ptr(W), _ptr(rb), _ptr(row_token),
                                      _ptr(row_w), _ptr(margin))
    if rc != 0:
        raise ValueError(f"moe_oracle_expert_choice failed ({rc})")
    return dict(row_token=row_token, row_w=row_w, margin=margin)


def routing_from_expert_choice(row_token, row_w, T):
    """Per-token (expert, weight) lists, expert ascending, padded with -1 / 0."""
    N, C = row_token.shape
    lists = [[] for _ in range(T)]
    for e in range(N):
        for j in range(C):
            lists[row_token[e, j]].append((e, row_w[e, j]))
    M = max(1, max(len(v) for v in lists))
    idx = np.full((T, M), -1, np.int32)
    w = np.zeros((T, M), np.float64)
    for t, v in enumerate(lists):
        for k, (e, ww) in enumerate(v):
            idx[t, k], w[t, k] = e, ww
    return idx, w


def layer_routed(hidden, idx, w, w_gate, w_up, w_down, ws_gate=None, ws_up=None, ws_down=None):
    """out[t] = sum_k w[t][k] E_{idx[t][k]}(x_t) (+ shared), slots with idx < 0 skipped."""
    lib = _load()
    x = _f32(hidden)
    n, d = x.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = _f64(w)
    M = idx.shape[1]
    N = len(w_gate)
    F = next(_bf16_bits(m).shape[0] for m in w_gate if m is not None)
    S = 0 if ws_gate is None else len(ws_gate)
    Fs = _bf16_bits(ws_gate[0]).shape[0] if S else 0
    g_arr, k1 = _ptr_array(w_gate, N)
    u_arr, k2 = _ptr_array(w_up, N)
    d_arr, k3 = _ptr_array(w_down, N)
    sg_arr, k4 = _ptr_array(ws_gate, max(S, 1))
    su_arr, k5 = _ptr_array(ws_up, max(S, 1))
    sd_arr, k6 = _ptr_array(ws_down, max(S, 1))
    out = np.empty((n, d), np.float64)
    rc = lib.moe_oracle_layer_routed(n, d, N, M, F, S, Fs, _ptr(x), _ptr(idx), _ptr(w),
                                     ctypes.cast(g_arr, ctypes.c_void_p), ctypes.cast(u_arr, ctypes.c_void_p),
                                     ctypes.cast(d_arr, ctypes.c_void_p),
                                     ctypes.cast(sg_arr, ctypes.c_void_p) if S else None,
                                     ctypes.cast(su_arr, ctypes.c_void_p) if S else None,
                                     ctypes.cast(sd_arr, ctypes.c_void_p) if S else None, _ptr(out))
    del k1, k2, k3, k4, k5, k6
    if rc != 0:
        raise ValueError(f"moe_oracle_layer_routed failed ({rc})")
    return out


def layer_routed_fp8(hidden, idx, w, q_gate, s_gate, q_up, s_up, q_down, s_down, qs_gate=None, ss_gate=None,
                     qs_up=None, ss_up=None, qs_down=None, ss_down=None):
    """layer_routed with FP8 E4M3 experts (codes + per-row scales, as layer_fp8)."""
    lib = _load()
    x = _f32(hidden)
    n, d = x.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = _f64(w)
    M = idx.shape[1]
    N = len(q_gate)
    F = next(_u8(m).shape[0] for m in q_gate if m is not None)
    S = 0 if qs_gate is None else len(qs_gate)
    Fs = _u8(qs_gate[0]).shape[0] if S else 0
    arrays, keepalive = [], []
    for mats, cnt, conv in ((q_gate, N, _u8), (q_up, N, _u8), (q_down, N, _u8), (s_gate, N, _f32),
                            (s_up, N, _f32), (s_down, N, _f32), (qs_gate, S, _u8), (qs_up, S, _u8),
                            (qs_down, S, _u8), (ss_gate, S, _f32), (ss_up, S, _f32),
                            (ss_down, S, _f32)):
        if cnt == 0:
            arrays.append(None)
            continue
        arr, k = _raw_ptr_array(mats, cnt, conv)
        keepalive.append((arr, k))
        arrays.append(ctypes.cast(arr, ctypes.c_void_p))
    out = np.empty((n, d), np.float64)
    rc = lib.moe_oracle_layer_routed_fp8(n, d, N, M, F, S, Fs, _ptr(x), _ptr(idx), _ptr(w), *arrays, _ptr(out))
    del keepalive
    if rc != 0:
        raise ValueError(f"moe_oracle_layer_routed_fp8 failed ({rc})")
    return out


def e2m1_value(code: int) -> float:
    """The value of one FP4 E2M1 code (0..15) as the oracle decodes it."""
    return float(_load().moe_oracle_e2m1_to_double(int(code)))


def e8m0_value(code: int) -> float:
    """The value of one E8M0 scale code (0..255) as the oracle decodes it."""
    return float(_load().moe_oracle_e8m0_to_double(int(code)))


def expert_ffn_mxfp4(x, q_gate, b_gate, q_up, b_up, q_down, b_down, return_h=False):
    """One SwiGLU expert with MXFP4 weights: packed E2M1 codes uint8 ([F][d/2],
    [F][d/2], [d][F/2]) and E8M0 block scales uint8 ([F][d/32], [F][d/32],
    [d][F/32]). Returns y (or (h, y))."""
    lib = _load()
    x = _f64(x)
    qg, qu, qd = _u8(q_gate), _u8(q_up), _u8(q_down)
    bg, bu, bd = _u8(b_gate), _u8(b_up), _u8(b_down)
    F, d2 = qg.shape
    d = 2 * d2
    assert x.shape == (d,) and qu.shape == (F, d2) and qd.shape == (d, F // 2)
    assert bg.shape == (F, d // 32) and bu.shape == (F, d // 32) and bd.shape == (d, F // 32)
    h = np.empty((F,), np.float64)
    y = np.empty((d,), np.float64)
    lib.moe_oracle_expert_ffn_mxfp4(d, F, _ptr(x), _ptr(qg), _ptr(bg), _ptr(qu), _ptr(bu), _ptr(qd),
                                    _ptr(bd), _ptr(h), _ptr(y))
    return (h, y) if return_h else y


def layer_mxfp4(hidden, w_router, q_gate, b_gate, q_up, b_up, q_down, b_down, K, score_fn=SOFTMAX,
                renormalize=1, router_bias=None, sel_bias=None, qs_gate=None, bs_gate=None, qs_up=None,
                bs_up=None, qs_down=None, bs_down=None, n_groups=0, topk_groups=0, keep=None):
    """The whole layer with MXFP4 expert weights (per-expert packed codes and
    E8M0 block scales; routed: q_*/b_*, shared: qs_*/bs_*). Otherwise as
    layer(). Returns dict(idx, w, margin, out)."""
    lib = _load()
    x = _f32(hidden)
    W = _f32(w_router)
    n, d = x.shape
    N = W.shape[1]
    F = next(_u8(m).shape[0] for m in q_gate if m is not None)
    S = 0 if qs_gate is None else len(qs_gate)
    Fs = _u8(qs_gate[0]).shape[0] if S else 0
    arrays, keepalive = [], []
    for mats, cnt in ((q_gate, N), (q_up, N), (q_down, N), (b_gate, N), (b_up, N), (b_down, N),
                      (qs_gate, S), (qs_up, S), (qs_down, S), (bs_gate, S), (bs_up, S), (bs_down, S)):
        if cnt == 0:
            arrays.append(None)
            continue
        arr, k = _raw_ptr_array(mats, cnt, _u8)
        keepalive.append((arr, k))
        arrays.append(ctypes.cast(arr, ctypes.c_void_p))
    rb, sb = _f32(router_bias), _f32(sel_bias)
    keep_a = None if keep is None else np.ascontiguousarray(keep, dtype=np.uint8)
    idx = np.empty((n, K), np.int32)
    w = np.empty((n, K), np.float64)
    margin = np.empty((n,), np.float64)
    out = np.empty((n, d), np.float64)
    rc = lib.moe_oracle_layer_mxfp4(n, d, N, K, F, S, Fs, score_fn, renormalize, n_groups, topk_groups,
                                    _ptr(x), _ptr(W), _ptr(rb), _ptr(sb), *arrays, _ptr(keep_a), _ptr(idx),
                                    _ptr(w), _ptr(margin), _ptr(out))
    del keepalive
    if rc != 0:
        raise ValueError(f"moe_oracle_layer_mxfp4 failed ({rc})")
    return dict(idx=idx, w=w, margin=margin, out=out)


def layer_routed_mxfp4(hidden, idx, w, q_gate, b_gate, q_up, b_up, q_down, b_down, qs_gate=None, bs_gate=None,
                       qs_up=None, bs_up=None, qs_down=None, bs_down=None):
    """layer_routed with MXFP4 experts (packed codes + E8M0 block scales, as layer_mxfp4)."""
    lib = _load()
    x = _f32(hidden)
    n, d = x.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = _f64(w)
    M = idx.shape[1]
    N = len(q_gate)
    F = next(_u8(m).shape[0] for m in q_gate if m is not None)
    S = 0 if qs_gate is None else len(qs_gate)
    Fs = _u8(qs_gate[0]).shape[0] if S else 0
    arrays, keepalive = [], []
    for mats, cnt in ((q_gate, N), (q_up, N), (q_down, N), (b_gate, N), (b_up, N), (b_down, N),
                      (qs_gate, S), (qs_up, S), (qs_down, S), (bs_gate, S), (bs_up, S), (bs_down, S)):
        if cnt == 0:
            arrays.append(None)
            continue
        arr, k = _raw_ptr_array(mats, cnt, _u8)
        keepalive.append((arr, k))
        arrays.append(ctypes.cast(arr, ctypes.c_void_p))
    out = np.empty((n, d), np.float64)
    rc = lib.moe_oracle_layer_routed_mxfp4(n, d, N, M, F, S, Fs, _ptr(x), _ptr(idx), _ptr(w), *arrays, _ptr(out))
    del keepalive
    if rc != 0:
        raise ValueError(f"moe_oracle_layer_routed_mxfp4 failed ({rc})")
    return out
