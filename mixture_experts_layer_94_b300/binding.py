"""Thin ctypes binding of libmoe.so (include/moe.h) for torch tensors.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Importing this module loads libmoe.so and raises if it is missing or
cannot be loaded; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from .inputs import MoEConfig

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "moe.h")

MOE_OK = 0
MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA = -1, -2, -3, -4
MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_BOUNDS = -5, -6
CALL_PERMUTE, CALL_GROUPED_SWIGLU, CALL_LAYER_FORWARD, CALL_ROUTER = 0, 1, 2, 3
SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1
DT_F32, DT_BF16 = 0, 1
ROUTING_TOKEN_CHOICE, ROUTING_EXPERT_CHOICE = 0, 1
EXPERT_BF16, EXPERT_FP8_E4M3, EXPERT_MXFP4 = 0, 1, 2
MOE_ERR_RANGE = -7


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("ffn", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("shared_ffn", ctypes.c_int32), ("score_fn", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("hidden_dtype", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("capacity_factor", ctypes.c_double), ("routing", ctypes.c_int32),
                ("expert_dtype", ctypes.c_int32)]


WEIGHT_FIELDS = ("w_router", "router_bias", "sel_bias", "w_gate", "w_up", "w_down", "ws_gate", "ws_up",
                 "ws_down", "w_gate_scale", "w_up_scale", "w_down_scale", "ws_gate_scale", "ws_up_scale",
                 "ws_down_scale", "mx_prep")


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so is not built ({LIB_PATH}); run "
                          "python -m mixture_experts_layer_94_b300.build")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    pp = ctypes.POINTER(Problem)
    sig = {
        "moe_status_string": ([i32], ctypes.c_char_p),
        "moe_problem_check": ([pp], i32),
        "moe_workspace_bytes": ([pp, i32], sz),
        "moe_router_topk": ([pp] + [P] * 8 + [sz, P], i32),
        "moe_permute": ([pp] + [P] * 8 + [sz, P], i32),
        "moe_grouped_swiglu": ([pp] + [P] * 8 + [sz, P], i32),
        "moe_grouped_swiglu_fp8": ([pp] + [P] * 11 + [sz, P], i32),
        "moe_grouped_swiglu_mxfp4": ([pp] + [P] * 11 + [sz, P], i32),
        "moe_combine": ([pp] + [P] * 6, i32),
        "moe_layer_forward": ([pp, ctypes.POINTER(Weights)] + [P] * 6 + [sz, P], i32),
        "moe_get_device_status": ([P, P], i32),
        "moe_layer_forward_profiled": ([pp, ctypes.POINTER(Weights)] + [P] * 3 + [sz, P, P], i32),
        "moe_layer_forward_kernel_count": ([pp, ctypes.POINTER(Weights)], i32),
        "moe_layer_small_batch": ([pp], i32),
        "moe_mxfp4_prep_bytes": ([pp], sz),
        "moe_mxfp4_prepare": ([pp, ctypes.POINTER(Weights), P, sz, P], i32),
        "moe_expert_choice_select": ([pp] + [P] * 7 + [sz, P], i32),
        "moe_expert_choice_capacity": ([pp], ctypes.c_int64),
        "moe_permute_static": ([pp] + [P] * 8, i32),
        "moe_debug_stall_wait": ([P, sz, ctypes.c_uint32, P], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def header_functions() -> list:
    """Names of the functions include/moe.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\*|moe_status_t|size_t|int32_t|int64_t)\s+(moe_\w+)\s*\(",
                                 text, re.M)))


def status_string(status: int) -> str:
    return lib.moe_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoEError(status, where)


def problem(cfg: MoEConfig = None, **kw) -> Problem:
    """A moe_problem_t from a workload config (fields may be overridden)."""
    f = {}
    if cfg is not None:
        f = dict(T=cfg.T, d_model=cfg.d, n_experts=cfg.N, top_k=cfg.K, ffn=cfg.F, n_shared=cfg.S,
                 shared_ffn=cfg.Fs, score_fn=cfg.score_fn, renormalize=cfg.renormalize,
                 hidden_dtype=DT_F32 if cfg.hidden_dtype == "f32" else DT_BF16, n_groups=cfg.n_groups,
                 topk_groups=cfg.topk_groups, capacity_factor=cfg.capacity_factor,
                 routing=ROUTING_EXPERT_CHOICE if cfg.routing == "expert" else ROUTING_TOKEN_CHOICE,
                 expert_dtype={"fp8": EXPERT_FP8_E4M3, "mxfp4": EXPERT_MXFP4}.get(cfg.expert_dtype, EXPERT_BF16))
    f.update(kw)
    return Problem(**f)


def problem_check(p: Problem) -> int:
    return int(lib.moe_problem_check(ctypes.byref(p)))


def workspace_bytes(p: Problem, call: int) -> int:
    return int(lib.moe_workspace_bytes(ctypes.byref(p), call))


def new_workspace(p: Problem, call: int, device="cuda") -> torch.Tensor:
    """Zero-filled workspace (its first 256 bytes are the device error word)."""
    n = workspace_bytes(p, call)
    if n == 0:
        raise ValueError("invalid problem")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _p(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def router_topk(p: Problem, hidden, w_router, topk_idx, topk_w, router_bias=None, sel_bias=None,
                logits=None, ws=None, stream=None):
    if ws is None:
        ws = new_workspace(p, CALL_ROUTER, hidden.device)
    _check(lib.moe_router_topk(ctypes.byref(p), _p(hidden), _p(w_router), _p(router_bias),
                               _p(sel_bias), _p(topk_idx), _p(topk_w), _p(logits), _p(ws), ws.numel(),
                               _stream(stream)), "moe_router_topk")


def expert_choice_capacity(cfg: MoEConfig, T: int = None) -> int:
    """Tokens every expert takes under expert-choice routing, as the library
    computes it (moe_expert_choice_capacity)."""
    c = int(lib.moe_expert_choice_capacity(ctypes.byref(problem(cfg, **({} if T is None else {"T": T})))))
    if c < 0:
        raise ValueError("invalid problem")
    return c


def expert_choice_select(p: Problem, hidden, w_router, row_token, row_w, offsets, router_bias=None,
                         ws=None, stream=None):
    if ws is None:
        ws = new_workspace(p, CALL_ROUTER, hidden.device)
    _check(lib.moe_expert_choice_select(ctypes.byref(p), _p(hidden), _p(w_router), _p(router_bias),
                                        _p(row_token), _p(row_w), _p(offsets), _p(ws), ws.numel(),
                                        _stream(stream)), "moe_expert_choice_select")


def permute(p: Problem, topk_idx, hidden, counts, offsets, perm_src, inv_row, x_perm, ws,
            stream=None):
    _check(lib.moe_permute(ctypes.byref(p), _p(topk_idx), _p(hidden), _p(counts), _p(offsets),
                           _p(perm_src), _p(inv_row), _p(x_perm), _p(ws), ws.numel(),
                           _stream(stream)), "moe_permute")


def grouped_swiglu(p: Problem, x_perm, offsets, w_gate, w_up, w_down, h_perm, y_perm, ws,
                   stream=None):
    _check(lib.moe_grouped_swiglu(ctypes.byref(p), _p(x_perm), _p(offsets), _p(w_gate), _p(w_up),
                                  _p(w_down), _p(h_perm), _p(y_perm), _p(ws), ws.numel(),
                                  _stream(stream)), "moe_grouped_swiglu")


def grouped_swiglu_fp8(p: Problem, x_perm, offsets, w_gate, w_gate_scale, w_up, w_up_scale, w_down,
                       w_down_scale, h_perm, y_perm, ws, stream=None):
    _check(lib.moe_grouped_swiglu_fp8(ctypes.byref(p), _p(x_perm), _p(offsets), _p(w_gate), _p(w_gate_scale),
                                      _p(w_up), _p(w_up_scale), _p(w_down), _p(w_down_scale), _p(h_perm),
                                      _p(y_perm), _p(ws), ws.numel(), _stream(stream)),
           "moe_grouped_swiglu_fp8")


def grouped_swiglu_mxfp4(p: Problem, x_perm, offsets, w_gate, w_gate_bscale, w_up, w_up_bscale, w_down,
                         w_down_bscale, h_perm, y_perm, ws, stream=None):
    _check(lib.moe_grouped_swiglu_mxfp4(ctypes.byref(p), _p(x_perm), _p(offsets), _p(w_gate), _p(w_gate_bscale),
                                        _p(w_up), _p(w_up_bscale), _p(w_down), _p(w_down_bscale), _p(h_perm),
                                        _p(y_perm), _p(ws), ws.numel(), _stream(stream)),
           "moe_grouped_swiglu_mxfp4")


def combine(p: Problem, y_perm, inv_row, topk_w, out, shared_out=None, stream=None):
    _check(lib.moe_combine(ctypes.byref(p), _p(y_perm), _p(inv_row), _p(topk_w), _p(shared_out),
                           _p(out), _stream(stream)), "moe_combine")


def weights_struct(w: dict) -> Weights:
    def ptr(k):
        t = w.get(k)
        return None if t is None else t.data_ptr()
    return Weights(*(ptr(k) for k in WEIGHT_FIELDS))


def layer_forward(p: Problem, weights: Weights, hidden, out, ws, topk_idx=None, topk_w=None,
                  counts=None, stream=None):
    _check(lib.moe_layer_forward(ctypes.byref(p), ctypes.byref(weights), _p(hidden), _p(out),
                                 _p(topk_idx), _p(topk_w), _p(counts), _p(ws), ws.numel(),
                                 _stream(stream)), "moe_layer_forward")


LAYER_STAGES = ("router_topk", "route_and_pack", "gemm_schedule", "gateup_swiglu_gemm",
                "down_scatter_gemm", "finalize")


def layer_forward_profiled(p: Problem, weights: Weights, hidden, out, ws, events, stream=None):
    """moe_layer_forward plus a cudaEventRecord before the first kernel and after
    each of the LAYER_STAGES stages (events: len(LAYER_STAGES) + 1 torch.cuda.Event)."""
    for e in events:  # torch creates the CUDA event lazily, on its first record
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * (len(LAYER_STAGES) + 1))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib.moe_layer_forward_profiled(ctypes.byref(p), ctypes.byref(weights), _p(hidden), _p(out),
                                          _p(ws), ws.numel(), arr, _stream(stream)),
           "moe_layer_forward_profiled")


def layer_small_batch(p: Problem) -> bool:
    """True when moe_layer_forward runs p's expert FFNs on the CUDA cores
    (decode-sized token-choice batches), False on the grouped GEMMs."""
    r = int(lib.moe_layer_small_batch(ctypes.byref(p)))
    if r < 0:
        raise ValueError("invalid problem")
    return r == 1


def layer_forward_kernel_count(p: Problem, weights: Weights = None) -> int:
    return int(lib.moe_layer_forward_kernel_count(ctypes.byref(p), None if weights is None
                                                  else ctypes.byref(weights)))


def mxfp4_prep_bytes(p: Problem) -> int:
    return int(lib.moe_mxfp4_prep_bytes(ctypes.byref(p)))


def mxfp4_prepare(p: Problem, weights: Weights, prep: torch.Tensor, stream=None):
    """Fill `prep` (a uint8 CUDA tensor of mxfp4_prep_bytes(p) bytes) with the
    MXFP4 weight preparation; set weights.mx_prep to use it."""
    _check(lib.moe_mxfp4_prepare(ctypes.byref(p), ctypes.byref(weights), _p(prep), prep.numel(),
                                 _stream(stream)), "moe_mxfp4_prepare")


def debug_stall_wait(ws, timeout_us: int, stream=None):
    """Failure-detection hook: a bounded wait nothing satisfies (see include/moe.h)."""
    _check(lib.moe_debug_stall_wait(_p(ws), ws.numel(), int(timeout_us), _stream(stream)),
           "moe_debug_stall_wait")


def get_device_status(ws, stream=None) -> int:
    return int(lib.moe_get_device_status(_p(ws), _stream(stream)))


class MoELayer:
    """One MoE FFN layer on the GPU: weights and workspace held on the device.

    weights: dict with w_router, router_bias, sel_bias, w_gate, w_up, w_down,
    ws_gate, ws_up, ws_down and, for FP8 / MXFP4 experts, the *_scale row or
    block scales (torch CUDA tensors or None). MXFP4 weights are prepared once
    here (moe_mxfp4_prepare) unless mx_prepare is False; every call then skips
    the per-call preparation.
    """

    def __init__(self, cfg: MoEConfig, weights: dict, T: int = None, device="cuda", mx_prepare: bool = True):
        self.cfg = cfg if T is None else cfg.with_(T=T)
        self.device = torch.device(device)
        self.w = {k: (None if v is None else v.to(self.device).contiguous())
                  for k, v in weights.items() if k in WEIGHT_FIELDS and k != "mx_prep"}
        self.ws_struct = weights_struct(self.w)
        self.mx_prep = None
        if cfg.expert_dtype == "mxfp4" and mx_prepare:
            p = problem(self.cfg)
            self.mx_prep = torch.empty(mxfp4_prep_bytes(p), dtype=torch.uint8, device=self.device)
            mxfp4_prepare(p, self.ws_struct, self.mx_prep)
            self.ws_struct.mx_prep = self.mx_prep.data_ptr()
        self._ws = {}

    def workspace(self, T: int) -> torch.Tensor:
        if T not in self._ws:
            self._ws[T] = new_workspace(problem(self.cfg, T=T), CALL_LAYER_FORWARD, self.device)
        return self._ws[T]

    def forward(self, hidden: torch.Tensor, out: torch.Tensor = None, topk_idx=None, topk_w=None,
                counts=None, stream=None) -> torch.Tensor:
        T = hidden.shape[0]
        if out is None:
            out = torch.empty(T, self.cfg.d, dtype=torch.bfloat16, device=self.device)
        layer_forward(problem(self.cfg, T=T), self.ws_struct, hidden, out, self.workspace(T),
                      topk_idx, topk_w, counts, stream)
        return out

    def status(self, T: int) -> int:
        return get_device_status(self.workspace(T))
