"""Failure detection on the GPU without a fault: a pipeline wait that nothing
satisfies gives up after its limit, reports MOE_ERR_TIMEOUT through the
workspace error word, and the CUDA context stays usable."""
import time

import pytest
import torch

from mixture_experts_layer_94_b300 import inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    from mixture_experts_layer_94_b300 import binding as B

    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.monotonic()
    B.debug_stall_wait(ws, 50_000)  # 50 ms limit
    st = B.get_device_status(ws)
    elapsed = time.monotonic() - t0
    assert st == -5, B.status_string(st)  # MOE_ERR_TIMEOUT
    assert elapsed < 1.0
    assert B.get_device_status(ws) == 0  # read-and-clear
    # the context is still usable: a small layer runs and reports no error
    cfg = inputs.TINY
    ins = inputs.make_inputs(cfg, seed=0)
    layer = B.MoELayer(cfg, {k: (None if v is None else v.cuda()) for k, v in ins.items()})
    out = layer.forward(ins["hidden"].cuda())
    torch.cuda.synchronize()
    assert layer.status(cfg.T) == 0 and torch.isfinite(out.float()).all()


def test_stall_hook_rejects_unbounded_limits():
    from mixture_experts_layer_94_b300 import binding as B

    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MoEError):
        B.debug_stall_wait(ws, 0)
    with pytest.raises(B.MoEError):
        B.debug_stall_wait(ws, 2_000_000)
