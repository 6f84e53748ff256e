"""Calls of the fused layer back to back on one stream, with no host
synchronisation between them, reusing one workspace.

Every kernel of the library starts early under programmatic dependent launch
and waits for its predecessor before touching global memory; a missing wait
would let one call's router, permutation or GEMMs read or overwrite another
call's workspace. Each call's output must equal the same call made alone (up
to the fp32 summation order of the down GEMM's atomic scatter).
"""
import pytest
import torch

from mixture_experts_layer_94_b300 import inputs
from tests import helpers as H

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from mixture_experts_layer_94_b300 import binding as B

CASES = {
    "bf16_decode": inputs.MoEConfig("bf16_decode", T=3, d=1024, N=128, K=8, F=256),
    "bf16_prefill_shared": inputs.MoEConfig("bf16_prefill_shared", T=700, d=512, N=16, K=4, F=384, S=1, Fs=256,
                                            score="sigmoid", sel_bias_var=0.1),
    "fp8_decode": inputs.MoEConfig("fp8_decode", T=5, d=1024, N=64, K=4, F=256, expert_dtype="fp8"),
    # single tokens: expert FFNs on the CUDA cores (FP8), on the GEMMs (MXFP4)
    "fp8_decode_T1_shared": inputs.MoEConfig("fp8_decode_T1_shared", T=1, d=1024, N=64, K=4, F=256, S=1, Fs=128,
                                             expert_dtype="fp8"),
    "mxfp4_decode_T1": inputs.MoEConfig("mxfp4_decode_T1", T=1, d=1024, N=64, K=4, F=256, expert_dtype="mxfp4"),
    "mxfp4_mixed": inputs.MoEConfig("mxfp4_mixed", T=40, d=512, N=32, K=4, F=320, S=1, Fs=128,
                                    expert_dtype="mxfp4"),
    "bf16_expert_choice": inputs.MoEConfig("bf16_expert_choice", T=256, d=512, N=8, K=2, F=256,
                                           routing="expert"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_back_to_back_calls_match_calls_made_alone(name):
    cfg = CASES[name]
    ins, dev = H.make_case(cfg)
    layer = B.MoELayer(cfg, dev)
    g = torch.Generator(device="cpu").manual_seed(7)
    hiddens = [dev["hidden"]] + [torch.randn(dev["hidden"].shape, generator=g).to(dev["hidden"].dtype).cuda()
                                 for _ in range(3)]
    alone = []
    for h in hiddens:
        alone.append(layer.forward(h).clone())
        torch.cuda.synchronize()
    outs = [torch.empty_like(alone[0]) for _ in hiddens]
    for h, o in zip(hiddens, outs):
        layer.forward(h, out=o)
    torch.cuda.synchronize()
    assert layer.status(cfg.T) == 0
    for i, (o, a) in enumerate(zip(outs, alone)):
        H.assert_same_but_summation_order(o, a, f"{name} call {i}")


@pytest.mark.parametrize("name", ["bf16_prefill_shared", "bf16_decode", "bf16_expert_choice"])
def test_calls_replayed_from_a_cuda_graph_match_eager_calls(name):
    """The layer captured into a CUDA graph and replayed on new inputs gives
    what eager calls give: every kernel's early start (programmatic dependent
    launch) becomes a graph edge, and the workspace and weights are bound at
    capture."""
    cfg = CASES[name]
    ins, dev = H.make_case(cfg)
    layer = B.MoELayer(cfg, dev)
    g = torch.Generator(device="cpu").manual_seed(11)
    xs = [torch.randn(dev["hidden"].shape, generator=g).to(dev["hidden"].dtype).cuda() for _ in range(2)]
    eager = [layer.forward(x).clone() for x in xs]
    torch.cuda.synchronize()
    static_in = xs[0].clone()
    static_out = torch.empty_like(eager[0])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # a first call outside capture (one-time launch attributes)
        layer.forward(static_in, out=static_out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(static_in, out=static_out)
    for x, e in zip(xs, eager):
        static_in.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        H.assert_same_but_summation_order(static_out, e, f"{name} graph replay")
    assert layer.status(cfg.T) == 0
