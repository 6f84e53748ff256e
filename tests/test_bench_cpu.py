"""The benchmark's host-side pieces on the CPU: the reference arm's JSON line
(the oracle on the host cores, no GPU needed) and the algorithmic work model
the roofline figures divide by, against closed forms of the layer's FLOPs and
bytes."""
import json
import os
import subprocess
import sys

import pytest

import bench
from mixture_experts_layer_94_b300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line_without_a_gpu():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["T"] == 64 and d["config"]["workload"]


def test_reference_arm_runs_on_rank_zero_only(capsys):
    # under torchrun every rank but 0 returns at once, printing nothing
    args = bench.argparse.Namespace(steps=1, warmup=0, gpus=2)
    cfg, desc = bench.WORKLOADS["tiny"]
    bench.run_reference(args, cfg, desc, world=2, rank=1)
    assert capsys.readouterr().out == ""


def test_work_model_matches_the_layers_closed_form():
    # Mixtral-shaped: router 2TdN, experts 6 d F T K; bytes: the 8 experts'
    # three bf16 matrices, the fp32 router, hidden in and out in bf16
    m = bench.work_model(inputs.MIXTRAL, counts=[1] * 8)
    T, d, N, K, F = 4096, 4096, 8, 2, 14336
    assert m["flops"] == 2 * T * d * N + 6 * d * F * T * K == 2886486458368
    assert m["bytes"] == 8 * 3 * d * F * 2 + 4 * d * N + T * d * (2 + 2) == 2885812224
    assert m["flops_gateup"] == 4 * d * F * T * K and m["bytes_gateup"] == 8 * 2 * d * F * 2
    # only experts that hold rows count: 8 of 128 at T = 1 (Qwen-shaped decode)
    q = inputs.QWEN_DECODE.with_(T=1)
    counts = [0] * 128
    for e in (3, 9, 17, 40, 41, 77, 100, 127):
        counts[e] = 1
    mq = bench.work_model(q, counts)
    assert mq["touched"] == 8 and mq["bytes_gateup"] == 8 * 2 * 4096 * 1536 * 2
    # DeepSeek-shaped: the shared expert's FLOPs and bytes are added in full
    ds = bench.work_model(inputs.DSV3, counts=[1] * 256)
    assert ds["flops"] == 2 * 8192 * 7168 * 256 + 6 * 7168 * 2048 * 8192 * 8 + 6 * 7168 * 2048 * 8192


@pytest.mark.parametrize("fmt,weight_bytes", [("fp8", 1), ("mxfp4", 0.5 + 1 / 32)])
def test_work_model_counts_the_stored_expert_bytes(fmt, weight_bytes):
    cfg = inputs.QWEN_DECODE.with_(T=1, expert_dtype=fmt)
    counts = [1] * 8 + [0] * 120
    m = bench.work_model(cfg, counts)
    d, F = 4096, 1536
    scales = (2 * F + d) * 4 if fmt == "fp8" else 0  # fp32 row scales of gate, up and down
    assert m["bytes_gateup"] + m["bytes_down"] == pytest.approx(8 * (3 * d * F * weight_bytes + scales))
