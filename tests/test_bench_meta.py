"""bench.py's description of what it measured (no GPU): the arithmetic type
and weight format per expert format, the workload config, the reference
arm's line shape, and the command line."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


@pytest.mark.parametrize("model,dtype,weights", [
    ("full", "f32 (bf16 weights and KV)", "bf16 random N(0,0.02)"),
    ("full_fp8", "fp8 E4M3 experts", "E4M3 codes"),
    ("full_fp4", "fp4 E2M1 experts", "E2M1 codes"),
])
def test_dtype_and_weights_text(model, dtype, weights):
    sh = synth.MODELS[model]
    assert dtype in bench.dtype_text(sh)
    assert weights in bench.weights_text(sh)


def test_workload_config_names_the_workload():
    inp = synth.make_inputs("full_bs1_8k")
    cfg = bench.workload_config(inp.workload, inp)
    assert cfg["workload"] == "full_bs1_8k" and cfg["global_batch"] == 1 and cfg["seq_len"] == 8192
    assert "128 experts top-8" in cfg["model"] and cfg["parallelism"].startswith("replicas")


def test_command_line(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert (a.gpus, a.impl, a.workload, a.service) == (1, "mine", "full_bs1_8k", 0) and a.warmup >= 3
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1",
                                      "--workload", "full_fp4_bs1_8k", "--service", "64"])
    a = bench.parse()
    assert (a.impl, a.steps, a.warmup, a.workload, a.service) == ("reference", 2, 1, "full_fp4_bs1_8k", 64)


def test_algorithmic_bytes_per_expert():
    # the roofline's per-expert bytes: codes plus scales for FP8 / FP4
    H, I = 2048, 768
    assert synth.MODELS["full"].expert_bytes() == 2 * 3 * H * I
    assert synth.MODELS["full_fp8"].expert_bytes() == 3 * H * I + 4 * (2 * I + H)
    assert synth.MODELS["full_fp4"].expert_bytes() == 3 * H * I // 2 + 3 * H * I // 16 + 4 * (2 * I + H)
