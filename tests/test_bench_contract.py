"""The benchmark's contract, checked on the CPU: the byte accounting behind every roofline
figure, and the JSON line of the reference arm (the CPU oracle) for a scan workload and a
neighbour-op workload."""
import json
import os
import socket
import subprocess
import sys

import bench
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_step_bytes():
    """State read and written once, plus q, k, v, o (bf16) and a, b, A_log, dt_bias."""
    inp = workloads.workload("bf16_decode_b256")
    B, H, D = 256, 32, 128
    state = B * H * D * D * 4
    io = 4 * B * H * D * 2 + 2 * B * H * 2
    assert bench.algorithmic_bytes(inp) == 2 * state + io + 2 * H * 4


def test_window_and_pool_bytes():
    win = workloads.workload("bf16_window_b256_t4")
    one = 256 * 32 * 128 * 128 * 4
    assert bench.io_bytes(win)["state_out"] == 4 * one
    slot = workloads.workload("bf16_slot_decode_b256")
    b = bench.io_bytes(slot)
    assert b["state_in"] == one and b["state_out"] == one and b["slots"] == 4 * 256


def test_per_key_gate_bytes():
    b = bench.io_bytes(workloads.workload("bf16_perkey_decode_b256"))
    assert b["a"] == 256 * 32 * 128 * 2 and b["params"] == 2 * 32 * 128 * 4


def test_neighbour_bytes():
    conv = workloads.any_workload("bf16_conv_decode_b256")
    b = bench.neighbour_io_bytes(conv)
    n = 256 * 12288 * 2
    assert b["x"] == n and b["y"] == n
    assert b["state_in"] == b["state_out"] == 256 * 3 * 12288 * 2
    assert b["weight"] == 12288 * 4 * 2 and b["bias"] == 0
    norm = workloads.any_workload("bf16_norm_gqa")
    b = bench.neighbour_io_bytes(norm)
    m = 2 * 8192 * 32 * 128 * 2
    assert b == {"x": m, "gate": m, "y": m, "scale": 128 * 2}


def test_rule_variant_bytes():
    """Rules without decay read no a, A_log or dt_bias; rules without the delta term no b;
    a shared beta is one value per token."""
    d = bench.io_bytes(workloads.workload("bf16_delta_prefill_t4096"))
    assert d["a"] == 0 and d["params"] == 0 and d["b"] == 4096 * 16 * 2
    sb = bench.io_bytes(workloads.workload("bf16_shared_beta_prefill_t4096"))
    assert sb["b"] == 4096 * 2 and sb["a"] == 4096 * 16 * 2
    pk = bench.io_bytes(workloads.workload("bf16_perkey_prefill_t4096"))
    assert pk["a"] == 4096 * 16 * 128 * 2 and pk["params"] == 2 * 16 * 128 * 4


def test_prefill_norm_bytes():
    """The prefill's bytes with o replaced by y, plus the gate and the norm scale."""
    inp = workloads.any_workload("varlen_bf16_prefill_norm")
    b = bench.prefill_norm_io_bytes(inp)
    o = 31979 * 16 * 128 * 2
    assert "o" not in b and b["y"] == o and b["gate"] == o and b["norm_scale"] == 128 * 2
    assert sum(b.values()) == bench.algorithmic_bytes(inp.prefill) + o + 128 * 2


def test_prefill_layer_bytes():
    """x, the conv's weight, bias and two states, a, b, the gate parameters, the states, the
    norm's scale and gate, and y."""
    inp = workloads.any_workload("varlen_bf16_prefill_layer")
    b = bench.prefill_layer_io_bytes(inp)
    T, C = inp.total_tokens, 2 * 16 * 128 + 16 * 128
    assert b["x"] == T * C * 2 and b["y"] == b["gate"] == T * 16 * 128 * 2
    assert b["conv_state_in"] == b["conv_state_out"] == 8 * 3 * C * 2
    assert b["state_in"] == b["state_out"] == 8 * 16 * 128 * 128 * 4


def test_reference_arm_prefill_layer_workload():
    d = _reference_line("varlen_bf16_prefill_layer")
    _check_line(d, "varlen_bf16_prefill_layer")
    assert d["unit"] == "tokens/s" and f"of {workloads.any_workload('varlen_bf16_prefill_layer').total_tokens} tokens" in d["cpu_baseline"]["sample"]


def test_neighbour_sample_is_bounded():
    inp = workloads.any_workload("bf16_conv_prefill_gqa")
    small, what = bench.neighbour_sample(inp)
    assert small.x.shape == (2, 8192, 512) and "512 of 8192" in what
    assert small.f64["x"].shape == (2, 8192, 512)


def _reference_line(name):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", name, "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def _check_line(d, name):
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["config"]["workload"] == name
    assert d["value"] > 0 and d["steps"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_scan_workload():
    d = _reference_line("tiny_f32_prefill")
    _check_line(d, "tiny_f32_prefill")
    assert d["unit"] == "tokens/s"


def test_reference_arm_neighbour_workload():
    d = _reference_line("bf16_conv_decode_b256")
    _check_line(d, "bf16_conv_decode_b256")
    assert d["unit"] == "GB/s"


def test_reference_arm_prefill_norm_workload():
    d = _reference_line("varlen_bf16_prefill_norm")
    _check_line(d, "varlen_bf16_prefill_norm")
    assert d["unit"] == "tokens/s" and "of 31979 tokens" in d["cpu_baseline"]["sample"]


def test_reference_arm_under_torchrun_prints_one_line():
    """Two ranks (gloo on the CPU): rank 0 alone runs the reference arm and prints its
    line; the other rank exits 0 without work."""
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--gpus", "2", "--impl", "reference", "--workload", "tiny_f32_prefill",
                        "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
