"""Host-side logic of the benchmark (no GPU): the algorithmic flop and byte models against
hand-counted values, the workload descriptions, and the rule that a recorded DRAM-traffic
figure is dropped once its kernel's sources change."""
import hashlib
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mesa_layer_gb300 import synth  # noqa: E402


def test_cg_flops_tiny_workload_by_hand():
    # 256 token-heads, 16 iterations plus the readout, each 2 d^2 + 2 d (C + 1) = 512 + 2080
    w = synth.workload("tiny_fp32_d16")
    iters = np.full((1, 1, 256), 16, dtype=np.int32)
    assert bench.cg_flops(w, iters) == 256 * 17 * 2592
    # the state sums add 4 d^2 per token-head: 45 088 per token-head in all
    assert (bench.cg_flops(w, iters) + bench.state_flops(w)) / 256 == 45088


def test_cg_flops_counts_each_tokens_own_iterations():
    w = synth.workload("fwd_fp32_d64", B=1, H=1, T=4)
    iters = np.array([[[0, 1, 5, 32]]], dtype=np.int32)
    per = 2 * 64 * 64 + 2 * 64 * 65
    assert bench.cg_flops(w, iters) == (1 + 2 + 6 + 33) * per


def test_tensor_core_issued_flops():
    w = synth.workload("fwd_bf16_d128", B=1, H=1, T=200)
    iters = np.full((1, 1, 200), 15, dtype=np.int32)
    iters[0, 0, 130] = 20  # the second 128-token chunk runs until its slowest token stops
    per_mma = 7 * 2.0 * 128 ** 3
    assert bench.tc_executed_flops(w, iters) == ((15 + 1) + (20 + 1)) * per_mma
    assert bench.tc_executed_flops(w, iters, readout=False) == (15 + 20) * per_mma


def test_decode_bytes_per_unit():
    w = synth.workload("decode_bf16_d128", B=1, H=1)
    # H and G (128 x 128 fp32 each) read and written, q, k, v read and out written in bf16,
    # gamma read and the iteration count written
    assert bench.decode_bytes(w) == 2 * 4 * (128 * 128 * 2) + 2 * (2 * 128 + 2 * 128) + 8
    ww = synth.workload("decode_warm_bf16_d128", B=1, H=1)
    assert bench.decode_bytes(ww) - bench.decode_bytes(w) == 2 * 4 * 128  # the start vector


def test_backward_flop_models():
    w = synth.workload("bwd_bf16_d128", B=1, H=1, T=64)
    d = 128
    assert bench.bwd_grad_flops(w) == 64 * (12 * d * d + 7 * d * 33)
    assert bench.bwd_rhs_flops(w) == 64 * (2 * d * d + 2 * d * 33)


def test_backward_split_flop_models():
    # with the row x state products on the tensor cores the gradient kernel keeps only the
    # intra-chunk work (7 d (C + 1) per token-head, C = 32); the products kernel counts five
    # d x d products (10 d^2) and issues 88 MMAs of 128 x 32 x 16 per 32-token chunk
    w = synth.workload("bwd_bf16_d128", B=1, H=1, T=64)
    assert bench.bwd_grad_flops(w, True) == 64 * 7 * 128 * 33
    assert bench.bwd_grad_flops(w) == 64 * (12 * 128 * 128 + 7 * 128 * 33)
    assert bench.bwd_sprod_flops(w) == 64 * 10 * 128 * 128
    assert bench.bwd_sprod_executed_flops(w) == 2 * 88 * 2 * 128 * 32 * 16


def test_preprocess_bytes():
    w = synth.workload("qkpre_bf16_d128", B=1, H=2, T=10)
    # q and k read and written in bf16, plus both tap arrays in fp32
    assert bench.preprocess_bytes(w) == 2 * 10 * 128 * 2 * 2 * 2 + 2 * 2 * 128 * 4 * 4


@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_workload_config_names_the_workload(name):
    w = synth.workload(name)
    cfg = bench.workload_config(w, {"extra": 1})
    assert cfg["workload"] == name and cfg["extra"] == 1
    assert cfg["parallelism"] == "replicas"
    if w.backward:
        assert "backward" in cfg["step"]
    if w.conv_taps:
        assert cfg["conv_taps"] == w.conv_taps
    if w.decode_steps:
        assert cfg["decode_steps"] == w.decode_steps and "T" not in cfg


def test_recorded_traffic_is_dropped_when_sources_change(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    h = hashlib.sha256()
    h.update(b"k.cu")
    h.update(b"kernel v1")
    rec = {"workloads": {"wl": {"kernel": "kern", "dram_bytes_per_launch": 123, "sources": ["k.cu"],
                                "sources_sha256": h.hexdigest()}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("wl", "kern") == 123
    assert bench.recorded_traffic("wl", "other_kernel") is None
    assert bench.recorded_traffic("other_workload", "kern") is None
    src.write_text("kernel v2")
    assert bench.recorded_traffic("wl", "kern") is None
