"""bench.py's algorithmic bytes (the numerator of every GB/s and roofline
fraction it reports) against the sizes of the arrays each operator must read
and write once, built here as numpy arrays of the right dtypes and shapes;
and the DeepSeek-V3 totals quoted with the results (21,643 (token, rank)
pairs and 32,768 valid entries)."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _arrays(T, H, E, R, K, n_pairs, n_valid):
    bf16, i32, f32, u8 = np.uint16, np.int32, np.float32, np.uint8
    return {
        "x": np.empty((T, H), bf16),
        "recv_rows": np.empty((n_pairs, H), bf16),          # only the rows the layout uses
        "recv_q": np.empty((n_pairs, H), u8),
        "recv_scales_fp8": np.empty((n_pairs, H // 128), f32),
        "recv_scales_mx": np.empty((n_pairs, H // 32), u8),
        "recv_slot": np.empty((T, R), i32),
        "y_rows": np.empty((n_valid, H), bf16),
        "out": np.empty((T, H), bf16),
        "expert_slot": np.empty((T, K), i32),
        "topk_w": np.empty((T, K), f32),
        "grad_w": np.empty((T, K), f32),
    }


@pytest.mark.parametrize("T,H,E,R,K,n_pairs,n_valid", [
    (4096, 7168, 256, 8, 8, 21643, 32768),
    (300, 256, 32, 8, 6, 1100, 1720),
    (16384, 2048, 64, 32, 6, 94369, 98304),
])
def test_bytes_are_the_arrays_read_and_written_once(T, H, E, R, K, n_pairs, n_valid):
    a = _arrays(T, H, E, R, K, n_pairs, n_valid)
    nb = lambda *names: sum(a[n].nbytes for n in names)
    ab = bench.algorithmic_bytes(T, H, E, R, K, n_pairs, n_valid, T * min(K, R))
    assert ab["dispatch"] == nb("x", "recv_rows", "recv_slot")
    assert ab["dispatch_fp8"] == nb("x", "recv_q", "recv_scales_fp8", "recv_slot")
    assert ab["dispatch_mxfp8"] == nb("x", "recv_q", "recv_scales_mx", "recv_slot")
    assert ab["combine"] == nb("y_rows", "out", "expert_slot", "topk_w")
    assert ab["dispatch_backward"] == nb("recv_rows", "x", "recv_slot")          # grad_recv in, grad_x out
    assert ab["combine_backward"] == nb("out", "y_rows", "y_rows", "expert_slot", "topk_w", "grad_w")
    # (grad_out in, y rows in, grad_y rows out, slots, weights, weight gradients out)


def test_deepseek_v3_totals():
    ab = bench.algorithmic_bytes(4096, 7168, 256, 8, 8, 21643, 32768, 32768)
    assert ab["dispatch"] == 369_125_376
    assert ab["combine"] == 528_744_448
    assert ab["dispatch_fp8"] == ab["dispatch_mxfp8"] == 218_836_384


def test_reference_arm_config_equals_the_gpu_arms():
    """The reference (CPU oracle) arm reports the same `config` object as the
    GPU arm when its per-step sample is the whole workload: built by the same
    function from the same pair count and capacity."""
    import argparse
    import oracle
    from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs
    wl = WORKLOADS["tiny"]
    ref = bench.run_reference(argparse.Namespace(workload="tiny", steps=3, warmup=3, gpus=1))
    inp = make_inputs(wl)
    L = oracle.layout(inp.topk_idx.numpy(), inp.topk_w.numpy(), wl.E, wl.R)
    assert ref["config"] == bench.step_config(wl, 0, L.n_pairs, L.capacity, 1)
    assert ref["config"]["T"] == wl.T and "first" not in ref["config"]["workload"]
    assert not ref["cpu_baseline"]["host_cpu"].startswith("0x")


def test_config_names_a_partial_sample():
    from combine_moe_dispatch_02_gb300.inputs import WORKLOADS
    wl = WORKLOADS["dsv3"]
    cfg = bench.step_config(wl, 0, 100, 800, 1, T_sample=100)
    assert "first 100 of 4096 tokens" in cfg["workload"] and cfg["T"] == 100
    assert bench.step_config(wl, 1, 21643, 32768, 1)["step"].startswith("layout + FP8")
