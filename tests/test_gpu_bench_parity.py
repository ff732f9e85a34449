"""Parity in the launch configuration the benchmark times.

bench.py times back-to-back gemm_run_ex launches:
- with GP_RUN_B_CONSTANT (and GP_RUN_INDEPENDENT for the weight-streaming
  runs);
- replayed from a CUDA graph;
- over rotating copies of A and packed B.
These tests drive that same code path (bench.Problem and bench.time_device)
on every workload at its full size, into outputs filled with a sentinel
first. They then check every output of every buffer it wrote against the
oracle.
"""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
import dense_gemm_preshuffle_gb300 as gp
from dense_gemm_preshuffle_gb300 import inputs

pytestmark = pytest.mark.gpu

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

TOL = 8e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_preshuffle_gb300 import build
    build.build()
    gp.load_library()


def fill_sentinel(prob):
    """NaN (float outputs) or INT32_MIN (int32 outputs, which no exact INT8
    or W4A8 result reaches): an output the timed launches never write fails
    the comparison."""
    for C in prob.C:
        if C.dtype == torch.int32:
            C.fill_(-2 ** 31)
        else:
            C.fill_(float("nan"))


def reference(ops):
    if ops.dtype in ("int8", "w4a8") or ops.M * ops.N * ops.K <= (1 << 31):
        return oracle.gemm_operands(ops)
    return oracle.gemm_dequantized(ops)  # the same values at full size


def check_outputs(prob, ops):
    """Every output of every buffer the timed launches wrote."""
    ref = reference(ops)
    for C in prob.C:
        if C.dtype == torch.int32:
            c = C.cpu().numpy().astype(np.int64)
            assert np.array_equal(c, ref), f"{int((c != ref).sum())} mismatching int32 outputs"
        else:
            c = C.float().cpu().numpy().astype(np.float64)
            err = oracle.max_rel_err(c, ref)
            assert err <= TOL, f"max rel err {err:.3e}"


@pytest.mark.parametrize("name", list(inputs.ALL_WORKLOADS))
def test_bench_launch_configuration_matches_oracle(name):
    dev = torch.device("cuda", 0)
    prob = bench.Problem(name, dev)
    fill_sentinel(prob)
    steps = 2 * len(prob.C) + 3  # every output buffer is written, some twice
    bench.time_device(prob, steps, 3, None, dev)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    ops = inputs.workload_operands(name)
    check_outputs(prob, ops)


@pytest.mark.parametrize("name", ["int8_16x7168x4096", "w4a8_16x7168x4096"])
def test_bench_independent_runs_match_oracle(name):
    dev = torch.device("cuda", 0)
    prob = bench.Problem(name, dev)
    prob.flags = gp.GP_RUN_B_CONSTANT | gp.GP_RUN_INDEPENDENT
    fill_sentinel(prob)
    bench.time_device(prob, 2 * len(prob.C) + 3, 3, None, dev)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    ops = inputs.workload_operands(name)
    check_outputs(prob, ops)


@pytest.mark.parametrize("name", ["int8_16x7168x4096", "fp8_128x256x512"])
def test_bench_end_to_end_leg_matches_oracle(name):
    """The end-to-end leg: host A (and its scales) copied in, gemm_run_ex, C
    copied out, every step, over the leg's concurrent streams.  Every step
    computes the same product, so every device output buffer and every host
    copy must equal the oracle's."""
    dev = torch.device("cuda", 0)
    prob = bench.Problem(name, dev)
    fill_sentinel(prob)
    rec = {}
    steps = 4 * bench.E2E_STREAMS
    bench.time_e2e(prob, steps, 3, dev, record=rec)
    torch.cuda.synchronize()
    assert gp.gemm_last_device_status() == 0
    ops = inputs.workload_operands(name)
    ref = oracle.gemm_operands(ops)
    written = rec["C"][:steps]  # step i writes buffer i mod len(C)
    outs = [c.cpu() for c in written] + list(rec["host_C"])
    assert len(rec["host_C"]) == bench.E2E_STREAMS
    for c in outs:
        if c.dtype == torch.int32:
            assert np.array_equal(c.numpy().astype(np.int64), ref)
        else:
            assert oracle.max_rel_err(c.float().numpy().astype(np.float64), ref) <= TOL
