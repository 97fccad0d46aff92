"""Device-side failure detection, without a GPU fault.

Every wait on the stream kernel's shared-memory pipeline, and the row kernel's
wait for the tile sums its cluster pushes, is bounded.  The test hook makes the
stream kernel's CTAs skip their first bulk copy, and the cluster row kernel
never push tile 0's sum -- barriers that nothing will complete -- with a 50 ms
bound: the kernel must come back on its own, report FRN_ERR_TIMEOUT through the
device status word, and leave the context usable (a normal call afterwards
matches the oracle).
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import assert_residual_exact, assert_y_close, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("groups", [0, 1])
def test_stalled_copy_times_out_and_context_survives(groups):
    inp = syn.make_inputs(2, 400, 4096, seed=80)
    p, r, g = dev_bf16(inp.partials), dev_bf16(inp.residual), dev_bf16(inp.gamma)
    assert frn.device_status(clear=True) in (frn.FRN_OK, frn.FRN_ERR_TIMEOUT)
    frn.set_kernel(frn.KERNEL_STREAM)
    frn.set_stream_groups(groups)
    try:
        frn.set_test_hooks(inject_stall=True, wait_limit_ns=50_000_000)
        frn.fused_reduce_rmsnorm(p, r, g, inp.eps)
        torch.cuda.synchronize()
        assert frn.device_status(clear=True) == frn.FRN_ERR_TIMEOUT
        assert frn.device_status() == frn.FRN_OK      # cleared
    finally:
        frn.set_test_hooks(False, 0)
    try:
        y, ro = frn.fused_reduce_rmsnorm(p, r, g, inp.eps)
        torch.cuda.synchronize()
    finally:
        frn.set_kernel(frn.KERNEL_AUTO)
        frn.set_stream_groups(0)
    assert frn.device_status() == frn.FRN_OK
    rro, ry = oracle.Oracle().reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, inp.eps)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)


@pytest.mark.parametrize("ctas", [2, 4])
def test_missing_cluster_push_times_out_and_context_survives(ctas):
    inp = syn.make_inputs(8, 6, 7168, seed=82, partial_std=0.5)
    p, r, g = dev_bf16(inp.partials), dev_bf16(inp.residual), dev_bf16(inp.gamma)
    assert frn.device_status(clear=True) in (frn.FRN_OK, frn.FRN_ERR_TIMEOUT)
    frn.set_kernel(frn.KERNEL_ROWS)
    frn.set_ctas_per_row(ctas)
    try:
        assert frn.query_launch(6, 7168, 8)[1] == ctas
        frn.set_test_hooks(inject_stall=True, wait_limit_ns=50_000_000)
        frn.fused_reduce_rmsnorm(p, r, g, inp.eps)
        torch.cuda.synchronize()
        assert frn.device_status(clear=True) == frn.FRN_ERR_TIMEOUT
        assert frn.device_status() == frn.FRN_OK
    finally:
        frn.set_test_hooks(False, 0)
    try:
        y, ro = frn.fused_reduce_rmsnorm(p, r, g, inp.eps)
        torch.cuda.synchronize()
    finally:
        frn.set_kernel(frn.KERNEL_AUTO)
        frn.set_ctas_per_row(0)
    assert frn.device_status() == frn.FRN_OK
    rro, ry = oracle.Oracle().reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, inp.eps)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)


def test_normal_calls_leave_status_clear():
    frn.device_status(clear=True)
    inp = syn.make_inputs(8, 512, 7168, seed=81, partial_std=0.5)
    frn.set_kernel(frn.KERNEL_STREAM)
    try:
        for _ in range(3):
            frn.fused_reduce_rmsnorm_quant_per_group(dev_bf16(inp.partials), dev_bf16(inp.residual),
                                                     dev_bf16(inp.gamma), inp.eps, 128, True)
        torch.cuda.synchronize()
    finally:
        frn.set_kernel(frn.KERNEL_AUTO)
    assert frn.device_status() == frn.FRN_OK
