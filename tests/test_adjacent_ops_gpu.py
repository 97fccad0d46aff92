"""The adjacent layer steps exposed on the same kernels: fused residual add +
RMSNorm of one activation (R = 1) and a plain RMSNorm, against the oracle,
under both kernels."""
import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import assert_residual_exact, assert_y_close, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[frn.KERNEL_ROWS, frn.KERNEL_STREAM], ids=["rows", "stream"])
def kernel(request):
    frn.set_kernel(request.param)
    yield request.param
    frn.set_kernel(frn.KERNEL_AUTO)


@pytest.mark.parametrize("T,H", [(1, 8), (7, 1000), (64, 7168), (300, 4096), (5, 16384)])
def test_fused_add_rmsnorm(T, H, kernel):
    inp = syn.make_inputs(1, T, H, seed=T + H)
    x, r, g = dev_bf16(inp.partials[0]), dev_bf16(inp.residual), dev_bf16(inp.gamma)
    y, ro = frn.fused_add_rmsnorm(x, r, g, inp.eps)
    rro, ry = oracle.Oracle().reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, inp.eps)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)


@pytest.mark.parametrize("T,H", [(1, 8), (7, 1000), (64, 7168), (300, 4096), (5, 16384)])
def test_rmsnorm(T, H, kernel):
    inp = syn.make_inputs(1, T, H, seed=2 * T + H)
    x, g = dev_bf16(inp.partials[0]), dev_bf16(inp.gamma)
    y = frn.rmsnorm(x, g, inp.eps)
    _, ry = oracle.Oracle().reduce_rmsnorm(inp.partials, None, inp.gamma, inp.eps)
    assert_y_close(host_bits(y), ry)
    # torch's own rms_norm in fp32 on the same input: within one bf16 ulp too
    ref = torch.nn.functional.rms_norm(x.float(), (H,), weight=g.float(), eps=inp.eps).to(torch.bfloat16)
    assert_y_close(host_bits(y), host_bits(ref))


def test_rmsnorm_writes_only_y():
    inp = syn.make_inputs(1, 9, 2048, seed=5)
    x, g = dev_bf16(inp.partials[0]), dev_bf16(inp.gamma)
    x_before = x.clone()
    y = frn.rmsnorm(x, g, inp.eps)
    torch.cuda.synchronize()
    assert torch.equal(x.view(torch.int16), x_before.view(torch.int16))
    assert y.shape == x.shape
