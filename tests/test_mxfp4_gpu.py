"""MXFP4 output variant (OCP MX: 32-element blocks, E8M0 scale, E2M1 elements)
against the oracle, under both kernels and both output variants.

Matching rule: residual_out bit-exact, y within one bf16 ulp (off by one on
at most 0.1% of elements); every block's E8M0 code and E2M1 codes equal the
oracle's OCP MX quantisation of the library's own y, and the oracle's own codes
wherever the block's y equals the oracle's."""
import os

import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import DevInputs, assert_mx_close, assert_residual_exact, assert_y_close, host_bits

pytestmark = pytest.mark.gpu

THREADS = max(1, os.cpu_count() or 1)   # the oracle splits rows over the host's cores


def check_mx(inp, what):
    d = DevInputs(inp)
    (qa, sa), roa = frn.fused_reduce_rmsnorm_mxfp4(d.partials, d.residual, d.gamma, inp.eps)
    (y, qb, sb), rob = frn.fused_reduce_rmsnorm_mxfp4(d.partials, d.residual, d.gamma, inp.eps, emit_bf16=True)
    yn, ron = frn.fused_reduce_rmsnorm(d.partials, d.residual, d.gamma, inp.eps)
    torch.cuda.synchronize()
    assert torch.equal(qa, qb) and torch.equal(sa, sb) and torch.equal(roa, rob) and torch.equal(roa, ron)
    assert torch.equal(y, yn)
    ro, yb, q, s = host_bits(rob), host_bits(y), host_bits(qb), host_bits(sb)
    rro, ry, rq, rs = oracle.Oracle().reduce_rmsnorm_mxfp4(inp.partials, inp.residual, inp.gamma, inp.eps,
                                                           threads=THREADS)
    assert_residual_exact(ro, rro, what)
    assert_y_close(yb, ry, what)
    assert_mx_close(host_bits(y), host_bits(qa), host_bits(sa), ry, rq, rs, what + " (A)")
    return assert_mx_close(yb, q, s, ry, rq, rs, what + " (B)")


@pytest.fixture(params=[frn.KERNEL_ROWS, frn.KERNEL_STREAM], ids=["rows", "stream"])
def kernel(request):
    frn.set_kernel(request.param)
    yield request.param
    frn.set_kernel(frn.KERNEL_AUTO)


@pytest.mark.parametrize("R,T,H", [(2, 4, 256), (8, 64, 7168), (4, 32, 4096), (3, 17, 1024), (1, 5, 32),
                                   (16, 3, 16384), (2, 300, 7168), (2, 700, 256), (8, 650, 1024), (8, 586, 7168),
                                   (16, 600, 4096)])
def test_mxfp4_parity(R, T, H, kernel):
    check_mx(syn.make_inputs(R, T, H, seed=R + T + H, partial_std=0.5), f"mx R={R} T={T} H={H} k={kernel}")


def test_mxfp4_prefill_outliers():
    """Every one of the 8192 rows of the prefill chunk."""
    check_mx(syn.config_prefill(seed=4), "mx prefill")


@pytest.mark.parametrize("scale", [2.0 ** -100, 2.0 ** -30, 2.0 ** 40])
def test_mxfp4_magnitudes_and_zero_blocks(scale):
    inp = syn.make_inputs(3, 6, 1024, seed=9)
    f = syn.bf16_bits_to_f32(inp.partials) * np.float32(scale)
    r = syn.bf16_bits_to_f32(inp.residual) * np.float32(scale)
    p, res = syn.f32_to_bf16_bits(f), syn.f32_to_bf16_bits(r)
    p[:, 2, 64:96] = 0
    res[2, 64:96] = 0
    inp = syn.Inputs(p, res, inp.gamma, 1e-30)
    check_mx(inp, f"mx scale {scale}")
    d = DevInputs(inp)
    (q, s), _ = frn.fused_reduce_rmsnorm_mxfp4(d.partials, d.residual, d.gamma, inp.eps)
    assert host_bits(s)[2, 2] == 0 and np.all(host_bits(q)[2, 32:48] == 0)


def test_mxfp4_rejects_bad_h():
    inp = syn.make_inputs(2, 2, 136, seed=1)
    d = DevInputs(inp)
    with pytest.raises(ValueError):
        frn.fused_reduce_rmsnorm_mxfp4(d.partials, d.residual, d.gamma, inp.eps)


def test_mxfp4_subnormal_y(kernel):
    """gamma among the bf16 subnormals makes y subnormal: the shared exponent
    clamps at E8M0's -127 (scale code 0) and the elements are y * 2^127."""
    inp = syn.make_inputs(2, 9, 2048, seed=12)
    rng = np.random.default_rng(5)
    g = rng.integers(1, 0x80, size=2048).astype(np.uint16)   # 1..127 * 2^-133
    g[::7] |= 0x8000
    inp = syn.Inputs(inp.partials, inp.residual, g, inp.eps)
    check_mx(inp, f"mx subnormal y k={kernel}")
    d = DevInputs(inp)
    (q, s), _ = frn.fused_reduce_rmsnorm_mxfp4(d.partials, d.residual, d.gamma, inp.eps)
    assert np.all(host_bits(s) == 0)
