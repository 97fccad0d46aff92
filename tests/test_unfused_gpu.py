"""The unfused comparison paths (3 kernels: reduce -> add + RMSNorm -> quant;
2 kernels: fused reduce + RMSNorm -> stand-alone quant, or reduce -> add +
RMSNorm without quant) return the same bits as the fused entry points, and
therefore match the oracle under the same rules."""
import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import DevInputs, assert_quant_close, assert_residual_exact, assert_y_close, gpu_norm, gpu_quant, \
    host_bits

pytestmark = pytest.mark.gpu

SHAPES = [(8, 64, 7168), (2, 300, 4096), (4, 32, 4096), (3, 17, 1024), (16, 5, 16384), (1, 9, 128)]


@pytest.mark.parametrize("R,T,H", SHAPES)
def test_unfused_norm_matches_fused(R, T, H):
    inp = syn.make_inputs(R, T, H, seed=90 + T, partial_std=0.5)
    d = DevInputs(inp)
    ro, y = gpu_norm(d)
    y2, ro2 = frn.unfused_reduce_rmsnorm(d.partials, d.residual, d.gamma, inp.eps, stages=2)
    assert np.array_equal(host_bits(ro2), ro) and np.array_equal(host_bits(y2), y)


@pytest.mark.parametrize("R,T,H", SHAPES)
@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("emit", [True, False])
def test_unfused_quant_matches_fused(R, T, H, stages, emit):
    inp = syn.make_inputs(R, T, H, seed=91 + T, partial_std=0.5)
    d = DevInputs(inp)
    base = gpu_quant(d, True)
    out, ro = frn.unfused_reduce_rmsnorm(d.partials, d.residual, d.gamma, inp.eps, stages=stages, quant=True,
                                         emit_bf16=emit)
    got_q, got_s = host_bits(out[-2]), host_bits(out[-1])
    assert np.array_equal(host_bits(ro), base[0])
    if emit:
        assert np.array_equal(host_bits(out[0]), base[1])
    assert np.array_equal(got_q, base[2]) and np.array_equal(got_s.view(np.uint32), base[3].view(np.uint32))


def test_unfused_against_oracle_no_residual():
    inp = syn.make_inputs(4, 40, 4096, seed=92, with_residual=False)
    d = DevInputs(inp)
    (y, q, s), ro = frn.unfused_reduce_rmsnorm(d.partials, None, d.gamma, inp.eps, stages=3, quant=True)
    rro, ry, rq, rs = oracle.Oracle().reduce_rmsnorm_quant(inp.partials, None, inp.gamma, inp.eps)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)
    assert_quant_close(host_bits(y), host_bits(q), host_bits(s), ry, rq, rs)


def test_workspace_checks():
    inp = syn.make_inputs(2, 8, 1024, seed=93)
    d = DevInputs(inp)
    need = frn.unfused_workspace_bytes(8, 1024, 3, True, False)
    assert need == 4 * 8 * 1024 + 2 * 8 * 1024
    assert frn.unfused_workspace_bytes(8, 1024, 3, False, True) == -1
    small = torch.empty((need - 16,), dtype=torch.uint8, device="cuda")
    with pytest.raises(frn.FrnError) as e:
        frn.unfused_reduce_rmsnorm(d.partials, d.residual, d.gamma, inp.eps, stages=3, quant=True, emit_bf16=False,
                                   workspace=small)
    assert e.value.status == frn.FRN_ERR_INVALID_ARG
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    with pytest.raises(frn.FrnError) as e:   # workspace aliasing an output
        frn.unfused_reduce_rmsnorm(d.partials, d.residual, d.gamma, inp.eps, stages=3, quant=True, emit_bf16=False,
                                   workspace=ws, residual_out=ws[:2 * 8 * 1024].view(torch.bfloat16).view(8, 1024))
    assert e.value.status == frn.FRN_ERR_INVALID_ARG
