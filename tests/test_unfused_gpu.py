"""The unfused comparison paths (3 kernels: reduce -> add + RMSNorm -> quant;
2 kernels: fused reduce + RMSNorm -> stand-alone quant, or reduce -> add +
RMSNorm without quant): each is compared with the oracle element by element,
with and without a residual, at a decode shape and at the prefill chunk, and
with the fused entry points bit for bit."""
import os

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


THREADS = max(1, os.cpu_count() or 1)
_CACHE = {}


def _workload(name, with_residual):
    """Decode (R=8, T=64, H=7168) or prefill (R=2, T=8192, H=7168, 1% outlier
    channels) inputs, on the host and the device, and the oracle's outputs."""
    key = (name, with_residual)
    if key not in _CACHE:
        if name == "decode":
            inp = syn.make_inputs(8, 64, 7168, seed=94, partial_std=0.5, with_residual=with_residual)
        else:
            inp = syn.make_inputs(2, 8192, 7168, seed=95, outlier_frac=0.01, with_residual=with_residual)
        ref = oracle.Oracle().reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps, 128,
                                                   threads=THREADS)
        _CACHE[key] = (inp, DevInputs(inp), ref)
    return _CACHE[key]


@pytest.mark.parametrize("with_residual", [True, False], ids=["residual", "no_residual"])
@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_two_stage_norm_against_oracle(name, with_residual):
    """reduce -> residual add + RMSNorm, element by element against the oracle."""
    inp, d, (rro, ry, _, _) = _workload(name, with_residual)
    y, ro = frn.unfused_reduce_rmsnorm(d.partials, d.residual, d.gamma, inp.eps, stages=2)
    assert_residual_exact(host_bits(ro), rro, f"2-stage norm {name}")
    assert_y_close(host_bits(y), ry, f"2-stage norm {name}")


@pytest.mark.parametrize("with_residual", [True, False], ids=["residual", "no_residual"])
@pytest.mark.parametrize("name", ["decode", "prefill"])
@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("emit", [True, False], ids=["B", "A"])
def test_quant_paths_against_oracle(name, with_residual, stages, emit):
    """2 kernels (fused reduce + RMSNorm -> stand-alone per-group quant) and 3
    kernels (reduce -> add + RMSNorm -> quant), both output variants, element by
    element against the oracle."""
    inp, d, (rro, ry, rq, rs) = _workload(name, with_residual)
    out, ro = frn.unfused_reduce_rmsnorm(d.partials, d.residual, d.gamma, inp.eps, stages=stages, quant=True,
                                         emit_bf16=emit)
    what = f"{stages}-stage quant {'B' if emit else 'A'} {name}"
    assert_residual_exact(host_bits(ro), rro, what)
    y = host_bits(out[0]) if emit else None
    if emit:
        assert_y_close(y, ry, what)
    assert_quant_close(y, host_bits(out[-2]), host_bits(out[-1]), ry, rq, rs, what)


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
