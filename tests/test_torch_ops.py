"""The torch custom ops: registered with fake implementations that give the
right shapes and dtypes without a GPU (CPU test), and on the GPU the same bits
as the plain binding, also inside torch.compile and a CUDA graph."""
import numpy as np
import pytest
import torch
from torch._subclasses.fake_tensor import FakeTensorMode

import reduce_residual_rmsnorm_fp32_gb300.torch_ops  # noqa: F401  (registers torch.ops.frn.*)
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn


def test_fake_impls_give_shapes_without_a_gpu():
    with FakeTensorMode():
        parts = [torch.empty((5, 256), dtype=torch.bfloat16) for _ in range(3)]
        res = torch.empty((5, 256), dtype=torch.bfloat16)
        g = torch.empty((256,), dtype=torch.bfloat16)
        y, ro = torch.ops.frn.fused_reduce_rmsnorm(parts, res, g, 1e-6)
        assert y.shape == (5, 256) and ro.dtype == torch.bfloat16
        y, q, s, ro = torch.ops.frn.fused_reduce_rmsnorm_quant_per_group(parts, None, g, 1e-6, 128, False)
        assert y.shape == (0, 256) and q.dtype == torch.float8_e4m3fn and s.shape == (5, 2)
        y, q, s, ro = torch.ops.frn.fused_reduce_rmsnorm_quant_per_group(parts, res, g, 1e-6, 128, True)
        assert y.shape == (5, 256)
        y, q, s, ro = torch.ops.frn.fused_reduce_rmsnorm_mxfp4(parts, res, g, 1e-6, False)
        assert y.shape == (0, 256) and q.shape == (5, 128) and q.dtype == torch.uint8 and s.shape == (5, 8)
        y, ro = torch.ops.frn.fused_add_rmsnorm(parts[0], res, g, 1e-6)
        assert y.shape == (5, 256) and ro.shape == (5, 256)
        assert torch.ops.frn.rmsnorm(parts[0], g, 1e-6).shape == (5, 256)


@pytest.mark.gpu
def test_ops_match_binding_in_compile_and_graph():
    import reduce_residual_rmsnorm_fp32_gb300 as frn
    from frn_testlib import dev_bf16
    inp = syn.make_inputs(4, 32, 4096, seed=3, partial_std=0.5)
    parts = [dev_bf16(inp.partials[r]) for r in range(4)]
    res, g = dev_bf16(inp.residual), dev_bf16(inp.gamma)
    (yb, qb, sb), rob = frn.fused_reduce_rmsnorm_quant_per_group(parts, res, g, inp.eps, 128, True)

    def f(ps, r, gg):
        return torch.ops.frn.fused_reduce_rmsnorm_quant_per_group(ps, r, gg, 1e-6, 128, True)

    y, q, s, ro = f(parts, res, g)
    for a, b in ((y, yb), (q, qb), (s, sb), (ro, rob)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    cf = torch.compile(f, fullgraph=True)
    y2, q2, s2, ro2 = cf(parts, res, g)
    assert torch.equal(q2.view(torch.uint8), qb.view(torch.uint8)) and torch.equal(ro2, rob)
    # inside a CUDA graph
    yg, rog = torch.ops.frn.fused_reduce_rmsnorm(parts, res, g, 1e-6)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        out = torch.ops.frn.fused_reduce_rmsnorm(parts, res, g, 1e-6)
    gr.replay()
    torch.cuda.synchronize()
    assert torch.equal(out[0], yg) and torch.equal(out[1], rog)


@pytest.mark.gpu
def test_mxfp4_and_adjacent_ops_match_binding():
    import reduce_residual_rmsnorm_fp32_gb300 as frn
    from frn_testlib import dev_bf16
    inp = syn.make_inputs(2, 16, 2048, seed=4, partial_std=0.5)
    parts = [dev_bf16(inp.partials[r]) for r in range(2)]
    res, g = dev_bf16(inp.residual), dev_bf16(inp.gamma)
    (yb, qb, sb), rob = frn.fused_reduce_rmsnorm_mxfp4(parts, res, g, inp.eps, True)
    y, q, s, ro = torch.compile(lambda ps, r, gg: torch.ops.frn.fused_reduce_rmsnorm_mxfp4(ps, r, gg, 1e-6, True),
                                fullgraph=True)(parts, res, g)
    assert torch.equal(y, yb) and torch.equal(q, qb) and torch.equal(s, sb) and torch.equal(ro, rob)
    ya, roa = frn.fused_add_rmsnorm(parts[0], res, g, inp.eps)
    y2, ro2 = torch.ops.frn.fused_add_rmsnorm(parts[0], res, g, 1e-6)
    assert torch.equal(y2, ya) and torch.equal(ro2, roa)
    assert torch.equal(torch.ops.frn.rmsnorm(parts[0], g, 1e-6), frn.rmsnorm(parts[0], g, inp.eps))
