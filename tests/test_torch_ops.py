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


# ----------------------------------------------------- ops vs the oracle --

def _op_inputs(R, T, H, with_residual, seed):
    from frn_testlib import dev_bf16
    inp = syn.make_inputs(R, T, H, seed=seed, partial_std=0.5, with_residual=with_residual)
    parts = [dev_bf16(inp.partials[r]) for r in range(R)]
    res = dev_bf16(inp.residual) if with_residual else None
    return inp, parts, res, dev_bf16(inp.gamma)


def _call(fn, compiled):
    return torch.compile(fn, fullgraph=True)() if compiled else fn()


@pytest.mark.gpu
@pytest.mark.parametrize("compiled", [False, True], ids=["eager", "compiled"])
@pytest.mark.parametrize("with_residual", [True, False], ids=["residual", "no_residual"])
@pytest.mark.parametrize("R,T,H", [(8, 64, 7168), (4, 32, 4096)])
def test_ops_against_oracle(R, T, H, with_residual, compiled):
    """Every torch.ops.frn.* output, eager and under torch.compile, element by
    element against the oracle under the matching rules."""
    import oracle
    from frn_testlib import (assert_mx_close, assert_quant_close, assert_residual_exact, assert_y_close,
                             host_bits)
    inp, parts, res, g = _op_inputs(R, T, H, with_residual, seed=R * 100 + T)
    orc = oracle.Oracle()
    rro, ry, rq, rs = orc.reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps, 128)
    _, _, rq4, re8 = orc.reduce_rmsnorm_mxfp4(inp.partials, inp.residual, inp.gamma, inp.eps)
    eps = inp.eps
    what = f"R={R} T={T} H={H} residual={with_residual} compiled={compiled}"

    y, ro = _call(lambda: torch.ops.frn.fused_reduce_rmsnorm(parts, res, g, eps), compiled)
    assert_residual_exact(host_bits(ro), rro, what)
    assert_y_close(host_bits(y), ry, what)
    y_lib = host_bits(y)     # the library's y: the MXFP4 variant without y quantises these bits
    for emit in (False, True):
        y, q, s, ro = _call(lambda: torch.ops.frn.fused_reduce_rmsnorm_quant_per_group(parts, res, g, eps, 128, emit),
                            compiled)
        assert_residual_exact(host_bits(ro), rro, what)
        yb = host_bits(y) if emit else None
        if emit:
            assert_y_close(yb, ry, what)
        else:
            assert y.shape == (0, H)
        assert_quant_close(yb, host_bits(q), host_bits(s), ry, rq, rs, what + f" fp8 emit={emit}")
        y, q4, e8, ro = _call(lambda: torch.ops.frn.fused_reduce_rmsnorm_mxfp4(parts, res, g, eps, emit), compiled)
        assert_residual_exact(host_bits(ro), rro, what)
        if emit:
            assert_y_close(host_bits(y), ry, what)
        if emit:
            assert np.array_equal(host_bits(y), y_lib), what
        assert_mx_close(y_lib, host_bits(q4), host_bits(e8), ry, rq4, re8, what + f" mxfp4 emit={emit}")
    # the adjacent ops: one activation plus the residual, and a plain RMSNorm
    one = syn.Inputs(inp.partials[:1], inp.residual, inp.gamma, eps)
    aro, ay = orc.reduce_rmsnorm(one.partials, one.residual, one.gamma, eps)
    y, ro = _call(lambda: torch.ops.frn.fused_add_rmsnorm(parts[0], res, g, eps), compiled)
    assert_residual_exact(host_bits(ro), aro, what + " fused_add_rmsnorm")
    assert_y_close(host_bits(y), ay, what + " fused_add_rmsnorm")
    _, ny = orc.reduce_rmsnorm(inp.partials[:1], None, inp.gamma, eps)
    y = _call(lambda: torch.ops.frn.rmsnorm(parts[0], g, eps), compiled)
    assert_y_close(host_bits(y), ny, what + " rmsnorm")
