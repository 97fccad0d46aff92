"""The no-allocation entry point (frn_unfused_reduce_rmsnorm_noalloc) against
the existing entry point with a caller-provided workspace.

It is meant for callers that cannot allocate device memory on the call path
(CUDA-graph capture in the default mode, engines that pre-reserve their memory,
plugins without an allocator), so its scratch is a fixed array in the library.
Two calls in a row, on different inputs, must both match the workspace path
(and hence the oracle rules), whatever the array held before; the largest size
the array holds runs and one row more is refused; a small case is compared
with the oracle itself; and the binding refuses malformed outputs before the
library is reached.  This file is collected last on purpose."""
import os

import pytest
import torch

import oracle
import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import DevInputs, assert_quant_close, assert_residual_exact, assert_y_close, host_bits

pytestmark = pytest.mark.gpu


def _outputs(T, H, quant, emit_y):
    ro = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda") if emit_y else None
    q = torch.empty((T, H), dtype=torch.float8_e4m3fn, device="cuda") if quant else None
    s = torch.empty((T, H // 128), dtype=torch.float32, device="cuda") if quant else None
    return ro, y, q, s


@pytest.mark.parametrize("stages,quant,emit_y", [(3, True, False), (3, True, True), (2, True, False),
                                                 (2, False, True)])
def test_noalloc_matches_workspace_path_twice(stages, quant, emit_y):
    R, T, H = 8, 64, 7168
    for call, seed in enumerate((501, 502)):      # two calls in a row, different inputs
        inp = syn.make_inputs(R, T, H, seed=seed + stages, partial_std=0.5)
        d = DevInputs(inp)
        ro, y, q, s = _outputs(T, H, quant, emit_y)
        frn.unfused_reduce_rmsnorm_noalloc(d.partials, d.residual, d.gamma, inp.eps, stages=stages,
                                           residual_out=ro, y=y, q=q, scales=s)
        if quant:
            (yref, qref, sref), roref = frn.unfused_reduce_rmsnorm(
                d.partials, d.residual, d.gamma, inp.eps, stages=stages, quant=True, emit_bf16=True)
            torch.cuda.synchronize()
            assert_residual_exact(host_bits(ro), host_bits(roref), f"call {call}")
            if emit_y:
                assert_y_close(host_bits(y), host_bits(yref), f"call {call}")
            assert_quant_close(host_bits(y if emit_y else yref), host_bits(q), host_bits(s), host_bits(yref),
                               host_bits(qref), host_bits(sref), f"call {call}")
        else:
            yref, roref = frn.unfused_reduce_rmsnorm(d.partials, d.residual, d.gamma, inp.eps, stages=stages)
            torch.cuda.synchronize()
            assert_residual_exact(host_bits(ro), host_bits(roref), f"call {call}")
            assert_y_close(host_bits(y), host_bits(yref), f"call {call}")


def test_noalloc_refuses_oversized_scratch():
    T, H = 512, 7168      # 3 stages, quant, no y: 6*T*H bytes > 16 MiB
    assert frn.unfused_workspace_bytes(T, H, 3, True, False) > frn.STATIC_WORKSPACE_BYTES
    inp = syn.make_inputs(2, T, H, seed=503)
    d = DevInputs(inp)
    ro, _, q, s = _outputs(T, H, True, False)
    with pytest.raises(frn.FrnError) as e:
        frn.unfused_reduce_rmsnorm_noalloc(d.partials, d.residual, d.gamma, inp.eps, stages=3, residual_out=ro,
                                           q=q, scales=s)
    assert e.value.status == frn.FRN_ERR_UNSUPPORTED
    assert "static workspace" in e.value.detail


def test_noalloc_size_limit_edge():
    """The largest call the array holds (3 stages, quant, no y, H = 7168:
    6 * T * H bytes of scratch, T = 390) runs and matches the workspace path;
    one more row (T = 391) is refused before anything is launched."""
    R, H = 2, 7168
    assert frn.unfused_workspace_bytes(390, H, 3, True, False) <= frn.STATIC_WORKSPACE_BYTES
    assert frn.unfused_workspace_bytes(391, H, 3, True, False) > frn.STATIC_WORKSPACE_BYTES
    inp = syn.make_inputs(R, 391, H, seed=504, partial_std=0.5)
    d = DevInputs(inp)
    ro, _, q, s = _outputs(390, H, True, False)
    first = [d.partials[r, :390] for r in range(R)]      # the first 390 rows of each partial
    frn.unfused_reduce_rmsnorm_noalloc(first, d.residual[:390], d.gamma, inp.eps, stages=3,
                                       residual_out=ro, q=q, scales=s)
    (yref, qref, sref), roref = frn.unfused_reduce_rmsnorm(first, d.residual[:390], d.gamma, inp.eps, stages=3,
                                                           quant=True, emit_bf16=True)
    torch.cuda.synchronize()
    assert_residual_exact(host_bits(ro), host_bits(roref), "T=390")
    assert_quant_close(host_bits(yref), host_bits(q), host_bits(s), host_bits(yref), host_bits(qref),
                       host_bits(sref), "T=390")
    ro, _, q, s = _outputs(391, H, True, False)
    with pytest.raises(frn.FrnError) as e:
        frn.unfused_reduce_rmsnorm_noalloc(d.partials, d.residual, d.gamma, inp.eps, stages=3, residual_out=ro,
                                           q=q, scales=s)
    assert e.value.status == frn.FRN_ERR_UNSUPPORTED


@pytest.mark.parametrize("stages,emit_y", [(3, False), (2, True)])
def test_noalloc_against_oracle(stages, emit_y):
    """A small quant case straight against the CPU oracle."""
    R, T, H = 4, 32, 4096
    inp = syn.make_inputs(R, T, H, seed=505 + stages, partial_std=0.5)
    d = DevInputs(inp)
    ro, y, q, s = _outputs(T, H, True, emit_y)
    frn.unfused_reduce_rmsnorm_noalloc(d.partials, d.residual, d.gamma, inp.eps, stages=stages, residual_out=ro,
                                       y=y, q=q, scales=s)
    torch.cuda.synchronize()
    rro, ry, rq, rs = oracle.Oracle().reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps, 128,
                                                           threads=max(1, os.cpu_count() or 1))
    assert_residual_exact(host_bits(ro), rro, "noalloc vs oracle")
    if emit_y:
        assert_y_close(host_bits(y), ry, "noalloc vs oracle")
    assert_quant_close(host_bits(y) if emit_y else None, host_bits(q), host_bits(s), ry, rq, rs,
                       "noalloc vs oracle")


def test_noalloc_checks_outputs_before_launch(monkeypatch):
    """The C side sees only pointers: a wrongly shaped or typed output is refused
    by the binding, and the library is never called."""
    R, T, H = 2, 8, 1024
    inp = syn.make_inputs(R, T, H, seed=507)
    d = DevInputs(inp)
    calls = []
    lib = frn.library()
    host_only = {"frn_unfused_workspace_bytes", "frn_status_string", "frn_last_error_detail"}

    class Spy:
        """Passes host-only queries through; any other entry point is a failure."""
        def __getattr__(self, name):
            if name in host_only:
                return getattr(lib, name)
            calls.append(name)
            raise AssertionError(f"library reached: {name}")
    monkeypatch.setattr(frn, "_lib", Spy())
    ro, y, q, s = _outputs(T, H, True, True)
    wide = torch.empty((T, 2 * H), dtype=torch.bfloat16, device="cuda")
    bad = [dict(residual_out=ro[:-1], y=y, q=q, scales=s),
           dict(residual_out=ro, y=y.float(), q=q, scales=s),
           dict(residual_out=ro, y=y, q=q[:, :-16], scales=s),
           dict(residual_out=ro, y=y, q=q, scales=s[:, :-1]),
           dict(residual_out=ro, y=y, q=q, scales=s.double()),
           dict(residual_out=wide[:, :H], y=y, q=q, scales=s),          # right shape, not contiguous
           dict(residual_out=ro, y=y, q=q.view(torch.int8), scales=s)]
    for kw in bad:
        with pytest.raises((ValueError, TypeError)):
            frn.unfused_reduce_rmsnorm_noalloc(d.partials, d.residual, d.gamma, inp.eps, stages=3, **kw)
        with pytest.raises((ValueError, TypeError)):
            frn.unfused_reduce_rmsnorm(d.partials, d.residual, d.gamma, inp.eps, stages=3, quant=True, **kw)
    with pytest.raises(ValueError):      # q without scales
        frn.unfused_reduce_rmsnorm_noalloc(d.partials, d.residual, d.gamma, inp.eps, stages=3, residual_out=ro,
                                           q=q)
    with pytest.raises(ValueError):      # gamma of the wrong length
        frn.unfused_reduce_rmsnorm_noalloc(d.partials, d.residual, d.gamma[:-8], inp.eps, stages=3,
                                           residual_out=ro, q=q, scales=s)
    assert calls == []
