"""The no-allocation entry point (frn_unfused_reduce_rmsnorm_noalloc) against
the existing entry point with a caller-provided workspace.

It is meant for callers that cannot allocate device memory on the call path
(CUDA-graph capture in the default mode, engines that pre-reserve their memory,
plugins without an allocator), so its scratch is a fixed array in the library.
Two calls in a row, on different inputs, must both match the workspace path
(and hence the oracle rules), whatever the array held before; sizes beyond the
array are refused.  This file is collected last on purpose."""
import pytest
import torch

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
