"""Bounds, poisoning and error handling on the GPU.

* Every output is surrounded by canary regions that must survive the call, and
  pre-filled with NaN / 0xFF so that an element the kernel forgets to write
  shows up as a mismatch (an uninitialised buffer is the accuracy bug that made
  the pages switch empty_like to zeros_like: "[AMD] Add AITER Custom
  All-Reduce", SGLang PR 13102, Modifications).
* Rejected arguments launch nothing (outputs stay poisoned) and leave the
  process usable.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import assert_quant_close, assert_residual_exact, assert_y_close, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

PAD = 4096  # bytes of canary on each side (keeps 16-byte alignment)


def guarded(shape, dtype, fill_byte):
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((PAD + n + PAD,), fill_byte, dtype=torch.uint8, device="cuda")
    view = raw[PAD:PAD + n].view(dtype).view(shape)
    return raw, view


def canaries_intact(raw, fill_byte):
    r = raw.cpu().numpy()
    return bool(np.all(r[:PAD] == fill_byte) and np.all(r[-PAD:] == fill_byte))


@pytest.mark.parametrize("R,T,H", [(8, 13, 7168), (2, 5, 4096), (3, 7, 1000), (1, 1, 8)])
def test_canaries_and_poison(R, T, H):
    inp = syn.make_inputs(R, T, H, seed=70)
    p, res, g = dev_bf16(inp.partials), dev_bf16(inp.residual), dev_bf16(inp.gamma)
    raw_ro, ro = guarded((T, H), torch.bfloat16, 0xFF)     # 0xFFFF bf16 = NaN
    raw_y, y = guarded((T, H), torch.bfloat16, 0xFF)
    frn.fused_reduce_rmsnorm(p, res, g, inp.eps, residual_out=ro, y=y)
    torch.cuda.synchronize()
    assert canaries_intact(raw_ro, 0xFF) and canaries_intact(raw_y, 0xFF)
    rro, ry = oracle.Oracle().reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, inp.eps)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)
    if H % 128:
        return
    raw_q, q = guarded((T, H), torch.uint8, 0xA5)
    raw_s, s = guarded((T, H // 128), torch.float32, 0xA5)
    raw_y2, y2 = guarded((T, H), torch.bfloat16, 0xFF)
    raw_ro2, ro2 = guarded((T, H), torch.bfloat16, 0xFF)
    frn.fused_reduce_rmsnorm_quant_per_group(p, res, g, inp.eps, 128, True, residual_out=ro2, y=y2, q=q, scales=s)
    torch.cuda.synchronize()
    for raw, fb in ((raw_q, 0xA5), (raw_s, 0xA5), (raw_y2, 0xFF), (raw_ro2, 0xFF)):
        assert canaries_intact(raw, fb)
    rro, ry, rq, rs = oracle.Oracle().reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps)
    assert_residual_exact(host_bits(ro2), rro)
    assert_quant_close(host_bits(y2), host_bits(q), host_bits(s), ry, rq, rs)


def test_rejected_calls_launch_nothing_and_process_stays_usable():
    inp = syn.make_inputs(2, 4, 256, seed=71)
    p, res, g = dev_bf16(inp.partials), dev_bf16(inp.residual), dev_bf16(inp.gamma)
    ro = torch.full((4, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full_like(ro, float("nan"))
    lib = frn.library()
    import ctypes
    arr = (ctypes.c_void_p * 2)(p[0].data_ptr(), p[1].data_ptr())
    bad = [
        (dict(R=0), frn.FRN_ERR_INVALID_ARG),
        (dict(R=17), frn.FRN_ERR_UNSUPPORTED),
        (dict(H=252), frn.FRN_ERR_UNSUPPORTED),
        (dict(eps=float("nan")), frn.FRN_ERR_INVALID_ARG),
        (dict(eps=-1.0), frn.FRN_ERR_INVALID_ARG),
        (dict(T=-1), frn.FRN_ERR_INVALID_ARG),
        (dict(y=None), frn.FRN_ERR_INVALID_ARG),
        (dict(gamma=None), frn.FRN_ERR_INVALID_ARG),
        (dict(y=y.data_ptr() + 2), frn.FRN_ERR_MISALIGNED),
        (dict(ro=p[0].data_ptr()), frn.FRN_ERR_INVALID_ARG),          # output aliases a partial
        (dict(y=ro.data_ptr()), frn.FRN_ERR_INVALID_ARG),             # two outputs overlap
        (dict(ro=res.data_ptr() + 16), frn.FRN_ERR_INVALID_ARG),      # partial overlap with residual
    ]
    for kw, want in bad:
        a = dict(R=2, res=res.data_ptr(), gamma=g.data_ptr(), ro=ro.data_ptr(), y=y.data_ptr(), T=4, H=256, eps=1e-6)
        a.update(kw)
        st = lib.fused_reduce_rmsnorm(arr, a["R"], a["res"], a["gamma"], a["ro"], a["y"], a["T"], a["H"], a["eps"],
                                      torch.cuda.current_stream().cuda_stream)
        assert st == want, (kw, frn.status_string(st), lib.frn_last_error_detail())
    torch.cuda.synchronize()
    assert torch.isnan(ro.float()).all() and torch.isnan(y.float()).all()
    # the process is still usable
    frn.fused_reduce_rmsnorm(p, res, g, inp.eps, residual_out=ro, y=y)
    torch.cuda.synchronize()
    rro, ry = oracle.Oracle().reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, inp.eps)
    assert_residual_exact(host_bits(ro), rro)


def test_quant_argument_errors():
    inp = syn.make_inputs(2, 4, 256, seed=72)
    p, res, g = dev_bf16(inp.partials), dev_bf16(inp.residual), dev_bf16(inp.gamma)
    with pytest.raises(frn.FrnError) as e:
        frn.fused_reduce_rmsnorm_quant_per_group(p, res, g, 1e-6, group_size=64)
    assert e.value.status == frn.FRN_ERR_UNSUPPORTED
    inp = syn.make_inputs(2, 4, 200, seed=73)
    with pytest.raises(ValueError):
        frn.fused_reduce_rmsnorm_quant_per_group(dev_bf16(inp.partials), None, dev_bf16(inp.gamma), 1e-6)
