"""torch custom ops over the C ABI, with fake (shape-only) implementations.

Registering the fused epilogue as opaque custom ops lets it sit inside
torch.compile graphs and CUDA graphs the way the vLLM pattern pass of the
"ROCm AITER fused all-reduce + RMSNorm" page (vLLM PR 37646 summary,
implementation breakdown items 1-2 and 5) swaps it in: the compiler sees the
op's output shapes through the fake implementation and never traces into it.
The real implementations call the same library entry points as the plain
binding; there is no other code path.

Ops (namespace ``frn``):
  fused_reduce_rmsnorm(partials[], residual?, gamma, eps) -> (y, residual_out)
  fused_reduce_rmsnorm_quant_per_group(partials[], residual?, gamma, eps, group_size, emit_bf16)
      -> (y_or_empty, q, scales, residual_out)   (y is a [0, H] tensor unless emit_bf16)
  fused_reduce_rmsnorm_mxfp4(partials[], residual?, gamma, eps, emit_bf16)
      -> (y_or_empty, q_fp4 uint8 [T, H/2], scales_e8m0 uint8 [T, H/32], residual_out)
  fused_add_rmsnorm(x, residual?, gamma, eps) -> (y, residual_out)
  rmsnorm(x, gamma, eps) -> y
"""
from __future__ import annotations

import torch

from . import fused_add_rmsnorm as _add_norm
from . import fused_reduce_rmsnorm as _fused
from . import fused_reduce_rmsnorm_mxfp4 as _fused_mx
from . import fused_reduce_rmsnorm_quant_per_group as _fused_quant
from . import rmsnorm as _rmsnorm


@torch.library.custom_op("frn::fused_reduce_rmsnorm", mutates_args=())
def fused_reduce_rmsnorm_op(partials: list[torch.Tensor], residual: torch.Tensor | None, gamma: torch.Tensor,
                            eps: float) -> tuple[torch.Tensor, torch.Tensor]:
    y, ro = _fused(list(partials), residual, gamma, eps)
    return y, ro


@fused_reduce_rmsnorm_op.register_fake
def _(partials, residual, gamma, eps):
    x = partials[0]
    return torch.empty_like(x), torch.empty_like(x)


@torch.library.custom_op("frn::fused_reduce_rmsnorm_quant_per_group", mutates_args=())
def fused_reduce_rmsnorm_quant_per_group_op(partials: list[torch.Tensor], residual: torch.Tensor | None,
                                            gamma: torch.Tensor, eps: float, group_size: int,
                                            emit_bf16: bool) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor,
                                                                      torch.Tensor]:
    out, ro = _fused_quant(list(partials), residual, gamma, eps, group_size, emit_bf16)
    if emit_bf16:
        y, q, s = out
    else:
        q, s = out
        y = ro.new_empty((0, ro.shape[1]))
    return y, q, s, ro


@fused_reduce_rmsnorm_quant_per_group_op.register_fake
def _(partials, residual, gamma, eps, group_size, emit_bf16):
    x = partials[0]
    T, H = x.shape
    y = torch.empty_like(x) if emit_bf16 else x.new_empty((0, H))
    q = x.new_empty((T, H), dtype=torch.float8_e4m3fn)
    s = x.new_empty((T, H // group_size), dtype=torch.float32)
    return y, q, s, torch.empty_like(x)


@torch.library.custom_op("frn::fused_reduce_rmsnorm_mxfp4", mutates_args=())
def fused_reduce_rmsnorm_mxfp4_op(partials: list[torch.Tensor], residual: torch.Tensor | None,
                                  gamma: torch.Tensor, eps: float,
                                  emit_bf16: bool) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor]:
    out, ro = _fused_mx(list(partials), residual, gamma, eps, emit_bf16)
    if emit_bf16:
        y, q, s = out
    else:
        q, s = out
        y = ro.new_empty((0, ro.shape[1]))
    return y, q, s, ro


@fused_reduce_rmsnorm_mxfp4_op.register_fake
def _(partials, residual, gamma, eps, emit_bf16):
    x = partials[0]
    T, H = x.shape
    y = torch.empty_like(x) if emit_bf16 else x.new_empty((0, H))
    q = x.new_empty((T, H // 2), dtype=torch.uint8)
    s = x.new_empty((T, H // 32), dtype=torch.uint8)
    return y, q, s, torch.empty_like(x)


@torch.library.custom_op("frn::fused_add_rmsnorm", mutates_args=())
def fused_add_rmsnorm_op(x: torch.Tensor, residual: torch.Tensor | None, gamma: torch.Tensor,
                         eps: float) -> tuple[torch.Tensor, torch.Tensor]:
    y, ro = _add_norm(x, residual, gamma, eps)
    return y, ro


@fused_add_rmsnorm_op.register_fake
def _(x, residual, gamma, eps):
    return torch.empty_like(x), torch.empty_like(x)


@torch.library.custom_op("frn::rmsnorm", mutates_args=())
def rmsnorm_op(x: torch.Tensor, gamma: torch.Tensor, eps: float) -> torch.Tensor:
    return _rmsnorm(x, gamma, eps)


@rmsnorm_op.register_fake
def _(x, gamma, eps):
    return torch.empty_like(x)
