"""Seeded synthetic inputs for the fused reduce + residual-add + RMSNorm epilogue.

This module is shared by the CUDA path's tests/benchmark and by the CPU oracle's
tests; it therefore holds none of the epilogue's arithmetic.  It draws float32
values with numpy's ``default_rng(seed)`` and converts them to bf16 bit patterns
with torch's round-to-nearest-even cast (a library routine).

Draw order for every workload: partials (R, T, H), then residual (T, H), then
gamma (H), then the outlier channel indices.  Outliers, where asked for, scale
the chosen hidden channels of every partial and every token before rounding.

The workloads mirror the shapes the pages care about: hidden sizes up to 7168
(DeepSeek-style, the vLLM eligibility gate), decode token counts up to 80, the
allreduce message sweep 32 KB..64 MB of the AITER custom-allreduce table, and a
prefill chunk.  No dataset is involved anywhere.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns (torch RNE cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact widening, via torch)."""
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float32).numpy()


@dataclass
class Inputs:
    partials: np.ndarray          # uint16 [R, T, H] bf16 bits
    residual: np.ndarray | None   # uint16 [T, H] bf16 bits, or None
    gamma: np.ndarray             # uint16 [H] bf16 bits
    eps: float
    outlier_channels: np.ndarray = field(default_factory=lambda: np.zeros(0, dtype=np.int64))

    @property
    def R(self) -> int:
        return self.partials.shape[0]

    @property
    def T(self) -> int:
        return self.partials.shape[1]

    @property
    def H(self) -> int:
        return self.partials.shape[2]


def make_inputs(R: int, T: int, H: int, seed: int = 0, partial_std: float = 1.0,
                residual_std: float = 1.0, gamma_lo: float = 0.5, gamma_hi: float = 1.5,
                eps: float = 1e-6, outlier_frac: float = 0.0, outlier_scale: float = 50.0,
                with_residual: bool = True) -> Inputs:
    rng = np.random.default_rng(seed)
    p = rng.standard_normal((R, T, H), dtype=np.float32)
    if partial_std != 1.0:
        p *= np.float32(partial_std)
    res = rng.standard_normal((T, H), dtype=np.float32)
    if residual_std != 1.0:
        res *= np.float32(residual_std)
    gamma = rng.uniform(gamma_lo, gamma_hi, size=H).astype(np.float32)
    chans = np.zeros(0, dtype=np.int64)
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * H))
        chans = np.sort(rng.choice(H, size=n_out, replace=False)).astype(np.int64)
        p[:, :, chans] *= np.float32(outlier_scale)
    return Inputs(partials=f32_to_bf16_bits(p),
                  residual=f32_to_bf16_bits(res) if with_residual else None,
                  gamma=f32_to_bf16_bits(gamma), eps=eps, outlier_channels=chans)


# --------------------------------------------------------------------------
# The five workloads.
# --------------------------------------------------------------------------

#: hidden size shared by the decode, sweep and prefill workloads
H_DEEPSEEK = 7168
DECODE_TOKENS = (8, 16, 32, 64)
#: per-partial allreduce message sizes of the custom-allreduce latency table
SWEEP_BYTES = tuple(32 * 1024 * 2 ** i for i in range(12))   # 32 KB .. 64 MB


def sweep_tokens(msg_bytes: int, H: int = H_DEEPSEEK) -> int:
    """Tokens of one bf16 [T, H] partial of ``msg_bytes`` bytes, rounded up, at least 1."""
    return max(1, math.ceil(msg_bytes / (2 * H)))


def config_small(seed: int = 0) -> Inputs:
    """R=2, T=4, H=256; partials and residual N(0,1); gamma U(0.5,1.5); no quant."""
    return make_inputs(2, 4, 256, seed=seed)


def config_decode(T: int, seed: int = 0) -> Inputs:
    """R=8, H=7168, decode T; partials N(0, 0.5) (0.5 read as the std), residual N(0,1)."""
    return make_inputs(8, T, H_DEEPSEEK, seed=seed, partial_std=0.5)


def config_quant(seed: int = 0) -> Inputs:
    """R=4, T=32, H=4096; distributions as the decode workload; per-group-128 FP8 quant."""
    return make_inputs(4, 32, 4096, seed=seed, partial_std=0.5)


def config_sweep(msg_bytes: int, seed: int = 0) -> Inputs:
    """R=8, H=7168, T from the per-partial message size; no quant."""
    return make_inputs(8, sweep_tokens(msg_bytes), H_DEEPSEEK, seed=seed, partial_std=0.5)


def config_prefill(seed: int = 0, T: int = 8192) -> Inputs:
    """R=2, T=8192, H=7168, per-group-128 FP8 quant; partials N(0,1) with a random 1% of
    hidden channels scaled x50 (outliers); residual N(0,1)."""
    return make_inputs(2, T, H_DEEPSEEK, seed=seed, partial_std=1.0, outlier_frac=0.01,
                       outlier_scale=50.0)


def algorithmic_bytes(R: int, T: int, H: int, mode: str = "norm", group_size: int = 128,
                      with_residual: bool = True) -> int:
    """Bytes a perfect kernel moves through HBM per call.

    mode: "norm" (residual_out + y), "quant_a" (residual_out + fp8 + scales),
    "quant_b" (residual_out + y + fp8 + scales), "mx_a" (residual_out + packed
    fp4 + E8M0 scales per 32), "mx_b" (the same + y).
    """
    n = T * H
    b = 2 * n * R + 2 * H + 2 * n          # partials + gamma + residual_out
    if with_residual:
        b += 2 * n
    if mode == "norm":
        b += 2 * n
    elif mode == "quant_a":
        b += n + 4 * (n // group_size)
    elif mode == "quant_b":
        b += 3 * n + 4 * (n // group_size)
    elif mode == "mx_a":
        b += n // 2 + n // 32
    elif mode == "mx_b":
        b += 2 * n + n // 2 + n // 32
    else:
        raise ValueError(mode)
    return b


def make_inputs_device(R: int, T: int, H: int, seed: int = 0, partial_std: float = 1.0,
                       residual_std: float = 1.0, gamma_lo: float = 0.5, gamma_hi: float = 1.5,
                       outlier_frac: float = 0.0, outlier_scale: float = 50.0, device="cuda"):
    """Same distributions and draw order as ``make_inputs``, drawn on the device with
    a seeded torch generator (a different random stream from the numpy one).  Used
    for large benchmark inputs that are never compared with the oracle.

    Returns bf16 device tensors (partials [R,T,H], residual [T,H], gamma [H]).
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    p = torch.randn((R, T, H), generator=g, device=device, dtype=torch.float32)
    if partial_std != 1.0:
        p.mul_(partial_std)
    res = torch.randn((T, H), generator=g, device=device, dtype=torch.float32)
    if residual_std != 1.0:
        res.mul_(residual_std)
    gamma = torch.rand((H,), generator=g, device=device, dtype=torch.float32) * (gamma_hi - gamma_lo) + gamma_lo
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * H))
        chans = torch.randperm(H, generator=g, device=device)[:n_out]
        p[:, :, chans] *= outlier_scale
    return p.to(torch.bfloat16), res.to(torch.bfloat16), gamma.to(torch.bfloat16)
