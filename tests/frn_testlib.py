"""Helpers shared by the GPU tests: move seeded inputs to the device, call the
library through its binding, and compare with the CPU oracle under the
matching rules:

* residual_out: bit-exact (same fixed-order fp32 sum, one RNE);
* y: within 1 bf16 ulp (|difference of ordered bit patterns| <= 1);
* fp8 codes: equal, except at most 1 e4m3 ulp on at most 0.1% of elements;
  and, given the library's y, exactly the oracle's quantisation of that y;
* scales: within 1e-6 relative of the oracle wherever the group's absmax y
  element has the same bits on both sides, and for every group within 1e-6 of
  absmax(y_gpu) / 448 (the GPU's own y) -- a 1-ulp flip of the absmax y
  element moves the scale by ~2^-8, which the 1e-6 rule cannot cover;
* MXFP4: every 32-block's E8M0 code and E2M1 codes equal the oracle's OCP MX
  quantisation of the library's own y (the same decision in the same
  precision), and the oracle's own codes wherever the block's y equals the
  oracle's; y is one ulp off the oracle's on at most 0.1% of elements.
"""
from __future__ import annotations

import numpy as np
import torch

import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300.synthetic import Inputs, bf16_bits_to_f32

Y_ULP_TOL = 1            # bf16 ulps
Q_ULP_TOL = 1            # e4m3 ulps
Q_MISMATCH_FRAC = 1e-3   # fraction of fp8 codes allowed to differ (by <= 1 ulp)
SCALE_RTOL = 1e-6
MX_Y_FLIP_FRAC = 1e-3     # fraction of y elements allowed one ulp off the oracle's (MXFP4 rule)


def dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.detach().view(torch.uint8).cpu().numpy()
    return t.detach().cpu().numpy()


class DevInputs:
    def __init__(self, inp: Inputs, device="cuda"):
        self.inp = inp
        self.partials = dev_bf16(inp.partials, device)
        self.residual = dev_bf16(inp.residual, device) if inp.residual is not None else None
        self.gamma = dev_bf16(inp.gamma, device)
        self.eps = inp.eps


def gpu_norm(d: DevInputs, **kw):
    y, ro = frn.fused_reduce_rmsnorm(d.partials, d.residual, d.gamma, d.eps, **kw)
    return host_bits(ro), host_bits(y)


def gpu_quant(d: DevInputs, emit_bf16: bool, **kw):
    out, ro = frn.fused_reduce_rmsnorm_quant_per_group(d.partials, d.residual, d.gamma, d.eps, 128,
                                                       emit_bf16, **kw)
    if emit_bf16:
        y, q, s = out
        return host_bits(ro), host_bits(y), host_bits(q), host_bits(s)
    q, s = out
    return host_bits(ro), None, host_bits(q), host_bits(s)


def ordered_bf16(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ordered_e4m3(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int32)
    return np.where(b & 0x80, -(b & 0x7F), b)


def assert_residual_exact(ro_gpu, ro_ref, what=""):
    bad = np.flatnonzero(ro_gpu.ravel() != ro_ref.ravel())
    assert bad.size == 0, f"{what}: residual_out differs at {bad.size} elements, first {bad[:5]}"


def assert_y_close(y_gpu, y_ref, what="") -> int:
    d = np.abs(ordered_bf16(y_gpu) - ordered_bf16(y_ref))
    assert d.max(initial=0) <= Y_ULP_TOL, f"{what}: y differs by {d.max()} ulps"
    return int((d > 0).sum())


def assert_quant_close(y_gpu, q_gpu, s_gpu, y_ref, q_ref, s_ref, what="", group=128) -> dict:
    T, H = q_ref.shape
    ng = H // group
    if y_gpu is not None:
        # the same decision in the same precision: the library's codes and
        # scales are the oracle's quantisation of the library's own y
        import oracle
        q_y, s_y = oracle.Oracle().quant_per_group(y_gpu, group)
        assert np.array_equal(q_gpu, q_y) and np.array_equal(s_gpu.view(np.uint32), s_y.view(np.uint32)), \
            f"{what}: fp8 codes or scales are not the oracle's quantisation of the library's y"
    # codes
    dq = np.abs(ordered_e4m3(q_gpu) - ordered_e4m3(q_ref))
    assert dq.max(initial=0) <= Q_ULP_TOL, f"{what}: fp8 codes differ by {dq.max()} ulps"
    frac = float((dq > 0).mean()) if dq.size else 0.0
    assert frac <= Q_MISMATCH_FRAC, f"{what}: {frac:.2e} of fp8 codes differ"
    # scales where the absmax y element agrees
    yr = np.abs(bf16_bits_to_f32(y_ref)).reshape(T, ng, group).max(-1)
    flips = 0
    if y_gpu is not None:
        yg = np.abs(bf16_bits_to_f32(y_gpu)).reshape(T, ng, group).max(-1)
        same = yg == yr
        flips = int((~same).sum())
        self_s = (yg / np.float32(448.0)).astype(np.float32)
        rel = np.abs(s_gpu - self_s) / np.maximum(np.abs(self_s), np.finfo(np.float32).tiny)
        assert np.all(rel <= SCALE_RTOL), f"{what}: scales not absmax(y)/448 of the GPU's y"
    else:
        same = np.abs(s_gpu - s_ref) <= SCALE_RTOL * np.abs(s_ref)
        flips = int((~same).sum())
    rel = np.abs(s_gpu - s_ref) / np.maximum(np.abs(s_ref), np.finfo(np.float32).tiny)
    assert np.all(rel[same] <= SCALE_RTOL), f"{what}: scales differ where absmax agrees"
    assert flips <= max(2, 0.001 * T * ng), f"{what}: {flips} groups with a flipped absmax"
    return {"code_mismatch_frac": frac, "absmax_flips": flips}


def mx_codes(q: np.ndarray) -> np.ndarray:
    """Packed E2M1 bytes [T, H/2] -> codes [T, H] (element 2i in the low nibble)."""
    T, Hh = q.shape
    return np.stack([q & 0xF, q >> 4], axis=-1).reshape(T, 2 * Hh)


def ordered_e2m1(c: np.ndarray) -> np.ndarray:
    c = c.astype(np.int32)
    return np.where(c & 0x8, -(c & 0x7), c & 0x7)


def assert_mx_close(y_gpu, q_gpu, s_gpu, y_ref, q_ref, s_ref, what="") -> int:
    """MXFP4 codes and E8M0 scales against the oracle.  y_gpu is the library's
    y for the same inputs (the variant's own, or the plain entry point's, which
    has the same bits); the caller checks it within one bf16 ulp of the
    oracle's y.  Every block's scale and codes must equal the oracle's OCP MX
    quantisation of y_gpu: the same decision, taken in the same precision.  (A
    one-ulp flip of a block's absmax across a power of two moves the block's
    shared exponent and with it every code of the block, so across such a flip
    the codes cannot be compared with the oracle's own.)  Where a whole block's
    y equals the oracle's, scale and codes must equal the oracle's own, and y
    may differ from the oracle's on at most 0.1 % of elements.  Returns the
    number of blocks whose y differs."""
    import oracle
    T, H = y_ref.shape
    q_y, s_y = oracle.Oracle().mxfp4(y_gpu)
    assert np.array_equal(q_gpu, q_y) and np.array_equal(s_gpu, s_y), \
        f"{what}: codes or scales are not the OCP MX quantisation of the library's y"
    c, rc = mx_codes(q_gpu).reshape(T, H // 32, 32), mx_codes(q_ref).reshape(T, H // 32, 32)
    same = np.all(y_gpu.reshape(T, H // 32, 32) == y_ref.reshape(T, H // 32, 32), axis=-1)
    assert np.array_equal(s_gpu[same], s_ref[same]), what
    assert np.array_equal(c[same], rc[same]), what
    flip_frac = float((y_gpu != y_ref).mean()) if y_ref.size else 0.0
    assert flip_frac <= MX_Y_FLIP_FRAC, f"{what}: y differs from the oracle's on {flip_frac:.2e} of elements"
    return int((~same).sum())
