"""Randomised shapes across the planner's regimes (GPU).

Each drawn (R, T, H, residual) runs through whatever launch the library plans
for it -- packed short rows, single and wide CTAs, clusters, two tiles a warp,
staged loads or the stream kernel, with or without the L2 prefetches -- and
every row of every output the shape supports (no quant; FP8 variants A and B
when H % 128 == 0; MXFP4 A and B when H % 32 == 0) is compared with the
oracle under the matching rules of frn_testlib.  The draw is seeded;
FRN_RANDOM_CASES sets how many shapes (default 40)."""
import os

import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import (DevInputs, assert_mx_close, assert_quant_close, assert_residual_exact, assert_y_close,
                         gpu_norm, gpu_quant, host_bits)

pytestmark = pytest.mark.gpu

THREADS = max(1, os.cpu_count() or 1)
N_CASES = int(os.environ.get("FRN_RANDOM_CASES", "40"))
MAX_ELEMENTS = 48 << 20     # R * T * H: keeps each case to a fraction of a second on the oracle


def draw(k: int):
    rng = np.random.default_rng(7000 + k)
    R = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 11, 16]))
    H = int(rng.choice([8 * int(rng.integers(1, 2049)), 256, 1024, 4096, 5120, 7168, 8192, 8448, 12288, 16384]))
    regime = rng.integers(0, 3)
    T = int(rng.integers(1, 80) if regime == 0 else rng.integers(80, 700) if regime == 1 else rng.integers(700, 5000))
    T = max(1, min(T, MAX_ELEMENTS // (R * H)))
    return R, T, H, bool(rng.random() < 0.85)


CASES = [draw(k) for k in range(N_CASES)]


@pytest.mark.parametrize("case", CASES, ids=[f"R{r}_T{t}_H{h}_{'res' if w else 'nores'}" for r, t, h, w in CASES])
def test_random_plan_against_oracle(case):
    R, T, H, with_residual = case
    inp = syn.make_inputs(R, T, H, seed=R * 100003 + T * 101 + H, partial_std=0.5, with_residual=with_residual)
    what = f"R={R} T={T} H={H} res={with_residual} launch={frn.query_launch(T, H, R, 0, with_residual)}"
    d = DevInputs(inp)
    orc = oracle.Oracle()
    ro, y = gpu_norm(d)
    rro, ry = orc.reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, inp.eps, threads=THREADS)
    assert_residual_exact(ro, rro, what)
    assert_y_close(y, ry, what)
    if H % 128 == 0:
        _, rq_y, rq, rs = orc.reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps, 128,
                                                   threads=THREADS)
        roA, _, qA, sA = gpu_quant(d, emit_bf16=False)
        roB, yB, qB, sB = gpu_quant(d, emit_bf16=True)
        assert np.array_equal(roA, ro) and np.array_equal(roB, ro) and np.array_equal(yB, y), what
        assert_quant_close(None, qA, sA, rq_y, rq, rs, what + " FP8 A")
        assert_quant_close(y, qA, sA, rq_y, rq, rs, what + " FP8 A, the library's y")
        assert_quant_close(yB, qB, sB, rq_y, rq, rs, what + " FP8 B")
    if H % 32 == 0:
        _, mx_y, mq, ms = orc.reduce_rmsnorm_mxfp4(inp.partials, inp.residual, inp.gamma, inp.eps, threads=THREADS)
        (qa, sa), roa = frn.fused_reduce_rmsnorm_mxfp4(d.partials, d.residual, d.gamma, inp.eps)
        (yb, qb, sb), rob = frn.fused_reduce_rmsnorm_mxfp4(d.partials, d.residual, d.gamma, inp.eps, emit_bf16=True)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(roa), ro) and np.array_equal(host_bits(rob), ro), what
        assert np.array_equal(host_bits(yb), y), what
        assert_mx_close(y, host_bits(qa), host_bits(sa), mx_y, mq, ms, what + " MXFP4 A")
        assert_mx_close(host_bits(yb), host_bits(qb), host_bits(sb), mx_y, mq, ms, what + " MXFP4 B")
