"""Stream-ordering guards (GPU).

A fused call must never read a partial before the kernel that produces it has
finished, and a later call must never clobber buffers an earlier one still
reads -- the failure the missing end_sync barrier caused in the fused
allreduce + RMSNorm kernels ("Fix: add missing end_sync barrier in fused
allreduce+rmsnorm kernel", AITER PR 4346).  Here the guarantee comes from stream
order plus a grid-dependency wait at the top of the kernel; these tests run a
deliberately slow producer right before each call, with and without
programmatic dependent launch, on one stream, across two streams joined by an
event, back to back on reused buffers, and inside CUDA graphs.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import assert_residual_exact, assert_y_close, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

R, T, H = 4, 16, 4096
SLEEP_CYCLES = 20_000_000   # ~10 ms of device time before the producer writes


@pytest.fixture(params=[True, False], ids=["pdl", "no_pdl"])
def pdl(request):
    frn.set_pdl(request.param)
    yield request.param
    frn.set_pdl(True)


def _ref(inp):
    return oracle.Oracle().reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, inp.eps)


def test_same_stream_slow_producer(pdl):
    inp = syn.make_inputs(R, T, H, seed=50)
    src = dev_bf16(inp.partials)
    buf = torch.zeros_like(src)
    res, gamma = dev_bf16(inp.residual), dev_bf16(inp.gamma)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(SLEEP_CYCLES)
        buf.copy_(src)                       # the producer
        y, ro = frn.fused_reduce_rmsnorm(buf, res, gamma, inp.eps)
    s.synchronize()
    rro, ry = _ref(inp)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)


@pytest.mark.parametrize("shape", [(4, 16, 4096), (8, 16, 7168), (8, 64, 7168), (2, 700, 256), (8, 586, 7168),
                                   (2, 700, 7168)],
                         ids=["single_cta", "cluster", "wide", "packed", "wide_waves", "r2_waves"])
def test_slow_producer_with_l2_prefetch_forced_on(shape):
    """The kernels prefetch their rows into L2 before the dependency wait (and,
    over several waves, the first wave's rows and rows further ahead).  With
    the prefetch forced on for every row-kernel shape and a slow producer that
    overwrites the partials (zeros before) only after ~10 ms, the prefetched
    lines hold the old zeros, yet every value the kernel reads after the wait is
    the producer's: L2 is where the producer's writes land."""
    R_, T_, H_ = shape
    inp = syn.make_inputs(R_, T_, H_, seed=52, partial_std=0.5)
    src = dev_bf16(inp.partials)
    buf = torch.zeros_like(src)
    res, gamma = dev_bf16(inp.residual), dev_bf16(inp.gamma)
    frn.set_l2_prefetch(2)
    frn.set_kernel(frn.KERNEL_ROWS)
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            torch.cuda._sleep(SLEEP_CYCLES)
            buf.copy_(src)                   # the producer
            y, ro = frn.fused_reduce_rmsnorm(buf, res, gamma, inp.eps)
        s.synchronize()
    finally:
        frn.set_kernel(frn.KERNEL_AUTO)
        frn.set_l2_prefetch(0)
    rro, ry = _ref(inp)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)


def test_two_streams_event(pdl):
    inp = syn.make_inputs(R, T, H, seed=51)
    src = dev_bf16(inp.partials)
    buf = torch.zeros_like(src)
    res, gamma = dev_bf16(inp.residual), dev_bf16(inp.gamma)
    ro = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(ro)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()
    with torch.cuda.stream(s1):
        torch.cuda._sleep(SLEEP_CYCLES)
        buf.copy_(src)
        ev.record(s1)
    s2.wait_event(ev)
    frn.fused_reduce_rmsnorm(buf, res, gamma, inp.eps, residual_out=ro, y=y, stream=s2)
    s2.synchronize()
    rro, ry = _ref(inp)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)


def _reuse_setup(n_iter):
    inps = [syn.make_inputs(R, T, H, seed=100 + i) for i in range(n_iter)]
    srcs = torch.stack([dev_bf16(i.partials) for i in inps])
    ress = torch.stack([dev_bf16(i.residual) for i in inps])
    gamma = dev_bf16(inps[0].gamma)
    buf = torch.zeros_like(srcs[0])
    rbuf = torch.zeros_like(ress[0])
    ro = torch.full((n_iter, T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full_like(ro, float("nan"))
    return inps, srcs, ress, gamma, buf, rbuf, ro, y


def _reuse_body(n_iter, srcs, ress, gamma, buf, rbuf, ro, y, eps):
    for i in range(n_iter):
        buf.copy_(srcs[i])          # overwrite the same partial buffers every call
        rbuf.copy_(ress[i])
        frn.fused_reduce_rmsnorm(buf, rbuf, gamma, eps, residual_out=ro[i], y=y[i])


def _reuse_check(inps, ro, y):
    orc = oracle.Oracle()
    roh, yh = host_bits(ro), host_bits(y)
    for i, inp in enumerate(inps):
        sub = syn.Inputs(inp.partials, inp.residual, inp.gamma, inp.eps)
        rro, ry = orc.reduce_rmsnorm(sub.partials, sub.residual, gamma_of(inps), sub.eps)
        assert_residual_exact(roh[i], rro, f"iteration {i}")
        assert_y_close(yh[i], ry, f"iteration {i}")


def gamma_of(inps):
    return inps[0].gamma


def test_back_to_back_reuse(pdl):
    n = 64
    inps, srcs, ress, gamma, buf, rbuf, ro, y = _reuse_setup(n)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(SLEEP_CYCLES // 4)
        _reuse_body(n, srcs, ress, gamma, buf, rbuf, ro, y, inps[0].eps)
    s.synchronize()
    _reuse_check(inps, ro, y)


def test_back_to_back_reuse_in_cuda_graph(pdl):
    n = 64
    inps, srcs, ress, gamma, buf, rbuf, ro, y = _reuse_setup(n)
    # warm up outside the capture (loads the kernels), then capture
    _reuse_body(2, srcs, ress, gamma, buf, rbuf, ro, y, inps[0].eps)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _reuse_body(n, srcs, ress, gamma, buf, rbuf, ro, y, inps[0].eps)
    for _ in range(2):
        ro.fill_(float("nan"))
        y.fill_(float("nan"))
        buf.zero_()
        g.replay()
        torch.cuda.synchronize()
        _reuse_check(inps, ro, y)


def test_quant_graph_replay_with_slow_producer(pdl):
    inp = syn.make_inputs(R, T, H, seed=52, partial_std=0.5)
    src = dev_bf16(inp.partials)
    buf = torch.zeros_like(src)
    res, gamma = dev_bf16(inp.residual), dev_bf16(inp.gamma)
    ro = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(ro)
    q = torch.empty((T, H), dtype=torch.float8_e4m3fn, device="cuda")
    sc = torch.empty((T, H // 128), dtype=torch.float32, device="cuda")

    def body():
        torch.cuda._sleep(SLEEP_CYCLES // 4)
        buf.copy_(src)
        frn.fused_reduce_rmsnorm_quant_per_group(buf, res, gamma, inp.eps, 128, True, residual_out=ro, y=y,
                                                 q=q, scales=sc)

    body()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    buf.zero_()
    q.zero_()
    g.replay()
    torch.cuda.synchronize()
    rro, ry, rq, rs = oracle.Oracle().reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)
    from frn_testlib import assert_quant_close
    assert_quant_close(host_bits(y), host_bits(q), host_bits(sc), ry, rq, rs)
