"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Covers the five workloads (small case; decode T in {8,16,32,64}; quant R=4
T=32 H=4096 in both output variants; the message-size sweep at H=7168, every
row of every size up to 64 MB per partial; the prefill chunk with outlier
channels, every row),
random shapes with ragged tails, and the edge cases: R=1, R=16, H=8, H=16384,
NULL residual, in-place residual, zero rows, huge and tiny magnitudes.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import (DevInputs, assert_quant_close, assert_residual_exact, assert_y_close, gpu_norm,
                         gpu_quant, host_bits, dev_bf16)

pytestmark = pytest.mark.gpu

ORC = None
THREADS = max(1, os.cpu_count() or 1)   # the oracle splits rows over the host's cores


def orc():
    global ORC
    if ORC is None:
        ORC = oracle.Oracle()
    return ORC


def ref_norm(inp):
    return orc().reduce_rmsnorm(inp.partials, inp.residual, inp.gamma, inp.eps, threads=THREADS)


def ref_quant(inp):
    return orc().reduce_rmsnorm_quant(inp.partials, inp.residual, inp.gamma, inp.eps, 128, threads=THREADS)


def check_norm(inp, what):
    d = DevInputs(inp)
    ro, y = gpu_norm(d)
    rro, ry = ref_norm(inp)
    assert_residual_exact(ro, rro, what)
    return assert_y_close(y, ry, what)


def check_quant(inp, what):
    d = DevInputs(inp)
    roA, _, qA, sA = gpu_quant(d, emit_bf16=False)
    roB, yB, qB, sB = gpu_quant(d, emit_bf16=True)
    ro_n, y_n = gpu_norm(d)
    # the two variants agree bit for bit, and B's y is the plain entry point's y
    assert np.array_equal(qA, qB) and np.array_equal(sA.view(np.uint32), sB.view(np.uint32)), what
    assert np.array_equal(roA, roB) and np.array_equal(roA, ro_n), what
    assert np.array_equal(yB, y_n), what
    rro, ry, rq, rs = ref_quant(inp)
    assert_residual_exact(roA, rro, what + " (A)")
    assert_residual_exact(roB, rro, what + " (B)")
    assert_y_close(yB, ry, what)
    assert_quant_close(None, qA, sA, ry, rq, rs, what + " (A)")
    return assert_quant_close(yB, qB, sB, ry, rq, rs, what + " (B)")


# ------------------------------------------------------------- workloads --

def test_small_case():
    check_norm(syn.config_small(), "R=2 T=4 H=256")


@pytest.mark.parametrize("T", syn.DECODE_TOKENS)
def test_decode(T):
    check_norm(syn.config_decode(T), f"decode T={T}")


def test_quant_both_variants():
    check_quant(syn.config_quant(), "quant R=4 T=32 H=4096")


@pytest.mark.parametrize("msg", syn.SWEEP_BYTES)
def test_sweep(msg):
    T = syn.sweep_tokens(msg)
    check_norm(syn.config_sweep(msg), f"sweep {msg} B (T={T})")


def test_prefill_outliers_quant():
    inp = syn.config_prefill()
    assert inp.outlier_channels.size == 72
    stats = check_quant(inp, "prefill R=2 T=8192 H=7168")
    # properties that hold at every row: each nonzero group reaches |q| = 448,
    # and the scales are the GPU's own absmax(y)/448
    d = DevInputs(inp)
    (y, q, s), _ = frn.fused_reduce_rmsnorm_quant_per_group(d.partials, d.residual, d.gamma, d.eps, 128, True)
    qf = q.view(torch.float8_e4m3fn).float().abs().view(inp.T, 56, 128)
    assert torch.all(qf.amax(-1)[s > 0] == 448.0)
    ya = y.float().abs().view(inp.T, 56, 128).amax(-1).cpu().numpy()
    assert np.array_equal(s.cpu().numpy(), ya / np.float32(448.0))
    # groups holding an outlier channel carry far larger scales than the rest
    outg = np.unique(inp.outlier_channels // 128)
    sn = s.cpu().numpy()
    rest = np.setdiff1d(np.arange(56), outg)
    if rest.size:
        assert np.median(sn[:, outg]) > 5 * np.median(sn[:, rest])
    assert stats["code_mismatch_frac"] <= 1e-3


# ----------------------------------------------------------- random shapes --

SHAPES = [
    (1, 1, 8), (1, 3, 24), (2, 7, 136), (3, 33, 1000), (5, 2, 2048), (8, 5, 7168), (13, 9, 4096),
    (16, 4, 7168), (2, 300, 256), (4, 17, 8200), (3, 3, 16384), (16, 2, 16384), (7, 65, 520),
    (2, 129, 7168), (1, 1025, 4096),
]


@pytest.fixture(params=[frn.KERNEL_ROWS, frn.KERNEL_STREAM], ids=["rows", "stream"])
def kernel(request):
    frn.set_kernel(request.param)
    yield request.param
    frn.set_kernel(frn.KERNEL_AUTO)


@pytest.mark.parametrize("R,T,H", SHAPES)
@pytest.mark.parametrize("with_residual", [True, False])
def test_random_shapes_norm(R, T, H, with_residual, kernel):
    inp = syn.make_inputs(R, T, H, seed=R * 1000 + T + H, with_residual=with_residual)
    check_norm(inp, f"R={R} T={T} H={H} res={with_residual} kernel={kernel}")


@pytest.mark.parametrize("R,T,H", [s for s in SHAPES if s[2] % 128 == 0])
def test_random_shapes_quant(R, T, H, kernel):
    inp = syn.make_inputs(R, T, H, seed=7 + R * 1000 + T + H, partial_std=0.5)
    check_quant(inp, f"quant R={R} T={T} H={H} kernel={kernel}")


@pytest.mark.parametrize("msg", [1 << 20, 64 << 20])
def test_sweep_each_kernel(msg, kernel):
    check_norm(syn.config_sweep(msg, seed=3), f"sweep {msg} B kernel={kernel}")


def test_prefill_each_kernel(kernel):
    inp = syn.config_prefill(seed=2)
    check_quant(inp, f"prefill kernel={kernel}")


@pytest.mark.parametrize("ctas", [1, 2, 3, 4, 5, 7, 8, 14, 16, "stream"])
@pytest.mark.parametrize("H", [7168, 4096, 16384])
def test_every_launch_shape_is_bit_identical(ctas, H):
    """Whatever number of CTAs a row is split over, and whichever kernel runs, every
    output has the same bits."""
    inp = syn.make_inputs(8, 11, H, seed=5, partial_std=0.5)
    d = DevInputs(inp)
    frn.set_kernel(frn.KERNEL_ROWS)
    try:
        base = gpu_quant(d, True)
        if ctas == "stream":
            frn.set_kernel(frn.KERNEL_STREAM)
        else:
            frn.set_ctas_per_row(ctas)
        got = gpu_quant(d, True)
    finally:
        frn.set_ctas_per_row(0)
        frn.set_kernel(frn.KERNEL_AUTO)
    for a, b in zip(base, got):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


@pytest.mark.parametrize("R", [2, 8])
def test_many_row_launches_are_bit_identical(R):
    """At 400 rows (beyond two waves of wide CTAs: rstd from one warp, and with
    R = 2 the one-wave-ahead L2 prefetch) the row kernel gives the bits of the
    stream kernel, and its first rows the bits of a 13-row call of the same
    rows (per-warp rstd, no ahead prefetch)."""
    inp = syn.make_inputs(R, 400, 7168, seed=8, partial_std=0.5)
    d = DevInputs(inp)
    few = DevInputs(syn.Inputs(inp.partials[:, :13], inp.residual[:13], inp.gamma, inp.eps))
    try:
        frn.set_kernel(frn.KERNEL_ROWS)
        rows = gpu_quant(d, True)
        rows_few = gpu_quant(few, True)
        frn.set_kernel(frn.KERNEL_STREAM)
        stream = gpu_quant(d, True)
    finally:
        frn.set_kernel(frn.KERNEL_AUTO)
    for a, b, c in zip(rows, stream, rows_few):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))
        assert np.array_equal(np.asarray(a)[:13].view(np.uint8), np.asarray(c).view(np.uint8))


@pytest.mark.parametrize("R,T,H,with_residual", [
    (8, 153, 7168, True),     # one row past a wave of wide rows
    (8, 400, 7000, True),     # ragged last tile
    (1, 1000, 7168, True),    # two wide rows an SM
    (3, 800, 5120, True),     # two 640-thread rows an SM
    (2, 5000, 256, True),     # packed short rows, eight to a CTA
    (2, 700, 7168, False),    # no residual: R loads a row
    (8, 1171, 7168, False),
    (12, 400, 16384, True),   # two tiles a warp, R > 8 in stages of four (FP8 output)
    (8, 400, 16384, True),    # two tiles a warp, partials in stages of four (FP8 output)
])
def test_prefetch_ahead_paths(R, T, H, with_residual):
    """Grids of more than one wave, where each CTA prefetches the rows a fixed
    distance ahead and the first wave its own rows before the dependency wait:
    every row against the oracle, and the same bits with every prefetch off."""
    inp = syn.make_inputs(R, T, H, seed=90 + R + T + H, partial_std=0.5, with_residual=with_residual)
    quant = H % 128 == 0 and with_residual
    assert frn.query_launch(T, H, R, 1 if quant else 0, with_residual)[0] == frn.KERNEL_ROWS
    if quant:
        check_quant(inp, f"ahead R={R} T={T} H={H}")
    else:
        check_norm(inp, f"ahead R={R} T={T} H={H} res={with_residual}")
    d = DevInputs(inp)
    base = gpu_quant(d, True) if quant else gpu_norm(d)
    frn.set_l2_prefetch(1)
    try:
        off = gpu_quant(d, True) if quant else gpu_norm(d)
    finally:
        frn.set_l2_prefetch(0)
    for a, b in zip(base, off):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


@pytest.mark.parametrize("R,T,H,with_residual", [
    (2, 400, 16384, True), (1, 320, 8200, True), (2, 333, 12288, True), (2, 310, 10000, True),
    (1, 500, 16384, False), (2, 304, 8448, True), (4, 330, 16384, True), (3, 400, 12288, True),
    (4, 310, 9000, False), (8, 330, 16384, True), (6, 300, 12288, True), (5, 200, 8448, True),
    (3, 200, 7168, True), (4, 400, 8192, False), (4, 333, 6656, True), (3, 160, 7800, True),
    (2, 2500, 7168, True), (7, 300, 16384, False), (5, 250, 12288, True), (16, 200, 5120, True),
    (12, 160, 12288, True), (10, 180, 5000, True), (16, 100, 5120, False), (9, 90, 16384, True),
    (12, 700, 5120, True), (10, 1000, 4096, True), (9, 100, 2312, True), (12, 500, 3072, True),
    (11, 470, 4096, True), (8, 200, 7168, True), (6, 240, 8192, False), (1, 400, 10240, True),
    (2, 330, 9728, False),
])
def test_two_tiles_per_warp(R, T, H, with_residual):
    """Rows of 33..64 tiles with R <= 8 at many rows (and of 26..32 tiles with
    R = 3 or 4 beyond one row per SM, R = 5..8 from one to 1.65 rows per SM,
    or R = 2 with FP8 A from 16 rows an SM;
    and of 17..64 tiles with R > 8 and an FP8 output, or up to 22 tiles) take
    one CTA per row, two tiles a warp: every row against the oracle, and
    the bits of the cluster and stream kernels (and, past 32 tiles, of a
    forced launch at decode size, prefetch on; at 26..32 tiles T <= 2 waves
    prefetches before the wait by itself)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    quant = H % 128 == 0 and with_residual
    plan = frn.plan_launch(T, H, R, 1 if quant else 0, with_residual, sms)
    assert plan["kernel"] == frn.KERNEL_ROWS and plan["tiles_per_warp"] == 2, plan
    inp = syn.make_inputs(R, T, H, seed=70 + R + T + H, partial_std=0.5, with_residual=with_residual)
    if quant:
        check_quant(inp, f"two tiles R={R} T={T} H={H}")
    else:
        check_norm(inp, f"two tiles R={R} T={T} H={H} res={with_residual}")
    d = DevInputs(inp)

    def outs():
        got = list(gpu_quant(d, True)) if quant else list(gpu_norm(d))
        if H % 32 == 0:
            (q4, sc4), ro4 = frn.fused_reduce_rmsnorm_mxfp4(d.partials, d.residual, d.gamma, d.eps, False)
            got += [host_bits(q4), host_bits(sc4), host_bits(ro4)]
        return got
    base = outs()
    for kernel, ctas in ((frn.KERNEL_STREAM, 0), (frn.KERNEL_ROWS, 4)):
        frn.set_kernel(kernel)
        frn.set_ctas_per_row(ctas)
        try:
            other = outs()
        finally:
            frn.set_ctas_per_row(0)
            frn.set_kernel(frn.KERNEL_AUTO)
        for a, b in zip(base, other):
            assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8)), (kernel, ctas)
    if -(-(H // 8) // 32) <= 32:
        return
    # a decode-sized call forced onto the same shape, with the prefetch before the wait
    few = DevInputs(syn.Inputs(inp.partials[:, :5], None if inp.residual is None else inp.residual[:5],
                               inp.gamma, inp.eps))
    frn.set_kernel(frn.KERNEL_ROWS)
    frn.set_ctas_per_row(1)
    frn.set_l2_prefetch(2)
    try:
        assert frn.plan_launch(5, H, R, 0, with_residual, sms)["tiles_per_warp"] == 2
        ro5, y5 = gpu_norm(few)
    finally:
        frn.set_l2_prefetch(0)
        frn.set_ctas_per_row(0)
        frn.set_kernel(frn.KERNEL_AUTO)
    ro_all, y_all = gpu_norm(d)
    assert np.array_equal(ro5, ro_all[:5]) and np.array_equal(y5, y_all[:5])


@pytest.mark.parametrize("H", [256, 512, 768, 1024])
@pytest.mark.parametrize("R", [1, 2, 8])
def test_packed_short_rows(H, R):
    """Short rows at many T share 256-thread CTAs (8 / ntiles rows each, the
    last CTA ragged): every row matches the oracle, and its bits are those of
    a one-row-per-CTA call of the same rows."""
    T = 613
    inp = syn.make_inputs(R, T, H, seed=14 + H + R, partial_std=0.5)
    kernel, ctas, threads, grid = frn.query_launch(T, H, R)
    ntiles = -(-H // 256)
    assert (kernel, ctas, threads, grid) == (frn.KERNEL_ROWS, 1, (8 // ntiles) * ntiles * 32,
                                             -(-T // (8 // ntiles)))
    if H % 128 == 0:
        check_quant(inp, f"packed H={H} R={R}")
    else:
        check_norm(inp, f"packed H={H} R={R}")
    d = DevInputs(inp)
    ro, y = gpu_norm(d)
    few = DevInputs(syn.Inputs(inp.partials[:, 600:], inp.residual[600:], inp.gamma, inp.eps))
    assert frn.query_launch(13, H, R)[2] == ntiles * 32
    ro_f, y_f = gpu_norm(few)
    assert np.array_equal(ro[600:], ro_f) and np.array_equal(y[600:], y_f)


@pytest.mark.parametrize("prefetch", [1, 2])
@pytest.mark.parametrize("ctas", [1, 3, 8])
@pytest.mark.parametrize("H", [7000, 16384, 2056])
def test_l2_prefetch_changes_no_bit(prefetch, ctas, H):
    """The L2 prefetch before the dependency wait (off, or forced on for every
    row launch, over ragged last tiles too) leaves every output bit as it is."""
    inp = syn.make_inputs(8, 13, H, seed=6, partial_std=0.5)
    d = DevInputs(inp)
    frn.set_kernel(frn.KERNEL_ROWS)
    frn.set_ctas_per_row(ctas)
    try:
        base = gpu_quant(d, True) if H % 128 == 0 else gpu_norm(d)
        frn.set_l2_prefetch(prefetch)
        got = gpu_quant(d, True) if H % 128 == 0 else gpu_norm(d)
    finally:
        frn.set_l2_prefetch(0)
        frn.set_ctas_per_row(0)
        frn.set_kernel(frn.KERNEL_AUTO)
    for a, b in zip(base, got):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


# ------------------------------------------------------------- edge cases --

def test_empty_T_is_noop():
    d = DevInputs(syn.make_inputs(2, 1, 256))
    p = d.partials[:, :0]
    ro = torch.full((0, 256), 1.0, dtype=torch.bfloat16, device="cuda")
    y, ro2 = frn.fused_reduce_rmsnorm([p[0], p[1]], None, d.gamma, 1e-6, residual_out=ro)
    assert y.shape == (0, 256) and ro2 is ro
    frn.fused_reduce_rmsnorm_quant_per_group([p[0], p[1]], None, d.gamma, 1e-6)
    torch.cuda.synchronize()


@pytest.mark.parametrize("kernel", [frn.KERNEL_ROWS, frn.KERNEL_STREAM])
def test_outputs_in_pinned_host_memory(kernel):
    """Outputs may live in pinned host memory (the kernel writes them over the
    host link): the same bits as device outputs."""
    inp = syn.make_inputs(4, 37, 4096, seed=9, partial_std=0.5)
    d = DevInputs(inp)
    T, H = 37, 4096
    pin = lambda dt, shape: torch.empty(shape, dtype=dt).pin_memory()
    frn.set_kernel(kernel)
    try:
        ro_h, y_h = pin(torch.bfloat16, (T, H)), pin(torch.bfloat16, (T, H))
        frn.fused_reduce_rmsnorm(d.partials, d.residual, d.gamma, d.eps, residual_out=ro_h, y=y_h)
        q_h, s_h = pin(torch.float8_e4m3fn, (T, H)), pin(torch.float32, (T, H // 128))
        ro2_h, y2_h = pin(torch.bfloat16, (T, H)), pin(torch.bfloat16, (T, H))
        frn.fused_reduce_rmsnorm_quant_per_group(d.partials, d.residual, d.gamma, d.eps, 128, True,
                                                 residual_out=ro2_h, y=y2_h, q=q_h, scales=s_h)
        torch.cuda.synchronize()
        ro_d, y_d = gpu_norm(d)
        ro2_d, y2_d, q_d, s_d = gpu_quant(d, True)
    finally:
        frn.set_kernel(frn.KERNEL_AUTO)
    for h, dv in ((ro_h, ro_d), (y_h, y_d), (ro2_h, ro2_d), (y2_h, y2_d), (q_h, q_d), (s_h, s_d)):
        assert np.array_equal(host_bits(h).view(np.uint8), np.asarray(dv).view(np.uint8))


def test_quant_subnormal_y(kernel):
    """gamma among the bf16 subnormals makes y and absmax/448 tiny (fp32
    subnormal scales): the kernels take the IEEE divides there and match the
    oracle's codes and scales."""
    inp = syn.make_inputs(2, 9, 2048, seed=13)
    rng = np.random.default_rng(6)
    g = rng.integers(1, 0x80, size=2048).astype(np.uint16)
    g[::5] |= 0x8000
    check_quant(syn.Inputs(inp.partials, inp.residual, g, inp.eps), f"quant subnormal y kernel={kernel}")


@pytest.mark.parametrize("T,H", [(19, 4096), (700, 512), (300, 7168)])
def test_in_place_residual(T, H, kernel):
    """residual_out == residual (in place), for every kernel and row shape."""
    inp = syn.make_inputs(4, T, H, seed=3)
    d = DevInputs(inp)
    rro, ry = ref_norm(inp)
    res = d.residual.clone()
    y, ro = frn.fused_reduce_rmsnorm(d.partials, res, d.gamma, inp.eps, residual_out=res)
    assert ro.data_ptr() == res.data_ptr()
    assert_residual_exact(host_bits(res), rro, f"in place T={T} H={H} kernel={kernel}")
    assert_y_close(host_bits(y), ry, f"in place T={T} H={H} kernel={kernel}")


@pytest.mark.parametrize("R,T,H", [(8, 16, 7168), (8, 5, 16384), (2, 400, 16384), (2, 320, 9000), (4, 300, 7168)])
def test_in_place_residual_cluster_and_two_tile(R, T, H):
    """residual_out == residual on the cluster shapes (which store residual_out
    before the tile sums cross the cluster) and on the two-tile shape."""
    inp = syn.make_inputs(R, T, H, seed=5, partial_std=0.5)
    d = DevInputs(inp)
    rro, ry = ref_norm(inp)
    res = d.residual.clone()
    y, ro = frn.fused_reduce_rmsnorm(d.partials, res, d.gamma, inp.eps, residual_out=res)
    assert ro.data_ptr() == res.data_ptr()
    assert_residual_exact(host_bits(res), rro, f"in place R={R} T={T} H={H}")
    assert_y_close(host_bits(y), ry, f"in place R={R} T={T} H={H}")


def test_separate_partial_allocations_and_repeats():
    """Partials as R separate tensors, including one pointer passed twice."""
    inp = syn.make_inputs(3, 9, 2048, seed=4)
    parts = [dev_bf16(inp.partials[r]) for r in range(3)]
    rep = np.stack([inp.partials[0], inp.partials[1], inp.partials[2], inp.partials[1]])
    rro, ry = orc().reduce_rmsnorm(rep, inp.residual, inp.gamma, inp.eps)
    y, ro = frn.fused_reduce_rmsnorm([parts[0], parts[1], parts[2], parts[1]], dev_bf16(inp.residual),
                                     dev_bf16(inp.gamma), inp.eps)
    assert_residual_exact(host_bits(ro), rro)
    assert_y_close(host_bits(y), ry)


def test_zero_rows_and_zero_groups():
    inp = syn.make_inputs(2, 6, 1024, seed=6)
    inp.partials[:, 2] = 0
    inp.residual[2] = 0
    inp.partials[:, 4, 128:256] = 0
    inp.residual[4, 128:256] = 0
    stats = check_quant(inp, "zero rows")
    d = DevInputs(inp)
    _, _, q, s = gpu_quant(d, True)
    assert np.all(q[2] == 0) and np.all(s[2] == 0)
    assert s[4, 1] == 0 and np.all(q[4, 128:256] == 0)
    assert stats["absmax_flips"] <= 2


@pytest.mark.parametrize("scale", [2.0 ** -60, 2.0 ** -20, 2.0 ** 20, 2.0 ** 50])
def test_magnitudes(scale):
    """Rows far from unit scale, within the range where fp32 sums of squares of a
    16384-wide row stay finite and normal."""
    inp = syn.make_inputs(3, 5, 4096, seed=8)
    f = syn.bf16_bits_to_f32(inp.partials) * np.float32(scale)
    r = syn.bf16_bits_to_f32(inp.residual) * np.float32(scale)
    inp = syn.Inputs(syn.f32_to_bf16_bits(f), syn.f32_to_bf16_bits(r), inp.gamma, 1e-30)
    check_quant(inp, f"scale {scale}")


def test_eps_matters():
    """Rows whose mean square is comparable to eps."""
    inp = syn.make_inputs(2, 8, 2048, seed=9, partial_std=1e-3, residual_std=1e-3)
    check_norm(syn.Inputs(inp.partials, inp.residual, inp.gamma, 1e-6), "eps ~ mean square")
    check_norm(syn.Inputs(inp.partials, inp.residual, inp.gamma, 0.5), "eps dominant")


@pytest.mark.parametrize("groups", [1, 2, 3, 4])
@pytest.mark.parametrize("R,T,H", [(4, 301, 4096), (8, 157, 7168), (2, 400, 1024), (3, 97, 256)])
def test_stream_consumer_groups(groups, R, T, H):
    """Every consumer-group count gives the same bits, and they match the oracle."""
    inp = syn.make_inputs(R, T, H, seed=11 + groups, partial_std=0.5)
    frn.set_kernel(frn.KERNEL_STREAM)
    frn.set_stream_groups(groups)
    try:
        check_quant(inp, f"stream groups={groups} R={R} T={T} H={H}") if H % 128 == 0 else \
            check_norm(inp, f"stream groups={groups} R={R} T={T} H={H}")
    finally:
        frn.set_stream_groups(0)
        frn.set_kernel(frn.KERNEL_AUTO)


def test_cluster_rows_prefetch_ahead_forced():
    """Cluster rows from two waves on prefetch the rows a fixed distance ahead.
    The planner gives such rows two tiles a warp instead, so clusters of 4 are
    forced: R = 12, T = 400, H = 16384 with an FP8 output against the oracle,
    and the same bits with every prefetch off and on the planner's choice."""
    R, T, H = 12, 400, 16384
    inp = syn.make_inputs(R, T, H, seed=95, partial_std=0.5)
    d = DevInputs(inp)
    auto = gpu_quant(d, True)
    frn.set_kernel(frn.KERNEL_ROWS)
    frn.set_ctas_per_row(4)
    try:
        assert frn.query_launch(T, H, R, 2)[1] == 4
        check_quant(inp, f"forced clusters R={R} T={T} H={H}")
        clusters = gpu_quant(d, True)
        frn.set_l2_prefetch(1)
        off = gpu_quant(d, True)
    finally:
        frn.set_l2_prefetch(0)
        frn.set_ctas_per_row(0)
        frn.set_kernel(frn.KERNEL_AUTO)
    for a, b, c in zip(auto, clusters, off):
        if a is not None:
            assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))
            assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(c).view(np.uint8))


@pytest.mark.parametrize("R,T,H", [(16, 600, 4096), (9, 500, 2048), (14, 1000, 4096), (16, 457, 3968),
                                   (12, 460, 1024)])
def test_staged_loads(R, T, H):
    """Rows whose partials are loaded in stages (two stages of two in flight),
    as the planner picks them: every row of every output against the oracle,
    and the same bits as the stream kernel."""
    quant = H % 128 == 0
    plan = frn.plan_launch(T, H, R, 1 if quant else 0, True,
                           torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["staged"] == 1, plan
    inp = syn.make_inputs(R, T, H, seed=40 + R + T, partial_std=0.5)
    got = check_quant(inp, f"staged R={R} T={T} H={H}") if quant else check_norm(inp, f"staged R={R} T={T} H={H}")
    d = DevInputs(inp)
    outs = [gpu_quant(d, True), gpu_quant(d, False)] if quant else [gpu_norm(d)]
    frn.set_kernel(frn.KERNEL_STREAM)
    try:
        ref = [gpu_quant(d, True), gpu_quant(d, False)] if quant else [gpu_norm(d)]
    finally:
        frn.set_kernel(frn.KERNEL_AUTO)
    for a_set, b_set in zip(outs, ref):
        for a, b in zip(a_set, b_set):
            if a is not None:
                assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


@pytest.mark.parametrize("R,T,H", [(2, 60, 16384), (8, 60, 12288), (1, 70, 8320), (12, 70, 16384)])
def test_wide_fp8_rows_on_clusters(R, T, H):
    """FP8 output on rows wider than 8192 below half a wave: the planner takes
    the row kernel's clusters; every row against the oracle, and the same bits
    as the stream kernel."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = frn.plan_launch(T, H, R, 1, True, sms)
    assert plan["kernel"] == frn.KERNEL_ROWS and plan["ctas_per_row"] > 1, plan
    inp = syn.make_inputs(R, T, H, seed=60 + R, partial_std=0.5)
    check_quant(inp, f"wide FP8 R={R} T={T} H={H}")
    d = DevInputs(inp)
    rows = [gpu_quant(d, True), gpu_quant(d, False)]
    frn.set_kernel(frn.KERNEL_STREAM)
    try:
        stream = [gpu_quant(d, True), gpu_quant(d, False)]
    finally:
        frn.set_kernel(frn.KERNEL_AUTO)
    for a_set, b_set in zip(rows, stream):
        for a, b in zip(a_set, b_set):
            if a is not None:
                assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))
