"""The launch planner's shapes, checked on the CPU for every hidden size.

frn_plan_launch runs the library's own kernel and launch-shape choice for a
given SM count without touching a device.  Every plan must fit the kernel
variant it selects: tiles covered with no empty CTA, thread counts within the
launch bounds of the instantiation the dispatcher picks, shared memory within
the opt-in limit, grids as the kernels index them."""
import itertools

import pytest

import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import _build

SMEM_LIMIT = 232448
TS = (1, 3, 8, 16, 33, 64, 127, 200, 300, 608, 1171, 2500, 8192, 65536)


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return frn.library()


def _check_plan(pl, T, H, R, quant, residual, sms, auto=True):
    ntiles = -(-(H // 8) // 32)
    what = (T, H, R, quant, residual, sms, pl)
    if auto and (ntiles <= 16 or (ntiles <= 32 and R <= 8)):
        assert pl["kernel"] == frn.KERNEL_ROWS, what                    # every row that fits one CTA
    if auto and ntiles > 32 and R <= 8 and 2 * T >= sms and not (quant == 3 and R <= 2):
        assert pl["kernel"] == frn.KERNEL_ROWS and pl["tiles_per_warp"] == 2, what
    if auto and 8 < ntiles <= 16 and R > 8:                            # against the staged CTA
        two = 2 * T >= sms and (R <= 10 or (R <= 12 and quant != 0 and T >= 3 * sms))
        assert pl["tiles_per_warp"] == (2 if two else 1) and (not two or not pl["staged"]), what
    if auto and ntiles > 16 and R > 8:                                  # no one-tile-a-warp CTA holds the row
        two = (quant in (1, 2) or ntiles <= 22) and 2 * T >= sms
        if two:
            assert pl["kernel"] == frn.KERNEL_ROWS and pl["tiles_per_warp"] == 2, what
        else:
            assert pl["kernel"] == frn.KERNEL_STREAM or pl["tiles_per_warp"] == 1, what
    if auto and 17 <= ntiles <= 32 and R <= 8:                          # rows a wide CTA could hold
        two = ntiles >= 26 and ((R in (3, 4) and T > sms) or (R == 2 and quant == 1 and T >= 16 * sms) or
                                (R >= 5 and sms < T and 20 * T <= 33 * sms))
        assert pl["tiles_per_warp"] == (2 if two else 1), what
    if pl["kernel"] == frn.KERNEL_ROWS:
        C, tpc, rows, thr = pl["ctas_per_row"], pl["tiles_per_cta"], pl["rows_per_cta"], pl["threads"]
        assert 1 <= C <= 16 and tpc >= 1 and rows >= 1, what
        assert C * tpc >= ntiles and (C - 1) * tpc < ntiles, what          # every tile, no empty CTA
        if pl["tiles_per_warp"] == 2:                                      # two tiles a warp, one CTA a row
            assert C == 1 and rows == 1 and tpc <= 64, what
            assert tpc > 32 or (tpc >= 26 and 2 <= R <= 8) or (tpc > 8 and R > 8), what
            assert thr == -(-tpc // 2) * 32 and not pl["staged"], what
        else:
            assert pl["tiles_per_warp"] == 1 and thr == rows * tpc * 32 and thr <= 1024, what
        assert tpc <= (64 if pl["tiles_per_warp"] == 2 else 32), what     # per-CTA tile-sum slots
        if rows > 1:                                                       # packed 256-thread variant
            assert C == 1 and tpc == ntiles and thr <= 256, what
        if thr > 512:                                                      # wide or two-tile: one CTA
            assert C == 1 and rows == 1 and (R <= 8 or pl["tiles_per_warp"] == 2), what
        if C > 1:                                                          # cluster variant: <= 512 threads
            assert thr <= 512 and rows == 1 and C <= 8, what
        assert pl["grid"] == -(-T // rows) * C, what
        assert pl["smem_bytes"] == 0, what
        if pl["staged"]:                                                   # staged loads: one CTA a row
            assert C == 1 and rows == 1 and R > 8 and ntiles <= 16 and T >= 3 * sms, what
    else:
        tpw, nc, g, slots = pl["tiles_per_warp"], pl["consumer_warps"], pl["groups"], pl["slots"]
        nslices = R + (1 if residual else 0)
        assert tpw in (1, 2, 4) and nc * tpw >= ntiles and (nc - 1) * tpw < ntiles, what
        assert 1 <= g <= 4 and pl["threads"] == (g * nc + 1) * 32 <= 704, what
        if pl["threads"] > 512:                                            # 544 / 704 variants are TPW 4
            assert tpw == 4, what
        assert g <= slots <= 32 and slots * 2 * H <= pl["smem_bytes"] <= SMEM_LIMIT, what
        assert pl["grid"] == min(T, sms), what
        assert nslices >= 1, what


def test_every_hidden_size_plans_a_valid_launch():
    n = 0
    for H in range(8, 16385, 8):
        for R, T in itertools.product((1, 2, 3, 4, 5, 6, 8, 10, 12, 16), TS):
            quants = [0] + ([1, 2] if H % 128 == 0 else []) + ([3, 4] if H % 32 == 0 else [])
            for quant in quants:
                for residual in (True, False):
                    if quant and not residual and H % 512:
                        continue   # thin the sample: residual-free quant on a quarter of H
                    pl = frn.plan_launch(T, H, R, quant, residual, 152)
                    _check_plan(pl, T, H, R, quant, residual, 152)
                    n += 1
    assert n > 300000, n


@pytest.mark.parametrize("sms", [1, 8, 132, 148])
def test_other_sm_counts(sms):
    for H, R, T in itertools.product(range(256, 16385, 1280), (1, 2, 4, 5, 8, 10, 16), TS):
        for residual in (True, False):
            _check_plan(frn.plan_launch(T, H, R, 0, residual, sms), T, H, R, 0, residual, sms)


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 8, 12, 16])
def test_forced_cluster_sizes(ctas):
    frn.set_kernel(frn.KERNEL_ROWS)
    frn.set_ctas_per_row(ctas)
    try:
        for H, R, T in itertools.product(range(8, 16385, 136), (1, 2, 8, 16), (1, 64, 4096)):
            pl = frn.plan_launch(T, H, R, 0, True, 152)
            ntiles = -(-(H // 8) // 32)
            assert pl["kernel"] == frn.KERNEL_ROWS
            C, tpc = pl["ctas_per_row"], pl["tiles_per_cta"]
            assert C * tpc >= ntiles and (C - 1) * tpc < ntiles and 1 <= C <= 16
            assert pl["threads"] <= (1024 if C == 1 else 512)
    finally:
        frn.set_ctas_per_row(0)
        frn.set_kernel(frn.KERNEL_AUTO)


def test_forced_stream_groups():
    frn.set_kernel(frn.KERNEL_STREAM)
    try:
        for groups in (1, 2, 3, 4):
            frn.set_stream_groups(groups)
            for H, R in itertools.product(range(8, 16385, 264), (1, 2, 8, 16)):
                pl = frn.plan_launch(4096, H, R, 0, True, 152)
                _check_plan(pl, 4096, H, R, 0, True, 152, auto=False)
                assert pl["groups"] <= groups
    finally:
        frn.set_stream_groups(0)
        frn.set_kernel(frn.KERNEL_AUTO)


def test_plan_rejects_bad_sizes():
    for args in ((0, 256, 2), (4, 100, 2), (4, 256, 0), (4, 256, 17), (4, 16392, 2)):
        with pytest.raises(frn.FrnError):
            frn.plan_launch(*args)


def test_query_launch_checks_sizes_then_needs_a_device():
    """frn_query_launch is frn_plan_launch with the current device's SM count:
    bad sizes are refused before any device is touched, and on a host without
    a GPU the SM-count lookup fails with FRN_ERR_CUDA."""
    import ctypes
    import torch
    lib = frn.library()
    k = ctypes.c_int()
    for bad in ((8, 7168, 0, 0), (8, 7168, 17, 0), (-1, 7168, 8, 0), (8, 7100, 8, 0), (8, 7168, 8, 5)):
        assert lib.frn_query_launch(*bad, 1, ctypes.byref(k), None, None, None) == frn.FRN_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert lib.frn_query_launch(8, 7168, 8, 0, 0, ctypes.byref(k), None, None, None) == frn.FRN_ERR_CUDA


def test_staged_plans():
    """Staged partial loads where they measured faster: R > 8 rows of up to 16
    tiles from three waves.  Wide rows (17-32 tiles, R <= 8) take the row
    kernel with every output at every T, loading all partials at once: a wide
    CTA a row, or, for 26..32 tiles with R = 3 or 4 beyond one row per SM,
    two tiles a warp on half the threads."""
    pl = frn.plan_launch(600, 4096, 16, 0, True, 152)
    assert pl["kernel"] == frn.KERNEL_ROWS and pl["staged"] == 1 and pl["threads"] == 512
    assert frn.plan_launch(300, 4096, 16, 0, True, 152)["staged"] == 0
    for quant in (0, 1, 2, 3, 4):
        for R, T in ((8, 586), (8, 1000), (5, 586), (4, 1519), (8, 1063), (8, 4682), (3, 1171), (4, 152),
                     (8, 200), (6, 250), (8, 251), (7, 152)):
            pl = frn.plan_launch(T, 7168, R, quant, True, 152)
            two = T > 152 and (R <= 4 or T <= 250)
            assert pl["kernel"] == frn.KERNEL_ROWS and pl["staged"] == 0, (R, T, quant)
            assert pl["threads"] == (448 if two else 896) and pl["tiles_per_warp"] == (2 if two else 1), (R, T, quant)
        # R = 2: two tiles a warp only with an FP8 output without y from 16 rows an SM
        assert frn.plan_launch(2432, 7168, 2, quant, True, 152)["tiles_per_warp"] == (2 if quant == 1 else 1)
        assert frn.plan_launch(2431, 7168, 2, quant, True, 152)["tiles_per_warp"] == 1
        # 25 tiles or fewer: two wide CTAs already fit an SM
        assert frn.plan_launch(1171, 6400, 4, quant, True, 152)["tiles_per_warp"] == 1
        assert frn.plan_launch(1171, 6656, 4, quant, True, 152)["threads"] == 13 * 32
    # rows wider than one CTA at many rows: one CTA a row, two tiles a warp, with R <= 8
    for quant in (0, 1, 3):
        pl = frn.plan_launch(1000, 16384, 8, quant, True, 152)
        assert pl["kernel"] == frn.KERNEL_ROWS and pl["tiles_per_warp"] == 2, quant
    # R > 8: two tiles a warp with an FP8 output, or up to 22 tiles; else the stream kernel
    assert frn.plan_launch(1000, 8192, 16, 0, True, 152)["kernel"] == frn.KERNEL_STREAM
    assert frn.plan_launch(1000, 16384, 12, 4, True, 152)["kernel"] == frn.KERNEL_STREAM
    assert frn.plan_launch(1000, 6144, 9, 3, True, 152)["kernel"] == frn.KERNEL_STREAM
    for R, H, quant in ((16, 8192, 1), (12, 16384, 2), (9, 5120, 0), (16, 5632, 4), (10, 4104, 3)):
        pl = frn.plan_launch(1000, H, R, quant, True, 152)
        assert pl["kernel"] == frn.KERNEL_ROWS and pl["tiles_per_warp"] == 2, (R, H, quant)
    assert frn.plan_launch(75, 16384, 16, 1, True, 152)["ctas_per_row"] == 4        # few rows: clusters
    assert frn.plan_launch(75, 5120, 16, 0, True, 152)["kernel"] == frn.KERNEL_ROWS
    for quant in (0, 1, 2, 4):
        pl = frn.plan_launch(8192, 16384, 2, quant, True, 152)
        assert pl["kernel"] == frn.KERNEL_ROWS and pl["tiles_per_warp"] == 2 and pl["threads"] == 1024
    assert frn.plan_launch(8192, 16384, 2, 3, True, 152)["kernel"] == frn.KERNEL_STREAM   # MXFP4 without y
    for R, quant in ((3, 0), (4, 1), (4, 3), (4, 4)):
        assert frn.plan_launch(4096, 16384, R, quant, True, 152)["tiles_per_warp"] == 2, (R, quant)
    for R in (5, 8):   # R = 5..8 in stages of four, every output
        for quant in (0, 2, 4):
            assert frn.plan_launch(2048, 16384, R, quant, True, 152)["tiles_per_warp"] == 2, (R, quant)
    assert frn.plan_launch(8192, 10000, 1, 0, True, 152)["threads"] == 20 * 32    # 40 tiles, ragged
    assert frn.plan_launch(75, 16384, 2, 0, True, 152)["tiles_per_warp"] == 1     # few rows: clusters
    assert frn.plan_launch(76, 16384, 4, 1, True, 152)["tiles_per_warp"] == 2


def test_cluster_sizes_for_heavy_rows():
    """Rows of more than 96 KB of loads spread over clusters at small T (up to
    7 CTAs at T <= 5, 4 up to T = 16, 2 up to T = 40), a divisor of the tile
    count; lighter rows, and heavy rows from T = 41 on, keep one CTA a row."""
    expect = {3: 7, 5: 7, 6: 4, 8: 4, 16: 4, 17: 2, 32: 2, 40: 2, 41: 1, 64: 1}
    for T, C in expect.items():
        assert frn.plan_launch(T, 7168, 8, 0, True, 152)["ctas_per_row"] == C, T
    assert frn.plan_launch(3, 4096, 8, 0, True, 152)["ctas_per_row"] == 1      # 72 KB a row
    assert frn.plan_launch(3, 16384, 2, 0, True, 152)["ctas_per_row"] == 4     # 7 does not divide 64 tiles
