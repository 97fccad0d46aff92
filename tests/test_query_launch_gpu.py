"""frn_query_launch on a GPU reports exactly what frn_plan_launch plans for the
device's SM count, with and without a residual (the stream kernel streams
R + 1 slices a row when a residual is passed, R otherwise)."""
import itertools

import pytest
import torch

import reduce_residual_rmsnorm_fp32_gb300 as frn

pytestmark = pytest.mark.gpu


def test_query_matches_plan_with_and_without_residual():
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    for T, H, R, quant, residual in itertools.product((1, 8, 64, 300, 1171, 8192), (256, 4096, 7168, 16384),
                                                      (1, 2, 8), (0, 1, 2, 3, 4), (True, False)):
        q = frn.query_launch(T, H, R, quant, residual)
        p = frn.plan_launch(T, H, R, quant, residual, sms)
        assert q == (p["kernel"], p["ctas_per_row"], p["threads"], p["grid"]), (T, H, R, quant, residual)
    assert frn.query_launch(0, 7168, 8)[3] == 0
