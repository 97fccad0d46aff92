"""The C ABI on a CPU host (no GPU): the library loads, exports every function
include/frn.h declares, and its host-side validation answers without touching
a device.  No call here launches a kernel."""
import ctypes
import os
import re

import pytest
import torch

import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "frn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return frn.library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fused_reduce_rmsnorm", "fused_reduce_rmsnorm_quant_per_group", "frn_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", frn.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.split() and l.split()[1] == "T"}
    ours = {n for n in exported if n.startswith("frn_") or n.startswith("fused_")}
    assert ours == set(declared_functions())


def test_status_strings_and_version(lib):
    assert frn.status_string(frn.FRN_OK) == "FRN_OK"
    assert frn.status_string(frn.FRN_ERR_CUDA) == "FRN_ERR_CUDA"
    assert frn.status_string(99) == "FRN_ERR_UNKNOWN"
    assert frn.version() >= 20000


def _call(lib, R=2, ptrs=(0x1000, 0x2000), res=0x3000, gamma=0x4000, ro=0x10000000, y=0x20000000, T=4, H=256,
          eps=1e-6):
    arr = (ctypes.c_void_p * max(len(ptrs), 1))(*ptrs)
    return lib.fused_reduce_rmsnorm(arr, R, res, gamma, ro, y, T, H, eps, None)


@pytest.mark.parametrize("kw,want", [
    (dict(R=0), frn.FRN_ERR_INVALID_ARG),
    (dict(R=17), frn.FRN_ERR_UNSUPPORTED),
    (dict(T=-3), frn.FRN_ERR_INVALID_ARG),
    (dict(H=0), frn.FRN_ERR_INVALID_ARG),
    (dict(H=100), frn.FRN_ERR_UNSUPPORTED),
    (dict(H=16392), frn.FRN_ERR_UNSUPPORTED),
    (dict(eps=float("inf")), frn.FRN_ERR_INVALID_ARG),
    (dict(eps=-1e-6), frn.FRN_ERR_INVALID_ARG),
    (dict(ptrs=(0x1000, 0)), frn.FRN_ERR_INVALID_ARG),
    (dict(ptrs=(0x1000, 0x2008)), frn.FRN_ERR_MISALIGNED),
    (dict(gamma=0), frn.FRN_ERR_INVALID_ARG),
    (dict(gamma=0x4004), frn.FRN_ERR_MISALIGNED),
    (dict(ro=0), frn.FRN_ERR_INVALID_ARG),
    (dict(y=0), frn.FRN_ERR_INVALID_ARG),
    (dict(y=0x10000010), frn.FRN_ERR_INVALID_ARG),     # y overlaps residual_out
    (dict(ro=0x1000), frn.FRN_ERR_INVALID_ARG),        # residual_out overlaps a partial
    (dict(ro=0x3010), frn.FRN_ERR_INVALID_ARG),        # partial overlap with the residual
    (dict(y=0x4000), frn.FRN_ERR_INVALID_ARG),         # y overlaps gamma
])
def test_validation_rejects_before_any_cuda_call(lib, kw, want):
    st = _call(lib, **kw)
    assert st == want, (kw, frn.status_string(st), lib.frn_last_error_detail())
    assert lib.frn_last_error_detail()


def test_quant_validation(lib):
    arr = (ctypes.c_void_p * 1)(0x1000)
    f = lib.fused_reduce_rmsnorm_quant_per_group
    assert f(arr, 1, None, 0x4000, 0x10000000, None, 0x20000000, 0x30000000, 4, 256, 1e-6, 64, None) \
        == frn.FRN_ERR_UNSUPPORTED
    assert f(arr, 1, None, 0x4000, 0x10000000, None, 0x20000000, 0x30000000, 4, 256, 1e-6, 96, None) \
        == frn.FRN_ERR_INVALID_ARG
    assert f(arr, 1, None, 0x4000, 0x10000000, None, 0x20000008, 0x30000000, 4, 256, 1e-6, 128, None) \
        == frn.FRN_ERR_MISALIGNED
    assert f(arr, 1, None, 0x4000, 0x10000000, None, 0x20000000, 0x30000002, 4, 256, 1e-6, 128, None) \
        == frn.FRN_ERR_MISALIGNED
    assert f(arr, 1, None, 0x4000, 0x10000000, None, None, 0x30000000, 4, 256, 1e-6, 128, None) \
        == frn.FRN_ERR_INVALID_ARG


def test_empty_T_is_ok_without_device(lib):
    assert _call(lib, T=0, ptrs=(0, 0), res=0, gamma=0, ro=0, y=0) == frn.FRN_OK


def test_launch_controls(lib):
    assert lib.frn_set_pdl(0) == frn.FRN_OK and lib.frn_set_pdl(1) == frn.FRN_OK
    assert lib.frn_set_ctas_per_row(17) == frn.FRN_ERR_INVALID_ARG
    assert lib.frn_set_ctas_per_row(3) == frn.FRN_OK and lib.frn_set_ctas_per_row(0) == frn.FRN_OK
    assert lib.frn_set_l2_prefetch(3) == frn.FRN_ERR_INVALID_ARG and lib.frn_set_l2_prefetch(-1) == frn.FRN_ERR_INVALID_ARG
    assert lib.frn_set_l2_prefetch(1) == frn.FRN_OK and lib.frn_set_l2_prefetch(0) == frn.FRN_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error path; a GPU would run the call")
def test_no_device_maps_to_cuda_error(lib):
    """A well-formed call on a host without a usable GPU fails with FRN_ERR_CUDA
    (the runtime's own error) instead of crashing."""
    st = _call(lib)
    assert st == frn.FRN_ERR_CUDA, frn.status_string(st)
    assert "cuda" in lib.frn_last_error_detail().decode().lower()


def test_binding_rejects_host_inputs():
    """Inputs must be CUDA tensors: the binding refuses host tensors before any
    library call (no CPU fallback)."""
    p = torch.zeros((2, 4, 256), dtype=torch.bfloat16)
    g = torch.ones((256,), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="must be on"):
        frn.fused_reduce_rmsnorm(p, None, g, 1e-6)
    with pytest.raises(ValueError, match="must be on"):
        frn.fused_reduce_rmsnorm_quant_per_group(p, None, g, 1e-6)


def test_floor_launch_validates_without_launching(lib):
    """Bad arguments to the measurement kernels are refused on the host."""
    arr = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    assert lib.frn_floor_launch(3, arr, 2, None, None, 64, 128, 1, 1, None) == frn.FRN_ERR_INVALID_ARG
    assert lib.frn_floor_launch(1, arr, 2, None, None, 64, 100, 1, 1, None) == frn.FRN_ERR_INVALID_ARG
    assert lib.frn_floor_launch(1, arr, 0, None, None, 64, 128, 1, 1, None) == frn.FRN_ERR_INVALID_ARG
    assert lib.frn_floor_launch(1, arr, 2, None, None, 40, 128, 1, 1, None) == frn.FRN_ERR_INVALID_ARG
    assert lib.frn_floor_launch(2, arr, 2, 0x3000, None, 64, 128, 1, 1, None) == frn.FRN_ERR_INVALID_ARG
    bad = (ctypes.c_void_p * 2)(0x1000, 0x2008)
    assert lib.frn_floor_launch(1, bad, 2, None, None, 64, 128, 1, 1, None) == frn.FRN_ERR_MISALIGNED
    assert lib.frn_floor_launch(0, None, 0, None, None, 0, 128, 0, 1, None) == frn.FRN_ERR_INVALID_ARG
