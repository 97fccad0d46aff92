"""Every entry point inside a CUDA graph, and several streams (and host
threads) calling the library at once: the results are the bits of plain eager
calls on one stream."""
import threading

import numpy as np
import pytest
import torch

import reduce_residual_rmsnorm_fp32_gb300 as frn
from reduce_residual_rmsnorm_fp32_gb300 import synthetic as syn
from frn_testlib import DevInputs

pytestmark = pytest.mark.gpu


def _all_entry_points(d, out):
    """One call of every entry point, writing into the preallocated `out` dict."""
    p, r, g, eps = d.partials, d.residual, d.gamma, d.eps
    frn.fused_reduce_rmsnorm(p, r, g, eps, residual_out=out["ro"], y=out["y"])
    frn.fused_reduce_rmsnorm_quant_per_group(p, r, g, eps, 128, True, residual_out=out["ro_q"], y=out["y_q"],
                                             q=out["q"], scales=out["s"])
    frn.fused_reduce_rmsnorm_mxfp4(p, r, g, eps, False, residual_out=out["ro_mx"], q=out["q4"],
                                   scales=out["e8"])
    frn.fused_add_rmsnorm(p[0], r, g, eps, residual_out=out["ro_add"], y=out["y_add"])
    frn.rmsnorm(p[0], g, eps, y=out["y_rms"])
    frn.unfused_reduce_rmsnorm(p, r, g, eps, stages=3, quant=True, emit_bf16=True, group_size=128,
                               workspace=out["ws"], residual_out=out["ro_u"], y=out["y_u"], q=out["q_u"],
                               scales=out["s_u"])


def _outputs(T, H, ws_bytes):
    bf = lambda: torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    return {"ro": bf(), "y": bf(), "ro_q": bf(), "y_q": bf(),
            "q": torch.empty((T, H), dtype=torch.float8_e4m3fn, device="cuda"),
            "s": torch.empty((T, H // 128), dtype=torch.float32, device="cuda"),
            "ro_mx": bf(), "q4": torch.empty((T, H // 2), dtype=torch.uint8, device="cuda"),
            "e8": torch.empty((T, H // 32), dtype=torch.uint8, device="cuda"),
            "ro_add": bf(), "y_add": bf(), "y_rms": bf(), "ro_u": bf(), "y_u": bf(),
            "q_u": torch.empty((T, H), dtype=torch.float8_e4m3fn, device="cuda"),
            "s_u": torch.empty((T, H // 128), dtype=torch.float32, device="cuda"),
            "ws": torch.empty((ws_bytes,), dtype=torch.uint8, device="cuda")}


def _same(a, b):
    for k in a:
        if k == "ws":
            continue
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k


@pytest.mark.parametrize("T,H", [(16, 7168), (700, 1024), (300, 4096)])
def test_every_entry_point_in_a_cuda_graph(T, H):
    d = DevInputs(syn.make_inputs(4, T, H, seed=31 + T, partial_std=0.5))
    ws = frn.unfused_workspace_bytes(T, H, 3, True, True)
    eager, graphed = _outputs(T, H, ws), _outputs(T, H, ws)
    _all_entry_points(d, eager)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _all_entry_points(d, graphed)          # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for v in graphed.values():
        v.zero_()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        _all_entry_points(d, graphed)
    for _ in range(3):
        gr.replay()
    torch.cuda.synchronize()
    _same(eager, graphed)


def test_concurrent_streams_and_host_threads():
    """Four host threads, each with its own CUDA stream and buffers, call every
    entry point 20 times; each thread's results are the eager single-stream ones."""
    T, H = 40, 7168
    inputs = [DevInputs(syn.make_inputs(2 + i, T, H, seed=40 + i, partial_std=0.5)) for i in range(4)]
    ws = frn.unfused_workspace_bytes(T, H, 3, True, True)
    ref = []
    for d in inputs:
        o = _outputs(T, H, ws)
        _all_entry_points(d, o)
        ref.append(o)
    torch.cuda.synchronize()
    outs = [_outputs(T, H, ws) for _ in inputs]
    errors = []

    def work(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(20):
                    _all_entry_points(inputs[i], outs[i])
            st.synchronize()
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for a, b in zip(ref, outs):
        _same(a, b)
    assert frn.device_status() == frn.FRN_OK
