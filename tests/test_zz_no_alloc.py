"""The allocation-free batched-decode entry point, moe_forward_decode_static.

Callers that cannot allocate device memory on their call path (a stream being captured into
a CUDA graph, a plugin whose host runtime owns every device allocation, a serving loop that
cannot take cudaMalloc's implicit device synchronisation) use this entry point instead of a
plan: its scratch lives in a fixed-size array inside the library. These tests call it
through the C ABI and hold its output to the plan-based moe_forward on the same inputs,
twice in a row, so the second call runs over the scratch contents the first one left.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import synth
import grouped_expert_ffn_gb300 as moe
from helpers import Y_MAX_REL, Y_RMSE_REL, weights_to, y_errors


def test_host_side_limits_need_no_gpu():
    lib = moe.lib()
    ws = moe.Weights(*([16] * 12))
    # more rows than the decode kernels take, and unsupported shapes, are refused on the host
    assert lib.moe_forward_decode_static(8, 2, 256, 128, 0, C.byref(ws), 16, 9, 16, 16, 16,
                                         None, None) == moe.MOE_ERR_CAPACITY
    assert lib.moe_forward_decode_static(8, 2, 100, 128, 0, C.byref(ws), 16, 4, 16, 16, 16,
                                         None, None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_forward_decode_static(300, 2, 256, 128, 0, C.byref(ws), 16, 4, 16, 16, 16,
                                         None, None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_forward_decode_static(8, 2, 256, 128, 0, None, 16, 4, 16, 16, 16,
                                         None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_decode_static(8, 2, 256, 128, 0, C.byref(ws), 18, 4, 16, 16, 16,
                                         None, None) == moe.MOE_ERR_INVALID_ARG


@pytest.mark.gpu
def test_static_decode_matches_moe_forward_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    wl = synth.WORKLOADS["decode"]
    sh = wl.shape
    d = synth.make_layer(wl, device="cpu")
    W = weights_to(d["weights"], "cuda")
    ws = moe.make_weights_struct(W)
    lay = moe.MoELayer(sh.E, sh.k, sh.H, sh.I, sh.Is, sh.T, W)
    lib = moe.lib()
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    second = synth.small_layer(5, sh.H, sh.E, sh.k, sh.I, sh.Is, seed=77, zipf_s=1.1, outliers=8)
    try:
        for x_cpu, lg_cpu in ((d["x"], d["logits"]), (second["x"], second["logits"])):
            T = x_cpu.shape[0]
            x = x_cpu.cuda()
            idx, w = lay.route(lg_cpu.cuda())
            y_ref = lay.forward(x, idx, w)
            y = torch.full((T, sh.H), float("nan"), device="cuda")
            st = lib.moe_forward_decode_static(
                sh.E, sh.k, sh.H, sh.I, sh.Is, C.byref(ws), x.data_ptr(), T, idx.data_ptr(),
                w.data_ptr(), y.data_ptr(), status.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
            assert st == moe.MOE_OK
            torch.cuda.synchronize()
            assert status[0].item() == 0
            assert torch.isfinite(y).all()
            mx, rm = y_errors(y.cpu().numpy(), y_ref.cpu().numpy().astype(np.float64))
            assert mx <= Y_MAX_REL and rm <= Y_RMSE_REL, (mx, rm)
    finally:
        lay.close()
