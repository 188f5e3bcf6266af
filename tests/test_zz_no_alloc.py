"""The allocation-free batched-decode entry point, moe_forward_decode_static.

Some callers cannot allocate device memory on their call path: a plugin whose host runtime
owns every device allocation and forbids its guests from calling cudaMalloc, or a serving
loop that cannot take cudaMalloc's implicit device synchronisation between steps. They use
this entry point instead of a plan: its scratch lives in a fixed-size array inside the
library. These tests call it through the C ABI and hold its output to the plan-based
moe_forward on the same inputs and to the CPU oracle, twice in a row per shape, so that the
second call runs over the scratch contents the first one left. This file is collected last,
so a run that stops at the first failure has already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import synth
import grouped_expert_ffn_gb300 as moe
from helpers import Y_MAX_REL, Y_RMSE_REL, oracle_layer, weights_to, y_errors


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


def _two_calls(sh, first, second):
    W = weights_to(first["weights"], "cuda")
    L = oracle_layer(first["weights"], sh)
    ws = moe.make_weights_struct(W)
    lay = moe.MoELayer(sh.E, sh.k, sh.H, sh.I, sh.Is, 8, W)
    lib = moe.lib()
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    try:
        for x_cpu, lg_cpu in ((first["x"], first["logits"]), (second["x"], second["logits"])):
            T = x_cpu.shape[0]
            x = x_cpu.cuda()
            idx, w = lay.route(lg_cpu.cuda())
            y_plan = lay.forward(x, idx, w)
            y = torch.full((T, sh.H), float("nan"), device="cuda")
            st = lib.moe_forward_decode_static(
                sh.E, sh.k, sh.H, sh.I, sh.Is, C.byref(ws), x.data_ptr(), T, idx.data_ptr(),
                w.data_ptr(), y.data_ptr(), status.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
            assert st == moe.MOE_OK
            torch.cuda.synchronize()
            assert status[0].item() == 0
            assert torch.isfinite(y).all()
            yh = y.cpu().numpy().astype(np.float64)
            # against the plan-based entry point on the same inputs
            mx, rm = y_errors(yh, y_plan.cpu().numpy().astype(np.float64))
            assert mx <= Y_MAX_REL and rm <= Y_RMSE_REL, (mx, rm)
            # and against the oracle (its own routing of the same logits)
            idx_o, w_o = oracle.route(lg_cpu, sh.k)
            assert (idx.cpu().numpy() == idx_o).all()
            y_o = oracle.forward(L, x_cpu, idx_o, w_o)
            mx, rm = y_errors(yh, y_o)
            assert mx <= Y_MAX_REL and rm <= Y_RMSE_REL, (mx, rm)
    finally:
        lay.close()


@pytest.mark.gpu
def test_static_decode_matches_moe_forward_and_oracle_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    wl = synth.WORKLOADS["decode"]
    sh = wl.shape
    first = synth.make_layer(wl, device="cpu")
    second = synth.small_layer(5, sh.H, sh.E, sh.k, sh.I, sh.Is, seed=77, zipf_s=1.1, outliers=8)
    _two_calls(sh, first, second)


@pytest.mark.gpu
@pytest.mark.parametrize("Is", [0, 384])
def test_static_decode_without_and_with_a_wider_shared_expert(Is):
    # no shared expert, and a shared expert wider than the routed ones (I_shared > I)
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    sh = synth.LayerShape(T=8, H=512, E=32, k=4, I=256, Is=Is)
    first = synth.small_layer(8, sh.H, sh.E, sh.k, sh.I, Is, seed=51 + Is, zipf_s=1.1)
    second = synth.small_layer(3, sh.H, sh.E, sh.k, sh.I, Is, seed=52 + Is, zipf_s=1.1)
    _two_calls(sh, first, second)
