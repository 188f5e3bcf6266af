"""The C-ABI library builds, loads on a machine without a GPU, exports every entry point
that include/moe.h declares, and rejects bad arguments on the host before touching a
device. No compute call runs here."""
import ctypes as C
import os
import subprocess

import pytest

import grouped_expert_ffn_gb300 as moe
from grouped_expert_ffn_gb300 import build as moe_build


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def test_exports_every_declared_symbol(lib):
    syms = moe.header_symbols()
    assert len(syms) >= 14
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [s for s in syms if s not in exported]
    assert not missing, missing
    for s in syms:
        assert hasattr(lib, s)


def test_status_strings(lib):
    for code in range(9):
        assert moe.status_string(code)
    assert moe.status_string(0) == "ok"


def test_plan_rejects_bad_shapes_on_host(lib):
    h = C.c_void_p()
    bad = [(0, 1, 64, 64, 0, 8), (8, 9, 64, 64, 0, 8), (8, 2, 64, 64, 0, 0), (8, 2, -64, 64, 0, 8),
           (8, 2, 64, 64, -64, 8)]
    for args in bad:
        assert lib.moe_plan(*args, C.byref(h)) == moe.MOE_ERR_INVALID_ARG, args
    unsup = [(300, 2, 64, 64, 0, 8), (8, 2, 100, 64, 0, 8), (8, 2, 64, 96, 0, 8),
             (8, 2, 64, 64, 32, 8), (16, 9, 64, 64, 0, 8), (8, 2, 16384, 64, 0, 8)]
    for args in unsup:
        assert lib.moe_plan(*args, C.byref(h)) == moe.MOE_ERR_UNSUPPORTED, args
    assert lib.moe_plan(8, 2, 64, 64, 0, 8, None) == moe.MOE_ERR_INVALID_ARG


def test_plan_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = C.c_void_p()
    assert lib.moe_plan(8, 2, 256, 128, 0, 16, C.byref(h)) == moe.MOE_ERR_NO_DEVICE
    assert h.value is None


def test_null_handles_rejected(lib):
    assert lib.moe_route(None, None, 4, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_forward(None, None, None, 4, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route_forward(None, None, None, 4, None, None, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_plan_destroy(None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_plan_set_decode_rows(None, 8) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_packed_destroy(None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_weights_nvfp4(None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_get_error(None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_tap_bytes(None, 0) == 0
    assert lib.moe_router_logits(None, None, 4, 64, 8, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_residual_add(None, None, 4, 64, None) == moe.MOE_ERR_INVALID_ARG
    # misaligned pointers are rejected before any launch
    assert lib.moe_router_logits(16 + 2, 32, 4, 64, 8, 64, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_residual_add(18, 32, 4, 64, None) == moe.MOE_ERR_INVALID_ARG


def test_binding_refuses_host_and_strided_tensors(lib):
    import torch
    import grouped_expert_ffn_gb300 as moe
    lg = torch.zeros((4, 8), dtype=torch.float32)
    idx = torch.zeros((4, 2), dtype=torch.int32)
    w = torch.zeros((4, 2), dtype=torch.float32)
    with pytest.raises(ValueError, match="not CUDA"):
        moe.moe_route(1, lg, idx, w, stream=0)
    with pytest.raises(ValueError, match="not contiguous"):
        moe.moe_route(1, torch.zeros((8, 4)).t(), idx, w, stream=0)
    with pytest.raises(ValueError, match="not CUDA"):
        moe.moe_residual_add(torch.zeros((2, 8), dtype=torch.bfloat16), torch.zeros((2, 8)), stream=0)
