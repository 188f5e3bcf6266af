"""GPU parity of the layer with NVFP4 expert weights (E2M1 codes, E4M3 block scales per 16
elements, fp32 matrix scales) against the CPU oracle's NVFP4 layer.

The weight-streaming kernels accumulate every row exactly (int64 in units of 2^-10), so the
fp64 accumulator taps must equal the oracle's exact sums bit for bit; the grouped tensor-core
GEMMs decode the weights exactly to fp16 and accumulate in fp32, so their accumulators are
held within 1e-4 * ||q|| * ||w'|| of the exact sums (q the activation or h codes, w' the
dequantised weight row without its matrix scale); the routing,
permutation and activation codes are bit-identical; requantised h codes may differ by one
at a rounding tie of exp (at most 1e-3 of them), and y is held to the int8 layer's
tolerances (max|dy| <= 1e-2 max|y_ref|, rms(dy) <= 5e-3 rms(y_ref))."""
import numpy as np
import pytest
import torch

import oracle
import synth
import grouped_expert_ffn_gb300 as moe
from helpers import check_layer, oracle_layer_nvfp4, weights_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.lib()


def _layer(T, H, E, k, I, Is, seed, zipf_s=1.1, outliers=8):
    sh = synth.LayerShape(T=T, H=H, E=E, k=k, I=I, Is=Is)
    d = synth.small_layer(T, H, E, k, I, Is, seed=seed, zipf_s=zipf_s, outliers=outliers)
    W = synth.make_weights_nvfp4(sh, seed)
    return sh, d, W


@pytest.mark.parametrize("T", [1, 3, 8, 9, 24, 64])
def test_nvfp4_decode_matches_the_oracle(T):
    # the 35B-A3B-shaped layer (H=2048, E=128, k=8, I=512, shared expert 512) with NVFP4
    # experts; above 8 rows an expert's rows take several passes
    sh, d, W = _layer(T, 2048, 128, 8, 512, 512, seed=90 + T)
    Wd = weights_to(W, "cuda")
    lay = moe.MoELayer(sh.E, sh.k, sh.H, sh.I, sh.Is, T, Wd)
    try:
        moe.moe_plan_set_decode_rows(lay.plan, 64)  # every T here on the streaming kernels
        st = check_layer(sh, d["x"], d["logits"], Wd, oracle_layer_nvfp4(W, sh), layer=lay)
        if T >= 24:
            assert st["tap"]["counts"].max() > 8  # some routed expert took more than one pass
    finally:
        lay.close()


def _random_bytes_weights(rng, E, H, I, Is):
    """Codes over every byte value, block scales over every finite non-negative E4M3 byte
    (zero, subnormals, 448) with whole zero-scale rows, matrix scales around 1e-3."""
    def codes(*s):
        return torch.from_numpy(rng.integers(0, 256, s).astype(np.uint8))

    def scales(*s):
        b = rng.integers(0, 127, s).astype(np.uint8)
        b.reshape(-1, s[-1])[::7] = 0  # every 7th row: all blocks zero
        return torch.from_numpy(b)

    def gs(*s):
        return torch.from_numpy(rng.uniform(5e-4, 2e-3, s).astype(np.float32))

    W = dict(w_gate=codes(E, I, H // 2), w_up=codes(E, I, H // 2), w_down=codes(E, H, I // 2),
             b_gate=scales(E, I, H // 16), b_up=scales(E, I, H // 16), b_down=scales(E, H, I // 16),
             g_gate=gs(E), g_up=gs(E), g_down=gs(E))
    if Is:
        W.update(sh_gate=codes(Is, H // 2), sh_up=codes(Is, H // 2), sh_down=codes(H, Is // 2),
                 sh_b_gate=scales(Is, H // 16), sh_b_up=scales(Is, H // 16),
                 sh_b_down=scales(H, Is // 16), sh_g=gs(3))
    return W


@pytest.mark.parametrize("T", [2, 8, 20])
def test_nvfp4_every_code_and_scale_byte(T):
    # full-range codes and block scales (subnormal and largest scales, zero blocks): the exact
    # int64 accumulation has no headroom problem and every decode rule is exercised
    H, E, k, I, Is = 512, 16, 4, 256, 128
    sh = synth.LayerShape(T=T, H=H, E=E, k=k, I=I, Is=Is)
    d = synth.small_layer(T, H, E, k, I, Is, seed=300 + T)
    W = _random_bytes_weights(np.random.default_rng(T), E, H, I, Is)
    check_layer(sh, d["x"], d["logits"], weights_to(W, "cuda"), oracle_layer_nvfp4(W, sh))


def test_nvfp4_largest_supported_shape():
    # H = 8192, I = I_shared = 4096: the largest exact sums the kernels form (a gate row sums
    # 8192 products); compared on every slot of 3 tokens
    T, H, E, k, I, Is = 3, 8192, 16, 4, 4096, 4096
    sh, d, W = _layer(T, H, E, k, I, Is, seed=310)
    check_layer(sh, d["x"], d["logits"], weights_to(W, "cuda"), oracle_layer_nvfp4(W, sh))


def test_nvfp4_route_forward_matches_route_then_forward():
    T, H, E, k, I, Is = 8, 2048, 128, 8, 512, 512
    sh, d, W = _layer(T, H, E, k, I, Is, seed=320)
    Wd = weights_to(W, "cuda")
    lay = moe.MoELayer(E, k, H, I, Is, T, Wd)
    try:
        x, lg = d["x"].cuda(), d["logits"].cuda()
        idx, w = lay.route(lg)
        y1 = lay.forward(x, idx, w)
        idx2 = torch.empty_like(idx)
        w2 = torch.empty_like(w)
        y2 = torch.empty_like(y1)
        moe.moe_route_forward(lay.plan, lay.packed, x, lg, idx2, w2, y2)
        torch.cuda.synchronize()
        assert moe.moe_get_error(lay.plan) == 0
        assert torch.equal(idx, idx2) and torch.equal(w, w2)
        assert (y1 - y2).abs().max().item() <= 1e-5 * y1.abs().max().item()
    finally:
        lay.close()


@pytest.mark.parametrize("bad", [0x7F, 0x80, 0xFE])
def test_nvfp4_bad_block_scale_sets_device_error(bad):
    # a NaN or negative block scale is found by the check moe_pack_weights_nvfp4 queues
    T, H, E, k, I = 4, 256, 8, 2, 128
    sh, d, W = _layer(T, H, E, k, I, 0, seed=330)
    W["b_down"][5, 17, 3] = bad
    lay = moe.MoELayer(E, k, H, I, 0, T, weights_to(W, "cuda"))
    try:
        assert moe.moe_get_error(lay.plan) == moe.MOE_ERR_DEVICE
        moe.moe_clear_error(lay.plan)
        assert moe.moe_get_error(lay.plan) == 0
    finally:
        lay.close()


@pytest.mark.parametrize("T", [40, 256])
def test_nvfp4_grouped_gemms_match_the_oracle(T):
    # above the decode threshold: the grouped tensor-core GEMMs (weights decoded exactly to
    # fp16, fp32 accumulation); T = 256 is the prefill chunk of the 35B-A3B-shaped layer
    sh, d, W = _layer(T, 2048, 128, 8, 512, 512, seed=350 + T)
    st = check_layer(sh, d["x"], d["logits"], weights_to(W, "cuda"), oracle_layer_nvfp4(W, sh),
                     acc_exact=False)
    assert st["tap"]["counts"].max() > 0


@pytest.mark.parametrize("T", [65, 77, 200])
def test_nvfp4_grouped_ragged_and_every_byte(T):
    # ragged token counts, a K (= I_shared = 192) that ends half-way through a 128-K stage,
    # and codes / block scales over every byte value
    H, E, k, I, Is = 512, 16, 4, 256, 192
    sh = synth.LayerShape(T=T, H=H, E=E, k=k, I=I, Is=Is)
    d = synth.small_layer(T, H, E, k, I, Is, seed=360 + T)
    W = _random_bytes_weights(np.random.default_rng(360 + T), E, H, I, Is)
    check_layer(sh, d["x"], d["logits"], weights_to(W, "cuda"), oracle_layer_nvfp4(W, sh),
                acc_exact=False)


def test_nvfp4_stream_and_grouped_paths_agree():
    # the same call through the exact streaming kernels and through the grouped GEMMs: the
    # permutation and activation codes are identical, the accumulators agree within the fp32
    # accumulation bound, y within the layer tolerance
    T, H, E, k, I, Is = 24, 2048, 128, 8, 512, 512
    sh, d, W = _layer(T, H, E, k, I, Is, seed=370)
    lay = moe.MoELayer(E, k, H, I, Is, T, weights_to(W, "cuda"))
    try:
        moe.moe_debug_enable(lay.plan, True)
        x = d["x"].cuda()
        idx, w = lay.route(d["logits"].cuda())
        out = {}
        for rows in (64, 0):
            moe.moe_plan_set_decode_rows(lay.plan, rows)
            y = lay.forward(x, idx, w)
            torch.cuda.synchronize()
            assert moe.moe_get_error(lay.plan) == 0
            out[rows] = (y.clone(), moe.moe_debug_tap(lay.plan, moe.TAP_PERM),
                         moe.moe_debug_tap(lay.plan, moe.TAP_QX),
                         moe.moe_debug_tap(lay.plan, moe.TAP_ACC_GU_F64))
        (ys, ps, qs, gs), (yg, pg, qg, gg) = out[64], out[0]
        assert (ps == pg).all() and (qs == qg).all()
        scale = np.abs(gs).max()
        assert np.abs(gs - gg).max() <= 2e-4 * scale
        assert (ys - yg).abs().max().item() <= 1e-2 * yg.abs().max().item()
    finally:
        lay.close()


def test_nvfp4_stress_dimensions_sampled():
    # the stress layer's dimensions (H = 4096, I = 1024, shared 2048, top_k 8, Zipf 1.5) with
    # 64 experts and 600 tokens on the grouped tensor-core GEMMs (several 128-row weight tiles
    # per expert, 32 K stages); oracle parity on 12 sampled tokens
    T, H, E, k, I, Is = 600, 4096, 64, 8, 1024, 2048
    sh = synth.LayerShape(T=T, H=H, E=E, k=k, I=I, Is=Is)
    d = synth.small_layer(T, H, E, k, I, Is, seed=380, zipf_s=1.5)
    W_dev = synth.make_weights_nvfp4(sh, 380, device="cuda")
    W = {n: v.cpu() for n, v in W_dev.items()}
    sample = np.random.default_rng(380).choice(T, 12, replace=False)
    check_layer(sh, d["x"], d["logits"], W_dev, oracle_layer_nvfp4(W, sh), sample=sample,
                acc_exact=False)


def test_nvfp4_pack_argument_errors():
    # host-side checks of moe_pack_weights_nvfp4: missing or misaligned arrays, and shared
    # expert arrays missing on a plan with a shared expert
    T, H, E, k, I, Is = 4, 256, 8, 2, 128, 64
    sh, d, W = _layer(T, H, E, k, I, Is, seed=390)
    Wd = weights_to(W, "cuda")
    plan = moe.moe_plan(E, k, H, I, Is, T)
    try:
        bad = dict(Wd)
        del bad["b_up"]
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_pack_weights_nvfp4(plan, bad)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
        bad = dict(Wd)
        bad["w_down"] = Wd["w_down"].data_ptr() + 8  # not 16-byte aligned
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_pack_weights_nvfp4(plan, bad)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
        bad = {n: v for n, v in Wd.items() if not n.startswith("sh_")}
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_pack_weights_nvfp4(plan, bad)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
        assert moe.moe_get_error(plan) == 0
    finally:
        moe.moe_plan_destroy(plan)
