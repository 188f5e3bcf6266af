"""Pins of the CPU oracle against things other than itself.

Every test here runs on the CPU. Each one checks the oracle against a hand-worked example,
a closed form, an invariant, a brute-force search or a library routine on a special case,
so that a dropped term, a wrong sign or index, or a transposed operand in the oracle fails
at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def layer_from_arrays(E, k, H, I, Is, **arrs):
    W = {}
    for key, v in arrs.items():
        dt = np.float32 if key.startswith("s_") or key.startswith("sh_s_") else np.int8
        W[key] = np.ascontiguousarray(np.array(v, dtype=dt))
    return oracle.Layer(W, E, k, H, I, Is), W


# ---------------------------------------------------------------- routing

def test_route_golden_ties():
    cases = json.load(open(os.path.join(GOLD, "route_ties.json")))["cases"]
    for c in cases:
        lg = np.array([c["logits"]], np.float32)
        idx, w = oracle.route(lg, c["k"])
        assert idx[0].tolist() == c["idx"], c
        sel = lg[0, idx[0]].astype(np.float64)
        closed = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        np.testing.assert_allclose(w[0], closed, rtol=0, atol=1e-7)
        if "w" in c:
            np.testing.assert_array_equal(w[0], np.array(c["w"], np.float32))


def test_route_all_equal_is_uniform():
    for E, k in [(8, 2), (128, 8), (5, 5), (3, 1)]:
        idx, w = oracle.route(np.full((4, E), 0.3, np.float32), k)
        assert (idx == np.arange(k)).all()
        assert (w == np.float32(1.0 / k)).all()


def test_route_k_equals_E_is_library_softmax():
    rng = np.random.default_rng(0)
    lg = rng.standard_normal((32, 16)).astype(np.float32)
    idx, w = oracle.route(lg, 16)
    order = np.argsort(-lg, axis=1, kind="stable")
    assert (idx == order).all()
    sm = torch.softmax(torch.from_numpy(lg).double(), dim=1).numpy()
    np.testing.assert_allclose(w, np.take_along_axis(sm, idx, 1), rtol=0, atol=1e-7)


def test_route_bruteforce_subsets():
    rng = np.random.default_rng(1)
    for trial in range(200):
        E = int(rng.integers(1, 7))
        k = int(rng.integers(1, E + 1))
        lg = rng.integers(-2, 3, size=(1, E)).astype(np.float32)  # many ties
        idx, w = oracle.route(lg, k)
        best = None
        for sub in itertools.combinations(range(E), k):
            s = float(lg[0, list(sub)].sum())
            if best is None or s > best[0]:        # combinations() is lexicographic: first wins ties
                best = (s, sub)
        assert tuple(sorted(idx[0].tolist())) == best[1]
        # slot order: logit descending, then id ascending
        keys = [(-lg[0, e], e) for e in idx[0]]
        assert keys == sorted(keys)


def test_route_library_topk_and_sum():
    rng = np.random.default_rng(2)
    lg = (rng.standard_normal((200, 64)) * 3).astype(np.float32)
    idx, w = oracle.route(lg, 8)
    tv, ti = torch.topk(torch.from_numpy(lg), 8, dim=1)
    assert (idx == ti.numpy()).all()          # distinct continuous draws: no ties
    assert np.abs(w.astype(np.float64).sum(1) - 1).max() <= 1e-6
    assert (np.diff(w, axis=1) <= 0).all()


# ---------------------------------------------------------------- activation quant

def test_quant_round_half_even_ties():
    # amax = 127 makes s = 1 exactly, so q = rne(x): the .5 cases land on even integers.
    row = [127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, 126.5, -0.5, 0.25, 0.0, -127.0]
    exp = [127, 2, 4, -2, -4, 0, 2, 126, 0, 0, 0, -127]
    x = bf16_bits([row])
    q, s = oracle.quant_rows(x)
    assert s[0] == np.float32(1.0)
    assert q[0].tolist() == exp


def test_quant_zero_row_and_extremes():
    rng = np.random.default_rng(3)
    xf = rng.standard_normal((20, 300)).astype(np.float32) * 3
    xf[5] = 0
    x = bf16_bits(xf)
    q, s = oracle.quant_rows(x)
    assert s[5] == 0 and (q[5] == 0).all()
    xr = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    for t in range(20):
        if t == 5:
            continue
        am = int(np.argmax(np.abs(xr[t].numpy())))
        assert abs(int(q[t, am])) == 127 and np.sign(q[t, am]) == np.sign(xr[t, am].item())
        assert np.abs(q[t]).max() <= 127
    # library: torch.round is round-half-even on the IEEE fp32 quotient
    sl = (xr.abs().amax(1) / 127.0)
    ql = torch.round(xr / torch.where(sl > 0, sl, torch.ones_like(sl))[:, None]).clamp(-127, 127)
    ql[5] = 0
    assert (torch.from_numpy(q.astype(np.float32)) == ql).all()
    assert (torch.from_numpy(s) == sl).all()


# ---------------------------------------------------------------- permutation

def test_permute_is_stable_sort_and_bijection():
    rng = np.random.default_rng(4)
    for T, E, k in [(16, 8, 2), (37, 128, 8), (1, 4, 4), (300, 256, 8)]:
        lg = rng.standard_normal((T, E)).astype(np.float32)
        idx, _ = oracle.route(lg, k)
        counts, offsets, perm = oracle.permute(idx, E)
        assert (counts == np.bincount(idx.ravel(), minlength=E)).all()
        assert counts.sum() == T * k and offsets[-1] == T * k
        assert (np.diff(offsets) >= 0).all()
        assert sorted(perm.tolist()) == list(range(T * k))
        assert (perm == np.argsort(idx.ravel(), kind="stable")).all()
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert (idx.ravel()[seg] == e).all()


# ---------------------------------------------------------------- integer GEMMs

def _tiny_layer(seed, T=5, H=64, E=4, k=2, I=32, Is=16):
    d = synth.small_layer(T, H, E, k, I, Is, seed)
    L = oracle.Layer(d["weights"], E, k, H, I, Is)
    idx, w = oracle.route(d["logits"], k)
    return d, L, idx, w


def test_gemm_accumulators_match_library_matmul():
    d, L, idx, w = _tiny_layer(5)
    W = {k_: v.numpy() for k_, v in d["weights"].items()}
    y, tp = oracle.forward(L, d["x"], idx, w, taps=True)
    qx = tp["qx"].astype(np.int64)
    T, S = tp["sh"].shape
    for t in range(T):
        for s in range(S):
            if s < L.k:
                e = idx[t, s]
                wg, wu, wd, I = W["w_gate"][e], W["w_up"][e], W["w_down"][e], L.I
            else:
                wg, wu, wd, I = W["sh_gate"], W["sh_up"], W["sh_down"], L.Is
            ag = wg.astype(np.int64) @ qx[t]
            au = wu.astype(np.int64) @ qx[t]
            assert (tp["acc_gu"][t, s, 0, :I] == ag).all()
            assert (tp["acc_gu"][t, s, 1, :I] == au).all()
            ad = wd.astype(np.int64) @ tp["hq"][t, s, :I].astype(np.int64)
            assert (tp["acc_d"][t, s] == ad).all()


@pytest.mark.parametrize("val", [127, -127])
def test_gemm_extremes_closed_form(val):
    # x constant -> q_x = 127 everywhere; weights all `val` -> acc = 127 * val * H.
    H, I, E, k = 128, 16, 2, 1
    lay, _ = layer_from_arrays(
        E, k, H, I, 0,
        w_gate=np.full((E, I, H), val), w_up=np.full((E, I, H), val),
        w_down=np.full((E, H, I), val), s_gate=np.full((E, I), 0.001),
        s_up=np.full((E, I), 0.001), s_down=np.full((E, H), 0.001))
    x = bf16_bits(np.full((1, H), 0.5))
    idx = np.array([[1]], np.int32)
    w = np.array([[1.0]], np.float32)
    y, tp = oracle.forward(lay, x, idx, w, taps=True)
    assert (tp["qx"] == 127).all()
    assert (tp["acc_gu"][0, 0] == 127 * val * H).all()
    # every h is equal -> q_h = +-127 (sign of h), acc_d = 127 * sign * val * I
    hs = int(np.sign(tp["hq"][0, 0, 0]))
    assert (tp["hq"][0, 0] == 127 * hs).all()
    assert (tp["acc_d"][0, 0] == 127 * hs * val * I).all()


# ---------------------------------------------------------------- whole layer

def test_golden_hand_layer():
    G = json.load(open(os.path.join(GOLD, "hand_layer.json")))
    lay, W = layer_from_arrays(2, 1, 4, 2, 0, w_gate=G["w_gate"], w_up=G["w_up"],
                               w_down=G["w_down"], s_gate=G["s_gate"], s_up=G["s_up"],
                               s_down=G["s_down"])
    x = bf16_bits([G["x"]])
    idx, w = oracle.route(np.array([G["logits"]], np.float32), G["top_k"])
    ex = G["expect"]
    assert idx[0].tolist() == ex["idx"] and w[0].tolist() == ex["w"]
    y, tp = oracle.forward(lay, x, idx, w, taps=True)
    assert tp["qx"][0].tolist() == ex["q_x"]
    assert tp["acc_gu"][0, 0, 0].tolist() == ex["acc_gate"]
    assert tp["acc_gu"][0, 0, 1].tolist() == ex["acc_up"]
    assert tp["hq"][0, 0].tolist() == ex["q_h"]
    assert tp["acc_d"][0, 0].tolist() == ex["acc_down"]
    # closed form in double
    sx = 1.0 / 127
    g = [32 * sx * 0.01, -95 * sx * 0.02]
    u = [64 * sx * 0.5, 127 * sx * 0.25]
    h = [gi / (1 + math.exp(-gi)) * ui for gi, ui in zip(g, u)]
    s_h = abs(h[1]) / 127
    yc = [a * s_h * sd for a, sd in zip(ex["acc_down"], G["s_down"][1])]
    np.testing.assert_allclose(y[0], yc, rtol=2e-6, atol=0)


@pytest.mark.parametrize("shape", [(16, 256, 8, 2, 128, 0), (7, 64, 6, 3, 32, 48), (3, 32, 4, 4, 16, 16)])
def test_dense_equals_sparse(shape):
    T, H, E, k, I, Is = shape
    d = synth.small_layer(T, H, E, k, I, Is, seed=11, zipf_s=1.1)
    L = oracle.Layer(d["weights"], E, k, H, I, Is)
    idx, w = oracle.route(d["logits"], k)
    ys = oracle.forward(L, d["x"], idx, w)
    yd = oracle.dense(L, d["x"], idx, w)
    np.testing.assert_allclose(ys, yd, rtol=1e-12, atol=1e-15 * np.abs(ys).max())


def _unquantised_reference(d, idx, w, E, k, H, I, Is):
    """The same layer with no activation quantisation (fp64 library matmuls on x and the
    dequantised weights); the oracle differs from it only by int8 activation error."""
    W = d["weights"]
    x = d["x"].double()

    def deq(q, s):
        return q.double() * s.double()[..., None]

    y = torch.zeros_like(x)
    for t in range(x.shape[0]):
        for j in range(k):
            e = int(idx[t, j])
            g = deq(W["w_gate"][e], W["s_gate"][e]) @ x[t]
            u = deq(W["w_up"][e], W["s_up"][e]) @ x[t]
            h = torch.nn.functional.silu(g) * u
            y[t] += float(w[t, j]) * (deq(W["w_down"][e], W["s_down"][e]) @ h)
        if Is:
            g = deq(W["sh_gate"], W["sh_s_gate"]) @ x[t]
            u = deq(W["sh_up"], W["sh_s_up"]) @ x[t]
            h = torch.nn.functional.silu(g) * u
            y[t] += deq(W["sh_down"], W["sh_s_down"]) @ h
    return y.numpy()


@pytest.mark.parametrize("shape", [(16, 256, 8, 2, 128, 0), (9, 128, 6, 3, 64, 96)])
def test_close_to_unquantised_layer(shape):
    T, H, E, k, I, Is = shape
    d = synth.small_layer(T, H, E, k, I, Is, seed=12)
    L = oracle.Layer(d["weights"], E, k, H, I, Is)
    idx, w = oracle.route(d["logits"], k)
    y = oracle.forward(L, d["x"], idx, w)
    yr = _unquantised_reference(d, idx, w, E, k, H, I, Is)
    rel = np.sqrt(((y - yr) ** 2).mean() / (yr ** 2).mean())
    assert rel < 3e-2, rel       # int8 activation + int8 h quantisation error only
    # a wrong slot weight or scale index would be far off; check per-token too
    per_tok = np.sqrt(((y - yr) ** 2).mean(1) / (yr ** 2).mean(1))
    assert per_tok.max() < 0.1


def test_single_expert_is_dense_swiglu_ffn():
    # E=1, k=1, no shared expert: the layer is one W8A8 SwiGLU FFN; its integer GEMMs are
    # library int64 matmuls and its activation is torch's SiLU.
    T, H, I = 6, 64, 48
    d = synth.small_layer(T, H, 1, 1, I, 0, seed=13)
    L = oracle.Layer(d["weights"], 1, 1, H, I, 0)
    idx, w = oracle.route(d["logits"], 1)
    assert (idx == 0).all() and (w == 1).all()
    y, tp = oracle.forward(L, d["x"], idx, w, taps=True)
    W = d["weights"]
    qx = torch.from_numpy(tp["qx"]).long()
    sx = torch.from_numpy(tp["sx"])
    ag = qx @ W["w_gate"][0].long().T
    au = qx @ W["w_up"][0].long().T
    g = (ag.float() * sx[:, None]) * W["s_gate"][0][None]
    u = (au.float() * sx[:, None]) * W["s_up"][0][None]
    h = torch.nn.functional.silu(g) * u
    hq = torch.from_numpy(tp["hq"][:, 0, :I]).long()
    sh = torch.from_numpy(tp["sh"][:, 0])
    # torch's SiLU may differ from g/(1+exp(-g)) in the last ulp: q_h may move by 1 at a tie
    assert (hq.float() - torch.round(h / sh[:, None])).abs().max() <= 1
    assert torch.allclose(sh, h.abs().amax(1) / 127, rtol=1e-6, atol=0)
    ad = hq @ W["w_down"][0].long().T
    assert (torch.from_numpy(tp["acc_d"][:, 0]).long() == ad).all()
    yl = (ad.float() * sh[:, None]) * W["s_down"][0][None]
    np.testing.assert_allclose(y, yl.double().numpy(), rtol=1e-6, atol=1e-9)


def test_token_permutation_equivariance():
    d = synth.small_layer(12, 64, 6, 2, 32, 16, seed=14)
    L = oracle.Layer(d["weights"], 6, 2, 64, 32, 16)
    idx, w = oracle.route(d["logits"], 2)
    y = oracle.forward(L, d["x"], idx, w)
    p = np.random.default_rng(0).permutation(12)
    yp = oracle.forward(L, d["x"][p], idx[p], w[p])
    np.testing.assert_array_equal(yp, y[p])


def test_shared_expert_alone():
    # Routed experts with zero weights contribute nothing; the shared one is a plain FFN
    # with weight 1 that matches the unquantised shared FFN up to int8 error.
    T, H, E, k, I, Is = 8, 128, 4, 2, 32, 64
    d = synth.small_layer(T, H, E, k, I, Is, seed=15)
    W = d["weights"]
    for key in ("w_gate", "w_up", "w_down"):
        W[key].zero_()
    for key in ("s_gate", "s_up", "s_down"):
        W[key].zero_()
    L = oracle.Layer(W, E, k, H, I, Is)
    idx, w = oracle.route(d["logits"], k)
    y = oracle.forward(L, d["x"], idx, w)
    yr = _unquantised_reference(d, idx, w, E, k, H, I, Is)
    rel = np.sqrt(((y - yr) ** 2).mean() / (yr ** 2).mean())
    assert rel < 3e-2


def test_router_logits_library_matmul():
    d = synth.make_layer(synth.Workload("p", synth.LayerShape(5, 96, 12, 2, 16, 0), 0,
                                        router="projection"))
    lg = oracle.router_logits(d["x"], d["w_router"])
    ref = d["x"].double() @ d["w_router"].double()
    np.testing.assert_allclose(lg, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_workload_properties():
    # Zipf skew readings: the decode rows share experts; the stress routing puts > 40% of
    # assignments on the top 4 experts and leaves some experts empty.
    dec = synth.WORKLOADS["decode"]
    lg = synth.make_logits(dec.shape.T, dec.shape.E, dec.seed, dec.zipf_s)
    idx, _ = oracle.route(lg, dec.shape.k)
    assert len(np.unique(idx)) < idx.size
    st = synth.WORKLOADS["stress"]
    lg = synth.make_logits(st.shape.T, st.shape.E, st.seed, st.zipf_s)
    idx, _ = oracle.route(lg, st.shape.k)
    c = np.bincount(idx.ravel(), minlength=st.shape.E)
    assert np.sort(c)[::-1][:4].sum() > 0.4 * idx.size
    assert (c == 0).any()


# ---------------------------------------------------------------- stacked-prefill layer input

def _bf16_to_f32(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).float()


def test_rmsnorm_constant_rows_closed_form():
    # a row of a constant c normalises to c / sqrt(c^2 + 1e-6) -> +-1 in bf16
    rows = np.array([[3.0] * 64, [-0.5] * 64, [1024.0] * 64], np.float32)
    _, x_in = oracle.rmsnorm_residual(bf16_bits(rows))
    f = _bf16_to_f32(x_in).numpy()
    assert (f[0] == 1.0).all() and (f[1] == -1.0).all() and (f[2] == 1.0).all()


def test_rmsnorm_matches_library_within_one_ulp():
    rng = np.random.default_rng(8)
    xf = (rng.standard_normal((40, 512)) * rng.uniform(0.1, 50, (40, 1))).astype(np.float32)
    # rows small enough that mean(x^2) is comparable to the 1e-6 epsilon, which then matters
    xf[30:] = (rng.standard_normal((10, 512)) * rng.uniform(2e-4, 2e-3, (10, 1))).astype(np.float32)
    x = bf16_bits(xf)
    _, x_in = oracle.rmsnorm_residual(x)
    xd = _bf16_to_f32(x).double()
    ref = torch.nn.functional.rms_norm(xd, (512,), eps=1e-6)
    got = _bf16_to_f32(x_in).double()
    ulp = ref.abs() * 2.0 ** -7      # bf16 spacing bound
    assert ((got - ref).abs() <= ulp).all()


def test_residual_is_fp32_add_rounded_to_bf16():
    rng = np.random.default_rng(9)
    x = bf16_bits(rng.standard_normal((7, 128)).astype(np.float32))
    y = rng.standard_normal((7, 128)) * 3
    x2, x_in = oracle.rmsnorm_residual(x, y)
    ref = (_bf16_to_f32(x) + torch.from_numpy(y).float()).to(torch.bfloat16)
    assert (torch.from_numpy(x2.view(np.int16)) == ref.view(torch.int16)).all()
    _, x_in2 = oracle.rmsnorm_residual(x2)
    assert (x_in == x_in2).all()


def test_residual_rounding_ties_go_to_even():
    # x + y landing exactly halfway between two bf16 neighbours rounds to the even one
    # (bf16 spacing is 2^-7 on [1, 2), 2^-6 on [2, 4), 2^-9 on [0.5, 1)); just above the
    # halfway point rounds up. Expected values worked by hand.
    cases = [  # (x, y, x + y rounded to bf16)
        (1.0, 2.0 ** -8, 1.0),
        (1.0078125, 2.0 ** -8, 1.015625),
        (-1.0, -(2.0 ** -8), -1.0),
        (-1.0078125, -(2.0 ** -8), -1.015625),
        (2.0, 2.0 ** -7, 2.0),
        (3.0, 2.0 ** -7, 3.0),
        (0.5, 2.0 ** -10, 0.5),
        (1.0, 2.0 ** -8 + 2.0 ** -20, 1.0078125),
    ]
    x = bf16_bits([[c[0] for c in cases]])
    y = np.array([[c[1] for c in cases]], np.float64)
    x2, _ = oracle.rmsnorm_residual(x, y)
    assert _bf16_to_f32(x2).numpy()[0].tolist() == [c[2] for c in cases]


# ---------------------------------------------------------------- NVFP4 expert weights

def _e2m1_table():
    return np.array(json.load(open(os.path.join(GOLD, "e2m1_codes.json")))["values"], np.float64)


def _e4m3_library(byte_array):
    """E4M3 bytes decoded by torch's float8_e4m3fn (a library routine)."""
    b = torch.from_numpy(np.ascontiguousarray(byte_array, np.uint8))
    return b.view(torch.float8_e4m3fn).double().numpy()


def test_e2m1_codes_golden_and_library():
    tab = _e2m1_table()
    got = np.array([oracle.e2m1_value(c) for c in range(16)])
    assert (got == tab).all() and (np.signbit(got) == np.signbit(tab)).all()
    # each E2M1 value re-encoded by bit placement as an E4M3 byte (exponent bias 1 -> 7,
    # the mantissa bit on top) and decoded by torch's float8_e4m3fn
    enc = []
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        enc.append((s << 7) | (((e + 6) << 3) | (m << 2) if e else (0x30 if m else 0)))
    assert (_e4m3_library(enc) == got).all()


def test_e4m3_every_byte_matches_library():
    lib_vals = _e4m3_library(np.arange(256))
    got = np.array([oracle.e4m3_value(b) for b in range(256)])
    nan = np.isnan(lib_vals)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2       # 0x7F and 0xFF
    assert (got[~nan] == lib_vals[~nan]).all()
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def _dequant_nvfp4(codes, scales):
    """w' = e2m1 * e4m3 of every element, decoded independently of the oracle: nibbles by
    numpy (element 2j low), values from the golden E2M1 table, scales by torch."""
    c = np.asarray(codes, np.uint8)
    nib = np.stack([c & 15, c >> 4], axis=-1).reshape(*c.shape[:-1], c.shape[-1] * 2)
    vals = _e2m1_table()[nib]
    sc = np.repeat(_e4m3_library(scales), 16, axis=-1)
    return vals * sc


def _random_nvfp4_layer(rng, E, k, H, I, Is):
    """Codes uniform over all bytes, block scales uniform over every finite non-negative
    E4M3 byte (subnormals and 448 included), matrix scales in [0.5, 2)."""
    W = dict(w_gate=rng.integers(0, 256, (E, I, H // 2)), w_up=rng.integers(0, 256, (E, I, H // 2)),
             w_down=rng.integers(0, 256, (E, H, I // 2)),
             b_gate=rng.integers(0, 127, (E, I, H // 16)), b_up=rng.integers(0, 127, (E, I, H // 16)),
             b_down=rng.integers(0, 127, (E, H, I // 16)),
             g_gate=rng.uniform(0.5, 2, E), g_up=rng.uniform(0.5, 2, E), g_down=rng.uniform(0.5, 2, E))
    if Is:
        W.update(sh_gate=rng.integers(0, 256, (Is, H // 2)), sh_up=rng.integers(0, 256, (Is, H // 2)),
                 sh_down=rng.integers(0, 256, (H, Is // 2)), sh_b_gate=rng.integers(0, 127, (Is, H // 16)),
                 sh_b_up=rng.integers(0, 127, (Is, H // 16)), sh_b_down=rng.integers(0, 127, (H, Is // 16)),
                 sh_g=rng.uniform(0.5, 2, 3))
    out = {}
    for key, v in W.items():
        out[key] = np.ascontiguousarray(v, np.float32 if key.startswith("g_") or key == "sh_g" else np.uint8)
    return out


@pytest.mark.parametrize("weights", ["random_bytes", "synth"])
def test_nvfp4_accumulators_match_library_matmul(weights):
    T, H, E, k, I, Is = 6, 64, 4, 2, 32, 48
    d = synth.small_layer(T, H, E, k, I, Is, seed=21)
    if weights == "synth":
        W = {key: v.numpy() for key, v in synth.make_weights_nvfp4(d["shape"], 21).items()}
    else:
        W = _random_nvfp4_layer(np.random.default_rng(21), E, k, H, I, Is)
    L = oracle.LayerNvfp4(W, E, k, H, I, Is)
    idx, w = oracle.route(d["logits"], k)
    y, tp = oracle.forward_nvfp4(L, d["x"], idx, w, taps=True)
    q, _ = oracle.quant_rows(d["x"])
    assert (tp["qx"] == q).all()
    qx = tp["qx"].astype(np.float64)
    for t in range(T):
        for s in range(k + 1):
            if s < k:
                e = idx[t, s]
                wg, wu = _dequant_nvfp4(W["w_gate"][e], W["b_gate"][e]), _dequant_nvfp4(W["w_up"][e], W["b_up"][e])
                wd, n = _dequant_nvfp4(W["w_down"][e], W["b_down"][e]), I
            else:
                wg, wu = _dequant_nvfp4(W["sh_gate"], W["sh_b_gate"]), _dequant_nvfp4(W["sh_up"], W["sh_b_up"])
                wd, n = _dequant_nvfp4(W["sh_down"], W["sh_b_down"]), Is
            # every term is a multiple of 2^-10 and every partial sum is far below 2^43:
            # the float64 matmul is exact in any summation order
            assert (tp["acc_gu"][t, s, 0, :n] == wg @ qx[t]).all()
            assert (tp["acc_gu"][t, s, 1, :n] == wu @ qx[t]).all()
            assert (tp["acc_d"][t, s] == wd @ tp["hq"][t, s, :n].astype(np.float64)).all()


def test_nvfp4_integer_weights_reduce_to_int8_layer():
    # Block scales 1.0 and codes of integer values (0, +-1, +-2, +-3, +-4, +-6): the NVFP4
    # layer is the int8 layer with those integers as weights and the matrix scale as every
    # channel's scale, bit for bit.
    T, H, E, k, I, Is = 7, 64, 5, 2, 32, 48
    rng = np.random.default_rng(22)
    d = synth.small_layer(T, H, E, k, I, Is, seed=22)
    int_codes = np.array([0, 2, 4, 5, 6, 7, 8, 10, 12, 13, 14, 15], np.uint8)
    tab = _e2m1_table()

    def mat(shape):
        c = rng.choice(int_codes, size=shape[:-1] + (shape[-1],))
        packed = (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
        return packed, tab[c].astype(np.int8), np.full(shape[:-1] + (shape[-1] // 16,), 0x38, np.uint8)

    g = rng.uniform(0.001, 0.01, (E, 3)).astype(np.float32)
    shg = rng.uniform(0.001, 0.01, 3).astype(np.float32)
    F, N = {}, {}
    for name, shape, r in (("gate", (E, I, H), 0), ("up", (E, I, H), 1), ("down", (E, H, I), 2)):
        F["w_" + name], N["w_" + name], F["b_" + name] = mat(shape)
        F["g_" + name] = np.ascontiguousarray(g[:, r])
        N["s_" + name] = np.ascontiguousarray(np.repeat(g[:, r:r + 1], shape[1], axis=1))
    for name, shape, r in (("gate", (Is, H), 0), ("up", (Is, H), 1), ("down", (H, Is), 2)):
        F["sh_" + name], N["sh_" + name], F["sh_b_" + name] = mat(shape)
        N["sh_s_" + name] = np.full(shape[0], shg[r], np.float32)
    F["sh_g"] = shg
    idx, w = oracle.route(d["logits"], k)
    y4, t4 = oracle.forward_nvfp4(oracle.LayerNvfp4(F, E, k, H, I, Is), d["x"], idx, w, taps=True)
    y8, t8 = oracle.forward(oracle.Layer(N, E, k, H, I, Is), d["x"], idx, w, taps=True)
    assert (t4["acc_gu"] == t8["acc_gu"]).all() and (t4["acc_d"] == t8["acc_d"]).all()
    assert (t4["hq"] == t8["hq"]).all()
    assert np.array_equal(y4, y8)


def test_golden_hand_layer_nvfp4():
    G = json.load(open(os.path.join(GOLD, "hand_layer_nvfp4.json")))
    E, k, H, I = 2, 1, 16, 16
    ex1 = G["expert1"]
    W = {}
    for name, rows, K in (("gate", I, H), ("up", I, H), ("down", H, I)):
        codes = np.zeros((E, rows, K // 2), np.uint8)
        sc = np.full((E, rows, K // 16), ex1["default_scale"], np.uint8)
        for r, b in ex1[name + "_rows"].items():
            codes[1, int(r)] = b
        for r, b in ex1[name + "_scales"].items():
            sc[1, int(r)] = b
        W["w_" + name], W["b_" + name] = codes, sc
        W["g_" + name] = np.array([1.0, ex1["g_" + name]], np.float32)
    lay = oracle.LayerNvfp4(W, E, k, H, I, 0)
    x = bf16_bits([G["x"]])
    idx, w = oracle.route(np.array([G["logits"]], np.float32), G["top_k"])
    ex = G["expect"]
    assert idx[0].tolist() == ex["idx"]
    y, tp = oracle.forward_nvfp4(lay, x, idx, w, taps=True)
    assert tp["qx"][0].tolist() == ex["q_x"]
    assert tp["acc_gu"][0, 0, 0].tolist() == ex["acc_gate"]
    assert tp["acc_gu"][0, 0, 1].tolist() == ex["acc_up"]
    assert tp["hq"][0, 0].tolist() == ex["q_h"]
    assert tp["acc_d"][0, 0].tolist() == ex["acc_down"]
    s_h = ex["h0"] / 127
    yc = [a * s_h * ex1["g_down"] for a in ex["acc_down"]]
    np.testing.assert_allclose(y[0], yc, rtol=2e-6, atol=0)


@pytest.mark.parametrize("bad", [0x7F, 0x80, 0xB8, 0xFF])
def test_nvfp4_rejects_negative_or_nan_block_scales(bad):
    T, H, E, k, I = 2, 32, 2, 1, 16
    W = _random_nvfp4_layer(np.random.default_rng(23), E, k, H, I, 0)
    W["b_down"][1, 3, 0] = bad
    d = synth.small_layer(T, H, E, k, I, 0, seed=23)
    idx = np.array([[0], [0]], np.int32)
    w = np.ones((T, 1), np.float32)
    lay = oracle.LayerNvfp4(W, E, k, H, I, 0)
    with pytest.raises(ValueError):
        oracle.forward_nvfp4(lay, d["x"], idx, w)


def test_nvfp4_synth_weights_close_to_their_fp32_draws():
    # the generator's NVFP4 quantisation of N(0, 0.02) draws: relative RMS error of an E2M1
    # element with an E4M3 block scale is about 10%; a wrong scale or nibble order is not
    g = torch.Generator().manual_seed(5)
    w = torch.randn((64, 256), generator=g) * 0.02
    gs = w.abs().amax() / (6 * 448)
    codes, bsc = synth.quantize_nvfp4_rows(w, gs)
    deq = _dequant_nvfp4(codes.numpy(), bsc.numpy()) * float(gs)
    rel = np.sqrt(((deq - w.double().numpy()) ** 2).mean() / (w.double().numpy() ** 2).mean())
    assert rel < 0.15, rel
