"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element.

Routing indices, permutation, activation codes and every int32 gate/up accumulator must be
bit-identical; requantised h codes may differ by one at a rounding tie caused by the last
ulp of exp (counted, at most 1e-3 of them); down accumulators must be bit-identical on every
row whose h codes agree; y must satisfy max|dy| <= 1e-2 max|y_ref| and
rms(dy) <= 5e-3 rms(y_ref)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import grouped_expert_ffn_gb300 as moe
from helpers import check_layer, oracle_layer, weights_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.lib()


def _host_layer(name):
    wl = synth.WORKLOADS[name]
    d = synth.make_layer(wl, device="cpu")
    return wl, d


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
def test_layer_parity_full(name):
    wl, d = _host_layer(name)
    sh = wl.shape
    W = weights_to(d["weights"], "cuda")
    st = check_layer(sh, d["x"], d["logits"], W, oracle_layer(d["weights"], sh))
    print(name, {k: v for k, v in st.items() if k in ("max_rel", "rmse_rel", "hq_diff", "hq_total")})


def test_stress_layer_sampled():
    # T=8192, E=256, Zipf 1.5: the persistent scheduler under heavy skew with empty experts.
    # Full oracle parity on a sample of tokens that includes, for every empty expert, the
    # first and last token of the nearest non-empty expert on each side (their rows sit at
    # the segment boundaries around the empty group); and every gate/up accumulator of the
    # heaviest expert's rows against the exact integer sums of the oracle's activation codes
    # with that expert's int8 weights (fp64 products and sums of integers below 2^53 are exact).
    wl = synth.WORKLOADS["stress"]
    sh = wl.shape
    W = synth.make_weights(sh, wl.seed, device="cuda")
    x = synth.make_activations(sh.T, sh.H, wl.seed, wl.outliers, "cpu")
    lg = synth.make_logits(sh.T, sh.E, wl.seed, wl.zipf_s, "cpu")
    L = oracle_layer(W, sh)
    idx_o, _ = oracle.route(lg, sh.k)
    counts_o = np.bincount(idx_o.ravel(), minlength=sh.E)
    toks_of = lambda e: np.nonzero((idx_o == e).any(axis=1))[0]
    edge = []
    for e in np.nonzero(counts_o == 0)[0]:
        for step in (-1, 1):
            n = e + step
            while 0 <= n < sh.E and counts_o[n] == 0:
                n += step
            if 0 <= n < sh.E:
                t = toks_of(n)
                edge += [t[0], t[-1]]
    rng = np.random.default_rng(0)
    sample = np.unique(np.concatenate([[0, sh.T - 1], rng.choice(sh.T, 22, replace=False),
                                       np.asarray(edge, np.int64)[:40]]))
    st = check_layer(sh, x, lg, W, L, sample=sample)
    counts = st["tap"]["counts"]
    assert (counts == 0).any() and np.sort(counts)[::-1][:4].sum() > 0.4 * sh.T * sh.k
    # every row of the heaviest expert
    e = int(np.argmax(counts_o))
    rows_tok = toks_of(e)
    q_o, _ = oracle.quant_rows(x)
    qx = q_o[rows_tok].astype(np.float64)
    ref_g = qx @ W["w_gate"][e].cpu().numpy().astype(np.float64).T
    ref_u = qx @ W["w_up"][e].cpu().numpy().astype(np.float64).T
    perm = st["tap"]["perm"]
    R = sh.T * sh.k + sh.T
    acc_gu = st["tap"]["acc_gu"].reshape(R, 2, max(sh.I, sh.Is))
    off = st["tap"]["offsets"]
    seg = np.arange(off[e], off[e + 1])
    assert (perm[seg] // sh.k == rows_tok).all()   # rows of expert e in token order
    rows = sh.T + seg                              # shared rows come first
    assert (acc_gu[rows, 0, :sh.I] == ref_g).all()
    assert (acc_gu[rows, 1, :sh.I] == ref_u).all()


def test_stack_layer0_sampled():
    # First layer of the stacked-prefill workload at full size (T=2600) in the bench's plan
    # configuration. The layer input is the RMS-normalised x; the router projection is checked
    # against the oracle's double-precision logits within the fp32 summation bound, and the
    # MoE layer is checked with both sides routing on the oracle's logits rounded to fp32.
    wl = synth.WORKLOADS["stack"]
    sh = wl.shape
    d = synth.make_layer(wl, device="cpu", with_weights=False)
    W = synth.make_weights(sh, synth.layer_seed(wl, 0), device="cuda")
    x_dev = d["x"].cuda()
    xin_dev = torch.empty_like(x_dev)
    moe.moe_rmsnorm_residual(x_dev, None, xin_dev)
    _, xin_o = oracle.rmsnorm_residual(d["x"])
    xin_g = xin_dev.cpu().view(torch.int16).numpy().view(np.uint16)
    diff = np.abs(xin_g.astype(np.int32) - xin_o.astype(np.int32))
    assert diff.max() <= 1 and (diff != 0).mean() < 1e-3
    x_in = torch.from_numpy(xin_o.view(np.int16)).view(torch.bfloat16)
    lg_dev = torch.empty((sh.T, sh.E), dtype=torch.float32, device="cuda")
    moe.moe_router_logits(x_in.cuda(), d["w_router"].cuda(), lg_dev)
    lg_o = oracle.router_logits(x_in, d["w_router"])
    bound = 2048 * 2.0 ** -24 * (np.abs(x_in.float().numpy()) @ np.abs(d["w_router"].numpy()))
    assert (np.abs(lg_dev.cpu().numpy() - lg_o) <= bound + 1e-6).all()
    lg = torch.from_numpy(lg_o.astype(np.float32))
    sample = np.arange(0, sh.T, 97)
    check_layer(sh, x_in, lg, W, oracle_layer(W, sh), sample=sample)


def test_rmsnorm_residual_matches_oracle():
    x = synth.make_activations(300, 2048, 11)
    y = torch.randn(300, 2048, generator=torch.Generator().manual_seed(2)) * 4
    xd, yd = x.cuda(), y.cuda()
    xin = torch.empty_like(xd)
    moe.moe_rmsnorm_residual(xd, yd, xin)
    x2_o, xin_o = oracle.rmsnorm_residual(x, y.double().numpy())
    assert (xd.cpu().view(torch.int16).numpy().view(np.uint16) == x2_o).all()
    g = xin.cpu().view(torch.int16).numpy().view(np.uint16).astype(np.int32)
    diff = np.abs(g - xin_o.astype(np.int32))
    assert diff.max() <= 1 and (diff != 0).mean() < 1e-3


@pytest.mark.parametrize("T", [1, 2, 5, 8, 9, 31, 129, 200])
def test_ragged_token_counts(T):
    sh = synth.LayerShape(T=T, H=256, E=16, k=4, I=128, Is=192)
    d = synth.small_layer(sh.T, sh.H, sh.E, sh.k, sh.I, sh.Is, seed=100 + T, zipf_s=1.1)
    W = weights_to(d["weights"], "cuda")
    check_layer(sh, d["x"], d["logits"], W, oracle_layer(d["weights"], sh), plan_tokens=256)


def test_all_tokens_one_expert_and_empty_experts():
    sh = synth.LayerShape(T=300, H=512, E=32, k=2, I=256, Is=0)
    d = synth.small_layer(sh.T, sh.H, sh.E, sh.k, sh.I, sh.Is, seed=7)
    lg = d["logits"].clone()
    lg[:, 0] += 50.0   # every token picks expert 0 first
    lg[:, 5] += 40.0   # and expert 5 second; the other 30 experts are empty
    W = weights_to(d["weights"], "cuda")
    st = check_layer(sh, d["x"], lg, W, oracle_layer(d["weights"], sh))
    c = st["tap"]["counts"]
    assert c[0] == 300 and c[5] == 300 and c.sum() == 600


def test_decode_and_prefill_give_identical_integers():
    # the same 8 tokens through the decode kernels (T=8) and inside a 9-token call on the
    # grouped GEMMs (the plan's threshold set to 8)
    d = synth.small_layer(9, 2048, 128, 8, 512, 512, seed=21, zipf_s=1.1, outliers=8)
    W = weights_to(d["weights"], "cuda")
    lay = moe.MoELayer(128, 8, 2048, 512, 512, 16, W)
    try:
        moe.moe_plan_set_decode_rows(lay.plan, 8)
        moe.moe_debug_enable(lay.plan, True)
        x = d["x"].cuda()
        lg = d["logits"].cuda()
        idx, w = lay.route(lg)
        y9 = lay.forward(x, idx, w)
        torch.cuda.synchronize()
        gu9 = moe.moe_debug_tap(lay.plan, moe.TAP_ACC_GU).reshape(-1, 2, 512)
        perm9 = moe.moe_debug_tap(lay.plan, moe.TAP_PERM)
        y8 = lay.forward(x[:8].contiguous(), idx[:8].contiguous(), w[:8].contiguous())
        torch.cuda.synchronize()
        gu8 = moe.moe_debug_tap(lay.plan, moe.TAP_ACC_GU).reshape(-1, 2, 512)
        perm8 = moe.moe_debug_tap(lay.plan, moe.TAP_PERM)
        from helpers import row_map
        r9 = row_map(perm9, 9, 8, True)
        r8 = row_map(perm8, 8, 8, True)
        for t in range(8):
            for s in range(9):
                assert (gu9[r9[t, s]] == gu8[r8[t, s]]).all()
        dy = (y9[:8] - y8).abs().max().item()
        assert dy <= 1e-5 * y9[:8].abs().max().item()
    finally:
        lay.close()


@pytest.mark.parametrize("T,E,k", [(9, 128, 8), (16, 128, 8), (33, 128, 8), (64, 128, 8),
                                   (64, 16, 4)])
def test_decode_kernels_up_to_64_rows_match_the_oracle(T, E, k):
    # the weight-streaming kernels above 8 rows: an expert's rows are taken 8 per pass (the
    # shared expert has all T rows; with E=16, k=4 every routed expert has about 16)
    sh = synth.LayerShape(T=T, H=2048, E=E, k=k, I=512, Is=512)
    d = synth.small_layer(T, 2048, E, k, 512, 512, seed=40 + T + E, zipf_s=1.1, outliers=8)
    W = weights_to(d["weights"], "cuda")
    lay = moe.MoELayer(E, k, 2048, 512, 512, T, W)
    try:
        moe.moe_plan_set_decode_rows(lay.plan, 64)
        st = check_layer(sh, d["x"], d["logits"], W, oracle_layer(d["weights"], sh), layer=lay)
        assert st["tap"]["counts"].max() > 8  # some routed expert took more than one pass
    finally:
        lay.close()


def _path_taps(lay, x, idx, w, rows):
    moe.moe_plan_set_decode_rows(lay.plan, rows)
    y = lay.forward(x, idx, w)
    torch.cuda.synchronize()
    assert moe.moe_get_error(lay.plan) == 0
    taps = {n: moe.moe_debug_tap(lay.plan, i) for n, i in (
        ("counts", moe.TAP_COUNTS), ("offsets", moe.TAP_OFFSETS), ("perm", moe.TAP_PERM),
        ("qx", moe.TAP_QX), ("sx", moe.TAP_SX), ("acc_gu", moe.TAP_ACC_GU), ("hq", moe.TAP_HQ),
        ("sh", moe.TAP_SH), ("acc_d", moe.TAP_ACC_D))}
    return y, taps


@pytest.mark.parametrize("T", [1, 3, 8, 9, 24, 64])
def test_decode_and_grouped_paths_give_identical_integers(T):
    # the same call through the weight-streaming kernels and through the grouped GEMMs, on
    # both sides of every dispatch threshold a plan can take: permutation, activation codes,
    # every gate/up and down accumulator, the h codes and their scales are bit-identical (the
    # two paths use the same rounding rules and the same h formula); y agrees up to the order
    # of the fp32 additions
    H, E, k, I, Is = 2048, 128, 8, 512, 512
    d = synth.small_layer(T, H, E, k, I, Is, seed=70 + T, zipf_s=1.1, outliers=8)
    W = weights_to(d["weights"], "cuda")
    lay = moe.MoELayer(E, k, H, I, Is, T, W)
    try:
        moe.moe_debug_enable(lay.plan, True)
        x = d["x"].cuda()
        idx, w = lay.route(d["logits"].cuda())
        y_s, ts = _path_taps(lay, x, idx, w, 64)
        y_g, tg = _path_taps(lay, x, idx, w, 0)
        for n in ("counts", "offsets", "perm", "qx", "sx"):
            assert (ts[n] == tg[n]).all(), n
        R = T * k + T
        ig = np.full(R, I)
        ig[:T] = Is  # shared rows first
        gu_s, gu_g = ts["acc_gu"].reshape(R, 2, -1), tg["acc_gu"].reshape(R, 2, -1)
        hq_s, hq_g = ts["hq"].reshape(R, -1), tg["hq"].reshape(R, -1)
        for r in range(R):
            assert (gu_s[r, :, :ig[r]] == gu_g[r, :, :ig[r]]).all(), r
            assert (hq_s[r, :ig[r]] == hq_g[r, :ig[r]]).all(), r
        assert (ts["sh"][:R] == tg["sh"][:R]).all()
        assert (ts["acc_d"].reshape(R, H) == tg["acc_d"].reshape(R, H)).all()
        assert (y_s - y_g).abs().max().item() <= 1e-5 * y_g.abs().max().item()
    finally:
        lay.close()


@pytest.mark.parametrize("T,rows", [(8, 32), (40, 32), (40, 0), (2600, 32)])
def test_route_forward_matches_route_then_forward(T, rows):
    # moe_route_forward (routing inside the forward's first kernel) against moe_route followed
    # by moe_forward: idx and w bit-identical, every tapped integer and scale bit-identical,
    # y equal up to the order of the fp32 additions; on the weight-streaming path (T <= rows)
    # and on the grouped GEMMs, twice in a row (the histogram kernel's counter returns to zero)
    H, E, k, I, Is = 2048, 128, 8, 512, 512
    d = synth.small_layer(T, H, E, k, I, Is, seed=90 + T, zipf_s=1.1, outliers=8)
    W = weights_to(d["weights"], "cuda")
    lay = moe.MoELayer(E, k, H, I, Is, T, W)
    names = (("counts", moe.TAP_COUNTS), ("offsets", moe.TAP_OFFSETS), ("perm", moe.TAP_PERM),
             ("qx", moe.TAP_QX), ("sx", moe.TAP_SX), ("acc_gu", moe.TAP_ACC_GU), ("hq", moe.TAP_HQ),
             ("sh", moe.TAP_SH), ("acc_d", moe.TAP_ACC_D))
    try:
        moe.moe_plan_set_decode_rows(lay.plan, rows)
        moe.moe_debug_enable(lay.plan, True)
        x = d["x"].cuda()
        lg = d["logits"].cuda()
        idx_r, w_r = lay.route(lg)
        y_r = lay.forward(x, idx_r, w_r)
        torch.cuda.synchronize()
        ref = {n: moe.moe_debug_tap(lay.plan, i) for n, i in names}
        for _ in range(2):
            idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
            w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
            y = torch.empty((T, H), dtype=torch.float32, device="cuda")
            moe.moe_route_forward(lay.plan, lay.packed, x, lg, idx, w, y)
            torch.cuda.synchronize()
            assert moe.moe_get_error(lay.plan) == 0
            assert torch.equal(idx, idx_r) and torch.equal(w, w_r)
            for n, i in names:
                assert (moe.moe_debug_tap(lay.plan, i) == ref[n]).all(), n
            assert (y - y_r).abs().max().item() <= 1e-5 * y_r.abs().max().item()
    finally:
        lay.close()


@pytest.mark.parametrize("T,rows", [(8, 32), (8, 0), (40, 0)])
def test_largest_supported_shape(T, rows):
    # H = 8192 and I = I_shared = 4096, the largest shapes a plan accepts: the decode kernels'
    # largest shared-memory staging (8 x H token codes, 8 x I h codes) and the grouped GEMMs'
    # longest reduction (the 1024-K chunked accumulators when the exactness bound needs them),
    # on the weight-streaming path and on the grouped GEMMs
    sh = synth.LayerShape(T=T, H=8192, E=4, k=2, I=4096, Is=4096)
    W = synth.make_weights(sh, 123, device="cuda")
    x = synth.make_activations(T, sh.H, 123, 0, "cpu")
    lg = synth.make_logits(T, sh.E, 123, 0.0, "cpu")
    lay = moe.MoELayer(sh.E, sh.k, sh.H, sh.I, sh.Is, T, W)
    try:
        moe.moe_plan_set_decode_rows(lay.plan, rows)
        check_layer(sh, x, lg, W, oracle_layer(W, sh), layer=lay)
    finally:
        lay.close()


def _tie_rows(x, seed):
    """Rows whose elements sit on (or next to) the rounding boundaries of the int8 code: with a
    power-of-two amax the scale is exact and (m + 1/2) * scale is an exact tie; with another
    amax the bf16 value nearest a tie lands a fraction of an ulp from it."""
    g = torch.Generator().manual_seed(seed)
    T, H = x.shape
    x = x.clone()
    for t in range(T):
        c = 2.0 ** (t % 9 - 4)
        m = torch.randint(-127, 127, (H,), generator=g).double() + 0.5
        if t % 3 == 2:  # non-exact scale: amax 100 c, targets next to (m + 1/2) * fl(amax / 127)
            s = float(np.float32(np.float32(100.0 * c) / np.float32(127.0)))
            row = m.clamp(-99.5, 99.5) * s
            row[0] = 100.0 * c
        else:
            row = m * c
            row[0] = -127.0 * c if t % 2 else 127.0 * c
        row[1::7] = torch.randint(-127, 128, (len(range(1, H, 7)),), generator=g).double() * c
        x[t] = row.to(torch.bfloat16)
    return x


@pytest.mark.parametrize("T", [8, 40])
def test_activation_codes_on_rounding_ties(T):
    # decode (T=8) and prefill (T=40) token quantisation at exact and near ties, bit-exact
    # against the oracle's round-half-even of the fp32 quotient, and the layer downstream
    sh = synth.LayerShape(T=T, H=1024, E=32, k=4, I=256, Is=256)
    d = synth.small_layer(T, 1024, 32, 4, 256, 256, seed=31 + T)
    x = _tie_rows(d["x"], 7 + T)
    W = weights_to(d["weights"], "cuda")
    q_o, s_o = oracle.quant_rows(x)
    xf = x.float().numpy()
    ties = np.abs(np.abs(xf / s_o[:, None]) % 1.0 - 0.5) < 1e-3
    assert ties.sum() > T * 1024 // 2  # most elements are (near) ties
    check_layer(sh, x, d["logits"], W, oracle_layer(d["weights"], sh))


def test_decode_after_a_smaller_plan_was_created():
    # The decode kernels' shared-memory limit is process-wide: creating a plan with small
    # shapes after one with large shapes must not break decode on the large plan.
    big = synth.LayerShape(T=8, H=4096, E=16, k=4, I=2048, Is=0)
    d = synth.small_layer(8, big.H, big.E, big.k, big.I, 0, seed=61, zipf_s=1.1)
    W = weights_to(d["weights"], "cuda")
    lay = moe.MoELayer(big.E, big.k, big.H, big.I, 0, 8, W)
    small = moe.moe_plan(8, 2, 256, 128, 0, 16)
    try:
        check_layer(big, d["x"], d["logits"], W, oracle_layer(d["weights"], big), layer=lay)
    finally:
        moe.moe_plan_destroy(small)
        lay.close()


def test_decode_threshold_range():
    lay_plan = moe.moe_plan(8, 2, 256, 128, 0, 16)
    try:
        for bad in (-1, 65):
            with pytest.raises(moe.MoeError):
                moe.moe_plan_set_decode_rows(lay_plan, bad)
        for ok in (0, 1, 32, 64):
            moe.moe_plan_set_decode_rows(lay_plan, ok)
    finally:
        moe.moe_plan_destroy(lay_plan)


def test_capacity_and_argument_errors():
    sh = synth.LayerShape(T=16, H=256, E=8, k=2, I=128, Is=0)
    d = synth.small_layer(16, 256, 8, 2, 128, 0, seed=3)
    W = weights_to(d["weights"], "cuda")
    lay = moe.MoELayer(8, 2, 256, 128, 0, 8, W)
    try:
        x = d["x"].cuda()
        lg = d["logits"].cuda()
        idx = torch.zeros((16, 2), dtype=torch.int32, device="cuda")
        w = torch.zeros((16, 2), dtype=torch.float32, device="cuda")
        with pytest.raises(moe.MoeError) as e:
            moe.moe_route(lay.plan, lg, idx, w)
        assert e.value.status == moe.MOE_ERR_CAPACITY
        y = torch.empty((16, 256), device="cuda")
        with pytest.raises(moe.MoeError) as e:
            moe.moe_forward(lay.plan, lay.packed, x, idx, w, y)
        assert e.value.status == moe.MOE_ERR_CAPACITY
        # misaligned output pointer
        yb = torch.empty(16 * 256 + 1, device="cuda")[1:]
        st = moe.lib().moe_forward(lay.plan, lay.packed, x[:8].data_ptr(), 8, idx.data_ptr(),
                                   w.data_ptr(), yb.data_ptr(), None)
        assert st == moe.MOE_ERR_INVALID_ARG
        # empty batch: refused on the host, nothing queued, no sticky error
        st = moe.lib().moe_route(lay.plan, lg.data_ptr(), 0, idx.data_ptr(), w.data_ptr(), None)
        assert st == moe.MOE_ERR_INVALID_ARG
        st = moe.lib().moe_forward(lay.plan, lay.packed, x.data_ptr(), 0, idx.data_ptr(),
                                   w.data_ptr(), y.data_ptr(), None)
        assert st == moe.MOE_ERR_INVALID_ARG
        assert moe.moe_get_error(lay.plan) == 0
    finally:
        lay.close()


def test_out_of_range_expert_sets_device_error():
    sh = synth.LayerShape(T=12, H=256, E=8, k=2, I=128, Is=0)
    d = synth.small_layer(12, 256, 8, 2, 128, 0, seed=4)
    W = weights_to(d["weights"], "cuda")
    lay = moe.MoELayer(8, 2, 256, 128, 0, 16, W)
    try:
        idx = torch.tensor([[0, 1]] * 11 + [[3, 99]], dtype=torch.int32, device="cuda")
        w = torch.full((12, 2), 0.5, device="cuda")
        lay.forward(d["x"].cuda(), idx, w)
        assert moe.moe_get_error(lay.plan) == moe.MOE_ERR_DEVICE
        moe.moe_clear_error(lay.plan)
        assert moe.moe_get_error(lay.plan) == 0
    finally:
        lay.close()


def test_bounded_wait_times_out_and_the_context_stays_usable():
    # Failure detection without a fault: a wait on a barrier that nothing completes gives up
    # after its limit and sets the plan's sticky MOE_ERR_TIMEOUT; the host reads it, clears
    # it, and the same plan then computes a full layer correctly.
    wl, d = _host_layer("tiny")
    sh = wl.shape
    W = weights_to(d["weights"], "cuda")
    lay = moe.MoELayer(sh.E, sh.k, sh.H, sh.I, sh.Is, sh.T, W)
    try:
        assert moe.moe_get_error(lay.plan) == 0
        moe.moe_selftest_wait_timeout(lay.plan)
        assert moe.moe_get_error(lay.plan) == moe.MOE_ERR_TIMEOUT
        assert moe.moe_get_error(lay.plan) == moe.MOE_ERR_TIMEOUT  # sticky
        moe.moe_clear_error(lay.plan)
        assert moe.moe_get_error(lay.plan) == 0
        check_layer(sh, d["x"], d["logits"], W, oracle_layer(d["weights"], sh), layer=lay)
    finally:
        lay.close()


def test_residual_add():
    x = synth.make_activations(37, 256, 5)
    y = torch.randn(37, 256, generator=torch.Generator().manual_seed(1))
    xd = x.cuda()
    moe.moe_residual_add(xd, y.cuda())
    ref = (x.float() + y).to(torch.bfloat16)
    assert torch.equal(xd.cpu().view(torch.int16), ref.view(torch.int16))


def test_adversarial_rows_take_the_exact_chunked_path():
    # Constant token rows quantise to +-127 everywhere and one gate row of expert 0 is all 127:
    # the gate accumulator reaches 2048 * 127^2 > 2^24, beyond what one fp32 accumulator holds
    # exactly, and the product of the row/weight sum-of-squares bounds exceeds 2^48, so the
    # kernel must take the 1024-K chunked accumulation; the int32 results stay bit-exact.
    sh = synth.LayerShape(T=40, H=2048, E=4, k=2, I=128, Is=128)
    d = synth.small_layer(sh.T, sh.H, sh.E, sh.k, sh.I, sh.Is, seed=31)
    W = d["weights"]
    W["w_gate"][0, 0, :] = 127
    W["w_up"][1, 3, :] = -127
    x = d["x"].float()
    x[:20] = 0.75                     # constant rows: every code is +127
    x[20:30] = -2.0                   # every code is -127
    x = x.to(torch.bfloat16)
    lg = d["logits"].clone()
    lg[:, 0] += 10.0                  # every token routes to expert 0
    Wd = weights_to(W, "cuda")
    layer = moe.MoELayer(sh.E, sh.k, sh.H, sh.I, sh.Is, sh.T, Wd)
    try:
        st = check_layer(sh, x, lg, Wd, oracle_layer(W, sh), layer=layer)
    finally:
        layer.close()
    gu = st["tap"]["acc_gu"]
    assert np.abs(gu).max() == 2048 * 127 * 127


def test_adversarial_rows_take_the_chunked_lists_at_k_4096():
    # H = I = 4096: with one accumulator the GEMMs take 192-row token tiles, but the exact
    # 1024-K chunked accumulation fits TMEM only with 96-row tiles, so the routing step also
    # builds both work lists in 96-row tiles and the GEMMs switch to them when the exactness
    # bound fails. Constant token rows (codes +-127) and an expert whose gate, up and down rows
    # are all 127 make the gate accumulators reach 4096 * 127^2 and the down accumulators pass
    # 2^24, so both GEMMs must take the chunked lists; every int32 stays bit-exact.
    sh = synth.LayerShape(T=40, H=4096, E=4, k=2, I=4096, Is=0)
    d = synth.small_layer(sh.T, sh.H, sh.E, sh.k, sh.I, sh.Is, seed=33)
    W = d["weights"]
    W["w_gate"][0] = 127
    W["w_up"][0] = 127
    W["w_down"][0] = 127
    x = d["x"].float()
    x[:20] = 0.75
    x[20:30] = -2.0
    x = x.to(torch.bfloat16)
    lg = d["logits"].clone()
    lg[:, 0] += 10.0                  # every token routes to expert 0
    Wd = weights_to(W, "cuda")
    layer = moe.MoELayer(sh.E, sh.k, sh.H, sh.I, sh.Is, sh.T, Wd)
    try:
        moe.moe_plan_set_decode_rows(layer.plan, 0)  # the grouped GEMMs
        st = check_layer(sh, x, lg, Wd, oracle_layer(W, sh), layer=layer,
                         sample=np.arange(0, sh.T, 3))
    finally:
        layer.close()
    assert np.abs(st["tap"]["acc_gu"]).max() == 4096 * 127 * 127
    # the h codes vary with the channels' weight scales, but the down sums still pass 2^24
    assert np.abs(st["tap"]["acc_d"]).max() > 1 << 24


@pytest.mark.parametrize("T", [2600, 77])
def test_router_tensor_core_projection(T):
    # bf16 x against the exact three-part bf16 split of the fp32 router weight: within the
    # fp32-accumulation bound of a 3H-term dot product of the oracle's double logits.
    H, E = 2048, 128
    x = synth.make_activations(T, H, 5)
    wr = synth.make_router_weight(H, E, 5)
    packed = moe.moe_router_pack(wr.cuda())
    lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
    moe.moe_router_logits_packed(x.cuda(), packed, lg)
    ref = oracle.router_logits(x, wr)
    mag = np.abs(x.float().numpy()) @ np.abs(wr.numpy())
    bound = (3 * H + 1) * 2.0 ** -23 * mag + 1e-6
    err = np.abs(lg.cpu().numpy() - ref)
    assert (err <= bound).all()
    assert np.sqrt((err ** 2).mean()) <= 5e-5 * np.sqrt((ref ** 2).mean())
