"""Shared test helpers: run one layer through the C ABI and compare it with the oracle.

Inputs come from synth (seeded); expected values come only from the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import grouped_expert_ffn_gb300 as moe

# Output tolerance of the layer (fp32 output against the oracle's double combine).
Y_MAX_REL = 1e-2      # max |dy| <= Y_MAX_REL * max |y_ref|
Y_RMSE_REL = 5e-3     # rms(dy) <= Y_RMSE_REL * rms(y_ref)
W_ABS = 1e-6          # routing weights
HQ_MISMATCH_FRAC = 1e-3
DOWN_SKIP_FRAC = 1e-3   # rows left out of the bit-exact down comparison by an h-code tie
SH_ULPS = 4             # h scales: amax / 127 of SiLU outputs that may differ in the last ulp


def weights_to(W: dict, device) -> dict:
    return {k: v.to(device).contiguous() for k, v in W.items()}


def oracle_layer(W: dict, sh: synth.LayerShape) -> oracle.Layer:
    return oracle.Layer({k: v.cpu() for k, v in W.items()}, sh.E, sh.k, sh.H, sh.I, sh.Is)


def y_errors(y, y_ref):
    y = np.asarray(y, np.float64)
    d = y - y_ref
    mx = np.abs(d).max() / max(np.abs(y_ref).max(), 1e-30)
    rm = np.sqrt((d ** 2).mean()) / max(np.sqrt((y_ref ** 2).mean()), 1e-30)
    return mx, rm


def row_map(perm: np.ndarray, T: int, k: int, has_shared: bool):
    """row[t, slot] in the library's row order (slot k = shared expert)."""
    T_sh = T if has_shared else 0
    rows = np.full((T, k + 1), -1, np.int64)
    if has_shared:
        rows[:, k] = np.arange(T)
    p = np.arange(T * k)
    rows[perm // k, perm % k] = T_sh + p
    return rows


def oracle_layer_nvfp4(W: dict, sh: synth.LayerShape) -> oracle.LayerNvfp4:
    return oracle.LayerNvfp4({k: v.cpu() for k, v in W.items()}, sh.E, sh.k, sh.H, sh.I, sh.Is)


_E2M1 = None


def nvfp4_row_norms(codes, scales) -> np.ndarray:
    """L2 norm of every weight row e2m1(code) * e4m3(block scale) (no matrix scale), decoded
    here from the E2M1 table of the OCP MX specification and torch's float8_e4m3fn."""
    global _E2M1
    if _E2M1 is None:
        import json
        import os
        _E2M1 = np.array(json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                                      "e2m1_codes.json")))["values"], np.float64)
    c = np.asarray(codes, np.uint8)
    sc = np.asarray(scales, np.uint8)
    lead = c.shape[:-1]
    c2 = c.reshape(-1, c.shape[-1])
    s2 = sc.reshape(-1, sc.shape[-1])
    out = np.empty(c2.shape[0])
    for a in range(0, c2.shape[0], 4096):
        cc = c2[a:a + 4096]
        nib = np.stack([cc & 15, cc >> 4], axis=-1).reshape(cc.shape[0], -1)
        sv = torch.from_numpy(np.ascontiguousarray(s2[a:a + 4096])).view(torch.float8_e4m3fn).double().numpy()
        v = _E2M1[nib] * np.repeat(sv, 16, axis=-1)
        out[a:a + 4096] = np.sqrt((v * v).sum(-1))
    return out.reshape(lead)


# Tensor-core accumulation of NVFP4 products (fp32, K/16 additions into the accumulator): the
# accumulators are compared within ACC_F32_REL * ||q|| * ||w'||, which bounds
# ACC_F32_REL * sum |q w'| from above (Cauchy-Schwarz) and is far above (K/16 + 1) * 2^-23 of it.
ACC_F32_REL = 1e-4


def check_layer(sh: synth.LayerShape, x_cpu, logits_cpu, W_dev: dict, L,
                sample=None, layer: moe.MoELayer | None = None, plan_tokens=None,
                acc_exact: bool = True):
    """Full parity of one layer call. Returns a dict of statistics. L is the oracle's layer:
    oracle.Layer (int8 weights) or oracle.LayerNvfp4 (NVFP4 weights; the accumulators are
    then the fp64 taps, compared bit-exactly with the oracle's exact sums, or, with
    acc_exact=False (the tensor-core path's fp32 accumulation), within ACC_F32_REL of the
    product of the two operand rows' norms)."""
    fp4 = isinstance(L, oracle.LayerNvfp4)
    tap_gu, tap_d = (moe.TAP_ACC_GU_F64, moe.TAP_ACC_D_F64) if fp4 else (moe.TAP_ACC_GU, moe.TAP_ACC_D)
    forward = oracle.forward_nvfp4 if fp4 else oracle.forward
    dev = torch.device("cuda")
    T, k, E, H = sh.T, sh.k, sh.E, sh.H
    own = layer is None
    if own:
        layer = moe.MoELayer(E, k, H, sh.I, sh.Is, plan_tokens or T, W_dev)
    try:
        x = x_cpu.to(dev)
        lg = logits_cpu.to(dev)
        idx_g, w_g = layer.route(lg)
        idx_o, w_o = oracle.route(logits_cpu, k)
        idx_g_h = idx_g.cpu().numpy()
        assert (idx_g_h == idx_o).all(), "routing indices differ"
        assert np.abs(w_g.cpu().numpy() - w_o).max() <= W_ABS
        moe.moe_debug_enable(layer.plan, True)
        y = layer.forward(x, idx_g, w_g)
        torch.cuda.synchronize()
        assert moe.moe_get_error(layer.plan) == 0
        tap = {n: moe.moe_debug_tap(layer.plan, i) for n, i in (
            ("counts", moe.TAP_COUNTS), ("offsets", moe.TAP_OFFSETS), ("perm", moe.TAP_PERM),
            ("qx", moe.TAP_QX), ("sx", moe.TAP_SX), ("acc_gu", tap_gu), ("hq", moe.TAP_HQ),
            ("sh", moe.TAP_SH), ("acc_d", tap_d))}
        counts, offsets, perm = oracle.permute(idx_o, E)
        assert (tap["counts"] == counts).all()
        assert (tap["offsets"] == offsets).all()
        assert (tap["perm"] == perm).all()
        q_o, s_o = oracle.quant_rows(x_cpu)
        assert (tap["qx"].reshape(T, H) == q_o).all()
        assert (tap["sx"] == s_o).all()

        toks = np.arange(T) if sample is None else np.asarray(sample)
        y_o, tp = forward(L, x_cpu[torch.from_numpy(toks)], idx_o[toks], w_o[toks], taps=True)
        has_sh = sh.Is > 0
        Imax = max(sh.I, sh.Is)
        R = T * k + (T if has_sh else 0)
        rows = row_map(perm, T, k, has_sh)
        acc_gu = tap["acc_gu"].reshape(R, 2, Imax)
        hq = tap["hq"].reshape(R, Imax)
        shs = tap["sh"]
        acc_d = tap["acc_d"].reshape(R, H)
        n_hq_diff = 0
        n_hq = 0
        n_rows_d = 0
        if not acc_exact:
            A = L.arrs
            norm_cache = {}

            def wnorms(e):
                """Row norms of (gate, up, down) of routed expert e, or of the shared expert
                (e None), decoded once per expert the sample touches."""
                if e not in norm_cache:
                    if e is None:
                        norm_cache[e] = [nvfp4_row_norms(A["sh_" + n], A["sh_b_" + n])
                                         for n in ("gate", "up", "down")]
                    else:
                        norm_cache[e] = [nvfp4_row_norms(A["w_" + n][e], A["b_" + n][e])
                                         for n in ("gate", "up", "down")]
                return norm_cache[e]
            qn = np.sqrt((tp["qx"].astype(np.float64) ** 2).sum(1))

        def acc_ok(got, ref, bound):
            if acc_exact:
                return (got == ref).all()
            return (np.abs(got - ref) <= ACC_F32_REL * bound).all()
        for i, t in enumerate(toks):
            for s in range(k + (1 if has_sh else 0)):
                Ig = sh.Is if s == k else sh.I
                r = rows[t, s]
                if acc_exact:
                    bgu = bd = None
                else:
                    wn = wnorms(None if s == k else int(idx_o[t, s]))
                    bgu = qn[i] * np.stack([wn[0][:Ig], wn[1][:Ig]])
                    hn = np.sqrt((tp["hq"][i, s, :Ig].astype(np.float64) ** 2).sum())
                    wdn = wn[2]  # norms of the down rows
                    bd = hn * wdn
                assert acc_ok(acc_gu[r, :, :Ig], tp["acc_gu"][i, s, :, :Ig], bgu), (t, s)
                dq = np.abs(hq[r, :Ig].astype(np.int32) - tp["hq"][i, s, :Ig].astype(np.int32))
                assert dq.max() <= 1, (t, s)
                n_hq_diff += int((dq != 0).sum())
                n_hq += Ig
                # the row's scale comes from an amax over SiLU outputs whose exp may differ in
                # the last ulp between the CUDA and host math libraries
                s_o = np.float32(tp["sh"][i, s])
                if acc_exact:
                    assert abs(float(shs[r]) - float(s_o)) <= SH_ULPS * float(np.spacing(s_o)), (t, s)
                else:  # the amax of h moves with the fp32 accumulation of g and u
                    assert abs(float(shs[r]) - float(s_o)) <= 1e-3 * float(s_o), (t, s)
                # the down accumulators depend only on the h codes (not on their scale): compared
                # bit-exactly on every row whose codes agree; with fp32 accumulation on every
                # row, the bound widened by what the differing codes can contribute
                # (||dq|| * ||w'||, Cauchy-Schwarz)
                if acc_exact and dq.max() == 0:
                    assert acc_ok(acc_d[r], tp["acc_d"][i, s], bd), (t, s)
                    n_rows_d += 1
                elif not acc_exact:
                    dqn = np.sqrt((dq.astype(np.float64) ** 2).sum())
                    assert (np.abs(acc_d[r] - tp["acc_d"][i, s]) <=
                            ACC_F32_REL * bd + dqn * wdn).all(), (t, s)
                    n_rows_d += 1
        assert n_hq_diff <= HQ_MISMATCH_FRAC * n_hq, (n_hq_diff, n_hq)
        # the bit-exact down check must have covered nearly every compared row (a run in which
        # many rows' h codes differed would otherwise skip it silently): at most 0.1% of the
        # rows, or 2 rows in a small sample, may be left out by a one-code tie difference
        n_rows = len(toks) * (k + (1 if has_sh else 0))
        assert n_rows - n_rows_d <= max(2, DOWN_SKIP_FRAC * n_rows), (n_rows_d, n_rows)
        yg = y.cpu().numpy().astype(np.float64)[toks]
        mx, rm = y_errors(yg, y_o)
        assert mx <= Y_MAX_REL and rm <= Y_RMSE_REL, (mx, rm)
        print(f"parity: y max_rel {mx:.2e} rmse_rel {rm:.2e}; h codes differing {n_hq_diff} of "
              f"{n_hq}; down rows compared bit-exactly {n_rows_d} of {n_rows}")
        return dict(max_rel=mx, rmse_rel=rm, hq_diff=n_hq_diff, hq_total=n_hq,
                    rows_down_exact=n_rows_d, y=y, idx=idx_g, w=w_g, tap=tap)
    finally:
        if own:
            layer.close()
