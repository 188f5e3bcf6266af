"""Seeded synthetic workloads for the grouped-expert MoE FFN layer.

This module only draws inputs. It holds none of the layer's arithmetic (no routing,
no activation quantisation, no GEMM, no combine), so both the CUDA path and the CPU
oracle can take their inputs from it without sharing any method code.

Inputs follow the workload recipes of the MoE layer this library serves:

* activations ``x``: bf16, N(0,1) drawn in fp32 and rounded to bf16 (round to nearest
  even); optionally a fixed set of outlier channels scaled x20 in fp32 before rounding;
* router logits: fp32 N(0,1), optionally plus a per-expert Zipf bias
  ``-s * ln(rank_e)`` where ``rank`` is a seeded random permutation of 1..E
  (the log of a Zipf(s) rank law, so low ranks are chosen by most tokens);
* expert weights: fp32 N(0, 0.02) quantised to int8 per output channel, symmetric,
  ``scale = amax/127`` in fp32 and ``q = round_half_even(w/scale)`` clamped to +-127.
  The weight quantisation is input preparation: the layer consumes int8 weights and
  fp32 scales.

Weight layout (row-major, all contiguous):

* ``w_gate``, ``w_up``: int8 [E, I, H]; ``s_gate``, ``s_up``: fp32 [E, I]
* ``w_down``: int8 [E, H, I]; ``s_down``: fp32 [E, H]
* shared expert (``Is > 0``): ``sh_gate``, ``sh_up`` int8 [Is, H], ``sh_down`` int8
  [H, Is] and fp32 scales ``sh_s_gate``, ``sh_s_up`` [Is], ``sh_s_down`` [H].

Draw order is fixed (x, outlier channels, logits, Zipf permutation, router weight,
then expert weights gate/up/down, then the shared expert) so a seed names one workload.
Generation runs with torch on the requested device; a CUDA generator and a CPU
generator give different (each reproducible) streams.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class LayerShape:
    T: int          # tokens
    H: int          # hidden size
    E: int          # routed experts
    k: int          # top_k
    I: int          # routed expert intermediate size
    Is: int         # shared expert intermediate size (0 = no shared expert)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    seed: int
    zipf_s: float = 0.0        # 0 = no Zipf bias on the logits
    outliers: int = 0          # number of outlier channels (x20)
    layers: int = 1            # >1: stacked layers with a router projection
    router: str = "logits"     # "logits": logits drawn directly; "projection": x @ W_r
    note: str = ""


# The five workloads of the layer (sizes and seeds as stated in each note).
WORKLOADS = {
    "tiny": Workload("tiny", LayerShape(T=16, H=256, E=8, k=2, I=128, Is=0), seed=0,
                     note="tiny MoE layer T16 H256 E8 k2 I128, no shared expert"),
    "decode": Workload("decode", LayerShape(T=8, H=2048, E=128, k=8, I=512, Is=512), seed=1,
                       zipf_s=1.1, outliers=8,
                       note="35B-A3B-shaped layer, batched decode C=8 rows, Zipf(1.1) routing skew"),
    "prefill": Workload("prefill", LayerShape(T=256, H=2048, E=128, k=8, I=512, Is=512), seed=2,
                        zipf_s=1.1, outliers=8,
                        note="35B-A3B-shaped layer, one 256-token prefill chunk"),
    "stack": Workload("stack", LayerShape(T=2600, H=2048, E=128, k=8, I=512, Is=512), seed=3,
                      layers=40, router="projection",
                      note="40-layer stacked prefill, T=2600, router = N(0,1) [H,E] projection, residual"),
    "stress": Workload("stress", LayerShape(T=8192, H=4096, E=256, k=8, I=1024, Is=2048), seed=4,
                       zipf_s=1.5,
                       note="load-imbalance stress layer T8192 H4096 E256 k8 I1024 Is2048, Zipf(1.5)"),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def quantize_weight_rows(w: torch.Tensor):
    """int8 symmetric per-output-channel quantisation of weight rows (last dim reduced).

    scale = amax/127 in fp32; q = round-half-even(w / scale) clamped to [-127, 127];
    an all-zero row gets scale 0 and q 0. Returns (q int8, scale fp32)."""
    w = w.float()
    amax = w.abs().amax(dim=-1, keepdim=True)
    s = amax / 127.0
    safe = torch.where(s > 0, s, torch.ones_like(s))
    q = torch.round(w / safe).clamp_(-127, 127)
    q = torch.where(s > 0, q, torch.zeros_like(q))
    return q.to(torch.int8), s.squeeze(-1).contiguous()


def _normal_q(shape, g, device, std=0.02, chunk_rows=None):
    """N(0,std) fp32 draws quantised per row, generated in slabs along dim 0 to bound
    the fp32 temporary."""
    out_q = torch.empty(shape, dtype=torch.int8, device=device)
    out_s = torch.empty(shape[:-1], dtype=torch.float32, device=device)
    n0 = shape[0]
    step = chunk_rows or n0
    for a in range(0, n0, step):
        b = min(n0, a + step)
        w = torch.randn((b - a,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32) * std
        q, s = quantize_weight_rows(w)
        out_q[a:b] = q
        out_s[a:b] = s
        del w
    return out_q, out_s


def make_weights(shape: LayerShape, seed: int, device="cpu", slab: int = 16) -> dict:
    """Quantised routed + shared expert weights for one layer (see module docstring)."""
    g = _gen(seed * 1000 + 17, device)
    E, H, I, Is = shape.E, shape.H, shape.I, shape.Is
    wg, sg = _normal_q((E, I, H), g, device, chunk_rows=slab)
    wu, su = _normal_q((E, I, H), g, device, chunk_rows=slab)
    wd, sd = _normal_q((E, H, I), g, device, chunk_rows=slab)
    W = dict(w_gate=wg, s_gate=sg, w_up=wu, s_up=su, w_down=wd, s_down=sd)
    if Is > 0:
        shg, shsg = _normal_q((Is, H), g, device)
        shu, shsu = _normal_q((Is, H), g, device)
        shd, shsd = _normal_q((H, Is), g, device)
        W.update(sh_gate=shg, sh_s_gate=shsg, sh_up=shu, sh_s_up=shsu,
                 sh_down=shd, sh_s_down=shsd)
    return W


def make_activations(T: int, H: int, seed: int, outliers: int = 0, device="cpu") -> torch.Tensor:
    """x bf16 [T, H] ~ N(0,1); `outliers` fixed channels (same for every token) x20."""
    g = _gen(seed * 1000 + 1, device)
    x = torch.randn((T, H), generator=g, device=device, dtype=torch.float32)
    if outliers:
        ch = torch.randperm(H, generator=g, device=device)[:outliers]
        x[:, ch] *= 20.0
    return x.to(torch.bfloat16)


def zipf_bias(E: int, s: float, g: torch.Generator, device) -> torch.Tensor:
    """Per-expert logit bias -s*ln(rank), rank = seeded permutation of 1..E."""
    perm = torch.randperm(E, generator=g, device=device)
    rank = torch.empty(E, dtype=torch.float32, device=device)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float32, device=device)
    return -s * torch.log(rank)


def make_logits(T: int, E: int, seed: int, zipf_s: float = 0.0, device="cpu") -> torch.Tensor:
    """Router logits fp32 [T, E] ~ N(0,1) (+ Zipf rank bias when zipf_s > 0)."""
    g = _gen(seed * 1000 + 2, device)
    logits = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
    if zipf_s > 0:
        logits = logits + zipf_bias(E, zipf_s, g, device)[None, :]
    return logits.contiguous()


def make_router_weight(H: int, E: int, seed: int, device="cpu") -> torch.Tensor:
    """Router projection W_r fp32 [H, E] ~ N(0,1) (stacked-prefill workload)."""
    g = _gen(seed * 1000 + 3, device)
    return torch.randn((H, E), generator=g, device=device, dtype=torch.float32)


def layer_seed(wl: Workload, layer: int) -> int:
    return wl.seed + layer


def make_layer(wl: Workload, device="cpu", layer: int = 0, with_weights: bool = True) -> dict:
    """One layer of a workload: x, logits (or router weight) and weights."""
    sh = wl.shape
    seed = layer_seed(wl, layer)
    d = {"shape": sh, "seed": seed}
    d["x"] = make_activations(sh.T, sh.H, seed, wl.outliers, device)
    if wl.router == "projection":
        d["w_router"] = make_router_weight(sh.H, sh.E, seed, device)
    else:
        d["logits"] = make_logits(sh.T, sh.E, seed, wl.zipf_s, device)
    if with_weights:
        d["weights"] = make_weights(sh, seed, device)
    return d


def small_layer(T, H, E, k, I, Is, seed, zipf_s=0.0, outliers=0, device="cpu") -> dict:
    """Ad-hoc small layer for tests (any shape)."""
    wl = Workload("adhoc", LayerShape(T, H, E, k, I, Is), seed, zipf_s, outliers)
    return make_layer(wl, device)


# NVFP4 expert weights. The same N(0, 0.02) draws quantised to NVFP4 instead of int8 (input
# preparation, as for int8): per weight matrix a fp32 scale gs = amax / (6 * 448); per block
# of 16 consecutive elements of a row an E4M3 scale = amax_block / (6 * gs) rounded to E4M3
# (torch's float8_e4m3fn conversion, round to nearest even); each element w / (scale * gs)
# rounded to the nearest E2M1 magnitude (0, 0.5, 1, 1.5, 2, 3, 4, 6; saturating at 6) with
# its sign. Codes are packed two per byte, element 2j in the low nibble.
_E2M1_BOUNDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def quantize_nvfp4_rows(w: torch.Tensor, gs: torch.Tensor):
    """NVFP4 codes (uint8 [..., K/2]) and E4M3 block scales (uint8 [..., K/16]) of weight
    rows w [..., K] under the matrix scale gs (fp32 scalar tensor)."""
    w = w.float()
    shp = w.shape
    blk = w.reshape(*shp[:-1], shp[-1] // 16, 16)
    bs = (blk.abs().amax(-1) / (6.0 * gs)).clamp_(max=448.0)
    bs8 = bs.to(torch.float8_e4m3fn)
    bsd = bs8.float()
    safe = torch.where(bsd > 0, bsd, torch.ones_like(bsd))
    v = blk / (safe * gs)[..., None]
    bounds = torch.tensor(_E2M1_BOUNDS, dtype=torch.float32, device=w.device)
    mag = torch.bucketize(v.abs(), bounds, right=False)
    mag = torch.where(bsd[..., None] > 0, mag, torch.zeros_like(mag))
    code = (mag | torch.where(v < 0, 8, 0)).to(torch.uint8).reshape(shp)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return packed.contiguous(), bs8.view(torch.uint8).contiguous()


def _normal_nvfp4(shape, g, device, std=0.02, chunk_rows=None):
    """N(0,std) fp32 draws [n0, rows, K] (or [rows, K]) quantised to NVFP4 with one matrix
    scale per index of dim 0 (per expert) or one for the whole 2-D matrix."""
    three = len(shape) == 3
    n0 = shape[0] if three else 1
    rows, K = shape[-2], shape[-1]
    codes = torch.empty((n0, rows, K // 2), dtype=torch.uint8, device=device)
    bsc = torch.empty((n0, rows, K // 16), dtype=torch.uint8, device=device)
    gsv = torch.empty((n0,), dtype=torch.float32, device=device)
    step = chunk_rows or n0
    for a in range(0, n0, step):
        b = min(n0, a + step)
        w = torch.randn((b - a, rows, K), generator=g, device=device, dtype=torch.float32) * std
        for i in range(b - a):
            am = w[i].abs().amax()
            gs = torch.where(am > 0, am / (6.0 * 448.0), torch.ones_like(am))
            codes[a + i], bsc[a + i] = quantize_nvfp4_rows(w[i], gs)
            gsv[a + i] = gs
        del w
    if not three:
        return codes[0], bsc[0], gsv
    return codes, bsc, gsv


def make_weights_nvfp4(shape: LayerShape, seed: int, device="cpu", slab: int = 16) -> dict:
    """NVFP4 routed + shared expert weights for one layer:
    w_gate, w_up uint8 [E, I, H/2], b_gate, b_up uint8 [E, I, H/16], g_gate, g_up fp32 [E];
    w_down uint8 [E, H, I/2], b_down uint8 [E, H, I/16], g_down fp32 [E]; shared expert
    sh_gate, sh_up [Is, H/2], sh_b_gate, sh_b_up [Is, H/16], sh_down [H, Is/2],
    sh_b_down [H, Is/16] and sh_g fp32 [3] (gate, up, down)."""
    g = _gen(seed * 1000 + 19, device)
    E, H, I, Is = shape.E, shape.H, shape.I, shape.Is
    wg, bg, gg = _normal_nvfp4((E, I, H), g, device, chunk_rows=slab)
    wu, bu, gu = _normal_nvfp4((E, I, H), g, device, chunk_rows=slab)
    wd, bd, gd = _normal_nvfp4((E, H, I), g, device, chunk_rows=slab)
    W = dict(w_gate=wg, b_gate=bg, g_gate=gg, w_up=wu, b_up=bu, g_up=gu,
             w_down=wd, b_down=bd, g_down=gd)
    if Is > 0:
        shg, shbg, shgg = _normal_nvfp4((Is, H), g, device)
        shu, shbu, shgu = _normal_nvfp4((Is, H), g, device)
        shd, shbd, shgd = _normal_nvfp4((H, Is), g, device)
        W.update(sh_gate=shg, sh_b_gate=shbg, sh_up=shu, sh_b_up=shbu, sh_down=shd,
                 sh_b_down=shbd, sh_g=torch.cat([shgg, shgu, shgd]).contiguous())
    return W


def weight_bytes_per_expert_nvfp4(H: int, I: int) -> int:
    """Bytes one NVFP4 expert occupies in HBM: packed codes plus E4M3 block scales."""
    return 3 * H * I // 2 + 3 * H * I // 16


def weight_bytes_per_expert(H: int, I: int) -> int:
    """Bytes one expert occupies in HBM: int8 gate+up+down plus fp32 scales."""
    return 3 * H * I + 4 * (2 * I + H)
