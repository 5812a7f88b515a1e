"""Workload recipes and seeded generators for the dropless MoE layer.

The five workloads are the layer shapes the MoE training pages revolve around:
a tiny fp32 layer, a mid-size bf16 layer, a DeepSeek-V3-shaped layer (256
routed experts, hidden 7168; MindSpore DeepSeek-V3 pre-training page, section
01.1), a Pangu-Ultra-MoE-shaped layer (hidden 7680, 256 routed + 1 shared
expert of width 2048, 8K sequence; reportify Pangu Ultra MoE summary) and an
adversarial-imbalance step at the Pangu shapes with T = 16384.

Recipe (every draw is seeded; seed = workload index, the tiny one is seed 0):

* draw order ``x, W_r, W13, W2, Ws13, Ws2, bias permutation, dY`` for the
  plain and Zipf-routed workloads; ``x, W13, W2, Ws13, Ws2, dY`` and then the
  logit construction for the adversarial one;
* ``x ~ N(0, 1)``, all weights ``~ N(0, 0.02)``, ``dY ~ N(0, 1)``, drawn in
  fp32 and rounded to bf16 (round-to-nearest-even) for the bf16 workloads;
  expert weights are drawn one expert at a time so that the fp32 temporaries
  stay small;
* the router weight ``W_r [d, E]`` stays fp32 (the pages keep the routing
  network in FP32);
* Zipf routing skew: a constant per-expert bias ``b_e = -s * ln(r_e)`` with
  ``r`` a seeded permutation of ``1..E``, so that ``exp(b_e)`` follows a
  rank-Zipf law with exponent ``s`` (s = 1.1 DeepSeek-V3-shaped, 0.8
  Pangu-shaped);
* adversarial routing: the router logits are the layer input.  Base logits
  ``N(0, 1)``; a quarter of the experts (64 of 256) are "dead" (logit -30 in
  every row); one "hot" expert is forced to the top in ceil(0.10 * T * k) rows
  chosen by a seeded permutation (logit = row max + 1) and is -30 elsewhere, so
  it holds exactly 10 % of the token copies; in ceil(0.01 * T) rows the
  (k+1)-th largest logit is overwritten with the k-th largest (an exact tie
  straddling the top-k boundary) and in a further ceil(0.005 * T) rows the 3rd
  largest is overwritten with the 2nd (a tie inside the top-k).

Replicas (one per rank of a multi-GPU run, data parallel): replica 0 is the draw
above; replica r > 0 keeps its weights, router and bias, and draws its own token
side (``x``, ``dY`` and, for the adversarial workload, the logit construction)
from a second generator seeded with ``seed + REPLICA_SEED_STRIDE * r``.

Expert weight layouts are K-major: ``W13 [E][2f][d]`` (gate rows ``0..f-1``,
up rows ``f..2f-1``), ``W2 [E][d][f]``; the shared experts use the same
layouts ``Ws13 [S][2f_s][d]``, ``Ws2 [S][d][f_s]``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

CONFIGS = {
    "tiny_fp32": dict(T=256, d=512, E=8, k=2, f=256, S=0, f_s=0, dtype="f32",
                      seed=0, bwd=True, routing="plain", zipf_s=0.0),
    "mid_bf16": dict(T=4096, d=2048, E=64, k=6, f=1408, S=2, f_s=1408, dtype="bf16",
                     seed=1, bwd=False, routing="plain", zipf_s=0.0),
    "dsv3_bf16": dict(T=8192, d=7168, E=256, k=8, f=2048, S=1, f_s=2048, dtype="bf16",
                      seed=2, bwd=True, routing="zipf", zipf_s=1.1),
    "pangu_bf16": dict(T=8192, d=7680, E=256, k=8, f=2048, S=1, f_s=2048, dtype="bf16",
                       seed=3, bwd=True, routing="zipf", zipf_s=0.8),
    "adversarial_bf16": dict(T=16384, d=7680, E=256, k=8, f=2048, S=1, f_s=2048, dtype="bf16",
                             seed=4, bwd=True, routing="adversarial", zipf_s=0.0),
}

DEAD_FRACTION = 0.25
HOT_COPY_FRACTION = 0.10
BOUNDARY_TIE_FRACTION = 0.01
INNER_TIE_FRACTION = 0.005
DEAD_LOGIT = -30.0
WEIGHT_STD = 0.02
REPLICA_SEED_STRIDE = 7919


def shrink(name: str, **overrides) -> dict:
    """The recipe of workload ``name`` with some sizes replaced (for small cases)."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    cfg["name"] = name if not overrides else name + "_" + "_".join(
        f"{k}{v}" for k, v in sorted(overrides.items()))
    return cfg


@dataclasses.dataclass
class Workload:
    cfg: dict
    x: torch.Tensor                      # [T, d] fp32 or bf16
    w_r: Optional[torch.Tensor]          # [d, E] fp32 (None when logits are the input)
    bias: Optional[torch.Tensor]         # [E] fp32 (Zipf skew) or None
    w13: torch.Tensor                    # [E, 2f, d]
    w2: torch.Tensor                     # [E, d, f]
    ws13: Optional[torch.Tensor]         # [S, 2f_s, d] or None
    ws2: Optional[torch.Tensor]          # [S, d, f_s] or None
    dy: torch.Tensor                     # [T, d]
    logits_in: Optional[torch.Tensor]    # [T, E] fp32 (adversarial) or None
    info: dict                           # which experts are dead/hot, tie rows

    @property
    def torch_dtype(self):
        return torch.float32 if self.cfg["dtype"] == "f32" else torch.bfloat16


def _normal(g, shape, std, device, dtype):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _expert_stack(g, n, shape, device, dtype):
    out = torch.empty((n,) + tuple(shape), device=device, dtype=dtype)
    for i in range(n):
        out[i] = _normal(g, shape, WEIGHT_STD, device, dtype)
    return out


def _adversarial_logits(g, T, E, k, device):
    base = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
    eperm = torch.randperm(E, generator=g, device=device)
    n_dead = int(E * DEAD_FRACTION)
    dead = eperm[:n_dead]
    hot = int(eperm[n_dead].item())
    rperm = torch.randperm(T, generator=g, device=device)
    n_hot = min(T, math.ceil(HOT_COPY_FRACTION * T * k))
    hot_rows = rperm[:n_hot]
    base[:, dead] = DEAD_LOGIT
    base[:, hot] = DEAD_LOGIT
    row_max = base.max(dim=1).values
    base[hot_rows, hot] = row_max[hot_rows] + 1.0

    tperm = torch.randperm(T, generator=g, device=device)
    n_bt = max(1, math.ceil(BOUNDARY_TIE_FRACTION * T))
    n_it = max(1, math.ceil(INNER_TIE_FRACTION * T))
    bt_rows = tperm[:n_bt]
    it_rows = tperm[n_bt:n_bt + n_it]
    # Rank the candidates of the chosen rows (descending, lower index first on
    # equal values) to know which entries to overwrite.
    if n_bt:
        sub = base[bt_rows]
        order = torch.sort(-sub, dim=1, stable=True).indices
        kth = order[:, k - 1]
        k1th = order[:, k]
        ar = torch.arange(sub.shape[0], device=device)
        sub[ar, k1th] = sub[ar, kth]
        base[bt_rows] = sub
    if n_it and k >= 3:
        sub = base[it_rows]
        order = torch.sort(-sub, dim=1, stable=True).indices
        ar = torch.arange(sub.shape[0], device=device)
        sub[ar, order[:, 2]] = sub[ar, order[:, 1]]
        base[it_rows] = sub
    info = dict(dead=sorted(int(i) for i in dead.tolist()), hot=hot, n_hot_rows=n_hot,
                boundary_tie_rows=sorted(int(i) for i in bt_rows.tolist()),
                inner_tie_rows=sorted(int(i) for i in it_rows.tolist()))
    return base, info


def make_workload(cfg, device="cpu", with_dy: bool = True, replica: int = 0) -> Workload:
    """Draw the inputs of one workload.  ``cfg`` is a name of CONFIGS or a dict.
    ``replica`` > 0: the same weights with that replica's own token batch."""
    if isinstance(cfg, str):
        cfg = dict(CONFIGS[cfg], name=cfg)
    cfg = dict(cfg)
    T, d, E, k, f, S, f_s = (cfg[n] for n in ("T", "d", "E", "k", "f", "S", "f_s"))
    dt = torch.float32 if cfg["dtype"] == "f32" else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(int(cfg["seed"]))
    x = _normal(g, (T, d), 1.0, device, dt)
    w_r = None
    if cfg["routing"] != "adversarial":
        w_r = _normal(g, (d, E), WEIGHT_STD, device, torch.float32)
    w13 = _expert_stack(g, E, (2 * f, d), device, dt)
    w2 = _expert_stack(g, E, (d, f), device, dt)
    ws13 = ws2 = None
    if S > 0:
        ws13 = _expert_stack(g, S, (2 * f_s, d), device, dt)
        ws2 = _expert_stack(g, S, (d, f_s), device, dt)
    bias = None
    info = {}
    if cfg["routing"] == "zipf":
        r = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
        bias = (-float(cfg["zipf_s"]) * torch.log(r)).to(torch.float32)
    dy = _normal(g, (T, d), 1.0, device, dt) if with_dy else None
    logits_in = None
    if cfg["routing"] == "adversarial":
        logits_in, info = _adversarial_logits(g, T, E, k, device)
    if replica > 0:
        gr = torch.Generator(device=device)
        gr.manual_seed(int(cfg["seed"]) + REPLICA_SEED_STRIDE * int(replica))
        x = _normal(gr, (T, d), 1.0, device, dt)
        dy = _normal(gr, (T, d), 1.0, device, dt) if with_dy else None
        if cfg["routing"] == "adversarial":
            logits_in, info = _adversarial_logits(gr, T, E, k, device)
    return Workload(cfg=cfg, x=x, w_r=w_r, bias=bias, w13=w13, w2=w2, ws13=ws13, ws2=ws2,
                    dy=dy, logits_in=logits_in, info=info)
