"""Helpers shared by the GPU parity tests: run the CUDA layer through the C ABI and the
fp64 oracle on the same seeded inputs, and compare.

Bars: bit-exact for routing indices, counts, offsets, dest, row_src and the permuted
rows; ||gpu - oracle|| / ||oracle|| <= 1e-5 for fp32 workloads and for the fp32 gates
and scores of every workload; <= 5e-3 for bf16 outputs and gradients, the score
gradients (dlogits, dW_r) included, except those of bf16 layers with fewer than 16 tokens
(<= 1e-2, see FEW_TOKENS below).

MOE_PARITY_LOG=<file> appends one JSON line per checked case with every measured error."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle as O

TOL = {"f32": 1e-5, "bf16": 5e-3}
GATE_TOL = 1e-5
# Score gradients (dlogits, dW_r) of a bf16 layer with fewer than FEW_TOKENS tokens. The
# gradient with respect to a gate, sum_f D * silu(a) * b, is formed from the bf16-rounded
# pre-activations a and b that the forward stores; over many tokens the rounding errors
# average to about 2.5e-3 of the score gradient, but for one token the error is a single
# draw and reaches 5-8e-3 (rounding the exact pre-activations to bf16 on the host gives the
# same error to three digits). Those tensors are held to this bar; every other case to TOL.
FEW_TOKENS = 16
FEW_TOKENS_SCORE_TOL = 1e-2


def rel(gpu, ref) -> float:
    a = O.as_f64(gpu)
    b = np.asarray(ref, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    nb = np.linalg.norm(b)
    na = np.linalg.norm(a - b)
    if nb == 0.0:
        return float(na)
    return float(na / nb)


def _to(t, dev="cuda"):
    return None if t is None else t.to(dev)


def run_gpu_layer(w, bwd=True, capacity=0, rearrange=0):
    from dropless_token_routing_gb300.api import LayerParams, MoELayer, get_device_error
    c = w.cfg
    params = LayerParams(w13=_to(w.w13), w2=_to(w.w2), w_r=_to(w.w_r), bias=_to(w.bias),
                         ws13=_to(w.ws13), ws2=_to(w.ws2))
    layer = MoELayer(params, c["T"], c["d"], c["E"], c["k"], c["f"], c["S"], c["f_s"],
                     w.torch_dtype, logits_input=w.logits_in is not None, capacity=capacity,
                     rearrange=rearrange)
    x = _to(w.x)
    layer.forward(x, _to(w.logits_in))
    grads = layer.backward(_to(w.dy)) if bwd else None
    torch.cuda.synchronize()
    err = get_device_error(layer.ws)
    return layer, grads, err


def oracle_layer(w, device_logits=None, bwd=True, capacity=0):
    """Oracle forward/backward with the top-k taken on the device's fp32 scores."""
    k = w.cfg["k"]
    if w.logits_in is not None:
        logits32 = w.logits_in.cpu().numpy()
    else:
        logits32 = device_logits.detach().cpu().numpy()
    bias32 = None if w.bias is None else w.bias.cpu().numpy()
    idx, gate = O.route_topk(O.selection_scores(logits32, bias32), k)
    x = O.as_f64(w.x)
    w13, w2, ws13, ws2 = (O.as_f64(t) for t in (w.w13, w.w2, w.ws13, w.ws2))
    fwd = O.layer_forward(x, idx, gate, w13, w2, ws13, ws2, capacity=capacity)
    res = dict(idx=idx, gate=gate, fwd=fwd)
    if bwd:
        res["bwd"] = O.layer_backward(x, idx, gate, fwd, O.as_f64(w.dy), w13, w2, ws13, ws2,
                                      w_r=O.as_f64(w.w_r))
    return res


def check_layer(w, bwd=True, report=None, capacity=0, rearrange=0):
    """Run both sides and assert every bar; returns a dict of the measured errors.
    capacity = C > 0 checks the drop-and-pad variant against the oracle's."""
    tol = TOL[w.cfg["dtype"]]
    layer, grads, err = run_gpu_layer(w, bwd=bwd, capacity=capacity, rearrange=rearrange)
    assert err == 0, f"device error {err}"
    s = layer.saved
    errs = {}
    if w.logits_in is None:
        ref_logits = O.router_logits(O.as_f64(w.x), O.as_f64(w.w_r))
        errs["logits"] = rel(s["logits"], ref_logits)
        assert errs["logits"] <= GATE_TOL, errs
    ref = oracle_layer(w, device_logits=s["logits"], bwd=bwd, capacity=capacity)
    fwd = ref["fwd"]
    # bit-exact routing and permutation
    assert np.array_equal(s["topk_idx"].cpu().numpy(), ref["idx"]), "topk_idx differs"
    assert np.array_equal(s["counts"].cpu().numpy(), fwd["counts"]), "counts differ"
    assert np.array_equal(s["offsets"].cpu().numpy(), fwd["offsets"]), "offsets differ"
    assert np.array_equal(s["dest"].cpu().numpy(), fwd["dest"]), "dest differs"
    assert np.array_equal(s["row_src"].cpu().numpy(), fwd["row_src"]), "row_src differs"
    src = torch.as_tensor(fwd["row_src"])
    xp = torch.zeros(len(src), w.x.shape[1], dtype=w.x.dtype)   # padding rows are zero
    xp[src >= 0] = w.x[src[src >= 0]]
    assert torch.equal(s["x_perm"].cpu(), xp), "x_perm differs"
    errs["topk_w"] = rel(s["topk_w"], ref["gate"])
    errs["w_perm"] = rel(s["w_perm"], fwd["w_perm"])
    errs["z"] = rel(s["z"], fwd["z"])
    errs["h"] = rel(s["h"], fwd["h"])
    errs["y"] = rel(layer.y, fwd["y"])
    if w.cfg["S"]:
        errs["z_sh"] = rel(s["z_sh"], np.concatenate(fwd["z_sh"], 0))
        errs["h_sh"] = rel(s["h_sh"], np.concatenate(fwd["h_sh"], 0))
    assert errs["topk_w"] <= GATE_TOL and errs["w_perm"] <= GATE_TOL, errs
    for n in ("z", "h", "y", "z_sh", "h_sh"):
        if n in errs:
            assert errs[n] <= tol, (n, errs)
    if bwd:
        b = ref["bwd"]
        errs["dx"] = rel(grads["dx"], b["dx"])
        errs["dw13"] = rel(grads["dw13"], b["dw13"])
        errs["dw2"] = rel(grads["dw2"], b["dw2"])
        if w.cfg["S"]:
            errs["dws13"] = rel(grads["dws13"], b["dws13"])
            errs["dws2"] = rel(grads["dws2"], b["dws2"])
        if grads["dw_r"] is not None:
            errs["dw_r"] = rel(grads["dw_r"], b["dw_r"])
        if grads["dlogits"] is not None:
            errs["dlogits"] = rel(grads["dlogits"], b["dscores"])
        # how far the score gradient dL_j = w_j (dgate_j - sum_i w_i dgate_i) cancels: the norm
        # of its terms w_j |dgate_j| over its own norm (reported, not a bar)
        errs["score_grad_cancellation"] = float(
            np.linalg.norm(ref["gate"] * b["dgate"]) / max(np.linalg.norm(b["dscores"]), 1e-300))
        _log(w, capacity, rearrange, errs)
        few = w.cfg["dtype"] == "bf16" and w.cfg["T"] < FEW_TOKENS
        for n in ("dx", "dw13", "dw2", "dws13", "dws2", "dw_r", "dlogits"):
            if n in errs:
                bar = FEW_TOKENS_SCORE_TOL if (few and n in ("dw_r", "dlogits")) else tol
                assert errs[n] <= bar, (n, errs)
        # experts without tokens keep exactly zero gradients
        empty = np.nonzero(fwd["counts"] == 0)[0]
        for e in empty:
            assert not grads["dw13"][int(e)].any() and not grads["dw2"][int(e)].any()
    if report is not None:
        report.update(errs)
    return layer, grads, errs


def _log(w, capacity, rearrange, errs):
    path = os.environ.get("MOE_PARITY_LOG")
    if path:
        with open(path, "a") as fh:
            fh.write(json.dumps({"case": w.cfg.get("name"), "capacity": capacity,
                                 "rearrange": rearrange, "errs": errs}) + "\n")
