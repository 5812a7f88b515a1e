"""Why the score gradients of a few-token bf16 layer get a wider bar (CPU, oracle only).

The device stores the SwiGLU pre-activations Z = [a | b] in bf16 and forms the gradient with
respect to a gate as dgate = sum_f D_f silu(a_f) b_f from them. Rounding the oracle's exact
pre-activations to bf16 (round to nearest even) and recomputing dgate and the score gradient
in fp64 shows the size of that one effect: about 2.5e-3 of the score gradient when many
tokens contribute, one draw of up to ~7e-3 for a single token. The bars of the GPU parity
tests follow from this: 5e-3 for every case with at least 16 tokens, 1e-2 below."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import make_workload, shrink


def _bf16(a):
    return torch.as_tensor(a, dtype=torch.float32).to(torch.bfloat16).double().numpy()


def _score_grad_error_from_bf16_z(cfg):
    """Relative error of the score gradient (and of dgate) when Z is rounded to bf16."""
    w = make_workload(cfg)
    k, f = cfg["k"], cfg["f"]
    logits = O.router_logits(O.as_f64(w.x), O.as_f64(w.w_r)).astype(np.float32)
    idx, gate = O.route_topk(O.selection_scores(logits, w.bias.numpy()), k)
    x, dy = O.as_f64(w.x), O.as_f64(w.dy)
    w13, w2 = O.as_f64(w.w13), O.as_f64(w.w2)
    exact = np.zeros(idx.shape)
    rounded = np.zeros(idx.shape)
    for e in np.unique(idx):
        t, j = np.nonzero(idx == e)
        Z = x[t] @ w13[e].T
        D = dy[t] @ w2[e]
        exact[t, j] = np.sum(D * O.silu(Z[:, :f]) * Z[:, f:], axis=1)
        Zr = _bf16(Z)
        rounded[t, j] = np.sum(D * O.silu(Zr[:, :f]) * Zr[:, f:], axis=1)
    dl, dlr = O.router_backward(gate, exact), O.router_backward(gate, rounded)
    return (float(np.linalg.norm(dlr - dl) / np.linalg.norm(dl)),
            float(np.linalg.norm(rounded - exact) / np.linalg.norm(exact)))


@pytest.mark.parametrize("over,lo,hi", [
    (dict(T=1, d=128, E=100, k=4, f=320, S=0, f_s=0), 5e-3, 1e-2),   # one token: above 5e-3
    (dict(T=1, d=256, E=8, k=2, f=128, f_s=128), 4e-3, 1e-2),
])
def test_one_token_score_gradient_error_comes_from_bf16_z(over, lo, hi):
    err, _ = _score_grad_error_from_bf16_z(shrink("pangu_bf16", **over))
    assert lo <= err <= hi, err


@pytest.mark.parametrize("over", [dict(T=640, d=512, E=16, k=4, f=256, f_s=256),
                                  dict(T=384, d=448, E=24, k=3, f=320, f_s=192)])
def test_many_token_score_gradient_error_is_within_the_plain_bar(over):
    err, dgate_err = _score_grad_error_from_bf16_z(shrink("pangu_bf16", **over))
    assert err <= 3.5e-3 and dgate_err <= 3.5e-3, (err, dgate_err)
