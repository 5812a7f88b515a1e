"""fp64 CPU oracle of one dropless MoE layer, forward and backward.

TEST INFRASTRUCTURE: this module is the independent reference the CUDA path is
checked against.  It is imported only by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; the library never calls it.

Sources (web pages on dropless MoE training; none of them prints formulas, so
each step below is the plainest reading of the text):

* routing = softmax -> top-k selection -> mask, as one fused step
  ("MoE operator optimisation: routing hardware acceleration and zero-copy
  communication", gtnt.cn, section 2.1); the router network stays FP32
  (same page, section 4.2);
* dropless: every token copy is kept, no capacity and no padding (Pangu Ultra
  MoE tech-report article, rjtj.cn, the dropless vs drop-and-pad comparison);
* rearrange / un-rearrange of token copies into expert-contiguous order
  (Huawei MoE training-operator article, feedman.me, section "Vector operator
  (VectorSort)", Fig. 3);
* layer output = weighted sum of the routed experts plus the shared expert
  (rjtj.cn article, the shared/routed contribution analysis; one shared
  expert per the reportify Pangu Ultra MoE summary);
* backward with the expert dW and dX computed separately (rjtj.cn article,
  adaptive-pipe overlap section; MindSpore DeepSeek-V3 page, section 01.2).

Readings taken where the pages are silent (the layer contract):

* top-k: the k largest scores, in descending order, equal scores resolved
  toward the lower expert index;
* gates: softmax over all E experts, picked at the top-k and renormalised over
  them, which equals ``exp(s_e - m) / sum_{i in top-k} exp(s_i - m)``; no
  routed scaling factor;
* order of the copies inside an expert segment: stable in the flattened copy
  index ``q = t*k + j``, i.e. ascending token;
* expert FFN: SwiGLU ``(silu(x W1^T) * (x W3^T)) W2^T`` with no biases,
  ``silu(a) = a / (1 + exp(-a))``;
* shared experts are added with weight 1 and are not gated;
* a per-expert score bias is a constant added before both selection and
  gating; it has no gradient;
* the top-k indices are constants of the backward (not differentiated).

Every floating-point value here is fp64, except the selection scores when the
caller passes fp32 logits: the top-k decision is then taken on the fp32 values
themselves (and ``logits + bias`` is formed with one fp32 rounding, as the
device does), because a decision that floating point makes must be made in the
same precision on both sides.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "silu", "silu_grad", "router_logits", "selection_scores", "route_topk",
    "expert_counts", "expert_offsets", "permutation", "capacity_permutation", "swiglu_rows",
    "layer_forward", "layer_backward", "router_backward", "as_f64",
    "balance_loss", "balance_loss_grad", "balance_loss_groups", "balance_loss_groups_grad",
    "coefficient_of_variation",
]


def as_f64(t):
    """Exact upcast of a torch tensor / numpy array (fp32 or bf16) to fp64 numpy."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        import torch  # local import: the oracle itself only needs numpy
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def silu(a):
    return a / (1.0 + np.exp(-a))


def silu_grad(a):
    s = 1.0 / (1.0 + np.exp(-a))
    return s * (1.0 + a * (1.0 - s))


def router_logits(x, w_r):
    """Router scores ``L = x W_r`` ([T, d] x [d, E]) in fp64."""
    return np.asarray(x, np.float64) @ np.asarray(w_r, np.float64)


def selection_scores(logits, bias=None):
    """Scores the top-k compares.

    fp32 logits (the device's own) keep fp32 and the bias is added with one
    fp32 rounding; fp64 logits stay fp64.
    """
    logits = np.asarray(logits)
    if logits.dtype == np.float32:
        if bias is None:
            return logits.copy()
        return (logits + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
    s = np.asarray(logits, np.float64)
    if bias is not None:
        s = s + np.asarray(bias, np.float64)[None, :]
    return s


def route_topk(scores, k):
    """Top-k selection and renormalised softmax gates.

    Returns ``idx [T, k]`` (int64; descending score, lower index first on equal
    scores) and ``w [T, k]`` (fp64, sums to 1 per row).
    """
    scores = np.asarray(scores)
    assert np.all(np.isfinite(scores)), "router scores must be finite"
    T, E = scores.shape
    assert 1 <= k <= E
    # A stable sort of the negated scores keeps equal scores in ascending
    # expert order; negation is exact in any binary float format.
    order = np.argsort(-scores, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int64)
    s = np.take_along_axis(scores, idx, axis=1).astype(np.float64)
    m = s[:, :1]  # the top-1 score is the row maximum
    ex = np.exp(s - m)
    w = ex / ex.sum(axis=1, keepdims=True)
    return idx, w


def expert_counts(idx, E):
    return np.bincount(np.asarray(idx).reshape(-1), minlength=E).astype(np.int64)


def expert_offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


def permutation(idx, E):
    """Stable counting sort of the copies ``q = t*k + j`` by expert.

    Returns ``dest [T*k]`` (position of copy q in the expert-contiguous order)
    and ``row_src [T*k]`` (token whose row sits at each position).
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    flat = idx.reshape(-1)
    offsets = expert_offsets(expert_counts(idx, E))
    fill = offsets[:-1].copy()
    dest = np.empty(T * k, np.int64)
    for q in range(T * k):          # ascending q: stable by construction
        e = flat[q]
        dest[q] = fill[e]
        fill[e] += 1
    row_src = np.empty(T * k, np.int64)
    row_src[dest] = np.arange(T * k) // k
    return dest, row_src


def capacity_permutation(idx, E, C):
    """Drop-and-pad rearrangement with C rows per expert.

    The pages compare dropless training with the drop-and-pad scheme, which gives
    every expert a fixed number of rows (the Pangu Ultra MoE tech-report article,
    rjtj.cn, the dropless vs drop-and-pad comparison; the CANN MoE page, gtnt.cn,
    section 4.3).  Reading taken: the copies of expert e keep the stable order of
    :func:`permutation`; the first C of them are kept and land in rows
    ``e*C .. e*C + C - 1``; later copies are dropped (``dest = -1``); rows left over
    are padding (``row_src = -1``) and hold zeros.

    Returns ``dest [T*k]`` and ``row_src [E*C]``.
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    flat = idx.reshape(-1)
    seen = np.zeros(E, np.int64)
    dest = np.full(T * k, -1, np.int64)
    row_src = np.full(E * C, -1, np.int64)
    for q in range(T * k):          # ascending q, as in the dropless order
        e = flat[q]
        r = seen[e]
        seen[e] += 1
        if r < C:
            dest[q] = e * C + r
            row_src[e * C + r] = q // k
    return dest, row_src


def swiglu_rows(X, w13, w2):
    """One expert on a block of rows: returns ``Z = [a | b]``, ``h``, ``Y``.

    ``w13`` is ``[2f, d]`` (gate rows first, then up rows), ``w2`` is ``[d, f]``.
    """
    X = np.asarray(X, np.float64)
    w13 = np.asarray(w13, np.float64)
    w2 = np.asarray(w2, np.float64)
    f = w13.shape[0] // 2
    Z = X @ w13.T
    a, b = Z[:, :f], Z[:, f:]
    h = silu(a) * b
    Y = h @ w2.T
    return Z, h, Y


def layer_forward(x, idx, w, w13, w2, ws13=None, ws2=None, capacity=0):
    """Dropless MoE forward on fp64 inputs.

    ``x [T, d]``, ``idx/w [T, k]`` from :func:`route_topk`, ``w13 [E, 2f, d]``,
    ``w2 [E, d, f]``, shared ``ws13 [S, 2f_s, d]``, ``ws2 [S, d, f_s]``.
    Returns a dict with ``y`` and every saved intermediate in the permuted
    order (``x_perm``, ``z``, ``h``, ``y_perm``), the shared parts
    (``z_sh[s]``, ``h_sh[s]``, ``y_sh``) and the routing bookkeeping.

    ``capacity = C > 0`` runs the drop-and-pad variant instead
    (:func:`capacity_permutation`): the permuted buffers have ``E*C`` rows, padding
    rows are zero, and a dropped copy adds nothing to its token's output (the gates
    of the kept copies are not renormalised).
    """
    x = np.asarray(x, np.float64)
    T, d = x.shape
    E = w13.shape[0]
    k = idx.shape[1]
    counts = expert_counts(idx, E)
    if capacity > 0:
        offsets = np.arange(E + 1, dtype=np.int64) * capacity
        dest, row_src = capacity_permutation(idx, E, capacity)
    else:
        offsets = expert_offsets(counts)
        dest, row_src = permutation(idx, E)
    R = len(row_src)
    x_perm = np.zeros((R, d))
    x_perm[row_src >= 0] = x[row_src[row_src >= 0]]
    f = w13.shape[1] // 2
    z = np.zeros((R, 2 * f))
    h = np.zeros((R, f))
    y_perm = np.zeros((R, d))
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            z[lo:hi], h[lo:hi], y_perm[lo:hi] = swiglu_rows(x_perm[lo:hi], w13[e], w2[e])
    w_perm = np.zeros(R)
    kept = dest >= 0
    w_perm[dest[kept]] = np.asarray(w, np.float64).reshape(-1)[kept]
    y_sh = np.zeros((T, d))
    z_sh, h_sh = [], []
    S = 0 if ws13 is None else ws13.shape[0]
    for s in range(S):
        zs, hs, ys = swiglu_rows(x, ws13[s], ws2[s])
        z_sh.append(zs)
        h_sh.append(hs)
        y_sh += ys
    y = np.zeros((T, d))
    dmat = dest.reshape(T, k)
    for j in range(k):
        on = dmat[:, j] >= 0                  # every copy in the dropless layer
        y[on] += np.asarray(w, np.float64)[on, j:j + 1] * y_perm[dmat[on, j]]
    y += y_sh
    return dict(y=y, counts=counts, offsets=offsets, dest=dest, row_src=row_src,
                x_perm=x_perm, z=z, h=h, y_perm=y_perm, w_perm=w_perm,
                z_sh=z_sh, h_sh=h_sh, y_sh=y_sh)


def router_backward(w, dgate):
    """Gradient of the loss w.r.t. the selected scores.

    With ``w_j = exp(s_j) / sum_i exp(s_i)`` over the top-k,
    ``dL_j = w_j * (dgate_j - sum_i w_i dgate_i)``; scores outside the top-k get 0.
    """
    w = np.asarray(w, np.float64)
    dgate = np.asarray(dgate, np.float64)
    return w * (dgate - np.sum(w * dgate, axis=1, keepdims=True))


def layer_backward(x, idx, w, fwd, dy, w13, w2, ws13=None, ws2=None, w_r=None):
    """Backward of :func:`layer_forward` given ``dy = dLoss/dy``.

    Returns ``dx``, ``dw13``, ``dw2``, ``dws13``, ``dws2``, ``dgate [T, k]``,
    ``dscores [T, E]`` (the gradient w.r.t. the router scores, i.e. the logits
    when they are the input) and ``dw_r`` (when ``w_r`` is given; its term is
    then also part of ``dx``).  The expert dX chain and the expert dW products
    are separate computations, as on the pages.
    """
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    T, d = x.shape
    E = w13.shape[0]
    k = idx.shape[1]
    f = w13.shape[1] // 2
    offsets, dest, row_src = fwd["offsets"], fwd["dest"], fwd["row_src"]
    w_perm = fwd["w_perm"]
    R = len(row_src)
    dy_perm = np.zeros((R, d))
    dy_perm[row_src >= 0] = dy[row_src[row_src >= 0]]
    dgate_perm = np.zeros(R)
    dz = np.zeros((R, 2 * f))
    dx_perm = np.zeros((R, d))
    dw13 = np.zeros(w13.shape)
    dw2 = np.zeros(w2.shape)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue          # an expert without tokens keeps zero gradients
        W13 = np.asarray(w13[e], np.float64)
        W2 = np.asarray(w2[e], np.float64)
        a, b = fwd["z"][lo:hi, :f], fwd["z"][lo:hi, f:]
        h = fwd["h"][lo:hi]
        D = dy_perm[lo:hi] @ W2                     # dLoss/d(h) before gating
        dgate_perm[lo:hi] = np.sum(D * h, axis=1)
        wr = w_perm[lo:hi, None]
        dz_e = np.concatenate([wr * D * b * silu_grad(a), wr * D * silu(a)], axis=1)
        dz[lo:hi] = dz_e
        # dX chain
        dx_perm[lo:hi] = dz_e @ W13
        # dW products
        dw2[e] = dy_perm[lo:hi].T @ (wr * h)
        dw13[e] = dz_e.T @ fwd["x_perm"][lo:hi]
    dx = np.zeros((T, d))
    dmat = dest.reshape(T, k)
    for j in range(k):
        on = dmat[:, j] >= 0                  # a dropped copy passes no gradient back
        dx[on] += dx_perm[dmat[on, j]]
    S = 0 if ws13 is None else ws13.shape[0]
    dws13 = np.zeros(ws13.shape) if S else None
    dws2 = np.zeros(ws2.shape) if S else None
    for s in range(S):
        fs = ws13.shape[1] // 2
        W13 = np.asarray(ws13[s], np.float64)
        W2 = np.asarray(ws2[s], np.float64)
        zs, hs = fwd["z_sh"][s], fwd["h_sh"][s]
        a, b = zs[:, :fs], zs[:, fs:]
        D = dy @ W2
        dzs = np.concatenate([D * b * silu_grad(a), D * silu(a)], axis=1)
        dx += dzs @ W13
        dws2[s] = dy.T @ hs
        dws13[s] = dzs.T @ x
    dgate = np.where(dest >= 0, dgate_perm[np.maximum(dest, 0)], 0.0).reshape(T, k)
    dsel = router_backward(w, dgate)
    dscores = np.zeros((T, E))
    np.put_along_axis(dscores, np.asarray(idx), dsel, axis=1)
    dw_r = None
    if w_r is not None:
        w_r = np.asarray(w_r, np.float64)
        dx += dscores @ w_r.T
        dw_r = x.T @ dscores
    return dict(dx=dx, dw13=dw13, dw2=dw2, dws13=dws13, dws2=dws2, dgate=dgate,
                dscores=dscores, dw_r=dw_r, dz=dz, dx_perm=dx_perm,
                dgate_perm=dgate_perm, dy_perm=dy_perm)


# ----------------------------------------------------------------------------- load balance
# The Pangu Ultra MoE tech-report article (rjtj.cn, load-balancing section) lists auxiliary
# balance losses at sequence, global-batch (DP group) and EP-group level without formulas; the
# CANN MoE page (gtnt.cn, section 4.3) adds a load term to the loss. Reading taken: the usual
# form L_aux = alpha * E * sum_e f_e * P_e over one micro-batch (a sequence of T tokens), with
# f_e = counts_e / (T k) the share of token copies routed to expert e and P_e the mean over
# tokens of the full softmax of the scores; the counts are constants of the gradient.

def _softmax_rows(scores):
    s = np.asarray(scores, np.float64)
    m = s.max(axis=1, keepdims=True)
    ex = np.exp(s - m)
    return ex / ex.sum(axis=1, keepdims=True)


def balance_loss(scores, counts, k, alpha):
    """Returns (P [E] mean softmax probability per expert, L_aux)."""
    p = _softmax_rows(scores)
    T, E = p.shape
    P = p.mean(axis=0)
    f = np.asarray(counts, np.float64) / (T * k)
    return P, alpha * E * float(np.sum(f * P))


def balance_loss_grad(scores, counts, k, alpha):
    """d L_aux / d scores [T, E] with the counts held constant."""
    p = _softmax_rows(scores)
    T, E = p.shape
    f = np.asarray(counts, np.float64) / (T * k)
    inner = (p * f[None, :]).sum(axis=1, keepdims=True)
    return alpha * E / T * p * (f[None, :] - inner)


def balance_loss_groups(scores, idx, k, alpha, group_len, n_groups=None, counts=None):
    """Sequence-level form: the tokens fall into groups of ``group_len`` consecutive tokens
    (one sequence each) and each group has its own balance term; the loss is their mean,
    ``L = alpha * E / n_groups * sum_g sum_e f_ge * P_ge`` with ``f_ge = counts_ge /
    (group_len * k)`` and ``P_ge`` the group's mean softmax probability. ``group_len = T``
    is the micro-batch form of :func:`balance_loss`. ``counts [G, E]`` may be given (e.g.
    summed over the ranks of a data-parallel group); by default they are the groups' own
    top-k counts. Returns (P [G, E], counts [G, E], L)."""
    p = _softmax_rows(scores)
    T, E = p.shape
    assert T % group_len == 0
    G = T // group_len
    n_groups = G if n_groups is None else n_groups
    P = p.reshape(G, group_len, E).mean(axis=1)
    if counts is None:
        counts = np.stack([expert_counts(np.asarray(idx)[g * group_len:(g + 1) * group_len], E)
                           for g in range(G)])
    f = np.asarray(counts, np.float64) / (group_len * k)
    return P, counts, alpha * E / n_groups * float(np.sum(f * P))


def balance_loss_groups_grad(scores, counts, k, alpha, group_len, n_groups=None):
    """d L / d scores [T, E] of :func:`balance_loss_groups`, counts held constant."""
    p = _softmax_rows(scores)
    T, E = p.shape
    G = -(-T // group_len)
    n_groups = G if n_groups is None else n_groups
    f = np.asarray(counts, np.float64).reshape(-1, E) / (group_len * k)
    fg = f[np.arange(T) // group_len]                     # each token's group
    inner = (p * fg).sum(axis=1, keepdims=True)
    return alpha * E / (n_groups * group_len) * p * (fg - inner)


def coefficient_of_variation(counts):
    """std / mean of the per-expert loads (the CANN page's cv(experts_load))."""
    c = np.asarray(counts, np.float64)
    return float(c.std() / c.mean())
