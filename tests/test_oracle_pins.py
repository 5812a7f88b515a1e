"""Pins of the fp64 oracle against things other than itself (CPU only).

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, an unstable sort, a wrong tie rule)
fails at least one of them:

* a closed-form hand-derived case (tests/golden/closed_form_tiny.json);
* brute force on tiny inputs in pure Python: every expert on every token,
  masked by a top-k found by sorting (-score, index) keys;
* E = 1, k = 1 reduces to a dense SwiGLU FFN (torch fp64 library ops);
* k = E reduces to a dense softmax mixture (scipy softmax);
* the permutation is a bijection, counts sum to T*k, offsets are the exclusive
  scan and each segment holds exactly its expert's copies in ascending token;
* renormalised gates sum to 1;
* central finite differences of the forward, for every input entry;
* torch autograd (fp64) of a dense masked formulation;
* dgate = <dY_t, Y_q> and the invariances under token permutation and
  expert relabelling;
* the SwiGLU derivative against central differences and the identity
  silu(a) - silu(-a) = a; the drop-and-pad rows against the dropless
  permutation cut at the capacity.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_layer(rng, T, d, E, k, f, S=0, f_s=0, scale=1.0):
    x = rng.standard_normal((T, d))
    w_r = rng.standard_normal((d, E)) * scale
    w13 = rng.standard_normal((E, 2 * f, d)) * 0.5
    w2 = rng.standard_normal((E, d, f)) * 0.5
    ws13 = rng.standard_normal((S, 2 * f_s, d)) * 0.5 if S else None
    ws2 = rng.standard_normal((S, d, f_s)) * 0.5 if S else None
    dy = rng.standard_normal((T, d))
    return x, w_r, w13, w2, ws13, ws2, dy


def _oracle_layer(x, w_r, w13, w2, ws13, ws2, k, logits=None, bias=None):
    L = O.router_logits(x, w_r) if logits is None else logits
    idx, w = O.route_topk(O.selection_scores(L, bias), k)
    fwd = O.layer_forward(x, idx, w, w13, w2, ws13, ws2)
    return idx, w, fwd


# ---------------------------------------------------------------- closed form
def _ev(s):
    return float(eval(str(s), {"ln3": math.log(3.0)}))


def test_closed_form_golden():
    g = json.load(open(os.path.join(GOLDEN, "closed_form_tiny.json")))
    x = np.array(g["x"], float)
    L = np.array([[_ev(v) for v in row] for row in g["logits"]])
    w13 = np.array([[[_ev(v) for v in r] for r in m] for m in g["w13"]])
    w2 = np.array([[[_ev(v) for v in r] for r in m] for m in g["w2"]])
    dy = np.array(g["dy"], float)
    idx, w = O.route_topk(O.selection_scores(L), g["k"])
    ex = g["expected"]
    assert idx.tolist() == ex["topk_idx"]
    np.testing.assert_allclose(w, [[_ev(v) for v in ex["topk_w"][0]]], rtol=0, atol=1e-15)
    fwd = O.layer_forward(x, idx, w, w13, w2)
    np.testing.assert_allclose(fwd["y_perm"][fwd["dest"][0], 0], _ev(ex["y_perm_expert0"]), atol=1e-14)
    np.testing.assert_allclose(fwd["y_perm"][fwd["dest"][1], 0], _ev(ex["y_perm_expert1"]), atol=1e-14)
    np.testing.assert_allclose(fwd["y"], [[_ev(v) for v in ex["y"][0]]], atol=1e-14)
    bwd = O.layer_backward(x, idx, w, fwd, dy, w13, w2)
    np.testing.assert_allclose(bwd["dgate"], [[_ev(v) for v in ex["dgate"][0]]], atol=1e-14)
    np.testing.assert_allclose(bwd["dscores"], [[_ev(v) for v in ex["dlogits"][0]]], atol=1e-14)


# ---------------------------------------------------------------- routing pins
def test_topk_tie_rule_and_order():
    s = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]])
    idx, w = O.route_topk(s, 2)
    assert idx.tolist() == [[1, 2]]
    np.testing.assert_allclose(w, [[0.5, 0.5]], atol=1e-16)
    idx, _ = O.route_topk(s, 4)
    assert idx.tolist() == [[1, 2, 4, 3]]
    # -0.0 and +0.0 compare equal: the lower index wins.
    s = np.array([[-0.0, 0.0, -1.0]], np.float32)
    assert O.route_topk(s, 1)[0].tolist() == [[0]]
    s = np.array([[0.0, -0.0, -1.0]], np.float32)
    assert O.route_topk(s, 1)[0].tolist() == [[0]]


def test_topk_matches_brute_force_sort_and_scipy_softmax():
    rng = np.random.default_rng(1)
    T, E, k = 64, 12, 4
    s = np.round(rng.standard_normal((T, E)) * 2) / 2   # many exact ties
    idx, w = O.route_topk(s, k)
    for t in range(T):
        ref = sorted(range(E), key=lambda e: (-s[t, e], e))[:k]
        assert idx[t].tolist() == ref
        p = scipy.special.softmax(s[t])
        sel = p[ref] / p[ref].sum()
        np.testing.assert_allclose(w[t], sel, rtol=1e-13)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-15)


def test_fp32_selection_scores_round_once():
    L = np.array([[1.0, 1.0 + 2 ** -23]], np.float32)
    b = np.array([2 ** -24, 0.0], np.float32)
    s = O.selection_scores(L, b)
    assert s.dtype == np.float32
    # 1 + 2^-24 rounds (ties-to-even) back to 1, so expert 1 stays ahead.
    assert O.route_topk(s, 1)[0].tolist() == [[1]]


@pytest.mark.parametrize("skew", [False, True])
def test_permutation_is_stable_bijection(skew):
    rng = np.random.default_rng(2)
    T, E, k = 97, 9, 3
    s = rng.standard_normal((T, E))
    if skew:
        s[:, 4] += 5.0          # one expert in every row
        s[:, 7] -= 50.0         # an expert with no tokens
    idx, _ = O.route_topk(s, k)
    counts = O.expert_counts(idx, E)
    offsets = O.expert_offsets(counts)
    dest, row_src = O.permutation(idx, E)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert np.all(np.diff(offsets) == counts)
    assert sorted(dest.tolist()) == list(range(T * k))
    assert np.all(row_src[dest] == np.arange(T * k) // k)
    for e in range(E):
        seg = row_src[offsets[e]:offsets[e + 1]]
        toks = [t for t in range(T) if e in idx[t]]
        assert seg.tolist() == toks          # exactly its copies, ascending token
    if skew:
        assert counts[4] == T and counts[7] == 0


# ---------------------------------------------------------------- forward pins
def _py_silu(a):
    return a / (1.0 + math.exp(-a))


def test_brute_force_dense_masked_forward():
    rng = np.random.default_rng(3)
    T, d, E, k, f, S, f_s = 10, 5, 6, 2, 3, 1, 2
    x, w_r, w13, w2, ws13, ws2, _ = _rand_layer(rng, T, d, E, k, f, S, f_s)
    _, _, fwd = _oracle_layer(x, w_r, w13, w2, ws13, ws2, k)

    def ffn(W13, W2, xt):          # pure-Python SwiGLU of one row
        ff = len(W13) // 2
        a = [sum(W13[i][c] * xt[c] for c in range(d)) for i in range(ff)]
        b = [sum(W13[ff + i][c] * xt[c] for c in range(d)) for i in range(ff)]
        hh = [_py_silu(a[i]) * b[i] for i in range(ff)]
        return [sum(W2[r][i] * hh[i] for i in range(ff)) for r in range(d)]

    for t in range(T):
        L = [sum(x[t, c] * w_r[c, e] for c in range(d)) for e in range(E)]
        sel = sorted(range(E), key=lambda e: (-L[e], e))[:k]
        m = max(L)
        den = sum(math.exp(L[e] - m) for e in sel)
        y = [0.0] * d
        for e in range(E):                      # every expert, masked
            out = ffn(w13[e].tolist(), w2[e].tolist(), x[t].tolist())
            g = math.exp(L[e] - m) / den if e in sel else 0.0
            y = [y[r] + g * out[r] for r in range(d)]
        for s in range(S):
            out = ffn(ws13[s].tolist(), ws2[s].tolist(), x[t].tolist())
            y = [y[r] + out[r] for r in range(d)]
        np.testing.assert_allclose(fwd["y"][t], y, rtol=1e-12, atol=1e-12)


def test_single_expert_top1_is_dense_swiglu():
    rng = np.random.default_rng(4)
    T, d, f = 33, 16, 8
    x, w_r, w13, w2, _, _, _ = _rand_layer(rng, T, d, 1, 1, f)
    idx, w, fwd = _oracle_layer(x, w_r, w13, w2, None, None, 1)
    assert np.all(idx == 0) and np.all(w == 1.0)
    assert fwd["counts"].tolist() == [T]
    assert fwd["dest"].tolist() == list(range(T))
    xt = torch.tensor(x)
    ref = (torch.nn.functional.silu(xt @ torch.tensor(w13[0, :f]).T)
           * (xt @ torch.tensor(w13[0, f:]).T)) @ torch.tensor(w2[0]).T
    np.testing.assert_allclose(fwd["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_topk_equal_E_is_softmax_mixture():
    rng = np.random.default_rng(5)
    T, d, E, f = 20, 7, 5, 4
    x, w_r, w13, w2, _, _, _ = _rand_layer(rng, T, d, E, E, f)
    _, _, fwd = _oracle_layer(x, w_r, w13, w2, None, None, E)
    p = scipy.special.softmax(x @ w_r, axis=1)
    xt = torch.tensor(x)
    ref = torch.zeros(T, d, dtype=torch.float64)
    for e in range(E):
        W13 = torch.tensor(w13[e])
        he = torch.nn.functional.silu(xt @ W13[:f].T) * (xt @ W13[f:].T)
        ref += torch.tensor(p[:, e:e + 1]) * (he @ torch.tensor(w2[e]).T)
    np.testing.assert_allclose(fwd["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- backward pins
def _loss(x, w_r, w13, w2, ws13, ws2, k, dy, logits=None, expect_idx=None):
    idx, _, fwd = _oracle_layer(x, w_r, w13, w2, ws13, ws2, k, logits=logits)
    if expect_idx is not None:
        assert np.array_equal(idx, expect_idx), "perturbation changed the top-k"
    return float(np.sum(fwd["y"] * dy))


def _fd(fn, arr, h=1e-6):
    g = np.zeros_like(arr)
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = arr[i]
        arr[i] = old + h
        lp = fn()
        arr[i] = old - h
        lm = fn()
        arr[i] = old
        g[i] = (lp - lm) / (2 * h)
    return g


def _margin_ok(s, k, margin):
    srt = -np.sort(-s, axis=1)
    return np.all(srt[:, k - 1] - srt[:, k] > margin)


@pytest.mark.parametrize("mode", ["router", "logits"])
def test_backward_central_differences(mode):
    rng = np.random.default_rng(6)
    T, d, E, k, f, S, f_s = 8, 6, 5, 2, 3, 1, 2
    for attempt in range(50):
        x, w_r, w13, w2, ws13, ws2, dy = _rand_layer(rng, T, d, E, k, f, S, f_s)
        logits = rng.standard_normal((T, E)) * 2 if mode == "logits" else None
        s = O.router_logits(x, w_r) if logits is None else logits
        if _margin_ok(s, k, 1e-3):
            break
    idx, w, fwd = _oracle_layer(x, w_r, w13, w2, ws13, ws2, k, logits=logits)
    bwd = O.layer_backward(x, idx, w, fwd, dy, w13, w2, ws13, ws2,
                           w_r=w_r if mode == "router" else None)

    def fn():
        return _loss(x, w_r, w13, w2, ws13, ws2, k, dy, logits=logits, expect_idx=idx)

    checks = [("dx", x), ("dw13", w13), ("dw2", w2), ("dws13", ws13), ("dws2", ws2)]
    if mode == "router":
        checks.append(("dw_r", w_r))
    else:
        checks.append(("dscores", logits))
    for name, arr in checks:
        num = _fd(fn, arr)
        ana = bwd[name]
        rel = np.linalg.norm(num - ana) / np.linalg.norm(ana)
        assert rel < 1e-6, (name, rel)


def test_backward_matches_torch_autograd_dense_formulation():
    rng = np.random.default_rng(7)
    T, d, E, k, f, S, f_s = 24, 10, 7, 3, 5, 2, 4
    x, w_r, w13, w2, ws13, ws2, dy = _rand_layer(rng, T, d, E, k, f, S, f_s)
    idx, w, fwd = _oracle_layer(x, w_r, w13, w2, ws13, ws2, k)
    bwd = O.layer_backward(x, idx, w, fwd, dy, w13, w2, ws13, ws2, w_r=w_r)
    tt = {n: torch.tensor(v, requires_grad=True)
          for n, v in dict(x=x, w_r=w_r, w13=w13, w2=w2, ws13=ws13, ws2=ws2).items()}
    L = tt["x"] @ tt["w_r"]
    mask = torch.zeros(T, E, dtype=torch.bool)
    mask[torch.arange(T)[:, None], torch.tensor(idx)] = True
    Lm = L.masked_fill(~mask, float("-inf"))
    gates = torch.softmax(Lm, dim=1)           # softmax restricted to the top-k
    y = torch.zeros(T, d, dtype=torch.float64)
    for e in range(E):
        he = (torch.nn.functional.silu(tt["x"] @ tt["w13"][e, :f].T)
              * (tt["x"] @ tt["w13"][e, f:].T))
        y = y + gates[:, e:e + 1] * (he @ tt["w2"][e].T)
    for s in range(S):
        hs = (torch.nn.functional.silu(tt["x"] @ tt["ws13"][s, :f_s].T)
              * (tt["x"] @ tt["ws13"][s, f_s:].T))
        y = y + hs @ tt["ws2"][s].T
    np.testing.assert_allclose(y.detach().numpy(), fwd["y"], rtol=1e-12, atol=1e-12)
    (y * torch.tensor(dy)).sum().backward()
    for name, key in [("x", "dx"), ("w_r", "dw_r"), ("w13", "dw13"), ("w2", "dw2"),
                      ("ws13", "dws13"), ("ws2", "dws2")]:
        np.testing.assert_allclose(bwd[key], tt[name].grad.numpy(), rtol=1e-10, atol=1e-11)


def test_dgate_is_inner_product_with_expert_output():
    rng = np.random.default_rng(8)
    T, d, E, k, f = 30, 8, 6, 3, 4
    x, w_r, w13, w2, _, _, dy = _rand_layer(rng, T, d, E, k, f)
    idx, w, fwd = _oracle_layer(x, w_r, w13, w2, None, None, k)
    bwd = O.layer_backward(x, idx, w, fwd, dy, w13, w2)
    for t in range(T):
        for j in range(k):
            Yq = fwd["y_perm"][fwd["dest"][t * k + j]]
            np.testing.assert_allclose(bwd["dgate"][t, j], dy[t] @ Yq, rtol=1e-12, atol=1e-12)
    # the router gradient of a renormalised softmax sums to zero per row
    np.testing.assert_allclose(bwd["dscores"].sum(1), 0.0, atol=1e-12)


def test_token_permutation_and_expert_relabelling_invariance():
    rng = np.random.default_rng(9)
    T, d, E, k, f, S, f_s = 40, 8, 7, 2, 5, 1, 3
    x, w_r, w13, w2, ws13, ws2, dy = _rand_layer(rng, T, d, E, k, f, S, f_s)
    idx, w, fwd = _oracle_layer(x, w_r, w13, w2, ws13, ws2, k)
    bwd = O.layer_backward(x, idx, w, fwd, dy, w13, w2, ws13, ws2, w_r=w_r)
    p = rng.permutation(T)
    idx2, w2_, fwd2 = _oracle_layer(x[p], w_r, w13, w2, ws13, ws2, k)
    bwd2 = O.layer_backward(x[p], idx2, w2_, fwd2, dy[p], w13, w2, ws13, ws2, w_r=w_r)
    np.testing.assert_allclose(fwd2["y"], fwd["y"][p], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bwd2["dx"], bwd["dx"][p], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(bwd2["dw13"], bwd["dw13"], rtol=1e-11, atol=1e-12)
    r = rng.permutation(E)            # expert e' = r[e]
    inv = np.argsort(r)
    idx3, _, fwd3 = _oracle_layer(x, w_r[:, inv], w13[inv], w2[inv], ws13, ws2, k)
    np.testing.assert_allclose(fwd3["y"], fwd["y"], rtol=1e-12, atol=1e-12)
    assert sorted(fwd3["counts"].tolist()) == sorted(fwd["counts"].tolist())


# ---------------------------------------------------------------- load-balance statistics
def test_balance_loss_closed_forms():
    T, E, k = 64, 8, 2
    s = np.zeros((T, E))                              # uniform router: P_e = 1/E
    counts = np.full(E, T * k // E)                   # perfectly balanced loads: f_e = 1/E
    P, L = O.balance_loss(s, counts, k, alpha=0.01)
    np.testing.assert_allclose(P, 1.0 / E, rtol=1e-15)
    np.testing.assert_allclose(L, 0.01, rtol=1e-14)   # alpha * E * E * (1/E)(1/E) = alpha
    assert O.coefficient_of_variation(counts) == 0.0
    # all copies on one expert with probability one there: L = alpha * E
    s = np.full((T, E), -1e3)
    s[:, 3] = 0.0
    counts = np.zeros(E)
    counts[3] = T * k
    _, L = O.balance_loss(s, counts, k, alpha=0.5)
    np.testing.assert_allclose(L, 0.5 * E, rtol=1e-12)
    np.testing.assert_allclose(O.coefficient_of_variation(counts), np.sqrt(E - 1), rtol=1e-12)


def test_balance_loss_gradient_central_differences():
    rng = np.random.default_rng(12)
    T, E, k = 9, 6, 2
    s = rng.standard_normal((T, E))
    counts = rng.integers(0, 5, E)
    g = O.balance_loss_grad(s, counts, k, alpha=0.3)
    num = np.zeros_like(s)
    h = 1e-6
    for t in range(T):
        for e in range(E):
            sp, sm = s.copy(), s.copy()
            sp[t, e] += h
            sm[t, e] -= h
            num[t, e] = (O.balance_loss(sp, counts, k, 0.3)[1] - O.balance_loss(sm, counts, k, 0.3)[1]) / (2 * h)
    assert np.linalg.norm(num - g) / np.linalg.norm(g) < 1e-7
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-14)   # softmax Jacobian rows sum to 0


def test_balance_groups_reduce_and_average():
    """One group of all T tokens is the micro-batch form; G groups average their own
    micro-batch terms (each evaluated on its slice alone)."""
    rng = np.random.default_rng(13)
    T, E, k, L = 48, 7, 2, 12
    s = rng.standard_normal((T, E)) * 1.5
    idx, _ = O.route_topk(s, k)
    P1, c1, l1 = O.balance_loss_groups(s, idx, k, 0.2, T)
    P0, l0 = O.balance_loss(s, O.expert_counts(idx, E), k, 0.2)
    np.testing.assert_allclose(P1[0], P0, rtol=1e-14)
    np.testing.assert_allclose(l1, l0, rtol=1e-14)
    P, c, lg = O.balance_loss_groups(s, idx, k, 0.2, L)
    per = [O.balance_loss(s[g * L:(g + 1) * L], O.expert_counts(idx[g * L:(g + 1) * L], E), k, 0.2)[1]
           for g in range(T // L)]
    np.testing.assert_allclose(lg, np.mean(per), rtol=1e-14)
    assert c.sum() == T * k and np.all(c.sum(axis=1) == L * k)


def test_balance_groups_gradient_central_differences():
    rng = np.random.default_rng(14)
    T, E, k, L = 12, 5, 2, 4
    s = rng.standard_normal((T, E))
    idx, _ = O.route_topk(s, k)
    _, counts, _ = O.balance_loss_groups(s, idx, k, 0.3, L)
    g = O.balance_loss_groups_grad(s, counts, k, 0.3, L)
    num = np.zeros_like(s)
    h = 1e-6
    for t in range(T):
        for e in range(E):
            sp, sm = s.copy(), s.copy()
            sp[t, e] += h
            sm[t, e] -= h
            num[t, e] = (O.balance_loss_groups(sp, idx, k, 0.3, L, counts=counts)[2] -
                         O.balance_loss_groups(sm, idx, k, 0.3, L, counts=counts)[2]) / (2 * h)
    assert np.linalg.norm(num - g) / np.linalg.norm(g) < 1e-7


# ---------------------------------------------------------------- drop-and-pad pins
def _kept_brute(idx, C):
    """Copy (t, j) is kept iff fewer than C copies of its expert come before it in
    token-major order (pure Python, no sort)."""
    T, k = len(idx), len(idx[0])
    kept = [[False] * k for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = idx[t][j]
            before = sum(1 for tt in range(T) for jj in range(k)
                         if (tt, jj) < (t, j) and idx[tt][jj] == e)
            kept[t][j] = before < C
    return kept


def test_capacity_brute_force_forward():
    rng = np.random.default_rng(31)
    T, d, E, k, f, S, f_s = 12, 5, 4, 2, 3, 1, 2
    x, w_r, w13, w2, ws13, ws2, _ = _rand_layer(rng, T, d, E, k, f, S, f_s)
    # a skewed router so that some experts overflow a capacity of 3
    w_r[:, 0] += 2.0 * np.sign(x.mean(0))
    idx, w = O.route_topk(O.selection_scores(O.router_logits(x, w_r)), k)
    C = 3
    assert O.expert_counts(idx, E).max() > C
    fwd = O.layer_forward(x, idx, w, w13, w2, ws13, ws2, capacity=C)
    kept = _kept_brute(idx.tolist(), C)

    def ffn(W13, W2, xt):
        ff = len(W13) // 2
        a = [sum(W13[i][c] * xt[c] for c in range(d)) for i in range(ff)]
        b = [sum(W13[ff + i][c] * xt[c] for c in range(d)) for i in range(ff)]
        hh = [_py_silu(a[i]) * b[i] for i in range(ff)]
        return [sum(W2[r][i] * hh[i] for i in range(ff)) for r in range(d)]

    for t in range(T):
        y = [0.0] * d
        for j in range(k):
            if kept[t][j]:
                e = int(idx[t, j])
                out = ffn(w13[e].tolist(), w2[e].tolist(), x[t].tolist())
                y = [y[r] + w[t, j] * out[r] for r in range(d)]
        for s in range(S):
            out = ffn(ws13[s].tolist(), ws2[s].tolist(), x[t].tolist())
            y = [y[r] + out[r] for r in range(d)]
        np.testing.assert_allclose(fwd["y"][t], y, rtol=1e-12, atol=1e-12)
    # layout: kept copies in rows e*C + rank, padding rows zero and marked -1
    dest, row_src = fwd["dest"], fwd["row_src"]
    assert sum(map(sum, kept)) == int(np.sum(dest >= 0))
    for q in range(T * k):
        t, j = divmod(q, k)
        assert (dest[q] >= 0) == kept[t][j]
        if dest[q] >= 0:
            assert dest[q] // C == idx[t, j] and row_src[dest[q]] == t
    pad = row_src < 0
    assert np.all(fwd["x_perm"][pad] == 0) and np.all(fwd["w_perm"][pad] == 0)


def test_capacity_at_least_max_count_equals_dropless():
    rng = np.random.default_rng(32)
    T, d, E, k, f = 40, 6, 5, 2, 4
    x, w_r, w13, w2, _, _, dy = _rand_layer(rng, T, d, E, k, f)
    idx, w = O.route_topk(O.selection_scores(O.router_logits(x, w_r)), k)
    C = int(O.expert_counts(idx, E).max())
    ref = O.layer_forward(x, idx, w, w13, w2)
    cap = O.layer_forward(x, idx, w, w13, w2, capacity=C)
    np.testing.assert_allclose(cap["y"], ref["y"], rtol=1e-12, atol=1e-12)
    assert np.all(cap["dest"] >= 0)
    # the segment of expert e holds the same rows, shifted from offsets[e] to e*C
    for e in range(E):
        lo, hi = ref["offsets"][e], ref["offsets"][e + 1]
        assert np.array_equal(cap["row_src"][e * C:e * C + hi - lo], ref["row_src"][lo:hi])
    rb = O.layer_backward(x, idx, w, ref, dy, w13, w2)
    cb = O.layer_backward(x, idx, w, cap, dy, w13, w2)
    for name in ("dx", "dw13", "dw2", "dgate", "dscores"):
        np.testing.assert_allclose(cb[name], rb[name], rtol=1e-11, atol=1e-12)


def test_capacity_backward_central_differences():
    rng = np.random.default_rng(33)
    T, d, E, k, f, S, f_s = 9, 5, 4, 2, 3, 1, 2
    C = 3
    for attempt in range(50):
        x, w_r, w13, w2, ws13, ws2, dy = _rand_layer(rng, T, d, E, k, f, S, f_s)
        logits = rng.standard_normal((T, E)) * 2
        logits[:, 1] += 1.5                  # expert 1 overflows
        idx0, _ = O.route_topk(O.selection_scores(logits), k)
        if _margin_ok(logits, k, 1e-3) and O.expert_counts(idx0, E).max() > C:
            break
    idx, w = O.route_topk(O.selection_scores(logits), k)
    fwd = O.layer_forward(x, idx, w, w13, w2, ws13, ws2, capacity=C)
    assert np.any(fwd["dest"] < 0)
    bwd = O.layer_backward(x, idx, w, fwd, dy, w13, w2, ws13, ws2)

    def fn():
        i2, w2_ = O.route_topk(O.selection_scores(logits), k)
        assert np.array_equal(i2, idx)
        return float(np.sum(O.layer_forward(x, i2, w2_, w13, w2, ws13, ws2, capacity=C)["y"] * dy))

    for name, arr in [("dx", x), ("dw13", w13), ("dw2", w2), ("dws13", ws13), ("dws2", ws2),
                      ("dscores", logits)]:
        num = _fd(fn, arr)
        ana = bwd[name]
        rel = np.linalg.norm(num - ana) / np.linalg.norm(ana)
        assert rel < 1e-6, (name, rel)
    # a dropped copy has no gate gradient
    assert np.all(bwd["dgate"].reshape(-1)[fwd["dest"] < 0] == 0)


# ---------------------------------------------------------------- helpers pinned directly
def test_silu_grad_is_the_derivative_of_silu():
    """silu'(a) against central differences of silu, at 0 (1/2), far out (0 and 1), and the
    identity silu(a) - silu(-a) = a, whose derivative gives silu'(a) + silu'(-a) = 1."""
    a = np.linspace(-12.0, 12.0, 481)
    h = 1e-5
    fd = (O.silu(a + h) - O.silu(a - h)) / (2 * h)
    assert np.max(np.abs(O.silu_grad(a) - fd)) < 1e-9
    assert O.silu_grad(np.array([0.0]))[0] == 0.5
    assert abs(O.silu_grad(np.array([40.0]))[0] - 1.0) < 1e-12
    assert abs(O.silu_grad(np.array([-40.0]))[0]) < 1e-12
    assert np.max(np.abs(O.silu(a) - O.silu(-a) - a)) < 1e-12
    assert np.max(np.abs(O.silu_grad(a) + O.silu_grad(-a) - 1.0)) < 1e-12


@pytest.mark.parametrize("C", [1, 2, 5, 40])
def test_capacity_permutation_is_the_dropless_order_cut_at_capacity(C):
    """The drop-and-pad rows are the dropless permutation's segments cut at C rows: copy q of
    rank r = dest[q] - offsets[e] in its expert's segment lands at row e*C + r when r < C and
    is dropped otherwise; each expert's first min(C, count) rows hold the dropless rows'
    tokens, the rest are padding."""
    rng = np.random.default_rng(7 + C)
    T, E, k = 37, 6, 3
    s = rng.standard_normal((T, E)) + np.array([2.0, 1.0, 0.0, 0.0, -1.0, -3.0])
    idx, _ = O.route_topk(s, k)
    dest, row_src = O.permutation(idx, E)
    counts = O.expert_counts(idx, E)
    off = O.expert_offsets(counts)
    flat = idx.reshape(-1)
    rank = dest - off[flat]
    dc, rc = O.capacity_permutation(idx, E, C)
    assert np.array_equal(dc, np.where(rank < C, flat * C + rank, -1))
    for e in range(E):
        n = min(C, counts[e])
        assert np.array_equal(rc[e * C:e * C + n], row_src[off[e]:off[e] + n])
        assert np.all(rc[e * C + n:(e + 1) * C] == -1)
    # every kept row is filled by exactly one copy
    kept = dc[dc >= 0]
    assert len(np.unique(kept)) == len(kept) == int(np.minimum(counts, C).sum())
