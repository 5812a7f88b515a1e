"""Model check of the top-k selection the routing kernel performs (no GPU).

The kernel ranks a token's scores on order-preserving 32-bit keys: a float's bits with the
sign bit set for x >= 0, all bits inverted for x < 0, taken of x + 0 so that -0 and +0 get
one key (they tie in a float comparison). Each of the k rounds takes the largest key, then
the lowest expert index holding it, and clears that expert's key to 0, below every finite
score. The functions below restate that arithmetic with numpy and check it against the
oracle's stable sort (descending score, lower index first on equal scores), including
exact ties and signed zeros at the top-k boundary.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O


def order_key(x):
    u = (np.asarray(x, np.float32) + np.float32(0.0)).view(np.uint32)
    return np.where(u & np.uint32(0x80000000), ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def key_value(key):
    key = np.asarray(key, np.uint32)
    u = np.where(key & np.uint32(0x80000000), key & np.uint32(0x7FFFFFFF), ~key).astype(np.uint32)
    return u.view(np.float32)


def select_by_keys(scores, k):
    T, E = scores.shape
    keys = order_key(scores)
    idx = np.empty((T, k), np.int64)
    val = np.empty((T, k), np.float32)
    for t in range(T):
        key = keys[t].copy()
        for j in range(k):
            m = key.max()
            i = int(np.flatnonzero(key == m).min())
            idx[t, j], val[t, j] = i, key_value(m)
            key[i] = 0
    return idx, val


def test_keys_preserve_the_float_order():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10,
        np.float32([0.0, -0.0, 1e-45, -1e-45, 1e-38, -1e-38, np.finfo(np.float32).max,
                    -np.finfo(np.float32).max, 1.0, -1.0]),
    ])
    kx = order_key(x).astype(np.int64)
    a, b = np.meshgrid(np.arange(x.size), np.arange(x.size), indexing="ij")
    sel = (a[:, :60].ravel(), b[:, :60].ravel())   # every value against the first 60
    xa, xb = x[sel[0]], x[sel[1]]
    ka, kb = kx[sel[0]], kx[sel[1]]
    assert np.array_equal(xa > xb, ka > kb)
    assert np.array_equal(xa == xb, ka == kb)     # -0 == +0 as floats and as keys
    # every finite score's key is above the cleared key 0
    assert kx.min() > 0
    # the key's value is the score, -0 read back as +0
    back = key_value(order_key(x))
    assert np.array_equal(back.view(np.uint32), (x + np.float32(0)).view(np.uint32))


@pytest.mark.parametrize("seed,T,E,k", [(0, 300, 64, 6), (1, 200, 256, 8), (2, 100, 24, 24),
                                        (3, 150, 1000, 32), (4, 50, 8, 1)])
def test_selection_matches_the_oracle(seed, T, E, k):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((T, E)).astype(np.float32)
    # dense exact ties: a quarter of the rows drawn from four values only
    s[: T // 4] = rng.choice(np.float32([-1.5, 0.25, 0.5, 2.0]), size=(T // 4, E))
    # signed zeros straddling the top-k boundary
    z = np.float32(-1e30) * np.ones((8, E), np.float32)
    z[:, : max(1, k - 1)] = 1.0
    z[:4, k - 1:] = np.where(np.arange(E - k + 1) % 2 == 0, np.float32(-0.0), np.float32(0.0))
    z[4:, k - 1:] = np.where(np.arange(E - k + 1) % 2 == 0, np.float32(0.0), np.float32(-0.0))
    s = np.concatenate([s, z[:, :E]])
    idx, val = select_by_keys(s, k)
    ref, _ = O.route_topk(s, k)
    assert np.array_equal(idx, ref)
    # the selected values are the scores themselves (zeros read back as +0)
    assert np.array_equal(val, np.take_along_axis(s, ref, axis=1) + np.float32(0))


def test_a_signed_zero_key_would_break_ties():
    """With -0 and +0 keyed apart (no `+ 0`), +0 would beat a -0 of lower index: the
    oracle's tie rule takes the lower index, so the canonicalisation is needed."""
    s = np.float32([[-0.0, 0.0, -1.0]])
    u = s.view(np.uint32)
    raw = np.where(u & np.uint32(0x80000000), ~u, u | np.uint32(0x80000000)).astype(np.uint32)
    assert raw[0, 1] > raw[0, 0]                 # the raw keys differ ...
    idx, _ = select_by_keys(s, 1)
    ref, _ = O.route_topk(s, 1)
    assert idx[0, 0] == ref[0, 0] == 0           # ... the canonical keys tie, lower index wins
