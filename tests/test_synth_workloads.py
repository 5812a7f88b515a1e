"""The seeded workload recipes produce what they promise (CPU only)."""
import math

import numpy as np
import torch

import oracle as O
from synth import make_workload, shrink


def test_seeded_and_deterministic():
    a = make_workload(shrink("tiny_fp32", T=16, d=32, f=16))
    b = make_workload(shrink("tiny_fp32", T=16, d=32, f=16))
    assert torch.equal(a.x, b.x) and torch.equal(a.w13, b.w13) and torch.equal(a.dy, b.dy)
    assert a.x.dtype == torch.float32 and a.w_r.dtype == torch.float32


def test_bf16_shapes_and_zipf_bias():
    w = make_workload(shrink("pangu_bf16", T=64, d=64, E=16, f=64))
    assert w.x.dtype == torch.bfloat16 and w.w13.shape == (16, 128, 64)
    assert w.w2.shape == (16, 64, 64) and w.ws13.shape == (1, 2 * 2048, 64)
    assert w.w_r.dtype == torch.float32
    # exp(b) is a rank-Zipf law: sorted exp(b) = r^-s for r = 1..E
    eb = np.sort(np.exp(w.bias.double().numpy()))[::-1]
    np.testing.assert_allclose(eb, np.arange(1, 17) ** -0.8, rtol=1e-6)


def test_adversarial_construction():
    cfg = shrink("adversarial_bf16", T=1024, d=64, E=32, f=64, f_s=64)
    w = make_workload(cfg)
    T, E, k = 1024, 32, 8
    L = w.logits_in.numpy()
    idx, _ = O.route_topk(O.selection_scores(L), k)
    counts = O.expert_counts(idx, E)
    assert all(counts[e] == 0 for e in w.info["dead"]) and len(w.info["dead"]) == E // 4
    assert counts[w.info["hot"]] == math.ceil(0.10 * T * k)
    for t in w.info["boundary_tie_rows"]:
        srt = np.sort(L[t])[::-1]
        assert srt[k - 1] == srt[k]           # exact tie straddling the top-k
    for t in w.info["inner_tie_rows"]:
        srt = np.sort(L[t])[::-1]
        assert srt[1] == srt[2]
    assert len(w.info["boundary_tie_rows"]) == math.ceil(0.01 * T)


def test_replicas_share_weights_and_draw_their_own_tokens():
    """Replica 0 is the plain draw; replica r > 0 keeps every weight and draws its own x, dY
    (and adversarial logits) from its own seed."""
    import torch
    cfg = shrink("pangu_bf16", T=32, d=64, E=16, k=4, f=64, f_s=64)
    a, a0, b = make_workload(cfg), make_workload(cfg, replica=0), make_workload(cfg, replica=1)
    for n in ("x", "dy", "w13", "w2", "ws13", "ws2", "w_r", "bias"):
        assert torch.equal(getattr(a, n), getattr(a0, n)), n
    for n in ("w13", "w2", "ws13", "ws2", "w_r", "bias"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n
    assert not torch.equal(a.x, b.x) and not torch.equal(a.dy, b.dy)
    adv = shrink("adversarial_bf16", T=64, d=64, E=32, k=8, f=64, f_s=64)
    c, d = make_workload(adv), make_workload(adv, replica=2)
    assert torch.equal(c.w13, d.w13) and not torch.equal(c.logits_in, d.logits_in)
    assert d.info["n_hot_rows"] == c.info["n_hot_rows"]
