"""GPU parity of the whole layer (moe_layer_fwd / moe_layer_bwd through the C ABI) against
the fp64 oracle, on the seeded workloads at sizes the oracle finishes in seconds that
still span several tiles and ragged tails."""
import numpy as np
import pytest
import torch

from synth import make_workload, shrink

pytestmark = pytest.mark.gpu

CASES = {
    # the tiny fp32 layer at its full size (T=256, d=512, E=8, top-2, f=256)
    "tiny_fp32": ("tiny_fp32", {}),
    # Pangu-shaped recipe, shrunk: Zipf(0.8) skew, 1 shared expert, ragged M tiles
    "pangu_small": ("pangu_bf16", dict(T=640, d=512, E=16, k=4, f=256, f_s=256)),
    # mid-size recipe, shrunk: 2 shared experts, f = 1408 (5.5 tiles of 256)
    "mid_small": ("mid_bf16", dict(T=384, d=1024, E=64, k=6, f=1408, f_s=1408)),
    # DeepSeek-shaped recipe, shrunk: E = 24 (not a multiple of 32), d = 448 and f = 320
    # (N tails in every GEMM), f_s = 192
    "dsv3_small": ("dsv3_bf16", dict(T=384, d=448, E=24, k=3, f=320, f_s=192)),
    # adversarial recipe, shrunk: logits are the input (dead experts, 10 % hot expert, ties)
    "adversarial_small": ("adversarial_bf16", dict(T=1024, d=256, E=32, k=8, f=256, f_s=256)),
}


@pytest.mark.parametrize("case", list(CASES))
def test_layer_matches_oracle(case):
    from layer_check import check_layer
    name, over = CASES[case]
    cfg = shrink(name, **over) if over else dict(__import__("synth").CONFIGS[name], name=name)
    w = make_workload(cfg)
    check_layer(w, bwd=True)


def test_layer_is_deterministic():
    from layer_check import run_gpu_layer
    w = make_workload(shrink("adversarial_bf16", T=512, d=256, E=32, k=8, f=256, f_s=256))
    a, ga, _ = run_gpu_layer(w)
    ya, dxa = a.y.clone(), ga["dx"].clone()
    dwa, dla = ga["dw13"].clone(), ga["dlogits"].clone()
    b, gb, _ = run_gpu_layer(w)
    assert torch.equal(ya, b.y) and torch.equal(dxa, gb["dx"])
    assert torch.equal(dwa, gb["dw13"]) and torch.equal(dla, gb["dlogits"])


def test_single_expert_top1_is_dense_ffn():
    """E = 1, k = 1: every copy goes to expert 0 in token order (routing reduces away)."""
    from layer_check import check_layer
    w = make_workload(shrink("pangu_bf16", T=300, d=256, E=1, k=1, f=256, S=0, f_s=0,
                             routing="plain"))
    layer, _, _ = check_layer(w)
    assert layer.saved["dest"].cpu().tolist() == list(range(300))


def test_top_k_equal_E():
    from layer_check import check_layer
    check_layer(make_workload(shrink("tiny_fp32", T=100, d=64, E=4, k=4, f=64)))


def test_single_token():
    from layer_check import check_layer
    check_layer(make_workload(shrink("pangu_bf16", T=1, d=256, E=8, k=2, f=128, f_s=128)))


def test_zero_tokens_is_noop_and_zero_grads():
    from dropless_token_routing_gb300.api import LayerParams, MoELayer, get_device_error
    w = make_workload(shrink("pangu_bf16", T=4, d=128, E=4, k=2, f=64, f_s=64))
    dev = "cuda"
    params = LayerParams(w13=w.w13.to(dev), w2=w.w2.to(dev), w_r=w.w_r.to(dev), bias=w.bias.to(dev),
                         ws13=w.ws13.to(dev), ws2=w.ws2.to(dev))
    layer = MoELayer(params, 0, 128, 4, 2, 64, 1, 64, torch.bfloat16)
    x = torch.empty(0, 128, dtype=torch.bfloat16, device=dev)
    layer.forward(x)
    g = layer.alloc_grads()
    for t in g.values():
        if t is not None:
            t.fill_(1.0)
    layer.backward(torch.empty(0, 128, dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    assert get_device_error(layer.ws) == 0
    assert layer.saved["counts"].sum().item() == 0 and layer.saved["offsets"].abs().sum().item() == 0
    for n in ("dw13", "dw2", "dws13", "dws2", "dw_r"):
        assert not g[n].any(), n


def test_selective_recompute_gives_identical_results():
    """x_perm and h not kept by the caller: the backward re-permutes x; bitwise the same."""
    from dropless_token_routing_gb300.api import LayerParams, MoELayer
    w = make_workload(shrink("pangu_bf16", T=700, d=512, E=16, k=4, f=256, f_s=256))
    c, dev = w.cfg, "cuda"
    to = lambda t: None if t is None else t.to(dev)  # noqa: E731
    out = []
    for rc in (False, True):
        params = LayerParams(w13=to(w.w13), w2=to(w.w2), w_r=to(w.w_r), bias=to(w.bias),
                             ws13=to(w.ws13), ws2=to(w.ws2))
        layer = MoELayer(params, c["T"], c["d"], c["E"], c["k"], c["f"], c["S"], c["f_s"],
                         torch.bfloat16, recompute=rc)
        y = layer.forward(to(w.x)).clone()
        g = {k_: v.clone() for k_, v in layer.backward(to(w.dy)).items() if v is not None}
        out.append((y, g))
    torch.cuda.synchronize()
    (y0, g0), (y1, g1) = out
    assert torch.equal(y0, y1)
    for k_ in g0:
        assert torch.equal(g0[k_], g1[k_]), k_


# ---------------------------------------------------------------- drop-and-pad variant
@pytest.mark.parametrize("case,cf", [("pangu_small", 1.0), ("pangu_small", 1.25),
                                     ("adversarial_small", 1.0), ("tiny_fp32", 0.75)])
def test_capacity_layer_matches_oracle(case, cf):
    """Drop-and-pad with C = ceil(cf * T * k / E) rows per expert against the oracle's
    capacity layer: bit-exact dest / row_src / offsets and zero padding rows, the usual
    float bars on y and every gradient (dropped copies pass nothing back)."""
    import math
    from layer_check import check_layer
    name, over = CASES[case]
    cfg = shrink(name, **over) if over else dict(__import__("synth").CONFIGS[name], name=name)
    C = math.ceil(cf * cfg["T"] * cfg["k"] / cfg["E"])
    layer, grads, _ = check_layer(make_workload(cfg), bwd=True, capacity=C)
    dest = layer.saved["dest"].cpu()
    counts = layer.saved["counts"].cpu()
    assert int((dest >= 0).sum()) == int(torch.clamp(counts, max=C).sum())
    if case == "adversarial_small":
        assert (dest < 0).any()        # the hot expert overflows


def test_capacity_at_max_count_reproduces_dropless_rows():
    """With C = the largest expert count nothing is dropped: every row's forward result is
    the dropless one bit for bit (a row's products do not depend on where it sits). dx agrees
    to rounding: the dropless bf16 path adds the router term to each dx row in the dX GEMM
    epilogue, the drop-and-pad path in the un-rearrangement. The dW products reduce over zero
    padding rows as well and agree to rounding."""
    from layer_check import run_gpu_layer
    w = make_workload(shrink("pangu_bf16", T=640, d=512, E=16, k=4, f=256, f_s=256))
    ref, gr, e0 = run_gpu_layer(w)
    C = int(ref.saved["counts"].max().item())
    cap, gc, e1 = run_gpu_layer(w, capacity=C)
    assert e0 == 0 and e1 == 0
    assert (cap.saved["dest"] >= 0).all()
    assert torch.equal(ref.y, cap.y)
    for n, tol in (("dx", 5e-3), ("dw13", 2e-3), ("dw2", 2e-3), ("dws13", 2e-3), ("dws2", 2e-3)):
        a, b = gr[n].float(), gc[n].float()
        assert (torch.linalg.norm(a - b) / torch.linalg.norm(a)).item() <= tol, n
    assert torch.allclose(gr["dw_r"], gc["dw_r"], rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------- fused rearrangement
@pytest.mark.parametrize("rearrange", [1, 2, 3])
@pytest.mark.parametrize("case", ["pangu_small", "dsv3_small", "adversarial_small"])
def test_fused_rearrangement_layer_matches_oracle(case, rearrange):
    """MOE_REARRANGE_GATHER (1): the expert GEMMs gather their token rows from x / dy by row_src
    (no rearranged copies of dY, x_perm kept only for the check); MOE_REARRANGE_SCATTER (2):
    the second expert GEMM writes its rows at their token-major slots and the combine reads
    each token's k rows as one block; 3: both. Every form meets every bar."""
    from layer_check import check_layer
    name, over = CASES[case]
    check_layer(make_workload(shrink(name, **over)), bwd=True, rearrange=rearrange)


@pytest.mark.parametrize("rearrange", [1, 2, 3])
def test_fused_rearrangement_matches_copies_bitwise(rearrange):
    """Gathered rows are the same bf16 values as the copied ones, fed in the same order, and the
    token-major rows are the same values the combine gathered by dest, summed in the same
    order: the forward, dX and dW results are bit-identical to the copy path."""
    from layer_check import run_gpu_layer
    w = make_workload(shrink("pangu_bf16", T=640, d=512, E=16, k=4, f=256, f_s=256))
    a, ga, e0 = run_gpu_layer(w)
    b, gb, e1 = run_gpu_layer(w, rearrange=rearrange)
    assert e0 == 0 and e1 == 0
    assert torch.equal(a.y, b.y) and torch.equal(a.saved["z"], b.saved["z"])
    for n in ("dx", "dw13", "dw2", "dws13", "dws2", "dw_r"):
        assert torch.equal(ga[n], gb[n]), n


# ---------------------------------------------------------------- limits
@pytest.mark.parametrize("case", ["bf16", "fp32"])
def test_layer_at_the_expert_and_topk_limits(case):
    """E = 1024 experts and k = 32 per token (the library's maxima): the chunk masks, the
    1024-wide scans, the 32-column top-k registers and the 1032-group tile schedule at full
    width, with most experts holding 0-3 rows; T = 333 leaves a ragged last chunk."""
    from layer_check import check_layer
    if case == "bf16":
        cfg = shrink("pangu_bf16", T=333, d=128, E=1024, k=32, f=64, f_s=64)
    else:
        cfg = shrink("tiny_fp32", T=333, d=64, E=1024, k=32, f=64)
    check_layer(make_workload(cfg), bwd=True)


def test_layer_step_replays_from_a_cuda_graph():
    """The whole forward + backward is asynchronous on one stream with no host wait, so it
    can be captured once in a CUDA graph and replayed: the replay gives the eager results bit
    for bit (after the first eager call has set up the kernels' attributes)."""
    from dropless_token_routing_gb300.api import LayerParams, MoELayer
    w = make_workload(shrink("pangu_bf16", T=640, d=512, E=16, k=4, f=256, f_s=256))
    c, dev = w.cfg, "cuda"
    to = lambda t: None if t is None else t.to(dev)  # noqa: E731
    params = LayerParams(w13=to(w.w13), w2=to(w.w2), w_r=to(w.w_r), bias=to(w.bias),
                         ws13=to(w.ws13), ws2=to(w.ws2))
    layer = MoELayer(params, c["T"], c["d"], c["E"], c["k"], c["f"], c["S"], c["f_s"], torch.bfloat16)
    x, dy = to(w.x), to(w.dy)
    y0 = layer.forward(x).clone()
    g0 = {k_: v.clone() for k_, v in layer.backward(dy).items() if v is not None}
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for t in list(layer.grads.values()) + [layer.y]:
            if t is not None:
                t.zero_()
        with torch.cuda.graph(graph, stream=s):
            layer.forward(x, stream=s)
            layer.backward(dy, stream=s)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.y, y0)
    for k_, v in g0.items():
        assert torch.equal(layer.grads[k_], v), k_


@pytest.mark.parametrize("k", [3, 8])
def test_combine_rows_longer_than_one_segment(k):
    """The combine's k <= 8 path hands each warp a segment of 1024 elements of one token's row:
    d = 1088 gives every row a full segment and a ragged one of 64 elements, in the forward
    combine and in the dX un-rearrangement."""
    from layer_check import check_layer
    check_layer(make_workload(shrink("pangu_bf16", T=100, d=1088, E=8, k=k, f=128, f_s=128)), bwd=True)


def test_experts_larger_than_one_tile_panel():
    """Groups of more than 16 M tiles (2048 rows) are walked in panels of 16 M tiles, the last
    one short (here 2 and 3 M tiles, the shared expert's last one a 64-row tile): T = 2200
    tokens on two experts and a shared expert, against the oracle."""
    from layer_check import check_layer
    check_layer(make_workload(shrink("pangu_bf16", T=2200, d=256, E=2, k=2, f=256, f_s=256)), bwd=True)


_THREADS_SCRIPT = r"""
import sys, threading
import torch
sys.path.insert(0, sys.argv[1])
from synth import make_workload, shrink
from dropless_token_routing_gb300.api import LayerParams, MoELayer

cfg = shrink("pangu_bf16", T=300, d=256, E=8, k=2, f=128, f_s=128)
ws = [make_workload(cfg, device="cuda", replica=r) for r in (0, 1)]
def build(w):
    p = LayerParams(w13=w.w13, w2=w.w2, w_r=w.w_r, bias=w.bias, ws13=w.ws13, ws2=w.ws2)
    c = w.cfg
    lay = MoELayer(p, c["T"], c["d"], c["E"], c["k"], c["f"], c["S"], c["f_s"], torch.bfloat16)
    lay.alloc_grads()
    return lay
layers = [build(w) for w in ws]
torch.cuda.synchronize()
out = [None, None]
gate = threading.Barrier(2)
def run(i):
    s = torch.cuda.Stream()
    gate.wait()   # both threads make their first library calls (one-time setup) at once
    for _ in range(3):
        y = layers[i].forward(ws[i].x, stream=s)
        g = layers[i].backward(ws[i].dy, stream=s)
    s.synchronize()
    out[i] = (y.clone(), {k: v.clone() for k, v in g.items() if v is not None})
th = [threading.Thread(target=run, args=(i,)) for i in (0, 1)]
for t in th: t.start()
for t in th: t.join()
for i in (0, 1):   # the same layers again, one after the other
    y = layers[i].forward(ws[i].x)
    g = layers[i].backward(ws[i].dy)
    torch.cuda.synchronize()
    assert torch.equal(y, out[i][0]), i
    for k, v in out[i][1].items():
        assert torch.equal(g[k], v), (i, k)
assert not torch.equal(out[0][0], out[1][0])
print("ok")
"""


def test_two_host_threads_call_the_library_at_once():
    """Two host threads, each with its own layer, workspace and stream, make their first calls
    into a freshly loaded library at the same moment (the per-device one-time setup runs under
    a lock) and run three steps; each thread's results equal the same layer run alone."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _THREADS_SCRIPT, root], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-2000:]


# ---------------------------------------------------------------- randomised shapes
def _random_shapes(n, seed):
    import random
    rng = random.Random(seed)
    out = []
    for i in range(n):
        bf16 = i % 3 != 2
        unit = 64 if bf16 else 8
        E = rng.choice([1, 2, 3, 7, 16, 33, 64, 100, 257])
        k = rng.randint(1, min(E, 32, 9))
        S = rng.choice([0, 0, 1, 2])
        cfg = dict(T=rng.choice([1, 5, 63, 64, 65, 200, 511, 700]), d=unit * rng.randint(1, 12),
                   E=E, k=k, f=unit * rng.randint(1, 8), S=S,
                   f_s=unit * rng.randint(1, 6) if S else 0)
        base = "pangu_bf16" if bf16 else "tiny_fp32"
        # the variants: dropless copies, drop-and-pad at a random capacity, fused row gathers
        variant = rng.choice(["copy", "copy", "capacity", "gather", "scatter"]) if bf16 else rng.choice(["copy", "capacity"])
        cap = max(1, int(cfg["T"] * k / E * rng.choice([0.5, 1.0, 1.5]))) if variant == "capacity" else 0
        out.append((base, cfg, cap, {"gather": 1, "scatter": 3}.get(variant, 0)))
    return out


@pytest.mark.parametrize("base,over,capacity,rearrange", _random_shapes(24, 2027))
def test_layer_on_random_shapes(base, over, capacity, rearrange):
    """Seeded random shapes (ragged everything: T from 1 to 700, d and f at any multiple of the
    vector unit, E up to 257, k up to 9, 0-2 shared experts, both dtypes), in the dropless,
    drop-and-pad, fused-gather and fused gather + scatter forms, each against the oracle at
    the usual bars."""
    from layer_check import check_layer
    cfg = shrink(base, **over)
    if cfg["S"] == 0:
        cfg["f_s"] = 0
    check_layer(make_workload(cfg), bwd=True, capacity=capacity, rearrange=rearrange)
