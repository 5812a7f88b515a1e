"""GPU parity of the individual C-ABI calls against the fp64 oracle, plus the device
error paths (expert ids out of range, a bounded wait that runs out)."""
import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu


def _api():
    from dropless_token_routing_gb300 import api
    return api


def _route(logits, k, bias=None):
    A = _api()
    T, E = logits.shape
    dims = A.make_dims(T, 64, E, k, 64, dtype=torch.float32)
    ws = A.Workspace(dims)
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    A.route_topk(logits, bias, k, idx, w, counts, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy()


@pytest.mark.parametrize("E,k", [(8, 2), (24, 3), (64, 6), (256, 8), (1000, 32), (5, 5), (33, 1)])
def test_route_topk_bitexact_with_ties(E, k):
    g = torch.Generator().manual_seed(E * 100 + k)
    T = 777
    # coarse values: many exact ties, including at the top-k boundary; a few -0.0 / +0.0
    L = (torch.randint(-6, 7, (T, E), generator=g).float() / 2).contiguous()
    L[::17, :3] = 0.0
    L[::19, 1] = -0.0
    bias = (torch.randint(-2, 3, (E,), generator=g).float() / 4)
    for b in (None, bias):
        idx, w, counts = _route(L.cuda(), k, None if b is None else b.cuda())
        s = O.selection_scores(L.numpy(), None if b is None else b.numpy())
        ridx, rw = O.route_topk(s, k)
        assert np.array_equal(idx, ridx)
        assert np.array_equal(counts, O.expert_counts(ridx, E))
        assert np.linalg.norm(w - rw) / np.linalg.norm(rw) <= 1e-5


def _permute(x, idx, E, w=None):
    A = _api()
    T, k = idx.shape
    d = x.shape[1]
    dt = x.dtype
    dims = A.make_dims(T, d, E, k, 64, dtype=dt)
    ws = A.Workspace(dims)
    Tk = T * k
    x_perm = torch.full((Tk, d), 7.0, dtype=dt, device="cuda")
    dest = torch.empty(Tk, dtype=torch.int32, device="cuda")
    row_src = torch.full((Tk,), -5, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    w_perm = torch.empty(Tk, dtype=torch.float32, device="cuda") if w is not None else None
    A.permute(x, idx, w, dims, x_perm, dest, row_src, offsets, w_perm, ws)
    err = A.get_device_error(ws)
    return x_perm, dest, row_src, offsets, w_perm, err


@pytest.mark.parametrize("T,E,k,skew", [(1, 8, 2, 0), (65, 3, 1, 0), (1000, 24, 3, 0),
                                         (3000, 256, 8, 1), (130, 7, 7, 0), (4097, 64, 6, 2)])
def test_permute_matches_stable_counting_sort(T, E, k, skew):
    g = torch.Generator().manual_seed(T + E)
    s = torch.randn(T, E, generator=g)
    if skew == 1:
        s[:, : E // 4] = -30.0           # dead experts
        s[: int(0.8 * T), E // 2] = 50.0  # hot expert
    if skew == 2:
        s[:, 5] += 3.0
    idx, _ = O.route_topk(s.numpy(), k)
    gate = torch.rand(T, k, generator=g)
    x = torch.randn(T, 64, generator=g).to(torch.bfloat16)
    x_perm, dest, row_src, offsets, w_perm, err = _permute(
        x.cuda(), torch.as_tensor(idx, dtype=torch.int32).cuda(), E, gate.cuda())
    assert err == 0
    rdest, rsrc = O.permutation(idx, E)
    assert np.array_equal(dest.cpu().numpy(), rdest)
    assert np.array_equal(row_src.cpu().numpy(), rsrc)
    assert np.array_equal(offsets.cpu().numpy(), O.expert_offsets(O.expert_counts(idx, E)))
    assert torch.equal(x_perm.cpu(), x[torch.as_tensor(rsrc)])
    wp = np.empty(T * k, np.float32)
    wp[rdest] = gate.numpy().reshape(-1)
    assert np.array_equal(w_perm.cpu().numpy(), wp)
    # gather-only mode and the unweighted / weighted combine
    A = _api()
    dims = A.make_dims(T, 64, E, k, 64, dtype=torch.bfloat16)
    again = torch.zeros_like(x_perm)
    A.permute_rows(x.cuda(), dest, dims, again)
    assert torch.equal(again, x_perm)
    y = torch.empty(T, 64, dtype=torch.bfloat16, device="cuda")
    A.unpermute_combine(x_perm, dest, None, None, dims, y)
    ref = O.as_f64(x) * k
    assert np.allclose(O.as_f64(y), ref, rtol=4e-3, atol=0)
    A.unpermute_combine(x_perm, dest, torch.as_tensor(gate).cuda(), x.cuda(), dims, y)
    ref = O.as_f64(x) * (gate.double().sum(1, keepdim=True).numpy() + 1.0)
    assert np.linalg.norm(O.as_f64(y) - ref) / np.linalg.norm(ref) <= 5e-3
    # the same rows in token-major order (dest NULL) give the same y bit for bit
    tok_major = x_perm[dest.long()]
    y2 = torch.empty_like(y)
    A.unpermute_combine(tok_major, None, torch.as_tensor(gate).cuda(), x.cuda(), dims, y2)
    assert torch.equal(y, y2)


@pytest.mark.parametrize("T,E,k,C", [(1000, 24, 3, 100), (3000, 256, 8, 90), (4097, 64, 6, 1),
                                     (130, 7, 7, 200)])
def test_capacity_permute_matches_oracle(T, E, k, C):
    """Drop-and-pad rearrangement: bit-exact dest / row_src / offsets / w_perm, kept rows
    moved exactly, padding rows zero."""
    A = _api()
    g = torch.Generator().manual_seed(T + E + C)
    s = torch.randn(T, E, generator=g)
    s[:, 3] += 2.0                                # one expert overflows
    idx, _ = O.route_topk(s.numpy(), k)
    gate = torch.rand(T, k, generator=g)
    x = torch.randn(T, 64, generator=g).to(torch.bfloat16)
    dims = A.make_dims(T, 64, E, k, 64, dtype=torch.bfloat16, capacity=C)
    ws = A.Workspace(dims)
    R = E * C
    x_perm = torch.full((R, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    dest = torch.empty(T * k, dtype=torch.int32, device="cuda")
    row_src = torch.full((R,), -5, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    w_perm = torch.full((R,), 3.0, dtype=torch.float32, device="cuda")
    A.permute(x.cuda(), torch.as_tensor(idx, dtype=torch.int32).cuda(), gate.cuda(), dims, x_perm,
              dest, row_src, offsets, w_perm, ws)
    assert A.get_device_error(ws) == 0
    rdest, rsrc = O.capacity_permutation(idx, E, C)
    assert np.array_equal(dest.cpu().numpy(), rdest)
    assert np.array_equal(row_src.cpu().numpy(), rsrc)
    assert np.array_equal(offsets.cpu().numpy(), np.arange(E + 1) * C)
    src = torch.as_tensor(rsrc)
    ref = torch.zeros(R, 64, dtype=torch.bfloat16)
    ref[src >= 0] = x[src[src >= 0]]
    assert torch.equal(x_perm.cpu(), ref)
    wp = np.zeros(R, np.float32)
    kept = rdest >= 0
    wp[rdest[kept]] = gate.numpy().reshape(-1)[kept]
    assert np.array_equal(w_perm.cpu().numpy(), wp)


@pytest.mark.parametrize("d,k,E", [(64, 16, 40), (1088, 12, 32), (448, 30, 64)])
def test_row_moves_when_a_row_ends_mid_warp(d, k, E):
    """Rows whose 16-byte vectors do not fill whole warp passes (d/8 = 8, 136, 56) with more
    copies per token than active lanes in the last pass: the scatter, the gather-only move and
    both combines must still place every copy."""
    A = _api()
    T = 300
    g = torch.Generator().manual_seed(d + k)
    idx, _ = O.route_topk(torch.randn(T, E, generator=g).numpy(), k)
    gate = torch.rand(T, k, generator=g)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    dims = A.make_dims(T, d, E, k, 64, dtype=torch.bfloat16)
    ws = A.Workspace(dims)
    x_perm = torch.zeros(T * k, d, dtype=torch.bfloat16, device="cuda")
    dest = torch.empty(T * k, dtype=torch.int32, device="cuda")
    row_src = torch.empty(T * k, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    A.permute(x.cuda(), torch.as_tensor(idx, dtype=torch.int32).cuda(), gate.cuda(), dims, x_perm, dest,
              row_src, offsets, None, ws)
    assert A.get_device_error(ws) == 0
    rdest, rsrc = O.permutation(idx, E)
    assert torch.equal(x_perm.cpu(), x[torch.as_tensor(rsrc)])
    again = torch.zeros_like(x_perm)
    A.permute_rows(x.cuda(), dest, dims, again)
    assert torch.equal(again, x_perm)
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    A.unpermute_combine(x_perm, dest, gate.cuda(), x.cuda(), dims, y)
    ref = O.as_f64(x) * (gate.double().sum(1, keepdim=True).numpy() + 1.0)
    assert np.linalg.norm(O.as_f64(y) - ref) / np.linalg.norm(ref) <= 5e-3


def test_permute_rejects_bad_expert_ids_without_writing_out_of_bounds():
    T, E, k = 200, 8, 2
    g = torch.Generator().manual_seed(3)
    idx, _ = O.route_topk(torch.randn(T, E, generator=g).numpy(), k)
    bad = idx.copy()
    bad[5, 0] = E          # out of range
    bad[9, 1] = -1         # negative
    bad[11, 1] = bad[11, 0]  # repeated within a row
    x = torch.randn(T, 64, generator=g).to(torch.bfloat16)
    x_perm, dest, row_src, offsets, _, err = _permute(
        x.cuda(), torch.as_tensor(bad, dtype=torch.int32).cuda(), E)
    from dropless_token_routing_gb300._native import STATUS_CODE
    assert err == STATUS_CODE["MOE_ERR_DEVICE_EXPERT_ID"]
    d = dest.cpu().numpy()
    assert d[5 * k + 0] == -1 and d[9 * k + 1] == -1 and d[11 * k + 1] == -1
    good = d[d >= 0]
    n_good = T * k - 3
    assert len(good) == n_good and sorted(good.tolist()) == list(range(n_good))
    assert offsets[-1].item() == n_good
    # rows past the valid copies were never written
    assert torch.all(x_perm[n_good:].float() == 7.0)
    assert torch.all(row_src[n_good:] == -5)


def test_bounded_wait_times_out_with_status():
    A = _api()
    from dropless_token_routing_gb300._native import STATUS_CODE
    dims = A.make_dims(1, 64, 2, 1, 64, dtype=torch.bfloat16)
    ws = A.Workspace(dims)
    A.debug_timeout_probe(ws, 2_000_000)  # 2 ms on a barrier nothing completes
    assert A.get_device_error(ws) == STATUS_CODE["MOE_ERR_DEVICE_TIMEOUT"]
    assert A.get_device_error(ws) == 0   # reading clears it
    # the context is still usable afterwards
    t = torch.ones(1024, device="cuda")
    assert t.sum().item() == 1024


def test_route_topk_bwd_matches_oracle():
    A = _api()
    T, E, k = 300, 40, 5
    g = torch.Generator().manual_seed(11)
    s = torch.randn(T, E, generator=g)
    idx, gate = O.route_topk(s.numpy(), k)
    dgate = torch.randn(T, k, generator=g)
    out = torch.empty(T, E, device="cuda")
    A.route_topk_bwd(torch.as_tensor(idx, dtype=torch.int32).cuda(),
                     torch.as_tensor(gate, dtype=torch.float32).cuda(), dgate.cuda(), E, out)
    ref = np.zeros((T, E))
    np.put_along_axis(ref, idx, O.router_backward(gate.astype(np.float32).astype(np.float64),
                                                  dgate.double().numpy()), axis=1)
    assert np.linalg.norm(out.cpu().double().numpy() - ref) / np.linalg.norm(ref) <= 1e-5


def test_balance_statistics_and_gradient_match_oracle():
    """moe_route_balance / moe_route_balance_bwd against the oracle's auxiliary balance loss."""
    A = _api()
    T, E, k, alpha = 1000, 64, 6, 0.01
    g = torch.Generator().manual_seed(21)
    L = torch.randn(T, E, generator=g) * 2
    bias = torch.randn(E, generator=g) * 0.5
    s32 = O.selection_scores(L.numpy(), bias.numpy())
    idx, _ = O.route_topk(s32, k)
    counts = O.expert_counts(idx, E)
    P_ref, L_ref = O.balance_loss(s32, counts, k, alpha)
    dims = A.make_dims(T, 64, E, k, 64, dtype=torch.float32)
    ws = A.Workspace(dims)
    Lg, bg = L.cuda(), bias.cuda()
    cg = torch.as_tensor(counts, dtype=torch.int32).cuda()
    P = torch.empty(E, device="cuda")
    aux = torch.empty(1, device="cuda")
    for _ in range(2):   # deterministic: the same bits twice
        A.route_balance(Lg, bg, cg, k, alpha, P, aux, ws)
        torch.cuda.synchronize()
        if _ == 0:
            P0, aux0 = P.clone(), aux.clone()
    assert torch.equal(P, P0) and torch.equal(aux, aux0)
    assert np.linalg.norm(P.cpu().double().numpy() - P_ref) / np.linalg.norm(P_ref) <= 1e-5
    assert abs(aux.item() - L_ref) / abs(L_ref) <= 1e-5
    # into zeros: the added term alone, compared with the oracle's gradient
    d0 = torch.zeros(T, E, device="cuda")
    A.route_balance_bwd(Lg, bg, cg, k, alpha, 1.7, d0)
    torch.cuda.synchronize()
    ref = 1.7 * O.balance_loss_grad(s32, counts, k, alpha)
    g0 = d0.cpu().double().numpy()
    assert np.linalg.norm(g0 - ref) / np.linalg.norm(ref) <= 1e-5
    # into an existing gradient: the call accumulates (one fp32 add, possibly fused)
    base = torch.randn(T, E, generator=g)
    d = base.clone().cuda()
    A.route_balance_bwd(Lg, bg, cg, k, alpha, 1.7, d)
    torch.cuda.synchronize()
    expect = base + d0.cpu()
    tol = 2 * torch.finfo(torch.float32).eps * (base.abs() + d0.cpu().abs()) + 1e-38
    assert torch.all((d.cpu() - expect).abs() <= tol)


@pytest.mark.parametrize("T,E,k,bias", [(1, 8, 2, False), (1000, 24, 3, True), (2053, 64, 6, True),
                                         (8192, 256, 8, True), (3000, 1000, 32, False)])
def test_route_with_fused_balance_is_bitwise_the_two_calls(T, E, k, bias):
    """moe_route_topk_balance gives the bits of moe_route_topk followed by moe_route_balance
    (indices, gates, counts, mean probabilities, loss), and the statistics match the oracle."""
    A = _api()
    alpha = 0.01
    g = torch.Generator().manual_seed(T + E)
    L = torch.randn(T, E, generator=g) * 2
    b = torch.randn(E, generator=g) * 0.5 if bias else None
    dims = A.make_dims(T, 64, E, k, 64, dtype=torch.float32)
    ws = A.Workspace(dims)
    Lg, bg = L.cuda(), (b.cuda() if bias else None)

    def outs():
        return (torch.empty(T, k, dtype=torch.int32, device="cuda"), torch.empty(T, k, device="cuda"),
                torch.empty(E, dtype=torch.int32, device="cuda"), torch.empty(E, device="cuda"),
                torch.empty(1, device="cuda"))
    i1, w1, c1, P1, a1 = outs()
    A.route_topk(Lg, bg, k, i1, w1, c1, ws)
    A.route_balance(Lg, bg, c1, k, alpha, P1, a1, ws)
    i2, w2, c2, P2, a2 = outs()
    A.route_topk_balance(Lg, bg, k, alpha, i2, w2, c2, P2, a2, ws)
    torch.cuda.synchronize()
    for u, v in ((i1, i2), (w1, w2), (c1, c2), (P1, P2), (a1, a2)):
        assert torch.equal(u, v)
    s32 = O.selection_scores(L.numpy(), b.numpy() if bias else None)
    idx, _ = O.route_topk(s32, k)
    assert np.array_equal(i2.cpu().numpy(), idx)
    counts = O.expert_counts(idx, E)
    P_ref, L_ref = O.balance_loss(s32, counts, k, alpha)
    assert np.linalg.norm(P2.cpu().double().numpy() - P_ref) / np.linalg.norm(P_ref) <= 1e-5
    assert abs(a2.item() - L_ref) / abs(L_ref) <= 1e-5


@pytest.mark.parametrize("T,E,k,L", [(1024, 64, 6, 256), (1000, 24, 3, 1000), (4096, 256, 8, 512)])
def test_balance_sequence_level_matches_oracle(T, E, k, L):
    """moe_route_balance_seq / _bwd (groups of L consecutive tokens) against the oracle."""
    A = _api()
    g = torch.Generator().manual_seed(T + L)
    Lg = torch.randn(T, E, generator=g) * 2
    bias = torch.randn(E, generator=g) * 0.5
    s32 = O.selection_scores(Lg.numpy(), bias.numpy())
    idx, _ = O.route_topk(s32, k)
    P_ref, c_ref, l_ref = O.balance_loss_groups(s32, idx, k, 0.01, L)
    G = T // L
    dims = A.make_dims(T, 64, E, k, 64, dtype=torch.float32)
    ws = A.Workspace(dims)
    lg, bg = Lg.cuda(), bias.cuda()
    ig = torch.as_tensor(idx, dtype=torch.int32).cuda()
    P = torch.empty(G, E, device="cuda")
    counts = torch.full((G, E), 7, dtype=torch.int32, device="cuda")
    aux = torch.empty(1, device="cuda")
    outs = []
    for _ in range(2):   # deterministic: the same bits twice
        A.route_balance_seq(lg, bg, ig, k, L, 0.01, P, counts, aux, ws)
        torch.cuda.synchronize()
        outs.append((P.clone(), counts.clone(), aux.clone()))
    assert all(torch.equal(a, b) for a, b in zip(outs[0], outs[1]))
    assert np.array_equal(counts.cpu().numpy(), c_ref)
    assert np.linalg.norm(P.cpu().double().numpy() - P_ref) / np.linalg.norm(P_ref) <= 1e-5
    assert abs(aux.item() - l_ref) / abs(l_ref) <= 1e-5
    d0 = torch.zeros(T, E, device="cuda")
    A.route_balance_seq_bwd(lg, bg, counts, k, L, G, 0.01, 1.3, d0)
    torch.cuda.synchronize()
    ref = 1.3 * O.balance_loss_groups_grad(s32, c_ref, k, 0.01, L)
    assert np.linalg.norm(d0.cpu().double().numpy() - ref) / np.linalg.norm(ref) <= 1e-5
