"""moe_permute_noalloc, the permutation for callers that cannot allocate device memory, gives
exactly what moe_permute gives (its scratch is a static device array instead of a
workspace). Collected last on purpose: it runs after every other test in the same process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else t.data_ptr()


def _outputs(T, d, E, k, dtype):
    Tk = T * k
    dev = "cuda"
    return dict(x_perm=torch.full((Tk, d), 3.0, dtype=dtype, device=dev),
                dest=torch.full((Tk,), -7, dtype=torch.int32, device=dev),
                row_src=torch.full((Tk,), -7, dtype=torch.int32, device=dev),
                offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
                w_perm=torch.full((Tk,), -1.0, dtype=torch.float32, device=dev))


@pytest.mark.parametrize("T,E,k,d,dtype", [(2000, 64, 6, 256, torch.bfloat16),
                                           (16384, 256, 8, 64, torch.bfloat16),
                                           (333, 8, 2, 64, torch.float32)])
def test_noalloc_permute_matches_workspace_permute_twice(T, E, k, d, dtype):
    from dropless_token_routing_gb300 import _native as N
    from dropless_token_routing_gb300.api import Workspace, make_dims, permute
    lib = N.lib()
    g = torch.Generator().manual_seed(T + E)
    scores = torch.randn(T, E, generator=g)
    scores[:, 3] += 2.0
    idx, gate = O.route_topk(scores.numpy(), k)
    x = torch.randn(T, d, generator=g).to(dtype).cuda()
    topk_idx = torch.as_tensor(idx, dtype=torch.int32).cuda()
    topk_w = torch.as_tensor(gate, dtype=torch.float32).cuda()
    dims = make_dims(T, d, E, k, 64, dtype=dtype)
    ref = _outputs(T, d, E, k, dtype)
    ws = Workspace(dims)
    permute(x, topk_idx, topk_w, dims, ref["x_perm"], ref["dest"], ref["row_src"], ref["offsets"],
            ref["w_perm"], ws)
    stream = torch.cuda.current_stream().cuda_stream
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):       # the static scratch keeps the previous call's contents
        out = _outputs(T, d, E, k, dtype)
        st = lib.moe_permute_noalloc(_p(x), _p(topk_idx), _p(topk_w), ctypes.byref(dims),
                                     _p(out["x_perm"]), _p(out["dest"]), _p(out["row_src"]),
                                     _p(out["offsets"]), _p(out["w_perm"]), _p(err), stream)
        assert st == 0, N.status_string(st)
        torch.cuda.synchronize()
        assert err.item() == 0
        for name in ("dest", "row_src", "offsets", "x_perm", "w_perm"):
            assert torch.equal(out[name], ref[name]), (call, name)
    assert np.array_equal(ref["dest"].cpu().numpy(), O.permutation(idx, E)[0])


def _noalloc(lib, x, topk_idx, topk_w, dims, out, err):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.moe_permute_noalloc(_p(x), _p(topk_idx), _p(topk_w), ctypes.byref(dims),
                                   _p(out["x_perm"]), _p(out["dest"]), _p(out["row_src"]),
                                   _p(out["offsets"]), _p(out["w_perm"]), _p(err), stream)


def test_noalloc_permute_reports_invalid_ids_like_the_workspace_permute():
    """An id outside [0, E) and an id repeated within a row are reported in the caller's error
    word; those copies get dest = -1 and move no row, exactly as in moe_permute."""
    from dropless_token_routing_gb300 import _native as N
    from dropless_token_routing_gb300.api import Workspace, get_device_error, make_dims, permute
    lib = N.lib()
    T, E, k, d = 300, 16, 4, 128
    g = torch.Generator().manual_seed(11)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    idx[5, 2] = E            # out of range
    idx[17, 0] = -1          # out of range
    idx[40, 3] = idx[40, 1]  # repeated within the row
    gate = torch.rand(T, k, generator=g, dtype=torch.float32)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16).cuda()
    topk_idx, topk_w = idx.cuda(), gate.cuda()
    dims = make_dims(T, d, E, k, 64, dtype=torch.bfloat16)
    ref = _outputs(T, d, E, k, torch.bfloat16)
    ws = Workspace(dims)
    permute(x, topk_idx, topk_w, dims, ref["x_perm"], ref["dest"], ref["row_src"], ref["offsets"],
            ref["w_perm"], ws)
    assert get_device_error(ws) == N.STATUS_CODE["MOE_ERR_DEVICE_EXPERT_ID"]
    dest = ref["dest"].cpu().view(T, k)
    assert dest[5, 2] == -1 and dest[17, 0] == -1 and dest[40, 3] == -1 and dest[40, 1] >= 0
    for call in range(2):
        out = _outputs(T, d, E, k, torch.bfloat16)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = _noalloc(lib, x, topk_idx, topk_w, dims, out, err)
        assert st == 0, N.status_string(st)
        torch.cuda.synchronize()
        assert err.item() == N.STATUS_CODE["MOE_ERR_DEVICE_EXPERT_ID"], call
        for name in ("dest", "row_src", "offsets", "x_perm", "w_perm"):
            assert torch.equal(out[name], ref[name]), (call, name)


def test_noalloc_permute_with_no_tokens_writes_zero_offsets():
    from dropless_token_routing_gb300 import _native as N
    from dropless_token_routing_gb300.api import make_dims
    lib = N.lib()
    E = 32
    dims = make_dims(0, 256, E, 4, 64, dtype=torch.bfloat16)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.moe_permute_noalloc(None, None, None, ctypes.byref(dims), None, None, None,
                                 _p(offsets), None, _p(err), stream)
    assert st == 0, N.status_string(st)
    torch.cuda.synchronize()
    assert not offsets.any() and err.item() == 0
