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


def test_noalloc_permute_rejects_problems_beyond_its_scratch():
    from dropless_token_routing_gb300 import _native as N
    from dropless_token_routing_gb300.api import make_dims
    lib = N.lib()
    fake = 0x10000  # never dereferenced: the size check comes first
    too_many_copies = make_dims(40000, 64, 16, 8, 64, dtype=torch.bfloat16)   # T*k > 262144
    st = lib.moe_permute_noalloc(fake, fake, fake, ctypes.byref(too_many_copies), fake, fake, fake,
                                 fake, fake, None, None)
    assert st == N.STATUS_CODE["MOE_ERR_WORKSPACE_TOO_SMALL"]
    too_many_cells = make_dims(8192, 64, 1024, 2, 64, dtype=torch.bfloat16)   # E*T/64 > 65536
    st = lib.moe_permute_noalloc(fake, fake, fake, ctypes.byref(too_many_cells), fake, fake, fake,
                                 fake, fake, None, None)
    assert st == N.STATUS_CODE["MOE_ERR_WORKSPACE_TOO_SMALL"]
