"""The C-ABI library loads, exports every function include/moe.h declares, and its
host-side argument checks reject bad calls before anything reaches a GPU (CPU only:
every call here fails validation, so no CUDA API is touched)."""
import ctypes
import os
import subprocess

import pytest

from dropless_token_routing_gb300 import builder as B

if not os.path.exists(B.LIB):
    B.build()

from dropless_token_routing_gb300 import _native as N  # noqa: E402

L = N.lib()
BAD = 0x1008    # not 16-byte aligned; never dereferenced
GOOD = 0x10000  # aligned fake address, never dereferenced on the paths tested here


def dims(**kw):
    base = dict(T=256, d=512, E=8, k=2, f=256, S=0, f_s=0, dtype=N.MOE_F32)
    base.update(kw)
    return N.MoeDims(*[base[n] for n in ("T", "d", "E", "k", "f", "S", "f_s", "dtype")])


def test_exports_every_header_function():
    names = N.header_functions()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)


def test_status_strings():
    for code, name in N.STATUS.items():
        s = N.status_string(code)
        assert s and s != "unknown status", name
    assert N.status_string(12345) == "unknown status"


def test_workspace_bytes_and_dims_validation():
    d = dims()
    assert L.moe_workspace_bytes(ctypes.byref(d)) > 256
    assert L.moe_workspace_bytes(ctypes.byref(dims(k=9))) == 0            # k > E
    assert L.moe_workspace_bytes(ctypes.byref(dims(E=2000, k=2))) == 0    # E > 1024
    assert L.moe_workspace_bytes(ctypes.byref(dims(dtype=7))) == 0
    assert L.moe_workspace_bytes(ctypes.byref(dims(d=100))) == 0          # fp32 needs d % 8
    assert L.moe_workspace_bytes(ctypes.byref(dims(dtype=N.MOE_BF16, d=96))) == 0  # bf16 d % 64
    assert L.moe_workspace_bytes(ctypes.byref(dims(T=-1))) == 0
    assert L.moe_workspace_bytes(ctypes.byref(dims(T=2**31))) == 0        # T must fit in int32
    assert L.moe_workspace_bytes(ctypes.byref(dims(T=2**62, k=8))) == 0   # rejected before T*k
    assert L.moe_workspace_bytes(ctypes.byref(dims(T=0))) >= 256         # T = 0 is valid
    big = dims(T=16384, d=7680, E=256, k=8, f=2048, S=1, f_s=2048, dtype=N.MOE_BF16)
    nb = L.moe_workspace_bytes(ctypes.byref(big))
    assert 4e9 < nb < 2e10


def test_rearrange_flags_are_validated():
    """moe_dims.rearrange takes the flags copy (0), gather (1), scatter (2) and both (3); the
    scatter form reserves one int32 per token copy for the token-major slots."""
    def with_rearrange(r, **kw):
        d = dims(dtype=N.MOE_BF16, **kw)
        d.rearrange = r
        return d
    sizes = {r: L.moe_workspace_bytes(ctypes.byref(with_rearrange(r))) for r in (0, 1, 2, 3)}
    assert all(v > 256 for v in sizes.values())
    assert sizes[2] >= sizes[0] + 4 * 256 * 2 and sizes[3] == sizes[2] and sizes[1] == sizes[0]
    for bad in (-1, 4, 7):
        assert L.moe_workspace_bytes(ctypes.byref(with_rearrange(bad))) == 0


def _code(name):
    return N.STATUS_CODE[name]


def test_host_argument_errors():
    d = dims()
    ws_n = L.moe_workspace_bytes(ctypes.byref(d))
    # bad top-k / dims on route_topk
    assert L.moe_route_topk(GOOD, None, 16, 8, 9, GOOD, GOOD, GOOD, GOOD, 256, None) == _code("MOE_ERR_BAD_TOPK")
    assert L.moe_route_topk(GOOD, None, 16, 8, 0, GOOD, GOOD, GOOD, GOOD, 256, None) == _code("MOE_ERR_BAD_TOPK")
    assert L.moe_route_topk(GOOD, None, 16, 0, 1, GOOD, GOOD, GOOD, GOOD, 256, None) == _code("MOE_ERR_BAD_DIMS")
    assert L.moe_route_topk(None, None, 16, 8, 2, GOOD, GOOD, GOOD, GOOD, 256, None) == _code("MOE_ERR_NULL_POINTER")
    assert L.moe_route_topk(BAD, None, 16, 8, 2, GOOD, GOOD, GOOD, GOOD, 256, None) == _code("MOE_ERR_MISALIGNED")
    assert L.moe_route_topk(GOOD, BAD, 16, 8, 2, GOOD, GOOD, GOOD, GOOD, 256, None) == _code("MOE_ERR_MISALIGNED")
    assert L.moe_route_topk(GOOD, None, 16, 8, 2, GOOD, GOOD, GOOD, GOOD + 16, 256, None) == _code("MOE_ERR_MISALIGNED")
    assert L.moe_route_topk(GOOD, None, 16, 8, 2, GOOD, GOOD, GOOD, GOOD, 128, None) == _code("MOE_ERR_WORKSPACE_TOO_SMALL")
    # permute: workspace too small, null output, unsupported dtype
    assert L.moe_permute(GOOD, GOOD, GOOD, ctypes.byref(d), GOOD, GOOD, GOOD, GOOD, GOOD, GOOD,
                         ws_n - 1, None) == _code("MOE_ERR_WORKSPACE_TOO_SMALL")
    assert L.moe_permute(GOOD, GOOD, GOOD, ctypes.byref(d), None, GOOD, GOOD, GOOD, GOOD, GOOD,
                         ws_n, None) == _code("MOE_ERR_NULL_POINTER")
    bad_dt = dims(dtype=3)
    assert L.moe_permute(GOOD, GOOD, GOOD, ctypes.byref(bad_dt), GOOD, GOOD, GOOD, GOOD, GOOD, GOOD,
                         ws_n, None) == _code("MOE_ERR_UNSUPPORTED_DTYPE")
    assert L.moe_permute_rows(GOOD, BAD, ctypes.byref(d), GOOD, None) == _code("MOE_ERR_MISALIGNED")
    # grouped GEMM: shared experts need their buffers
    ds = dims(S=1, f_s=64)
    ws_s = L.moe_workspace_bytes(ctypes.byref(ds))
    assert L.moe_grouped_swiglu_fwd(GOOD, None, GOOD, GOOD, GOOD, GOOD, GOOD, ctypes.byref(ds), GOOD,
                                    GOOD, GOOD, GOOD, GOOD, GOOD, GOOD, ws_s, None) == _code("MOE_ERR_NULL_POINTER")
    assert L.moe_unpermute_combine(GOOD, GOOD, BAD, None, ctypes.byref(d), GOOD, None) == _code("MOE_ERR_MISALIGNED")
    # dest NULL (token-major rows) is refused for drop-and-pad, where copies can be dropped
    dc = dims()
    dc.capacity = 4
    assert L.moe_unpermute_combine(GOOD, None, None, None, ctypes.byref(dc), GOOD, None) == _code("MOE_ERR_NULL_POINTER")
    assert L.moe_route_topk_bwd(GOOD, GOOD, GOOD, 4, 8, 9, GOOD, None) == _code("MOE_ERR_BAD_TOPK")
    # routing with the balance statistics: T >= 1, the statistics' workspace, a loss output
    rb = L.moe_route_topk_balance
    a = 0.01
    assert rb(GOOD, None, 0, 8, 2, a, GOOD, GOOD, GOOD, None, GOOD, GOOD, 4096, None) == _code("MOE_ERR_BAD_DIMS")
    assert rb(GOOD, None, 16, 8, 9, a, GOOD, GOOD, GOOD, None, GOOD, GOOD, 4096, None) == _code("MOE_ERR_BAD_TOPK")
    assert rb(GOOD, None, 16, 8, 2, a, GOOD, GOOD, GOOD, None, None, GOOD, 4096, None) == _code("MOE_ERR_NULL_POINTER")
    assert rb(GOOD, None, 16, 8, 2, a, GOOD, GOOD, GOOD, BAD, GOOD, GOOD, 4096, None) == _code("MOE_ERR_MISALIGNED")
    # 16 tokens -> 2 partial rows of 8 experts and one loss share: 256 + 68 bytes
    assert rb(GOOD, None, 16, 8, 2, a, GOOD, GOOD, GOOD, None, GOOD, GOOD, 256 + 67, None) == \
        _code("MOE_ERR_WORKSPACE_TOO_SMALL")
    assert rb(GOOD, None, 16, 8, 2, a, GOOD, GOOD, GOOD, None, GOOD, GOOD + 16, 4096, None) == _code("MOE_ERR_MISALIGNED")
    # layer calls: router weights or logits must be given; grads need dlogits without W_r
    p = N.LayerParams(None, None, GOOD, GOOD, None, None)
    s = N.LayerSaved(*([GOOD] * 13))
    assert L.moe_layer_fwd(ctypes.byref(p), GOOD, None, ctypes.byref(d), ctypes.byref(s), GOOD, GOOD,
                           ws_n, None) == _code("MOE_ERR_NULL_POINTER")
    g = N.LayerGrads(GOOD, GOOD, GOOD, None, None, None, None)
    assert L.moe_layer_bwd(ctypes.byref(p), ctypes.byref(s), GOOD, GOOD, ctypes.byref(d), ctypes.byref(g),
                           GOOD, ws_n, None) == _code("MOE_ERR_NULL_POINTER")
    assert L.moe_layer_fwd(None, GOOD, None, ctypes.byref(d), ctypes.byref(s), GOOD, GOOD, ws_n,
                           None) == _code("MOE_ERR_NULL_POINTER")
    assert L.moe_debug_timeout_probe(GOOD + 16, 256, 1000, None) == _code("MOE_ERR_MISALIGNED")


def test_import_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib
    import sys
    monkeypatch.setattr(B, "LIB", str(tmp_path / "missing.so"))
    sys.modules.pop("dropless_token_routing_gb300._native", None)
    try:
        with pytest.raises(ImportError):
            importlib.import_module("dropless_token_routing_gb300._native")
    finally:
        monkeypatch.undo()
        sys.modules.pop("dropless_token_routing_gb300._native", None)
        importlib.import_module("dropless_token_routing_gb300._native")


def test_noalloc_permute_rejects_bad_calls_before_launching():
    """The workspace-free permutation checks sizes, widths and pointers on the host; every call
    here is rejected before any CUDA API is touched (the fake addresses are never used)."""
    def bf16(**kw):
        return dims(dtype=N.MOE_BF16, f=64, **kw)

    def call(dm, x_perm=GOOD, dest=GOOD, dev_err=None):
        return L.moe_permute_noalloc(GOOD, GOOD, GOOD, ctypes.byref(dm), x_perm, dest, GOOD, GOOD,
                                     GOOD, dev_err, None)

    assert call(bf16(T=40000, d=64, E=16, k=8)) == _code("MOE_ERR_WORKSPACE_TOO_SMALL")   # T*k > 2^18
    assert call(bf16(T=8192, d=64, E=1024, k=2)) == _code("MOE_ERR_WORKSPACE_TOO_SMALL")  # E*T/64 > 2^16
    assert call(bf16(T=2 ** 62, d=64, E=16, k=8)) == _code("MOE_ERR_WORKSPACE_TOO_SMALL")  # T*k overflows
    assert call(bf16(T=256, d=72, E=16, k=2)) == _code("MOE_ERR_BAD_DIMS")                 # bf16: d % 64
    ok = bf16(T=256, d=128, E=16, k=2)
    assert call(ok, dev_err=GOOD + 2) == _code("MOE_ERR_MISALIGNED")   # not a 32-bit atomic's word
    assert call(ok, x_perm=BAD) == _code("MOE_ERR_MISALIGNED")
    assert call(ok, dest=None) == _code("MOE_ERR_NULL_POINTER")


def test_workspace_grows_with_every_dimension_and_the_capacity_tables():
    """moe_workspace_bytes is monotone in T, d, f, E, k and the shared experts, and the
    drop-and-pad variant adds its dropless index tables (two int32 per token copy and the
    dropless offsets) to permuted buffers of E*C rows."""
    base = dict(T=1024, d=512, E=16, k=4, f=256, S=1, f_s=256, dtype=N.MOE_BF16)

    def ws(capacity=0, **kw):
        d = dims(**{**base, **kw})
        d.capacity = capacity
        return L.moe_workspace_bytes(ctypes.byref(d))

    w0 = ws()
    for kw in (dict(T=2048), dict(d=1024), dict(f=512), dict(E=32), dict(k=8), dict(S=2), dict(f_s=512)):
        assert ws(**kw) > w0, kw
    Tk = base["T"] * base["k"]
    # E*C == T*k: the same permuted rows, plus the three dropless tables
    assert ws(capacity=Tk // base["E"]) >= w0 + 8 * Tk
    # a larger capacity only adds rows
    assert ws(capacity=2 * Tk // base["E"]) > ws(capacity=Tk // base["E"])
