"""C-ABI checks that need no GPU: the library builds and loads, exports exactly
the entry points include/mkmoe.h declares, sizes its workspace, and rejects
bad arguments synchronously (before any CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

import dispatch_ffn_combine_gb300 as mk
from dispatch_ffn_combine_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return mk.load_library()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^MK_API\s+[\w\s\*]+?\b(mk_\w+)\s*\(", txt, flags=re.M))
    return names


def test_exports_match_header(lib):
    declared = _declared()
    assert declared == set(mk.ENTRY_POINTS)
    out = subprocess.run(["nm", "-D", "--defined-only", mk.LIB_PATH], capture_output=True, text=True, check=True)
    exported = {ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln}
    assert exported == declared, (exported ^ declared)


def test_workspace_size(lib):
    n = mk.workspace_size(32768, 7168, 256, 8, 2048)
    S = 32768 * 8
    # at least x_perm + h + P + the host staging buffers
    assert n >= 2 * S * 7168 + 2 * S * 2048 + 2 * S * 7168 + 2 * 2 * 32768 * 7168
    assert mk.workspace_size(0, 256, 8, 2, 512) > 0
    for bad in [(16, 100, 8, 2, 512), (16, 256, 0, 1, 512), (16, 256, 8, 9, 512), (16, 256, 4, 5, 512),
                (16, 256, 300, 2, 512), (16, 256, 8, 2, 500), (-1, 256, 8, 2, 512)]:
        assert mk.workspace_size(*bad) == 0, bad


def test_status_strings(lib):
    for s in range(7):
        assert mk.status_string(s).startswith("MK_")
    assert "unknown" in mk.status_string(99)


def _vp(v):
    return ctypes.c_void_p(v)


def test_layer_rejects_bad_arguments(lib):
    A = _vp(0x10000)  # never dereferenced: every case fails validation first
    T, d, E, k, f = 64, 256, 8, 2, 512
    need = mk.workspace_size(T, d, E, k, f)
    L = lib.mk_moe_layer
    ok_args = [A, A, None, A, A, A, T, d, E, k, f, A, A, need, None, None]

    def call(**over):
        args = list(ok_args)
        names = ["x", "wg", "bias", "w1", "w3", "w2", "T", "d", "E", "k", "f", "y", "ws", "wsb", "opts", "s"]
        for key, v in over.items():
            args[names.index(key)] = v
        return L(*args)

    assert call(d=100) == mk.MK_ERR_INVALID_ARG
    assert call(f=96) == mk.MK_ERR_INVALID_ARG
    assert call(k=0) == mk.MK_ERR_INVALID_ARG
    assert call(k=9, E=16) == mk.MK_ERR_INVALID_ARG
    assert call(E=257) == mk.MK_ERR_INVALID_ARG
    assert call(T=-5) == mk.MK_ERR_INVALID_ARG
    assert call(x=None) == mk.MK_ERR_INVALID_ARG
    assert call(w2=None) == mk.MK_ERR_INVALID_ARG
    assert call(x=_vp(0x10008)) == mk.MK_ERR_INVALID_ARG  # not 16-byte aligned
    assert call(ws=None) == mk.MK_ERR_WORKSPACE
    assert call(ws=_vp(0x10080)) == mk.MK_ERR_WORKSPACE  # not 256-byte aligned
    assert call(wsb=need - 1) == mk.MK_ERR_WORKSPACE
    assert call(T=1 << 28, k=8) == mk.MK_ERR_UNSUPPORTED  # T*k >= 2^31
    opts = mk.MkMoeOpts()
    opts.trace_cap = 4  # a record count without a buffer
    assert call(opts=ctypes.pointer(opts)) == mk.MK_ERR_INVALID_ARG
    opts = mk.MkMoeOpts()
    opts.path = 5
    assert call(opts=ctypes.pointer(opts)) == mk.MK_ERR_INVALID_ARG
    opts = mk.MkMoeOpts()
    opts.mover_ctas = -2
    assert call(opts=ctypes.pointer(opts)) == mk.MK_ERR_INVALID_ARG
    opts = mk.MkMoeOpts()
    opts.inject = 7
    assert call(opts=ctypes.pointer(opts)) == mk.MK_ERR_INVALID_ARG
    # T == 0 is a no-op that enqueues nothing
    assert call(T=0, wsb=mk.workspace_size(0, d, E, k, f)) == mk.MK_OK


def test_other_entry_points_reject_bad_arguments(lib):
    A = _vp(0x10000)
    T, d, E, k = 64, 256, 8, 2
    need = mk.workspace_size(T, d, E, k, 64)
    assert lib.mk_moe_route(None, A, None, T, d, E, k, A, A, None, A, need, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_moe_route(A, A, None, T, 96, E, k, A, A, None, A, need, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_moe_route(A, A, None, T, d, E, k, A, A, None, A, need - 1, None) == mk.MK_ERR_WORKSPACE
    assert lib.mk_moe_dispatch(A, A, None, T, d, E, k, None, A, None, A, A, A, need, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_moe_dispatch(A, A, None, T, d, E, 9, A, A, None, A, A, A, need, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_moe_expert_ffn(A, A, None, A, A, A, T, d, E, 100, A, A, A, 4096, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_moe_expert_ffn(A, A, None, A, A, A, T, d, E, 512, A, A, A, 16, None) == mk.MK_ERR_WORKSPACE
    assert lib.mk_moe_combine(A, A, T, d, 9, A, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_moe_combine(None, A, T, d, k, A, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_moe_combine(A, A, 0, d, k, A, None) == mk.MK_OK
    assert lib.mk_moe_last_device_error(None, None, None) == mk.MK_ERR_WORKSPACE
    assert lib.mk_moe_route_approx_logits(None, T, d, E, k, A, None) == mk.MK_ERR_WORKSPACE
    assert lib.mk_moe_route_approx_logits(A, T, d, E, k, None, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_moe_route_approx_logits(A, T, 100, E, k, A, None) == mk.MK_ERR_INVALID_ARG


def test_dispatch_gemm_entry_points_reject_bad_arguments(lib):
    A = _vp(0x10000)  # never dereferenced: every case fails validation first
    T, d, E, k, n = 64, 256, 8, 2, 512
    need = mk.dispatch_gemm_workspace_size(T, d, E, k)
    # the routing and dispatch regions plus the dispatched rows, and less than the layer's
    assert T * k * d * 2 < need < mk.workspace_size(T, d, E, k, n)
    assert mk.dispatch_gemm_workspace_size(T, 100, E, k) == 0
    assert mk.dispatch_gemm_workspace_size(T, d, E, 9) == 0
    G = lib.mk_moe_dispatch_gemm
    ok = [A, A, None, A, T, d, E, k, n, A, A, A, None, A, need, None]
    names = ["x", "wg", "bias", "w", "T", "d", "E", "k", "n", "out", "off", "row_token", "row_weight", "ws", "wsb",
             "s"]

    def call(**over):
        args = list(ok)
        for key, v in over.items():
            args[names.index(key)] = v
        return G(*args)

    assert call(n=96) == mk.MK_ERR_INVALID_ARG
    assert call(d=100) == mk.MK_ERR_INVALID_ARG
    assert call(k=0) == mk.MK_ERR_INVALID_ARG
    assert call(w=None) == mk.MK_ERR_INVALID_ARG
    assert call(out=None) == mk.MK_ERR_INVALID_ARG
    assert call(row_token=None) == mk.MK_ERR_INVALID_ARG
    assert call(w=_vp(0x10008)) == mk.MK_ERR_INVALID_ARG  # not 16-byte aligned
    assert call(ws=None) == mk.MK_ERR_WORKSPACE
    assert call(wsb=need - 1) == mk.MK_ERR_WORKSPACE
    assert call(T=1 << 28, k=8) == mk.MK_ERR_UNSUPPORTED
    Q = lib.mk_moe_grouped_gemm
    assert Q(A, A, None, A, T, d, E, 96, A, A, 4096, None) == mk.MK_ERR_INVALID_ARG
    assert Q(A, A, None, None, T, d, E, n, A, A, 4096, None) == mk.MK_ERR_INVALID_ARG
    assert Q(A, A, None, A, T, d, E, n, A, A, 16, None) == mk.MK_ERR_WORKSPACE
    assert Q(A, A, None, A, 0, d, E, n, A, A, 4096, None) == mk.MK_OK


def test_workspace_regions(lib):
    """Every region the layer leaves filled lies inside the workspace, starts
    256-byte aligned, has the bytes of its documented shape, and no two
    overlap."""
    for T, d, E, k, f in [(32768, 7168, 256, 8, 2048), (300, 128, 256, 1, 64), (1, 64, 3, 3, 64)]:
        total = mk.workspace_size(T, d, E, k, f)
        spans = []
        for name, (_, dtype, shape) in mk.WS_REGIONS.items():
            off, nb = mk.mk_moe_workspace_region(T, d, E, k, f, name)
            n = 1
            for s in shape(T, d, E, k, f):
                n *= s
            esz = 2 if dtype.is_floating_point and dtype.itemsize == 2 else 4
            assert nb == n * esz, name
            assert off % 256 == 0 and off + nb <= total, name
            spans.append((off, off + nb, name))
        spans.sort()
        for (a0, a1, na), (b0, b1, nb_) in zip(spans, spans[1:]):
            assert a1 <= b0, (na, nb_)
    off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    R = lib.mk_moe_workspace_region
    assert R(64, 256, 8, 2, 512, 9, ctypes.byref(off), ctypes.byref(nb)) == mk.MK_ERR_INVALID_ARG
    assert R(64, 100, 8, 2, 512, 0, ctypes.byref(off), ctypes.byref(nb)) == mk.MK_ERR_INVALID_ARG
    assert R(64, 256, 8, 2, 512, 0, None, ctypes.byref(nb)) == mk.MK_ERR_INVALID_ARG


def test_noalloc_router_rejects_bad_arguments(lib):
    """The no-alloc router runs mk_moe_route's checks in the same order (sizes,
    pointers, alignment) before its own limit on T * E, so both entry points
    answer the same for the same arguments."""
    A = _vp(0x10000)  # never dereferenced: every case fails validation first
    N = lib.mk_moe_route_noalloc
    T, d, E, k = 64, 256, 8, 2
    assert N(A, A, None, T, 96, E, k, A, A, None, None) == mk.MK_ERR_INVALID_ARG
    assert N(A, A, None, T, d, E, 9, A, A, None, None) == mk.MK_ERR_INVALID_ARG
    assert N(A, A, None, -1, d, E, k, A, A, None, None) == mk.MK_ERR_INVALID_ARG
    assert N(None, A, None, 0, d, E, k, A, A, None, None) == mk.MK_ERR_INVALID_ARG  # pointers before T == 0
    assert N(A, A, None, T, d, E, k, None, A, None, None) == mk.MK_ERR_INVALID_ARG
    assert N(_vp(0x10008), A, None, T, d, E, k, A, A, None, None) == mk.MK_ERR_INVALID_ARG
    assert N(A, A, None, 8193, 64, 256, 2, A, A, None, None) == mk.MK_ERR_UNSUPPORTED  # T * E > 2^21
    assert N(A, A, None, 1 << 28, 64, 8, 8, A, A, None, None) == mk.MK_ERR_UNSUPPORTED  # T * k >= 2^31
    assert lib.mk_moe_route(None, A, None, 0, d, E, k, A, A, None, A, 1 << 20, None) == mk.MK_ERR_INVALID_ARG
