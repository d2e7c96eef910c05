"""GB300-native fused MoE layer: route -> dispatch -> grouped SwiGLU FFN -> combine.

A thin binding over the C ABI of ``libmkmoe.so`` (``include/mkmoe.h``).  Every
step of the layer runs in the library's sm_103a kernels; this module only
marshals torch tensors (device memory, streams) into the C calls, with the
same names.  There is no fallback: if the library is missing or the device is
not sm_103, calls raise.

    import dispatch_ffn_combine_gb300 as mk
    y = mk.mk_moe_layer(x, wg, bias, w1, w3, w2, k)      # torch CUDA tensors
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmkmoe.so")

MK_OK = 0
MK_ERR_INVALID_ARG = 1
MK_ERR_WORKSPACE = 2
MK_ERR_UNSUPPORTED = 3
MK_ERR_CUDA = 4
MK_ERR_TIMEOUT = 5
MK_ERR_BOUNDS = 6

PHASES = ("route_logits", "topk", "count", "scan", "scatter", "gemm1", "gemm2", "combine")

# Every entry point the header declares (checked against the library's exports).
ENTRY_POINTS = (
    "mk_moe_workspace_size", "mk_moe_route", "mk_moe_dispatch", "mk_moe_expert_ffn", "mk_moe_combine",
    "mk_moe_layer", "mk_moe_layer_host", "mk_moe_layer_host_async", "mk_moe_last_device_error",
    "mk_moe_status_string",
    "mk_moe_layer_routing", "mk_moe_route_noalloc", "mk_moe_layer_trace_count", "mk_moe_route_fallbacks",
    "mk_moe_grouped_gemm", "mk_moe_dispatch_gemm_workspace_size", "mk_moe_dispatch_gemm",
    "mk_moe_route_approx_logits", "mk_moe_workspace_region", "mk_moe_ep_regroup_workspace_size",
    "mk_moe_ep_regroup",
)
_SIZE_RESULT = ("mk_moe_workspace_size", "mk_moe_dispatch_gemm_workspace_size", "mk_moe_ep_regroup_workspace_size")

_lock = threading.Lock()
_lib = None


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class MkMoeOpts(ctypes.Structure):
    _fields_ = [("timeout_ns", ctypes.c_uint64), ("phase_events", ctypes.POINTER(ctypes.c_void_p)),
                ("inject", ctypes.c_int), ("path", ctypes.c_int), ("mover_ctas", ctypes.c_int),
                ("trace_cap", ctypes.c_int), ("trace", ctypes.c_void_p), ("gather_rows", ctypes.c_int)]


MK_INJECT_STALL_GEMM1 = 1
MK_INJECT_ROUTE_ZERO_BOUND = 2
MK_INJECT_DROP_TILE_SIGNAL = 3
MK_PATH_STEPS = 0
MK_PATH_FUSED = 1
MK_PATH_TILES = 2


def load_library():
    """Load libmkmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m dispatch_ffn_combine_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        lib.mk_moe_workspace_size.restype = SZ
        lib.mk_moe_workspace_size.argtypes = [I64, I, I, I, I]
        lib.mk_moe_status_string.restype = ctypes.c_char_p
        lib.mk_moe_status_string.argtypes = [I]
        lib.mk_moe_route.argtypes = [P, P, P, I64, I, I, I, P, P, P, P, SZ, P]
        lib.mk_moe_dispatch.argtypes = [P, P, P, I64, I, I, I, P, P, P, P, P, P, SZ, P]
        lib.mk_moe_expert_ffn.argtypes = [P, P, P, P, P, P, I64, I, I, I, P, P, P, SZ, P]
        lib.mk_moe_combine.argtypes = [P, P, I64, I, I, P, P]
        lib.mk_moe_layer.argtypes = [P, P, P, P, P, P, I64, I, I, I, I, P, P, SZ, ctypes.POINTER(MkMoeOpts), P]
        lib.mk_moe_layer_host.argtypes = lib.mk_moe_layer.argtypes
        lib.mk_moe_layer_host_async.argtypes = lib.mk_moe_layer.argtypes + [P]
        lib.mk_moe_last_device_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
        lib.mk_moe_layer_routing.argtypes = [P, I64, I, I, I, I, P, P, P, P, P]
        lib.mk_moe_route_noalloc.argtypes = [P, P, P, I64, I, I, I, P, P, P, P]
        lib.mk_moe_layer_trace_count.argtypes = [P, I64, I, I, I, I, P, ctypes.POINTER(ctypes.c_uint32)]
        lib.mk_moe_route_fallbacks.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
        lib.mk_moe_grouped_gemm.argtypes = [P, P, P, P, I64, I, I, I, P, P, SZ, P]
        lib.mk_moe_dispatch_gemm_workspace_size.restype = SZ
        lib.mk_moe_dispatch_gemm_workspace_size.argtypes = [I64, I, I, I]
        lib.mk_moe_dispatch_gemm.argtypes = [P, P, P, P, I64, I, I, I, I, P, P, P, P, P, SZ, P]
        lib.mk_moe_route_approx_logits.argtypes = [P, I64, I, I, I, P, P]
        lib.mk_moe_workspace_region.argtypes = [I64, I, I, I, I, I, ctypes.POINTER(SZ), ctypes.POINTER(SZ)]
        lib.mk_moe_ep_regroup_workspace_size.restype = SZ
        lib.mk_moe_ep_regroup_workspace_size.argtypes = [I, I]
        lib.mk_moe_ep_regroup.argtypes = [P, P, P, I, I, I64, I, I, P, P, SZ, P]
        for name in ENTRY_POINTS:
            if name not in _SIZE_RESULT + ("mk_moe_status_string",):
                getattr(lib, name).restype = I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().mk_moe_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != MK_OK:
        raise MoEError(status, what)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, shape, name, device=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t


def workspace_size(T: int, d: int, E: int, k: int, ffn: int) -> int:
    return int(load_library().mk_moe_workspace_size(T, d, E, k, ffn))


def alloc_workspace(T: int, d: int, E: int, k: int, ffn: int, device="cuda") -> torch.Tensor:
    n = workspace_size(T, d, E, k, ffn)
    if n == 0:
        raise ValueError("invalid sizes for the MoE layer")
    return torch.empty(n, dtype=torch.uint8, device=device)


def mk_moe_route(x, wg, bias, k, topk_ids=None, topk_w=None, expert_counts=None, ws=None, stream=None):
    """Router: returns (topk_ids [T,k] int32, topk_w [T,k] fp32, expert_counts [E] int32)."""
    T, d = x.shape
    E = wg.shape[0]
    _need(x, torch.bfloat16, (T, d), "x")
    _need(wg, torch.float32, (E, d), "wg")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    dev = x.device
    topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    topk_w = torch.empty((T, k), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    expert_counts = torch.empty(E, dtype=torch.int32, device=dev) if expert_counts is None else expert_counts
    ws = alloc_workspace(T, d, E, k, 64, dev) if ws is None else ws
    st = load_library().mk_moe_route(_p(x), _p(wg), _p(bias), T, d, E, k, _p(topk_ids), _p(topk_w),
                                     _p(expert_counts), _p(ws), ws.numel(), _stream(stream))
    _check(st, "mk_moe_route")
    return topk_ids, topk_w, expert_counts


def mk_moe_route_noalloc(x, wg, bias, k, topk_ids, topk_w, expert_counts=None, stream=None):
    """Router for callers that cannot allocate device memory: no workspace, the
    logits go to a static 8 MiB device array inside the library (T*E <= 2**21).
    The outputs must be passed in; nothing is allocated by this call."""
    T, d = x.shape
    E = wg.shape[0]
    _need(x, torch.bfloat16, (T, d), "x")
    _need(wg, torch.float32, (E, d), "wg")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    _need(topk_ids, torch.int32, (T, k), "topk_ids")
    _need(topk_w, torch.float32, (T, k), "topk_w")
    if expert_counts is not None:
        _need(expert_counts, torch.int32, (E,), "expert_counts")
    st = load_library().mk_moe_route_noalloc(_p(x), _p(wg), _p(bias), T, d, E, k, _p(topk_ids), _p(topk_w),
                                             _p(expert_counts), _stream(stream))
    _check(st, "mk_moe_route_noalloc")
    return topk_ids, topk_w, expert_counts


def mk_moe_dispatch(x, topk_ids, topk_w, E, ws=None, stream=None, out=None):
    """Dispatch: returns dict(expert_offsets, row_token, row_weight, slot_row, x_perm)."""
    T, d = x.shape
    k = topk_ids.shape[1]
    _need(x, torch.bfloat16, (T, d), "x")
    _need(topk_ids, torch.int32, (T, k), "topk_ids")
    if topk_w is not None:
        _need(topk_w, torch.float32, (T, k), "topk_w")
    dev = x.device
    o = out or {}
    res = {
        "expert_offsets": o.get("expert_offsets", torch.empty(E + 1, dtype=torch.int32, device=dev)),
        "row_token": o.get("row_token", torch.empty(T * k, dtype=torch.int32, device=dev)),
        "row_weight": o.get("row_weight", torch.empty(T * k, dtype=torch.float32, device=dev)),
        "slot_row": o.get("slot_row", torch.empty((T, k), dtype=torch.int32, device=dev)),
        "x_perm": o.get("x_perm", torch.empty((T * k, d), dtype=torch.bfloat16, device=dev)),
    }
    ws = alloc_workspace(T, d, E, k, 64, dev) if ws is None else ws
    st = load_library().mk_moe_dispatch(_p(x), _p(topk_ids), _p(topk_w), T, d, E, k, _p(res["expert_offsets"]),
                                        _p(res["row_token"]), _p(res["row_weight"]), _p(res["slot_row"]),
                                        _p(res["x_perm"]), _p(ws), ws.numel(), _stream(stream))
    _check(st, "mk_moe_dispatch")
    return res


def mk_moe_expert_ffn(x_perm, expert_offsets, row_weight, w1, w3, w2, h=None, P=None, ws=None, stream=None):
    """Grouped expert FFN on dispatched rows: returns (h [S,ffn] bf16, P [S,d] bf16)."""
    S, d = x_perm.shape
    E, f, _ = w1.shape
    _need(x_perm, torch.bfloat16, (S, d), "x_perm")
    _need(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    if row_weight is not None:
        _need(row_weight, torch.float32, (S,), "row_weight")
    _need(w1, torch.bfloat16, (E, f, d), "w1")
    _need(w3, torch.bfloat16, (E, f, d), "w3")
    _need(w2, torch.bfloat16, (E, d, f), "w2")
    dev = x_perm.device
    h = torch.empty((S, f), dtype=torch.bfloat16, device=dev) if h is None else h
    P = torch.empty((S, d), dtype=torch.bfloat16, device=dev) if P is None else P
    ws = torch.empty(256 + 4 * (E + 1), dtype=torch.uint8, device=dev) if ws is None else ws
    st = load_library().mk_moe_expert_ffn(_p(x_perm), _p(expert_offsets), _p(row_weight), _p(w1), _p(w3), _p(w2),
                                          S, d, E, f, _p(h), _p(P), _p(ws), ws.numel(), _stream(stream))
    _check(st, "mk_moe_expert_ffn")
    return h, P


def mk_moe_grouped_gemm(x_perm, expert_offsets, w, row_weight=None, out=None, ws=None, stream=None):
    """Grouped GEMM on dispatched rows: out[r] = row_weight[r] * x_perm[r] @ w[e].T for the
    rows r of expert e (row_weight None = 1); returns out [S, n] bf16."""
    S, d = x_perm.shape
    E, n, _ = w.shape
    _need(x_perm, torch.bfloat16, (S, d), "x_perm")
    _need(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _need(w, torch.bfloat16, (E, n, d), "w")
    if row_weight is not None:
        _need(row_weight, torch.float32, (S,), "row_weight")
    dev = x_perm.device
    out = torch.empty((S, n), dtype=torch.bfloat16, device=dev) if out is None else out
    _need(out, torch.bfloat16, (S, n), "out")
    ws = torch.empty(256 + 4 * (E + 1), dtype=torch.uint8, device=dev) if ws is None else ws
    st = load_library().mk_moe_grouped_gemm(_p(x_perm), _p(expert_offsets), _p(row_weight), _p(w), S, d, E, n,
                                            _p(out), _p(ws), ws.numel(), _stream(stream))
    _check(st, "mk_moe_grouped_gemm")
    return out


def dispatch_gemm_workspace_size(T: int, d: int, E: int, k: int) -> int:
    return int(load_library().mk_moe_dispatch_gemm_workspace_size(T, d, E, k))


def alloc_dispatch_gemm_workspace(T: int, d: int, E: int, k: int, device="cuda") -> torch.Tensor:
    n = dispatch_gemm_workspace_size(T, d, E, k)
    if n == 0:
        raise ValueError("invalid sizes for Dispatch + GEMM")
    return torch.empty(n, dtype=torch.uint8, device=device)


def mk_moe_dispatch_gemm(x, wg, bias, w, k, out=None, ws=None, stream=None, row_weight=True):
    """MoE Dispatch + GEMM: route, dispatch, and each expert's GEMM on its rows.

    Returns dict(out [T*k, n] bf16 rows grouped by expert, expert_offsets [E+1],
    row_token [T*k], row_weight [T*k] fp32 or None when row_weight=False)."""
    T, d = x.shape
    E, n, _ = w.shape
    _need(x, torch.bfloat16, (T, d), "x")
    _need(wg, torch.float32, (E, d), "wg")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    _need(w, torch.bfloat16, (E, n, d), "w")
    dev = x.device
    o = out or {}
    res = {
        "out": o.get("out", torch.empty((T * k, n), dtype=torch.bfloat16, device=dev)),
        "expert_offsets": o.get("expert_offsets", torch.empty(E + 1, dtype=torch.int32, device=dev)),
        "row_token": o.get("row_token", torch.empty(T * k, dtype=torch.int32, device=dev)),
        "row_weight": (o.get("row_weight", torch.empty(T * k, dtype=torch.float32, device=dev))
                       if row_weight else None),
    }
    _need(res["out"], torch.bfloat16, (T * k, n), "out")
    ws = alloc_dispatch_gemm_workspace(T, d, E, k, dev) if ws is None else ws
    st = load_library().mk_moe_dispatch_gemm(_p(x), _p(wg), _p(bias), _p(w), T, d, E, k, n, _p(res["out"]),
                                             _p(res["expert_offsets"]), _p(res["row_token"]), _p(res["row_weight"]),
                                             _p(ws), ws.numel(), _stream(stream))
    _check(st, "mk_moe_dispatch_gemm")
    return res


def mk_moe_combine(P, slot_row, y=None, stream=None):
    """Combine: y[t] = sum_j P[slot_row[t, j]] (fp32, ascending j) -> bf16 [T, d]."""
    T, k = slot_row.shape
    d = P.shape[1]
    _need(P, torch.bfloat16, (T * k, d), "P")
    _need(slot_row, torch.int32, (T, k), "slot_row")
    y = torch.empty((T, d), dtype=torch.bfloat16, device=P.device) if y is None else y
    st = load_library().mk_moe_combine(_p(P), _p(slot_row), T, d, k, _p(y), _stream(stream))
    _check(st, "mk_moe_combine")
    return y


def _opts(phase_events, timeout_ns, inject=0, path=MK_PATH_STEPS, mover_ctas=0, trace=None, gather_rows=False):
    if (phase_events is None and not timeout_ns and not inject and path == MK_PATH_STEPS and mover_ctas == 0
            and trace is None and not gather_rows):
        return None
    o = MkMoeOpts()
    o.gather_rows = 1 if gather_rows else 0
    if trace is not None:
        if trace.dtype != torch.int32 or trace.dim() != 2 or trace.shape[1] != 8 or not trace.is_cuda:
            raise ValueError("trace must be a CUDA int32 tensor of shape [records, 8]")
        o.trace = trace.data_ptr()
        o.trace_cap = trace.shape[0]
    o.timeout_ns = int(timeout_ns or 0)
    o.inject = int(inject)
    o.path = int(path)
    o.mover_ctas = int(mover_ctas)
    if phase_events is not None:
        if len(phase_events) != len(PHASES) + 1:
            raise ValueError(f"phase_events needs {len(PHASES) + 1} events")
        arr = (ctypes.c_void_p * len(phase_events))(*[ctypes.c_void_p(e.cuda_event) for e in phase_events])
        o._keep = arr
        o.phase_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    return ctypes.pointer(o)


def _layer_shapes(x, wg, bias, w1, w3, w2, device=True):
    T, d = x.shape
    E, f, _ = w1.shape
    _need(x, torch.bfloat16, (T, d), "x", device=device)
    _need(wg, torch.float32, (E, d), "wg")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    _need(w1, torch.bfloat16, (E, f, d), "w1")
    _need(w3, torch.bfloat16, (E, f, d), "w3")
    _need(w2, torch.bfloat16, (E, d, f), "w2")
    return T, d, E, f


def mk_moe_layer(x, wg, bias, w1, w3, w2, k, y=None, ws=None, phase_events=None, timeout_ns=0, stream=None,
                 inject=0, path=MK_PATH_STEPS, mover_ctas=0, trace=None, gather_rows=False):
    """The whole layer on device tensors; returns y [T, d] bf16.

    path: MK_PATH_STEPS (one kernel per step, default), MK_PATH_FUSED (one
    persistent kernel) or MK_PATH_TILES (one kernel per step, launched as
    programmatic dependents and synchronised per tile by data-tile
    semaphores).  mover_ctas: fused-path SM split, 0 = adaptive.  gather_rows:
    kernel-per-step path, gemm1 gathers its rows from x (no dispatched copy)."""
    T, d, E, f = _layer_shapes(x, wg, bias, w1, w3, w2)
    y = torch.empty((T, d), dtype=torch.bfloat16, device=x.device) if y is None else y
    ws = alloc_workspace(T, d, E, k, f, x.device) if ws is None else ws
    st = load_library().mk_moe_layer(_p(x), _p(wg), _p(bias), _p(w1), _p(w3), _p(w2), T, d, E, k, f, _p(y), _p(ws),
                                     ws.numel(),
                                     _opts(phase_events, timeout_ns, inject, path, mover_ctas, trace, gather_rows),
                                     _stream(stream))
    _check(st, "mk_moe_layer")
    return y


def mk_moe_layer_host(x_host, wg, bias, w1, w3, w2, k, y_host, ws, phase_events=None, timeout_ns=0, stream=None,
                      path=MK_PATH_STEPS, mover_ctas=0, gather_rows=False):
    """The layer on host buffers (pinned for asynchronous copies): x_host in, y_host out."""
    T, d, E, f = _layer_shapes(x_host, wg, bias, w1, w3, w2, device=False)
    _need(y_host, torch.bfloat16, (T, d), "y_host", device=False)
    st = load_library().mk_moe_layer_host(_p(x_host), _p(wg), _p(bias), _p(w1), _p(w3), _p(w2), T, d, E, k, f,
                                          _p(y_host), _p(ws), ws.numel(),
                                          _opts(phase_events, timeout_ns, 0, path, mover_ctas,
                                                gather_rows=gather_rows), _stream(stream))
    _check(st, "mk_moe_layer_host")
    return y_host


def mk_moe_layer_host_async(x_host, wg, bias, w1, w3, w2, k, y_host, ws, y_ready, phase_events=None, timeout_ns=0,
                            stream=None, path=MK_PATH_STEPS, mover_ctas=0, gather_rows=False):
    """The layer on host buffers with y's download off `stream`: y_ready (a
    torch.cuda.Event) is recorded once y_host holds the output; wait for it
    before reading y_host."""
    T, d, E, f = _layer_shapes(x_host, wg, bias, w1, w3, w2, device=False)
    _need(y_host, torch.bfloat16, (T, d), "y_host", device=False)
    s = torch.cuda.current_stream() if stream is None else stream
    if y_ready.cuda_event == 0:  # torch creates the event on its first record
        y_ready.record(s)
    st = load_library().mk_moe_layer_host_async(_p(x_host), _p(wg), _p(bias), _p(w1), _p(w3), _p(w2), T, d, E, k,
                                                f, _p(y_host), _p(ws), ws.numel(),
                                                _opts(phase_events, timeout_ns, 0, path, mover_ctas, gather_rows=gather_rows),
                                                ctypes.c_void_p(s.cuda_stream), ctypes.c_void_p(y_ready.cuda_event))
    _check(st, "mk_moe_layer_host_async")
    return y_host


def mk_moe_last_device_error(ws, stream=None):
    """(status, site) of the device-side errors of the last call on ws (synchronises)."""
    detail = ctypes.c_uint32(0)
    st = load_library().mk_moe_last_device_error(_p(ws), _stream(stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def mk_moe_route_fallbacks(ws, stream=None):
    """Tokens of the last router run on ws whose logits all took the fixed-order
    fallback (the candidate filter's bound did not hold; synchronises)."""
    n = ctypes.c_uint32(0)
    _check(load_library().mk_moe_route_fallbacks(_p(ws), _stream(stream), ctypes.byref(n)), "mk_moe_route_fallbacks")
    return int(n.value)


def mk_moe_route_approx_logits(ws, T, d, E, k, stream=None):
    """The approximate logits [T, E] fp32 the last candidate-filter router run on ws left there."""
    out = torch.empty((T, E), dtype=torch.float32, device=ws.device)
    _check(load_library().mk_moe_route_approx_logits(_p(ws), T, d, E, k, _p(out), _stream(stream)),
           "mk_moe_route_approx_logits")
    return out


def mk_moe_layer_trace_count(ws, T, d, E, k, ffn, stream=None):
    """Number of task records the last fused layer call on ws wrote (synchronises)."""
    n = ctypes.c_uint32(0)
    _check(load_library().mk_moe_layer_trace_count(_p(ws), T, d, E, k, ffn, _stream(stream), ctypes.byref(n)),
           "mk_moe_layer_trace_count")
    return int(n.value)


TRACE_KINDS = {2: "route", 3: "dispatch", 5: "combine", 6: "gemm"}


def mk_moe_layer_routing(ws, T, d, E, k, ffn, stream=None):
    """Routing tables the last mk_moe_layer call left in ws: (ids, w, offsets, slot_row)."""
    dev = ws.device
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    slot = torch.empty((T, k), dtype=torch.int32, device=dev)
    st = load_library().mk_moe_layer_routing(_p(ws), T, d, E, k, ffn, _p(ids), _p(w), _p(off), _p(slot),
                                             _stream(stream))
    _check(st, "mk_moe_layer_routing")
    return ids, w, off, slot


# Workspace regions (mk_ws_region): name -> (id, dtype, shape(T, d, E, k, ffn))
WS_REGIONS = {
    "ids": (0, torch.int32, lambda T, d, E, k, f: (T, k)),
    "w": (1, torch.float32, lambda T, d, E, k, f: (T, k)),
    "offsets": (2, torch.int32, lambda T, d, E, k, f: (E + 1,)),
    "row_token": (3, torch.int32, lambda T, d, E, k, f: (T * k,)),
    "row_weight": (4, torch.float32, lambda T, d, E, k, f: (T * k,)),
    "slot_row": (5, torch.int32, lambda T, d, E, k, f: (T, k)),
    "x_perm": (6, torch.bfloat16, lambda T, d, E, k, f: (T * k, d)),
    "h": (7, torch.bfloat16, lambda T, d, E, k, f: (T * k, f)),
    "P": (8, torch.bfloat16, lambda T, d, E, k, f: (T * k, d)),
}


def mk_moe_workspace_region(T, d, E, k, ffn, region):
    """(offset, bytes) of a workspace region (host arithmetic, no GPU call)."""
    rid = WS_REGIONS[region][0] if isinstance(region, str) else int(region)
    off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(load_library().mk_moe_workspace_region(T, d, E, k, ffn, rid, ctypes.byref(off), ctypes.byref(nb)),
           "mk_moe_workspace_region")
    return int(off.value), int(nb.value)


def workspace_view(ws, T, d, E, k, ffn, region):
    """A typed view (no copy) of a region the last mk_moe_layer call on ws filled."""
    _, dtype, shape = WS_REGIONS[region]
    off, nb = mk_moe_workspace_region(T, d, E, k, ffn, region)
    return ws[off:off + nb].view(dtype).view(shape(T, d, E, k, ffn))


def mk_moe_ep_regroup(rows_in, counts, to_expert_major, rows_out=None, expert_offsets=None, ws=None, stream=None):
    """Rows between source-major [q][e][rows] and expert-major [e][q][rows]
    order (expert parallelism).  counts: int32 [G, E_local] on the device;
    expert_offsets: optional int32 [E_local + 1] output (expert-major starts)."""
    import math

    G, El = counts.shape
    _need(counts, torch.int32, (G, El), "counts")
    if not rows_in.is_contiguous() or not rows_in.is_cuda:
        raise ValueError("rows_in must be a contiguous CUDA tensor")
    rows = rows_in.shape[0]
    row_bytes = math.prod(rows_in.shape[1:]) * rows_in.element_size()
    rows_out = torch.empty_like(rows_in) if rows_out is None else rows_out
    if expert_offsets is not None:
        _need(expert_offsets, torch.int32, (El + 1,), "expert_offsets")
    if ws is None:
        n = int(load_library().mk_moe_ep_regroup_workspace_size(G, El))
        if n == 0:
            raise ValueError("invalid G, E_local for the regroup")
        ws = torch.empty(n, dtype=torch.uint8, device=rows_in.device)
    st = load_library().mk_moe_ep_regroup(_p(rows_in), _p(rows_out), _p(counts), G, El, rows, row_bytes,
                                          1 if to_expert_major else 0, _p(expert_offsets), _p(ws), ws.numel(),
                                          _stream(stream))
    _check(st, "mk_moe_ep_regroup")
    return rows_out
