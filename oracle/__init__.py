"""CPU oracle for the MoE dispatch -> FFN -> combine layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``dispatch_ffn_combine_gb300``) never does and shares no code
with it; the two meet only through the seeded input generators, which hold
none of the layer's arithmetic.

The arithmetic lives in ``oracle.c`` (plain C, OpenMP over tokens); this module
builds it with gcc on first use and wraps it with numpy arrays.  The readings
of the pages it follows (router order R1, tie-break, slot order, row order,
SwiGLU convention) are stated at the top of ``oracle.c``.

Parity status of each function:
  router_logits      pinned (exact integer cases, hand-worked order cases,
                     fp64 error bound)
  topk               pinned (brute-force rank definition, ties, k=1, closed forms)
  dispatch           pinned (brute-force O(S^2) positions, invariants)
  expert_ffn / layer pinned (E=1,k=1 dense SwiGLU vs torch fp64, identical
                     experts, k=E full mixture, power-of-two scaling)
  expert_linear      pinned (torch fp64 matmul, permutation and power-of-two
                     expert matrices)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc); returns the path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _declare(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.oracle_num_threads.restype = I
    lib.oracle_set_num_threads.argtypes = [I]
    lib.oracle_router_logits.argtypes = [P, P, P, I64, I, I, P]
    lib.oracle_router_logits_f64.argtypes = [P, P, P, I64, I, I, P]
    lib.oracle_topk.argtypes = [P, I64, I, I, P, P]
    lib.oracle_dispatch.argtypes = [P, I64, I, I, P, P, P, P]
    lib.oracle_expert_ffn.argtypes = [P, P, P, P, I, I, P, P, I64, P]
    lib.oracle_layer.argtypes = [P, P, P, P, P, P, I64, I, I, I, I, P, I64, P, P, P]
    lib.oracle_expert_linear.argtypes = [P, P, I, I, P, P, I64, P]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def compile_variant(src_text: str, out_path: str) -> None:
    """Compile a modified copy of oracle.c (used only by the planted-mistake
    tests, which check that the pins catch plausible errors)."""
    src = out_path + ".c"
    with open(src, "w") as fh:
        fh.write(src_text)
    subprocess.run(["gcc", *CFLAGS, "-o", out_path, src, "-lm"], check=True)


def use_library(path):
    """Switch this module to another build of oracle.c; returns the previous
    handle so a test can restore it (``restore_library``)."""
    global _lib
    with _lock:
        prev = _lib
        _lib = _declare(ctypes.CDLL(path))
        return prev


def restore_library(handle) -> None:
    global _lib
    with _lock:
        _lib = handle


def source_text() -> str:
    with open(_SRC) as fh:
        return fh.read()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """bf16 data as its raw 16-bit patterns (numpy uint16, C-contiguous)."""
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 arrays are passed as uint16 bit patterns")
    return np.ascontiguousarray(a)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def router_logits(x_bits, wg, bias=None) -> np.ndarray:
    """fp32 gate logits [T, E] in the R1 order (see oracle.c)."""
    x_bits = _u16(x_bits)
    wg = _f32(wg)
    bias = _f32(bias)
    T, d = x_bits.shape
    E = wg.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    _load().oracle_router_logits(_ptr(x_bits), _ptr(wg), _ptr(bias), T, d, E, _ptr(out))
    return out


def router_logits_f64(x_bits, wg, bias=None) -> np.ndarray:
    x_bits = _u16(x_bits)
    wg = _f32(wg)
    bias = _f32(bias)
    T, d = x_bits.shape
    E = wg.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    _load().oracle_router_logits_f64(_ptr(x_bits), _ptr(wg), _ptr(bias), T, d, E, _ptr(out))
    return out


def topk(logits, k: int):
    """(ids [T,k] int32, weights [T,k] fp64) from fp32 logits [T,E]."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    _load().oracle_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w))
    return ids, w


def dispatch(ids, E: int):
    """(counts [E], offsets [E+1], row_token [T*k], slot_row [T,k]) from ids [T,k]."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    row_token = np.empty(T * k, dtype=np.int32)
    slot_row = np.empty((T, k), dtype=np.int32)
    _load().oracle_dispatch(_ptr(ids), T, E, k, _ptr(counts), _ptr(offsets), _ptr(row_token), _ptr(slot_row))
    return counts, offsets, row_token, slot_row


def expert_ffn(x_bits, w1_bits, w3_bits, w2_bits, tokens, experts) -> np.ndarray:
    """fp64 FFN_e(x_t) for each (tokens[p], experts[p]) pair -> [npairs, d]."""
    x_bits, w1_bits, w3_bits, w2_bits = map(_u16, (x_bits, w1_bits, w3_bits, w2_bits))
    d = x_bits.shape[1]
    f = w1_bits.shape[1]
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    experts = np.ascontiguousarray(experts, dtype=np.int32)
    out = np.empty((tokens.shape[0], d), dtype=np.float64)
    _load().oracle_expert_ffn(_ptr(x_bits), _ptr(w1_bits), _ptr(w3_bits), _ptr(w2_bits), d, f,
                              _ptr(tokens), _ptr(experts), tokens.shape[0], _ptr(out))
    return out


def expert_linear(x_bits, w_bits, tokens, experts) -> np.ndarray:
    """fp64 W_e x_t for each (tokens[p], experts[p]) pair -> [npairs, n]; w is [E, n, d]."""
    x_bits, w_bits = map(_u16, (x_bits, w_bits))
    d = x_bits.shape[1]
    n = w_bits.shape[1]
    if w_bits.shape[2] != d:
        raise ValueError("w must be [E, n, d]")
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    experts = np.ascontiguousarray(experts, dtype=np.int32)
    out = np.empty((tokens.shape[0], n), dtype=np.float64)
    _load().oracle_expert_linear(_ptr(x_bits), _ptr(w_bits), d, n, _ptr(tokens), _ptr(experts), tokens.shape[0],
                                 _ptr(out))
    return out


def dispatch_gemm(x_bits, wg, bias, w_bits, k: int):
    """MoE Dispatch + GEMM on all tokens: route (R1-R4), dispatch (R5), then each
    expert's linear map on its rows.  Returns (out [T*k, n] fp64 in dispatched row
    order, offsets [E+1], row_token [T*k], row_weight [T*k] fp64)."""
    x_bits = _u16(x_bits)
    E = np.asarray(wg).shape[0]
    ids, wts = topk(router_logits(x_bits, wg, bias), k)
    _, offsets, row_token, slot_row = dispatch(ids, E)
    row_expert = np.empty(row_token.shape[0], dtype=np.int32)
    row_weight = np.empty(row_token.shape[0], dtype=np.float64)
    row_expert[slot_row.ravel()] = ids.ravel()
    row_weight[slot_row.ravel()] = wts.ravel()
    out = expert_linear(x_bits, w_bits, row_token, row_expert)
    return out, offsets, row_token, row_weight


def layer(x_bits, wg, bias, w1_bits, w3_bits, w2_bits, k: int, tokens=None):
    """The full layer for the listed tokens (default: all).

    Returns (y [ntok, d] fp64, ids [ntok, k] int32, weights [ntok, k] fp64)."""
    x_bits, w1_bits, w3_bits, w2_bits = map(_u16, (x_bits, w1_bits, w3_bits, w2_bits))
    wg = _f32(wg)
    bias = _f32(bias)
    T, d = x_bits.shape
    E, f, _ = w1_bits.shape
    if not (1 <= k <= min(E, 64)):
        raise ValueError("k out of range")
    if tokens is None:
        tokens = np.arange(T, dtype=np.int64)
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    n = tokens.shape[0]
    y = np.empty((n, d), dtype=np.float64)
    ids = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k), dtype=np.float64)
    _load().oracle_layer(_ptr(x_bits), _ptr(wg), _ptr(bias), _ptr(w1_bits), _ptr(w3_bits), _ptr(w2_bits),
                         T, d, E, k, f, _ptr(tokens), n, _ptr(y), _ptr(ids), _ptr(w))
    return y, ids, w
