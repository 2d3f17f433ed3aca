"""CPU oracle for the W4A16 verify linear, the speculative accept step, and the
tree-masked verify attention with its KV compaction.

TEST INFRASTRUCTURE ONLY: imported by `tests/`, by `__graft_entry__.smoke()`
and by the benchmark's CPU-baseline leg, never by the library. It is plain C
(`w4a16_oracle.c`, fp64 arithmetic) behind ctypes, and shares no code with the
CUDA path. Every function states the page passage it follows in the C file.

Parity pins: every function here is pinned by `tests/test_oracle_pins.py`
against closed forms, library routines, brute force and the pages' worked
example. One convention is pinned only by its distributional property: the
extra token drawn from the (K+1)-th target row when all K drafts are accepted
(pinned by the output-distribution test, not by a printed value).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(dt):
    return np.ctypeslib.ndpointer(dtype=dt, flags="C_CONTIGUOUS")


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            i64, i32 = ctypes.c_int64, ctypes.c_int
            L.oracle_bf16_round.argtypes = [ctypes.c_float]
            L.oracle_bf16_round.restype = ctypes.c_uint16
            L.oracle_bf16_round_f64.argtypes = [ctypes.c_double]
            L.oracle_bf16_round_f64.restype = ctypes.c_uint16
            L.oracle_f16_round.argtypes = [ctypes.c_float]
            L.oracle_f16_round.restype = ctypes.c_uint16
            L.oracle_unpack_codes.argtypes = [_P(np.uint32), i64, i64, _P(np.int8)]
            L.oracle_pack_codes.argtypes = [_P(np.int8), i64, i64, _P(np.uint32)]
            L.oracle_dequantize.argtypes = [_P(np.uint32), _P(np.uint16), i64, i64, _P(np.float32)]
            L.oracle_quantize.argtypes = [_P(np.float32), i64, i64, _P(np.uint32), _P(np.uint16)]
            L.oracle_linear.argtypes = [_P(np.uint16), i64, i64, _P(np.uint32), _P(np.uint16), i64,
                                        _P(np.uint16), ctypes.c_void_p]
            L.oracle_linear_cols.argtypes = [_P(np.uint16), i64, i64, _P(np.uint32), _P(np.uint16), i64,
                                             _P(np.int64), i64, _P(np.uint16), ctypes.c_void_p]
            L.oracle_spec_accept_seq.argtypes = [_P(np.float32), _P(np.float32), _P(np.int32), _P(np.float32),
                                                 i32, i32, i32, _P(np.int32), _P(np.int32), _P(np.float64),
                                                 _P(np.float64), _P(np.float64)]
            L.oracle_greedy_tree.argtypes = [_P(np.float32), _P(np.int32), _P(np.int32), i32, i32, i32,
                                             _P(np.int32), _P(np.int32), _P(np.int32)]
            L.oracle_spec_accept_tree.argtypes = [_P(np.float32), _P(np.float32), _P(np.int32), _P(np.int32),
                                                  _P(np.float32), i32, i32, i32, _P(np.int32), _P(np.int32),
                                                  _P(np.int32), _P(np.float64), _P(np.float64)]
            L.oracle_tree_attention.argtypes = [_P(np.uint16), _P(np.uint16), _P(np.uint16), _P(np.int32),
                                                ctypes.c_void_p, i32, i32, i32, i32, i32, i32, ctypes.c_double,
                                                _P(np.float64), ctypes.c_void_p]
            L.oracle_kv_compact.argtypes = [_P(np.uint16), _P(np.uint16), _P(np.int32), ctypes.c_void_p,
                                            _P(np.int32), i32, i32, i32, i32, i32, i32, _P(np.int32)]
            L.oracle_greedy_chain.argtypes = [_P(np.float32), _P(np.int32), i32, i32, i32, _P(np.int32),
                                              _P(np.int32)]
            L.oracle_num_threads.restype = ctypes.c_int
            L.oracle_set_num_threads.argtypes = [ctypes.c_int]
            L.oracle_set_num_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> int:
    """Threads of the oracle's parallel loops from now on; returns the count in effect."""
    return int(lib().oracle_set_num_threads(int(n)))


def bf16_round(f: float) -> int:
    return int(lib().oracle_bf16_round(float(f)))


def bf16_round_f64(v: float) -> int:
    """bf16 bits of a double, rounded to nearest even in one step."""
    return int(lib().oracle_bf16_round_f64(float(v)))


def f16_round(f: float) -> int:
    return int(lib().oracle_f16_round(float(f)))


def pack_codes(codes: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.int8)
    N, K = codes.shape
    out = np.empty((N, K // 8), dtype=np.uint32)
    lib().oracle_pack_codes(codes, N, K, out)
    return out


def unpack_codes(qweight: np.ndarray, K: int) -> np.ndarray:
    qweight = _c(qweight, np.uint32)
    N = qweight.shape[0]
    out = np.empty((N, K), dtype=np.int8)
    lib().oracle_unpack_codes(qweight, N, K, out)
    return out


def dequantize(qweight: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    qweight, scales = _c(qweight, np.uint32), _c(scales, np.uint16)
    N = qweight.shape[0]
    out = np.empty((N, K), dtype=np.float32)
    lib().oracle_dequantize(qweight, scales, N, K, out)
    return out


def quantize(w: np.ndarray):
    """w [N,K] float32 -> (qweight [N,K/8] uint32, scales [N,K/128] fp16 bits as uint16)."""
    w = _c(w, np.float32)
    N, K = w.shape
    qw = np.empty((N, K // 8), dtype=np.uint32)
    sc = np.empty((N, K // 128), dtype=np.uint16)
    lib().oracle_quantize(w, N, K, qw, sc)
    return qw, sc


def linear(x_bf16: np.ndarray, qweight: np.ndarray, scales: np.ndarray, want_y: bool = False):
    """out[M,N] bf16 bits = bf16(x . W^T); optional fp64 sums y[M,N]."""
    x_bf16, qweight, scales = _c(x_bf16, np.uint16), _c(qweight, np.uint32), _c(scales, np.uint16)
    M, K = x_bf16.shape
    N = qweight.shape[0]
    out = np.empty((M, N), dtype=np.uint16)
    y = np.empty((M, N), dtype=np.float64) if want_y else None
    lib().oracle_linear(x_bf16, M, K, qweight, scales, N, out, None if y is None else y.ctypes.data)
    return (out, y) if want_y else out


def linear_cols(x_bf16, qweight, scales, cols, want_y: bool = False):
    """out[M, len(cols)] for the chosen output columns only."""
    x_bf16, qweight, scales = _c(x_bf16, np.uint16), _c(qweight, np.uint32), _c(scales, np.uint16)
    cols = _c(cols, np.int64)
    M, K = x_bf16.shape
    N = qweight.shape[0]
    out = np.empty((M, len(cols)), dtype=np.uint16)
    y = np.empty((M, len(cols)), dtype=np.float64) if want_y else None
    lib().oracle_linear_cols(x_bf16, M, K, qweight, scales, N, cols, len(cols), out,
                             None if y is None else y.ctypes.data)
    return (out, y) if want_y else out


def spec_accept_seq(p, q, d, u):
    """Stochastic acceptance of a sequence draft. Returns
    (accepted_len[B], next_token[B], alpha[B,K], margin_alpha[B], margin_cdf[B]):
    margin_alpha = min |u_i - alpha_i| over the evaluated drafts, margin_cdf =
    distance of u*S from the nearer end of the drawn token's CDF interval, / S."""
    p, q, d, u = _c(p, np.float32), _c(q, np.float32), _c(d, np.int32), _c(u, np.float32)
    B, K1, V = p.shape
    K = K1 - 1
    assert q.shape == (B, K, V) and d.shape == (B, K) and u.shape == (B, K + 1)
    acc = np.empty(B, dtype=np.int32)
    nxt = np.empty(B, dtype=np.int32)
    alpha = np.empty((B, K), dtype=np.float64)
    margin_alpha = np.empty(B, dtype=np.float64)
    margin_cdf = np.empty(B, dtype=np.float64)
    lib().oracle_spec_accept_seq(p, q, d, u, B, K, V, acc, nxt, alpha, margin_alpha, margin_cdf)
    return acc, nxt, alpha, margin_alpha, margin_cdf


def greedy_tree(p, draft, parents, want_node: bool = False):
    """Greedy tree verification. p [B,n,V], draft [B,n], parents [B,n] (or [n]).
    Returns (accepted_len, next_token) and, with want_node, the deepest
    accepted node's index."""
    p, draft = _c(p, np.float32), _c(draft, np.int32)
    B, n, V = p.shape
    parents = _parents(parents, B, n)
    acc = np.empty(B, dtype=np.int32)
    nxt = np.empty(B, dtype=np.int32)
    node = np.empty(B, dtype=np.int32)
    lib().oracle_greedy_tree(p, draft, parents, B, n, V, acc, nxt, node)
    return (acc, nxt, node) if want_node else (acc, nxt)


def spec_accept_tree(p, q, d, parents, u):
    """Stochastic acceptance of a token tree (multi-step speculative
    sampling). p, q [B,n,V] logits at every node, d [B,n], parents [B,n] (or
    [n]), u [B,n] (u[:, j] tests node j, u[:, 0] draws the next token).
    Returns (accepted_len, next_token, accepted_node, margin_alpha, margin_cdf)."""
    p, q, d, u = _c(p, np.float32), _c(q, np.float32), _c(d, np.int32), _c(u, np.float32)
    B, n, V = p.shape
    assert q.shape == (B, n, V) and d.shape == (B, n) and u.shape == (B, n)
    par = _parents(parents, B, n)
    acc, nxt, node = (np.empty(B, dtype=np.int32) for _ in range(3))
    ma, mc = np.empty(B, dtype=np.float64), np.empty(B, dtype=np.float64)
    lib().oracle_spec_accept_tree(p, q, d, par, u, B, n, V, acc, nxt, node, ma, mc)
    return acc, nxt, node, ma, mc


def _parents(parents, B, n):
    parents = np.asarray(parents, dtype=np.int32)
    if parents.ndim == 1:
        parents = np.broadcast_to(parents, (B, n))
    return _c(parents, np.int32)


def tree_attention(q, k_cache, v_cache, lens, parents=None, scale=None, want_abs: bool = False):
    """Tree-masked attention of the verify pass. q bf16 bits [B,n,H,D];
    caches bf16 bits [B,Hkv,Lcap,D] holding the prefix at 0..lens-1 and the
    tree nodes at lens..lens+n-1; parents [B,n] / [n] or None (chain).
    Returns fp64 [B,n,H,D] (and, with want_abs, the softmax-weighted sum of
    |v|, same shape)."""
    q, k_cache, v_cache = _c(q, np.uint16), _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    B, n, H, D = q.shape
    _, Hkv, Lcap, _ = k_cache.shape
    lens = _c(lens, np.int32)
    assert k_cache.shape == v_cache.shape == (B, Hkv, Lcap, D) and lens.shape == (B,)
    assert int(lens.max()) + n <= Lcap and H % Hkv == 0
    par = None if parents is None else _parents(parents, B, n)
    out = np.empty((B, n, H, D), dtype=np.float64)
    absw = np.empty((B, n, H, D), dtype=np.float64) if want_abs else None
    lib().oracle_tree_attention(q, k_cache, v_cache, lens, None if par is None else par.ctypes.data, B, n, H, Hkv, D,
                                Lcap, float(D ** -0.5 if scale is None else scale), out,
                                None if absw is None else absw.ctypes.data)
    return (out, absw) if want_abs else out


def kv_compact(k_cache, v_cache, lens, parents, accepted_node):
    """Moves the accepted root path's keys/values to lens..lens+depth (copies;
    caches bf16 bits [layers,B,Hkv,Lcap,D]). Returns (k, v, new_lens)."""
    k = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    v = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    nl, B, Hkv, Lcap, D = k.shape
    node = _c(accepted_node, np.int32)
    lens = _c(lens, np.int32)
    n = int(np.asarray(parents).shape[-1]) if parents is not None else int(node.max()) + 1
    par = None if parents is None else _parents(parents, B, n)
    new_lens = np.empty(B, dtype=np.int32)
    lib().oracle_kv_compact(k, v, lens, None if par is None else par.ctypes.data, node, B, n, Hkv, D, Lcap, nl,
                            new_lens)
    return k, v, new_lens


def greedy_chain(p, draft):
    """Greedy sequence verification. p [B,K+1,V], draft [B,K]."""
    p, draft = _c(p, np.float32), _c(draft, np.int32)
    B, K1, V = p.shape
    acc = np.empty(B, dtype=np.int32)
    nxt = np.empty(B, dtype=np.int32)
    lib().oracle_greedy_chain(p, draft, B, K1 - 1, V, acc, nxt)
    return acc, nxt
