"""CPU oracle of the CSA2 decode path -- TEST INFRASTRUCTURE ONLY.

Only tests/, the smoke check (`__graft_entry__.smoke`) and the benchmark's
CPU-baseline / reference arm may import this package. The product path (the
`sparse_attention_fp4_mxfp4_gb300` package and its CUDA library) never does,
and this package never imports it.

Thin ctypes wrappers around oracle.cpp, which holds the arithmetic and cites
the pages it follows. All results are fp64 (formats are exact).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "_oracle.so")

THREADS = max(1, min(64, os.cpu_count() or 1))


def build(force: bool = False) -> str:
    """Compile oracle.cpp (IEEE arithmetic: no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                               _SRC, "-o", tmp, "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        alt = os.environ.get("CSA2_ORACLE_LIB")  # a deliberately mutated build, see tests
        if alt:
            L = ctypes.CDLL(alt)
        else:
            build()
            L = ctypes.CDLL(_LIB)
        i64, i32, p, d, f = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double, ctypes.c_float
        L.orc_e2m1_value.argtypes, L.orc_e2m1_value.restype = [i32], d
        L.orc_e4m3_value.argtypes, L.orc_e4m3_value.restype = [i32], d
        L.orc_e4m3_encode.argtypes, L.orc_e4m3_encode.restype = [f], i32
        L.orc_e4m3_encode_array.argtypes = [p, i64, p, i32]
        L.orc_mxfp4_quant.argtypes = [p, i64, p, p, i32]
        L.orc_mxfp4_dequant.argtypes = [p, p, i64, p]
        L.orc_fp8_quant.argtypes = [p, i64, p]
        L.orc_fp8_dequant.argtypes = [p, i64, p]
        L.orc_index_scores.argtypes = [p, p, i32, i32, p, i64, p, i32]
        L.orc_block_max.argtypes = [p, i64, i32, p]
        L.orc_topk.argtypes, L.orc_topk.restype = [p, i64, i64, p], i64
        L.orc_full_indexer.argtypes = [p, p, i32, i32, p, i64, i32, i64, i64, p, p, p, p, i32]
        L.orc_full_indexer.restype = i64
        L.orc_reindex.argtypes = [p, p, i32, i32, p, i64, i32, p, i64, i64, p, p, i32]
        L.orc_reindex.restype = i64
        L.orc_window_positions.argtypes, L.orc_window_positions.restype = [i64, i64, i64, p], i64
        L.orc_sparse_attention.argtypes = [p, i32, i32, p, i64, p, i64, d, p, p]
        L.orc_output_derotate.argtypes = [p, i64, i32, i64]
        L.orc_compress.argtypes = [p, p, i32, i32, i64, p]
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a) -> int:
    return a.ctypes.data if a is not None and a.size else 0


# ---- formats -----------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return lib().orc_e4m3_value(int(byte))


def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> E4M3 bytes (RNE, saturating to +-448)."""
    x = _c(x, np.float32).ravel()
    out = np.empty(x.size, np.uint8)
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(out), THREADS)
    return out


def mxfp4_quant(x):
    """fp32 values [..., n] (n % 16 == 0) -> (codes uint8 [..., n/2], scales uint8 [..., n/16])."""
    x = _c(x, np.float32)
    n = x.size
    assert n % 16 == 0
    codes = np.empty(n // 2, np.uint8)
    scales = np.empty(n // 16, np.uint8)
    lib().orc_mxfp4_quant(_p(x), n, _p(codes), _p(scales), THREADS)
    shp = x.shape[:-1]
    return codes.reshape(*shp, x.shape[-1] // 2), scales.reshape(*shp, x.shape[-1] // 16)


def mxfp4_dequant(codes, scales) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    n = codes.size * 2
    assert scales.size * 16 == n
    out = np.empty(n, np.float64)
    lib().orc_mxfp4_dequant(_p(codes), _p(scales), n, _p(out))
    return out.reshape(*codes.shape[:-1], codes.shape[-1] * 2)


def fp8_quant(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_fp8_quant(_p(x), x.size, _p(out))
    return out


def fp8_dequant(b) -> np.ndarray:
    b = _c(b, np.uint8)
    out = np.empty(b.shape, np.float64)
    lib().orc_fp8_dequant(_p(b), b.size, _p(out))
    return out


# ---- indexer -----------------------------------------------------------------

def index_scores(qhat, w, keys) -> np.ndarray:
    """qhat fp64 [H, D], w [H], keys fp64 [n, D] (already dequantised) -> fp64 [n]."""
    qhat = _c(qhat, np.float64)
    w = _c(w, np.float64)
    keys = _c(keys, np.float64)
    H, D = qhat.shape
    n = keys.shape[0]
    out = np.empty(n, np.float64)
    lib().orc_index_scores(_p(qhat), _p(w), H, D, _p(keys), n, _p(out), THREADS)
    return out


def block_max(s, block=8) -> np.ndarray:
    s = _c(s, np.float64)
    out = np.empty((s.size + block - 1) // block, np.float64)
    lib().orc_block_max(_p(s), s.size, block, _p(out))
    return out


def topk(s, k) -> np.ndarray:
    s = _c(s, np.float64)
    out = np.empty(min(k, s.size), np.int64)
    m = lib().orc_topk(_p(s), s.size, k, _p(out))
    return out[:m]


def full_indexer(qidx_bf16, w, keys_bf16, t, n_pool=2048, k=512, block=8, want_scores=True,
                 threads=None):
    """Full-mode indexer for one query at position t.

    qidx_bf16: uint16 [H, D]; w: fp32 [H]; keys_bf16: uint16 [>= t+1, D].
    Returns dict(scores fp64 [t+1] | None, blockmax fp64 [ceil((t+1)/block)],
    pool int32 [n_pool], topk int32 [k]) with -1 padding.
    """
    q = _c(qidx_bf16, np.uint16)
    w = _c(w, np.float32)
    keys = _c(keys_bf16, np.uint16)
    H, D = q.shape
    assert keys.shape[0] >= t + 1 and keys.shape[1] == D
    n = t + 1
    scores = np.empty(n, np.float64) if want_scores else None
    bm = np.empty((n + block - 1) // block, np.float64)
    pool = np.empty(n_pool, np.int32)
    tk = np.empty(k, np.int32)
    lib().orc_full_indexer(_p(q), _p(w), H, D, _p(keys), t, block, n_pool, k, _p(scores), _p(bm),
                           _p(pool), _p(tk), threads or THREADS)
    return dict(scores=scores, blockmax=bm, pool=pool, topk=tk)


def reindex(qidx_bf16, w, keys_bf16, t, pool, k=512, block=8, threads=None):
    """Reindex-mode indexer for one query at position t over a given pool.

    Returns dict(pos_scores fp64 [n_pool*block] (-inf off-pool/non-causal), topk int32 [k]).
    """
    q = _c(qidx_bf16, np.uint16)
    w = _c(w, np.float32)
    keys = _c(keys_bf16, np.uint16)
    pool = _c(pool, np.int32)
    H, D = q.shape
    ps = np.empty(pool.size * block, np.float64)
    tk = np.empty(k, np.int32)
    lib().orc_reindex(_p(q), _p(w), H, D, _p(keys), t, block, _p(pool), pool.size, k, _p(ps), _p(tk),
                      threads or THREADS)
    return dict(pos_scores=ps, topk=tk)


# ---- attention ---------------------------------------------------------------

def window_positions(t, n_ctx, window=128) -> np.ndarray:
    out = np.empty(window, np.int64)
    m = lib().orc_window_positions(t, n_ctx, window, _p(out))
    return out[:m]


def sparse_attention(q_bf16, main_rows_bf16, win_rows_bf16, tau):
    """One query: q uint16 [H, D]; raw bf16 rows of the selected main entries
    [n_main, D] and of the window entries [n_win, D]. Returns (out fp64 [H, D], lse fp64 [H])."""
    q = _c(q_bf16, np.uint16)
    H, D = q.shape
    mr = _c(main_rows_bf16, np.uint16).reshape(-1, D)
    wr = _c(win_rows_bf16, np.uint16).reshape(-1, D)
    out = np.empty((H, D), np.float64)
    lse = np.empty(H, np.float64)
    lib().orc_sparse_attention(_p(q), H, D, _p(mr), mr.shape[0], _p(wr), wr.shape[0], float(tau),
                               _p(out), _p(lse))
    return out, lse


def output_derotate(rows, t):
    """Rows fp64 [n, D] (or [D]) of attention output for query position t, with
    the last 64 channels rotated back by t (pairs 2i, 2i+1; see oracle.cpp)."""
    a = np.array(rows, dtype=np.float64, order="C", copy=True)
    D = a.shape[-1]
    lib().orc_output_derotate(_p(a), a.size // D, D, int(t))
    return a


# ---- compressed entries (encoder-side CSA2, m tokens per entry) ---------------

def compress(x_bf16, z_bf16):
    """x, z: uint16 (bf16 bits) [n, m, D] candidates and compression logits of
    each entry's m tokens. Returns uint16 [n, D]: per channel the softmax over
    the m tokens of z weighting x, in fp64, rounded once to bf16."""
    x = _c(x_bf16, np.uint16)
    z = _c(z_bf16, np.uint16)
    assert x.shape == z.shape and x.ndim == 3
    n, m, D = x.shape
    out = np.empty((n, D), np.uint16)
    lib().orc_compress(_p(x), _p(z), m, D, n, _p(out))
    return out


def entry_limit(t, m):
    """Complete entries visible to a token at position t: floor((t + 1) / m)."""
    return (t + 1) // m
