"""Python binding of libcsa2.so, the GB300 (sm_103a) CSA2 decode hot path.

Argument marshalling only: every step runs in the CUDA library. Functions
carry the C ABI's names (include/csa2.h documents arguments, layouts and
errors) and take torch tensors; device pointers, sizes and the current CUDA
stream are passed through. A failing call raises Csa2Error with the library's
message. There is no CPU fallback: importing this package fails loudly when
the library has not been built.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

# Constants of include/csa2.h.
(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_DEVICE_BOUNDS,
 ERR_DEVICE_RANGE) = range(8)
LATENT_DIM, Q_HEADS, IDX_HEADS, IDX_DIM = 512, 64, 32, 128
TOPK, POOL_BLOCKS, BLOCK, WINDOW, PAGE_TOKENS = 512, 2048, 8, 128, 128
MAIN_ENTRY_BYTES, IDX_ENTRY_BYTES, MAX_NQ = 288, 72, 8
MAX_PREFILL_NQ, MAX_TOKENS = 4096, 65535
PLANE_MAIN, PLANE_INDEX = 0, 1
OUT_F32, OUT_BF16 = 0, 1
OUT_DEROTATE = 0x100  # OR'ed into out_dtype: rotate the output back by the query position
MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2
OP_INDEXER_FULL, OP_INDEXER_REINDEX, OP_SPARSE_ATTN, OP_DECODE_LAYER = 1, 2, 3, 4

# Exported entry points of include/csa2.h.
EXPORTS = (
    "csa2_status_string", "csa2_last_error", "csa2_version", "csa2_page_bytes", "csa2_ring_bytes",
    "csa2_workspace_bytes", "csa2_append_kv", "csa2_decode_appends", "csa2_compress_append", "csa2_append_swa", "csa2_quant_fp8_entries",
    "csa2_ring_refill", "csa2_quant_mxfp4",
    "csa2_dequant_mxfp4", "csa2_quant_fp8", "csa2_indexer_scan", "csa2_block_topk",
    "csa2_indexer_reindex", "csa2_indexer_reindex_noalloc", "csa2_indexer_full", "csa2_sparse_attn", "csa2_sparse_attn_prefill", "csa2_decode_layer",
    "csa2_decode_group", "csa2_check_device_status", "csa2_debug_force_wait_timeout",
)


class Csa2Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"csa2 status {status}: {msg}")
        self.status = status


class AppendLayer(ctypes.Structure):
    """csa2_append_layer of include/csa2.h."""
    _fields_ = [
        ("swa", ctypes.c_void_p), ("ring_idx", ctypes.c_void_p), ("n_rings", ctypes.c_int64),
        ("rings", ctypes.c_void_p), ("q_idx", ctypes.c_void_p), ("q_n", ctypes.c_int64),
        ("q_codes", ctypes.c_void_p), ("q_scales", ctypes.c_void_p),
    ]


class LayerArgs(ctypes.Structure):
    """csa2_layer_args of include/csa2.h."""
    _fields_ = [
        ("mode", ctypes.c_int), ("B", ctypes.c_int), ("n_q", ctypes.c_int),
        ("max_ctx", ctypes.c_int64), ("seq_len", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
        ("max_pages", ctypes.c_int), ("n_pages", ctypes.c_int64), ("main_pages", ctypes.c_void_p),
        ("idx_pages", ctypes.c_void_p), ("rings", ctypes.c_void_p), ("ring_idx", ctypes.c_void_p),
        ("n_rings", ctypes.c_int64), ("q_idx_codes", ctypes.c_void_p), ("q_idx_scales", ctypes.c_void_p),
        ("w", ctypes.c_void_p), ("q", ctypes.c_void_p), ("pool", ctypes.c_void_p), ("topk", ctypes.c_void_p),
        ("softmax_scale", ctypes.c_float), ("out_dtype", ctypes.c_int), ("out", ctypes.c_void_p),
        ("lse", ctypes.c_void_p), ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t),
        ("swa_chunk", ctypes.c_void_p), ("tokens_per_entry", ctypes.c_int),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    p, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    psz = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "csa2_status_string": ([i32], ctypes.c_char_p),
        "csa2_last_error": ([], ctypes.c_char_p),
        "csa2_version": ([], i32),
        "csa2_page_bytes": ([i32, psz], i32),
        "csa2_ring_bytes": ([psz], i32),
        "csa2_workspace_bytes": ([i32, i32, i32, i64, psz], i32),
        "csa2_append_kv": ([p, p, p, p, i32, p, i32, i32, i64, p, p, p], i32),
        "csa2_decode_appends": ([p, p, p, p, i32, p, i32, i32, i64, p, p, p, i32, p], i32),
        "csa2_compress_append": ([p, p, p, p, p, p, i32, i32, p, p, i32, i32, i64, p, p, p], i32),
        "csa2_append_swa": ([p, p, p, i32, i64, p, p], i32),
        "csa2_quant_fp8_entries": ([p, i32, p, p], i32),
        "csa2_ring_refill": ([p, p, i32, i32, p, i64, p, p], i32),
        "csa2_quant_mxfp4": ([p, i64, p, p, p], i32),
        "csa2_dequant_mxfp4": ([p, p, i64, p, p], i32),
        "csa2_quant_fp8": ([p, i64, p, p], i32),
        "csa2_indexer_scan": ([p, p, p, p, i32, i32, i64, p, i32, i64, p, p, i64, i32, p], i32),
        "csa2_block_topk": ([p, p, i32, i32, i64, p, i32, p], i32),
        "csa2_indexer_reindex": ([p, p, p, p, i32, i32, p, i32, i64, p, p, p, p, sz, i32, p], i32),
        "csa2_indexer_reindex_noalloc": ([p, p, p, p, i32, i32, p, i32, i64, p, p, p, i32, p], i32),
        "csa2_indexer_full": ([p, p, p, p, i32, i32, i64, p, i32, i64, p, p, p, p, sz, i32, p], i32),
        "csa2_sparse_attn": ([p, p, p, i32, i32, p, i32, i64, p, p, p, i64, f32, i32, p, p, p, sz, i32, p], i32),
        "csa2_sparse_attn_prefill": ([p, p, p, i32, i32, p, i32, i64, p, p, p, i64, p, f32, i32, p, p, p, sz, i32,
                                      p], i32),
        "csa2_decode_layer": ([ctypes.POINTER(LayerArgs), p], i32),
        "csa2_decode_group": ([ctypes.POINTER(LayerArgs), i32, p], i32),
        "csa2_check_device_status": ([p, ctypes.POINTER(ctypes.c_int)], i32),
        "csa2_debug_force_wait_timeout": ([i32, p], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes, fn.restype = args, res
    return L


lib = _load()


def _check(status: int):
    if status != OK:
        raise Csa2Error(status, lib.csa2_last_error().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtype, ndim=None):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: {t.dim()} dims, expected {ndim}")


# ---- size queries -------------------------------------------------------------

def csa2_page_bytes(plane: int) -> int:
    n = ctypes.c_size_t()
    _check(lib.csa2_page_bytes(plane, ctypes.byref(n)))
    return n.value


def csa2_ring_bytes() -> int:
    n = ctypes.c_size_t()
    _check(lib.csa2_ring_bytes(ctypes.byref(n)))
    return n.value


def csa2_workspace_bytes(op: int, B: int, n_q: int, max_ctx: int) -> int:
    n = ctypes.c_size_t()
    _check(lib.csa2_workspace_bytes(op, B, n_q, max_ctx, ctypes.byref(n)))
    return n.value


# ---- append -------------------------------------------------------------------

def csa2_append_kv(latent, idx_key, seq_idx, pos, block_table, main_pages, idx_pages, stream=None):
    """latent bf16 [T,512], idx_key bf16 [T,128], seq_idx int32 [T], pos int64 [T],
    block_table int32 [B,max_pages], main_pages uint8 [P,36864], idx_pages uint8 [P,9216]."""
    _need(latent, "latent", torch.bfloat16, 2)
    _need(idx_key, "idx_key", torch.bfloat16, 2)
    _need(seq_idx, "seq_idx", torch.int32, 1)
    _need(pos, "pos", torch.int64, 1)
    _need(block_table, "block_table", torch.int32, 2)
    T = latent.shape[0]
    if latent.shape[1] != LATENT_DIM or idx_key.shape != (T, IDX_DIM) or seq_idx.numel() != T or pos.numel() != T:
        raise ValueError("append_kv: inconsistent shapes")
    _check(lib.csa2_append_kv(_ptr(latent), _ptr(idx_key), _ptr(seq_idx), _ptr(pos), T, _ptr(block_table),
                              block_table.shape[0], block_table.shape[1], main_pages.shape[0],
                              _ptr(main_pages), _ptr(idx_pages), _stream(stream)))


def csa2_decode_appends(latent, idx_key, seq_idx, pos, block_table, main_pages, idx_pages, layers, stream=None):
    """One launch for a decode step's stores and query quantisations: csa2_append_kv(latent, idx_key, seq_idx,
    pos, ...) and, per entry of `layers` (dicts with optional keys swa, ring_idx, rings and q_idx, q_codes,
    q_scales), csa2_append_swa(swa, ring_idx, pos, rings) and csa2_quant_mxfp4(q_idx, q_codes, q_scales)."""
    _need(latent, "latent", torch.bfloat16, 2)
    _need(idx_key, "idx_key", torch.bfloat16, 2)
    _need(seq_idx, "seq_idx", torch.int32, 1)
    _need(pos, "pos", torch.int64, 1)
    _need(block_table, "block_table", torch.int32, 2)
    T = latent.shape[0]
    if latent.shape[1] != LATENT_DIM or idx_key.shape != (T, IDX_DIM) or seq_idx.numel() != T or pos.numel() != T:
        raise ValueError("decode_appends: inconsistent shapes")
    arr = (AppendLayer * max(1, len(layers)))()
    for a, L in zip(arr, layers):
        swa, q_idx = L.get("swa"), L.get("q_idx")
        if swa is not None:
            _need(swa, "swa", torch.bfloat16, 2)
            _need(L["ring_idx"], "ring_idx", torch.int32, 1)
            if swa.shape != (T, LATENT_DIM) or L["ring_idx"].numel() != T:
                raise ValueError("decode_appends: inconsistent window shapes")
            a.swa, a.ring_idx, a.n_rings, a.rings = _ptr(swa), _ptr(L["ring_idx"]), L["rings"].shape[0], _ptr(L["rings"])
        if q_idx is not None:
            _need(q_idx, "q_idx", torch.bfloat16)
            n = q_idx.numel()
            if L["q_codes"].numel() != n // 2 or L["q_scales"].numel() != n // 16:
                raise ValueError("decode_appends: inconsistent query code shapes")
            a.q_idx, a.q_n, a.q_codes, a.q_scales = _ptr(q_idx), n, _ptr(L["q_codes"]), _ptr(L["q_scales"])
    _check(lib.csa2_decode_appends(_ptr(latent), _ptr(idx_key), _ptr(seq_idx), _ptr(pos), T, _ptr(block_table),
                                   block_table.shape[0], block_table.shape[1], main_pages.shape[0], _ptr(main_pages),
                                   _ptr(idx_pages), ctypes.cast(arr, ctypes.c_void_p), len(layers), _stream(stream)))


def csa2_compress_append(kv, kv_gate, idx_key, idx_gate, seq_idx, pos, m, tail, block_table, main_pages, idx_pages,
                         stream=None):
    """Encoder-side append at m tokens per entry: kv, kv_gate bf16 [T,512], idx_key, idx_gate bf16 [T,128],
    seq_idx int32 [T], pos int64 [T] (each sequence's rows consecutive positions), tail bf16 [B,m-1,1280]
    (None for m = 1). Entries go to the pages at entry e = pos // m."""
    for t, n in ((kv, "kv"), (kv_gate, "kv_gate"), (idx_key, "idx_key"), (idx_gate, "idx_gate")):
        _need(t, n, torch.bfloat16, 2)
    _need(seq_idx, "seq_idx", torch.int32, 1)
    _need(pos, "pos", torch.int64, 1)
    T = kv.shape[0]
    _check(lib.csa2_compress_append(_ptr(kv), _ptr(kv_gate), _ptr(idx_key), _ptr(idx_gate), _ptr(seq_idx), _ptr(pos),
                                    T, m, _ptr(tail), _ptr(block_table), block_table.shape[0], block_table.shape[1],
                                    main_pages.shape[0], _ptr(main_pages), _ptr(idx_pages), _stream(stream)))


def csa2_append_swa(x, ring_idx, pos, rings, stream=None):
    """x bf16 [T,512], ring_idx int32 [T], pos int64 [T], rings uint8 [R,128,512]."""
    _need(x, "x", torch.bfloat16, 2)
    _need(ring_idx, "ring_idx", torch.int32, 1)
    _need(pos, "pos", torch.int64, 1)
    T = x.shape[0]
    _check(lib.csa2_append_swa(_ptr(x), _ptr(ring_idx), _ptr(pos), T, rings.shape[0], _ptr(rings),
                               _stream(stream)))


def csa2_quant_fp8_entries(x, out=None, stream=None):
    """x bf16 [T,512] -> E4M3 uint8 [T,512] (a prefill chunk's own window entries)."""
    _need(x, "x", torch.bfloat16, 2)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib.csa2_quant_fp8_entries(_ptr(x), x.shape[0], _ptr(out), _stream(stream)))
    return out


def csa2_ring_refill(entries, seq_len, ring_idx, rings, stream=None):
    """entries uint8 [B,n,512] (E4M3, positions seq_len-n .. seq_len-1), ring_idx int32 [B]:
    the last min(n,128) entries of each sequence into their ring slots."""
    _need(entries, "entries", torch.uint8, 3)
    _need(ring_idx, "ring_idx", torch.int32, 1)
    B, n = entries.shape[0], entries.shape[1]
    _check(lib.csa2_ring_refill(_ptr(entries), _ptr(seq_len), B, n, _ptr(ring_idx), rings.shape[0], _ptr(rings),
                                _stream(stream)))


# ---- codecs -------------------------------------------------------------------

def csa2_quant_mxfp4(x, codes=None, scales=None, stream=None):
    """bf16 [..., n] (n % 16 == 0) -> (codes uint8 [..., n/2], scales uint8 [..., n/16])."""
    _need(x, "x", torch.bfloat16)
    n = x.numel()
    if codes is None:
        codes = torch.empty(*x.shape[:-1], x.shape[-1] // 2, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(*x.shape[:-1], x.shape[-1] // 16, dtype=torch.uint8, device=x.device)
    _check(lib.csa2_quant_mxfp4(_ptr(x), n, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def csa2_dequant_mxfp4(codes, scales, out=None, stream=None):
    n = codes.numel() * 2
    if out is None:
        out = torch.empty(*codes.shape[:-1], codes.shape[-1] * 2, dtype=torch.float32, device=codes.device)
    _check(lib.csa2_dequant_mxfp4(_ptr(codes), _ptr(scales), n, _ptr(out), _stream(stream)))
    return out


def csa2_quant_fp8(x, out=None, stream=None):
    _need(x, "x", torch.float32)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib.csa2_quant_fp8(_ptr(x), x.numel(), _ptr(out), _stream(stream)))
    return out


# ---- indexer ------------------------------------------------------------------

def csa2_indexer_scan(q_codes, q_scales, w, seq_len, max_ctx, block_table, n_pages, idx_pages,
                      block_max, stream=None, m=1):
    """q_codes uint8 [B,n_q,32,64], q_scales uint8 [B,n_q,32,8], w fp32 [B,n_q,32],
    seq_len int64 [B] -> block_max fp32 [B,n_q,max_blocks]."""
    B, n_q = w.shape[0], w.shape[1]
    _check(lib.csa2_indexer_scan(_ptr(q_codes), _ptr(q_scales), _ptr(w), _ptr(seq_len), B, n_q, max_ctx,
                                 _ptr(block_table), block_table.shape[1], n_pages, _ptr(idx_pages),
                                 _ptr(block_max), block_max.shape[-1], m, _stream(stream)))


def csa2_block_topk(block_max, seq_len, pool, stream=None, m=1):
    B, n_q = block_max.shape[0], block_max.shape[1]
    _check(lib.csa2_block_topk(_ptr(block_max), _ptr(seq_len), B, n_q, block_max.shape[-1], _ptr(pool), m,
                               _stream(stream)))


def csa2_indexer_reindex(q_codes, q_scales, w, seq_len, block_table, n_pages, idx_pages, pool, topk, ws,
                         stream=None, m=1):
    B, n_q = w.shape[0], w.shape[1]
    _check(lib.csa2_indexer_reindex(_ptr(q_codes), _ptr(q_scales), _ptr(w), _ptr(seq_len), B, n_q,
                                    _ptr(block_table), block_table.shape[1], n_pages, _ptr(idx_pages),
                                    _ptr(pool), _ptr(topk), _ptr(ws), ws.numel() * ws.element_size(), m,
                                    _stream(stream)))


def csa2_indexer_reindex_noalloc(q_codes, q_scales, w, seq_len, block_table, n_pages, idx_pages, pool, topk,
                                 stream=None, m=1):
    """csa2_indexer_reindex without a workspace (scores kept in the library's
    fixed device array; at most 64 query tokens per call)."""
    B, n_q = w.shape[0], w.shape[1]
    _check(lib.csa2_indexer_reindex_noalloc(_ptr(q_codes), _ptr(q_scales), _ptr(w), _ptr(seq_len), B, n_q,
                                            _ptr(block_table), block_table.shape[1], n_pages, _ptr(idx_pages),
                                            _ptr(pool), _ptr(topk), m, _stream(stream)))


def csa2_indexer_full(q_codes, q_scales, w, seq_len, max_ctx, block_table, n_pages, idx_pages, pool, topk,
                      ws, stream=None, m=1):
    B, n_q = w.shape[0], w.shape[1]
    _check(lib.csa2_indexer_full(_ptr(q_codes), _ptr(q_scales), _ptr(w), _ptr(seq_len), B, n_q, max_ctx,
                                 _ptr(block_table), block_table.shape[1], n_pages, _ptr(idx_pages),
                                 _ptr(pool), _ptr(topk), _ptr(ws), ws.numel() * ws.element_size(), m,
                                 _stream(stream)))


# ---- attention ----------------------------------------------------------------

def csa2_sparse_attn(q, topk, seq_len, block_table, n_pages, main_pages, rings, ring_idx, out, lse, ws,
                     softmax_scale=1.0 / math.sqrt(LATENT_DIM), stream=None, derotate=False, m=1):
    """q bf16 [B,n_q,64,512], topk int32 [B,n_q,512] -> out [B,n_q,64,512] (fp32 or bf16), lse fp32 [B,n_q,64].
    derotate: rotate the output's last 64 channels back by the token position (CSA2_OUT_DEROTATE)."""
    _need(q, "q", torch.bfloat16, 4)
    B, n_q = q.shape[0], q.shape[1]
    out_dtype = (OUT_F32 if out.dtype == torch.float32 else OUT_BF16) | (OUT_DEROTATE if derotate else 0)
    _check(lib.csa2_sparse_attn(_ptr(q), _ptr(topk), _ptr(seq_len), B, n_q, _ptr(block_table),
                                block_table.shape[1], n_pages, _ptr(main_pages), _ptr(rings), _ptr(ring_idx),
                                rings.shape[0], softmax_scale, out_dtype, _ptr(out), _ptr(lse), _ptr(ws),
                                ws.numel() * ws.element_size(), m, _stream(stream)))


def csa2_sparse_attn_prefill(q, topk, seq_len, block_table, n_pages, main_pages, rings, ring_idx, swa_chunk, out,
                             lse, ws=None, softmax_scale=1.0 / math.sqrt(LATENT_DIM), stream=None, derotate=False,
                             m=1):
    """As csa2_sparse_attn, with the exact causal window: swa_chunk uint8 [B,n_q,512] holds the E4M3
    window entries of the call's own positions, the rings the 128 positions before them."""
    _need(q, "q", torch.bfloat16, 4)
    _need(swa_chunk, "swa_chunk", torch.uint8, 3)
    B, n_q = q.shape[0], q.shape[1]
    out_dtype = (OUT_F32 if out.dtype == torch.float32 else OUT_BF16) | (OUT_DEROTATE if derotate else 0)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib.csa2_sparse_attn_prefill(_ptr(q), _ptr(topk), _ptr(seq_len), B, n_q, _ptr(block_table),
                                        block_table.shape[1], n_pages, _ptr(main_pages), _ptr(rings),
                                        _ptr(ring_idx), rings.shape[0], _ptr(swa_chunk), softmax_scale, out_dtype,
                                        _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, m, _stream(stream)))


# ---- dispatcher ---------------------------------------------------------------

def layer_args(mode, *, B, n_q, max_ctx, seq_len, block_table, n_pages, main_pages, idx_pages, rings,
               ring_idx, q, out, ws, q_idx_codes=None, q_idx_scales=None, w=None, pool=None, topk=None,
               lse=None, softmax_scale=1.0 / math.sqrt(LATENT_DIM), derotate=False, swa_chunk=None,
               m=1) -> LayerArgs:
    a = LayerArgs()
    a.mode, a.B, a.n_q, a.max_ctx = mode, B, n_q, max_ctx
    a.seq_len, a.block_table, a.max_pages, a.n_pages = _ptr(seq_len), _ptr(block_table), block_table.shape[1], n_pages
    a.main_pages, a.idx_pages = _ptr(main_pages), _ptr(idx_pages)
    a.rings, a.ring_idx, a.n_rings = _ptr(rings), _ptr(ring_idx), rings.shape[0]
    a.q_idx_codes, a.q_idx_scales, a.w, a.q = _ptr(q_idx_codes), _ptr(q_idx_scales), _ptr(w), _ptr(q)
    a.pool, a.topk = _ptr(pool), _ptr(topk)
    a.softmax_scale = softmax_scale
    a.out_dtype = (OUT_F32 if out.dtype == torch.float32 else OUT_BF16) | (OUT_DEROTATE if derotate else 0)
    a.out, a.lse = _ptr(out), _ptr(lse)
    a.ws, a.ws_bytes = _ptr(ws), ws.numel() * ws.element_size()
    a.swa_chunk = _ptr(swa_chunk)
    a.tokens_per_entry = m
    return a


def csa2_decode_layer(args: LayerArgs, stream=None):
    _check(lib.csa2_decode_layer(ctypes.byref(args), _stream(stream)))


def csa2_decode_group(layers, stream=None):
    arr = (LayerArgs * len(layers))(*layers)
    _check(lib.csa2_decode_group(arr, len(layers), _stream(stream)))


def csa2_check_device_status(stream=None) -> int:
    """Waits for the stream and returns (and clears) the device status code."""
    st = ctypes.c_int(0)
    _check(lib.csa2_check_device_status(_stream(stream), ctypes.byref(st)))
    return st.value


def csa2_debug_force_wait_timeout(site: int, stream=None):
    """Test utility: bounded waits at the given internal site give up at once
    (CSA2_ERR_DEVICE_TIMEOUT); 0 turns it off."""
    _check(lib.csa2_debug_force_wait_timeout(site, _stream(stream)))


def device_status_message() -> str:
    return lib.csa2_last_error().decode()
