"""The C-ABI library loads and exports every entry point that include/csa2.h
declares; host-only calls (sizes, status strings, argument validation) work
without a GPU. No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


@pytest.fixture(scope="module")
def lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_csa2_build", os.path.join(ROOT, "sparse_attention_fp4_mxfp4_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return ctypes.CDLL(mod.build())


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(csa2_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared()
    for must in ("csa2_append_kv", "csa2_append_swa", "csa2_indexer_full", "csa2_indexer_reindex",
                 "csa2_indexer_scan", "csa2_block_topk", "csa2_sparse_attn", "csa2_decode_layer",
                 "csa2_decode_group", "csa2_check_device_status", "csa2_workspace_bytes"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_symbol():
    import sparse_attention_fp4_mxfp4_gb300 as m
    assert sorted(m.EXPORTS) == declared()


def test_size_queries(lib):
    n = ctypes.c_size_t()
    assert lib.csa2_page_bytes(0, ctypes.byref(n)) == 0 and n.value == 36864
    assert lib.csa2_page_bytes(1, ctypes.byref(n)) == 0 and n.value == 9216
    assert lib.csa2_page_bytes(7, ctypes.byref(n)) == 1
    assert lib.csa2_ring_bytes(ctypes.byref(n)) == 0 and n.value == 65536
    lib.csa2_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                         ctypes.POINTER(ctypes.c_size_t)]
    assert lib.csa2_workspace_bytes(3, 64, 1, 65536, ctypes.byref(n)) == 0
    assert n.value == 64 * 5 * 64 * 512 * 4 + 64 * 5 * 64 * 8
    assert lib.csa2_workspace_bytes(2, 64, 1, 131072, ctypes.byref(n)) == 0 and n.value == 64 * 16384 * 4
    assert lib.csa2_workspace_bytes(3, 1, 0, 100, ctypes.byref(n)) == 1
    # Prefill shapes: up to 4096 tokens per sequence and 65535 per call; the
    # attention needs no partial-output workspace from 256 tokens on.
    assert lib.csa2_workspace_bytes(3, 1, 4096, 100, ctypes.byref(n)) == 0 and n.value == 0
    assert lib.csa2_workspace_bytes(3, 1, 255, 100, ctypes.byref(n)) == 0
    assert n.value == 255 * 5 * 64 * 512 * 4 + 255 * 5 * 64 * 8
    assert lib.csa2_workspace_bytes(2, 2, 1000, 100, ctypes.byref(n)) == 0 and n.value == 2000 * 16384 * 4
    assert lib.csa2_workspace_bytes(3, 1, 4097, 100, ctypes.byref(n)) == 2
    assert lib.csa2_workspace_bytes(3, 17, 4000, 100, ctypes.byref(n)) == 2  # 68000 tokens


def test_prefill_and_refill_host_checks(lib):
    p, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.csa2_last_error.restype = ctypes.c_char_p
    lib.csa2_sparse_attn.argtypes = [p, p, p, i32, i32, p, i32, i64, p, p, p, i64, f32, i32, p, p, p, sz, i32, p]
    lib.csa2_sparse_attn_prefill.argtypes = [p, p, p, i32, i32, p, i32, i64, p, p, p, i64, p, f32, i32, p, p, p,
                                             sz, i32, p]
    x = p(4096)  # an aligned non-null address; no call below reaches the device
    # The decode attention keeps its 8-token limit (its window comes from the ring alone).
    assert lib.csa2_sparse_attn(x, x, x, 1, 9, x, 1, 1, x, x, x, 1, 0.05, 0, x, None, None, 0, 1, None) == 2
    assert lib.csa2_sparse_attn(x, x, x, 1, 1, x, 1, 1, x, x, x, 1, 0.05, 0, x, None, None, 0, 3, None) == 2  # m = 3
    assert lib.csa2_sparse_attn_prefill(x, x, x, 1, 9, x, 1, 1, x, x, x, 1, None, 0.05, 0, x, None, None, 0,
                                        1, None) == 1
    assert b"swa_chunk" in lib.csa2_last_error()
    assert lib.csa2_sparse_attn_prefill(x, x, x, 1, 9, x, 1, 1, x, x, x, 1, p(4100), 0.05, 0, x, None, None, 0,
                                        1, None) == 1
    assert lib.csa2_sparse_attn_prefill(x, x, x, 1, 4097, x, 1, 1, x, x, x, 1, x, 0.05, 0, x, None, None, 0,
                                        1, None) == 2
    lib.csa2_ring_refill.argtypes = [p, p, i32, i32, p, i64, p, p]
    assert lib.csa2_ring_refill(None, None, 1, 0, None, 1, None, None) == 0  # nothing to do
    assert lib.csa2_ring_refill(None, x, 1, 4, x, 1, x, None) == 1
    assert b"entries" in lib.csa2_last_error()
    assert lib.csa2_ring_refill(x, x, 1, 4, x, 0, x, None) == 1
    assert lib.csa2_ring_refill(x, x, 1, -1, x, 1, x, None) == 1
    lib.csa2_quant_fp8_entries.argtypes = [p, i32, p, p]
    assert lib.csa2_quant_fp8_entries(p(4104), 2, x, None) == 1
    assert lib.csa2_quant_fp8_entries(None, 0, None, None) == 0


def test_status_strings_and_null_checks(lib):
    lib.csa2_status_string.restype = ctypes.c_char_p
    lib.csa2_last_error.restype = ctypes.c_char_p
    assert lib.csa2_status_string(0) == b"ok"
    assert lib.csa2_status_string(5).startswith(b"a bounded device wait")
    p = ctypes.c_void_p
    lib.csa2_append_kv.argtypes = [p, p, p, p, ctypes.c_int, p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, p, p, p]
    assert lib.csa2_append_kv(None, None, None, None, 4, None, 1, 1, 1, None, None, None) == 1
    assert b"latent" in lib.csa2_last_error()
    assert lib.csa2_append_kv(None, None, None, None, 0, None, 1, 1, 1, None, None, None) == 0  # nothing to do
    lib.csa2_quant_mxfp4.argtypes = [p, ctypes.c_int64, p, p, p]
    assert lib.csa2_quant_mxfp4(p(16), 17, p(16), p(16), None) == 1
    assert lib.csa2_decode_group(None, 1, None) == 1


def test_tokens_per_entry_and_compressor_host_checks(lib):
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.csa2_last_error.restype = ctypes.c_char_p
    x = p(4096)  # an aligned non-null address; no call below reaches the device
    lib.csa2_compress_append.argtypes = [p, p, p, p, p, p, i32, i32, p, p, i32, i32, i64, p, p, p]
    assert lib.csa2_compress_append(None, None, None, None, None, None, 0, 2, None, None, 1, 1, 1, None, None,
                                    None) == 0  # nothing to do
    assert lib.csa2_compress_append(x, x, x, x, x, x, 4, 3, x, x, 1, 1, 1, x, x, None) == 2  # m = 3
    assert b"m = 3" in lib.csa2_last_error()
    assert lib.csa2_compress_append(x, x, x, x, x, x, 4, 2, None, x, 1, 1, 1, x, x, None) == 1
    assert b"tail" in lib.csa2_last_error()
    # m = 1 needs no tail
    assert lib.csa2_compress_append(x, x, x, x, x, x, 4, 1, None, None, 1, 1, 1, x, x, None) == 1
    assert b"block_table" in lib.csa2_last_error()
    lib.csa2_indexer_scan.argtypes = [p, p, p, p, i32, i32, i64, p, i32, i64, p, p, i64, i32, p]
    assert lib.csa2_indexer_scan(x, x, x, x, 1, 1, 100, x, 1, 1, x, x, 13, 4, None) == 2  # m = 4
    # at m = 2 the block maxima cover ceil(max_ctx / 2 / 8) blocks
    assert lib.csa2_indexer_scan(x, x, x, x, 1, 1, 1600, x, 1, 1, x, x, 99, 2, None) == 1
    assert b"max_blocks" in lib.csa2_last_error()
    lib.csa2_block_topk.argtypes = [p, p, i32, i32, i64, p, i32, p]
    assert lib.csa2_block_topk(x, x, 1, 1, 10, x, 0, None) == 2


def test_decode_appends_host_checks(lib):
    """csa2_decode_appends rejects bad arguments before any device work."""
    import sparse_attention_fp4_mxfp4_gb300 as m
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.csa2_decode_appends.argtypes = [p, p, p, p, i32, p, i32, i32, i64, p, p, p, i32, p]
    x = p(4096)  # an aligned non-null address; no call below reaches the device
    layers = (m.AppendLayer * 17)()
    assert lib.csa2_decode_appends(x, x, x, x, -1, x, 1, 1, 1, x, x, layers, 1, None) == 1    # T < 0
    assert lib.csa2_decode_appends(x, x, x, x, 1, x, 1, 1, 1, x, x, layers, -1, None) == 1    # n_layers < 0
    assert lib.csa2_decode_appends(x, x, x, x, 1, x, 1, 1, 1, x, x, layers, 17, None) == 2    # > 16 layers
    assert lib.csa2_decode_appends(x, x, x, x, 1, x, 1, 1, 1, x, x, None, 1, None) == 1       # layers NULL
    assert lib.csa2_decode_appends(p(4100), x, x, x, 1, x, 1, 1, 1, x, x, layers, 0, None) == 1  # latent unaligned
    assert lib.csa2_decode_appends(x, x, x, x, 1, x, 0, 1, 1, x, x, layers, 0, None) == 1     # B < 1
    layers[0].swa, layers[0].ring_idx, layers[0].rings, layers[0].n_rings = 4096, None, 4096, 1
    assert lib.csa2_decode_appends(x, x, x, x, 1, x, 1, 1, 1, x, x, layers, 1, None) == 1     # ring_idx NULL
    layers[0].swa = None
    layers[0].q_idx, layers[0].q_n, layers[0].q_codes, layers[0].q_scales = 4096, 24, 4096, 4096
    assert lib.csa2_decode_appends(x, x, x, x, 1, x, 1, 1, 1, x, x, layers, 1, None) == 1     # q_n % 16
    layers[0].q_n, layers[0].q_codes = 32, 4100
    assert lib.csa2_decode_appends(x, x, x, x, 1, x, 1, 1, 1, x, x, layers, 1, None) == 1     # codes unaligned
    # Nothing to do: no launch at all.
    assert lib.csa2_decode_appends(None, None, None, None, 0, None, 0, 0, 0, None, None, None, 0, None) == 0
