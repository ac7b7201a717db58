"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

Holds none of the method's arithmetic: it only draws numbers (see gen.cpp for
the generator's definition). Both sides receive exactly the arrays returned
here, so a parity failure can never come from two generators disagreeing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.cpp")
_LIB = os.path.join(_HERE, "_synth.so")

# Tensor ids of the counter streams (per-layer tensors add the layer index).
LATENT = 1      # main-KV latent entries, (seq, pos) -> 512 bf16
IDXKEY = 2      # indexer keys, (seq, pos) -> 128 bf16
KVGATE = 3      # compression logits of the latent candidates (m > 1), (seq, pos) -> 512 bf16
IDXGATE = 4     # compression logits of the indexer-key candidates (m > 1), (seq, pos) -> 128 bf16
Q = 16          # attention queries, (seq, t) -> 64 x 512 bf16        (+ layer)
IDXQ = 32       # indexer queries, (seq, t) -> 32 x 128 bf16          (+ layer)
W = 48          # indexer head weights, (seq, t) -> 32 fp32 U(0,1)    (+ layer)
SWA = 64        # sliding-window entries, (seq, pos) -> 512 bf16      (+ layer)
TOPK = 96       # uniform top-512 positions, (seq, t)
POOL = 112      # uniform pool of 2048 blocks, (seq, t)               (+ layer)

DEFAULT_THREADS = max(1, min(32, os.cpu_count() or 1))


def build(force: bool = False) -> str:
    """Compile gen.cpp into _synth.so (plain g++, no fast-math, no FMA contraction)."""
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
        build()
        L = ctypes.CDLL(_LIB)
        i64, u64, u32, i32, p = ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p
        L.synth_normal_bf16.argtypes = [u64, u32, i64, i64, i64, i32, p, i32]
        L.synth_normal_bf16_rows.argtypes = [u64, u32, p, p, i64, i32, p, i32]
        L.synth_latent_bf16.argtypes = [u64, u32, i64, i64, i64, p, i32]
        L.synth_latent_bf16_rows.argtypes = [u64, u32, p, p, i64, p, i32]
        L.synth_uniform_f32.argtypes = [u64, u32, i64, i64, i64, i32, ctypes.c_double, ctypes.c_double, p]
        L.synth_sample_sorted.argtypes = [u64, u32, i64, i64, i64, i64, p]
        L.synth_sample_sorted.restype = i64
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def normal(seed, tensor, seq, pos0, n, dim, out=None, threads=DEFAULT_THREADS) -> np.ndarray:
    """bf16 bit patterns (uint16) [n, dim] of N(0,1) draws for rows (seq, pos0..pos0+n)."""
    out = np.empty((n, dim), np.uint16) if out is None else out
    lib().synth_normal_bf16(seed, tensor, seq, pos0, n, dim, _ptr(out), threads)
    return out


def normal_rows(seed, tensor, seqs, poss, dim, threads=DEFAULT_THREADS) -> np.ndarray:
    seqs = np.ascontiguousarray(seqs, np.int64)
    poss = np.ascontiguousarray(poss, np.int64)
    out = np.empty((len(seqs), dim), np.uint16)
    lib().synth_normal_bf16_rows(seed, tensor, _ptr(seqs), _ptr(poss), len(seqs), dim, _ptr(out), threads)
    return out


def latent(seed, seq, pos0, n, tensor=LATENT, out=None, threads=DEFAULT_THREADS) -> np.ndarray:
    """bf16 bit patterns [n, 512]: RMSNormed, post-RoPE latents (recipe in gen.cpp)."""
    out = np.empty((n, 512), np.uint16) if out is None else out
    lib().synth_latent_bf16(seed, tensor, seq, pos0, n, _ptr(out), threads)
    return out


def latent_rows(seed, seqs, poss, tensor=LATENT, threads=DEFAULT_THREADS) -> np.ndarray:
    seqs = np.ascontiguousarray(seqs, np.int64)
    poss = np.ascontiguousarray(poss, np.int64)
    out = np.empty((len(seqs), 512), np.uint16)
    lib().synth_latent_bf16_rows(seed, tensor, _ptr(seqs), _ptr(poss), len(seqs), _ptr(out), threads)
    return out


def uniform(seed, tensor, seq, pos0, n, dim, lo=0.0, hi=1.0) -> np.ndarray:
    out = np.empty((n, dim), np.float32)
    lib().synth_uniform_f32(seed, tensor, seq, pos0, n, dim, lo, hi, _ptr(out))
    return out


def sample_sorted(seed, tensor, seq, pos, rng, k) -> np.ndarray:
    """k distinct ints uniform without replacement in [0, rng), ascending."""
    out = np.empty(max(0, min(k, rng)), np.int32)
    m = lib().synth_sample_sorted(seed, tensor, seq, pos, rng, k, _ptr(out) if out.size else 0)
    assert m == out.size
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)
