"""Seeded synthetic inputs for the DGQ tests and benchmark.

Host generation goes through ``libsynth.so`` (gcc), device generation through
``libsynth_dev.so`` (nvcc); both are built from ``synth_core.h`` and produce the same
bits.  This module carries no part of the DGQ method: it only draws the tensors
(piecewise-sigma Gaussian K/V, Gaussian Q and current-step K/V) and the per-config
metadata (sequence lengths, block tables, variance spans).  Both the oracle and the
CUDA path read their inputs from here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SRC = os.path.join(HERE, "synth.c")
DEV_SRC = os.path.join(HERE, "synth_dev.cu")
CORE = os.path.join(HERE, "synth_core.h")
HOST_LIB = os.path.join(HERE, "libsynth.so")
DEV_LIB = os.path.join(HERE, "libsynth_dev.so")
MAX_SPANS = 5

STREAM_K, STREAM_V, STREAM_Q, STREAM_KNEW, STREAM_VNEW = 1, 2, 3, 4, 5
STREAM_SPAN, STREAM_CODES, STREAM_META = 6, 7, 8
RULE_SET3, RULE_U, RULE_PERM5 = 0, 1, 2


def _stale(lib: str, *srcs: str) -> bool:
    return not os.path.exists(lib) or any(os.path.getmtime(lib) < os.path.getmtime(s) for s in srcs)


def build_host(force: bool = False) -> str:
    if force or _stale(HOST_LIB, HOST_SRC, CORE):
        tmp = HOST_LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", HOST_SRC, "-o", tmp, "-lm"])
        os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build_device(force: bool = False, nvcc: str = "nvcc") -> str:
    if force or _stale(DEV_LIB, DEV_SRC, CORE):
        tmp = DEV_LIB + f".{os.getpid()}.tmp"
        subprocess.check_call([nvcc, "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-fmad=false", "-prec-div=true", "-prec-sqrt=true",
                               "-Xcompiler", "-fPIC,-ffp-contract=off", "-shared", DEV_SRC, "-o", tmp])
        os.replace(tmp, DEV_LIB)
    return DEV_LIB


_host = None
_dev = None


def host() -> ctypes.CDLL:
    global _host
    if _host is None:
        build_host()
        L = ctypes.CDLL(HOST_LIB)
        P, u64, u32, i32, i64 = (ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32,
                                 ctypes.c_int64)
        L.synth_hash_c.argtypes = [u64, u64]
        L.synth_hash_c.restype = u64
        L.synth_key_c.argtypes = [u64, u32, u32, u32, u32]
        L.synth_key_c.restype = u64
        L.synth_normal_c.argtypes = [u64, u64]
        L.synth_normal_c.restype = ctypes.c_float
        L.synth_bf16_c.argtypes = [ctypes.c_float]
        L.synth_bf16_c.restype = ctypes.c_uint16
        L.synth_spans.argtypes = [u64, u32, u32, u32, i32, i32, P, P]
        L.synth_spans.restype = i32
        L.synth_fill_pair.argtypes = [u64, u32, u32, u32, u32, i32, i32, i32, P, P, P, i64]
        L.synth_fill_pair.restype = None
        L.synth_fill_layer.argtypes = [u64, u32, u32, i32, i32, i32, P, P, P, P, P]
        L.synth_fill_layer.restype = None
        L.synth_fill_heads.argtypes = [u64, u32, u32, i32, i32, i32, ctypes.c_float, P]
        L.synth_fill_heads.restype = None
        L.synth_fill_bytes.argtypes = [u64, u32, u32, i64, P]
        L.synth_fill_bytes.restype = None
        L.synth_permutation.argtypes = [u64, u32, i64, P]
        L.synth_permutation.restype = None
        _host = L
    return _host


def device() -> ctypes.CDLL:
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError("libsynth_dev.so is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(DEV_LIB)
        P, u64, u32, i32, i64 = (ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32,
                                 ctypes.c_int64)
        L.synth_dev_fill_layer.argtypes = [u64, u32, u32, i32, i32, i32, P, P, P, P, i64, P, P]
        L.synth_dev_fill_layer.restype = ctypes.c_int
        L.synth_dev_fill_heads.argtypes = [u64, u32, u32, i32, i32, i32, ctypes.c_float, P, P]
        L.synth_dev_fill_heads.restype = ctypes.c_int
        L.synth_dev_fill_bytes.argtypes = [u64, u32, u32, i64, P, P]
        L.synth_dev_fill_bytes.restype = ctypes.c_int
        _dev = L
    return _dev


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def hash64(key: int, ctr: int) -> int:
    return int(host().synth_hash_c(key & (2**64 - 1), ctr & (2**64 - 1)))


def key(seed: int, stream: int, layer: int, req: int, head: int) -> int:
    return int(host().synth_key_c(seed, stream, layer, req, head))


def spans(seed: int, layer: int, req: int, head: int, L: int, rule: int):
    start = np.zeros(MAX_SPANS, dtype=np.int32)
    sigma = np.zeros(MAX_SPANS, dtype=np.float32)
    n = host().synth_spans(seed, layer, req, head, L, rule, _p(start), _p(sigma))
    return int(n), start, sigma


def span_tables(seed: int, layer: int, seq_lens, num_heads: int, rule: int):
    """Per-(request, head) span tables of one layer: (n [B*H], start [B*H*5], sigma [B*H*5])."""
    B = len(seq_lens)
    n = np.zeros(B * num_heads, dtype=np.int32)
    st = np.zeros((B * num_heads, MAX_SPANS), dtype=np.int32)
    sg = np.zeros((B * num_heads, MAX_SPANS), dtype=np.float32)
    for b in range(B):
        for h in range(num_heads):
            i = b * num_heads + h
            n[i], st[i], sg[i] = spans(seed, layer, b, h, int(seq_lens[b]), rule)
    return n, st.reshape(-1), sg.reshape(-1)


def fill_pair(seed, stream, layer, req, head, L, n_spans, start, sigma, D=128) -> np.ndarray:
    out = np.zeros((max(L, 1), D), dtype=np.uint16)
    start = np.ascontiguousarray(start, dtype=np.int32)
    sigma = np.ascontiguousarray(sigma, dtype=np.float32)
    host().synth_fill_pair(seed, stream, layer, req, head, L, D, n_spans, _p(start), _p(sigma),
                           _p(out), D)
    return out[:L]


def fill_layer(seed, stream, layer, cu_seqlens, num_heads, tables, D=128) -> np.ndarray:
    """Host copy of one layer's packed K or V, [T, H, D] uint16 (bf16 bits)."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    n, st, sg = tables
    T = int(cu[-1])
    out = np.zeros((max(T, 1), num_heads, D), dtype=np.uint16)
    host().synth_fill_layer(seed, stream, layer, cu.shape[0] - 1, num_heads, D, _p(cu), _p(n),
                            _p(st), _p(sg), _p(out))
    return out[:T]


def fill_heads(seed, stream, layer, B, H, sigma, D=128) -> np.ndarray:
    out = np.zeros((B, H, D), dtype=np.uint16)
    host().synth_fill_heads(seed, stream, layer, B, H, D, float(sigma), _p(out))
    return out


def fill_bytes(seed, stream, layer, n) -> np.ndarray:
    out = np.zeros(max(n, 1), dtype=np.uint8)
    host().synth_fill_bytes(seed, stream, layer, n, _p(out))
    return out[:n]


def permutation(seed, stream, n) -> np.ndarray:
    out = np.zeros(max(n, 1), dtype=np.int32)
    host().synth_permutation(seed, stream, n, _p(out))
    return out[:n]


# ---- device fillers (torch tensors; bench / GPU tests only) ------------------------------

def dev_fill_layer(seed, stream, layer, cu_seqlens_dev, num_heads, tables_dev, total_tokens,
                   out, stream_ptr=0, D=128):
    n, st, sg = tables_dev
    rc = device().synth_dev_fill_layer(seed, stream, layer, cu_seqlens_dev.numel() - 1, num_heads, D,
                                       cu_seqlens_dev.data_ptr(), n.data_ptr(), st.data_ptr(),
                                       sg.data_ptr(), total_tokens, out.data_ptr(), stream_ptr)
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_layer failed: {rc}")


def dev_fill_heads(seed, stream, layer, B, H, sigma, out, stream_ptr=0, D=128):
    rc = device().synth_dev_fill_heads(seed, stream, layer, B, H, D, float(sigma), out.data_ptr(),
                                       stream_ptr)
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_heads failed: {rc}")


def dev_fill_bytes(seed, stream, layer, n, out, stream_ptr=0):
    rc = device().synth_dev_fill_bytes(seed, stream, layer, n, out.data_ptr(), stream_ptr)
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill_bytes failed: {rc}")
