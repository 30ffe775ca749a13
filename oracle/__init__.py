"""CPU oracle for DGQ KV-cache compression and INT8 paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import this package.  The product library
(``int8_group_quantized_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, fp32 steps exactly as
the DGQ article's compress() describes them, fp64 attention); this module only builds
that file with gcc and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")
D = 128
MAX_SEG = 5

# One record per (request, KV head), 128 bytes, as written by oracle_compress.
SEG_DTYPE = np.dtype(
    [
        ("n_seg", "<i4"),
        ("seq_len", "<i4"),
        ("start", "<i4", (MAX_SEG,)),
        ("k_min", "<f4", (MAX_SEG,)),
        ("k_scale", "<f4", (MAX_SEG,)),
        ("v_min", "<f4", (MAX_SEG,)),
        ("v_scale", "<f4", (MAX_SEG,)),
        ("k_inv_last", "<f4"),
        ("v_inv_last", "<f4"),
        ("pad", "<i4", (3,)),
    ]
)
assert SEG_DTYPE.itemsize == 128


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2 -ffp-contract=off)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".{os.getpid()}.tmp"
    subprocess.check_call(
        ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
         SRC, "-o", tmp, "-lm"]
    )
    os.replace(tmp, LIB)
    return LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        L.oracle_ngroups.argtypes = [i32]
        L.oracle_ngroups.restype = i32
        L.oracle_token_variance.argtypes = [P]
        L.oracle_token_variance.restype = ctypes.c_float
        L.oracle_window_means.argtypes = [P, i32, P]
        L.oracle_window_means.restype = None
        L.oracle_boundaries.argtypes = [P, i32, i32, P]
        L.oracle_boundaries.restype = i32
        L.oracle_boundaries_ex.argtypes = [P, i32, i32, i32, ctypes.c_float, P]
        L.oracle_boundaries_ex.restype = i32
        L.oracle_encode.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_float]
        L.oracle_encode.restype = ctypes.c_uint8
        L.oracle_compress_pair.argtypes = [P, P, i64, i32, P, P, P]
        L.oracle_compress_pair.restype = None
        L.oracle_compress.argtypes = [P, P, P, i32, i32, i32, P, i32, P, P, P]
        L.oracle_compress.restype = None
        L.oracle_compress_pair_ex.argtypes = [P, P, i64, i32, i32, ctypes.c_float, P, P, P]
        L.oracle_compress_pair_ex.restype = None
        L.oracle_compress_ex.argtypes = [P, P, P, i32, i32, i32, P, i32, i32, ctypes.c_float, P, P, P]
        L.oracle_compress_ex.restype = None
        L.oracle_compress_split.argtypes = [P, P, P, i32, i32, i32, P, i32, i32, ctypes.c_float, P, P, P, P]
        L.oracle_compress_split.restype = None
        L.oracle_append_split.argtypes = [P, P, i32, i32, i32, P, i32, P, P, P, P]
        L.oracle_append_split.restype = i32
        L.oracle_dequant_pair.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, ctypes.c_int, P]
        L.oracle_dequant_pair.restype = None
        L.oracle_paged_decode_attn.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, P]
        L.oracle_paged_decode_attn.restype = None
        L.oracle_append.argtypes = [P, P, i32, i32, i32, P, i32, P, P, P]
        L.oracle_append.restype = i32
        L.oracle_resegment_flags.argtypes = [i32]
        L.oracle_resegment_flags.restype = i32
        L.oracle_append_resegment.argtypes = [P, P, i32, i32, i32, P, i32, P, P, P, P, P, P, i32, i32,
                                              ctypes.c_float, P]
        L.oracle_append_resegment.restype = i32
        L.oracle_decode_attn_unquantised.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, P]
        L.oracle_decode_attn_unquantised.restype = None
        for name in ("oracle_dequant_fixed64", "oracle_dequant_sym_int8", "oracle_dequant_fp8_e4m3"):
            getattr(L, name).argtypes = [P, i64, i32, P]
            getattr(L, name).restype = None
        L.oracle_decode_attn_dense.argtypes = [P, P, P, P, P, i32, i32, i32, P]
        L.oracle_decode_attn_dense.restype = None
        L.oracle_compress_bytes_written.argtypes = [i32, i32]
        L.oracle_compress_bytes_written.restype = i64
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def ngroups(L: int) -> int:
    return int(lib().oracle_ngroups(int(L)))


def token_variance(k_row: np.ndarray) -> np.float32:
    k_row = np.ascontiguousarray(k_row, dtype=np.uint16)
    assert k_row.shape == (D,)
    return np.float32(lib().oracle_token_variance(_p(k_row)))


def window_means(var: np.ndarray) -> np.ndarray:
    var = np.ascontiguousarray(var, dtype=np.float32)
    L = var.shape[0]
    out = np.zeros((L + 15) // 16, dtype=np.float32)
    lib().oracle_window_means(_p(var), L, _p(out))
    return out


def boundaries(means: np.ndarray, L: int, max_groups: int = MAX_SEG, min_var: float = 0.0) -> list[int]:
    means = np.ascontiguousarray(means, dtype=np.float32)
    start = np.zeros(MAX_SEG, dtype=np.int32)
    n = lib().oracle_boundaries_ex(_p(means), means.shape[0], int(L), int(max_groups), float(min_var), _p(start))
    return [int(x) for x in start[:n]]


def encode(x: float, mn: float, inv: float) -> int:
    return int(lib().oracle_encode(float(x), float(mn), float(inv)))


def compress_pair(k: np.ndarray, v: np.ndarray, max_groups: int = MAX_SEG, min_var: float = 0.0):
    """k, v: [L, 128] bf16 bit patterns (uint16).  Returns (record, k_codes, v_codes)."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    L = k.shape[0]
    rec = np.zeros(1, dtype=SEG_DTYPE)
    kc = np.zeros((max(L, 1), D), dtype=np.uint8)
    vc = np.zeros((max(L, 1), D), dtype=np.uint8)
    lib().oracle_compress_pair_ex(_p(k), _p(v), D, L, int(max_groups), float(min_var), _p(rec), _p(kc), _p(vc))
    return rec[0], kc[:L], vc[:L]


def compress(k, v, cu_seqlens, num_kv_heads, block_size, block_tables, num_blocks, fill=0, max_groups=MAX_SEG,
             min_var=0.0):
    """One layer.  k, v: [T, Hkv, 128] uint16; block_tables [B, max_blocks] int32.
    Returns (k_pool, v_pool, table) with pools [num_blocks, Hkv, bs, 128] uint8 (slots
    the call does not write keep `fill`) and table [B, Hkv] SEG_DTYPE."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    B = cu.shape[0] - 1
    kp = np.full((num_blocks, num_kv_heads, block_size, D), fill, dtype=np.uint8)
    vp = np.full((num_blocks, num_kv_heads, block_size, D), fill, dtype=np.uint8)
    table = np.zeros((B, num_kv_heads), dtype=SEG_DTYPE)
    lib().oracle_compress_ex(_p(k), _p(v), _p(cu), B, num_kv_heads, block_size, _p(bt), bt.shape[1],
                             int(max_groups), float(min_var), _p(kp), _p(vp), _p(table))
    return kp, vp, table


def compress_split(k, v, cu_seqlens, num_kv_heads, block_size, block_tables, num_blocks, fill=0,
                   max_groups=MAX_SEG, min_var=0.0):
    """One layer with independent V segmentation (V segmented by the same rule on V's own
    variance).  Returns (k_pool, v_pool, k_table, v_table): k_table holds K's segments and K
    parameters, v_table V's segments and V parameters (the other tensor's fields 0)."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    B = cu.shape[0] - 1
    kp = np.full((num_blocks, num_kv_heads, block_size, D), fill, dtype=np.uint8)
    vp = np.full((num_blocks, num_kv_heads, block_size, D), fill, dtype=np.uint8)
    kt = np.zeros((B, num_kv_heads), dtype=SEG_DTYPE)
    vt = np.zeros((B, num_kv_heads), dtype=SEG_DTYPE)
    lib().oracle_compress_split(_p(k), _p(v), _p(cu), B, num_kv_heads, block_size, _p(bt), bt.shape[1],
                                int(max_groups), float(min_var), _p(kp), _p(vp), _p(kt), _p(vt))
    return kp, vp, kt, vt


def append(k_new, v_new, block_size, block_tables, k_pool, v_pool, table):
    """One decode step's token per (request, KV head) into the cache, in place.  k_new, v_new:
    [B, Hkv, 128] uint16; pools [num_blocks, Hkv, bs, 128] uint8; table [B, Hkv] SEG_DTYPE.
    Returns the number of pairs skipped for want of a block-table column."""
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    for a in (k_pool, v_pool, table):
        assert a.flags["C_CONTIGUOUS"]
    B, Hkv = k_new.shape[0], k_new.shape[1]
    return int(lib().oracle_append(_p(k_new), _p(v_new), B, Hkv, int(block_size), _p(bt), bt.shape[1],
                                   _p(k_pool), _p(v_pool), _p(table)))


RESEG_WINDOW = 1   # the appended token completed a 16-token window
RESEG_NGROUPS = 2  # the length crossed an n_groups threshold


def resegment_flags(L: int) -> int:
    """Trigger bits of appending token L (the cache grows from L to L + 1 tokens)."""
    return int(lib().oracle_resegment_flags(int(L)))


def append_resegment(k_new, v_new, block_size, block_tables, k_pool, v_pool, table, k_hist, v_hist, hist_cu,
                     mask=RESEG_WINDOW | RESEG_NGROUPS, max_groups=MAX_SEG, min_var=0.0):
    """append, then every request with a pair whose trigger bits meet `mask` compressed again from
    its bf16 history (k_hist, v_hist packed [T, Hkv, 128] uint16 with its L + 1 tokens on rows
    hist_cu[b] ..).  Pools and table in place.  Returns (flags [B, Hkv] int32, skipped)."""
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    kh = np.ascontiguousarray(k_hist, dtype=np.uint16)
    vh = np.ascontiguousarray(v_hist, dtype=np.uint16)
    cu = np.ascontiguousarray(hist_cu, dtype=np.int32)
    for a in (k_pool, v_pool, table):
        assert a.flags["C_CONTIGUOUS"]
    B, Hkv = k_new.shape[0], k_new.shape[1]
    flags = np.zeros((B, Hkv), dtype=np.int32)
    skipped = lib().oracle_append_resegment(_p(k_new), _p(v_new), B, Hkv, int(block_size), _p(bt), bt.shape[1],
                                            _p(k_pool), _p(v_pool), _p(table), _p(kh), _p(vh), _p(cu), int(mask),
                                            int(max_groups), float(min_var), _p(flags))
    return flags, int(skipped)


def append_split(k_new, v_new, block_size, block_tables, k_pool, v_pool, k_table, v_table):
    """append with independent V segmentation: K's codes and record from k_table, V's from
    v_table, in place.  Returns the number of pairs skipped for want of a block-table column."""
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    for a in (k_pool, v_pool, k_table, v_table):
        assert a.flags["C_CONTIGUOUS"]
    B, Hkv = k_new.shape[0], k_new.shape[1]
    return int(lib().oracle_append_split(_p(k_new), _p(v_new), B, Hkv, int(block_size), _p(bt), bt.shape[1],
                                         _p(k_pool), _p(v_pool), _p(k_table), _p(v_table)))


def dequant_pair(pool, table, block_tables, b, h, L, which_v):
    pool = np.ascontiguousarray(pool, dtype=np.uint8)
    table = np.ascontiguousarray(table)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    Hkv, bs = pool.shape[1], pool.shape[2]
    out = np.zeros((max(L, 1), D), dtype=np.float64)
    lib().oracle_dequant_pair(_p(pool), _p(table), _p(bt), b, h, Hkv, bs, bt.shape[1], L,
                              int(which_v), _p(out))
    return out[:L]


def paged_decode_attn(q, k_new, v_new, k_pool, v_pool, table, block_tables, seq_lens):
    """fp64 decode attention; q [B, Hq, 128], k_new/v_new [B, Hkv, 128] uint16."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kn = np.ascontiguousarray(k_new, dtype=np.uint16)
    vn = np.ascontiguousarray(v_new, dtype=np.uint16)
    kp = np.ascontiguousarray(k_pool, dtype=np.uint8)
    vp = np.ascontiguousarray(v_pool, dtype=np.uint8)
    table = np.ascontiguousarray(table)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq = q.shape[0], q.shape[1]
    Hkv, bs = kp.shape[1], kp.shape[2]
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lib().oracle_paged_decode_attn(_p(q), _p(kn), _p(vn), _p(kp), _p(vp), _p(table), _p(bt),
                                   _p(sl), B, Hq, Hkv, bs, bt.shape[1], _p(out))
    return out


def decode_attn_unquantised(q, k_new, v_new, k, v, cu_seqlens, seq_lens):
    """fp64 decode attention over the original bf16 K/V (packed [T, Hkv, 128] uint16, request b
    on rows cu_seqlens[b] ..), for the fidelity of the compressed cache."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kn = np.ascontiguousarray(k_new, dtype=np.uint16)
    vn = np.ascontiguousarray(v_new, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq = q.shape[0], q.shape[1]
    Hkv = kn.shape[1]
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lib().oracle_decode_attn_unquantised(_p(q), _p(kn), _p(vn), _p(k if k.size else np.zeros(1, np.uint16)),
                                         _p(v if v.size else np.zeros(1, np.uint16)), _p(cu), _p(sl), B, Hq, Hkv,
                                         _p(out))
    return out


COMPARISON_QUANTISERS = ("fixed64", "sym_int8", "fp8_e4m3")


def dequant_comparison(x, scheme: str) -> np.ndarray:
    """x: [L, 128] bf16 bits of one (request, head) pair -> fp64 values after a comparison
    quantiser (fixed64 / sym_int8 / fp8_e4m3) and its dequantisation."""
    assert scheme in COMPARISON_QUANTISERS
    x = np.ascontiguousarray(x, dtype=np.uint16)
    L = x.shape[0]
    out = np.zeros((max(L, 1), D), dtype=np.float64)
    getattr(lib(), "oracle_dequant_" + scheme)(_p(x), D, L, _p(out))
    return out[:L]


def decode_attn_dense(q, k_new, v_new, kd, vd):
    """fp64 decode attention of one request: q [Hq, 128], k_new/v_new [Hkv, 128] bf16 bits,
    kd/vd [L, Hkv, 128] fp64 (dequantised keys and values)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kn = np.ascontiguousarray(k_new, dtype=np.uint16)
    vn = np.ascontiguousarray(v_new, dtype=np.uint16)
    kd = np.ascontiguousarray(kd, dtype=np.float64)
    vd = np.ascontiguousarray(vd, dtype=np.float64)
    Hq, Hkv = q.shape[0], kn.shape[0]
    L = kd.shape[0]
    out = np.zeros((Hq, D), dtype=np.float64)
    lib().oracle_decode_attn_dense(_p(q), _p(kn), _p(vn), _p(kd if kd.size else np.zeros(1)),
                                   _p(vd if vd.size else np.zeros(1)), L, Hq, Hkv, _p(out))
    return out


def compress_bytes_written(L: int, Hkv: int) -> int:
    return int(lib().oracle_compress_bytes_written(int(L), int(Hkv)))
