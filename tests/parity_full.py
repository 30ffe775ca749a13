"""Host side of the whole-workload parity tests: one layer of a workload drawn on the host by the
seeded generator and run through the CPU oracle, every request of it.  The generator and the
oracle are single-threaded C; their calls release the GIL, so independent requests run on a
thread pool (each call writes only its own rows, blocks and records).  No arithmetic of the
method is done here: the pieces are the oracle's own C functions, called per request."""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

import oracle
import synth
from synth import configs

D = 128
REC = 128  # bytes per segment record


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


@dataclass
class HostLayer:
    lens: np.ndarray
    cu: np.ndarray
    bt: np.ndarray
    num_blocks: int
    k: np.ndarray      # [T, Hkv, 128] bf16 bits
    v: np.ndarray
    q: np.ndarray      # [B, Hq, 128]
    knew: np.ndarray   # [B, Hkv, 128]
    vnew: np.ndarray
    kp: np.ndarray = None     # oracle pools [num_blocks, Hkv, bs, 128]
    vp: np.ndarray = None
    table: np.ndarray = None  # oracle records [B, Hkv]
    out: np.ndarray = None    # oracle fp64 attention [B, Hq, 128]


def draw_layer(w: configs.Workload, layer: int) -> HostLayer:
    """Every request's K and V of one layer, drawn on the host (bit-identical to the device
    generator the benchmark uses)."""
    lens = configs.seq_lens(w)
    bt, nb = configs.block_tables(w, lens)
    cu = configs.cu_seqlens(lens)
    B, Hkv = w.batch, w.hkv
    n, st, sg = synth.span_tables(w.seed, layer, lens, Hkv, w.rule)
    T = int(cu[-1])
    k = np.zeros((max(T, 1), Hkv, D), dtype=np.uint16)
    v = np.zeros_like(k)
    lib = synth.host()
    st = np.ascontiguousarray(st, dtype=np.int32)
    sg = np.ascontiguousarray(sg, dtype=np.float32)

    def fill(b):
        L = int(lens[b])
        for h in range(Hkv):
            p = b * Hkv + h
            for arr, stream in ((k, synth.STREAM_K), (v, synth.STREAM_V)):
                dst = arr.ctypes.data + ((int(cu[b]) * Hkv + h) * D) * 2
                lib.synth_fill_pair(w.seed, stream, layer, b, h, L, D, int(n[p]),
                                    st.ctypes.data + p * synth.MAX_SPANS * 4,
                                    sg.ctypes.data + p * synth.MAX_SPANS * 4, dst, Hkv * D)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(B)))
    q = synth.fill_heads(w.seed, synth.STREAM_Q, layer, B, w.hq, 1.0)
    kn = synth.fill_heads(w.seed, synth.STREAM_KNEW, layer, B, Hkv, 0.15)
    vn = synth.fill_heads(w.seed, synth.STREAM_VNEW, layer, B, Hkv, 0.15)
    return HostLayer(lens, cu, bt, nb, k[:T], v[:T], q, kn, vn)


def oracle_layer(w: configs.Workload, hl: HostLayer) -> HostLayer:
    """The oracle's compression of every request into pools laid out like the GPU's (same block
    table), and its fp64 decode attention of every request and query head."""
    lib = oracle.lib()
    B, Hq, Hkv, bs = w.batch, w.hq, w.hkv, w.block_size
    mb = hl.bt.shape[1]
    kp = np.zeros((hl.num_blocks, Hkv, bs, D), dtype=np.uint8)
    vp = np.zeros_like(kp)
    table = np.zeros((B, Hkv), dtype=oracle.SEG_DTYPE)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    k = np.ascontiguousarray(hl.k)
    v = np.ascontiguousarray(hl.v)
    bt = np.ascontiguousarray(hl.bt, dtype=np.int32)
    lens = np.ascontiguousarray(hl.lens, dtype=np.int32)
    cus = [np.array([0, int(L)], dtype=np.int32) for L in lens]

    def one(b):
        row = int(hl.cu[b]) * Hkv * D * 2
        lib.oracle_compress_ex(k.ctypes.data + row, v.ctypes.data + row, cus[b].ctypes.data, 1, Hkv, bs,
                               bt.ctypes.data + b * mb * 4, mb, oracle.MAX_SEG, ctypes.c_float(0.0),
                               kp.ctypes.data, vp.ctypes.data, table.ctypes.data + b * Hkv * REC)
        lib.oracle_paged_decode_attn(hl.q.ctypes.data + b * Hq * D * 2, hl.knew.ctypes.data + b * Hkv * D * 2,
                                     hl.vnew.ctypes.data + b * Hkv * D * 2, kp.ctypes.data, vp.ctypes.data,
                                     table.ctypes.data + b * Hkv * REC, bt.ctypes.data + b * mb * 4,
                                     lens.ctypes.data + b * 4, 1, Hq, Hkv, bs, mb,
                                     out.ctypes.data + b * Hq * D * 8)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(B)))
    hl.kp, hl.vp, hl.table, hl.out = kp, vp, table, out
    return hl
