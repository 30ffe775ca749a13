"""The five synthetic workloads (shapes, seeds, length mixes, block placement).

Shapes follow the sources: Llama-3-8B-like decode (32 layers, 32 query heads, 8 KV heads,
head dim 128) as in the DGQ article's storage example (section 3.3), 100 concurrent
requests of up to 2048 tokens with d_model 4096 / 32 heads as in the PagedAttention
article's memory model, block size 64 for sequences past 32K as in that article's
long-context configuration, and a 128K single sequence as in the DGQ article's headline
case.  No dataset or trained weight is used anywhere: every tensor is drawn by `synth`.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import (RULE_PERM5, RULE_SET3, RULE_U, STREAM_META, hash64, key, permutation)

D = 128


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    layers: int
    batch: int
    hq: int
    hkv: int
    block_size: int
    rule: int           # variance-span rule for K/V (synth RULE_*)
    lens: tuple         # ("fixed", L0, L1, ...) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    placement: str      # "perm32" | "contiguous" | "shuffled"
    head_dim: int = D


WORKLOADS = {
    1: Workload("tiny b2 hq4 hkv2 L{37,300} bs16", 0, 1, 2, 4, 2, 16, RULE_SET3,
                ("fixed", 37, 300), "perm32"),
    2: Workload("llama3-8b decode b32 L2048 bs16", 1, 32, 32, 32, 8, 16, RULE_U,
                ("fixed", 2048), "contiguous"),
    3: Workload("mha decode b100 L~U[256,2048] bs16", 2, 32, 100, 32, 32, 16, RULE_U,
                ("uniform", 256, 2048), "shuffled"),
    4: Workload("long context b1 L131072 bs64", 3, 32, 1, 32, 8, 64, RULE_PERM5,
                ("fixed", 131072), "contiguous"),
    5: Workload("mixed serving b64 L~logU[128,32768] bs64", 4, 32, 64, 32, 8, 64, RULE_U,
                ("loguniform", 128, 32768), "shuffled"),
    # the prefill compress case that rides with workload 5
    "5p": Workload("prefill compress b1 L16384 bs64", 4, 32, 1, 32, 8, 64, RULE_U,
                   ("fixed", 16384), "contiguous"),
}


def seq_lens(w: Workload) -> np.ndarray:
    kind = w.lens[0]
    if kind == "fixed":
        vals = list(w.lens[1:])
        if len(vals) == 1:
            vals = vals * w.batch
        assert len(vals) == w.batch
        return np.asarray(vals, dtype=np.int32)
    lo, hi = w.lens[1], w.lens[2]
    out = np.zeros(w.batch, dtype=np.int32)
    for b in range(w.batch):
        h = hash64(key(w.seed, STREAM_META, 0, b, 0), 0)
        if kind == "uniform":
            out[b] = lo + h % (hi - lo + 1)
        else:  # log-uniform in [lo, hi)
            u = (h >> 11) * 2.0 ** -53
            out[b] = min(hi, int(lo * (hi / lo) ** u))
    return out


def block_tables(w: Workload, lens: np.ndarray):
    """Returns (block_tables [B, max_blocks] int32, num_blocks).  Unused entries are 0."""
    bs = w.block_size
    nblk = [(int(L) + bs - 1) // bs for L in lens]
    max_blocks = max(1, max(nblk))
    total = sum(nblk)
    if w.placement == "perm32":
        num_blocks = 32
        assert total <= num_blocks
        order = permutation(w.seed, STREAM_META, num_blocks)
    elif w.placement == "contiguous":
        num_blocks = max(total, 1)
        order = np.arange(num_blocks, dtype=np.int32)
    else:
        num_blocks = max(total, 1)
        order = permutation(w.seed, STREAM_META, num_blocks)
    bt = np.zeros((w.batch, max_blocks), dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = order[off:off + n]
        off += n
    return bt, num_blocks


def cu_seqlens(lens: np.ndarray) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    return cu
