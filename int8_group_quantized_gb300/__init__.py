"""DGQ INT8 paged KV cache on GB300: Python binding of ``libdgq.so``.

Argument marshalling only.  Every step of compression and decode attention runs in the
library's CUDA kernels; the functions here take torch CUDA tensors (or raw device
addresses), pass pointers and sizes through the C ABI declared in ``include/dgq.h`` and
raise :class:`DGQError` on a non-OK status.  There is no CPU fallback: if ``libdgq.so``
is missing the import of any entry point fails loudly.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

HEAD_DIM = 128
MAX_SEG = 5
SEG_RECORD_BYTES = 128

# dgq_format: the method's own encoding and the comparison encodings on the same cache layout
FORMAT_DGQ = 0
FORMAT_FIXED64 = 1
FORMAT_SYM_INT8 = 2
FORMAT_FP8_E4M3 = 3
FORMATS = {"dgq": FORMAT_DGQ, "fixed64": FORMAT_FIXED64, "sym_int8": FORMAT_SYM_INT8, "fp8_e4m3": FORMAT_FP8_E4M3}

__all__ = [
    "DGQError", "lib", "dgq_compress", "dgq_compress_paged", "dgq_compress_workspace_size", "dgq_append",
    "dgq_append_workspace_size",
    "dgq_paged_decode_attn", "dgq_encode_format", "dgq_encode_format_workspace_size",
    "dgq_paged_decode_attn_format", "FORMATS", "dgq_prefill_workspace_size", "dgq_prefill_chunk_stats",
    "dgq_prefill_finish", "dgq_paged_decode_attn_split", "dgq_append_split", "dgq_append_ex",
    "dgq_prefill_finish_ex", "RESEG_WINDOW", "RESEG_NGROUPS",
    "dgq_attn_workspace_size", "dgq_workspace_init", "dgq_workspace_error", "BlockPool",
    "seg_record_dtype",
]


class DGQError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = lib().dgq_status_str(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what}: {msg} (status {status})" if what else f"{msg} (status {status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libdgq.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is not built: run __graft_entry__.build() first")
        L = ctypes.CDLL(_build.LIB)
        P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.dgq_status_str.argtypes = [ctypes.c_int]
        L.dgq_status_str.restype = ctypes.c_char_p
        L.dgq_compress.argtypes = [P, P, i32, P, i32, i32, i32, i32, i32, P, i32, P, P, i32, P, P, sz, P]
        L.dgq_compress.restype = ctypes.c_int
        L.dgq_compress_ex.argtypes = [P, P, i32, P, i32, i32, i32, i32, i32, P, i32, P, P, i32, P, P, sz,
                                      ctypes.POINTER(CompressOptions), P]
        L.dgq_compress_ex.restype = ctypes.c_int
        L.dgq_compress_paged.argtypes = [P, P, i32, P, i32, P, i32, i32, i32, i32, i32, P, i32, P, P, i32, P, P, sz,
                                         ctypes.POINTER(CompressOptions), P]
        L.dgq_compress_paged.restype = ctypes.c_int
        L.dgq_compress_workspace_size.argtypes = [i32, i32, i32]
        L.dgq_compress_workspace_size.restype = sz
        L.dgq_paged_decode_attn.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                            P, P, sz, P]
        L.dgq_paged_decode_attn.restype = ctypes.c_int
        L.dgq_paged_decode_attn_noalloc.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                    i32, P, P]
        L.dgq_paged_decode_attn_noalloc.restype = ctypes.c_int
        L.dgq_encode_format.argtypes = [i32, P, P, i32, P, i32, i32, i32, i32, i32, P, i32, P, P, i32, P, P, P, P,
                                        sz, P]
        L.dgq_encode_format.restype = ctypes.c_int
        L.dgq_encode_format_workspace_size.argtypes = [i32, i32]
        L.dgq_encode_format_workspace_size.restype = sz
        L.dgq_paged_decode_attn_format.argtypes = [i32, P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                                   i32, i32, P, P, sz, P]
        L.dgq_paged_decode_attn_format.restype = ctypes.c_int
        L.dgq_prefill_workspace_size.argtypes = [i32, i32]
        L.dgq_prefill_workspace_size.restype = sz
        L.dgq_prefill_chunk_stats.argtypes = [P, P, i32, P, i32, P, P, i32, i32, i32, i32, i32, P, i32, i32, P, sz,
                                              P]
        L.dgq_prefill_chunk_stats.restype = ctypes.c_int
        L.dgq_prefill_finish.argtypes = [P, P, i32, P, i32, P, i32, i32, i32, i32, i32, P, i32, P, i32, P, P, i32, P,
                                         P, P, P, sz, P]
        L.dgq_prefill_finish_ex.argtypes = [P, P, i32, P, i32, P, i32, i32, i32, i32, i32, P, i32, P, i32, P, P, i32,
                                            P, P, P, P, i32, P, sz, P]
        L.dgq_prefill_finish_ex.restype = ctypes.c_int
        L.dgq_paged_decode_attn_split.argtypes = [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                  i32, P, P, sz, P]
        L.dgq_paged_decode_attn_split.restype = ctypes.c_int
        L.dgq_prefill_finish.restype = ctypes.c_int
        L.dgq_append.argtypes = [P, P, i32, i32, i32, i32, P, i32, P, P, i32, P, P, sz, P]
        L.dgq_append_ex.argtypes = [P, P, i32, i32, i32, i32, P, i32, P, P, i32, P, P, P, sz, P]
        L.dgq_append_ex.restype = ctypes.c_int
        L.dgq_append_split.argtypes = [P, P, i32, i32, i32, i32, P, i32, P, P, i32, P, P, P, sz, P]
        L.dgq_append_split.restype = ctypes.c_int
        L.dgq_append.restype = ctypes.c_int
        L.dgq_append_workspace_size.argtypes = []
        L.dgq_append_workspace_size.restype = sz
        L.dgq_attn_workspace_size.argtypes = [i32, i32, i32, i32]
        L.dgq_attn_workspace_size.restype = sz
        L.dgq_workspace_init.argtypes = [P, sz, P]
        L.dgq_workspace_init.restype = ctypes.c_int
        L.dgq_workspace_error.argtypes = [P, P, ctypes.POINTER(i32)]
        L.dgq_workspace_error.restype = ctypes.c_int
        L.dgq_pool_create.argtypes = [i32]
        L.dgq_pool_create.restype = P
        L.dgq_pool_destroy.argtypes = [P]
        L.dgq_pool_destroy.restype = None
        L.dgq_pool_alloc.argtypes = [P, i32, P]
        L.dgq_pool_alloc.restype = ctypes.c_int
        L.dgq_pool_free.argtypes = [P, P, i32]
        L.dgq_pool_free.restype = ctypes.c_int
        L.dgq_pool_num_free.argtypes = [P]
        L.dgq_pool_num_free.restype = i32
        L.dgq_pool_alloc_table_row.argtypes = [P, i32, i32, P, i32, i32]
        L.dgq_pool_alloc_table_row.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(x) -> int:
    """Device address of a torch tensor (or a raw integer address)."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _nbytes(x) -> int:
    return x.numel() * x.element_size()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != 0:
        raise DGQError(status, what)


def seg_record_dtype():
    """numpy structured dtype of one dgq_seg_record (128 bytes)."""
    import numpy as np
    dt = np.dtype([("n_seg", "<i4"), ("seq_len", "<i4"), ("start", "<i4", (MAX_SEG,)),
                   ("k_min", "<f4", (MAX_SEG,)), ("k_scale", "<f4", (MAX_SEG,)),
                   ("v_min", "<f4", (MAX_SEG,)), ("v_scale", "<f4", (MAX_SEG,)),
                   ("k_inv_last", "<f4"), ("v_inv_last", "<f4"), ("pad", "<i4", (3,))])
    assert dt.itemsize == SEG_RECORD_BYTES
    return dt


def dgq_compress_workspace_size(batch: int, max_seqlen: int, num_kv_heads: int) -> int:
    return int(lib().dgq_compress_workspace_size(batch, max_seqlen, num_kv_heads))


def dgq_attn_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, max_seqlen: int) -> int:
    return int(lib().dgq_attn_workspace_size(batch, num_q_heads, num_kv_heads, max_seqlen))


def dgq_workspace_init(workspace, stream=None) -> None:
    _check(lib().dgq_workspace_init(_ptr(workspace), _nbytes(workspace), _stream(stream)), "dgq_workspace_init")


def dgq_workspace_error(workspace, stream=None) -> int:
    """Synchronises the stream; returns the device-side error word (0 = none)."""
    code = ctypes.c_int32(0)
    st = lib().dgq_workspace_error(_ptr(workspace), _stream(stream), ctypes.byref(code))
    if st not in (0, -6):
        raise DGQError(st, "dgq_workspace_error")
    return int(code.value)


class CompressOptions(ctypes.Structure):
    """dgq_compress_options: group-selection settings (segment cap 1..5, variance floor >= 0)."""
    _fields_ = [("max_groups", ctypes.c_int32), ("min_var", ctypes.c_float)]


def dgq_compress(k, v, cu_seqlens, max_seqlen, block_size, block_tables, k_pool, v_pool, seg_table,
                 workspace, stream=None, max_groups=MAX_SEG, min_var=0.0) -> None:
    """k, v: bf16 [T, Hkv, 128]; cu_seqlens int32 [B+1]; block_tables int32 [B, max_blocks];
    k_pool, v_pool uint8 [num_blocks, Hkv, bs, 128]; seg_table uint8 [B, Hkv, 128] (records);
    workspace uint8 (dgq_compress_workspace_size bytes).  All CUDA tensors.  max_groups /
    min_var: group-selection settings (dgq_compress_ex); the defaults are the plain method."""
    B = cu_seqlens.shape[0] - 1
    Hkv = k.shape[1]
    args = (_ptr(k), _ptr(v), k.shape[0], _ptr(cu_seqlens), B, int(max_seqlen), Hkv, k.shape[2], int(block_size),
            _ptr(block_tables), block_tables.shape[1], _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(seg_table),
            _ptr(workspace), _nbytes(workspace))
    if max_groups == MAX_SEG and min_var == 0.0:
        _check(lib().dgq_compress(*args, _stream(stream)), "dgq_compress")
    else:
        opts = CompressOptions(int(max_groups), float(min_var))
        _check(lib().dgq_compress_ex(*args, ctypes.byref(opts), _stream(stream)), "dgq_compress_ex")


def dgq_append_workspace_size() -> int:
    return int(lib().dgq_append_workspace_size())


def dgq_append(k_new, v_new, block_size, block_tables, k_pool, v_pool, seg_table, workspace, stream=None) -> None:
    """k_new, v_new bf16 [B, Hkv, 128]; block_tables int32 [B, max_blocks]; pools uint8
    [num_blocks, Hkv, bs, 128] and seg_table uint8 [B, Hkv, 128] updated in place; workspace
    uint8 (dgq_append_workspace_size bytes).  All CUDA tensors."""
    B, Hkv, D = k_new.shape
    _check(lib().dgq_append(_ptr(k_new), _ptr(v_new), B, Hkv, D, int(block_size), _ptr(block_tables),
                            block_tables.shape[1], _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(seg_table),
                            _ptr(workspace), _nbytes(workspace), _stream(stream)), "dgq_append")


RESEG_WINDOW = 1   # dgq_append_ex: the appended token completed a 16-token window
RESEG_NGROUPS = 2  # the length reached a threshold of the n_groups rule (2048, 16384)


def dgq_append_ex(k_new, v_new, block_size, block_tables, k_pool, v_pool, seg_table, resegment_flags, workspace,
                  stream=None) -> None:
    """dgq_append, writing each pair's re-segmentation bits into resegment_flags (int32 CUDA tensor
    [B, Hkv], or None)."""
    B, Hkv, D = k_new.shape
    _check(lib().dgq_append_ex(_ptr(k_new), _ptr(v_new), B, Hkv, D, int(block_size), _ptr(block_tables),
                               block_tables.shape[1], _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(seg_table),
                               _ptr(resegment_flags), _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "dgq_append_ex")


def dgq_append_split(k_new, v_new, block_size, block_tables, k_pool, v_pool, k_seg_table, v_seg_table, workspace,
                     stream=None) -> None:
    """dgq_append for a cache with independent V segmentation (K's and V's record tables)."""
    B, Hkv, D = k_new.shape
    _check(lib().dgq_append_split(_ptr(k_new), _ptr(v_new), B, Hkv, D, int(block_size), _ptr(block_tables),
                                  block_tables.shape[1], _ptr(k_pool), _ptr(v_pool), k_pool.shape[0],
                                  _ptr(k_seg_table), _ptr(v_seg_table), _ptr(workspace), _nbytes(workspace),
                                  _stream(stream)), "dgq_append_split")


def dgq_compress_paged(k_src, v_src, src_block_tables, cu_seqlens, max_seqlen, block_size, block_tables, k_pool,
                       v_pool, seg_table, workspace, stream=None, max_groups=MAX_SEG, min_var=0.0) -> None:
    """k_src, v_src: bf16 paged cache [num_src_blocks, Hkv, bs, 128]; src_block_tables int32
    [B, max_src_blocks]; cu_seqlens int32 [B+1] (lengths only); the rest as dgq_compress."""
    B = cu_seqlens.shape[0] - 1
    Hkv = k_src.shape[1]
    opts = CompressOptions(int(max_groups), float(min_var))
    _check(lib().dgq_compress_paged(_ptr(k_src), _ptr(v_src), k_src.shape[0], _ptr(src_block_tables),
                                    src_block_tables.shape[1], _ptr(cu_seqlens), B, int(max_seqlen), Hkv,
                                    k_src.shape[3], int(block_size), _ptr(block_tables), block_tables.shape[1],
                                    _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(seg_table), _ptr(workspace),
                                    _nbytes(workspace), ctypes.byref(opts), _stream(stream)), "dgq_compress_paged")


def dgq_paged_decode_attn(q, k_new, v_new, k_pool, v_pool, seg_table, block_tables, seq_lens, max_seqlen,
                          out, workspace, stream=None) -> None:
    """q bf16 [B, Hq, 128]; k_new, v_new bf16 [B, Hkv, 128]; pools / seg_table / block_tables as
    written by dgq_compress; seq_lens int32 [B]; out bf16 [B, Hq, 128]."""
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    _check(lib().dgq_paged_decode_attn(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                       _ptr(seg_table), _ptr(block_tables), _ptr(seq_lens), int(max_seqlen),
                                       B, Hq, Hkv, D, k_pool.shape[2], block_tables.shape[1], k_pool.shape[0],
                                       _ptr(out), _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "dgq_paged_decode_attn")


def dgq_prefill_workspace_size(batch: int, num_kv_heads: int) -> int:
    return int(lib().dgq_prefill_workspace_size(batch, num_kv_heads))


PREFILL_V_VARIANCE = 1


def dgq_prefill_chunk_stats(k_src, v_src, src_block_tables, chunk_begin, chunk_end, max_seqlen, window_stats,
                            workspace, stream=None, v_variance=False) -> None:
    """Window statistics of tokens [chunk_begin[b], chunk_end[b]) of each request (int32 CUDA
    tensors [B]) from the bf16 paged cache k_src / v_src [num_src_blocks, Hkv, bs, 128] into
    window_stats fp32 [B, Hkv, max_windows, 8]; workspace: dgq_prefill_workspace_size bytes.
    v_variance: also V's mean variance (for independent V segmentation)."""
    B = chunk_begin.shape[0]
    _, Hkv, bs, D = k_src.shape
    _check(lib().dgq_prefill_chunk_stats(_ptr(k_src), _ptr(v_src), k_src.shape[0], _ptr(src_block_tables),
                                         src_block_tables.shape[1], _ptr(chunk_begin), _ptr(chunk_end), B,
                                         int(max_seqlen), Hkv, D, bs, _ptr(window_stats), window_stats.shape[2],
                                         PREFILL_V_VARIANCE if v_variance else 0, _ptr(workspace),
                                         _nbytes(workspace), _stream(stream)),
           "dgq_prefill_chunk_stats")


def dgq_prefill_finish(k_src, v_src, src_block_tables, seq_lens, max_seqlen, window_stats, block_tables, k_pool,
                       v_pool, seg_table, workspace, stream=None, max_groups=MAX_SEG, min_var=0.0,
                       v_seg_table=None) -> None:
    """Segmentation from window_stats and codes of every token [0, seq_lens[b]) into the INT8
    pools / records (as dgq_compress_paged with the same settings would write them).  With
    v_seg_table (uint8 [B, Hkv, 128]): independent V segmentation, V's records there."""
    B = seq_lens.shape[0]
    _, Hkv, bs, D = k_src.shape
    opts = CompressOptions(int(max_groups), float(min_var))
    _check(lib().dgq_prefill_finish(_ptr(k_src), _ptr(v_src), k_src.shape[0], _ptr(src_block_tables),
                                    src_block_tables.shape[1], _ptr(seq_lens), B, int(max_seqlen), Hkv, D, bs,
                                    _ptr(window_stats), window_stats.shape[2], _ptr(block_tables),
                                    block_tables.shape[1], _ptr(k_pool), _ptr(v_pool), k_pool.shape[0],
                                    _ptr(seg_table), _ptr(v_seg_table), ctypes.byref(opts), _ptr(workspace),
                                    _nbytes(workspace), _stream(stream)), "dgq_prefill_finish")


def dgq_prefill_finish_ex(k_src, v_src, src_block_tables, seq_lens, max_seqlen, window_stats, block_tables, k_pool,
                          v_pool, seg_table, workspace, pair_flags, flag_mask=RESEG_WINDOW | RESEG_NGROUPS,
                          stream=None, max_groups=MAX_SEG, min_var=0.0, v_seg_table=None) -> None:
    """dgq_prefill_finish for the requests with a pair whose pair_flags (int32 CUDA tensor [B, Hkv],
    e.g. from dgq_append_ex) meet flag_mask; every other request is left untouched."""
    B = seq_lens.shape[0]
    _, Hkv, bs, D = k_src.shape
    opts = CompressOptions(int(max_groups), float(min_var))
    _check(lib().dgq_prefill_finish_ex(_ptr(k_src), _ptr(v_src), k_src.shape[0], _ptr(src_block_tables),
                                       src_block_tables.shape[1], _ptr(seq_lens), B, int(max_seqlen), Hkv, D, bs,
                                       _ptr(window_stats), window_stats.shape[2], _ptr(block_tables),
                                       block_tables.shape[1], _ptr(k_pool), _ptr(v_pool), k_pool.shape[0],
                                       _ptr(seg_table), _ptr(v_seg_table), ctypes.byref(opts), _ptr(pair_flags),
                                       int(flag_mask), _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "dgq_prefill_finish_ex")


def dgq_paged_decode_attn_split(q, k_new, v_new, k_pool, v_pool, k_seg_table, v_seg_table, block_tables, seq_lens,
                                max_seqlen, out, workspace, stream=None) -> None:
    """dgq_paged_decode_attn over a cache with independent V segmentation (K's and V's record
    tables as dgq_prefill_finish wrote them)."""
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    _check(lib().dgq_paged_decode_attn_split(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                             _ptr(k_seg_table), _ptr(v_seg_table), _ptr(block_tables),
                                             _ptr(seq_lens), int(max_seqlen), B, Hq, Hkv, D, k_pool.shape[2],
                                             block_tables.shape[1], k_pool.shape[0], _ptr(out), _ptr(workspace),
                                             _nbytes(workspace), _stream(stream)), "dgq_paged_decode_attn_split")


def _format_id(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def dgq_encode_format_workspace_size(batch: int, num_kv_heads: int) -> int:
    return int(lib().dgq_encode_format_workspace_size(batch, num_kv_heads))


def dgq_encode_format(fmt, k, v, cu_seqlens, max_seqlen, block_size, block_tables, k_pool, v_pool, seg_table,
                      workspace, k_params=None, v_params=None, stream=None) -> None:
    """A comparison encoding ("fixed64", "sym_int8", "fp8_e4m3") of bf16 [T, Hkv, 128] rows into
    the paged cache; k_params / v_params fp32 [num_blocks, Hkv, bs, 4] for "fixed64" (else
    None); the other arguments as dgq_compress (workspace: dgq_encode_format_workspace_size)."""
    B = cu_seqlens.shape[0] - 1
    Hkv = k.shape[1]
    _check(lib().dgq_encode_format(_format_id(fmt), _ptr(k), _ptr(v), k.shape[0], _ptr(cu_seqlens), B,
                                   int(max_seqlen), Hkv, k.shape[2], int(block_size), _ptr(block_tables),
                                   block_tables.shape[1], _ptr(k_pool), _ptr(v_pool), k_pool.shape[0],
                                   _ptr(seg_table), _ptr(k_params), _ptr(v_params), _ptr(workspace),
                                   _nbytes(workspace), _stream(stream)), "dgq_encode_format")


def dgq_paged_decode_attn_format(fmt, q, k_new, v_new, k_pool, v_pool, seg_table, block_tables, seq_lens,
                                 max_seqlen, out, workspace, k_params=None, v_params=None, stream=None) -> None:
    """dgq_paged_decode_attn over a cache written in format `fmt` (a FORMATS key or id)."""
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    _check(lib().dgq_paged_decode_attn_format(_format_id(fmt), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
                                              _ptr(v_pool), _ptr(seg_table), _ptr(k_params), _ptr(v_params),
                                              _ptr(block_tables), _ptr(seq_lens), int(max_seqlen), B, Hq, Hkv, D,
                                              k_pool.shape[2], block_tables.shape[1], k_pool.shape[0], _ptr(out),
                                              _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "dgq_paged_decode_attn_format")


def dgq_paged_decode_attn_noalloc(q, k_new, v_new, k_pool, v_pool, seg_table, block_tables, seq_lens,
                                  max_seqlen, out, stream=None) -> None:
    """dgq_paged_decode_attn without a workspace: the scratch is the library's own fixed
    device array (for callers that cannot allocate).  Same arguments otherwise."""
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    _check(lib().dgq_paged_decode_attn_noalloc(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                               _ptr(seg_table), _ptr(block_tables), _ptr(seq_lens),
                                               int(max_seqlen), B, Hq, Hkv, D, k_pool.shape[2],
                                               block_tables.shape[1], k_pool.shape[0], _ptr(out), _stream(stream)),
           "dgq_paged_decode_attn_noalloc")


class BlockPool:
    """Host free list of physical block ids (dgq_pool_*)."""

    def __init__(self, num_blocks: int):
        self._h = lib().dgq_pool_create(num_blocks)
        if not self._h:
            raise DGQError(-1, "dgq_pool_create")

    def close(self) -> None:
        if self._h:
            lib().dgq_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, n: int) -> list[int]:
        buf = (ctypes.c_int32 * max(n, 1))()
        _check(lib().dgq_pool_alloc(self._h, n, buf), "dgq_pool_alloc")
        return list(buf[:n])

    def free(self, ids) -> None:
        ids = list(ids)
        buf = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(lib().dgq_pool_free(self._h, buf, len(ids)), "dgq_pool_free")

    def num_free(self) -> int:
        return int(lib().dgq_pool_num_free(self._h))

    def alloc_table_row(self, length: int, block_size: int, table, row: int) -> None:
        """table: C-contiguous int32 numpy array [rows, max_blocks]."""
        _check(lib().dgq_pool_alloc_table_row(self._h, length, block_size, table.ctypes.data, row,
                                              table.shape[1]), "dgq_pool_alloc_table_row")
