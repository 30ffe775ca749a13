"""The C ABI on the host: the library loads, exports every function include/dgq.h declares,
rejects bad arguments before any launch, and keeps the block pool consistent.  CPU only."""
import ctypes
import os
import re

import numpy as np
import pytest

from int8_group_quantized_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, INVALID, UNSUPPORTED, WORKSPACE, POOL_EXHAUSTED = 0, -1, -2, -3, -5


@pytest.fixture(scope="module")
def L():
    _build.build()
    import int8_group_quantized_gb300 as dgq
    return dgq.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dgq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(dgq_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"dgq_compress", "dgq_paged_decode_attn", "dgq_pool_alloc"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert L.dgq_status_str(s)
    assert L.dgq_status_str(-99) == b"unknown status"


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced: checks fail first


def _compress(L, **kw):
    a = dict(k=FAKE, v=FAKE, T=337, cu=FAKE, batch=2, max_seqlen=300, hkv=2, d=128, bs=16, bt=FAKE,
             max_blocks=19, kp=FAKE, vp=FAKE, nb=32, table=FAKE, ws=FAKE, wsb=1 << 30, stream=0)
    a.update(kw)
    return L.dgq_compress(a["k"], a["v"], a["T"], a["cu"], a["batch"], a["max_seqlen"], a["hkv"], a["d"], a["bs"],
                          a["bt"], a["max_blocks"], a["kp"], a["vp"], a["nb"], a["table"], a["ws"], a["wsb"],
                          a["stream"])


def test_compress_rejects_bad_arguments_before_launch(L):
    assert _compress(L, d=64) == UNSUPPORTED
    assert _compress(L, bs=8) == UNSUPPORTED
    assert _compress(L, bs=128) == UNSUPPORTED
    assert _compress(L, k=0) == INVALID
    assert _compress(L, table=0) == INVALID
    assert _compress(L, k=FAKE + 2) == INVALID           # misaligned
    assert _compress(L, batch=0) == INVALID
    assert _compress(L, batch=8193) == INVALID            # above the per-call limit of 8192 requests
    assert _compress(L, max_seqlen=305) == INVALID       # > max_blocks * bs
    assert _compress(L, T=-1) == INVALID
    assert _compress(L, ws=0) == WORKSPACE
    need = L.dgq_compress_workspace_size(2, 300, 2)
    assert need > 0
    assert _compress(L, wsb=need - 1) == WORKSPACE


def test_compress_ex_rejects_bad_settings(L):
    import ctypes
    from int8_group_quantized_gb300 import CompressOptions
    L.dgq_compress_ex.restype = ctypes.c_int

    def call(mg, mv):
        o = CompressOptions(mg, mv)
        return L.dgq_compress_ex(FAKE, FAKE, 300, FAKE, 2, 300, 2, 128, 16, FAKE, 19, FAKE, FAKE, 64, FAKE, FAKE,
                                 1 << 30, ctypes.byref(o), None)
    for mg, mv in ((0, 0.0), (6, 0.0), (-1, 0.0), (3, -0.5), (3, float("nan")), (3, float("inf"))):
        assert call(mg, mv) == INVALID, (mg, mv)


def _attn(L, **kw):
    a = dict(q=FAKE, kn=FAKE, vn=FAKE, kp=FAKE, vp=FAKE, table=FAKE, bt=FAKE, lens=FAKE, max_seqlen=300,
             batch=2, hq=4, hkv=2, d=128, bs=16, max_blocks=19, nb=32, out=FAKE, ws=FAKE, wsb=1 << 30, stream=0)
    a.update(kw)
    return L.dgq_paged_decode_attn(a["q"], a["kn"], a["vn"], a["kp"], a["vp"], a["table"], a["bt"], a["lens"],
                                   a["max_seqlen"], a["batch"], a["hq"], a["hkv"], a["d"], a["bs"],
                                   a["max_blocks"], a["nb"], a["out"], a["ws"], a["wsb"], a["stream"])


def test_attn_rejects_bad_arguments_before_launch(L):
    assert _attn(L, d=256) == UNSUPPORTED
    assert _attn(L, bs=48) == UNSUPPORTED
    assert _attn(L, hq=6, hkv=4) == INVALID              # Hq not a multiple of Hkv
    assert _attn(L, hq=48, hkv=3) == UNSUPPORTED         # G = 16
    assert _attn(L, q=0) == INVALID
    assert _attn(L, out=FAKE + 8) == INVALID
    assert _attn(L, max_seqlen=400) == INVALID
    assert _attn(L, batch=-1) == INVALID


def _append(L, **kw):
    a = dict(kn=FAKE, vn=FAKE, batch=2, hkv=2, d=128, bs=16, bt=FAKE, max_blocks=19, kp=FAKE, vp=FAKE, nb=32,
             table=FAKE, ws=FAKE, wsb=256, stream=0)
    a.update(kw)
    return L.dgq_append(a["kn"], a["vn"], a["batch"], a["hkv"], a["d"], a["bs"], a["bt"], a["max_blocks"], a["kp"],
                        a["vp"], a["nb"], a["table"], a["ws"], a["wsb"], a["stream"])


def test_append_rejects_bad_arguments_before_launch(L):
    assert L.dgq_append_workspace_size() == 256
    assert _append(L, d=64) == UNSUPPORTED
    assert _append(L, bs=24) == UNSUPPORTED
    assert _append(L, kn=0) == INVALID
    assert _append(L, table=FAKE + 4) == INVALID         # misaligned
    assert _append(L, batch=0) == INVALID
    assert _append(L, max_blocks=0) == INVALID
    assert _append(L, ws=0) == WORKSPACE
    assert _append(L, wsb=255) == WORKSPACE
    # the split variant needs V's record table
    args = (FAKE, FAKE, 2, 2, 128, 16, FAKE, 19, FAKE, FAKE, 32, FAKE)
    assert L.dgq_append_split(*args, 0, FAKE, 256, 0) == INVALID
    assert L.dgq_append_split(*args, FAKE + 4, FAKE, 256, 0) == INVALID
    assert L.dgq_append_split(FAKE, FAKE, 2, 2, 64, 16, FAKE, 19, FAKE, FAKE, 32, FAKE, FAKE, FAKE, 256,
                              0) == UNSUPPORTED
    # the variant that reports re-segmentation bits: same checks, plus an aligned flags array
    assert L.dgq_append_ex(*args, FAKE + 4, FAKE, 256, 0) == INVALID
    assert L.dgq_append_ex(FAKE, FAKE, 2, 2, 64, 16, FAKE, 19, FAKE, FAKE, 32, FAKE, FAKE, FAKE, 256,
                           0) == UNSUPPORTED
    assert L.dgq_append_ex(*args, FAKE, 0, 256, 0) == WORKSPACE


def _encode(L, **kw):
    a = dict(fmt=1, k=FAKE, v=FAKE, T=337, cu=FAKE, batch=2, max_seqlen=300, hkv=2, d=128, bs=16, bt=FAKE,
             max_blocks=19, kp=FAKE, vp=FAKE, nb=32, table=FAKE, kpar=FAKE, vpar=FAKE, ws=FAKE, wsb=1 << 20, stream=0)
    a.update(kw)
    return L.dgq_encode_format(a["fmt"], a["k"], a["v"], a["T"], a["cu"], a["batch"], a["max_seqlen"], a["hkv"],
                               a["d"], a["bs"], a["bt"], a["max_blocks"], a["kp"], a["vp"], a["nb"], a["table"],
                               a["kpar"], a["vpar"], a["ws"], a["wsb"], a["stream"])


def test_encode_format_rejects_bad_arguments_before_launch(L):
    for fmt in (0, 4, -1):                               # DGQ itself is dgq_compress; unknown ids
        assert _encode(L, fmt=fmt) == INVALID, fmt
    assert _encode(L, kpar=0) == INVALID                 # fixed groups need their parameter arrays
    assert _encode(L, vpar=FAKE + 4) == INVALID
    assert _encode(L, d=64) == UNSUPPORTED
    assert _encode(L, bs=8) == UNSUPPORTED
    assert _encode(L, k=0) == INVALID
    assert _encode(L, T=-1) == INVALID
    assert _encode(L, max_seqlen=305) == INVALID         # > max_blocks * bs
    assert _encode(L, ws=0) == WORKSPACE
    need = L.dgq_encode_format_workspace_size(2, 2)
    assert need >= 256 + 2 * 2 * 8
    assert _encode(L, wsb=need - 1) == WORKSPACE
    assert L.dgq_encode_format_workspace_size(0, 2) == 0


def test_attn_format_rejects_bad_arguments_before_launch(L):
    def call(fmt, kpar=FAKE, vpar=FAKE, d=128):
        return L.dgq_paged_decode_attn_format(fmt, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, kpar, vpar, FAKE, FAKE, 300,
                                              2, 4, 2, d, 16, 19, 32, FAKE, FAKE, 1 << 30, 0)
    assert call(5) == INVALID
    assert call(-1) == INVALID
    assert call(1, kpar=0) == INVALID                    # fixed groups need their parameter arrays
    assert call(1, vpar=FAKE + 8) == INVALID
    for fmt in (0, 1, 2, 3):
        assert call(fmt, d=64) == UNSUPPORTED, fmt


def test_prefill_calls_reject_bad_arguments_before_launch(L):
    def stats(**kw):
        a = dict(k=FAKE, v=FAKE, nsrc=32, sbt=FAKE, msrc=19, beg=FAKE, end=FAKE, batch=2, max_seqlen=300, hkv=2,
                 d=128, bs=16, st=FAKE, mw=19, flags=0, ws=FAKE, wsb=1 << 20)
        a.update(kw)
        return L.dgq_prefill_chunk_stats(a["k"], a["v"], a["nsrc"], a["sbt"], a["msrc"], a["beg"], a["end"],
                                         a["batch"], a["max_seqlen"], a["hkv"], a["d"], a["bs"], a["st"], a["mw"],
                                         a["flags"], a["ws"], a["wsb"], 0)

    def finish(**kw):
        a = dict(k=FAKE, v=FAKE, nsrc=32, sbt=FAKE, msrc=19, lens=FAKE, batch=2, max_seqlen=300, hkv=2, d=128,
                 bs=16, st=FAKE, mw=19, bt=FAKE, mb=19, kp=FAKE, vp=FAKE, nb=32, table=FAKE, vtable=None, ws=FAKE,
                 wsb=1 << 20)
        a.update(kw)
        return L.dgq_prefill_finish(a["k"], a["v"], a["nsrc"], a["sbt"], a["msrc"], a["lens"], a["batch"],
                                    a["max_seqlen"], a["hkv"], a["d"], a["bs"], a["st"], a["mw"], a["bt"], a["mb"],
                                    a["kp"], a["vp"], a["nb"], a["table"], a["vtable"], None, a["ws"], a["wsb"], 0)
    for call in (stats, finish):
        assert call(d=64) == UNSUPPORTED
        assert call(bs=48) == UNSUPPORTED
        assert call(k=0) == INVALID
        assert call(st=0) == INVALID
        assert call(st=FAKE + 4) == INVALID                  # misaligned statistics array
        assert call(mw=18) == INVALID                        # fewer windows than ceil(300 / 16)
        assert call(max_seqlen=305) == INVALID               # > max_src_blocks * bs
        assert call(batch=0) == INVALID
        assert call(ws=0) == WORKSPACE
        assert call(wsb=L.dgq_prefill_workspace_size(2, 2) - 1) == WORKSPACE
    assert stats(beg=0) == INVALID
    assert stats(flags=2) == INVALID                     # unknown flag bits
    assert finish(vtable=FAKE + 8) == INVALID            # misaligned V record table
    assert finish(lens=0) == INVALID
    assert finish(mb=18) == INVALID                          # destination table too short for 300 tokens
    assert finish(table=FAKE + 8) == INVALID

    def finish_ex(flags=FAKE, d=128, ws=FAKE):
        return L.dgq_prefill_finish_ex(FAKE, FAKE, 32, FAKE, 19, FAKE, 2, 300, 2, d, 16, FAKE, 19, FAKE, 19, FAKE,
                                       FAKE, 32, FAKE, None, None, flags, 3, ws, 1 << 20, 0)
    assert finish_ex(flags=FAKE + 4) == INVALID           # misaligned flags
    assert finish_ex(d=64) == UNSUPPORTED
    assert finish_ex(ws=0) == WORKSPACE
    assert L.dgq_prefill_workspace_size(2, 2) == 256 + 2 * 2 * 2 * 128

    def split(vtable=FAKE, d=128):
        return L.dgq_paged_decode_attn_split(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, vtable, FAKE, FAKE, 300, 2, 4, 2,
                                             d, 16, 19, 32, FAKE, FAKE, 1 << 30, 0)
    assert split(vtable=0) == INVALID
    assert split(vtable=FAKE + 4) == INVALID
    assert split(d=64) == UNSUPPORTED


def test_workspace_size_is_monotone(L):
    a = L.dgq_compress_workspace_size(4, 1000, 8)
    b = L.dgq_compress_workspace_size(4, 2000, 8)
    c = L.dgq_compress_workspace_size(8, 2000, 8)
    assert 0 < a < b < c
    assert L.dgq_compress_workspace_size(0, 10, 1) == 0


def test_block_pool_alloc_free_exhaust():
    import int8_group_quantized_gb300 as dgq
    _build.build()
    pool = dgq.BlockPool(10)
    assert pool.num_free() == 10
    a = pool.alloc(4)
    assert a == [0, 1, 2, 3] and pool.num_free() == 6
    with pytest.raises(dgq.DGQError) as e:
        pool.alloc(7)  # all or nothing
    assert e.value.status == POOL_EXHAUSTED and pool.num_free() == 6
    b = pool.alloc(6)
    assert sorted(a + b) == list(range(10)) and pool.num_free() == 0
    pool.free([3, 1])
    assert pool.num_free() == 2
    with pytest.raises(dgq.DGQError):
        pool.free([3])        # already free
    with pytest.raises(dgq.DGQError):
        pool.free([0, 0])     # duplicate id: nothing freed
    with pytest.raises(dgq.DGQError):
        pool.free([10])       # out of range
    assert pool.num_free() == 2
    assert sorted(pool.alloc(2)) == [1, 3]
    pool.close()


def test_block_pool_table_rows():
    import int8_group_quantized_gb300 as dgq
    _build.build()
    pool = dgq.BlockPool(32)
    table = np.full((2, 19), -1, dtype=np.int32)
    pool.alloc_table_row(37, 16, table, 0)
    pool.alloc_table_row(300, 16, table, 1)
    used = np.concatenate([table[0, :3], table[1, :19]])
    assert len(set(used.tolist())) == 22 and pool.num_free() == 10
    assert np.all(table[0, 3:] == 0)
    with pytest.raises(dgq.DGQError):
        pool.alloc_table_row(400, 16, table, 0)  # 25 blocks > 19 columns
