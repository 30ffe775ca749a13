"""Pins for the oracle's decode-step append: the new token of each (request, KV head) is
encoded with the last segment's min and 255 / (max - min), its codes held to [0, 255]; a
request with no token yet gets a one-token first segment.  Each check ties the oracle to a
closed form, an invariant or to its compress path on data where the segment is unchanged.
CPU only."""
import numpy as np
import pytest

import oracle

D = 128


def bf16_bits(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def bf16_float(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def empty_state(B, Hkv, bs, max_blocks, nb):
    kp = np.zeros((nb, Hkv, bs, D), dtype=np.uint8)
    vp = np.zeros_like(kp)
    table = np.zeros((B, Hkv), dtype=oracle.SEG_DTYPE)
    bt = np.arange(B * max_blocks, dtype=np.int32).reshape(B, max_blocks) % nb
    return kp, vp, table, bt


def test_first_token_is_its_own_segment():
    # n_seg == 0: the token alone sets min/max; its min -> 0, its max -> 255, and the codes
    # are the textbook per-tensor asymmetric uint8 codes of its 128 values
    rng = np.random.default_rng(1)
    kp, vp, table, bt = empty_state(1, 1, 16, 2, 2)
    xk = bf16_bits(rng.standard_normal(D).astype(np.float32) * 0.3)
    xv = bf16_bits(rng.standard_normal(D).astype(np.float32) * 2.0)
    assert oracle.append(xk[None, None], xv[None, None], 16, bt, kp, vp, table) == 0
    rec = table[0, 0]
    assert rec["n_seg"] == 1 and rec["seq_len"] == 1 and list(rec["start"]) == [0, 1, 1, 1, 1]
    for x, pool, mn_f, sc_f, inv_f in ((xk, kp, "k_min", "k_scale", "k_inv_last"),
                                       (xv, vp, "v_min", "v_scale", "v_inv_last")):
        f = bf16_float(x)
        mn, mx = np.float32(f.min()), np.float32(f.max())
        r = np.float32(mx - mn)
        assert rec[mn_f][0] == mn and rec[sc_f][0] == np.float32(r / np.float32(255))
        assert rec[inv_f] == np.float32(np.float32(255) / r)
        codes = pool[bt[0, 0], 0, 0]
        assert codes[np.argmin(f)] == 0 and codes[np.argmax(f)] == 255
        err = np.abs(mn + codes.astype(np.float64) * rec[sc_f][0] - f)
        assert err.max() <= 0.5 * rec[sc_f][0] * (1 + 2**-10) + 2**-22 * (abs(mn) + abs(mx))


def test_in_range_token_gets_the_codes_compress_gives_it():
    # 40 tokens: windows 0-1 quiet, window 2 loud -> one cut at 32 for 40 and for 41 tokens.
    # A 41st token inside segment 1's range leaves its min/max unchanged, so appending it to
    # the 40-token cache must give exactly the codes compressing all 41 tokens gives it.
    rng = np.random.default_rng(2)
    for trial in range(20):
        quiet = rng.standard_normal((32, D)).astype(np.float32) * 0.02
        loud = rng.standard_normal((9, D)).astype(np.float32) * 1.0
        kf = np.concatenate([quiet, loud])
        vf = rng.standard_normal((41, D)).astype(np.float32)
        vf[:40, 0], vf[:40, 1] = 5.0, -5.0       # V range fixed by earlier tokens
        kf[32, 0], kf[32, 1] = 4.0, -4.0         # K range of segment 1 fixed by token 32
        kf[40] = np.clip(kf[40], -3.9, 3.9)
        vf[40] = np.clip(vf[40], -4.9, 4.9)
        k, v = bf16_bits(kf), bf16_bits(vf)
        rec41, kc41, vc41 = oracle.compress_pair(k, v)
        assert list(rec41["start"][:rec41["n_seg"]]) == [0, 32]
        bs = 16
        cu = np.array([0, 40], dtype=np.int32)
        bt = np.array([[3, 0, 2, 1]], dtype=np.int32)
        kp, vp, table = oracle.compress(k[:40, None], v[:40, None], cu, 1, bs, bt, 4)
        assert oracle.append(k[40][None, None], v[40][None, None], bs, bt, kp, vp, table) == 0
        blk = bt[0, 40 // bs]
        assert np.array_equal(kp[blk, 0, 40 % bs], kc41[40])
        assert np.array_equal(vp[blk, 0, 40 % bs], vc41[40])
        got = table[0, 0]
        assert got["seq_len"] == 41 and list(got["start"]) == [0, 32, 41, 41, 41]
        for f in ("n_seg", "k_min", "k_scale", "v_min", "v_scale", "k_inv_last", "v_inv_last"):
            assert np.array_equal(got[f], rec41[f]), f


def test_out_of_range_values_clamp():
    k = bf16_bits(np.tile(np.linspace(-1.0, 1.0, D, dtype=np.float32), (16, 1)))
    cu = np.array([0, 16], dtype=np.int32)
    bt = np.array([[0, 1]], dtype=np.int32)
    kp, vp, table = oracle.compress(k[:, None], k[:, None], cu, 1, 16, bt, 2)
    x = np.zeros(D, dtype=np.float32)
    x[:4] = [7.0, 1.0, -1.0, -9.0]          # above max, at max, at min, below min
    xb = bf16_bits(x)
    assert oracle.append(xb[None, None], xb[None, None], 16, bt, kp, vp, table) == 0
    assert list(kp[1, 0, 0, :4]) == [255, 255, 0, 0]
    assert list(vp[1, 0, 0, :4]) == [255, 255, 0, 0]


def test_flat_last_segment_encodes_zero():
    k = np.tile(bf16_bits(np.full(D, 0.25)), (16, 1))
    cu = np.array([0, 16], dtype=np.int32)
    bt = np.array([[0, 1]], dtype=np.int32)
    kp, vp, table = oracle.compress(k[:, None], k[:, None], cu, 1, 16, bt, 2)
    assert table[0, 0]["k_inv_last"] == 0 and table[0, 0]["k_scale"][0] == 0
    x = bf16_bits(np.random.default_rng(3).standard_normal(D).astype(np.float32))
    oracle.append(x[None, None], x[None, None], 16, bt, kp, vp, table)
    assert np.all(kp[1, 0, 0] == 0) and np.all(vp[1, 0, 0] == 0)


def test_repeated_appends_walk_blocks_and_skip_without_a_column():
    # two requests x two heads, 37 appends from empty with bs 16 -> blocks 0, 1, 2 of each
    # row; a third request whose table has no column for its next slot is skipped
    rng = np.random.default_rng(4)
    B, Hkv, bs = 3, 2, 16
    nb = 9
    bt = np.array([[4, 0, 7], [2, 8, 5], [1, 3, 6]], dtype=np.int32)
    kp = np.full((nb, Hkv, bs, D), 0xEE, dtype=np.uint8)
    vp = kp.copy()
    table = np.zeros((B, Hkv), dtype=oracle.SEG_DTYPE)
    table[2, :]["seq_len"] = 48          # 48 / 16 == 3 == max_blocks: no column
    table[2, :]["n_seg"] = 1
    table[2, :]["start"] = [0, 48, 48, 48, 48]
    for step in range(37):
        k = bf16_bits(rng.standard_normal((B, Hkv, D)).astype(np.float32))
        assert oracle.append(k, k, bs, bt, kp, vp, table) == Hkv
    for b in range(2):
        for h in range(Hkv):
            assert table[b, h]["seq_len"] == 37 and table[b, h]["n_seg"] == 1
            assert list(table[b, h]["start"]) == [0, 37, 37, 37, 37]
            for t in range(37):
                assert not np.all(kp[bt[b, t // bs], h, t % bs] == 0xEE)
            assert np.all(kp[bt[b, 2], h, 37 % bs:] == 0xEE)   # slots past the end untouched
    assert np.all(table[2, :]["seq_len"] == 48)
    for blk in bt[2]:
        assert np.all(kp[blk] == 0xEE)
