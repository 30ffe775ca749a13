"""Pins for the oracle's re-segmentation after a decode-step append: the trigger bits follow the
length rule's thresholds and the 16-token windows (DGQ article, sections 2.2 and 3.2), a
re-segmented request is exactly a fresh compression of its grown bf16 history, every other
request is exactly the plain append, and crossing 2048 / 16384 changes the segment count.
CPU only."""
import numpy as np
import pytest

import oracle
import synth
from synth import configs

D = 128
GOLDEN_THRESHOLDS = {2048, 16384}  # tests/golden/ngroups.txt: the rule changes there and only there


def test_trigger_bits_closed_form():
    # bit 1: the appended token L closes the window [L - 15, L]; bit 2: the length L + 1 reaches
    # a threshold of the length rule (for every L >= 16384 the rule gives 5, so none above)
    for L in list(range(0, 4200)) + list(range(16300, 16500)) + [32766, 32767, 65535, 131071, 1 << 20]:
        want = (1 if (L + 1) % 16 == 0 else 0) | (2 if (L + 1) in GOLDEN_THRESHOLDS else 0)
        assert oracle.resegment_flags(L) == want, L


def _history(lens, Hkv, seed, steps):
    """bf16 K/V of each request for its first lens[b] + steps tokens (synth, rule U), packed."""
    full = np.asarray(lens, dtype=np.int32) + steps
    cu = configs.cu_seqlens(full)
    tabs = synth.span_tables(seed, 0, full, Hkv, synth.RULE_U)
    k = synth.fill_layer(seed, synth.STREAM_K, 0, cu, Hkv, tabs)
    v = synth.fill_layer(seed, synth.STREAM_V, 0, cu, Hkv, tabs)
    return k, v, cu


def _prefix(x, cu, lens):
    """The first lens[b] rows of each request of a packed array, packed again."""
    parts = [x[cu[b]:cu[b] + int(L)] for b, L in enumerate(lens)]
    return np.concatenate(parts) if parts else x[:0]


def _state(lens, Hkv, bs, steps, seed):
    k, v, cu = _history(lens, Hkv, seed, steps)
    lens = np.asarray(lens, dtype=np.int32)
    nblk = [(int(L) + steps + bs - 1) // bs for L in lens]
    mb = max(nblk)
    perm = synth.permutation(seed, synth.STREAM_META, sum(nblk))
    bt = np.zeros((len(lens), mb), dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n]
        off += n
    cu0 = configs.cu_seqlens(lens)
    kp, vp, table = oracle.compress(_prefix(k, cu, lens), _prefix(v, cu, lens), cu0, Hkv, bs, bt, sum(nblk))
    return k, v, cu, bt, sum(nblk), kp, vp, table


@pytest.mark.parametrize("mask", [oracle.RESEG_WINDOW | oracle.RESEG_NGROUPS, oracle.RESEG_NGROUPS])
def test_resegmented_requests_equal_a_fresh_compress(mask):
    lens, Hkv, bs, steps = [2040, 300, 1000, 16380, 5], 2, 16, 9
    k, v, cu, bt, nb, kp, vp, table = _state(lens, Hkv, bs, steps, seed=31)
    for s in range(steps):
        cur = np.asarray(lens, dtype=np.int32) + s  # cached tokens before this step
        knew = np.stack([k[cu[b] + int(L)] for b, L in enumerate(cur)])
        vnew = np.stack([v[cu[b] + int(L)] for b, L in enumerate(cur)])
        grown = cur + 1
        kh, vh = _prefix(k, cu, grown), _prefix(v, cu, grown)
        hcu = configs.cu_seqlens(grown)
        # the plain append of the same token, for the requests that are not re-segmented
        kp_a, vp_a, tab_a = kp.copy(), vp.copy(), table.copy()
        assert oracle.append(knew, vnew, bs, bt, kp_a, vp_a, tab_a) == 0
        flags, skipped = oracle.append_resegment(knew, vnew, bs, bt, kp, vp, table, kh, vh, hcu, mask=mask)
        assert skipped == 0
        assert np.array_equal(flags, np.array([[oracle.resegment_flags(int(L))] * Hkv for L in cur]))
        fresh_kp, fresh_vp, fresh_tab = oracle.compress(kh, vh, hcu, Hkv, bs, bt, nb)
        for b in range(len(lens)):
            redo = bool(flags[b].any() and (flags[b] & mask).any())
            ref_tab, ref_kp, ref_vp = (fresh_tab, fresh_kp, fresh_vp) if redo else (tab_a, kp_a, vp_a)
            assert table[b].tobytes() == ref_tab[b].tobytes(), (s, b, redo)
            t = np.arange(int(grown[b]))
            blk, slot = bt[b, t // bs], t % bs
            assert np.array_equal(kp[blk, :, slot], ref_kp[blk, :, slot]), (s, b)
            assert np.array_equal(vp[blk, :, slot], ref_vp[blk, :, slot]), (s, b)


def test_crossing_thresholds_changes_the_segment_count():
    # 2047 -> 2048 tokens: 2 -> 3 segments; 16383 -> 16384: 3 -> 5 (planted spans give distinct
    # jumps, so the rule's count is reached)
    for L0, n0, n1 in ((2047, 2, 3), (16383, 3, 5)):
        k, v, cu, bt, nb, kp, vp, table = _state([L0], 1, 64, 1, seed=40 + L0 % 7)
        assert table[0, 0]["n_seg"] == n0
        kh, vh = k[:L0 + 1], v[:L0 + 1]
        flags, _ = oracle.append_resegment(k[L0:L0 + 1][None], v[L0:L0 + 1][None], 64, bt, kp, vp, table, kh,
                                           vh, np.array([0, L0 + 1], np.int32))
        assert flags[0, 0] == oracle.RESEG_WINDOW | oracle.RESEG_NGROUPS
        assert table[0, 0]["n_seg"] == n1 and table[0, 0]["seq_len"] == L0 + 1


def test_empty_mask_is_the_plain_append():
    lens, Hkv, bs = [31, 47, 2047], 2, 32
    k, v, cu, bt, nb, kp, vp, table = _state(lens, Hkv, bs, 1, seed=33)
    knew = np.stack([k[cu[b] + L] for b, L in enumerate(lens)])
    vnew = np.stack([v[cu[b] + L] for b, L in enumerate(lens)])
    kp_a, vp_a, tab_a = kp.copy(), vp.copy(), table.copy()
    oracle.append(knew, vnew, bs, bt, kp_a, vp_a, tab_a)
    grown = np.asarray(lens, np.int32) + 1
    flags, _ = oracle.append_resegment(knew, vnew, bs, bt, kp, vp, table, _prefix(k, cu, grown),
                                       _prefix(v, cu, grown), configs.cu_seqlens(grown), mask=0)
    assert flags[:, 0].tolist() == [1, 1, 3]
    assert np.array_equal(kp, kp_a) and np.array_equal(vp, vp_a) and table.tobytes() == tab_a.tobytes()
