"""Pins for the oracle's independent V segmentation (a group-selection variant: V segmented by
the same rule on its own variance).  Checks: identical K and V reduce to the shared path; the
two tensors' roles swap with the inputs; planted variance steps in K and in V land as each
tensor's own boundaries; each V segment's extremes encode to 0 and 255; appending through split
tables that carry the shared segmentation equals the shared append.  CPU only."""
import numpy as np

import oracle

D = 128


def bf16_bits(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def layer(lens, hkv, seed, steps_k=None, steps_v=None):
    """Packed [T, Hkv, 128] bf16 K and V; optional planted sigma steps {token: sigma} per tensor."""
    rng = np.random.default_rng(seed)
    T = int(sum(lens))
    out = []
    for steps in (steps_k, steps_v):
        sig = np.full(T, 0.2, dtype=np.float32)
        if steps:
            off = 0
            for L in lens:
                for t0, s in sorted(steps.items()):
                    if t0 < L:
                        sig[off + t0:off + L] = s
                off += L
        out.append(bf16_bits(rng.standard_normal((T, hkv, D)).astype(np.float32) * sig[:, None, None]))
    return out


def paging(lens, bs):
    nblk = [(L + bs - 1) // bs for L in lens]
    bt = np.zeros((len(lens), max(1, max(nblk))), dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = np.arange(off, off + n)
        off += n
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return cu, bt, off + 1


def test_identical_k_and_v_reduce_to_the_shared_segmentation():
    lens, hkv, bs = [37, 300, 0, 3000], 2, 16
    k, _ = layer(lens, hkv, 1)
    cu, bt, nb = paging(lens, bs)
    kp, vp, table = oracle.compress(k, k, cu, hkv, bs, bt, nb)
    skp, svp, kt, vt = oracle.compress_split(k, k, cu, hkv, bs, bt, nb)
    assert np.array_equal(skp, kp) and np.array_equal(svp, vp)
    for f in ("n_seg", "seq_len", "start"):
        assert np.array_equal(kt[f], table[f]) and np.array_equal(vt[f], table[f])
    for f in ("k_min", "k_scale", "k_inv_last"):
        assert np.array_equal(kt[f], table[f])
    for f in ("v_min", "v_scale", "v_inv_last"):
        assert np.array_equal(vt[f], table[f])
    for f in ("v_min", "v_scale", "v_inv_last"):
        assert not kt[f].any()
    for f in ("k_min", "k_scale", "k_inv_last"):
        assert not vt[f].any()


def test_roles_swap_with_the_inputs():
    lens, hkv, bs = [500, 2100, 40], 3, 32
    k, v = layer(lens, hkv, 2, steps_k={128: 0.5, 1024: 0.05}, steps_v={256: 0.03, 1600: 0.6})
    cu, bt, nb = paging(lens, bs)
    kp, vp, kt, vt = oracle.compress_split(k, v, cu, hkv, bs, bt, nb)
    kp2, vp2, kt2, vt2 = oracle.compress_split(v, k, cu, hkv, bs, bt, nb)
    assert np.array_equal(kp, vp2) and np.array_equal(vp, kp2)
    assert np.array_equal(kt["start"], vt2["start"]) and np.array_equal(vt["start"], kt2["start"])
    assert np.array_equal(kt["k_min"], vt2["v_min"]) and np.array_equal(kt["k_scale"], vt2["v_scale"])
    assert np.array_equal(vt["v_min"], kt2["k_min"]) and np.array_equal(vt["v_scale"], kt2["k_scale"])
    # and the K side is the shared path's K side
    _, _, table = oracle.compress(k, v, cu, hkv, bs, bt, nb)
    assert np.array_equal(kt["start"], table["start"]) and np.array_equal(kt["k_min"], table["k_min"])


def test_planted_steps_land_on_each_tensors_own_boundaries():
    # L = 2100 -> n_groups 3: two boundaries each; K steps at 512 / 1536, V steps at 256 / 1024
    lens, hkv, bs = [2100], 1, 16
    k, v = layer(lens, hkv, 3, steps_k={512: 0.47, 1536: 0.03}, steps_v={256: 0.5, 1024: 0.03})
    cu, bt, nb = paging(lens, bs)
    _, _, kt, vt = oracle.compress_split(k, v, cu, hkv, bs, bt, nb)
    assert list(kt[0, 0]["start"][:3]) == [0, 512, 1536] and kt[0, 0]["n_seg"] == 3
    assert list(vt[0, 0]["start"][:3]) == [0, 256, 1024] and vt[0, 0]["n_seg"] == 3


def test_v_segment_extremes_encode_to_0_and_255():
    lens, hkv, bs = [2100], 1, 16
    k, v = layer(lens, hkv, 4, steps_v={256: 0.5, 1024: 0.03})
    cu, bt, nb = paging(lens, bs)
    _, vp, _, vt = oracle.compress_split(k, v, cu, hkv, bs, bt, nb)
    rec = vt[0, 0]
    x = (v[:, 0, :].astype(np.uint32) << 16).view(np.float32)
    codes = vp[bt[0, np.arange(2100) // bs], 0, np.arange(2100) % bs]
    starts = list(rec["start"][:rec["n_seg"]]) + [2100]
    for s in range(rec["n_seg"]):
        seg = slice(starts[s], starts[s + 1])
        assert np.float32(x[seg].min()) == rec["v_min"][s]
        assert codes[seg][x[seg] == x[seg].min()].max() == 0
        assert codes[seg][x[seg] == x[seg].max()].min() == 255


def test_split_append_equals_shared_append_on_shared_segments():
    """Split tables that carry the shared segmentation (K's fields in one, V's in the other):
    appending through them gives the shared append's codes and the same fields."""
    lens, hkv, bs = [37, 300, 0, 2100], 2, 16
    k, v = layer(lens, hkv, 5)
    cu, bt, nb = paging(lens, bs)
    bt = np.concatenate([bt, np.full((len(lens), 2), -1, dtype=np.int32)], axis=1)
    for b, L in enumerate(lens):  # one more block per request for the appended tokens
        n = (L + bs - 1) // bs
        bt[b, n] = nb + b
    nb += len(lens)
    kp, vp, table = oracle.compress(k, v, cu, hkv, bs, bt, nb)
    kt, vt = table.copy(), table.copy()
    for f in ("v_min", "v_scale", "v_inv_last"):
        kt[f] = 0
    for f in ("k_min", "k_scale", "k_inv_last"):
        vt[f] = 0
    rng = np.random.default_rng(6)
    skp, svp = kp.copy(), vp.copy()
    for step in range(3):
        kn = bf16_bits(rng.standard_normal((len(lens), hkv, D)).astype(np.float32) * 0.3)
        vn = bf16_bits(rng.standard_normal((len(lens), hkv, D)).astype(np.float32) * 0.3)
        assert oracle.append(kn, vn, bs, bt, kp, vp, table) == 0
        assert oracle.append_split(kn, vn, bs, bt, skp, svp, kt, vt) == 0
    assert np.array_equal(skp, kp) and np.array_equal(svp, vp)
    for f in ("n_seg", "seq_len", "start", "k_min", "k_scale", "k_inv_last"):
        assert np.array_equal(kt[f], table[f]), f
    for f in ("n_seg", "seq_len", "start", "v_min", "v_scale", "v_inv_last"):
        assert np.array_equal(vt[f], table[f]), f
