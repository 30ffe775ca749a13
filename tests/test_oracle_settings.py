"""Pins for the oracle's group-selection settings ([DGQ] section 5.3): a cap on the number of
segments and a variance floor under which windows are not separated.  Each check ties the
selection to a closed form, brute force over candidate sets, or a planted structure.  CPU only."""
import itertools

import numpy as np

import oracle

D = 128
L_FIVE = 20000  # n_groups(L) = 5


def bf16_bits(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def brute_force_starts(means, k, min_var):
    """The k largest jumps |m[w+1] - m[w]| among windows w not between two quiet windows
    (keys: jump descending, then window ascending), by enumerating every candidate subset."""
    m = np.asarray(means, dtype=np.float32)
    cand = [w for w in range(len(m) - 1) if m[w] >= min_var or m[w + 1] >= min_var]
    jumps = {w: float(np.float32(abs(np.float32(m[w + 1] - m[w])))) for w in cand}
    k = min(k, len(cand))
    best, best_key = None, None
    for sub in itertools.combinations(cand, k):
        key = sorted(((jumps[w], -w) for w in sub), reverse=True)
        if best_key is None or key > best_key:
            best, best_key = sub, key
    return [0] + sorted(16 * (w + 1) for w in best)


def test_cap_and_floor_match_brute_force_on_tiny_inputs():
    rng = np.random.default_rng(1)
    for trial in range(300):
        W = int(rng.integers(1, 9))
        means = rng.choice([0.0, 0.01, 0.02, 0.05, 0.3, 0.31, 1.0], W).astype(np.float32)
        if trial % 2:
            means = (rng.random(W) * 0.1).astype(np.float32)
        max_groups = int(rng.integers(1, 6))
        min_var = float(rng.choice([0.0, 0.015, 0.04, 0.5, 2.0]))
        k = min(5, max_groups, W) - 1
        got = oracle.boundaries(means, L_FIVE, max_groups, min_var)
        assert got == brute_force_starts(means, k, np.float32(min_var)), (means, max_groups, min_var)


def test_one_group_is_one_segment():
    rng = np.random.default_rng(2)
    k = bf16_bits(rng.standard_normal((300, D)).astype(np.float32) * np.repeat([0.1, 1.0, 0.2], 100)[:, None])
    rec, kc, _ = oracle.compress_pair(k, k, max_groups=1)
    assert rec["n_seg"] == 1 and list(rec["start"]) == [0, 300, 300, 300, 300]
    f = (k.astype(np.uint32) << 16).view(np.float32)
    assert rec["k_min"][0] == f.min() and rec["k_scale"][0] == np.float32(np.float32(f.max() - f.min()) / 255)


def test_cap_keeps_the_largest_jumps_of_the_rule():
    # a 20000-token pair: the rule gives 5 segments; capping at m keeps the m - 1 largest jumps
    rng = np.random.default_rng(3)
    means = (rng.random(1250) ** 3).astype(np.float32)
    full = oracle.boundaries(means, L_FIVE)
    assert len(full) == 5
    m = means
    jumps = np.abs(m[1:] - m[:-1]).astype(np.float32)
    order = sorted(range(len(jumps)), key=lambda w: (-jumps[w], w))
    for cap in (1, 2, 3, 4, 5):
        want = [0] + sorted(16 * (w + 1) for w in order[:cap - 1])
        assert oracle.boundaries(means, L_FIVE, cap) == want


def test_floor_above_every_window_gives_one_segment():
    rng = np.random.default_rng(4)
    k = bf16_bits(rng.standard_normal((4096, D)).astype(np.float32) * 0.3)
    rec, _, _ = oracle.compress_pair(k, k, min_var=100.0)
    assert rec["n_seg"] == 1


def test_floor_keeps_boundaries_off_quiet_transitions():
    # 16384 tokens in spans of 2048 with sigma 0.1 / 0.4 alternating around one louder span
    # (sigma 0.6): window variance means ~0.01 / ~0.16 / ~0.36.  The rule gives 4 boundaries.
    # Without a floor the two edges of the loud span and two of the quiet 0.1 / 0.4 transitions
    # (jumps ~0.15, far above the window-to-window noise) are taken; with a floor of 0.25 no
    # boundary may separate two quiet windows, so the other two fall inside the loud span.
    rng = np.random.default_rng(5)
    sig = np.repeat([0.1, 0.4, 0.1, 0.4, 0.6, 0.1, 0.4, 0.1], 2048).astype(np.float32)
    k = bf16_bits(rng.standard_normal((16384, D)).astype(np.float32) * sig[:, None])
    loud = (8192, 10240)
    quiet_edges = {2048, 4096, 6144, 12288, 14336}
    rec0, _, _ = oracle.compress_pair(k, k)
    s0 = set(int(x) for x in rec0["start"][1:rec0["n_seg"]])
    assert rec0["n_seg"] == 5 and set(loud) <= s0 and len(s0 & quiet_edges) == 2, rec0["start"]
    rec1, _, _ = oracle.compress_pair(k, k, min_var=0.25)
    s1 = set(int(x) for x in rec1["start"][1:rec1["n_seg"]])
    assert rec1["n_seg"] == 5 and set(loud) <= s1 and not (s1 & quiet_edges), rec1["start"]
    assert all(loud[0] <= x <= loud[1] for x in s1)
