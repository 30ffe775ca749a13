"""Pins for the CPU oracle: each check ties it to something other than itself --
a value the DGQ article fixes, a closed form, an invariant, a textbook special case or
brute force on tiny inputs.  CPU only."""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 128


def bf16_bits(x):
    """fp32 values -> bf16 bit patterns (round to nearest even)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def bf16_float(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def gauss_rows(rng, L, sigma):
    return bf16_bits(rng.standard_normal((L, D)).astype(np.float32) * np.float32(sigma))


# --- a1: n_groups ---------------------------------------------------------------------

def _golden_pairs(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_ngroups_golden_table():
    for L, n in _golden_pairs("ngroups.txt"):
        assert oracle.ngroups(int(L)) == int(n), L


def test_ngroups_integer_form():
    # floor(log2(L/1024)) == bit_length(L) - 11 for integer L >= 1024
    for L in list(range(1, 40000, 7)) + [2**k + d for k in range(11, 24) for d in (-1, 0, 1)]:
        want = 2 if L < 2048 else 3 if L < 16384 else min(5, (L.bit_length() - 11) + 2)
        assert oracle.ngroups(L) == want, L


# --- a2: per-token variance -------------------------------------------------------------

def test_variance_matches_fp64_population_variance():
    rng = np.random.default_rng(11)
    for sigma in (0.03, 0.15, 0.47, 3.0):
        rows = gauss_rows(rng, 64, sigma)
        for r in rows:
            got = float(oracle.token_variance(r))
            x = bf16_float(r).astype(np.float64)
            want = float(np.mean((x - x.mean()) ** 2))  # population variance (divide by D)
            assert abs(got - want) <= 2e-6 * want + 1e-30, (got, want)


def test_variance_closed_forms():
    assert oracle.token_variance(bf16_bits(np.full(D, 0.7))) == 0.0
    # half +a, half -a: mean 0, variance a^2 exactly
    a = 0.5
    row = bf16_bits(np.r_[np.full(D // 2, a), np.full(D // 2, -a)])
    assert oracle.token_variance(row) == np.float32(a * a)
    # one spike of height h on zeros: var = h^2/D - (h/D)^2
    h = 2.0
    row = bf16_bits(np.r_[np.float32(h), np.zeros(D - 1)])
    want = h * h / D - (h / D) ** 2
    assert abs(float(oracle.token_variance(row)) - want) <= 1e-7


# --- a3: window means -------------------------------------------------------------------

def test_window_means_vs_fp64_and_partial_window():
    rng = np.random.default_rng(5)
    for L in (1, 15, 16, 17, 37, 300, 1000):
        var = rng.random(L).astype(np.float32)
        got = oracle.window_means(var)
        assert got.shape == ((L + 15) // 16,)
        for w in range(got.shape[0]):
            seg = var[16 * w:16 * w + 16].astype(np.float64)
            assert abs(float(got[w]) - seg.mean()) <= 1e-6 * seg.mean() + 1e-12


def test_window_mean_of_equal_values_is_exact():
    var = np.full(37, 0.25, dtype=np.float32)  # last window holds 5 tokens
    got = oracle.window_means(var)
    assert np.all(got == np.float32(0.25))


# --- a4: boundaries ---------------------------------------------------------------------

def _planted(L, spans, seed=0):
    """K whose sigma steps at the given window-aligned starts; returns K rows."""
    rng = np.random.default_rng(seed)
    k = np.zeros((L, D), dtype=np.uint16)
    edges = [s for s, _ in spans] + [L]
    for (s, sg), e in zip(spans, edges[1:]):
        k[s:e] = gauss_rows(rng, e - s, sg)
    return k


@pytest.mark.parametrize("L,spans", [
    (300, [(0, 0.03), (112, 0.47)]),                                   # n_groups 2
    (4096, [(0, 0.03), (1024, 0.47), (2560, 0.15)]),                   # n_groups 3
    (20000, [(0, 0.15), (3200, 0.47), (8000, 0.03), (12800, 0.47), (16000, 0.08)]),  # 5
])
def test_boundaries_recover_planted_variance_steps(L, spans):
    # magnitudes 0.03 / 0.15 / 0.47 are the article's own example (section 2.2)
    k = _planted(L, spans)
    rec, _, _ = oracle.compress_pair(k, k)
    assert rec["n_seg"] == len(spans)
    assert list(rec["start"][:rec["n_seg"]]) == [s for s, _ in spans]


def _brute_force_starts(means, L):
    W = len(means)
    k = min(oracle.ngroups(L), W) - 1
    jumps = [abs(np.float32(means[w + 1]) - np.float32(means[w])) for w in range(W - 1)]
    best = None
    for subset in itertools.combinations(range(W - 1), k):
        total = sum(Fraction(float(jumps[w])) for w in subset)
        key = (-total, subset)  # max total jump, then the lexicographically first subset
        if best is None or key < best:
            best = key
    return [0] + [16 * (w + 1) for w in best[1]]


def test_boundaries_brute_force_tiny():
    rng = np.random.default_rng(3)
    for trial in range(300):
        W = int(rng.integers(1, 9))
        L = 16 * (W - 1) + int(rng.integers(1, 17))
        if trial % 3 == 0:  # force ties
            means = rng.integers(0, 3, W).astype(np.float32)
        else:
            means = rng.random(W).astype(np.float32)
        # n_groups depends on L alone, so the same W means are cut for 2, 3 and 5 groups
        for L_eff in (L, L + 3000, L + 20000):
            got = oracle.boundaries(means, L_eff)
            assert got == _brute_force_starts(means, L_eff), (means, L_eff)


_HUGE = Fraction(2) ** 200  # exceeds any sum of finite fp32 jumps (each < 2^129)


def _brute_force_starts_nonfinite(means, L):
    """Brute force for means that may be +inf: a jump between two infinite means (NaN) is no
    candidate; an infinite jump outranks every finite total; the count is capped by the
    candidates left.  Maximum total jump, then the lexicographically first subset."""
    W = len(means)
    k = min(oracle.ngroups(L), W) - 1
    jumps = {}
    for w in range(W - 1):
        j = abs(np.float32(means[w + 1]) - np.float32(means[w]))
        if not np.isnan(j):
            jumps[w] = _HUGE if np.isinf(j) else Fraction(float(j))
    k = min(k, len(jumps))
    best = None
    for subset in itertools.combinations(sorted(jumps), k):
        key = (-sum(jumps[w] for w in subset), subset)
        if best is None or key < best:
            best = key
    return [0] + [16 * (w + 1) for w in best[1]]


def test_boundaries_skip_undefined_jumps():
    # two adjacent overflowed windows: inf - inf has no value, so the cut goes to the infinite
    # jump after them, not to the first (undefined) candidate
    inf = np.float32(np.inf)
    with np.errstate(invalid="ignore"):
        assert oracle.boundaries(np.array([inf, inf, 1.0], np.float32), 40) == [0, 32]
        # only undefined jumps: no candidate, one segment
        assert oracle.boundaries(np.array([inf, inf], np.float32), 32) == [0]
        # three segments wanted, two candidates (the jumps either side of an infinite run)
        assert oracle.boundaries(np.array([1.0, inf, inf, inf, 2.0], np.float32), 3000) == [0, 16, 64]


def test_boundaries_brute_force_with_overflowed_windows():
    rng = np.random.default_rng(4)
    with np.errstate(invalid="ignore"):
        for trial in range(300):
            W = int(rng.integers(1, 9))
            L = 16 * (W - 1) + int(rng.integers(1, 17))
            means = rng.integers(0, 3, W).astype(np.float32) if trial % 2 else rng.random(W).astype(np.float32)
            means[rng.random(W) < 0.4] = np.inf
            for L_eff in (L, L + 3000, L + 20000):
                got = oracle.boundaries(means, L_eff)
                assert got == _brute_force_starts_nonfinite(means, L_eff), (means, L_eff)


def test_variance_overflow_closed_form():
    # a row of +-a has mean 0 and variance a^2; for a = 2^60 every step is exact, for a = 2^63
    # the squares (2^126) are finite but their fp32 sum (2^133) overflows, so the variance is +inf
    row = np.where(np.arange(D) % 2 == 0, 1.0, -1.0).astype(np.float32)
    assert oracle.token_variance(bf16_bits(row * np.float32(2.0 ** 60))) == np.float32(2.0 ** 120)
    assert np.isposinf(oracle.token_variance(bf16_bits(row * np.float32(2.0 ** 63))))


def test_overflowed_windows_cut_at_the_finite_edge():
    # finite bf16 rows large enough to overflow the fp32 variance in windows 0..1, ordinary rows
    # after: the only defined jump that is infinite is the one between windows 1 and 2
    rng = np.random.default_rng(9)
    L = 300
    k = gauss_rows(rng, L, 0.1)
    sign = np.where(rng.random((32, D)) < 0.5, -1.0, 1.0).astype(np.float32)
    k[:32] = bf16_bits(sign * np.float32(2.0 ** 63))
    rec, kc, _ = oracle.compress_pair(k, k)
    assert rec["n_seg"] == 2 and list(rec["start"][:2]) == [0, 32]
    # the overflowed segment holds two values: its codes are exactly 0 and 255
    assert set(np.unique(kc[:32]).tolist()) == {0, 255}


def test_single_window_is_one_segment():
    k = gauss_rows(np.random.default_rng(1), 16, 0.3)
    rec, _, _ = oracle.compress_pair(k, k)
    assert rec["n_seg"] == 1 and rec["start"][0] == 0


# --- a5/a6: segment min/max and codes ------------------------------------------------------

def _compress_random(L, seed):
    n = synth.spans(seed, 0, 0, 0, L, synth.RULE_U)
    k = synth.fill_pair(seed, synth.STREAM_K, 0, 0, 0, L, *n)
    v = synth.fill_pair(seed, synth.STREAM_V, 0, 0, 0, L, *n)
    return k, v, oracle.compress_pair(k, v)


@pytest.mark.parametrize("L", [1, 5, 16, 37, 300, 2048, 5000, 17000])
def test_segment_min_max_brute_force(L):
    k, v, (rec, kc, vc) = _compress_random(L, L)
    n = rec["n_seg"]
    st = list(rec["start"][:n]) + [L]
    for s in range(n):
        for x, mn_field, sc_field in ((k, "k_min", "k_scale"), (v, "v_min", "v_scale")):
            xs = bf16_float(x[st[s]:st[s + 1]])
            mn, mx = np.float32(xs.min()), np.float32(xs.max())
            assert rec[mn_field][s] == mn
            r = np.float32(mx - mn)
            assert rec[sc_field][s] == (np.float32(r / np.float32(255)) if r != 0 else 0)


@pytest.mark.parametrize("L", [3, 37, 300, 2048, 17000])
def test_code_invariants(L):
    k, v, (rec, kc, vc) = _compress_random(L, 100 + L)
    n = rec["n_seg"]
    st = list(rec["start"][:n]) + [L]
    for x, codes, mnf, scf in ((k, kc, "k_min", "k_scale"), (v, vc, "v_min", "v_scale")):
        for s in range(n):
            xs = bf16_float(x[st[s]:st[s + 1]]).astype(np.float64)
            cs = codes[st[s]:st[s + 1]].astype(np.int64)
            mn, sc = float(rec[mnf][s]), float(rec[scf][s])
            mx = xs.max()
            if sc > 0:
                assert cs[xs == xs.min()].max() == 0
                assert cs[xs == mx].min() == 255
                err = np.abs(mn + cs * sc - xs)
                bound = 0.5 * sc * (1 + 2**-10) + 2**-22 * (abs(mn) + abs(mx))
                assert err.max() <= bound
                order = np.argsort(xs.ravel(), kind="stable")
                assert np.all(np.diff(cs.ravel()[order]) >= 0)  # monotone in x
            else:
                assert np.all(cs == 0)


def test_round_half_to_even_closed_form():
    # one flat-range segment with min 0, max 255 -> inv == 1 exactly; x = k + 0.5 ties
    vals = np.zeros(D, dtype=np.float32)
    vals[1] = 255.0
    vals[2:10] = [0.5, 1.5, 2.5, 3.5, 4.5, 253.5, 254.5, 100.0]
    k = np.tile(bf16_bits(vals), (4, 1))
    rec, kc, _ = oracle.compress_pair(k, k)
    assert rec["n_seg"] == 1 and rec["k_min"][0] == 0 and rec["k_scale"][0] == np.float32(1.0)
    assert list(kc[0, :10]) == [0, 255, 0, 2, 2, 4, 4, 254, 254, 100]


def test_rounded_product_ties_round_half_to_even():
    # x where the fp32 product (x - min) * inv is exactly k + 0.5 but the exact product is not:
    # the method rounds the product first, then half to even, so these codes must differ from
    # the integer nearest to the exact product (what one fused multiply-add rounding gives) in
    # every case where k + 0.5 was rounded toward the odd side
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    finite = np.isfinite(vals)
    rng = np.random.default_rng(4)
    lo_pool = bits[finite & (vals > -2.0) & (vals < -0.01)]
    hi_pool = bits[finite & (vals > 0.01) & (vals < 3.0)]
    checked = flipped = 0
    while flipped < 20:
        ab, bb = rng.choice(lo_pool), rng.choice(hi_pool)
        a, b = vals[ab], vals[bb]
        inside = finite & (vals >= a) & (vals <= b)
        xv = vals[inside]
        p = (xv - a).astype(np.float32).astype(np.float64) * np.float64(np.float32(255.0) / np.float32(b - a))
        u = p.astype(np.float32).astype(np.float64)
        tie = (u - np.floor(u) == 0.5) & (p != u)
        if not tie.any():
            continue
        row = np.resize(bits[inside][tie], D).astype(np.uint16)
        row[0], row[1] = ab, bb
        rec, kc, _ = oracle.compress_pair(np.tile(row, (16, 1)), np.tile(row, (16, 1)))
        assert rec["n_seg"] == 1 and rec["k_min"][0] == a
        xs = (row[2:].astype(np.uint32) << 16).view(np.float32)
        pe = (xs - a).astype(np.float32).astype(np.float64) * np.float64(np.float32(255.0) / np.float32(b - a))
        ue = pe.astype(np.float32).astype(np.float64)
        even = 2 * np.round(ue / 2)        # ue = k + 0.5 -> the even one of k, k + 1
        assert np.all(kc[0, 2:] == even)
        checked += xs.size
        flipped += int((even != np.rint(pe)).sum())
    assert checked > 0


def test_flat_segment_codes_zero_and_decode_to_min():
    # 20 tokens = 2 windows -> 2 segments (a zero jump is still a boundary), both flat
    k = np.tile(bf16_bits(np.full(D, -0.375)), (20, 1))
    rec, kc, _ = oracle.compress_pair(k, k)
    assert rec["n_seg"] == 2 and list(rec["start"][:2]) == [0, 16]
    assert np.all(rec["k_scale"][:2] == 0) and np.all(rec["k_min"][:2] == np.float32(-0.375))
    assert np.all(kc == 0)


def test_negative_zero_min_is_stored_as_positive_zero():
    vals = np.abs(np.random.default_rng(2).standard_normal(D)).astype(np.float32)
    vals[0] = -0.0
    vals[1] = 0.0
    k = np.tile(bf16_bits(vals), (3, 1))
    rec, _, _ = oracle.compress_pair(k, k)
    assert rec["k_min"][0] == 0 and not np.signbit(rec["k_min"][0])


def test_single_segment_matches_torch_per_tensor_affine_quantization():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    k = gauss_rows(rng, 16, 0.2)  # one window -> one segment
    rec, kc, _ = oracle.compress_pair(k, k)
    x = torch.from_numpy(bf16_float(k).copy())
    mn, mx = float(x.min()), float(x.max())
    scale = (mx - mn) / 255.0
    zp = int(round(-mn / scale))
    tq = torch.quantize_per_tensor(x, scale, zp, torch.quint8).int_repr().numpy().astype(np.int64)
    assert np.abs(tq - kc.astype(np.int64)).max() <= 1  # textbook asymmetric uint8, +-1 code


# --- a6/a7: paging and bytes ---------------------------------------------------------------

def _batch(Ls, Hkv, bs, seed, shuffle=True, extra_blocks=3):
    lens = np.asarray(Ls, dtype=np.int32)
    cu = np.zeros(len(Ls) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    tabs = synth.span_tables(seed, 0, lens, Hkv, synth.RULE_U)
    k = synth.fill_layer(seed, synth.STREAM_K, 0, cu, Hkv, tabs)
    v = synth.fill_layer(seed, synth.STREAM_V, 0, cu, Hkv, tabs)
    nblk = [(L + bs - 1) // bs for L in Ls]
    num_blocks = sum(nblk) + extra_blocks
    order = synth.permutation(seed, synth.STREAM_META, num_blocks) if shuffle else np.arange(num_blocks)
    bt = np.zeros((len(Ls), max(1, max(nblk))), dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = order[off:off + n]
        off += n
    return lens, cu, k, v, bt, num_blocks


@pytest.mark.parametrize("bs", [16, 32, 64])
def test_paged_scatter_gathers_back_and_counts_bytes(bs):
    Ls, Hkv = [37, 300, 1, 64], 2
    lens, cu, k, v, bt, nb = _batch(Ls, Hkv, bs, seed=bs)
    kp, vp, table = oracle.compress(k, v, cu, Hkv, bs, bt, nb, fill=0xA5)
    written = 0
    touched = np.zeros(kp.shape[:3], dtype=bool)
    for b, L in enumerate(Ls):
        for h in range(Hkv):
            rec, kc, vc = oracle.compress_pair(k[cu[b]:cu[b + 1], h], v[cu[b]:cu[b + 1], h])
            assert table[b, h].tobytes() == rec.tobytes()
            for t in range(L):
                blk = bt[b, t // bs]
                assert np.array_equal(kp[blk, h, t % bs], kc[t])
                assert np.array_equal(vp[blk, h, t % bs], vc[t])
                touched[blk, h, t % bs] = True
        written += oracle.compress_bytes_written(L, Hkv)
    assert np.all(kp[~touched] == 0xA5) and np.all(vp[~touched] == 0xA5)
    assert written == 2 * int(touched.sum()) * D + table.nbytes


def test_storage_formula_golden():
    g = {r[0]: int(r[1]) for r in _golden_pairs("storage_formula.txt")}
    layers, heads, L = g["layers"], g["heads"], g["seq_len"]
    per_layer = oracle.compress_bytes_written(L, heads)
    body = layers * (per_layer - 128 * heads)
    assert body == g["dgq_body_bytes"]
    assert 2 * body == g["fp16_bytes"]
    marker = layers * heads * L // 8
    assert marker == g["dgq_marker_bytes"] and round(marker / 1e6) == g["marker_printed_mb"]


# --- a8-a10: attention ------------------------------------------------------------------------

def _attn_numpy(q, kn, vn, kdq, vdq):
    """Independent fp64 attention for one (request, query head): kdq/vdq [L, D]."""
    keys = np.vstack([kdq, bf16_float(kn)[None].astype(np.float64)])
    vals = np.vstack([vdq, bf16_float(vn)[None].astype(np.float64)])
    s = keys @ bf16_float(q).astype(np.float64) / math.sqrt(D)
    p = np.exp(s - s.max())
    return (p / p.sum()) @ vals


def _decode_case(Ls, Hq, Hkv, bs, seed):
    lens, cu, k, v, bt, nb = _batch(Ls, Hkv, bs, seed)
    kp, vp, table = oracle.compress(k, v, cu, Hkv, bs, bt, nb)
    q = synth.fill_heads(seed, synth.STREAM_Q, 0, len(Ls), Hq, 1.0)
    kn = synth.fill_heads(seed, synth.STREAM_KNEW, 0, len(Ls), Hkv, 0.15)
    vn = synth.fill_heads(seed, synth.STREAM_VNEW, 0, len(Ls), Hkv, 0.15)
    return lens, bt, kp, vp, table, q, kn, vn


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (4, 4), (8, 1)])
def test_attention_matches_numpy_brute_force(Hq, Hkv):
    Ls, bs = [37, 300, 0, 16], 16
    lens, bt, kp, vp, table, q, kn, vn = _decode_case(Ls, Hq, Hkv, bs, seed=Hq * 10 + Hkv)
    out = oracle.paged_decode_attn(q, kn, vn, kp, vp, table, bt, lens)
    G = Hq // Hkv
    for b, L in enumerate(Ls):
        for hq in range(Hq):
            h = hq // G
            kdq = oracle.dequant_pair(kp, table, bt, b, h, L, False)
            vdq = oracle.dequant_pair(vp, table, bt, b, h, L, True)
            want = _attn_numpy(q[b, hq], kn[b, h], vn[b, h], kdq.reshape(L, D), vdq.reshape(L, D))
            np.testing.assert_allclose(out[b, hq], want, rtol=1e-12, atol=1e-13)


def test_attention_empty_cache_returns_current_value():
    lens, bt, kp, vp, table, q, kn, vn = _decode_case([0, 5], 4, 2, 16, seed=4)
    out = oracle.paged_decode_attn(q, kn, vn, kp, vp, table, bt, lens)
    for hq in range(4):
        assert np.array_equal(out[0, hq], bf16_float(vn[0, hq // 2]).astype(np.float64))


def test_attention_two_keys_closed_form():
    lens, bt, kp, vp, table, q, kn, vn = _decode_case([1], 2, 1, 16, seed=8)
    out = oracle.paged_decode_attn(q, kn, vn, kp, vp, table, bt, lens)
    kdq = oracle.dequant_pair(kp, table, bt, 0, 0, 1, False)[0]
    vdq = oracle.dequant_pair(vp, table, bt, 0, 0, 1, True)[0]
    for hq in range(2):
        qq = bf16_float(q[0, hq]).astype(np.float64)
        s0 = qq @ kdq / math.sqrt(D)
        s1 = qq @ bf16_float(kn[0, 0]).astype(np.float64) / math.sqrt(D)
        p0 = 1.0 / (1.0 + math.exp(s1 - s0))  # softmax over two scores
        want = p0 * vdq + (1 - p0) * bf16_float(vn[0, 0]).astype(np.float64)
        np.testing.assert_allclose(out[0, hq], want, rtol=1e-12, atol=1e-14)


def test_attention_equal_keys_give_uniform_average():
    L, bs = 40, 16
    lens, bt, kp, vp, table, q, kn, vn = _decode_case([L], 1, 1, bs, seed=12)
    kp[:] = 77  # every cached key identical within its segment ...
    table = table.copy()
    table["k_min"][:] = 0.125
    table["k_scale"][:] = 0.0  # ... and across segments: every cached key == 0.125
    kn[:] = bf16_bits(np.full(D, 0.125))  # the current key equals them too
    out = oracle.paged_decode_attn(q, kn, vn, kp, vp, table, bt, lens)
    vdq = oracle.dequant_pair(vp, table, bt, 0, 0, L, True)
    want = (vdq.sum(0) + bf16_float(vn[0, 0])) / (L + 1)
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-12, atol=1e-14)


def test_attention_invariant_under_physical_block_permutation():
    Ls, Hq, Hkv, bs = [37, 300], 4, 2, 16
    lens, bt, kp, vp, table, q, kn, vn = _decode_case(Ls, Hq, Hkv, bs, seed=21)
    out = oracle.paged_decode_attn(q, kn, vn, kp, vp, table, bt, lens)
    perm = np.random.default_rng(0).permutation(kp.shape[0]).astype(np.int32)  # new id of block i
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    out2 = oracle.paged_decode_attn(q, kn, vn, kp2, vp2, table, perm[bt], lens)
    assert np.array_equal(out, out2)


def test_gqa_equals_mha_with_duplicated_kv_heads():
    Ls, Hq, Hkv, bs = [37, 300], 4, 2, 16
    lens, bt, kp, vp, table, q, kn, vn = _decode_case(Ls, Hq, Hkv, bs, seed=31)
    out = oracle.paged_decode_attn(q, kn, vn, kp, vp, table, bt, lens)
    G = Hq // Hkv
    idx = np.arange(Hq) // G
    out_mha = oracle.paged_decode_attn(q, kn[:, idx], vn[:, idx], np.ascontiguousarray(kp[:, idx]),
                                       np.ascontiguousarray(vp[:, idx]),
                                       np.ascontiguousarray(table[:, idx]), bt, lens)
    assert np.array_equal(out, out_mha)


# --- fidelity context: attention over the unquantised bf16 K/V ------------------------------

def test_unquantised_attention_matches_numpy_brute_force():
    rng = np.random.default_rng(21)
    lens = np.array([3, 0, 9], dtype=np.int32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    B, Hq, Hkv = 3, 4, 2
    k = bf16_bits(rng.standard_normal((cu[-1], Hkv, D)).astype(np.float32))
    v = bf16_bits(rng.standard_normal((cu[-1], Hkv, D)).astype(np.float32))
    q = bf16_bits(rng.standard_normal((B, Hq, D)).astype(np.float32))
    kn = bf16_bits(rng.standard_normal((B, Hkv, D)).astype(np.float32))
    vn = bf16_bits(rng.standard_normal((B, Hkv, D)).astype(np.float32))
    got = oracle.decode_attn_unquantised(q, kn, vn, k, v, cu, lens)
    f = lambda a: bf16_float(a).astype(np.float64)
    for b in range(B):
        for hq in range(Hq):
            h = hq // (Hq // Hkv)
            keys = np.concatenate([f(k[cu[b]:cu[b + 1], h]), f(kn[b, h])[None]])
            vals = np.concatenate([f(v[cu[b]:cu[b + 1], h]), f(vn[b, h])[None]])
            s = keys @ f(q[b, hq]) / math.sqrt(D)
            p = np.exp(s - s.max())
            want = (p[:, None] * vals).sum(0) / p.sum()
            assert np.allclose(got[b, hq], want, rtol=1e-12, atol=1e-12)


def test_unquantised_attention_equals_cache_attention_when_codes_are_exact():
    # every value on the grid q / 16 with 0 and 255 / 16 in each segment: scale = 1/16 and
    # inv = 16 exactly, so every code decodes to its value and the two attentions coincide
    rng = np.random.default_rng(22)
    L, Hkv, Hq, bs = 40, 1, 2, 16
    grid = rng.integers(0, 256, (L, Hkv, D)).astype(np.float32) / 16
    grid[:, :, 0], grid[:, :, 1] = 0.0, 255 / 16
    k = bf16_bits(grid)
    v = bf16_bits(grid[::-1].copy())
    cu = np.array([0, L], dtype=np.int32)
    bt = np.array([[2, 0, 1]], dtype=np.int32)
    kp, vp, table = oracle.compress(k, v, cu, Hkv, bs, bt, 3)
    assert np.all(table["k_scale"][0, 0][:table["n_seg"][0, 0]] == np.float32(1 / 16))
    q = bf16_bits(rng.standard_normal((1, Hq, D)).astype(np.float32) * 0.2)
    kn = bf16_bits(rng.standard_normal((1, Hkv, D)).astype(np.float32))
    lens = np.array([L], dtype=np.int32)
    cache = oracle.paged_decode_attn(q, kn, kn, kp, vp, table, bt, lens)
    raw = oracle.decode_attn_unquantised(q, kn, kn, k, v, cu, lens)
    assert np.array_equal(cache, raw)
