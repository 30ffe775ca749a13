"""dgq_compress on the GPU against the CPU oracle: codes, segment records and block gathers
bit-exact, across lengths that hit every n_groups branch, ragged tails, empty requests and
all block sizes."""
import numpy as np
import pytest

from dgq_cases import Case, assert_compress_equal, table_to_numpy

pytestmark = pytest.mark.gpu


def run(case, fill=0):
    kp, vp, table = case.oracle_compress()
    case.gpu_compress(fill=fill)
    assert_compress_equal(case, kp, vp, table, case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(),
                          table_to_numpy(case.d_table))
    return kp, vp, table


def test_tiny_workload():
    run(Case([37, 300], hq=4, hkv=2, bs=16, seed=0, rule=0))


@pytest.mark.parametrize("bs", [16, 32, 64])
def test_lengths_across_ngroups_branches(bs):
    lens = [1, 15, 16, 17, 37, 300, 2047, 2048, 2049, 5000, 16383, 16384, 20000]
    run(Case(lens, hq=8, hkv=2, bs=bs, seed=bs))


def test_empty_requests_and_single_tokens():
    case = Case([0, 1, 0, 33, 0], hq=2, hkv=2, bs=16, seed=5)
    run(case)
    tab = table_to_numpy(case.d_table)
    assert tab[0, 0]["n_seg"] == 0 and tab[1, 0]["n_seg"] == 1 and tab[3, 1]["n_seg"] == 2


def test_untouched_slots_keep_their_bytes():
    case = Case([37, 300], hq=4, hkv=2, bs=16, seed=7)
    run(case, fill=0xA5)
    kp = case.d_kp.cpu().numpy()
    touched = np.zeros(kp.shape[:3], dtype=bool)
    for b, L in enumerate(case.lens):
        for t in range(L):
            touched[case.bt[b, t // 16], :, t % 16] = True
    assert np.all(kp[~touched] == 0xA5)


def test_many_short_pairs_cluster_path():
    # every request <= 4096 tokens: pairs segmented inside thread-block clusters; 512 pairs,
    # several per cluster and per shared-memory slot
    rng = np.random.default_rng(1)
    lens = rng.integers(1, 3000, 64).tolist()
    run(Case(lens, hq=32, hkv=8, bs=16, seed=11))


def test_many_pairs_two_cta_clusters():
    # at least 1024 pairs: the cluster path uses clusters of two CTAs; ragged lengths up to the
    # longest pair it takes, empty and one-token requests, shuffled blocks
    rng = np.random.default_rng(2)
    lens = rng.integers(1, 700, 130).tolist()
    lens[3], lens[7], lens[11], lens[20] = 0, 1, 4096, 16
    run(Case(lens, hq=16, hkv=8, bs=16, seed=13))


def test_short_pairs_cluster_path_edges():
    # the longest pair the cluster path takes (4096 tokens = 256 windows), one-window pairs,
    # empty requests, a partial last window, block size 64
    lens = [4096, 1, 0, 16, 17, 4095, 2048, 0, 255, 3333]
    run(Case(lens, hq=4, hkv=4, bs=64, seed=12))


def test_many_pairs_several_chunks_grid_path():
    # one request above 4096 tokens sends the call through the grid-wide kernel: ~50 K windows
    # in several 8192-window chunks, pairs crossing chunk and CTA-share edges
    rng = np.random.default_rng(2)
    lens = rng.integers(1, 3000, 64).tolist() + [5000]
    run(Case(lens, hq=32, hkv=8, bs=16, seed=14))


def test_grid_path_many_chunks():
    # 160 K windows: five 32768-window chunks, pairs of 1250 windows crossing chunk edges
    case = Case([20000] * 16, hq=8, hkv=8, bs=64, seed=15)
    run(case)
    assert compress_path(case) == PATH_GRID


def test_repeated_calls_reuse_workspace():
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case([100, 2500, 40], hq=4, hkv=4, bs=32, seed=13)
    kp, vp, table = run(case)
    for _ in range(3):  # same workspace, the epoch/flag protocol must reset itself
        case.d_kp.zero_()
        case.d_vp.zero_()
        dgq.dgq_compress(case.d_k, case.d_v, case.d_cu, case.max_seqlen, case.bs, case.d_bt, case.d_kp,
                         case.d_vp, case.d_table, case.d_cws)
        torch.cuda.synchronize()
        assert dgq.dgq_workspace_error(case.d_cws) == 0
        assert_compress_equal(case, kp, vp, table, case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(),
                              table_to_numpy(case.d_table))


def test_planted_boundaries_on_gpu():
    # K with sigma steps at window-aligned tokens (0.03 / 0.47 / 0.15 as in the DGQ example)
    import torch
    case = Case([4096], hq=1, hkv=1, bs=64, seed=3)
    rng = np.random.default_rng(0)
    k = np.zeros((4096, 1, 128), dtype=np.float32)
    for (s, e, sg) in ((0, 1024, 0.03), (1024, 2560, 0.47), (2560, 4096, 0.15)):
        k[s:e] = rng.standard_normal((e - s, 1, 128)) * sg
    bits = k.view(np.uint32)
    case.k = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    case.v = case.k.copy()
    run(case)
    tab = table_to_numpy(case.d_table)
    assert tab[0, 0]["n_seg"] == 3 and list(tab[0, 0]["start"][:3]) == [0, 1024, 2560]


def _tie_segments(n, rng):
    """n segments (min, max, xs) as bf16 bit patterns, xs in [min, max], chosen so that the fp32
    product (x - min) * (255 / (max - min)) rounds to exactly k + 0.5 although the exact product
    is not k + 0.5: there the method's two roundings (product, then to an integer, half to even)
    and a single fused rounding give different codes whenever k + 0.5 is closer to the odd
    neighbour."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    finite = np.isfinite(vals)
    lo_pool = bits[finite & (vals > -2.0) & (vals < -0.01)]
    hi_pool = bits[finite & (vals > 0.01) & (vals < 3.0)]
    out, flips = [], 0
    while len(out) < n:
        ab, bb = rng.choice(lo_pool), rng.choice(hi_pool)
        a, b = vals[ab], vals[bb]
        inside = finite & (vals >= a) & (vals <= b)
        xv = vals[inside]
        d = (xv - a).astype(np.float32)
        inv = np.float32(255.0) / np.float32(b - a)
        p = d.astype(np.float64) * np.float64(inv)       # exact: 24 x 24 bits
        u = p.astype(np.float32).astype(np.float64)
        tie = (u - np.floor(u) == 0.5) & (p != u)
        if tie.sum() >= 2:
            double = np.rint(u[tie])                      # the method: round the product, then half-even
            single = np.rint(p[tie])                      # one fused rounding
            flips += int((double != single).sum())
            out.append((ab, bb, bits[inside][tie]))
    return out, flips


def test_codes_at_rounding_ties():
    # every code of these segments sits where rounding the product once instead of twice would
    # change it: the codes must match the oracle's two IEEE roundings bit for bit
    lens = [32] * 4
    case = Case(lens, hq=2, hkv=2, bs=16, seed=21)
    rng = np.random.default_rng(21)
    segs, flips = _tie_segments(2 * 2 * len(lens) * 2, rng)  # (K, V) x heads x requests x 2 segments
    assert flips > 0
    it = iter(segs)
    for arr in (case.k, case.v):
        for b in range(len(lens)):
            for h in range(2):
                for s in range(2):  # L = 32: two windows, one cut, segments of 16 tokens
                    ab, bb, xs = next(it)
                    vals = np.resize(xs, 16 * 128).astype(np.uint16)
                    vals[0], vals[1] = ab, bb
                    r0 = case.cu[b] + 16 * s
                    arr[r0:r0 + 16, h, :] = vals.reshape(16, 128)
    run(case)


PATH_GRID, PATH_CLUSTER = 1, 2


def compress_path(case):
    """Which compress kernel the case's last call ran (word 1 of the workspace header)."""
    return int(case.d_cws[4:8].cpu().numpy().view(np.uint32)[0])


def test_paths_taken():
    # requests of at most 4096 tokens go to the cluster kernel, longer ones to the grid-wide one
    short = Case([37, 300, 4096], hq=4, hkv=2, bs=16, seed=35)
    run(short)
    assert compress_path(short) == PATH_CLUSTER
    lng = Case([37, 4097], hq=4, hkv=2, bs=16, seed=36)
    run(lng)
    assert compress_path(lng) == PATH_GRID
