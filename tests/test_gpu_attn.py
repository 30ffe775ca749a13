"""dgq_paged_decode_attn on the GPU against the oracle's fp64 attention over the same
dequantised cache (max |diff| <= 1e-2, mean |diff| <= 1e-3), plus invariants: bitwise
stability under physical-block permutation and across runs, GQA group sizes, empty caches,
ragged tails, and a cache of arbitrary codes that did not come from compression."""
import numpy as np
import pytest

import oracle
import synth
from dgq_cases import Case, assert_attn_close, bf16_to_f32, table_to_numpy

pytestmark = pytest.mark.gpu


def compress_and_attend(case):
    kp, vp, table = case.oracle_compress()
    case.gpu_compress()
    ref = case.oracle_attn(kp, vp, table)
    got = case.gpu_attn()
    assert_attn_close(ref, got)
    return ref, got


def test_tiny_workload():
    compress_and_attend(Case([37, 300], hq=4, hkv=2, bs=16, seed=0, rule=0))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (16, 2)])
def test_group_sizes(hq, hkv):
    compress_and_attend(Case([5, 64, 65, 700, 3000], hq=hq, hkv=hkv, bs=16, seed=hq + hkv))


@pytest.mark.parametrize("bs", [16, 32, 64])
def test_block_sizes_and_ragged_tails(bs):
    compress_and_attend(Case([1, 63, 64, 65, 129, 1000, 4097], hq=8, hkv=2, bs=bs, seed=40 + bs))


def test_empty_cache_returns_current_value():
    case = Case([0, 3, 0], hq=4, hkv=2, bs=16, seed=9)
    ref, got = compress_and_attend(case)
    vn = bf16_to_f32(case.vnew)
    for hq in range(4):
        assert np.array_equal(got[0, hq], vn[0, hq // 2])  # softmax over one key: exactly v_new


def test_long_sequence_many_pieces():
    compress_and_attend(Case([40000, 100], hq=8, hkv=2, bs=64, seed=17))


def test_block_permutation_is_bitwise_invariant():
    import torch
    case = Case([37, 300, 1200], hq=8, hkv=2, bs=16, seed=21)
    kp, vp, table = case.oracle_compress()
    case.gpu_compress()
    out1 = case.gpu_attn()
    perm = np.random.default_rng(5).permutation(case.num_blocks).astype(np.int64)  # new id of block i
    dev = case.d_kp.device
    tperm = torch.from_numpy(perm).to(dev)
    kp2 = torch.empty_like(case.d_kp)
    vp2 = torch.empty_like(case.d_vp)
    kp2[tperm] = case.d_kp
    vp2[tperm] = case.d_vp
    case.d_bt = torch.from_numpy(perm[case.bt].astype(np.int32)).to(dev)
    out2 = case.gpu_attn(kp=kp2, vp=vp2)
    assert np.array_equal(out1, out2)


def test_run_to_run_determinism():
    case = Case([3000, 70, 9000], hq=8, hkv=2, bs=32, seed=23)
    case.gpu_compress()
    a = case.gpu_attn()
    b = case.gpu_attn()
    assert np.array_equal(a, b)


def test_arbitrary_codes_and_records():
    """Decode alone: random codes, random (valid) segment records, no compression involved."""
    import torch
    case = Case([37, 300, 2000], hq=8, hkv=4, bs=16, seed=31)
    n = case.num_blocks * case.hkv * case.bs * 128
    kp = synth.fill_bytes(31, synth.STREAM_CODES, 0, n).reshape(case.num_blocks, case.hkv, case.bs, 128)
    vp = synth.fill_bytes(32, synth.STREAM_CODES, 0, n).reshape(case.num_blocks, case.hkv, case.bs, 128)
    table = np.zeros((case.B, case.hkv), dtype=oracle.SEG_DTYPE)
    rng = np.random.default_rng(3)
    for b, L in enumerate(case.lens):
        for h in range(case.hkv):
            W = (L + 15) // 16
            k = min(oracle.ngroups(int(L)), W) - 1
            cuts = sorted(rng.choice(np.arange(1, W), size=k, replace=False).tolist()) if k else []
            rec = table[b, h]
            rec["n_seg"], rec["seq_len"] = k + 1, L
            rec["start"][:] = L
            rec["start"][:k + 1] = [0] + [16 * c for c in cuts]
            rec["k_min"][:k + 1] = rng.uniform(-2, 0, k + 1)
            rec["k_scale"][:k + 1] = rng.uniform(0, 0.02, k + 1)
            rec["v_min"][:k + 1] = rng.uniform(-2, 0, k + 1)
            rec["v_scale"][:k + 1] = rng.uniform(0, 0.02, k + 1)
            if k:
                rec["v_scale"][1] = 0.0  # flat segments with non-zero codes decode to min
                rec["k_scale"][k] = 0.0
    ref = case.oracle_attn(kp, vp, table)
    dev = torch.device("cuda:0")
    case.d_bt = torch.from_numpy(case.bt).to(dev)
    case.d_lens = torch.from_numpy(case.lens).to(dev)
    d_table = torch.from_numpy(table.view(np.uint8).reshape(case.B, case.hkv, 128).copy()).to(dev)
    got = case.gpu_attn(table=d_table, kp=torch.from_numpy(kp).to(dev), vp=torch.from_numpy(vp).to(dev))
    assert_attn_close(ref, got)


MERGE_BLOCK, MERGE_WARP = 3, 4  # word 1 of the decode workspace header: the merge kernel that ran


@pytest.mark.parametrize("lens,hq,hkv,expect", [
    # 256 pairs of 13 tiles over at most 3 CTAs per SM: at least one pair per two decode CTAs, so
    # the one-warp-per-item merge runs, and each pair is split over two or three CTAs
    ([200] * 128, 8, 2, MERGE_WARP),
    # 16 pairs of 188 tiles: each split over dozens of CTAs, merged by whole CTAs
    ([3000] * 8, 8, 2, MERGE_BLOCK),
])
def test_both_merge_kernels_with_split_pairs(lens, hq, hkv, expect):
    case = Case(lens, hq=hq, hkv=hkv, bs=16, seed=61 + len(lens))
    compress_and_attend(case)
    assert int(case.d_aws[4:8].cpu().numpy().view(np.uint32)[0]) == expect


def _empty_slices(lens, hkv, ncta, piece_cost):
    """CTAs of the decode kernel whose slice holds no tile when the flat tile list (16-token tiles,
    at least one per pair) is split evenly by cost, a pair costing its tiles plus piece_cost: a
    model of the launch layout, used only to show that a case reaches the path it is meant for."""
    tiles = [max(1, -(-int(L) // 16)) for L in lens for _ in range(hkv)]
    C = sum(tiles) + piece_cost * len(tiles)
    starts, pos = [], 0  # cost position of every tile
    for n in tiles:
        starts.extend(range(pos + piece_cost, pos + piece_cost + n))
        pos += piece_cost + n
    held = set(((p + 1) * ncta - 1) // C for p in starts)
    return ncta - len(held)


@pytest.mark.parametrize("B,lmax,expect", [
    (150, 100, MERGE_WARP),   # 300 short pairs: one pair per two CTAs or more, warp merge
    (100, 200, MERGE_BLOCK),  # 200 short pairs: fewer, block merge
])
def test_split_pairs_around_empty_slices(B, lmax, expect):
    # Many short pairs: the per-piece charge of the cost split exceeds some CTAs' share of the
    # total cost, so those CTAs hold no tile although the tiles outnumber the CTAs; the merges must
    # skip their slots.  Word 3 of the decode workspace header is 0 when some slice is empty.
    import torch
    lens = np.random.default_rng(B).integers(0, lmax + 1, B).astype(np.int32)
    hkv = 2
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    ncta = min(3 * nsm, B * hkv * -(-int(lens.max()) // 16))
    assert sum(hkv * max(1, -(-int(L) // 16)) for L in lens) >= ncta
    assert _empty_slices(lens, hkv, ncta, piece_cost=10) > 0  # the kernel's charge per piece end
    case = Case(lens, hq=8, hkv=hkv, bs=16, seed=90 + B)
    compress_and_attend(case)
    words = case.d_aws[:16].cpu().numpy().view(np.uint32)
    assert int(words[1]) == expect and int(words[3]) == 0
