"""Compression in two phases for chunked prefill on the GPU: window statistics taken chunk by
chunk from a bf16 paged cache, then segmentation and codes in one finishing call, give the same
records and codes, bit for bit, as the oracle compressing each complete request -- for any chunk
schedule (uniform, ragged, out of order), block size and group-selection setting."""
import numpy as np
import pytest

from dgq_cases import Case, assert_compress_equal, table_to_numpy
from test_gpu_paged_source import paged_source

pytestmark = pytest.mark.gpu


def schedule_uniform(lens, C):
    """Chunks of C tokens (C a multiple of 16) across all requests at once."""
    n = (int(max(lens)) + C - 1) // C
    return [(np.minimum(c * C, lens), np.minimum((c + 1) * C, lens)) for c in range(max(n, 1))]


def schedule_ragged(lens, seed):
    """Per request, random window-aligned cut points; chunk c of every request in call c."""
    rng = np.random.default_rng(seed)
    cuts = []
    for L in lens:
        W = (int(L) + 15) // 16
        inner = sorted(set(rng.integers(1, max(W, 2), size=rng.integers(0, 5)).tolist())) if W > 1 else []
        cuts.append([0] + [16 * w for w in inner if 16 * w < L] + [int(L)])
    n = max(len(c) - 1 for c in cuts)
    out = []
    for i in range(n):
        beg = np.array([c[min(i, len(c) - 1)] for c in cuts], dtype=np.int32)
        end = np.array([c[min(i + 1, len(c) - 1)] for c in cuts], dtype=np.int32)
        out.append((beg, end))
    return out


def run_chunked(case, schedule, src_seed, max_groups=5, min_var=0.0):
    import torch
    import int8_group_quantized_gb300 as dgq
    dev = torch.device("cuda:0")
    ks, vs, sbt = paged_source(case, seed=src_seed)
    d_ks = torch.from_numpy(ks.view(np.int16)).to(dev).view(torch.bfloat16)
    d_vs = torch.from_numpy(vs.view(np.int16)).to(dev).view(torch.bfloat16)
    d_sbt = torch.from_numpy(sbt).to(dev)
    d_bt = torch.from_numpy(case.bt).to(dev)
    d_lens = torch.from_numpy(case.lens).to(dev)
    W = (case.max_seqlen + 15) // 16
    stats = torch.full((case.B, case.hkv, W, 8), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.zeros(dgq.dgq_prefill_workspace_size(case.B, case.hkv), dtype=torch.uint8, device=dev)
    shape = (case.num_blocks, case.hkv, case.bs, 128)
    kp = torch.zeros(shape, dtype=torch.uint8, device=dev)
    vp = torch.zeros(shape, dtype=torch.uint8, device=dev)
    table = torch.full((case.B, case.hkv, 128), 0x77, dtype=torch.uint8, device=dev)
    for beg, end in schedule:
        dgq.dgq_prefill_chunk_stats(d_ks, d_vs, d_sbt, torch.from_numpy(np.asarray(beg, np.int32)).to(dev),
                                    torch.from_numpy(np.asarray(end, np.int32)).to(dev), case.max_seqlen, stats, ws)
    dgq.dgq_prefill_finish(d_ks, d_vs, d_sbt, d_lens, case.max_seqlen, stats, d_bt, kp, vp, table, ws,
                           max_groups=max_groups, min_var=min_var)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    return kp.cpu().numpy(), vp.cpu().numpy(), table_to_numpy(table)


def check(case, schedule, src_seed, max_groups=5, min_var=0.0):
    kp, vp, table = case.oracle_compress(max_groups=max_groups, min_var=min_var)
    g_kp, g_vp, g_table = run_chunked(case, schedule, src_seed, max_groups, min_var)
    assert_compress_equal(case, kp, vp, table, g_kp, g_vp, g_table)


@pytest.mark.parametrize("bs", [16, 32, 64])
def test_uniform_chunks_match_oracle(bs):
    case = Case([37, 300, 0, 1, 16, 129, 2500], hq=4, hkv=2, bs=bs, seed=110 + bs)
    check(case, schedule_uniform(case.lens, 256), src_seed=bs)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_ragged_chunks_match_oracle(seed):
    rng = np.random.default_rng(seed)
    case = Case(rng.integers(0, 1500, 9).tolist(), hq=8, hkv=2, bs=16, seed=120 + seed)
    check(case, schedule_ragged(case.lens, seed), src_seed=seed)


def test_chunks_out_of_order_and_whole_request():
    case = Case([700, 33, 2048], hq=4, hkv=4, bs=32, seed=130)
    sched = schedule_uniform(case.lens, 512)
    check(case, sched[::-1], src_seed=5)
    check(case, [(np.zeros(3, np.int32), case.lens)], src_seed=5)  # one chunk: the whole prompt


def test_long_request_segmentation_over_many_windows():
    # 20000 tokens: 1250 windows, more than one strided pass of the segmentation CTA; five segments
    case = Case([20000, 100], hq=8, hkv=2, bs=64, seed=131)
    check(case, schedule_uniform(case.lens, 4096), src_seed=6)


@pytest.mark.parametrize("max_groups,min_var", [(3, 0.0), (5, 0.05), (2, 0.01)])
def test_group_settings_match_oracle(max_groups, min_var):
    case = Case([3000, 17000, 40], hq=4, hkv=2, bs=16, seed=132)
    check(case, schedule_uniform(case.lens, 1024), src_seed=7, max_groups=max_groups, min_var=min_var)


def test_misaligned_chunk_is_flagged():
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case([300], hq=2, hkv=1, bs=16, seed=133)
    dev = torch.device("cuda:0")
    ks, vs, sbt = paged_source(case, seed=8)
    d_ks = torch.from_numpy(ks.view(np.int16)).to(dev).view(torch.bfloat16)
    d_vs = torch.from_numpy(vs.view(np.int16)).to(dev).view(torch.bfloat16)
    stats = torch.zeros((1, 1, 19, 8), dtype=torch.float32, device=dev)
    ws = torch.zeros(dgq.dgq_prefill_workspace_size(1, 1), dtype=torch.uint8, device=dev)
    beg = torch.tensor([8], dtype=torch.int32, device=dev)  # not a window boundary
    end = torch.tensor([100], dtype=torch.int32, device=dev)
    dgq.dgq_prefill_chunk_stats(d_ks, d_vs, torch.from_numpy(sbt).to(dev), beg, end, 300, stats, ws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 6  # kErrBadLength
    assert not stats.any()


def test_window_statistics_bit_exact():
    """The statistics array itself against the oracle, window by window: K's and V's mean
    variance (balanced fp32 sums, as the oracle fixes them) and the K/V extremes, bit for bit."""
    import torch
    import int8_group_quantized_gb300 as dgq
    import oracle
    case = Case([37, 300, 1, 2100], hq=4, hkv=2, bs=16, seed=134)
    dev = torch.device("cuda:0")
    ks, vs, sbt = paged_source(case, seed=10)
    d_ks = torch.from_numpy(ks.view(np.int16)).to(dev).view(torch.bfloat16)
    d_vs = torch.from_numpy(vs.view(np.int16)).to(dev).view(torch.bfloat16)
    W = (case.max_seqlen + 15) // 16
    stats = torch.full((case.B, case.hkv, W, 8), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.zeros(dgq.dgq_prefill_workspace_size(case.B, case.hkv), dtype=torch.uint8, device=dev)
    for beg, end in schedule_ragged(case.lens, 11):
        dgq.dgq_prefill_chunk_stats(d_ks, d_vs, torch.from_numpy(sbt).to(dev),
                                    torch.from_numpy(np.asarray(beg, np.int32)).to(dev),
                                    torch.from_numpy(np.asarray(end, np.int32)).to(dev), case.max_seqlen, stats, ws,
                                    v_variance=True)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    got = stats.cpu().numpy()
    for b in range(case.B):
        L = int(case.lens[b])
        rows = slice(int(case.cu[b]), int(case.cu[b + 1]))
        for h in range(case.hkv):
            k, v = case.k[rows, h], case.v[rows, h]
            km = oracle.window_means(np.array([oracle.token_variance(r) for r in k], dtype=np.float32))
            vm = oracle.window_means(np.array([oracle.token_variance(r) for r in v], dtype=np.float32))
            kf = (k.astype(np.uint32) << 16).view(np.float32)
            vf = (v.astype(np.uint32) << 16).view(np.float32)
            nw = (L + 15) // 16
            want = np.zeros((nw, 8), dtype=np.float32)
            want[:, 0], want[:, 5] = km, vm
            for w in range(nw):
                want[w, 1], want[w, 2] = kf[16 * w:16 * w + 16].min(), kf[16 * w:16 * w + 16].max()
                want[w, 3], want[w, 4] = vf[16 * w:16 * w + 16].min(), vf[16 * w:16 * w + 16].max()
            assert np.array_equal(got[b, h, :nw].view(np.uint32), want.view(np.uint32)), (b, h)
