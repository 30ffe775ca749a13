"""dgq_compress_paged on the GPU: compressing K/V read straight from a bf16 paged cache gives the
same records and codes, bit for bit, as the oracle compressing the same tokens in packed rows, on
both compress kernels and all block sizes; a source block id outside the cache is flagged."""
import numpy as np
import pytest

from dgq_cases import Case, assert_compress_equal, table_to_numpy

pytestmark = pytest.mark.gpu


def paged_source(case, seed, extra=3):
    """A bf16 paged cache holding the case's K and V through a shuffled source block table;
    slots past each request's end hold junk."""
    rng = np.random.default_rng(seed)
    nblk = [(int(L) + case.bs - 1) // case.bs for L in case.lens]
    nsrc = sum(nblk) + extra
    order = rng.permutation(nsrc).astype(np.int32)
    sbt = np.zeros((case.B, max(1, max(nblk))), dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        sbt[b, :n] = order[off:off + n]
        off += n
    ks = rng.integers(0, 1 << 16, (nsrc, case.hkv, case.bs, 128)).astype(np.uint16) & 0x3FFF  # junk
    vs = rng.integers(0, 1 << 16, (nsrc, case.hkv, case.bs, 128)).astype(np.uint16) & 0x3FFF
    for b in range(case.B):
        L = int(case.lens[b])
        t = np.arange(L)
        ks[sbt[b, t // case.bs], :, t % case.bs] = case.k[case.cu[b]:case.cu[b] + L]
        vs[sbt[b, t // case.bs], :, t % case.bs] = case.v[case.cu[b]:case.cu[b] + L]
    return ks, vs, sbt


def run_paged(case, ks, vs, sbt):
    import torch
    import int8_group_quantized_gb300 as dgq
    kp, vp, table = case.oracle_compress()
    case.gpu_compress()  # allocates the device buffers (and checks the packed path once more)
    case.d_kp.zero_()
    case.d_vp.zero_()
    case.d_table.zero_()
    dev = torch.device("cuda:0")
    d_ks = torch.from_numpy(ks.view(np.int16)).to(dev).view(torch.bfloat16)
    d_vs = torch.from_numpy(vs.view(np.int16)).to(dev).view(torch.bfloat16)
    d_sbt = torch.from_numpy(sbt).to(dev)
    dgq.dgq_compress_paged(d_ks, d_vs, d_sbt, case.d_cu, case.max_seqlen, case.bs, case.d_bt, case.d_kp,
                           case.d_vp, case.d_table, case.d_cws)
    torch.cuda.synchronize()
    return kp, vp, table, d_ks, d_vs, d_sbt


@pytest.mark.parametrize("bs", [16, 32, 64])
@pytest.mark.parametrize("lens", [[37, 300, 0, 4096, 1, 2047], [5000, 37, 20000, 0, 16]])
def test_paged_source_matches_oracle(bs, lens):
    import int8_group_quantized_gb300 as dgq
    case = Case(lens, hq=4, hkv=2, bs=bs, seed=80 + bs)
    ks, vs, sbt = paged_source(case, seed=bs)
    kp, vp, table, *_ = run_paged(case, ks, vs, sbt)
    assert dgq.dgq_workspace_error(case.d_cws) == 0
    assert_compress_equal(case, kp, vp, table, case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(),
                          table_to_numpy(case.d_table))


def test_paged_source_many_pairs():
    import int8_group_quantized_gb300 as dgq
    rng = np.random.default_rng(9)
    case = Case(rng.integers(1, 3000, 48).tolist(), hq=16, hkv=8, bs=16, seed=90)
    ks, vs, sbt = paged_source(case, seed=9)
    kp, vp, table, *_ = run_paged(case, ks, vs, sbt)
    assert dgq.dgq_workspace_error(case.d_cws) == 0
    assert_compress_equal(case, kp, vp, table, case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(),
                          table_to_numpy(case.d_table))


def test_paged_source_flags_block_outside_the_cache():
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case([300, 40], hq=2, hkv=2, bs=16, seed=91)
    ks, vs, sbt = paged_source(case, seed=91)
    sbt[0, 4] = ks.shape[0] + 2
    run_paged(case, ks, vs, sbt)
    assert dgq.dgq_workspace_error(case.d_cws) == 5
