"""Device-side guards against inconsistent inputs that only the GPU sees (block-table entries
and request lengths live in device memory): each kernel turns them into an error word in the
workspace and keeps every access inside its buffers; the workspace works again once
re-initialised."""
import numpy as np
import pytest

from dgq_cases import Case

pytestmark = pytest.mark.gpu
ERR_BAD_BLOCK, ERR_BAD_LENGTH = 5, 6


def fresh_ws(dgq, ws):
    dgq.dgq_workspace_init(ws)


def test_decode_flags_block_id_outside_the_pools():
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case([300, 37], hq=4, hkv=2, bs=16, seed=70)
    case.gpu_compress()
    case.gpu_attn()
    bad = case.d_bt.clone()
    bad[0, 3] = case.num_blocks + 7
    dgq.dgq_paged_decode_attn(case.d_q, case.d_knew, case.d_vnew, case.d_kp, case.d_vp, case.d_table, bad,
                              case.d_lens, case.max_seqlen, case.d_out, case.d_aws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(case.d_aws) == ERR_BAD_BLOCK
    fresh_ws(dgq, case.d_aws)
    case.gpu_attn()  # a valid call on the re-initialised workspace succeeds


def test_decode_flags_length_beyond_the_block_table():
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case([300, 37], hq=4, hkv=2, bs=16, seed=71)
    case.gpu_compress()
    case.gpu_attn()
    lens = case.d_lens.clone()
    lens[1] = case.max_blocks * case.bs + 100
    dgq.dgq_paged_decode_attn(case.d_q, case.d_knew, case.d_vnew, case.d_kp, case.d_vp, case.d_table, case.d_bt,
                              lens, case.max_seqlen, case.d_out, case.d_aws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(case.d_aws) == ERR_BAD_LENGTH


@pytest.mark.parametrize("lens", [[300, 2000], [300, 5000]])  # cluster kernel, grid-wide kernel
def test_compress_flags_block_id_outside_the_pools(lens):
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case(lens, hq=4, hkv=2, bs=16, seed=72)
    case.gpu_compress()
    bad = case.d_bt.clone()
    bad[1, 2] = -3
    dgq.dgq_compress(case.d_k, case.d_v, case.d_cu, case.max_seqlen, case.bs, bad, case.d_kp, case.d_vp,
                     case.d_table, case.d_cws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(case.d_cws) == ERR_BAD_BLOCK
    fresh_ws(dgq, case.d_cws)
    case.gpu_compress()


@pytest.mark.parametrize("lens,claimed", [([300, 2000], 1000), ([300, 5000], 4500)])
def test_compress_flags_request_longer_than_max_seqlen(lens, claimed):
    # max_seqlen sizes the workspace and picks the kernel; a longer request is refused on the GPU
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case(lens, hq=4, hkv=2, bs=16, seed=73)
    case.gpu_compress()
    dgq.dgq_compress(case.d_k, case.d_v, case.d_cu, claimed, case.bs, case.d_bt, case.d_kp, case.d_vp,
                     case.d_table, case.d_cws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(case.d_cws) == ERR_BAD_LENGTH
    fresh_ws(dgq, case.d_cws)
    case.gpu_compress()


def test_append_flags_block_id_outside_the_pools():
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case([20, 40], hq=2, hkv=2, bs=16, seed=74)
    case.gpu_compress()
    before = case.d_table.clone()
    bad = case.d_bt.clone()
    bad[0, 1] = case.num_blocks  # slot 20 of request 0 lies in column 1
    ws = torch.zeros(dgq.dgq_append_workspace_size(), dtype=torch.uint8, device="cuda:0")
    k = torch.zeros((2, 2, 128), dtype=torch.bfloat16, device="cuda:0")
    dgq.dgq_append(k, k, case.bs, bad, case.d_kp, case.d_vp, case.d_table, ws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == ERR_BAD_BLOCK
    assert torch.equal(case.d_table[0], before[0])
