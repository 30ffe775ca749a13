"""The per-call limits: a batch of the largest size the calls accept (8192 requests; the kernels
keep per-request prefixes on chip) through compression on both kernels, the two-phase path,
decode attention and the append, against the oracle -- codes and records bit-exact, attention
within the tolerance."""
import numpy as np
import pytest

import oracle
from dgq_cases import Case, assert_attn_close, assert_compress_equal, table_to_numpy
from test_gpu_append import grow_tables
from test_gpu_compress import PATH_CLUSTER, PATH_GRID, compress_path
from test_gpu_prefill import run_chunked, schedule_uniform

pytestmark = pytest.mark.gpu
MAX_BATCH = 8192


def _lens(seed, long_len=None):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 48, MAX_BATCH)
    lens[::97] = 0
    if long_len:
        lens[MAX_BATCH // 2] = long_len
    return lens.tolist()


@pytest.mark.parametrize("long_len,path", [(None, PATH_CLUSTER), (5000, PATH_GRID)])
def test_largest_batch_compress_decode_append(long_len, path):
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case(_lens(81 + bool(long_len), long_len), hq=4, hkv=2, bs=16, seed=81)
    grow_tables(case, 1)  # a fresh block for each request whose next token starts one
    kp, vp, table = case.oracle_compress()
    case.gpu_compress()
    assert compress_path(case) == path
    assert_compress_equal(case, kp, vp, table, case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(),
                          table_to_numpy(case.d_table))
    assert_attn_close(case.oracle_attn(kp, vp, table), case.gpu_attn())
    # one appended token per pair (every request has room in its last block or a fresh one)
    assert oracle.append(case.knew, case.vnew, case.bs, case.bt, kp, vp, table) == 0
    ws = torch.zeros(dgq.dgq_append_workspace_size(), dtype=torch.uint8, device="cuda:0")
    dgq.dgq_append(case.d_knew, case.d_vnew, case.bs, case.d_bt, case.d_kp, case.d_vp, case.d_table, ws)
    torch.cuda.synchronize()
    assert np.array_equal(case.d_kp.cpu().numpy(), kp) and np.array_equal(case.d_vp.cpu().numpy(), vp)
    assert table_to_numpy(case.d_table).tobytes() == table.tobytes()


def test_largest_batch_two_phase():
    case = Case(_lens(83), hq=2, hkv=2, bs=16, seed=83)
    kp, vp, table = case.oracle_compress()
    g_kp, g_vp, g_table = run_chunked(case, schedule_uniform(case.lens, 32), src_seed=83)
    assert_compress_equal(case, kp, vp, table, g_kp, g_vp, g_table)
