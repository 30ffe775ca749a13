"""dgq_append on the GPU against the CPU oracle: after a compress, several decode steps'
tokens appended through the C ABI give the same pools and records bit for bit (codes of
in-range and clamped values, one-token first segments of empty requests, new blocks at
block edges), and decode attention over the grown cache matches the oracle's."""
import numpy as np
import pytest

import oracle
import synth
from dgq_cases import Case, assert_attn_close, bf16_to_f32, first_record_diff, table_to_numpy

pytestmark = pytest.mark.gpu
D = 128


def grow_tables(case, steps):
    """Extend the case's block table with fresh blocks for `steps` more tokens per request."""
    need = [(int(L) + steps + case.bs - 1) // case.bs for L in case.lens]
    have = [(int(L) + case.bs - 1) // case.bs for L in case.lens]
    mb = max(max(need), case.max_blocks)
    bt = np.zeros((case.B, mb), dtype=np.int32)
    bt[:, :case.max_blocks] = case.bt
    nxt = case.num_blocks
    for b in range(case.B):
        for j in range(have[b], need[b]):
            bt[b, j] = nxt
            nxt += 1
    case.bt, case.max_blocks, case.num_blocks = bt, mb, nxt


def step_tokens(seed, step, B, hkv, outliers=True):
    """The step's new K and V, bf16 bit patterns [B, Hkv, 128]: with `outliers`, wide values
    plus one far above and one far below every segment (they clamp); without, values of the
    spread of a decode step's own key and value (sigma 0.15)."""
    k = synth.fill_heads(seed, synth.STREAM_KNEW, 100 + step, B, hkv, 0.5 if outliers else 0.15)
    v = synth.fill_heads(seed, synth.STREAM_VNEW, 100 + step, B, hkv, 1.5 if outliers else 0.15)
    if outliers:
        k[:, :, 0] = 0x4120  # 10.0: above any segment built from the synthetic data
        v[:, :, 1] = 0xC120  # -10.0: below
    return k, v


def run_appends(case, steps, seed, outliers=True):
    import torch
    import int8_group_quantized_gb300 as dgq
    kp, vp, table = case.oracle_compress()
    case.gpu_compress()
    ws = torch.zeros(dgq.dgq_append_workspace_size(), dtype=torch.uint8, device="cuda:0")
    dev = torch.device("cuda:0")
    for s in range(steps):
        k, v = step_tokens(seed, s, case.B, case.hkv, outliers)
        assert oracle.append(k, v, case.bs, case.bt, kp, vp, table) == 0
        dk = torch.from_numpy(k.view(np.int16)).to(dev).view(torch.bfloat16)
        dv = torch.from_numpy(v.view(np.int16)).to(dev).view(torch.bfloat16)
        dgq.dgq_append(dk, dv, case.bs, case.d_bt, case.d_kp, case.d_vp, case.d_table, ws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    g_table = table_to_numpy(case.d_table)
    assert g_table.tobytes() == table.tobytes(), first_record_diff(table, g_table)
    g_kp, g_vp = case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy()
    assert np.array_equal(g_kp, kp), f"K pool differs at {np.argwhere(g_kp != kp)[:3].tolist()}"
    assert np.array_equal(g_vp, vp), f"V pool differs at {np.argwhere(g_vp != vp)[:3].tolist()}"
    return kp, vp, table


@pytest.mark.parametrize("bs", [16, 32, 64])
def test_appends_match_oracle(bs):
    # lengths at, just past and just before block edges, an empty request, a long one
    lens = [0, 1, bs - 1, bs, bs + 1, 37, 300, 2048, 5000]
    case = Case(lens, hq=8, hkv=2, bs=bs, seed=bs + 1)
    steps = bs + 3  # every request crosses at least one block edge
    grow_tables(case, steps)
    run_appends(case, steps, seed=bs)


def test_many_pairs_one_step():
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 3000, 64).tolist()
    case = Case(lens, hq=32, hkv=8, bs=16, seed=6)
    grow_tables(case, 1)
    run_appends(case, 1, seed=7)


def test_decode_attention_over_appended_cache():
    # tokens in the data's own spread (no planted outliers): outputs keep the magnitude the
    # attention tolerance is stated for (bf16 output rounding alone is 0.03 at |out| >= 8)
    import torch
    lens = [0, 15, 16, 300, 1000]
    case = Case(lens, hq=16, hkv=4, bs=16, seed=8)
    steps = 20
    grow_tables(case, steps)
    kp, vp, table = run_appends(case, steps, seed=9, outliers=False)
    case.lens = case.lens + steps
    case.d_lens = torch.from_numpy(case.lens).to("cuda:0")
    case.max_seqlen = int(case.lens.max())
    ref = case.oracle_attn(kp, vp, table)
    got = case.gpu_attn()
    assert_attn_close(ref, got)


def test_missing_block_column_is_flagged_and_nothing_written():
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case([32, 20], hq=2, hkv=2, bs=16, seed=10)  # request 0 full: no column for slot 32
    case.gpu_compress()
    before_kp, before_tab = case.d_kp.clone(), case.d_table.clone()
    ws = torch.zeros(dgq.dgq_append_workspace_size(), dtype=torch.uint8, device="cuda:0")
    k, v = step_tokens(11, 0, case.B, case.hkv)
    dk = torch.from_numpy(k.view(np.int16)).cuda().view(torch.bfloat16)
    dv = torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16)
    dgq.dgq_append(dk, dv, case.bs, case.d_bt, case.d_kp, case.d_vp, case.d_table, ws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) != 0
    assert torch.equal(case.d_table[0], before_tab[0])            # request 0 untouched
    assert table_to_numpy(case.d_table)[1, 0]["seq_len"] == 21    # request 1 appended
    blk0 = case.bt[0]
    assert torch.equal(case.d_kp[torch.from_numpy(blk0).long().cuda()],
                       before_kp[torch.from_numpy(blk0).long().cuda()])
