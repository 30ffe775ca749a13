"""Independent V segmentation on the GPU (two-phase compress with V's variance, then the decode
kernel's split instance) against the oracle: K and V pools and both record tables bit-exact,
decode attention within tolerance of fp64 attention over the K- and V-segmented caches."""
import numpy as np
import pytest

import oracle
from dgq_cases import Case, D, assert_attn_close, bf16_to_f32, table_to_numpy
from test_gpu_paged_source import paged_source
from test_gpu_prefill import schedule_ragged, schedule_uniform

pytestmark = pytest.mark.gpu


def restructure_v(case: Case, seed: int):
    """Give V a variance structure of its own: per request, one random window-aligned span of V
    scaled up by 3 and one scaled down by 4 (in bf16), so V's boundaries differ from K's."""
    rng = np.random.default_rng(seed)
    v = bf16_to_f32(case.v).copy()
    for b, L in enumerate(case.lens):
        W = int(L) // 16
        if W < 4:
            continue
        a, c = sorted(rng.choice(np.arange(1, W), 2, replace=False))
        r0 = int(case.cu[b])
        v[r0 + 16 * a:r0 + 16 * c] *= 3.0
        v[r0 + 16 * c:r0 + int(L)] *= 0.25
    bits = v.view(np.uint32).astype(np.uint64)
    case.v = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)


def run_split(case, schedule, src_seed, max_groups=5, min_var=0.0):
    import torch
    import int8_group_quantized_gb300 as dgq
    dev = torch.device("cuda:0")
    ks, vs, sbt = paged_source(case, seed=src_seed)
    d_ks = torch.from_numpy(ks.view(np.int16)).to(dev).view(torch.bfloat16)
    d_vs = torch.from_numpy(vs.view(np.int16)).to(dev).view(torch.bfloat16)
    d_sbt = torch.from_numpy(sbt).to(dev)
    case.d_bt = torch.from_numpy(case.bt).to(dev)
    case.d_lens = torch.from_numpy(case.lens).to(dev)
    W = (case.max_seqlen + 15) // 16
    stats = torch.full((case.B, case.hkv, W, 8), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.zeros(dgq.dgq_prefill_workspace_size(case.B, case.hkv), dtype=torch.uint8, device=dev)
    shape = (case.num_blocks, case.hkv, case.bs, 128)
    case.d_kp = torch.zeros(shape, dtype=torch.uint8, device=dev)
    case.d_vp = torch.zeros(shape, dtype=torch.uint8, device=dev)
    case.d_kt = torch.full((case.B, case.hkv, 128), 0x77, dtype=torch.uint8, device=dev)
    case.d_vt = torch.full((case.B, case.hkv, 128), 0x77, dtype=torch.uint8, device=dev)
    for beg, end in schedule:
        dgq.dgq_prefill_chunk_stats(d_ks, d_vs, d_sbt, torch.from_numpy(np.asarray(beg, np.int32)).to(dev),
                                    torch.from_numpy(np.asarray(end, np.int32)).to(dev), case.max_seqlen, stats, ws,
                                    v_variance=True)
    dgq.dgq_prefill_finish(d_ks, d_vs, d_sbt, case.d_lens, case.max_seqlen, stats, case.d_bt, case.d_kp, case.d_vp,
                           case.d_kt, ws, max_groups=max_groups, min_var=min_var, v_seg_table=case.d_vt)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    return (case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(), table_to_numpy(case.d_kt),
            table_to_numpy(case.d_vt))


def assert_split_equal(case, ref, got):
    kp, vp, kt, vt = ref
    g_kp, g_vp, g_kt, g_vt = got
    assert g_kt.tobytes() == kt.tobytes(), "K records differ"
    assert g_vt.tobytes() == vt.tobytes(), "V records differ"
    for b in range(case.B):
        L = int(case.lens[b])
        t = np.arange(L)
        blk, slot = case.bt[b, t // case.bs], t % case.bs
        for h in range(case.hkv):
            assert np.array_equal(kp[blk, h, slot], g_kp[blk, h, slot]), f"K codes differ: request {b} head {h}"
            assert np.array_equal(vp[blk, h, slot], g_vp[blk, h, slot]), f"V codes differ: request {b} head {h}"


def oracle_split_attn(case, kp, vp, kt, vt):
    out = np.zeros((case.B, case.hq, D))
    for b in range(case.B):
        L = int(case.lens[b])
        kd = np.stack([oracle.dequant_pair(kp, kt, case.bt, b, h, L, False) for h in range(case.hkv)], axis=1)
        vd = np.stack([oracle.dequant_pair(vp, vt, case.bt, b, h, L, True) for h in range(case.hkv)], axis=1)
        out[b] = oracle.decode_attn_dense(case.q[b], case.knew[b], case.vnew[b], kd.reshape(L, case.hkv, D),
                                          vd.reshape(L, case.hkv, D))
    return out


def gpu_split_attn(case):
    import torch
    import int8_group_quantized_gb300 as dgq
    dev = torch.device("cuda:0")
    d_q = torch.from_numpy(case.q.view(np.int16)).to(dev).view(torch.bfloat16)
    d_kn = torch.from_numpy(case.knew.view(np.int16)).to(dev).view(torch.bfloat16)
    d_vn = torch.from_numpy(case.vnew.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.zeros((case.B, case.hq, D), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(dgq.dgq_attn_workspace_size(case.B, case.hq, case.hkv, case.max_seqlen), dtype=torch.uint8,
                     device=dev)
    dgq.dgq_paged_decode_attn_split(d_q, d_kn, d_vn, case.d_kp, case.d_vp, case.d_kt, case.d_vt, case.d_bt,
                                    case.d_lens, case.max_seqlen, out, ws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    return bf16_to_f32(out.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


CASES = {
    "mixed_bs16": dict(lens=[37, 300, 0, 1, 2100, 129], hq=8, hkv=2, bs=16, seed=140),
    "long_bs64": dict(lens=[20000, 700], hq=4, hkv=2, bs=64, seed=141),
    "mha_bs32": dict(lens=[3000, 33, 5000], hq=4, hkv=4, bs=32, seed=142),
}


@pytest.mark.parametrize("name", list(CASES))
def test_split_compress_and_decode_match_oracle(name):
    case = Case(**CASES[name])
    restructure_v(case, seed=CASES[name]["seed"])
    ref = oracle.compress_split(case.k, case.v, case.cu, case.hkv, case.bs, case.bt, case.num_blocks)
    got = run_split(case, schedule_uniform(case.lens, 1024), src_seed=7)
    assert_split_equal(case, ref, got)
    # the V segmentations really differ from K's somewhere
    assert any(not np.array_equal(ref[2][b, h]["start"], ref[3][b, h]["start"])
               for b in range(case.B) for h in range(case.hkv) if case.lens[b] >= 2048)
    assert_attn_close(oracle_split_attn(case, *ref), gpu_split_attn(case))


def test_split_with_settings_and_ragged_chunks():
    case = Case([17000, 2500, 90], hq=8, hkv=2, bs=16, seed=143)
    restructure_v(case, seed=143)
    ref = oracle.compress_split(case.k, case.v, case.cu, case.hkv, case.bs, case.bt, case.num_blocks,
                                max_groups=4, min_var=0.02)
    got = run_split(case, schedule_ragged(case.lens, 9), src_seed=8, max_groups=4, min_var=0.02)
    assert_split_equal(case, ref, got)
    assert_attn_close(oracle_split_attn(case, *ref), gpu_split_attn(case))


def test_v_variance_statistics_leave_the_shared_path_unchanged():
    """Statistics taken with V's variance, finished without a V table: the method's shared
    segmentation, identical to the oracle's compress."""
    import torch
    import int8_group_quantized_gb300 as dgq
    from dgq_cases import assert_compress_equal
    case = Case([300, 2100], hq=4, hkv=2, bs=16, seed=144)
    restructure_v(case, seed=144)
    kp, vp, table = case.oracle_compress()
    dev = torch.device("cuda:0")
    ks, vs, sbt = paged_source(case, seed=9)
    d_ks = torch.from_numpy(ks.view(np.int16)).to(dev).view(torch.bfloat16)
    d_vs = torch.from_numpy(vs.view(np.int16)).to(dev).view(torch.bfloat16)
    d_sbt = torch.from_numpy(sbt).to(dev)
    stats = torch.zeros((case.B, case.hkv, (case.max_seqlen + 15) // 16, 8), dtype=torch.float32, device=dev)
    ws = torch.zeros(dgq.dgq_prefill_workspace_size(case.B, case.hkv), dtype=torch.uint8, device=dev)
    shape = (case.num_blocks, case.hkv, case.bs, 128)
    g_kp = torch.zeros(shape, dtype=torch.uint8, device=dev)
    g_vp = torch.zeros(shape, dtype=torch.uint8, device=dev)
    g_t = torch.zeros((case.B, case.hkv, 128), dtype=torch.uint8, device=dev)
    zeros = torch.zeros(case.B, dtype=torch.int32, device=dev)
    lens = torch.from_numpy(case.lens).to(dev)
    dgq.dgq_prefill_chunk_stats(d_ks, d_vs, d_sbt, zeros, lens, case.max_seqlen, stats, ws, v_variance=True)
    dgq.dgq_prefill_finish(d_ks, d_vs, d_sbt, lens, case.max_seqlen, stats, torch.from_numpy(case.bt).to(dev),
                           g_kp, g_vp, g_t, ws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    assert_compress_equal(case, kp, vp, table, g_kp.cpu().numpy(), g_vp.cpu().numpy(), table_to_numpy(g_t))


def test_split_append_matches_oracle_and_decodes():
    """Three decode steps appended through both record tables (one empty request among them), then
    the split decode over L + 3 tokens: pools and records bit-exact, attention within tolerance."""
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case([37, 300, 0, 2100, 129], hq=4, hkv=2, bs=16, seed=145, extra_blocks=8)
    restructure_v(case, seed=145)
    kp, vp, kt, vt = oracle.compress_split(case.k, case.v, case.cu, case.hkv, case.bs, case.bt, case.num_blocks)
    run_split(case, schedule_uniform(case.lens, 512), src_seed=11)
    # room for three more tokens per request: one of the unused blocks where a new block starts
    bt = np.concatenate([case.bt, np.zeros((case.B, 1), dtype=np.int32)], axis=1)
    used = {int(case.bt[b, i]) for b, L in enumerate(case.lens) for i in range((int(L) + case.bs - 1) // case.bs)}
    free = iter(sorted(set(range(case.num_blocks)) - used))
    for b, L in enumerate(case.lens):
        for t in range(int(L), int(L) + 3):
            if t % case.bs == 0:
                bt[b, t // case.bs] = next(free)
    case.bt = bt
    dev = torch.device("cuda:0")
    case.d_bt = torch.from_numpy(bt).to(dev)
    ws = torch.zeros(dgq.dgq_append_workspace_size(), dtype=torch.uint8, device=dev)
    rng = np.random.default_rng(146)
    for step in range(3):
        kn = bf16_bits_np(rng.standard_normal((case.B, case.hkv, D)).astype(np.float32) * 0.3)
        vn = bf16_bits_np(rng.standard_normal((case.B, case.hkv, D)).astype(np.float32) * 0.3)
        assert oracle.append_split(kn, vn, case.bs, bt, kp, vp, kt, vt) == 0
        d_kn = torch.from_numpy(kn.view(np.int16)).to(dev).view(torch.bfloat16)
        d_vn = torch.from_numpy(vn.view(np.int16)).to(dev).view(torch.bfloat16)
        dgq.dgq_append_split(d_kn, d_vn, case.bs, case.d_bt, case.d_kp, case.d_vp, case.d_kt, case.d_vt, ws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    case.lens = case.lens + 3
    case.d_lens = torch.from_numpy(case.lens).to(dev)
    case.max_seqlen = int(case.lens.max())
    assert_split_equal(case, (kp, vp, kt, vt), (case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(),
                                                table_to_numpy(case.d_kt), table_to_numpy(case.d_vt)))
    assert_attn_close(oracle_split_attn(case, kp, vp, kt, vt), gpu_split_attn(case))


def bf16_bits_np(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
