"""Full-size parity: one layer of each workload at its full shape, compressed and decoded by the
same calls and launch configuration the benchmark times, checked on sampled requests the oracle
computes one by one -- every code and record of the sampled requests bit-exact, and their
decode outputs (all query heads) within the attention tolerance."""
import numpy as np
import pytest

import oracle
import synth
from synth import configs
from dgq_cases import assert_attn_close, bf16_to_f32

pytestmark = pytest.mark.gpu
D = 128


def sampled(B):
    return sorted({0, B // 2, B - 1})


@pytest.mark.parametrize("cfg", ["2", "3", "4", "5", "5p"])
def test_full_size_sampled_requests(cfg):
    import torch
    import int8_group_quantized_gb300 as dgq
    w = configs.WORKLOADS[int(cfg) if cfg.isdigit() else cfg]
    lens = configs.seq_lens(w)
    bt, nb = configs.block_tables(w, lens)
    cu = configs.cu_seqlens(lens)
    B, Hq, Hkv, bs = w.batch, w.hq, w.hkv, w.block_size
    T, ms = int(cu[-1]), int(lens.max())
    dev = torch.device("cuda:0")
    sp = torch.cuda.current_stream().cuda_stream
    d_cu, d_bt, d_len = (torch.from_numpy(x).to(dev) for x in (cu, bt, lens))
    tabs = tuple(torch.from_numpy(x).to(dev) for x in synth.span_tables(w.seed, 0, lens, Hkv, w.rule))
    k = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    synth.dev_fill_layer(w.seed, synth.STREAM_K, 0, d_cu, Hkv, tabs, T, k, sp)
    synth.dev_fill_layer(w.seed, synth.STREAM_V, 0, d_cu, Hkv, tabs, T, v, sp)
    q = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    kn = torch.empty((B, Hkv, D), dtype=torch.bfloat16, device=dev)
    vn = torch.empty_like(kn)
    synth.dev_fill_heads(w.seed, synth.STREAM_Q, 0, B, Hq, 1.0, q, sp)
    synth.dev_fill_heads(w.seed, synth.STREAM_KNEW, 0, B, Hkv, 0.15, kn, sp)
    synth.dev_fill_heads(w.seed, synth.STREAM_VNEW, 0, B, Hkv, 0.15, vn, sp)
    kp = torch.zeros((nb, Hkv, bs, D), dtype=torch.uint8, device=dev)
    vp = torch.zeros_like(kp)
    table = torch.zeros((B, Hkv, 128), dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    cws = torch.zeros(dgq.dgq_compress_workspace_size(B, ms, Hkv), dtype=torch.uint8, device=dev)
    aws = torch.zeros(dgq.dgq_attn_workspace_size(B, Hq, Hkv, ms), dtype=torch.uint8, device=dev)
    dgq.dgq_compress(k, v, d_cu, ms, bs, d_bt, kp, vp, table, cws, sp)
    dgq.dgq_paged_decode_attn(q, kn, vn, kp, vp, table, d_bt, d_len, ms, out, aws, sp)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(cws) == 0 and dgq.dgq_workspace_error(aws) == 0
    g_tab = table.cpu().numpy().reshape(-1).view(dgq.seg_record_dtype()).reshape(B, Hkv)
    q_h = q.view(torch.int16).cpu().numpy().view(np.uint16)
    kn_h = kn.view(torch.int16).cpu().numpy().view(np.uint16)
    vn_h = vn.view(torch.int16).cpu().numpy().view(np.uint16)
    out_h = bf16_to_f32(out.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)

    for b in sampled(B):
        L = int(lens[b])
        kr = np.zeros((L, Hkv, D), dtype=np.uint16)
        vr = np.zeros_like(kr)
        for h in range(Hkv):
            n, st, sg = synth.spans(w.seed, 0, b, h, L, w.rule)
            kr[:, h] = synth.fill_pair(w.seed, synth.STREAM_K, 0, b, h, L, n, st, sg)
            vr[:, h] = synth.fill_pair(w.seed, synth.STREAM_V, 0, b, h, L, n, st, sg)
        nbr = max(1, (L + bs - 1) // bs)
        btr = np.arange(nbr, dtype=np.int32)[None]
        okp, ovp, otab = oracle.compress(kr, vr, np.array([0, L], dtype=np.int32), Hkv, bs, btr, nbr)
        assert g_tab[b].tobytes() == otab[0].tobytes(), f"request {b}: records differ"
        if L:
            t = np.arange(L)
            blocks = torch.from_numpy(bt[b, t // bs].astype(np.int64)).to(dev)
            slots = torch.from_numpy((t % bs).astype(np.int64)).to(dev)
            gk = kp[blocks, :, slots].cpu().numpy()          # [L, Hkv, D]
            gv = vp[blocks, :, slots].cpu().numpy()
            ok = okp[btr[0, t // bs], :, t % bs]
            ov = ovp[btr[0, t // bs], :, t % bs]
            assert np.array_equal(gk, ok), f"request {b}: K codes differ"
            assert np.array_equal(gv, ov), f"request {b}: V codes differ"
        ref = oracle.paged_decode_attn(q_h[b:b + 1], kn_h[b:b + 1], vn_h[b:b + 1], okp, ovp, otab, btr,
                                       np.array([L], dtype=np.int32))
        assert_attn_close(ref[0], out_h[b])


@pytest.mark.parametrize("cfg", ["2", "4", "5p"])
def test_full_size_two_phase_sampled_requests(cfg):
    """The two-phase compression at full size, chunked as the benchmark chunks it (about 64 MB of
    K/V per statistics call): the sampled requests' records and codes bit-exact with the oracle."""
    import torch
    import int8_group_quantized_gb300 as dgq
    w = configs.WORKLOADS[int(cfg) if cfg.isdigit() else cfg]
    lens = configs.seq_lens(w)
    bt, nb = configs.block_tables(w, lens)
    cu = configs.cu_seqlens(lens)
    B, Hkv, bs = w.batch, w.hkv, w.block_size
    T, ms = int(cu[-1]), int(lens.max())
    dev = torch.device("cuda:0")
    sp = torch.cuda.current_stream().cuda_stream
    d_cu, d_bt, d_len = (torch.from_numpy(x).to(dev) for x in (cu, bt, lens))
    tabs = tuple(torch.from_numpy(x).to(dev) for x in synth.span_tables(w.seed, 0, lens, Hkv, w.rule))
    k = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    synth.dev_fill_layer(w.seed, synth.STREAM_K, 0, d_cu, Hkv, tabs, T, k, sp)
    synth.dev_fill_layer(w.seed, synth.STREAM_V, 0, d_cu, Hkv, tabs, T, v, sp)
    # the bf16 paged cache the prefill writes, laid out like the INT8 pools
    ks = torch.zeros((nb, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
    vs = torch.zeros_like(ks)
    blk = torch.from_numpy(np.concatenate([bt[b, np.arange(int(L)) // bs] for b, L in enumerate(lens)])
                           .astype(np.int64)).to(dev)
    slot = torch.from_numpy(np.concatenate([np.arange(int(L)) % bs for L in lens]).astype(np.int64)).to(dev)
    ks[blk, :, slot, :] = k
    vs[blk, :, slot, :] = v
    C = int(min(16384, max(16, (64 << 20) // (B * Hkv * 512)))) // 16 * 16
    stats = torch.zeros((B, Hkv, (ms + 15) // 16, 8), dtype=torch.float32, device=dev)
    ws = torch.zeros(dgq.dgq_prefill_workspace_size(B, Hkv), dtype=torch.uint8, device=dev)
    for c in range((ms + C - 1) // C):
        beg = torch.from_numpy(np.minimum(c * C, lens).astype(np.int32)).to(dev)
        end = torch.from_numpy(np.minimum((c + 1) * C, lens).astype(np.int32)).to(dev)
        dgq.dgq_prefill_chunk_stats(ks, vs, d_bt, beg, end, ms, stats, ws, sp)
    kp = torch.zeros((nb, Hkv, bs, D), dtype=torch.uint8, device=dev)
    vp = torch.zeros_like(kp)
    table = torch.zeros((B, Hkv, 128), dtype=torch.uint8, device=dev)
    dgq.dgq_prefill_finish(ks, vs, d_bt, d_len, ms, stats, d_bt, kp, vp, table, ws, sp)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    g_tab = table.cpu().numpy().reshape(-1).view(dgq.seg_record_dtype()).reshape(B, Hkv)
    for b in sampled(B):
        L = int(lens[b])
        kr = np.zeros((L, Hkv, D), dtype=np.uint16)
        vr = np.zeros_like(kr)
        for h in range(Hkv):
            n, st, sg = synth.spans(w.seed, 0, b, h, L, w.rule)
            kr[:, h] = synth.fill_pair(w.seed, synth.STREAM_K, 0, b, h, L, n, st, sg)
            vr[:, h] = synth.fill_pair(w.seed, synth.STREAM_V, 0, b, h, L, n, st, sg)
        nbr = max(1, (L + bs - 1) // bs)
        btr = np.arange(nbr, dtype=np.int32)[None]
        okp, ovp, otab = oracle.compress(kr, vr, np.array([0, L], dtype=np.int32), Hkv, bs, btr, nbr)
        assert g_tab[b].tobytes() == otab[0].tobytes(), f"request {b}: records differ"
        if L:
            t = np.arange(L)
            blocks = torch.from_numpy(bt[b, t // bs].astype(np.int64)).to(dev)
            slots = torch.from_numpy((t % bs).astype(np.int64)).to(dev)
            assert np.array_equal(kp[blocks, :, slots].cpu().numpy(), okp[btr[0, t // bs], :, t % bs])
            assert np.array_equal(vp[blocks, :, slots].cpu().numpy(), ovp[btr[0, t // bs], :, t % bs])
