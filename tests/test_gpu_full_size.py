"""Whole-workload parity: the first and the last layer of every workload at its full shape,
compressed and decoded by the same calls and launch configuration the benchmark times, and
compared with the oracle over every request -- every record and every code byte-exact (the whole
INT8 pools, which start zeroed on both sides, so untouched slots are compared too), every query
head's decode output within the attention tolerance (max |diff| over the layer, mean |diff| per
request).  The two-phase compression (statistics per prefill chunk, chunked as the benchmark
chunks it, then the finish) is held to the same bytes."""
import numpy as np
import pytest

from synth import configs
import synth
from dgq_cases import ATTN_MAX_ABS, ATTN_MEAN_ABS, bf16_to_f32
from parity_full import draw_layer, oracle_layer

pytestmark = pytest.mark.gpu
D = 128


def _dev_bf16(a, dev):
    import torch
    return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)


def _check_pools(what, hl, g_kp, g_vp, g_tab):
    if g_tab.tobytes() != hl.table.tobytes():
        bad = [idx for idx in np.ndindex(hl.table.shape) if g_tab[idx].tobytes() != hl.table[idx].tobytes()]
        raise AssertionError(f"{what}: {len(bad)} records differ, first {bad[0]}: oracle {hl.table[bad[0]]} "
                             f"gpu {g_tab[bad[0]]}")
    for name, ref, got in (("K", hl.kp, g_kp), ("V", hl.vp, g_vp)):
        if not np.array_equal(ref, got):
            bad = np.argwhere(ref != got)
            raise AssertionError(f"{what}: {name} pool differs in {len(bad)} bytes, first at "
                                 f"[block, head, slot, d] = {bad[0].tolist()}")


def _check_attn(hl, got):
    diff = np.abs(hl.out - got)
    assert np.isfinite(got).all()
    assert diff.max() <= ATTN_MAX_ABS, f"max |diff| {diff.max():.3e}"
    per_req = diff.reshape(diff.shape[0], -1).mean(axis=1)
    assert per_req.max() <= ATTN_MEAN_ABS, f"request {int(per_req.argmax())}: mean |diff| {per_req.max():.3e}"


def _layers(w):
    return sorted({0, w.layers - 1})


@pytest.mark.parametrize("cfg", ["2", "3", "4", "5", "5p"])
def test_full_size_every_request(cfg):
    import torch
    import int8_group_quantized_gb300 as dgq
    w = configs.WORKLOADS[int(cfg) if cfg.isdigit() else cfg]
    B, Hq, Hkv, bs = w.batch, w.hq, w.hkv, w.block_size
    dev = torch.device("cuda:0")
    sp = torch.cuda.current_stream().cuda_stream
    for layer in _layers(w):
        hl = oracle_layer(w, draw_layer(w, layer))
        T, ms, nb = int(hl.cu[-1]), int(hl.lens.max()), hl.num_blocks
        d_cu, d_bt, d_len = (torch.from_numpy(x).to(dev) for x in (hl.cu, hl.bt, hl.lens))
        k, v = _dev_bf16(hl.k, dev), _dev_bf16(hl.v, dev)
        # the benchmark draws the same tensors on the device: the generator gives the same bits
        tabs = tuple(torch.from_numpy(x).to(dev) for x in synth.span_tables(w.seed, layer, hl.lens, Hkv, w.rule))
        kd = torch.empty_like(k)
        synth.dev_fill_layer(w.seed, synth.STREAM_K, layer, d_cu, Hkv, tabs, T, kd, sp)
        torch.cuda.synchronize()
        assert torch.equal(kd.view(torch.int16), k.view(torch.int16)), "device generator differs from the host's"
        del kd
        q, kn, vn = (_dev_bf16(x, dev) for x in (hl.q, hl.knew, hl.vnew))
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
        rec = dgq.seg_record_dtype()
        _check_pools(f"layer {layer} one-shot", hl, kp.cpu().numpy(), vp.cpu().numpy(),
                     table.cpu().numpy().reshape(-1).view(rec).reshape(B, Hkv))
        _check_attn(hl, bf16_to_f32(out.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64))

        # two-phase: the bf16 paged cache a prefill writes (laid out like the INT8 pools), window
        # statistics chunk by chunk (about 64 MB of K/V per call, as the benchmark chunks it), finish
        ks = torch.zeros((nb, Hkv, bs, D), dtype=torch.bfloat16, device=dev)
        vs = torch.zeros_like(ks)
        blk = torch.from_numpy(np.concatenate([hl.bt[b, np.arange(int(L)) // bs] for b, L in enumerate(hl.lens)])
                               .astype(np.int64)).to(dev)
        slot = torch.from_numpy(np.concatenate([np.arange(int(L)) % bs for L in hl.lens]).astype(np.int64)).to(dev)
        ks[blk, :, slot, :] = k
        vs[blk, :, slot, :] = v
        del k, v
        C = int(min(16384, max(16, (64 << 20) // (B * Hkv * 512)))) // 16 * 16
        stats = torch.zeros((B, Hkv, (ms + 15) // 16, 8), dtype=torch.float32, device=dev)
        ws = torch.zeros(dgq.dgq_prefill_workspace_size(B, Hkv), dtype=torch.uint8, device=dev)
        for c in range((ms + C - 1) // C):
            beg = torch.from_numpy(np.minimum(c * C, hl.lens).astype(np.int32)).to(dev)
            end = torch.from_numpy(np.minimum((c + 1) * C, hl.lens).astype(np.int32)).to(dev)
            dgq.dgq_prefill_chunk_stats(ks, vs, d_bt, beg, end, ms, stats, ws, sp)
        kp.zero_()
        vp.zero_()
        table.zero_()
        dgq.dgq_prefill_finish(ks, vs, d_bt, d_len, ms, stats, d_bt, kp, vp, table, ws, sp)
        torch.cuda.synchronize()
        assert dgq.dgq_workspace_error(ws) == 0
        _check_pools(f"layer {layer} two-phase", hl, kp.cpu().numpy(), vp.cpu().numpy(),
                     table.cpu().numpy().reshape(-1).view(rec).reshape(B, Hkv))
        del ks, vs, kp, vp, stats
        torch.cuda.empty_cache()
