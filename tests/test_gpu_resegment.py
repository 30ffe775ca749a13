"""Re-segmentation after decode-step appends on the GPU, step by step against the oracle: each
step appends every request's token (dgq_append_ex, which reports the re-segmentation bits of
every pair), writes the token into the bf16 paged history, takes the statistics of each window a
request just completed and re-encodes exactly the flagged requests from their history
(dgq_prefill_finish_ex).  Flags, records and every pool byte must equal the oracle's
append-then-re-segment step; lengths cross 2048 and 16384 and fill windows on the way.  At the
end, dgq_compress_paged over the whole grown history must equal the oracle's compress of it."""
import numpy as np
import pytest

import oracle
import synth
from synth import configs
from dgq_cases import table_to_numpy

pytestmark = pytest.mark.gpu
D = 128


def _prefix(x, cu, lens):
    return np.concatenate([x[cu[b]:cu[b] + int(L)] for b, L in enumerate(lens)])


@pytest.mark.parametrize("mask", [oracle.RESEG_WINDOW | oracle.RESEG_NGROUPS, oracle.RESEG_NGROUPS])
def test_appends_with_resegmentation_match_oracle(mask):
    o_tab, redone = run_resegment_steps([2040, 300, 1000, 16380, 5, 2047, 0], 2, 16, 10, 51, mask)
    assert redone == (3 if mask == oracle.RESEG_NGROUPS else 5)  # the steps did re-segment
    assert o_tab[0, 0]["n_seg"] == 3 and o_tab[3, 0]["n_seg"] == 5  # 2048 and 16384 crossed


def run_resegment_steps(lens0, Hkv, bs, steps, seed, mask):
    """`steps` decode steps with re-segmentation on the GPU, each checked against the oracle;
    then the one-shot compress of the grown history.  Returns the oracle's final records and the
    number of request re-segmentations."""
    import torch
    import int8_group_quantized_gb300 as dgq
    dev = torch.device("cuda:0")
    lens0 = np.asarray(lens0, dtype=np.int32)
    full = lens0 + steps
    cu = configs.cu_seqlens(full)
    tabs = synth.span_tables(seed, 0, full, Hkv, synth.RULE_U)
    k = synth.fill_layer(seed, synth.STREAM_K, 0, cu, Hkv, tabs)
    v = synth.fill_layer(seed, synth.STREAM_V, 0, cu, Hkv, tabs)
    B = len(lens0)
    nblk = [(int(L) + bs - 1) // bs for L in full]
    nb = sum(nblk)
    perm = synth.permutation(seed, synth.STREAM_META, nb)
    bt = np.zeros((B, max(nblk)), dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n]
        off += n
    max_seqlen = int(full.max())
    W = (max_seqlen + 15) // 16

    # oracle state: the prefix compressed, then the steps
    cu0 = configs.cu_seqlens(lens0)
    o_kp, o_vp, o_tab = oracle.compress(_prefix(k, cu, lens0), _prefix(v, cu, lens0), cu0, Hkv, bs, bt, nb)

    # GPU state: the bf16 paged history (slots not yet generated hold junk), its window statistics
    # and the INT8 cache of the prefix, compressed in two phases
    rng = np.random.default_rng(seed)
    hk = (rng.integers(0, 1 << 16, (nb, Hkv, bs, D)) & 0x3FFF).astype(np.uint16)
    hv = (rng.integers(0, 1 << 16, (nb, Hkv, bs, D)) & 0x3FFF).astype(np.uint16)
    for b, L in enumerate(lens0):
        t = np.arange(int(L))
        hk[bt[b, t // bs], :, t % bs] = k[cu[b]:cu[b] + L]
        hv[bt[b, t // bs], :, t % bs] = v[cu[b]:cu[b] + L]
    d_hk = torch.from_numpy(hk.view(np.int16)).to(dev).view(torch.bfloat16)
    d_hv = torch.from_numpy(hv.view(np.int16)).to(dev).view(torch.bfloat16)
    d_bt = torch.from_numpy(bt).to(dev)
    d_cur = torch.from_numpy(lens0.copy()).to(dev)
    kp = torch.zeros((nb, Hkv, bs, D), dtype=torch.uint8, device=dev)
    vp = torch.zeros_like(kp)
    table = torch.zeros((B, Hkv, 128), dtype=torch.uint8, device=dev)
    stats = torch.zeros((B, Hkv, W, 8), dtype=torch.float32, device=dev)
    pws = torch.zeros(dgq.dgq_prefill_workspace_size(B, Hkv), dtype=torch.uint8, device=dev)
    aws = torch.zeros(dgq.dgq_append_workspace_size(), dtype=torch.uint8, device=dev)
    flags = torch.full((B, Hkv), -1, dtype=torch.int32, device=dev)
    zero = torch.zeros(B, dtype=torch.int32, device=dev)
    dgq.dgq_prefill_chunk_stats(d_hk, d_hv, d_bt, zero, d_cur, max_seqlen, stats, pws)
    dgq.dgq_prefill_finish(d_hk, d_hv, d_bt, d_cur, max_seqlen, stats, d_bt, kp, vp, table, pws)
    torch.cuda.synchronize()
    assert table_to_numpy(table).tobytes() == o_tab.tobytes()

    redone = 0
    for s in range(steps):
        cur = lens0 + s
        knew = np.stack([k[cu[b] + int(L)] for b, L in enumerate(cur)])
        vnew = np.stack([v[cu[b] + int(L)] for b, L in enumerate(cur)])
        grown = cur + 1
        o_flags, skipped = oracle.append_resegment(knew, vnew, bs, bt, o_kp, o_vp, o_tab, _prefix(k, cu, grown),
                                                   _prefix(v, cu, grown), configs.cu_seqlens(grown), mask=mask)
        assert skipped == 0
        # the decode loop on the GPU: no host round trip between its calls
        d_kn = torch.from_numpy(knew.view(np.int16)).to(dev).view(torch.bfloat16)
        d_vn = torch.from_numpy(vnew.view(np.int16)).to(dev).view(torch.bfloat16)
        dgq.dgq_append_ex(d_kn, d_vn, bs, d_bt, kp, vp, table, flags, aws)
        blk = d_bt[torch.arange(B, device=dev), (d_cur // bs).long()].long()
        d_hk[blk, :, (d_cur % bs).long()] = d_kn  # the step's own bf16 K/V into the history
        d_hv[blk, :, (d_cur % bs).long()] = d_vn
        d_cur += 1
        done = (flags & dgq.RESEG_WINDOW).amax(dim=1) > 0  # requests that completed a window
        beg = torch.where(done, d_cur - 16, zero)
        end = torch.where(done, d_cur, zero)
        dgq.dgq_prefill_chunk_stats(d_hk, d_hv, d_bt, beg, end, max_seqlen, stats, pws)
        dgq.dgq_prefill_finish_ex(d_hk, d_hv, d_bt, d_cur, max_seqlen, stats, d_bt, kp, vp, table, pws, flags,
                                  flag_mask=mask)
        torch.cuda.synchronize()
        assert dgq.dgq_workspace_error(aws) == 0 and dgq.dgq_workspace_error(pws) == 0
        assert np.array_equal(flags.cpu().numpy(), o_flags), (s, flags.cpu().numpy(), o_flags)
        g_tab = table_to_numpy(table)
        assert g_tab.tobytes() == o_tab.tobytes(), s
        assert np.array_equal(kp.cpu().numpy(), o_kp) and np.array_equal(vp.cpu().numpy(), o_vp), s
        redone += int(((o_flags & mask).max(axis=1) > 0).sum())
    final_tab = o_tab.copy()

    # the whole grown history through the one-shot compress from the paged cache
    grown = lens0 + steps
    f_kp, f_vp, f_tab = oracle.compress(_prefix(k, cu, grown), _prefix(v, cu, grown), configs.cu_seqlens(grown),
                                        Hkv, bs, bt, nb)
    cws = torch.zeros(dgq.dgq_compress_workspace_size(B, max_seqlen, Hkv), dtype=torch.uint8, device=dev)
    kp.zero_()
    vp.zero_()
    d_cu = torch.from_numpy(configs.cu_seqlens(grown)).to(dev)
    dgq.dgq_compress_paged(d_hk, d_hv, d_bt, d_cu, max_seqlen, bs, d_bt, kp, vp, table, cws)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(cws) == 0
    assert table_to_numpy(table).tobytes() == f_tab.tobytes()
    assert np.array_equal(kp.cpu().numpy(), f_kp) and np.array_equal(vp.cpu().numpy(), f_vp)
    return final_tab, redone
