"""Shared helpers for the GPU parity tests: seeded inputs from `synth`, the CUDA path through
the C ABI binding, and element-wise comparison with the CPU oracle."""
from __future__ import annotations

import numpy as np

import oracle
import synth

D = 128
ATTN_MAX_ABS = 1e-2   # tolerance on decode attention vs the fp64 oracle (max |diff|)
ATTN_MEAN_ABS = 1e-3  # and mean |diff|


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


class Case:
    """One layer: batch of requests with given lengths, paged with a block table."""

    def __init__(self, lens, hq, hkv, bs, seed, layer=0, rule=synth.RULE_U, shuffle=True, extra_blocks=2):
        self.lens = np.asarray(lens, dtype=np.int32)
        self.B = len(lens)
        self.hq, self.hkv, self.bs, self.seed, self.layer = hq, hkv, bs, seed, layer
        self.cu = np.zeros(self.B + 1, dtype=np.int32)
        self.cu[1:] = np.cumsum(self.lens)
        self.tabs = synth.span_tables(seed, layer, self.lens, hkv, rule)
        self.k = synth.fill_layer(seed, synth.STREAM_K, layer, self.cu, hkv, self.tabs)
        self.v = synth.fill_layer(seed, synth.STREAM_V, layer, self.cu, hkv, self.tabs)
        self.q = synth.fill_heads(seed, synth.STREAM_Q, layer, self.B, hq, 1.0)
        self.knew = synth.fill_heads(seed, synth.STREAM_KNEW, layer, self.B, hkv, 0.15)
        self.vnew = synth.fill_heads(seed, synth.STREAM_VNEW, layer, self.B, hkv, 0.15)
        nblk = [(int(L) + bs - 1) // bs for L in self.lens]
        self.max_blocks = max(1, max(nblk))
        self.num_blocks = sum(nblk) + extra_blocks
        order = (synth.permutation(seed, synth.STREAM_META, self.num_blocks) if shuffle
                 else np.arange(self.num_blocks, dtype=np.int32))
        self.bt = np.zeros((self.B, self.max_blocks), dtype=np.int32)
        off = 0
        for b, n in enumerate(nblk):
            self.bt[b, :n] = order[off:off + n]
            off += n
        self.max_seqlen = int(max(1, self.lens.max()))

    # ---- oracle -------------------------------------------------------------------------
    def oracle_compress(self, max_groups=oracle.MAX_SEG, min_var=0.0):
        return oracle.compress(self.k, self.v, self.cu, self.hkv, self.bs, self.bt, self.num_blocks,
                               max_groups=max_groups, min_var=min_var)

    def oracle_attn(self, kp, vp, table):
        return oracle.paged_decode_attn(self.q, self.knew, self.vnew, kp, vp, table, self.bt, self.lens)

    # ---- CUDA path ---------------------------------------------------------------------------
    def gpu_compress(self, fill=0, max_groups=oracle.MAX_SEG, min_var=0.0):
        import torch
        import int8_group_quantized_gb300 as dgq
        dev = torch.device("cuda:0")
        self.d_k = torch.from_numpy(self.k.view(np.int16)).to(dev).view(torch.bfloat16)
        self.d_v = torch.from_numpy(self.v.view(np.int16)).to(dev).view(torch.bfloat16)
        if self.k.shape[0] == 0:
            self.d_k = torch.zeros((1, self.hkv, D), dtype=torch.bfloat16, device=dev)
            self.d_v = torch.zeros((1, self.hkv, D), dtype=torch.bfloat16, device=dev)
        self.d_cu = torch.from_numpy(self.cu).to(dev)
        self.d_bt = torch.from_numpy(self.bt).to(dev)
        self.d_lens = torch.from_numpy(self.lens).to(dev)
        shape = (self.num_blocks, self.hkv, self.bs, D)
        self.d_kp = torch.full(shape, fill, dtype=torch.uint8, device=dev)
        self.d_vp = torch.full(shape, fill, dtype=torch.uint8, device=dev)
        self.d_table = torch.zeros((self.B, self.hkv, 128), dtype=torch.uint8, device=dev)
        wsz = dgq.dgq_compress_workspace_size(self.B, self.max_seqlen, self.hkv)
        self.d_cws = torch.zeros(wsz, dtype=torch.uint8, device=dev)
        dgq.dgq_compress(self.d_k, self.d_v, self.d_cu, self.max_seqlen, self.bs, self.d_bt, self.d_kp,
                         self.d_vp, self.d_table, self.d_cws, max_groups=max_groups, min_var=min_var)
        torch.cuda.synchronize()
        assert dgq.dgq_workspace_error(self.d_cws) == 0

    def gpu_attn(self, table=None, kp=None, vp=None):
        import torch
        import int8_group_quantized_gb300 as dgq
        dev = torch.device("cuda:0")
        self.d_q = torch.from_numpy(self.q.view(np.int16)).to(dev).view(torch.bfloat16)
        self.d_knew = torch.from_numpy(self.knew.view(np.int16)).to(dev).view(torch.bfloat16)
        self.d_vnew = torch.from_numpy(self.vnew.view(np.int16)).to(dev).view(torch.bfloat16)
        self.d_out = torch.zeros((self.B, self.hq, D), dtype=torch.bfloat16, device=dev)
        wsz = dgq.dgq_attn_workspace_size(self.B, self.hq, self.hkv, self.max_seqlen)
        if not hasattr(self, "d_aws") or self.d_aws.numel() < wsz:
            self.d_aws = torch.zeros(wsz, dtype=torch.uint8, device=dev)
        dgq.dgq_paged_decode_attn(self.d_q, self.d_knew, self.d_vnew,
                                  self.d_kp if kp is None else kp, self.d_vp if vp is None else vp,
                                  self.d_table if table is None else table, self.d_bt, self.d_lens,
                                  self.max_seqlen, self.d_out, self.d_aws)
        torch.cuda.synchronize()
        assert dgq.dgq_workspace_error(self.d_aws) == 0
        return bf16_to_f32(self.d_out.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def table_to_numpy(d_table):
    import int8_group_quantized_gb300 as dgq
    raw = d_table.cpu().numpy()
    return raw.reshape(-1).view(dgq.seg_record_dtype()).reshape(d_table.shape[:2])


def assert_compress_equal(case: Case, kp, vp, table, g_kp, g_vp, g_table):
    """Bit-exact: every record, and every code of every written slot (tokens < L)."""
    assert g_table.tobytes() == table.tobytes(), first_record_diff(table, g_table)
    for b in range(case.B):
        L = int(case.lens[b])
        if L == 0:
            continue
        t = np.arange(L)
        blk = case.bt[b, t // case.bs]
        slot = t % case.bs
        for h in range(case.hkv):
            for ref, got, name in ((kp, g_kp, "K"), (vp, g_vp, "V")):
                r = ref[blk, h, slot]
                g = got[blk, h, slot]
                if not np.array_equal(r, g):
                    bad = np.argwhere(r != g)
                    raise AssertionError(f"{name} codes differ for request {b} head {h}: "
                                         f"{len(bad)} bytes, first at token/d {bad[0].tolist()} "
                                         f"oracle {r[tuple(bad[0])]} gpu {g[tuple(bad[0])]}")


def first_record_diff(table, g_table):
    for idx in np.ndindex(table.shape):
        if table[idx].tobytes() != g_table[idx].tobytes():
            return f"record {idx}: oracle {table[idx]} gpu {g_table[idx]}"
    return "records equal"


def assert_attn_close(ref, got):
    diff = np.abs(ref - got)
    assert np.isfinite(got).all()
    assert diff.max() <= ATTN_MAX_ABS, f"max |diff| {diff.max():.3e}"
    assert diff.mean() <= ATTN_MEAN_ABS, f"mean |diff| {diff.mean():.3e}"
    return diff.max(), diff.mean()
