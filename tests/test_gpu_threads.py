"""Calls from several host threads at once: each thread compresses and decodes its own batch on
its own stream and workspaces through the C ABI (the binding releases the interpreter lock during
the calls), and every result equals the oracle's -- codes and records bit-exact, attention within
the tolerance.  The library keeps no state shared between host threads."""
import threading

import numpy as np
import pytest

from dgq_cases import Case, assert_attn_close, assert_compress_equal, bf16_to_f32, table_to_numpy

pytestmark = pytest.mark.gpu


def _run(case, errors, idx):
    import torch
    import int8_group_quantized_gb300 as dgq
    try:
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            k = torch.from_numpy(case.k.view(np.int16)).to(dev).view(torch.bfloat16)
            v = torch.from_numpy(case.v.view(np.int16)).to(dev).view(torch.bfloat16)
            cu, bt, lens = (torch.from_numpy(x).to(dev) for x in (case.cu, case.bt, case.lens))
            q, kn, vn = (torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
                         for x in (case.q, case.knew, case.vnew))
            shape = (case.num_blocks, case.hkv, case.bs, 128)
            kp = torch.zeros(shape, dtype=torch.uint8, device=dev)
            vp = torch.zeros_like(kp)
            table = torch.zeros((case.B, case.hkv, 128), dtype=torch.uint8, device=dev)
            out = torch.zeros((case.B, case.hq, 128), dtype=torch.bfloat16, device=dev)
            cws = torch.zeros(dgq.dgq_compress_workspace_size(case.B, case.max_seqlen, case.hkv), dtype=torch.uint8,
                              device=dev)
            aws = torch.zeros(dgq.dgq_attn_workspace_size(case.B, case.hq, case.hkv, case.max_seqlen),
                              dtype=torch.uint8, device=dev)
            for _ in range(5):  # several calls, interleaved with the other threads'
                dgq.dgq_compress(k, v, cu, case.max_seqlen, case.bs, bt, kp, vp, table, cws, stream)
                dgq.dgq_paged_decode_attn(q, kn, vn, kp, vp, table, bt, lens, case.max_seqlen, out, aws, stream)
            stream.synchronize()
            assert dgq.dgq_workspace_error(cws, stream) == 0 and dgq.dgq_workspace_error(aws, stream) == 0
            errors[idx] = (kp.cpu().numpy(), vp.cpu().numpy(), table_to_numpy(table),
                           bf16_to_f32(out.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64))
    except BaseException as e:  # reported by the main thread
        errors[idx] = e


def test_concurrent_host_threads():
    cases = [Case([300, 2048, 37], hq=8, hkv=2, bs=16, seed=71),       # cluster compress, 4-CTA clusters
             Case([5000, 100], hq=4, hkv=4, bs=64, seed=72),           # grid-wide compress
             Case([700] * 130, hq=16, hkv=8, bs=16, seed=73),          # 2-CTA clusters, warp merge
             Case([1, 64, 129], hq=4, hkv=1, bs=32, seed=74)]
    res = [None] * len(cases)
    threads = [threading.Thread(target=_run, args=(c, res, i)) for i, c in enumerate(cases)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for case, r in zip(cases, res):
        if isinstance(r, BaseException):
            raise r
        kp, vp, table = case.oracle_compress()
        assert_compress_equal(case, kp, vp, table, r[0], r[1], r[2])
        assert_attn_close(case.oracle_attn(kp, vp, table), r[3])
