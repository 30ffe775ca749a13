"""The library's calls inside CUDA graphs: decode (both merges of split pairs), the decode-step
append and compress (cluster path and grid-wide cooperative path) captured with
torch.cuda.graph and replayed give exactly the bytes the same calls give launched directly.
The calls keep no host-side state between launches and leave their workspaces ready for the
next call, so a replay is a call."""
import numpy as np
import pytest

from dgq_cases import Case
from test_gpu_append import grow_tables, step_tokens

pytestmark = pytest.mark.gpu


def _capture(fn):
    """fn() run once on a side stream (first-call setup outside the capture), then captured."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("lens", [[200] * 128, [3000] * 8])  # warp merge / block merge
def test_decode_graph_replays_equal_calls(lens):
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case(lens, hq=8, hkv=2, bs=16, seed=70 + len(lens))
    case.gpu_compress()
    case.gpu_attn()
    eager = case.d_out.clone()
    out = torch.zeros_like(case.d_out)
    ws = torch.zeros_like(case.d_aws)
    g = _capture(lambda: dgq.dgq_paged_decode_attn(case.d_q, case.d_knew, case.d_vnew, case.d_kp, case.d_vp,
                                                   case.d_table, case.d_bt, case.d_lens, case.max_seqlen, out, ws))
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert dgq.dgq_workspace_error(ws) == 0
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("lens", [[37, 300, 1000, 4000], [5000, 300, 9000]])  # cluster / grid-wide
def test_compress_graph_replays_equal_calls(lens):
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case(lens, hq=8, hkv=2, bs=16, seed=80 + len(lens))
    case.gpu_compress()
    ref = (case.d_kp.clone(), case.d_vp.clone(), case.d_table.clone())
    kp, vp, tab = torch.zeros_like(case.d_kp), torch.zeros_like(case.d_vp), torch.zeros_like(case.d_table)
    ws = torch.zeros_like(case.d_cws)
    g = _capture(lambda: dgq.dgq_compress(case.d_k, case.d_v, case.d_cu, case.max_seqlen, case.bs, case.d_bt, kp, vp,
                                          tab, ws))
    for _ in range(3):
        for t in (kp, vp, tab):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert dgq.dgq_workspace_error(ws) == 0
        assert torch.equal(kp, ref[0]) and torch.equal(vp, ref[1]) and torch.equal(tab, ref[2])


def test_append_graph_replays_equal_calls():
    # one captured append replayed twice equals two appends of the same token called directly
    import torch
    import int8_group_quantized_gb300 as dgq
    case = Case([40, 300, 1023], hq=8, hkv=2, bs=16, seed=88)
    grow_tables(case, 2)
    case.gpu_compress()
    dev = case.d_kp.device
    k, v = step_tokens(88, 0, case.B, case.hkv)
    d_k = torch.from_numpy(k.view(np.int16)).to(dev).view(torch.bfloat16)
    d_v = torch.from_numpy(v.view(np.int16)).to(dev).view(torch.bfloat16)
    state = lambda: (case.d_kp.clone(), case.d_vp.clone(), case.d_table.clone())
    start = state()
    ws = torch.zeros(dgq.dgq_append_workspace_size(), dtype=torch.uint8, device=dev)
    want = []
    for _ in range(2):
        dgq.dgq_append(d_k, d_v, case.bs, case.d_bt, case.d_kp, case.d_vp, case.d_table, ws)
        torch.cuda.synchronize()
        want.append(state())
    kp, vp, tab = (t.clone() for t in start)
    g = _capture(lambda: dgq.dgq_append(d_k, d_v, case.bs, case.d_bt, kp, vp, tab, ws))
    for t, s in zip((kp, vp, tab), start):  # the side-stream setup call appended once: start over
        t.copy_(s)
    for w in want:
        g.replay()
        torch.cuda.synchronize()
        assert dgq.dgq_workspace_error(ws) == 0
        assert torch.equal(kp, w[0]) and torch.equal(vp, w[1]) and torch.equal(tab, w[2])
