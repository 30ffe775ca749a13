"""The no-allocation decode attention (dgq_paged_decode_attn_noalloc), for callers that may not
allocate device memory while they run and so cannot pass a workspace: its output through the
C ABI must match the regular entry point's, call after call, on the library's fixed scratch.

This file is collected last on purpose (its name sorts after every other test file), so a
run that stops at its first failure has run every other test before it.  It also passes on
its own in a fresh process: nothing here depends on state left by other tests."""
import numpy as np
import pytest

from dgq_cases import Case, assert_attn_close, bf16_to_f32

pytestmark = pytest.mark.gpu


def _noalloc_out(case, dgq, torch):
    out = torch.full_like(case.d_out, float("nan"))
    dgq.dgq_paged_decode_attn_noalloc(case.d_q, case.d_knew, case.d_vnew, case.d_kp, case.d_vp, case.d_table,
                                      case.d_bt, case.d_lens, case.max_seqlen, out)
    torch.cuda.synchronize()
    return bf16_to_f32(out.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


@pytest.mark.parametrize("lens,hq,hkv,bs,seed", [
    ([37, 300], 4, 2, 16, 0),                       # tiny, ragged, two KV heads
    ([1000, 17, 0, 2500, 640], 32, 8, 64, 5),       # GQA 4, an empty request, several CTAs per pair
])
def test_noalloc_matches_workspace_entry_point_twice(lens, hq, hkv, bs, seed):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import int8_group_quantized_gb300 as dgq
    case = Case(lens, hq=hq, hkv=hkv, bs=bs, seed=seed)
    case.gpu_compress()
    ref = case.gpu_attn()  # regular entry point, caller-owned workspace
    first = _noalloc_out(case, dgq, torch)
    second = _noalloc_out(case, dgq, torch)  # the scratch keeps the first call's contents
    assert_attn_close(ref, first)
    assert_attn_close(ref, second)


def test_noalloc_second_problem_after_first():
    """Two different problems back to back on the shared scratch: each matches its own
    regular-entry-point result."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import int8_group_quantized_gb300 as dgq
    for lens, hq, hkv, bs, seed in (([900, 33], 8, 1, 32, 7), ([64, 128, 4096], 16, 4, 16, 8)):
        case = Case(lens, hq=hq, hkv=hkv, bs=bs, seed=seed)
        case.gpu_compress()
        assert_attn_close(case.gpu_attn(), _noalloc_out(case, dgq, torch))


def test_noalloc_rejects_problem_beyond_scratch_limit():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import int8_group_quantized_gb300 as dgq
    L = dgq.lib()
    limit = 8 << 20
    # a batch whose workspace exceeds the fixed array; no pointer is touched before the check
    batch, hq, hkv = 4096, 64, 8
    assert dgq.dgq_attn_workspace_size(batch, hq, hkv, 1024) > limit
    fake = 0x10000
    st = L.dgq_paged_decode_attn_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, 1024, batch, hq, hkv,
                                         128, 16, 64, 1 << 16, fake, None)
    assert st == -7
    assert b"scratch" in L.dgq_status_str(st)
