"""The no-allocation decode attention (dgq_paged_decode_attn_noalloc), for callers that may not
allocate device memory while they run and so cannot pass a workspace: it runs the regular entry
point's kernels with the same launch shapes on the library's fixed scratch, so its output through
the C ABI must equal the regular entry point's bit for bit, call after call (a stale-scratch bug
that perturbs a few heads cannot hide under a tolerance), and lie within the attention tolerance
of the oracle's fp64 attention over the same cache.

This file is collected last on purpose (its name sorts after every other test file), so a
run that stops at its first failure has run every other test before it.  It also passes on
its own in a fresh process: nothing here depends on state left by other tests."""
import numpy as np
import pytest

from dgq_cases import Case, assert_attn_close, assert_compress_equal, bf16_to_f32, table_to_numpy

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
    kp, vp, table = case.oracle_compress()
    case.gpu_compress()
    assert_compress_equal(case, kp, vp, table, case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(),
                          table_to_numpy(case.d_table))
    ref = case.gpu_attn()  # regular entry point, caller-owned workspace
    first = _noalloc_out(case, dgq, torch)
    second = _noalloc_out(case, dgq, torch)  # the scratch keeps the first call's contents
    assert np.array_equal(first, ref), "no-allocation output differs from the regular entry point's"
    assert np.array_equal(second, ref), "second no-allocation call differs from the regular entry point's"
    assert_attn_close(case.oracle_attn(kp, vp, table), first)


def test_noalloc_second_problem_after_first():
    """Two different problems back to back on the shared scratch: each matches its own
    regular-entry-point result."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import int8_group_quantized_gb300 as dgq
    for lens, hq, hkv, bs, seed in (([900, 33], 8, 1, 32, 7), ([64, 128, 4096], 16, 4, 16, 8)):
        case = Case(lens, hq=hq, hkv=hkv, bs=bs, seed=seed)
        kp, vp, table = case.oracle_compress()
        case.gpu_compress()
        ref = case.gpu_attn()  # regular entry point (also allocates the output buffer)
        got = _noalloc_out(case, dgq, torch)
        assert np.array_equal(got, ref)
        assert_attn_close(case.oracle_attn(kp, vp, table), got)


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
