"""The comparison encodings on the GPU -- fixed 64-value groups, symmetric INT8, FP8 E4M3 -- against
the oracle's comparison quantisers.  Bit-exact: every stored code, decoded by its format's
definition, equals the oracle's dequantised value, and slots past each request's end stay
untouched.  Attention: the decode kernel over each cache matches the oracle's fp64 attention over
the same dequantised values within the attention tolerance."""
import numpy as np
import pytest

import oracle
from dgq_cases import D, Case, assert_attn_close, bf16_to_f32

pytestmark = pytest.mark.gpu

FILL = 0xAB  # pool bytes before encoding: slots that must stay untouched keep it


def e4m3_values() -> np.ndarray:
    """fp64 value of every E4M3 byte from the format's definition: sign bit, 4 exponent bits
    (bias 7), 3 mantissa bits; exponent 0 is subnormal (m / 8 * 2^-6); 0x7F / 0xFF are NaN."""
    out = np.zeros(256)
    for byte in range(256):
        s, e, m = byte >> 7, (byte >> 3) & 15, byte & 7
        if e == 15 and m == 7:
            v = np.nan
        elif e == 0:
            v = m / 8 * 2.0 ** -6
        else:
            v = (1 + m / 8) * 2.0 ** (e - 7)
        out[byte] = -v if s else v
    return out


def gpu_encode(case: Case, fmt: str, fill=FILL, par_fill=-7.0):
    import torch
    import int8_group_quantized_gb300 as dgq
    dev = torch.device("cuda:0")
    d_k = torch.from_numpy(case.k.view(np.int16)).to(dev).view(torch.bfloat16)
    d_v = torch.from_numpy(case.v.view(np.int16)).to(dev).view(torch.bfloat16)
    if case.k.shape[0] == 0:
        d_k = d_v = torch.zeros((1, case.hkv, D), dtype=torch.bfloat16, device=dev)
    case.d_cu = torch.from_numpy(case.cu).to(dev)
    case.d_bt = torch.from_numpy(case.bt).to(dev)
    case.d_lens = torch.from_numpy(case.lens).to(dev)
    shape = (case.num_blocks, case.hkv, case.bs, D)
    case.d_kp = torch.full(shape, fill, dtype=torch.uint8, device=dev)
    case.d_vp = torch.full(shape, fill, dtype=torch.uint8, device=dev)
    case.d_kpar = case.d_vpar = None
    if fmt == "fixed64":
        case.d_kpar = torch.full((*shape[:3], 4), par_fill, dtype=torch.float32, device=dev)
        case.d_vpar = torch.full((*shape[:3], 4), par_fill, dtype=torch.float32, device=dev)
    case.d_table = torch.full((case.B, case.hkv, 128), 0x5A, dtype=torch.uint8, device=dev)
    ws = torch.zeros(dgq.dgq_encode_format_workspace_size(case.B, case.hkv), dtype=torch.uint8, device=dev)
    dgq.dgq_encode_format(fmt, d_k, d_v, case.d_cu, case.max_seqlen, case.bs, case.d_bt, case.d_kp, case.d_vp,
                          case.d_table, ws, case.d_kpar, case.d_vpar)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    from dgq_cases import table_to_numpy
    kpar = case.d_kpar.cpu().numpy() if case.d_kpar is not None else None
    vpar = case.d_vpar.cpu().numpy() if case.d_vpar is not None else None
    return case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(), table_to_numpy(case.d_table), kpar, vpar


def decode_stored(case: Case, fmt, pool, par, rec, b, h, is_v):
    """[L, 128] fp64 values of the GPU's stored codes of (b, h), by the format's definition."""
    L = int(case.lens[b])
    t = np.arange(L)
    blk, slot = case.bt[b, t // case.bs], t % case.bs
    codes = pool[blk, h, slot].astype(np.float64)
    if fmt == "fixed64":
        p = par[blk, h, slot].astype(np.float64)  # [L, 4]: min0, scale0, min1, scale1
        out = np.empty((L, D))
        out[:, :64] = p[:, 0:1] + codes[:, :64] * p[:, 1:2]
        out[:, 64:] = p[:, 2:3] + codes[:, 64:] * p[:, 3:4]
        return out
    if fmt == "sym_int8":
        s = np.float64(rec["v_scale" if is_v else "k_scale"][0])
        return (codes - 128.0) * s
    return e4m3_values()[pool[blk, h, slot]]


def check_encoding(case: Case, fmt: str):
    kp, vp, table, kpar, vpar = gpu_encode(case, fmt)
    written = np.zeros(kp.shape[:3], dtype=bool)
    for b in range(case.B):
        L = int(case.lens[b])
        for h in range(case.hkv):
            rec = table[b, h]
            assert rec["seq_len"] == L and rec["n_seg"] == (1 if L else 0), (b, h, rec)
            assert list(rec["start"]) == [0] + [L] * 4, rec
            assert rec["k_inv_last"] == 0 and rec["v_inv_last"] == 0 and not rec["pad"].any()
            if L == 0:
                continue
            rows = slice(int(case.cu[b]), int(case.cu[b + 1]))
            for is_v, x, pool, par in ((False, case.k, kp, kpar), (True, case.v, vp, vpar)):
                want = oracle.dequant_comparison(x[rows, h, :], fmt)
                got = decode_stored(case, fmt, pool, par, rec, b, h, is_v)
                bad = np.argwhere(~(got == want))
                assert len(bad) == 0, (f"{fmt} {'V' if is_v else 'K'} request {b} head {h}: {len(bad)} values "
                                       f"differ, first {bad[0].tolist()}: oracle {want[tuple(bad[0])]!r} "
                                       f"gpu {got[tuple(bad[0])]!r}")
                mn, sc = rec["v_min" if is_v else "k_min"][0], rec["v_scale" if is_v else "k_scale"][0]
                if fmt == "sym_int8":
                    assert mn == np.float32(-128.0) * sc and not (sc == 0 and np.signbit(mn))
                else:
                    assert (mn, sc) == (0.0, 1.0)
            t = np.arange(L)
            written[case.bt[b, t // case.bs], h, t % case.bs] = True
    assert (kp[~written] == FILL).all() and (vp[~written] == FILL).all()
    if kpar is not None:
        assert (kpar[~written] == -7.0).all() and (vpar[~written] == -7.0).all()


def gpu_attn_format(case: Case, fmt: str):
    import torch
    import int8_group_quantized_gb300 as dgq
    dev = torch.device("cuda:0")
    d_q = torch.from_numpy(case.q.view(np.int16)).to(dev).view(torch.bfloat16)
    d_kn = torch.from_numpy(case.knew.view(np.int16)).to(dev).view(torch.bfloat16)
    d_vn = torch.from_numpy(case.vnew.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.zeros((case.B, case.hq, D), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(dgq.dgq_attn_workspace_size(case.B, case.hq, case.hkv, case.max_seqlen), dtype=torch.uint8,
                     device=dev)
    dgq.dgq_paged_decode_attn_format(fmt, d_q, d_kn, d_vn, case.d_kp, case.d_vp, case.d_table, case.d_bt,
                                     case.d_lens, case.max_seqlen, out, ws, case.d_kpar, case.d_vpar)
    torch.cuda.synchronize()
    assert dgq.dgq_workspace_error(ws) == 0
    return bf16_to_f32(out.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def oracle_attn_format(case: Case, fmt: str):
    out = np.zeros((case.B, case.hq, D))
    for b in range(case.B):
        rows = slice(int(case.cu[b]), int(case.cu[b + 1]))
        L = int(case.lens[b])
        kd = np.zeros((L, case.hkv, D))
        vd = np.zeros((L, case.hkv, D))
        for h in range(case.hkv):
            kd[:, h] = oracle.dequant_comparison(case.k[rows, h, :], fmt)
            vd[:, h] = oracle.dequant_comparison(case.v[rows, h, :], fmt)
        out[b] = oracle.decode_attn_dense(case.q[b], case.knew[b], case.vnew[b], kd, vd)
    return out


CASES = {
    # ragged lengths over several 16-token tiles and one 256-token encoder slice, an empty and a
    # one-token request, shuffled blocks
    "mixed_bs16_gqa4": dict(lens=[37, 300, 0, 1, 16, 129], hq=8, hkv=2, bs=16, seed=101),
    "bs64_gqa8": dict(lens=[700, 65, 128], hq=16, hkv=2, bs=64, seed=102),
    "mha_bs32": dict(lens=[5, 250, 33], hq=4, hkv=4, bs=32, seed=103),
    # several encoder slices per pair and a split pair in the decode kernel
    "long_bs16": dict(lens=[3000], hq=8, hkv=1, bs=16, seed=104),
}


@pytest.mark.parametrize("fmt", ["fixed64", "sym_int8", "fp8_e4m3"])
@pytest.mark.parametrize("name", list(CASES))
def test_encoding_matches_oracle(fmt, name):
    check_encoding(Case(**CASES[name]), fmt)


@pytest.mark.parametrize("fmt", ["fixed64", "sym_int8", "fp8_e4m3"])
@pytest.mark.parametrize("name", list(CASES))
def test_decode_attention_matches_oracle(fmt, name):
    case = Case(**CASES[name])
    gpu_encode(case, fmt)
    assert_attn_close(oracle_attn_format(case, fmt), gpu_attn_format(case, fmt))


def test_fp8_saturation_and_subnormals():
    """Values past 448 saturate; values below half the smallest subnormal flush to +-0; the
    subnormal range keeps its 2^-9 step (inputs planted in a one-request cache)."""
    case = Case(lens=[32], hq=2, hkv=1, bs=16, seed=105)
    special = np.array([500.0, -1000.0, 448.0, 464.0, 2.0 ** -10, -(2.0 ** -11), 3 * 2.0 ** -10, 0.0,
                        -0.0, 2.0 ** -7, 1.0625, 1.1875, 240.0, -240.0, 2.0 ** -9, 0.1], dtype=np.float32)
    bits = special.view(np.uint32).astype(np.uint64)
    bits = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    case.k[0, 0, :16] = bits
    case.v[3, 0, 100:116] = bits
    check_encoding(case, "fp8_e4m3")


@pytest.mark.parametrize("fmt", ["fixed64", "fp8_e4m3", "sym_int8"])
@pytest.mark.parametrize("fill", [0x7F, 0xFF])
def test_decode_ignores_whatever_lies_past_the_end(fmt, fill):
    """Slots past each request's end are never written and may hold any bytes: E4M3 NaN patterns
    (0x7F, 0xFF) in the codes and NaN in the fixed groups' parameters must not reach the output
    (their softmax weight is 0, and 0 * NaN is NaN).  Ragged lengths leave partial tiles; G = 1 and
    G = 4."""
    for kw in (dict(lens=[37, 300, 1, 129, 250], hq=4, hkv=4, bs=16, seed=106),
               dict(lens=[700, 65, 17, 3], hq=16, hkv=4, bs=64, seed=107)):
        case = Case(**kw)
        gpu_encode(case, fmt, fill=fill, par_fill=float("nan"))
        got = gpu_attn_format(case, fmt)
        assert np.isfinite(got).all()
        assert_attn_close(oracle_attn_format(case, fmt), got)
