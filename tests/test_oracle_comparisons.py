"""Pins for the oracle's comparison quantisers (fidelity context): fixed 64-dim-group INT8,
symmetric per-tensor INT8 and FP8 E4M3, each against values its format represents exactly, its
error bound, and the format's rounding rules; and the dense attention against the paged one.
CPU only."""
import numpy as np

import oracle

D = 128


def bf16_bits(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


def f(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def test_fixed64_two_valued_groups_round_trip_and_error_bound():
    rng = np.random.default_rng(1)
    # groups whose range is 255 * 2^-k (scale exactly 2^-k): both values decode exactly
    x = np.where(rng.random((10, D)) < 0.5, -2.0, -2.0 + 255 / 128).astype(np.float32)
    x[:, :64] = np.where(rng.random((10, 64)) < 0.5, 0.0, 255 / 64)
    x[:, 0], x[:, 1], x[:, 64], x[:, 65] = 0.0, 255 / 64, -2.0, -2.0 + 255 / 128
    assert np.array_equal(oracle.dequant_comparison(bf16_bits(x), "fixed64"), x.astype(np.float64))
    g = bf16_bits(rng.standard_normal((50, D)).astype(np.float32))
    got = oracle.dequant_comparison(g, "fixed64")
    xv = f(g)
    for half in (slice(0, 64), slice(64, 128)):
        blk = xv[:, half]
        scale = (blk.max(1) - blk.min(1)) / 255
        assert np.all(np.abs(got[:, half] - blk).max(1) <= 0.5 * scale * (1 + 2**-10) + 1e-6)


def test_symmetric_int8_grid_round_trips():
    # max |x| = 127 / 128 -> scale = 1/128 exactly; every k / 128 round-trips
    rng = np.random.default_rng(2)
    k = rng.integers(-127, 128, (20, D)).astype(np.float32)
    k[0, 0] = 127
    x = k / 128
    assert np.array_equal(oracle.dequant_comparison(bf16_bits(x), "sym_int8"), x.astype(np.float64))
    g = bf16_bits(rng.standard_normal((30, D)).astype(np.float32))
    got = oracle.dequant_comparison(g, "sym_int8")
    scale = np.float32(np.abs(f(g)).max().astype(np.float32) / np.float32(127))
    assert np.abs(got - f(g)).max() <= 0.5 * scale * (1 + 2**-10)


def test_fp8_e4m3_rounding():
    # E4M3 numbers round-trip; midpoints go to the even mantissa; 448 caps; 2^-9 is the step
    exact = np.array([0.0, 1.0, 1.125, -0.75, 448.0, -448.0, 2.0**-9, 3 * 2.0**-9, 240.0, 0.1015625])
    assert np.array_equal(oracle.dequant_comparison(bf16_bits(np.resize(exact, D))[None], "fp8_e4m3")[0],
                          np.resize(exact, D))
    cases = {1.0625: 1.0,        # halfway 1.0 / 1.125 -> even mantissa 1.0
             1.1875: 1.25,       # halfway 1.125 / 1.25 -> 1.25 (mantissa 010)
             500.0: 448.0,       # saturates
             -1000.0: -448.0,
             2.0**-10: 0.0,      # halfway 0 / 2^-9 -> 0
             3 * 2.0**-10: 2.0**-8}  # halfway 2^-9 / 2^-8 -> 2^-8 (even)
    xs = np.resize(np.array(list(cases), dtype=np.float32), D)
    want = np.resize(np.array(list(cases.values())), D)
    assert np.array_equal(oracle.dequant_comparison(bf16_bits(xs)[None], "fp8_e4m3")[0], want)


def test_dense_attention_equals_paged_attention_on_the_same_values():
    rng = np.random.default_rng(3)
    L, Hq, Hkv, bs = 40, 4, 2, 16
    k = bf16_bits(rng.standard_normal((L, Hkv, D)).astype(np.float32) * 0.3)
    v = bf16_bits(rng.standard_normal((L, Hkv, D)).astype(np.float32))
    cu = np.array([0, L], dtype=np.int32)
    bt = np.array([[1, 2, 0]], dtype=np.int32)
    kp, vp, table = oracle.compress(k, v, cu, Hkv, bs, bt, 3)
    q = bf16_bits(rng.standard_normal((1, Hq, D)).astype(np.float32))
    kn = bf16_bits(rng.standard_normal((1, Hkv, D)).astype(np.float32))
    lens = np.array([L], dtype=np.int32)
    paged = oracle.paged_decode_attn(q, kn, kn, kp, vp, table, bt, lens)[0]
    kd = np.stack([oracle.dequant_pair(kp, table, bt, 0, h, L, False) for h in range(Hkv)], axis=1)
    vd = np.stack([oracle.dequant_pair(vp, table, bt, 0, h, L, True) for h in range(Hkv)], axis=1)
    dense = oracle.decode_attn_dense(q[0], kn[0], kn[0], kd, vd)
    assert np.allclose(dense, paged, rtol=1e-12, atol=1e-12)
