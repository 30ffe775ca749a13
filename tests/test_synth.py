"""The seeded input generator: determinism, distribution and span rules.  CPU only."""
import numpy as np

import synth
from synth import configs


def test_normal_stream_moments_and_determinism():
    k = synth.key(7, synth.STREAM_K, 0, 0, 0)
    x = np.array([synth.host().synth_normal_c(k, i) for i in range(100000)])
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02
    assert synth.host().synth_normal_c(k, 123) == synth.host().synth_normal_c(k, 123)


def test_bf16_round_to_nearest_even():
    f = synth.host().synth_bf16_c
    assert f(1.0) == 0x3F80
    assert f(1.0 + 2.0 ** -8) == 0x3F80        # tie -> even (mantissa ...0)
    assert f(1.0 + 3 * 2.0 ** -8) == 0x3F82    # tie -> even (mantissa ...10)
    assert f(-2.5) == 0xC020


def test_span_rules():
    for rule, counts in ((synth.RULE_SET3, {3}), (synth.RULE_U, {3, 4, 5}), (synth.RULE_PERM5, {5})):
        for h in range(40):
            n, st, sg = synth.spans(3, 1, 2, h, 1000, rule)
            assert n in counts and st[0] == 0 and np.all(np.diff(st[:n]) >= 0) and st[n - 1] < 1000
            if rule == synth.RULE_SET3:
                assert set(sg[:n].tolist()) <= {float(np.float32(x)) for x in (0.03, 0.15, 0.47)}
            elif rule == synth.RULE_U:
                assert np.all((sg[:n] >= 0.03) & (sg[:n] <= 0.5))
            else:
                assert sorted(sg[:n].tolist()) == [float(np.float32(x)) for x in (0.03, 0.08, 0.15, 0.3, 0.47)]


def test_fill_layer_matches_fill_pair():
    lens = np.array([5, 40], dtype=np.int32)
    cu = configs.cu_seqlens(lens)
    tabs = synth.span_tables(1, 2, lens, 3, synth.RULE_U)
    lay = synth.fill_layer(1, synth.STREAM_V, 2, cu, 3, tabs)
    for b in range(2):
        for h in range(3):
            i = b * 3 + h
            pair = synth.fill_pair(1, synth.STREAM_V, 2, b, h, int(lens[b]), tabs[0][i],
                                   tabs[1][5 * i:5 * i + 5], tabs[2][5 * i:5 * i + 5])
            assert np.array_equal(lay[cu[b]:cu[b + 1], h], pair)


def test_workload_metadata():
    w = configs.WORKLOADS[1]
    lens = configs.seq_lens(w)
    bt, nb = configs.block_tables(w, lens)
    assert list(lens) == [37, 300] and nb == 32
    used = np.concatenate([bt[0, :3], bt[1, :19]])
    assert len(set(used.tolist())) == 22 and used.max() < 32
    w3 = configs.WORKLOADS[3]
    l3 = configs.seq_lens(w3)
    assert l3.min() >= 256 and l3.max() <= 2048
    bt3, nb3 = configs.block_tables(w3, l3)
    assert nb3 == int(sum((l3 + 15) // 16))
    w5 = configs.WORKLOADS[5]
    l5 = configs.seq_lens(w5)
    assert l5.min() >= 128 and l5.max() <= 32768
