"""The threaded host driver of the whole-workload parity tests gives exactly what the plain,
batched oracle and generator give (it only calls them per request, in parallel).  CPU only."""
import numpy as np

import oracle
import synth
from synth import configs
from parity_full import draw_layer, oracle_layer


def test_threaded_driver_equals_batched_oracle():
    for wid, layer in ((1, 0), (3, 5)):
        w = configs.WORKLOADS[wid]
        hl = draw_layer(w, layer)
        if wid == 3:  # a sub-batch of the MHA workload keeps this quick
            keep = 6
            w = configs.Workload(w.name, w.seed, w.layers, keep, w.hq, w.hkv, w.block_size, w.rule, w.lens,
                                 w.placement)
            T = int(hl.cu[keep])
            hl.lens, hl.cu, hl.bt = hl.lens[:keep], hl.cu[:keep + 1], hl.bt[:keep]
            hl.k, hl.v = hl.k[:T], hl.v[:T]
            hl.q, hl.knew, hl.vnew = hl.q[:keep], hl.knew[:keep], hl.vnew[:keep]
        tabs = synth.span_tables(w.seed, layer, hl.lens, w.hkv, w.rule)
        assert np.array_equal(synth.fill_layer(w.seed, synth.STREAM_K, layer, hl.cu, w.hkv, tabs), hl.k)
        assert np.array_equal(synth.fill_layer(w.seed, synth.STREAM_V, layer, hl.cu, w.hkv, tabs), hl.v)
        oracle_layer(w, hl)
        kp, vp, tab = oracle.compress(hl.k, hl.v, hl.cu, w.hkv, w.block_size, hl.bt, hl.num_blocks)
        assert np.array_equal(kp, hl.kp) and np.array_equal(vp, hl.vp)
        assert tab.tobytes() == hl.table.tobytes()
        out = oracle.paged_decode_attn(hl.q, hl.knew, hl.vnew, kp, vp, tab, hl.bt, hl.lens)
        assert np.array_equal(out, hl.out)
