"""Finite bf16 inputs whose fp32 variance overflows: windows of values near +-2^63 have an
infinite mean variance, two such windows side by side have no defined jump (inf - inf), and
such a pair of windows is no boundary candidate (the DGQ article's boundaries sit at the largest
variance jumps, section 2.2; the undefined jump is read as no jump at all).  Records and codes of
every compression path -- the cluster kernel, the grid-wide kernel (short and long pairs) and the
two-phase finish -- must equal the oracle's byte for byte on such inputs."""
import numpy as np
import pytest

from dgq_cases import Case, assert_compress_equal, table_to_numpy
from test_gpu_compress import PATH_CLUSTER, PATH_GRID, compress_path
from test_gpu_prefill import run_chunked, schedule_uniform

pytestmark = pytest.mark.gpu

BIG = (0x5F00, 0xDF00, 0x5F40, 0xDF40)  # bf16 bits of +-2^63 and +-1.5 * 2^63


def plant(case, rng, runs):
    """runs: (request, head, first window, windows) -> huge values in K and V there."""
    for b, h, w0, n in runs:
        L = int(case.lens[b])
        t0, t1 = case.cu[b] + 16 * w0, case.cu[b] + min(L, 16 * (w0 + n))
        for arr in (case.k, case.v):
            arr[t0:t1, h] = rng.choice(np.array(BIG, dtype=np.uint16), size=(t1 - t0, 128))


def overflow_case(lens, hkv, bs, seed, runs):
    case = Case(lens, hq=hkv, hkv=hkv, bs=bs, seed=seed)
    plant(case, np.random.default_rng(seed), runs)
    return case


def check_one_shot(case, expect_path):
    kp, vp, table = case.oracle_compress()
    case.gpu_compress()
    assert compress_path(case) == expect_path
    assert_compress_equal(case, kp, vp, table, case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(),
                          table_to_numpy(case.d_table))
    return table


RUNS_SHORT = [(0, 0, 0, 2),      # overflowed first two windows: the cut goes after them
              (0, 1, 5, 3),      # a run in the middle: two infinite jumps, one undefined
              (1, 0, 0, 256),    # every window overflowed: no candidate, one segment
              (2, 1, 100, 50), (2, 0, 10, 1)]
RUNS_LONG = RUNS_SHORT[:2] + [(1, 0, 0, 1250), (1, 1, 300, 40), (1, 1, 900, 2), (2, 0, 0, 4)]


def test_overflow_cluster_path():
    case = overflow_case([300, 4096, 2500], hkv=2, bs=16, seed=41, runs=RUNS_SHORT)
    table = check_one_shot(case, PATH_CLUSTER)
    assert table[0, 0]["n_seg"] == 2 and table[0, 0]["start"][1] == 32
    assert table[1, 0]["n_seg"] == 1


def test_overflow_grid_path_short_and_long_pairs():
    # the 20000-token request (1250 windows) takes the long-pair segmentation of the grid kernel
    case = overflow_case([300, 20000, 4000], hkv=2, bs=64, seed=42, runs=RUNS_LONG)
    table = check_one_shot(case, PATH_GRID)
    assert table[1, 0]["n_seg"] == 1


@pytest.mark.parametrize("lens,runs", [([300, 4096, 2500], RUNS_SHORT), ([300, 20000, 4000], RUNS_LONG)])
def test_overflow_two_phase_finish(lens, runs):
    case = overflow_case(lens, hkv=2, bs=16, seed=43, runs=runs)
    kp, vp, table = case.oracle_compress()
    g_kp, g_vp, g_table = run_chunked(case, schedule_uniform(case.lens, 1024), src_seed=43)
    assert_compress_equal(case, kp, vp, table, g_kp, g_vp, g_table)
