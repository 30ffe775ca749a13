"""dgq_compress_ex on the GPU against the oracle: the segment cap and the variance floor give
the same records and codes bit for bit, on both compress kernels (requests up to 4096 tokens
and longer ones)."""
import numpy as np
import pytest

from dgq_cases import Case, assert_compress_equal, table_to_numpy

pytestmark = pytest.mark.gpu


def run(case, max_groups, min_var):
    kp, vp, table = case.oracle_compress(max_groups=max_groups, min_var=min_var)
    case.gpu_compress(max_groups=max_groups, min_var=min_var)
    assert_compress_equal(case, kp, vp, table, case.d_kp.cpu().numpy(), case.d_vp.cpu().numpy(),
                          table_to_numpy(case.d_table))
    return table


@pytest.mark.parametrize("max_groups", [1, 2, 3, 5])
def test_cap_cluster_path(max_groups):
    case = Case([37, 300, 2048, 4096, 1, 0, 1500], hq=8, hkv=2, bs=16, seed=40 + max_groups)
    table = run(case, max_groups, 0.0)
    assert table["n_seg"].max() <= max_groups


@pytest.mark.parametrize("min_var", [0.05, 0.3, 1e9])
def test_floor_cluster_path(min_var):
    case = Case([300, 2048, 4096, 17, 3333], hq=4, hkv=4, bs=32, seed=50)
    table = run(case, 5, min_var)
    if min_var >= 1e9:
        assert np.all(table["n_seg"][table["seq_len"] > 0] == 1)


@pytest.mark.parametrize("max_groups,min_var", [(3, 0.0), (5, 0.05), (2, 0.3), (5, 1e9)])
def test_settings_grid_path(max_groups, min_var):
    case = Case([5000, 20000, 37, 16384], hq=8, hkv=2, bs=64, seed=60)
    table = run(case, max_groups, min_var)
    assert table["n_seg"].max() <= max_groups
