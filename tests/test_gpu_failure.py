"""Device-side failure detection without a GPU fault: one tile is made to skip
publishing its look-back status, the waiting tiles give up after a short
bounded wait, the error is recorded in the work buffer and read back on the
host, and the CUDA context stays usable for the next call."""
import numpy as np
import pytest

import oracle
from sorting_lsd_radix_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sorting_lsd_radix_gb300 import build as gbuild
    gbuild.build()
    from sorting_lsd_radix_gb300 import gbsort
    gbsort.load()
    yield gbsort
    gbsort.gbs_debug_set_lookback_fault(-1, 0, 0)


def test_lookback_timeout_is_reported_and_context_survives(g):
    tile = g.gbs_debug_radix_tile_keys(4)
    n = 6 * tile + 5
    keys = wl.uniform_u32(n, wl.seed_for(60))
    t = torch.from_numpy(keys).cuda()
    g.gbs_debug_set_lookback_fault(1, 2, 1 << 12)  # pass 1, tile 2 never publishes
    try:
        out, temp = g.gbs_sort_keys(t, begin_bit=0, end_bit=24, return_temp=True)
        assert g.gbs_get_status(temp) == g.GBS_ERR_TIMEOUT
    finally:
        g.gbs_debug_set_lookback_fault(-1, 0, 0)
    out2 = g.gbs_sort_keys(t, begin_bit=0, end_bit=24, temp=temp)
    assert g.gbs_get_status(temp) == g.GBS_OK
    assert np.array_equal(out2.cpu().numpy(), oracle.sort_keys(keys, 0, 24))


def test_invalid_arguments_launch_nothing(g):
    t = torch.zeros(100, dtype=torch.uint32, device="cuda")
    with pytest.raises(g.GbsError) as e:
        g.gbs_sort_keys(t, begin_bit=4, end_bit=2)
    assert e.value.status == g.GBS_ERR_INVALID_ARG
    with pytest.raises(g.GbsError) as e:
        g.gbs_sort_pairs(t, torch.zeros(100, dtype=torch.uint32, device="cuda"), begin_bit=0, end_bit=33)
    assert e.value.status == g.GBS_ERR_INVALID_ARG
    assert g.gbs_debug_last_launch_count() == 0
