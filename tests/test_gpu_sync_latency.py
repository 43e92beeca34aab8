"""lf_sync_latency: the one-hop flag and grid-barrier microbenchmark runs,
finishes inside its bounded waits, and reports plausible times."""
import math

import pytest

from conftest import cuda_available

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    return pm


@pytest.mark.parametrize("n_ctas", [2, 37, 148])
def test_flag_hop_and_grid_barrier(pm, n_ctas):
    import torch
    n_ctas = min(n_ctas, torch.cuda.get_device_properties(0).multi_processor_count)
    hop = pm.sync_latency_ns(0, n_ctas, 50)
    bar = pm.sync_latency_ns(1, n_ctas, 50)
    for v in (hop, bar):
        assert math.isfinite(v) and 10.0 < v < 1e6
