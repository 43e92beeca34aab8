"""The Python binding's argument checks that need no GPU (CPU only): host
tensors are refused before any call reaches the library, and the
per-layer window list is checked and marshalled."""
import pytest

from synthetic import MODELS, make_weights


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    return pm


def test_host_tensors_are_refused(pm):
    cfg = MODELS["tiny"]
    with pytest.raises(ValueError, match="contiguous CUDA"):
        pm.Decoder(cfg, make_weights(cfg, 0), 64)


def test_layer_window_needs_one_entry_per_layer(pm):
    cfg = MODELS["tiny"]
    with pytest.raises(ValueError):
        pm._windows(cfg, [16])
    assert list(pm._windows(cfg, [16, 0])) == [16, 0]
    assert pm._windows(cfg, None) is None
