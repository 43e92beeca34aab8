"""The C-ABI library loads and exports every symbol include/lf.h declares;
host-side argument checks (no GPU needed, no compute call)."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "lf.h")


def _declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"LF_API\s+[\w\s\*]*?\b(lf_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    return pm


def test_header_declares_the_public_entry_points():
    syms = _declared_symbols()
    for name in ("lf_create", "lf_prefill", "lf_decode", "lf_destroy", "lf_sync", "lf_reset"):
        assert name in syms


def test_library_exports_every_declared_symbol(pm):
    L = pm.lib()
    for name in _declared_symbols():
        assert hasattr(L, name), name
    assert set(pm.EXPORTS) == set(_declared_symbols())


def test_abi_version_and_error_strings(pm):
    assert pm.lib().lf_abi_version() == 6
    for code, name in pm.STATUS_NAMES.items():
        assert pm.error_string(code).startswith(name)


def test_create_rejects_bad_arguments_before_touching_the_gpu(pm):
    L = pm.lib()
    h = C.c_void_p()
    w = pm.lf_weights(*([0x1000] * 12))
    assert L.lf_create(None, C.byref(w), C.byref(h)) == 1
    good = dict(n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=1024, vocab=4096,
                max_seq=64, rope_theta=10000.0, rms_eps=1e-5, wait_timeout_ns=0, n_ctas=0, fault_step=-1)
    cases = [(dict(head_dim=96), 7), (dict(n_kv_heads=3), 7), (dict(d_model=300), 7), (dict(ffn_dim=1000), 7),
             (dict(n_layers=0), 1), (dict(max_seq=0), 1), (dict(n_heads=64, n_kv_heads=4), 7)]
    for change, expect in cases:
        cfg = pm.lf_config(**{**good, **change})
        assert L.lf_create(C.byref(cfg), C.byref(w), C.byref(h)) == expect, change
    wnull = pm.lf_weights(*([0x1000] * 11 + [0]))
    cfg = pm.lf_config(**good)
    assert L.lf_create(C.byref(cfg), C.byref(wnull), C.byref(h)) == 1
    # bulk copies read the weights: every pointer must be 16-byte aligned
    wodd = pm.lf_weights(*([0x1000] * 3 + [0x1008] + [0x1000] * 8))
    assert L.lf_create(C.byref(cfg), C.byref(wodd), C.byref(h)) == 1
    # more than 64 column groups of 256 in one vector
    cfg = pm.lf_config(**{**good, "ffn_dim": 256 * 65})
    assert L.lf_create(C.byref(cfg), C.byref(w), C.byref(h)) == 7
    # a negative sliding window
    win = (C.c_int32 * 2)(16, -1)
    cfg = pm.lf_config(**{**good, "layer_window": win})
    assert L.lf_create(C.byref(cfg), C.byref(w), C.byref(h)) == 1
    # weight formats: unknown -> NOT_SUPPORTED; FP8 needs every scale array, FP16 takes none
    cfg = pm.lf_config(**{**good, "weight_format": 7})
    assert L.lf_create(C.byref(cfg), C.byref(w), C.byref(h)) == 7
    cfg = pm.lf_config(**{**good, "weight_format": pm.WEIGHTS_FP8_E4M3})
    assert L.lf_create(C.byref(cfg), C.byref(w), C.byref(h)) == 1
    w8 = pm.lf_weights(*([0x1000] * 12 + [0x2000] * 7 + [0]))
    assert L.lf_create(C.byref(cfg), C.byref(w8), C.byref(h)) == 1
    cfg = pm.lf_config(**good)
    assert L.lf_create(C.byref(cfg), C.byref(w8), C.byref(h)) == 1
    # a prefill block below LF_PREFILL_AUTO (-1)
    cfg = pm.lf_config(**{**good, "prefill_block": -2})
    assert L.lf_create(C.byref(cfg), C.byref(w), C.byref(h)) == 1
    # MXFP4: every block-scale pointer is needed (any byte address); no batched prefill
    cfg = pm.lf_config(**{**good, "weight_format": pm.WEIGHTS_MXFP4})
    assert L.lf_create(C.byref(cfg), C.byref(w), C.byref(h)) == 1
    w4 = pm.lf_weights(*([0x1000] * 12 + [0x2001] * 7 + [0]))
    assert L.lf_create(C.byref(cfg), C.byref(w4), C.byref(h)) == 1
    # mixture of experts: limits on the expert counts, FP16 only, the router pointer required
    for change, expect in [(dict(n_experts=-1), 1), (dict(n_experts=65, top_k_experts=2), 7),
                           (dict(n_experts=8, top_k_experts=0), 7), (dict(n_experts=8, top_k_experts=9), 7),
                           (dict(n_experts=2, top_k_experts=3), 7),
                           (dict(n_experts=8, top_k_experts=2, weight_format=pm.WEIGHTS_FP8_E4M3), 7),
                           (dict(n_experts=8, top_k_experts=8, ffn_dim=4096), 7),
                           (dict(n_experts=8, top_k_experts=2), 1)]:      # no w_router
        cfg = pm.lf_config(**{**good, **change})
        assert L.lf_create(C.byref(cfg), C.byref(w), C.byref(h)) == expect, change
    wr = pm.lf_weights(*([0x1000] * 12 + [0] * 8 + [0x1008]))           # router not 16-byte aligned
    cfg = pm.lf_config(**{**good, "n_experts": 8, "top_k_experts": 2})
    assert L.lf_create(C.byref(cfg), C.byref(wr), C.byref(h)) == 1
    wr = pm.lf_weights(*([0x1000] * 12 + [0] * 8 + [0x1000]))           # a router on a dense model
    assert L.lf_create(C.byref(pm.lf_config(**good)), C.byref(wr), C.byref(h)) == 1


def test_noalloc_rejects_batched_prefill_before_touching_the_gpu(pm):
    L = pm.lib()
    good = dict(n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=1024, vocab=4096,
                max_seq=64, rope_theta=10000.0, rms_eps=1e-5, wait_timeout_ns=0, n_ctas=0, fault_step=-1,
                prefill_block=32)
    cfg = pm.lf_config(**good)
    w = pm.lf_weights(*([0x1000] * 12))
    sp = pm.lf_sampling(0.0, 0, None, None)
    assert L.lf_generate_noalloc(C.byref(cfg), C.byref(w), 0x1000, 8, 4, C.byref(sp), 0, 0x1000, None) == 7


def test_calls_on_a_null_handle_are_rejected(pm):
    L = pm.lib()
    sp = pm.lf_sampling(0.0, 0, None, None)
    assert L.lf_prefill(None, None, 4, None) == 1
    assert L.lf_decode(None, 4, C.byref(sp), 0, None, None) == 1
    assert L.lf_sync(None) == 1
    assert L.lf_reset(None) == 1
    assert L.lf_set_schedule(None, 0) == 1
    L.lf_destroy(None)


def test_sync_latency_rejects_bad_arguments_before_touching_the_gpu(pm):
    L = pm.lib()
    v = C.c_double()
    assert L.lf_sync_latency(2, 8, 10, C.byref(v)) == 1
    assert L.lf_sync_latency(0, 1, 10, C.byref(v)) == 1
    assert L.lf_sync_latency(1, 8, 0, C.byref(v)) == 1
    assert L.lf_sync_latency(0, 8, 10, None) == 1
