"""lf_generate_noalloc: a whole request without any device allocation.

It is meant for callers that cannot call cudaMalloc when a request arrives
(for instance a plugin inside a host framework that owns all device memory
through its own pool).  Its scratch is one static device array shared by all
calls, so this file checks it against the handle-based path (lf_create +
lf_prefill + lf_decode) on two calls in a row, with different prompts and
sampling, so that stale contents from the first call would show in the
second.  The file is named to be collected last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from conftest import cuda_available
from parity import check_tokens, compare_logits
from synthetic import WORKLOADS, make_prompt, make_weights

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    return pm


def _cfg(pm, m, max_seq, window=None):
    win = (C.c_int32 * m.n_layers)(*window) if window is not None else None
    return pm.lf_config(m.n_layers, m.d_model, m.n_heads, m.n_kv_heads, m.head_dim, m.ffn_dim, m.vocab, max_seq,
                        m.rope_theta, m.rms_eps, 0, 0, -1, win)


def _noalloc(pm, cfg, weights, prompt, n_steps, T, k, seed):
    w = pm.lf_weights(*[int(weights[n].data_ptr()) for n in pm.WEIGHT_FIELDS])
    out = torch.full((n_steps,), -1, dtype=torch.int32, device="cuda")
    lg = torch.full((n_steps, cfg.vocab), float("nan"), dtype=torch.float32, device="cuda")
    sp = pm.lf_sampling(T, k, int(lg.data_ptr()), None)
    st = pm.lib().lf_generate_noalloc(C.byref(cfg), C.byref(w), int(prompt.data_ptr()), prompt.numel(), n_steps,
                                      C.byref(sp), seed, int(out.data_ptr()),
                                      int(torch.cuda.current_stream().cuda_stream))
    assert st == 0, pm.error_string(st)
    return out.cpu().numpy(), lg.cpu().numpy()


def _handle_path(pm, model, weights, max_seq, prompt, n_steps, T, k, seed, window=None):
    dec = pm.Decoder(model, weights, max_seq, layer_window=window)
    dec.prefill(prompt)
    lg = torch.empty((n_steps, model.vocab), dtype=torch.float32, device="cuda")
    toks = dec.decode(n_steps, temperature=T, top_k=k, seed=seed, debug_logits=lg)
    assert dec.sync() == 0
    dec.close()
    return toks.cpu().numpy(), lg.cpu().numpy()


def test_noalloc_matches_the_handle_path_on_two_calls_in_a_row(pm):
    wl = WORKLOADS["tiny"]
    m = wl.model
    weights = make_weights(m, wl.weight_seed, device="cuda")
    cfg = _cfg(pm, m, wl.max_seq)
    runs = [(make_prompt(m.vocab, wl.prompt_len, wl.prompt_seed).cuda(), wl.decode_steps, 0.0, 0, 0),
            (make_prompt(m.vocab, 40, 4321).cuda(), 48, 0.8, 20, 99)]
    for prompt, n, T, k, seed in runs:
        toks, lg = _noalloc(pm, cfg, weights, prompt, n, T, k, seed)
        ref_toks, ref_lg = _handle_path(pm, m, weights, wl.max_seq, prompt, n, T, k, seed)
        compare_logits(lg, ref_lg)
        check_tokens(toks, ref_lg, T, k, seed, prompt.numel() - 1)
        assert np.all((toks >= 0) & (toks < m.vocab))


def test_noalloc_with_sliding_windows_matches_the_handle_path(pm):
    wl = WORKLOADS["tiny"]
    m = wl.model
    weights = make_weights(m, wl.weight_seed, device="cuda")
    window = [29, 0]
    cfg = _cfg(pm, m, wl.max_seq, window)
    prompt = make_prompt(m.vocab, wl.prompt_len, wl.prompt_seed).cuda()
    toks, lg = _noalloc(pm, cfg, weights, prompt, 24, 0.0, 0, 0)
    ref_toks, ref_lg = _handle_path(pm, m, weights, wl.max_seq, prompt, 24, 0.0, 0, 0, window)
    compare_logits(lg, ref_lg)
    check_tokens(toks, ref_lg, 0.0, 0, 0, prompt.numel() - 1)


def test_noalloc_rejects_requests_beyond_its_scratch(pm):
    wl = WORKLOADS["tiny"]
    m = wl.model
    weights = make_weights(m, wl.weight_seed, device="cuda")
    cfg = _cfg(pm, m, 32768)           # a 32k-position KV cache needs 64 MiB of scratch
    w = pm.lf_weights(*[int(weights[n].data_ptr()) for n in pm.WEIGHT_FIELDS])
    prompt = make_prompt(m.vocab, 8, 1).cuda()
    out = torch.empty(4, dtype=torch.int32, device="cuda")
    sp = pm.lf_sampling(0.0, 0, None, None)
    st = pm.lib().lf_generate_noalloc(C.byref(cfg), C.byref(w), int(prompt.data_ptr()), 8, 4, C.byref(sp), 0,
                                      int(out.data_ptr()), int(torch.cuda.current_stream().cuda_stream))
    assert st == 3   # LF_ERR_CAPACITY


def test_noalloc_refuses_a_capturing_stream(pm):
    """Every call copies from pageable host memory and synchronizes its
    stream, which a CUDA graph capture cannot hold: on a capturing stream the
    call returns LF_ERR_NOT_SUPPORTED before it queues any work."""
    wl = WORKLOADS["tiny"]
    m = wl.model
    weights = make_weights(m, wl.weight_seed, device="cuda")
    cfg = _cfg(pm, m, 64)
    w = pm.lf_weights(*[int(weights[n].data_ptr()) for n in pm.WEIGHT_FIELDS])
    prompt = make_prompt(m.vocab, 8, 1).cuda()
    out = torch.empty(4, dtype=torch.int32, device="cuda")
    sp = pm.lf_sampling(0.0, 0, None, None)
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        graph.capture_begin()
        try:
            st = pm.lib().lf_generate_noalloc(C.byref(cfg), C.byref(w), int(prompt.data_ptr()), 8, 4, C.byref(sp), 0,
                                              int(out.data_ptr()), int(side.cuda_stream))
        finally:
            graph.capture_end()
    assert st == 7   # LF_ERR_NOT_SUPPORTED
