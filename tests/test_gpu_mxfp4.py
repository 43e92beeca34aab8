"""MXFP4 weights (E2M1 codes, E8M0 scales per 32 elements) on the GPU against the
oracle's MXFP4 decoder, through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
from conftest import cuda_available
from parity import check_tokens, compare_logits
from synthetic import MODELS, WORKLOADS, ModelConfig, make_prompt, make_weights_mxfp4

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    return pm


def _setup(pm, cfg, wseed, max_seq, gains="ones", **kw):
    wg = make_weights_mxfp4(cfg, wseed, device="cuda", gains=gains)
    wc = {k: v.cpu() for k, v in wg.items()}
    dec = pm.Decoder(cfg, wg, max_seq, **kw)
    orc = oracle.OracleDecoder(cfg, wc, max_seq, layer_window=kw.get("layer_window"))
    return dec, orc, wg


def _forced_run(dec, orc, cfg, prompt, n_steps, force_seed, T=0.0, top_k=0, seed=0):
    force = make_prompt(cfg.vocab, n_steps, force_seed)
    dec.prefill(prompt.cuda())
    lg = torch.empty((n_steps, cfg.vocab), dtype=torch.float32, device="cuda")
    toks = dec.decode(n_steps, temperature=T, top_k=top_k, seed=seed, debug_logits=lg, force_tokens=force.cuda())
    assert dec.sync() == 0
    orc.prefill(prompt.numpy())
    _, ref = orc.decode(n_steps, T, top_k, seed, force_tokens=force.numpy())
    return toks.cpu().numpy(), lg.cpu().numpy(), ref


@pytest.mark.parametrize("cfg,gains,window", [
    (MODELS["tiny"], "random", None),
    (MODELS["small"].with_(n_layers=4), "ones", None),
    (ModelConfig("gqa128-mxfp4", 2, 512, 8, 2, 128, 1024, 3000), "random", [300, 0]),
])
def test_mxfp4_forced_parity(pm, cfg, gains, window):
    dec, orc, _ = _setup(pm, cfg, 41, 600, gains=gains, layer_window=window)
    prompt = make_prompt(cfg.vocab, 500, 42)
    toks, lg, ref = _forced_run(dec, orc, cfg, prompt, 32, 43)
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, 499)


def test_mxfp4_sampled_tokens_match_under_the_same_philox_stream(pm):
    cfg = MODELS["tiny"]
    dec, orc, _ = _setup(pm, cfg, 44, 200)
    prompt = make_prompt(cfg.vocab, 20, 45)
    toks, lg, ref = _forced_run(dec, orc, cfg, prompt, 48, 46, T=0.8, top_k=50, seed=1234)
    compare_logits(lg, ref)
    assert check_tokens(toks, ref, 0.8, 50, 1234, 19) > 12


def test_mxfp4_schedules_are_bitwise_identical(pm):
    cfg = MODELS["tiny"]
    wg = make_weights_mxfp4(cfg, 47, device="cuda")
    prompt = make_prompt(cfg.vocab, 30, 3).cuda()
    outs = []
    for sched in (pm.SCHED_FLAGS, pm.SCHED_GRID_BARRIER, pm.SCHED_MULTI_KERNEL):
        dec = pm.Decoder(cfg, wg, 64)
        dec.set_schedule(sched)
        dec.prefill(prompt)
        lg = torch.empty((16, cfg.vocab), dtype=torch.float32, device="cuda")
        t = dec.decode(16, debug_logits=lg)
        assert dec.sync() == 0
        outs.append((t.cpu().numpy(), lg.cpu().numpy()))
        dec.close()
    for t, lg in outs[1:]:
        assert np.array_equal(t, outs[0][0]) and np.array_equal(lg, outs[0][1])


def test_full_size_2p3b_mxfp4_parity(pm):
    """The ~2.3B decoder with MXFP4 weights at full size and the bench's grid."""
    wl = WORKLOADS["2.3b-mxfp4"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, wl.weight_seed, 64)
    prompt = make_prompt(cfg.vocab, 24, wl.prompt_seed)
    toks, lg, ref = _forced_run(dec, orc, cfg, prompt, 8, 57)
    compare_logits(lg, ref)
    assert check_tokens(toks, ref, 0.0, 0, 0, 23) >= 6


def test_mxfp4_decoder_reports_its_format(pm):
    cfg = MODELS["tiny"]
    dec, _, _ = _setup(pm, cfg, 49, 64)
    assert dec.mxfp4 and not dec.fp8
    # the stream holds 144 bytes per row of 256 weights (codes, scales, padding)
    L, d, F, V, Q, KV = cfg.n_layers, cfg.d_model, cfg.ffn_dim, cfg.vocab, cfg.q_dim, cfg.kv_dim
    groups = L * ((Q + 2 * KV) * d + d * Q + 3 * d * F) // 256 + V * d // 256
    assert dec.info()["weight_stream_bytes"] == 144 * groups


@pytest.mark.parametrize("cfg,window", [
    (MODELS["tiny"], None),
    (ModelConfig("gqa128-mxpf", 2, 512, 8, 2, 128, 1024, 3000), [100, 0]),
])
def test_mxfp4_batched_prefill_parity(pm, cfg, window):
    """The batched prefill on the FP16-decoded MXFP4 weights, then the MXFP4 decode kernel."""
    dec, orc, _ = _setup(pm, cfg, 50, 300, gains="random", layer_window=window, prefill_block=48)
    assert dec.info()["prefill_block"] == 48
    prompt = make_prompt(cfg.vocab, 230, 51)
    toks, lg, ref = _forced_run(dec, orc, cfg, prompt, 16, 52)
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, 229)


def test_mxfp4_batched_prefill_rejects_scales_outside_the_exact_range(pm):
    cfg = MODELS["tiny"]
    wg = make_weights_mxfp4(cfg, 53, device="cuda")
    wg["w_up_scale"][1, 3, 2] = 150          # 2^23: not exact in FP16
    with pytest.raises(pm.LFError):
        pm.Decoder(cfg, wg, 64, prefill_block=16)
    pm.Decoder(cfg, wg, 64).close()          # the step-wise prefill takes any scale
