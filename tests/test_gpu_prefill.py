"""Batched prefill (lf_config.prefill_block > 0) on the GPU: the prompt's
forward passes run over blocks of positions (tensor-core GEMMs and a causal
flash-style attention), then the monokernel decodes from the cache they
filled.  The decode logits must match the oracle's, which runs the same
prompt one position at a time (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
from conftest import cuda_available
from parity import check_tokens, compare_logits
from synthetic import MODELS, WORKLOADS, ModelConfig, make_prompt, make_weights, make_weights_fp8

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    return pm


def _setup(pm, cfg, wseed, max_seq, block, gains="random", fp8=False, **kw):
    make = make_weights_fp8 if fp8 else make_weights
    wg = make(cfg, wseed, device="cuda", gains=gains)
    wc = {k: v.cpu() for k, v in wg.items()}
    dec = pm.Decoder(cfg, wg, max_seq, prefill_block=block, **kw)
    orc = oracle.OracleDecoder(cfg, wc, max_seq, layer_window=kw.get("layer_window"))
    return dec, orc, wg


def _forced_decode(dec, cfg, n_steps, force):
    lg = torch.empty((n_steps, cfg.vocab), dtype=torch.float32, device="cuda")
    toks = dec.decode(n_steps, debug_logits=lg, force_tokens=force.cuda())
    assert dec.sync() == 0
    return toks.cpu().numpy(), lg.cpu().numpy()


@pytest.mark.parametrize("cfg,block,prompt_len,window", [
    # MHA, hd 64: three full blocks and a ragged tail
    (MODELS["tiny"], 48, 150, None),
    # GQA 16 / 4, hd 64, several blocks of 64 query rows
    (MODELS["small"].with_(n_layers=4), 64, 200, None),
    # hd 128, GQA 8 / 2, a window that reaches back across blocks next to a full layer
    (ModelConfig("gqa128-pf", 2, 512, 8, 2, 128, 1024, 3000), 128, 500, [300, 0]),
    # one position per block
    (MODELS["tiny"], 1, 20, None),
    # a block larger than the whole cache (capped at max_seq), windows below and above the prompt
    (MODELS["tiny"], 4096, 64, [37, 1000]),
])
def test_batched_prefill_then_decode_matches_the_oracle(pm, cfg, block, prompt_len, window):
    n = 16
    dec, orc, _ = _setup(pm, cfg, 61, prompt_len + n + 1, block, layer_window=window)
    info = dec.info()
    assert info["prefill_block"] == min(block, prompt_len + n + 1) and info["prefill_bytes"] > 0
    prompt = make_prompt(cfg.vocab, prompt_len, 62)
    force = make_prompt(cfg.vocab, n, 63)
    dec.prefill(prompt.cuda())
    toks, lg = _forced_decode(dec, cfg, n, force)
    orc.prefill(prompt.numpy())
    _, ref = orc.decode(n, force_tokens=force.numpy())
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, prompt_len - 1)


def test_batched_prefill_continues_a_sequence(pm):
    """prefill, decode, prefill again (the pending token runs first), decode."""
    cfg = MODELS["tiny"]
    dec, orc, _ = _setup(pm, cfg, 64, 200, 16)
    p1, p2 = make_prompt(cfg.vocab, 37, 65), make_prompt(cfg.vocab, 41, 66)
    f1, f2 = make_prompt(cfg.vocab, 5, 67), make_prompt(cfg.vocab, 12, 68)
    dec.prefill(p1.cuda())
    _forced_decode(dec, cfg, 5, f1)
    dec.prefill(p2.cuda())
    toks, lg = _forced_decode(dec, cfg, 12, f2)
    orc.prefill(p1.numpy())
    orc.decode(5, force_tokens=f1.numpy())
    orc.prefill(p2.numpy())
    _, ref = orc.decode(12, force_tokens=f2.numpy())
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, 37 + 5 + 40)


def test_batched_prefill_with_fp8_weights(pm):
    cfg = ModelConfig("gqa128-fp8pf", 2, 512, 8, 2, 128, 1024, 3000)
    n = 16
    dec, orc, _ = _setup(pm, cfg, 69, 300, 64, fp8=True, layer_window=[100, 0])
    prompt = make_prompt(cfg.vocab, 230, 70)
    force = make_prompt(cfg.vocab, n, 71)
    dec.prefill(prompt.cuda())
    toks, lg = _forced_decode(dec, cfg, n, force)
    orc.prefill(prompt.numpy())
    _, ref = orc.decode(n, force_tokens=force.numpy())
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, 229)


def test_batched_prefill_reports_a_bad_token_and_recovers(pm):
    cfg = MODELS["tiny"]
    dec, _, _ = _setup(pm, cfg, 72, 64, 16)
    prompt = make_prompt(cfg.vocab, 30, 73)
    bad = prompt.clone()
    bad[7] = cfg.vocab + 3
    dec.prefill(bad.cuda())
    assert dec.sync() == 1    # LF_ERR_INVALID_ARG, latched
    dec.reset()
    dec.prefill(prompt.cuda())
    dec.decode(4)
    assert dec.sync() == 0


def test_full_size_2p3b_batched_prefill_parity(pm):
    """The ~2.3B decoder at full size: a prompt of several blocks, then decode
    steps against the oracle on a sequence it can follow."""
    wl = WORKLOADS["2.3b"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, wl.weight_seed, 64, 16, gains="ones")
    prompt = make_prompt(cfg.vocab, 40, wl.prompt_seed)
    force = make_prompt(cfg.vocab, 8, 74)
    dec.prefill(prompt.cuda())
    toks, lg = _forced_decode(dec, cfg, 8, force)
    orc.prefill(prompt.numpy())
    _, ref = orc.decode(8, force_tokens=force.numpy())
    compare_logits(lg, ref)
    assert check_tokens(toks, ref, 0.0, 0, 0, 39) >= 6


def test_full_size_2p3b_long_prompt_batched_equals_stepwise(pm):
    """At 8,192 cached positions (too long for the oracle), the batched
    prefill and the monokernel's step-by-step prefill of the same prompt
    must give the same decode logits within the oracle tolerance."""
    wl = WORKLOADS["2.3b"]
    cfg = wl.model
    n, plen = 8, 8192
    wg = make_weights(cfg, wl.weight_seed, device="cuda")
    prompt = make_prompt(cfg.vocab, plen, 75).cuda()
    force = make_prompt(cfg.vocab, n, 76)
    out = []
    for block in (0, 1024):
        dec = pm.Decoder(cfg, wg, plen + n + 1, prefill_block=block)
        dec.prefill(prompt)
        out.append(_forced_decode(dec, cfg, n, force))
        dec.close()
    (t0, l0), (t1, l1) = out
    compare_logits(l1, l0)
    check_tokens(t1, l0, 0.0, 0, 0, plen - 1)


def test_automatic_prefill_block_fits_the_attention_in_one_wave(pm):
    """prefill_block = LF_PREFILL_AUTO: the library picks the largest multiple
    of 128 up to 1024 whose attention grid ((block / 128) x heads CTAs) fills
    its waves of SMs to at least 80 % of the best such block's (896 for 20
    heads on 152 SMs), and the batched prefill it runs, here over two blocks,
    still matches the oracle."""
    cfg = ModelConfig("auto-20h", 1, 768, 20, 5, 128, 1024, 3000)
    n, prompt_len = 8, 960
    dec, orc, _ = _setup(pm, cfg, 71, prompt_len + n + 1, pm.PREFILL_AUTO)
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    def fill(b):
        k = b // 128 * cfg.n_heads
        return k / (-(-k // sms) * sms)

    best = max(fill(b) for b in range(128, 1025, 128))
    want = next(b for b in range(1024, 127, -128) if fill(b) >= 0.8 * best)
    assert dec.info()["prefill_block"] == min(want, prompt_len + n + 1)
    if sms == 152:
        assert want == 896
    prompt = make_prompt(cfg.vocab, prompt_len, 72)
    force = make_prompt(cfg.vocab, n, 73)
    dec.prefill(prompt.cuda())
    toks, lg = _forced_decode(dec, cfg, n, force)
    orc.prefill(prompt.numpy())
    _, ref = orc.decode(n, force_tokens=force.numpy())
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, prompt_len - 1)
