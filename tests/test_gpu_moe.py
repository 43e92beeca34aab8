"""Mixture-of-experts FFN on the GPU against the oracle, through the C ABI
(needs a GB300): the kernel chooses each layer's experts from its own router
logits and streams only their rows; the decode logits (and with them the
expert choices) must match the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from conftest import cuda_available
from parity import check_tokens, compare_logits
from synthetic import MODELS, WORKLOADS, ModelConfig, make_prompt, make_weights

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    return pm


def _setup(pm, cfg, wseed, max_seq, gains="random", **kw):
    wg = make_weights(cfg, wseed, device="cuda", gains=gains)
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


@pytest.mark.parametrize("cfg,window", [
    # 6 experts of 512 units, 2 active, MHA hd 64
    (ModelConfig("moe-a", 2, 256, 4, 4, 64, 512, 4096, n_experts=6, top_k_experts=2), None),
    # top-1 of 4 (gate exactly 1), GQA 8/2 x 128, a sliding window next to a full layer
    (ModelConfig("moe-b", 2, 512, 8, 2, 128, 256, 3000, n_experts=4, top_k_experts=1), [40, 0]),
    # 16 experts, 4 active (h of 4 x 1,024 units), GQA 16/4 x 64
    (ModelConfig("moe-c", 3, 1024, 16, 4, 64, 1024, 8000, n_experts=16, top_k_experts=4), None),
    # 64 experts (two router logits per lane), 8 active
    (ModelConfig("moe-d", 1, 256, 4, 4, 64, 256, 2000, n_experts=64, top_k_experts=8), None),
    # d 2,048 with 16 experts (wider router rows)
    (ModelConfig("moe-e", 1, 2048, 16, 4, 128, 512, 2000, n_experts=16, top_k_experts=2), None),
])
def test_moe_forced_parity(pm, cfg, window):
    dec, orc, _ = _setup(pm, cfg, 81, 200, layer_window=window)
    prompt = make_prompt(cfg.vocab, 100, 82)
    toks, lg, ref = _forced_run(dec, orc, cfg, prompt, 24, 83)
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, 99)


def test_moe_sampled_tokens_match_under_the_same_philox_stream(pm):
    cfg = ModelConfig("moe-a", 2, 256, 4, 4, 64, 512, 4096, n_experts=6, top_k_experts=2)
    dec, orc, _ = _setup(pm, cfg, 84, 200)
    prompt = make_prompt(cfg.vocab, 20, 85)
    toks, lg, ref = _forced_run(dec, orc, cfg, prompt, 48, 86, T=0.8, top_k=50, seed=1234)
    compare_logits(lg, ref)
    assert check_tokens(toks, ref, 0.8, 50, 1234, 19) > 12


def test_moe_grid_barrier_schedule_is_bitwise_identical_and_multi_kernel_is_refused(pm):
    cfg = ModelConfig("moe-a", 2, 256, 4, 4, 64, 512, 4096, n_experts=6, top_k_experts=2)
    wg = make_weights(cfg, 87, device="cuda")
    prompt = make_prompt(cfg.vocab, 30, 3).cuda()
    outs = []
    for sched in (pm.SCHED_FLAGS, pm.SCHED_GRID_BARRIER):
        dec = pm.Decoder(cfg, wg, 64)
        dec.set_schedule(sched)
        dec.prefill(prompt)
        lg = torch.empty((16, cfg.vocab), dtype=torch.float32, device="cuda")
        t = dec.decode(16, debug_logits=lg)
        assert dec.sync() == 0
        outs.append((t.cpu().numpy(), lg.cpu().numpy()))
        if sched == pm.SCHED_FLAGS:
            with pytest.raises(pm.LFError):
                dec.set_schedule(pm.SCHED_MULTI_KERNEL)
        dec.close()
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_one_expert_equals_the_dense_decoder_bitwise(pm):
    """E = 1, top-1: gate 1.0, the same rows streamed in the same tiles as the
    dense model whose FFN is that expert, so the logits are bit-identical."""
    cfg = ModelConfig("moe-1", 2, 256, 4, 4, 64, 1024, 4096, n_experts=1, top_k_experts=1)
    wg = make_weights(cfg, 88, device="cuda")
    dense = cfg.with_(n_experts=0, top_k_experts=0)
    wd = {k: v for k, v in wg.items() if k != "w_router"}
    for n in ("w_gate", "w_up", "w_down"):
        wd[n] = wg[n][:, 0].contiguous()
    prompt = make_prompt(cfg.vocab, 30, 4).cuda()
    outs = []
    for c, w in ((cfg, wg), (dense, wd)):
        dec = pm.Decoder(c, w, 64)
        dec.prefill(prompt)
        lg = torch.empty((12, cfg.vocab), dtype=torch.float32, device="cuda")
        t = dec.decode(12, debug_logits=lg)
        assert dec.sync() == 0
        outs.append((t.cpu().numpy(), lg.cpu().numpy()))
        dec.close()
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_full_size_moe_parity(pm):
    """The 8-expert, 2-active decoder with the ~2.3B's attention at full size
    (6.3B expert parameters, 2.3B active per token) and the bench's grid."""
    wl = WORKLOADS["moe-8x"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, wl.weight_seed, 64, gains="ones")
    prompt = make_prompt(cfg.vocab, 24, wl.prompt_seed)
    toks, lg, ref = _forced_run(dec, orc, cfg, prompt, 8, 89)
    compare_logits(lg, ref)
    assert check_tokens(toks, ref, 0.0, 0, 0, 23) >= 6


@pytest.mark.parametrize("cfg,window", [
    (ModelConfig("moe-a", 2, 256, 4, 4, 64, 512, 4096, n_experts=6, top_k_experts=2), None),
    (ModelConfig("moe-b", 2, 512, 8, 2, 128, 256, 3000, n_experts=4, top_k_experts=1), [40, 0]),
    (ModelConfig("moe-c", 3, 1024, 16, 4, 64, 1024, 8000, n_experts=16, top_k_experts=4), None),
    (ModelConfig("moe-d", 1, 256, 4, 4, 64, 256, 2000, n_experts=64, top_k_experts=8), None),
])
def test_moe_batched_prefill_parity(pm, cfg, window):
    """The batched prefill routes the block's tokens and runs one GEMM per
    expert; the decode that follows must match the oracle."""
    dec, orc, _ = _setup(pm, cfg, 95, 200, layer_window=window, prefill_block=32)
    assert dec.info()["prefill_block"] == 32
    prompt = make_prompt(cfg.vocab, 100, 96)
    toks, lg, ref = _forced_run(dec, orc, cfg, prompt, 16, 97)
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, 99)
