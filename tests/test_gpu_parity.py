"""CUDA monokernel vs the CPU oracle, through the C ABI (needs a GB300)."""
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


def _setup(pm, cfg, wseed, max_seq, gains="ones", **kw):
    wg = make_weights(cfg, wseed, device="cuda", gains=gains)
    wc = {k: v.cpu() for k, v in wg.items()}
    dec = pm.Decoder(cfg, wg, max_seq, **kw)
    orc = oracle.OracleDecoder(cfg, wc, max_seq, layer_window=kw.get("layer_window"))
    return dec, orc, wg


def _forced_run(pm, dec, orc, cfg, prompt, n_steps, force_seed, T=0.0, top_k=0, seed=0):
    """Both sides: prefill `prompt`, then n_steps decode steps fed a fixed seeded
    token sequence (teacher forcing).  Returns (gpu tokens, gpu logits, oracle logits)."""
    force = make_prompt(cfg.vocab, n_steps, force_seed)
    dec.prefill(prompt.cuda())
    lg = torch.empty((n_steps, cfg.vocab), dtype=torch.float32, device="cuda")
    toks = dec.decode(n_steps, temperature=T, top_k=top_k, seed=seed, debug_logits=lg, force_tokens=force.cuda())
    assert dec.sync() == 0
    orc.prefill(prompt.numpy())
    _, ref = orc.decode(n_steps, T, top_k, seed, force_tokens=force.numpy())
    return toks.cpu().numpy(), lg.cpu().numpy(), ref


@pytest.mark.parametrize("gains", ["ones", "random"])
def test_tiny_forced_logits_and_greedy_tokens(pm, gains):
    wl = WORKLOADS["tiny"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, wl.weight_seed, wl.max_seq, gains=gains)
    prompt = make_prompt(cfg.vocab, wl.prompt_len, wl.prompt_seed)
    toks, lg, ref = _forced_run(pm, dec, orc, cfg, prompt, wl.decode_steps, 77)
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, wl.prompt_len - 1)


def test_tiny_free_running_greedy_matches_until_a_near_tie(pm):
    """Both sides decode greedily on their own; tokens must agree until the
    first step whose oracle margin is within 0.05, where the GPU's token must
    be one of the near-best ones (after that the sequences may diverge)."""
    wl = WORKLOADS["tiny"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, wl.weight_seed, wl.max_seq)
    prompt = make_prompt(cfg.vocab, wl.prompt_len, wl.prompt_seed)
    dec.prefill(prompt.cuda())
    gpu = dec.decode(wl.decode_steps).cpu().numpy()
    assert dec.sync() == 0
    lg = None
    for t in prompt.numpy():
        lg = orc.forward(int(t))
    for i in range(wl.decode_steps):
        best = int(np.argmax(lg))
        if gpu[i] != best:
            top2 = np.sort(lg)[-2:]
            assert top2[1] - top2[0] <= 0.05 and lg[gpu[i]] >= lg[best] - 0.05, f"step {i}"
            break
        lg = orc.forward(best)


def test_small_forced_parity(pm):
    wl = WORKLOADS["small"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, wl.weight_seed, wl.max_seq)
    prompt = make_prompt(cfg.vocab, wl.prompt_len, wl.prompt_seed)
    toks, lg, ref = _forced_run(pm, dec, orc, cfg, prompt, 48, 78)
    compare_logits(lg, ref)
    assert check_tokens(toks, ref, 0.0, 0, 0, wl.prompt_len - 1) > 24


def test_hd128_gqa_shape_parity(pm):
    cfg = ModelConfig("gqa128", 2, 512, 8, 2, 128, 1024, 3000)
    dec, orc, _ = _setup(pm, cfg, 21, 200, gains="random")
    prompt = make_prompt(cfg.vocab, 100, 22)
    toks, lg, ref = _forced_run(pm, dec, orc, cfg, prompt, 40, 23)
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, 99)


@pytest.mark.parametrize("T,k", [(0.8, 50), (1.0, 0), (0.7, 2)])
def test_sampled_tokens_match_under_the_same_philox_stream(pm, T, k):
    wl = WORKLOADS["tiny"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, 5, 200)
    prompt = make_prompt(cfg.vocab, 20, 9)
    toks, lg, ref = _forced_run(pm, dec, orc, cfg, prompt, 64, 10, T=T, top_k=k, seed=1234)
    compare_logits(lg, ref)
    assert check_tokens(toks, ref, T, k, 1234, 19) > 16


@pytest.mark.parametrize("n_ctas", [3, 7, 64])
def test_small_grids_give_the_same_logits(pm, n_ctas):
    wl = WORKLOADS["tiny"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, wl.weight_seed, 128, n_ctas=n_ctas)
    assert dec.info()["n_ctas"] == n_ctas
    prompt = make_prompt(cfg.vocab, 40, 31)
    toks, lg, ref = _forced_run(pm, dec, orc, cfg, prompt, 24, 32)
    compare_logits(lg, ref)


def test_schedules_are_bitwise_identical(pm):
    wl = WORKLOADS["tiny"]
    cfg = wl.model
    wg = make_weights(cfg, 0, device="cuda")
    prompt = make_prompt(cfg.vocab, 30, 3).cuda()
    force = make_prompt(cfg.vocab, 20, 4).cuda()
    outs = []
    for sched in (pm.SCHED_FLAGS, pm.SCHED_GRID_BARRIER, pm.SCHED_MULTI_KERNEL):
        dec = pm.Decoder(cfg, wg, 64)
        dec.set_schedule(sched)
        dec.prefill(prompt)
        lg = torch.empty((20, cfg.vocab), dtype=torch.float32, device="cuda")
        t = dec.decode(20, temperature=0.9, top_k=10, seed=7, debug_logits=lg, force_tokens=force)
        assert dec.sync() == 0
        outs.append((t.cpu().numpy(), lg.cpu().numpy()))
        dec.close()
    for t, lg in outs[1:]:
        assert np.array_equal(t, outs[0][0])
        assert np.array_equal(lg, outs[0][1])


def test_decode_calls_compose_and_repeat_bitwise(pm):
    wl = WORKLOADS["tiny"]
    cfg = wl.model
    wg = make_weights(cfg, 0, device="cuda")
    prompt = make_prompt(cfg.vocab, 16, 1).cuda()
    dec = pm.Decoder(cfg, wg, 128)
    runs = []
    for split in (None, 11, None):
        dec.reset()
        dec.prefill(prompt)
        if split is None:
            runs.append(dec.decode(40, temperature=0.9, top_k=20, seed=99).cpu().numpy())
        else:
            a = dec.decode(split, temperature=0.9, top_k=20, seed=99).cpu().numpy()
            b = dec.decode(40 - split, temperature=0.9, top_k=20, seed=99).cpu().numpy()
            runs.append(np.concatenate([a, b]))
        assert dec.sync() == 0
    assert np.array_equal(runs[0], runs[1]) and np.array_equal(runs[0], runs[2])


def test_prefill_in_two_calls_equals_one(pm):
    cfg = MODELS["tiny"]
    wg = make_weights(cfg, 0, device="cuda")
    prompt = make_prompt(cfg.vocab, 33, 8).cuda()
    dec = pm.Decoder(cfg, wg, 96)
    dec.prefill(prompt)
    a = dec.decode(10).cpu().numpy()
    dec.reset()
    dec.prefill(prompt[:20].contiguous())
    dec.prefill(prompt[20:].contiguous())
    b = dec.decode(10).cpu().numpy()
    assert dec.sync() == 0
    assert np.array_equal(a, b)


def test_generate_with_host_buffers(pm):
    cfg = MODELS["tiny"]
    wg = make_weights(cfg, 0, device="cuda")
    prompt = make_prompt(cfg.vocab, 12, 8)
    dec = pm.Decoder(cfg, wg, 64)
    host = dec.generate(prompt.numpy(), 16)
    dec.reset()
    dec.prefill(prompt.cuda())
    dev = dec.decode(16).cpu().numpy()
    assert np.array_equal(host, dev)


def test_errors_capacity_state_and_top_k(pm):
    cfg = MODELS["tiny"]
    wg = make_weights(cfg, 0, device="cuda")
    dec = pm.Decoder(cfg, wg, 16)
    with pytest.raises(pm.LFError) as e:
        dec.decode(1)
    assert e.value.status == 8
    dec.prefill(make_prompt(cfg.vocab, 8, 1).cuda())
    with pytest.raises(pm.LFError) as e:
        dec.decode(10)
    assert e.value.status == 3
    with pytest.raises(pm.LFError) as e:
        dec.decode(2, temperature=1.0, top_k=65)
    assert e.value.status == 7
    dec.decode(9)
    assert dec.sync() == 0
    assert dec.info()["position"] == 16


def test_bounded_wait_runs_out_and_the_handle_recovers(pm):
    """A readiness signal that is never published (test hook) makes the
    consumers' bounded waits expire: the kernel returns, lf_sync reports
    LF_ERR_TIMEOUT, and after lf_reset the same handle decodes correctly."""
    cfg = MODELS["tiny"]
    wg = make_weights(cfg, 0, device="cuda")
    prompt = make_prompt(cfg.vocab, 10, 2).cuda()
    ref = pm.Decoder(cfg, wg, 64)
    ref.prefill(prompt)
    want = ref.decode(6).cpu().numpy()
    dec = pm.Decoder(cfg, wg, 64, wait_timeout_ns=200_000_000, fault_step=3)
    dec.prefill(prompt)
    dec.decode(6)
    assert dec.sync() == 6
    with pytest.raises(pm.LFError) as e:
        dec.decode(1)
    assert e.value.status == 8
    dec.reset()
    dec.set_schedule(pm.SCHED_MULTI_KERNEL)   # the fault hook only acts in the persistent schedules
    dec.prefill(prompt)
    got = dec.decode(6).cpu().numpy()
    assert dec.sync() == 0
    assert np.array_equal(got, want)


@pytest.mark.parametrize("cfg,prompt_len,wseed", [
    (MODELS["tiny"], 3000, 0),                                        # 38 pieces per KV head
    (ModelConfig("gqa128-long", 1, 512, 8, 2, 128, 1024, 2000), 2000, 24),
])
def test_long_context_parity(pm, cfg, prompt_len, wseed):
    """Split-KV attention over thousands of cached positions: many pieces,
    several combine batches, hd 64 (MHA) and hd 128 (GQA)."""
    n = 12
    dec, orc, _ = _setup(pm, cfg, wseed, prompt_len + n)
    prompt = make_prompt(cfg.vocab, prompt_len, wseed + 100)
    toks, lg, ref = _forced_run(pm, dec, orc, cfg, prompt, n, wseed + 200)
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, prompt_len - 1)


def test_full_size_2p3b_decoder_parity(pm):
    """The ~2.3B workload's decoder at its full size and launch configuration
    (the bench's grid), on a short sequence the oracle can follow."""
    wl = WORKLOADS["2.3b"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, wl.weight_seed, 64)
    prompt = make_prompt(cfg.vocab, 24, wl.prompt_seed)
    toks, lg, ref = _forced_run(pm, dec, orc, cfg, prompt, 8, 55)
    compare_logits(lg, ref)
    assert check_tokens(toks, ref, 0.0, 0, 0, 23) >= 6


def test_full_size_8b_sampled_parity(pm):
    """The 8B-shape workload's decoder at full size, sampled in-kernel at
    T = 0.8, top-k 50 with its Philox seed, against the oracle's choice."""
    wl = WORKLOADS["8b"]
    cfg = wl.model
    dec, orc, _ = _setup(pm, cfg, wl.weight_seed, 32)
    prompt = make_prompt(cfg.vocab, 8, wl.prompt_seed)
    toks, lg, ref = _forced_run(pm, dec, orc, cfg, prompt, 6, 56, T=wl.temperature, top_k=wl.top_k,
                                seed=wl.sample_seed)
    compare_logits(lg, ref)
    check_tokens(toks, ref, wl.temperature, wl.top_k, wl.sample_seed, 7)


# ---- sliding-window attention (shivam2003.com, "Why GQA and sliding windows")

@pytest.mark.parametrize("cfg,window,prompt_len,steps", [
    # MHA, windows below, at and above the context, one window not a multiple of the 32-position sub-block
    (MODELS["tiny"], [37, 0], 64, 24),
    # GQA 16/4 x 64, windowed and full layers interleaved (the pages: 10 of 15 layers windowed)
    (MODELS["small"].with_(n_layers=6), [100, 100, 0, 100, 100, 0], 160, 24),
    # hd 128, the window spans several split-KV pieces and moves across them step by step
    (ModelConfig("gqa128w", 2, 512, 8, 2, 128, 1024, 3000), [700, 1], 900, 40),
])
def test_sliding_window_parity(pm, cfg, window, prompt_len, steps):
    dec, orc, _ = _setup(pm, cfg, 31, prompt_len + steps + 1, gains="random", layer_window=window)
    prompt = make_prompt(cfg.vocab, prompt_len, 32)
    toks, lg, ref = _forced_run(pm, dec, orc, cfg, prompt, steps, 33)
    compare_logits(lg, ref)
    check_tokens(toks, ref, 0.0, 0, 0, prompt_len - 1)


def test_window_covering_the_context_is_bitwise_full_attention(pm):
    wl = WORKLOADS["tiny"]
    cfg = wl.model
    wg = make_weights(cfg, wl.weight_seed, device="cuda")
    prompt = make_prompt(cfg.vocab, wl.prompt_len, wl.prompt_seed).cuda()
    out = []
    for win in (None, [wl.max_seq, wl.max_seq + 7]):
        dec = pm.Decoder(cfg, wg, wl.max_seq, layer_window=win)
        dec.prefill(prompt)
        lg = torch.empty((16, cfg.vocab), dtype=torch.float32, device="cuda")
        toks = dec.decode(16, debug_logits=lg)
        assert dec.sync() == 0
        out.append((toks.cpu(), lg.cpu()))
        dec.close()
    assert torch.equal(out[0][0], out[1][0]) and torch.equal(out[0][1], out[1][1])
