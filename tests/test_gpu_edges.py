"""Edge cases of the decode path on the GPU against the oracle (needs a
GB300): GQA group sizes 2 and 8, the longest supported vectors (d_model or
ffn_dim of 16,384 = 64 slices), a one-token prompt, and a cache filled to its
last position -- each with the prompt run step by step and batched."""
import numpy as np
import pytest
import torch

import oracle
from conftest import cuda_available
from parity import check_tokens, compare_logits
from synthetic import MODELS, ModelConfig, make_prompt, make_weights

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    return pm


def _run(pm, cfg, wseed, prompt_len, n_steps, max_seq, block, gains="random"):
    wg = make_weights(cfg, wseed, device="cuda", gains=gains)
    dec = pm.Decoder(cfg, wg, max_seq, prefill_block=block)
    orc = oracle.OracleDecoder(cfg, {k: v.cpu() for k, v in wg.items()}, max_seq)
    prompt = make_prompt(cfg.vocab, prompt_len, wseed + 1)
    force = make_prompt(cfg.vocab, n_steps, wseed + 2)
    dec.prefill(prompt.cuda())
    lg = torch.empty((n_steps, cfg.vocab), dtype=torch.float32, device="cuda")
    toks = dec.decode(n_steps, debug_logits=lg, force_tokens=force.cuda())
    assert dec.sync() == 0
    orc.prefill(prompt.numpy())
    _, ref = orc.decode(n_steps, force_tokens=force.numpy())
    compare_logits(lg.cpu().numpy(), ref)
    check_tokens(toks.cpu().numpy(), ref, 0.0, 0, 0, prompt_len - 1)
    dec.close()


@pytest.mark.parametrize("block", [0, 32])
@pytest.mark.parametrize("cfg", [
    ModelConfig("g2", 2, 512, 8, 4, 64, 1024, 3000),      # two query heads per KV head
    ModelConfig("g8", 2, 1024, 8, 1, 128, 1024, 3000),    # eight query heads per KV head, one KV head
])
def test_group_sizes(pm, cfg, block):
    _run(pm, cfg, 91, 90, 16, 128, block)


@pytest.mark.parametrize("cfg", [
    ModelConfig("wide-ffn", 1, 256, 4, 4, 64, 16384, 1000),   # h: 64 slices of 256
    ModelConfig("wide-d", 1, 16384, 4, 4, 64, 256, 1000),     # the residual stream: 64 slices
])
def test_longest_vectors(pm, cfg):
    _run(pm, cfg, 92, 20, 8, 32, 0)


@pytest.mark.parametrize("block", [0, 16])
def test_one_token_prompt(pm, block):
    _run(pm, MODELS["tiny"], 93, 1, 12, 16, block)


@pytest.mark.parametrize("block", [0, 16])
def test_cache_filled_to_its_last_position(pm, block):
    # prompt of 40 (39 prefilled positions) + 25 decode steps = 64 positions = max_seq
    _run(pm, MODELS["tiny"], 94, 40, 25, 64, block)
