"""Full-size parity: the CUDA path against the oracle at each decode workload's
stated prompt length (needs a GB300).

The oracle cannot follow a 2,048- or 32,768-token prompt inside a test, so its
logits and tokens are stored (tests/golden/<case>.npz, written by
tests/golden/make_full_size_goldens.py, which calls only the oracle).  The GPU
prefills the same seeded prompt, then decodes with the oracle's tokens fed
back (teacher forcing), so every step's logits are compared on the oracle's
own prefix: logits max-abs <= 2e-2 and RMS <= 2e-3, the GPU's own token equal
to the oracle's wherever the oracle's margin exceeds 0.05.
"""
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN, cuda_available
from parity import check_tokens, compare_logits
from synthetic import MODELS, make_prompt, make_weights

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    from persistent_monokernel_gb300 import build
    build.build()
    return pm


def _golden(case):
    path = os.path.join(GOLDEN, case + ".npz")
    if not os.path.exists(path):
        pytest.skip(f"{case}.npz not generated")
    return np.load(path)


_WEIGHTS = {}


def _weights(model, seed):
    key = (model.name, seed)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()
        torch.cuda.empty_cache()
        _WEIGHTS[key] = make_weights(model, seed, device="cuda")
    return _WEIGHTS[key]


def _run(pm, case, prefill_block):
    g = _golden(case)
    model = MODELS[str(g["model"])]
    prompt = make_prompt(model.vocab, g["prompt"].size, int(g["prompt_seed"]))
    assert np.array_equal(prompt.numpy(), g["prompt"]), "the seeded prompt generator changed"
    ref_tokens, ref = g["tokens"], g["logits"]
    n = ref_tokens.size
    T, top_k, seed = float(g["temperature"]), int(g["top_k"]), int(g["sample_seed"])
    w = _weights(model, int(g["weight_seed"]))
    dec = pm.Decoder(model, w, prompt.numel() + n, prefill_block=prefill_block)
    try:
        dec.prefill(prompt.cuda())
        lg = torch.empty((n, model.vocab), dtype=torch.float32, device="cuda")
        force = torch.from_numpy(ref_tokens.astype(np.int32)).cuda()
        toks = dec.decode(n, temperature=T, top_k=top_k, seed=seed, debug_logits=lg, force_tokens=force)
        assert dec.sync() == 0
    finally:
        torch.cuda.synchronize()
        dec.close()
    max_abs, rms = compare_logits(lg.cpu().numpy(), ref)
    exact = check_tokens(toks.cpu().numpy(), ref, T, top_k, seed, int(g["first_pos"]))
    assert exact >= n // 2, f"only {exact} of {n} steps had a decisive oracle margin"
    return max_abs, rms


@pytest.mark.parametrize("prefill_block", [0, 1024])
def test_2p3b_at_its_512_token_prompt(pm, prefill_block):
    """The ~2.3B decoder (25 layers, d_model 2560, 20/5 heads x 128), 511
    prompt positions then 16 greedy steps, with the prompt run as monokernel
    steps and as the batched prefill."""
    _run(pm, "2p3b_p512", prefill_block)


@pytest.mark.parametrize("prefill_block", [0, 1024])
def test_8b_at_its_2048_token_prompt_sampled(pm, prefill_block):
    """The 8B-shaped decoder after 2,047 prompt positions, 8 steps sampled in
    the kernel at temperature 0.8, top-k 50, Philox seed 1234."""
    _run(pm, "8b_p2048", prefill_block)


@pytest.mark.parametrize("prefill_block", [1024, 4096])
def test_32k_context_attention_shape(pm, prefill_block):
    """Two layers with the ~2.3B's attention shape after a 32,768-token prompt:
    every KV head's 32,768 positions split over 30 pieces of ~1,092 on 152
    CTAs, K/V streamed past L2 (84 MB per layer at full depth)."""
    _run(pm, "attn2l_p32768", prefill_block)
