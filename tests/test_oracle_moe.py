"""Pins of the oracle's mixture-of-experts FFN (CPU only): the routing rule on
hand-worked cases, the one-expert model against the pinned dense decoder, a
model whose experts are all equal against the dense decoder, and the whole
decoder against an FP64 brute force."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MODELS, ModelConfig, make_prompt, make_weights
from test_oracle_decoder import _brute_force_logits

MOECFG = ModelConfig("m", 2, 64, 4, 2, 16, 96, 50, n_experts=6, top_k_experts=2)


@pytest.mark.parametrize("logits,k,sel,gates", [
    ([1.0, 3.0, 2.0, 3.0], 2, [1, 3], [0.5, 0.5]),             # a tie: the lower index first
    ([1.0, 3.0, 2.0, 3.0], 3, [1, 3, 2], None),
    ([0.0, math.log(3.0)], 2, [1, 0], [0.75, 0.25]),            # softmax over the chosen logits
    ([5.0, -1.0, 7.0], 1, [2], [1.0]),                         # top-1: gate exactly 1
    ([-2.0, -2.0, -2.0], 2, [0, 1], [0.5, 0.5]),
])
def test_route_hand_worked_cases(logits, k, sel, gates):
    s, g = oracle.route(np.array(logits, dtype=np.float32), k)
    assert list(s) == sel
    if gates is not None:
        np.testing.assert_allclose(g, gates, rtol=1e-6, atol=0)
    assert abs(float(np.sum(g)) - 1.0) < 1e-6


def _dense_view(cfg_moe, w, expert):
    """The dense model whose FFN is expert `expert` of every layer."""
    cfg = cfg_moe.with_(n_experts=0, top_k_experts=0)
    wd = {k: v for k, v in w.items() if k != "w_router"}
    for n in ("w_gate", "w_up", "w_down"):
        wd[n] = w[n][:, expert].contiguous()
    return cfg, wd


def test_one_expert_top_one_equals_the_dense_decoder_bitwise():
    cfg = MOECFG.with_(n_experts=1, top_k_experts=1)
    w = make_weights(cfg, 3, gains="random")
    cfg_d, wd = _dense_view(cfg, w, 0)
    tokens = make_prompt(cfg.vocab, 7, 4).numpy()
    om = oracle.OracleDecoder(cfg, w, 8)
    od = oracle.OracleDecoder(cfg_d, wd, 8)
    for t in tokens:
        np.testing.assert_array_equal(om.forward(int(t)), od.forward(int(t)))


def test_equal_experts_give_the_dense_decoder():
    """Gates sum to one, so k copies of the same expert reproduce it (to FP32
    rounding of the weighted sum): a wrong gate, a gate applied twice or an
    expert dropped shows up."""
    cfg = MOECFG
    w = make_weights(cfg, 5, gains="random")
    for n in ("w_gate", "w_up", "w_down"):
        w[n] = w[n][:, :1].expand(-1, cfg.n_experts, -1, -1).contiguous()
    cfg_d, wd = _dense_view(cfg, w, 0)
    tokens = make_prompt(cfg.vocab, 6, 6).numpy()
    om = oracle.OracleDecoder(cfg, w, 8)
    od = oracle.OracleDecoder(cfg_d, wd, 8)
    for t in tokens:
        np.testing.assert_allclose(om.forward(int(t)), od.forward(int(t)), atol=2e-6, rtol=0)


def test_moe_decoder_matches_float64_brute_force():
    cfg = MOECFG
    w = make_weights(cfg, 7, gains="random")
    wn = {k: v.numpy() for k, v in w.items()}
    tokens = make_prompt(cfg.vocab, 9, 8).numpy()
    o = oracle.OracleDecoder(cfg, w, 9)
    got = np.array([o.forward(int(t)) for t in tokens])
    ref = _brute_force_logits(cfg, wn, tokens)
    np.testing.assert_allclose(got, ref, atol=2e-4, rtol=0)


def test_moe_routing_uses_more_than_one_expert_pair():
    """The synthetic router spreads tokens over experts (so the tests above
    exercise several expert choices)."""
    cfg = MOECFG
    w = make_weights(cfg, 7, gains="random")
    wr = w["w_router"].to(torch.float32).numpy()
    xs = np.random.default_rng(0).standard_normal((40, cfg.d_model)).astype(np.float32)
    pairs = {tuple(oracle.route(wr[0] @ x, 2)[0]) for x in xs}
    assert len(pairs) > 5
