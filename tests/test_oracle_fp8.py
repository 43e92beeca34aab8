"""Pins of the oracle's weight-only FP8 path (CPU only): the E4M3 decode
against its format definition and an independent library cast, the scaled
matvec against an FP64 brute force, and the whole FP8 decoder against the
already pinned FP16 decoder on weights both formats represent exactly."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import FP8_MATRICES, MODELS, ModelConfig, make_prompt, make_weights, make_weights_fp8
from test_oracle_decoder import _brute_force_logits

TINYCFG = ModelConfig("t", 2, 16, 4, 2, 4, 24, 50)


def test_e4m3_decode_matches_torch_float8_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle.e4m3_to_float(int(c)) for c in range(256)], dtype=np.float32)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(nan, np.isnan(got))   # S.1111.111 only
    np.testing.assert_array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("code,value", [(0x00, 0.0), (0x80, -0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),
                                        (0x08, 2.0 ** -6), (0x38, 1.0), (0xB8, -1.0), (0x3C, 1.5),
                                        (0x7E, 448.0), (0xFE, -448.0), (0x40, 2.0)])
def test_e4m3_closed_forms(code, value):
    got = oracle.e4m3_to_float(code)
    assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value)


def test_fp8_matvec_exact_on_integers_and_within_the_fp32_bound():
    rng = np.random.default_rng(3)
    # codes 0x38..0x50 decode to small integers and halves; scale 1, integer x: every sum is exact
    C = rng.integers(0x38, 0x51, size=(7, 40)).astype(np.uint8)
    x = rng.integers(-3, 4, size=40).astype(np.float32)
    dec = np.vectorize(oracle.e4m3_to_float)(C).astype(np.float64)
    np.testing.assert_array_equal(oracle.matvec_fp8(C, np.ones(7, np.float32), x), (dec @ x).astype(np.float32))
    # random codes and scales: within the FP32 summation bound of the FP64 result
    C = rng.integers(0, 256, size=(9, 300)).astype(np.uint8)
    C[(C & 0x7F) == 0x7F] = 0x10                          # no NaN codes
    s = rng.uniform(1e-4, 1e-2, size=9).astype(np.float32)
    x = rng.standard_normal(300).astype(np.float32)
    dec = np.vectorize(oracle.e4m3_to_float)(C).astype(np.float64)
    ref = s.astype(np.float64) * (dec @ x.astype(np.float64))
    bound = 300 * 2.0 ** -24 * s * (np.abs(dec) @ np.abs(x)) * 2 + 1e-30
    assert np.all(np.abs(oracle.matvec_fp8(C, s, x) - ref) <= bound)


def _pow2_fp8_model(cfg, seed):
    """FP8 weights whose per-row scales are powers of two (2^-9..2^-11, by row),
    and the FP16 weights decode(codes) * scale, which FP16 holds exactly."""
    w8 = make_weights_fp8(cfg, seed)
    w16 = make_weights(cfg, seed, projections=False)
    for n in FP8_MATRICES:
        sc = w8[n + "_scale"]
        k = torch.arange(sc.numel()).view(sc.shape) % 3
        w8[n + "_scale"] = torch.pow(2.0, -(9 + k).to(torch.float32))
        dec = w8[n].view(torch.float8_e4m3fn).to(torch.float32)
        w16[n] = (dec * w8[n + "_scale"].unsqueeze(-1)).to(torch.float16)
        assert torch.equal(w16[n].to(torch.float32), dec * w8[n + "_scale"].unsqueeze(-1))
    return w8, w16


def test_fp8_decoder_equals_the_fp16_decoder_on_exactly_representable_weights():
    """Scaling by a power of two commutes with FP32 rounding, so decode(C)
    times a power-of-two row scale gives the FP16 path's sums bit for bit: a
    wrong matrix, row or layer of scales shows up as a difference."""
    cfg = MODELS["tiny"]
    w8, w16 = _pow2_fp8_model(cfg, 5)
    tokens = make_prompt(cfg.vocab, 6, 8).numpy()
    o8 = oracle.OracleDecoder(cfg, w8, 8)
    o16 = oracle.OracleDecoder(cfg, w16, 8)
    for t in tokens:
        np.testing.assert_array_equal(o8.forward(int(t)), o16.forward(int(t)))


def test_fp8_decoder_matches_float64_brute_force():
    cfg = TINYCFG
    w8 = make_weights_fp8(cfg, 21, gains="random")
    deq = {k: v.numpy() for k, v in w8.items() if not k.endswith("_scale")}
    for n in FP8_MATRICES:
        dec = w8[n].view(torch.float8_e4m3fn).to(torch.float64)
        deq[n] = (dec * w8[n + "_scale"].to(torch.float64).unsqueeze(-1)).numpy()
    tokens = make_prompt(cfg.vocab, 9, 22).numpy()
    o = oracle.OracleDecoder(cfg, w8, 9)
    got = np.array([o.forward(int(t)) for t in tokens])
    ref = _brute_force_logits(cfg, deq, tokens)
    np.testing.assert_allclose(got, ref, atol=2e-4, rtol=0)
