"""Pins of the oracle's MXFP4 path (CPU only): the E2M1 element and E8M0
scale decodes against the format's value table, the packed-nibble order, the
block-scaled matvec against an FP64 brute force, and the whole MXFP4 decoder
against the already pinned FP16 decoder on the same (exactly representable)
weights."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import FP8_MATRICES, MODELS, ModelConfig, make_prompt, make_weights, make_weights_mxfp4
from test_oracle_decoder import _brute_force_logits

TINYCFG = ModelConfig("t", 2, 64, 4, 2, 16, 96, 50)

# OCP Microscaling formats, E2M1 element encodings 0000 .. 1111
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_decode_matches_the_format_table():
    for code, value in enumerate(E2M1_TABLE):
        got = oracle.e2m1_to_float(code)
        assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value), code


@pytest.mark.parametrize("code,value", [(127, 1.0), (128, 2.0), (126, 0.5), (120, 2.0 ** -7), (0, 2.0 ** -127),
                                        (254, 2.0 ** 127), (1, 2.0 ** -126)])
def test_e8m0_closed_forms(code, value):
    assert oracle.e8m0_to_float(code) == value


def test_e8m0_255_is_nan():
    assert math.isnan(oracle.e8m0_to_float(255))


def _decode_f64(codes, scales):
    """Independent decode: lookup of each nibble in the value table times 2^(E - 127)."""
    tab = np.array(E2M1_TABLE, dtype=np.float64)
    lo = tab[codes & 15]
    hi = tab[codes >> 4]
    el = np.empty(codes.shape[:-1] + (2 * codes.shape[-1],), dtype=np.float64)
    el[..., 0::2] = lo
    el[..., 1::2] = hi
    sc = np.ldexp(1.0, scales.astype(np.int64) - 127)
    return el * np.repeat(sc, 32, axis=-1)


def test_packed_element_order_low_nibble_first():
    # row 0: element 0 = 1.0 (code 2), element 1 = -6.0 (code 15); scale 2^0
    codes = np.zeros((1, 16), dtype=np.uint8)
    codes[0, 0] = 2 | (15 << 4)
    scales = np.full((1, 1), 127, dtype=np.uint8)
    x = np.zeros(32, dtype=np.float32)
    x[0] = 1.0
    assert oracle.matvec_mxfp4(codes, scales, x)[0] == 1.0
    x[:] = 0.0
    x[1] = 1.0
    assert oracle.matvec_mxfp4(codes, scales, x)[0] == -6.0
    # the second block of a row uses the second scale byte
    codes = np.zeros((1, 32), dtype=np.uint8)
    codes[0, 16] = 2                      # element 32 = 1.0
    scales = np.array([[127, 130]], dtype=np.uint8)
    x = np.zeros(64, dtype=np.float32)
    x[32] = 1.0
    assert oracle.matvec_mxfp4(codes, scales, x)[0] == 8.0


def test_mxfp4_matvec_matches_float64_brute_force():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, size=(13, 96)).astype(np.uint8)        # 192 columns
    scales = rng.integers(110, 140, size=(13, 6)).astype(np.uint8)
    x = rng.standard_normal(192).astype(np.float32)
    W = _decode_f64(codes, scales)
    ref = W @ x.astype(np.float64)
    bound = 192 * 2.0 ** -24 * (np.abs(W) @ np.abs(x)) * 2 + 1e-30
    got = oracle.matvec_mxfp4(codes, scales, x)
    assert np.all(np.abs(got - ref) <= bound)
    # integer inputs with small scales: every partial sum is exact
    xi = rng.integers(-3, 4, size=192).astype(np.float32)
    s1 = np.full((13, 6), 127, dtype=np.uint8)
    np.testing.assert_array_equal(oracle.matvec_mxfp4(codes, s1, xi),
                                  (_decode_f64(codes, s1) @ xi.astype(np.float64)).astype(np.float32))


def _as_fp16_model(cfg, w4):
    """The FP16 decoder whose projections are the decoded MXFP4 weights (every
    one of them is exactly an FP16 value at these scales)."""
    w16 = make_weights(cfg, 0, projections=False)
    for k in ("embed", "attn_norm", "ffn_norm", "final_norm"):
        w16[k] = w4[k]
    for n in FP8_MATRICES:
        dec = _decode_f64(w4[n].numpy(), w4[n + "_scale"].numpy())
        t = torch.from_numpy(dec).to(torch.float16)
        assert np.array_equal(t.to(torch.float64).numpy(), dec)
        w16[n] = t
    return w16


def test_mxfp4_decoder_equals_the_fp16_decoder_on_the_decoded_weights():
    """decode(C, S) is exact in FP32 and in FP16 here, so both decoders form
    the same products in the same order: a wrong nibble, block, row, matrix or
    layer of scales shows up as a difference."""
    cfg = MODELS["tiny"]
    w4 = make_weights_mxfp4(cfg, 7, gains="random")
    w16 = _as_fp16_model(cfg, w4)
    tokens = make_prompt(cfg.vocab, 6, 9).numpy()
    o4 = oracle.OracleDecoder(cfg, w4, 8)
    o16 = oracle.OracleDecoder(cfg, w16, 8)
    assert o4.mxfp4 and not o4.fp8
    for t in tokens:
        np.testing.assert_array_equal(o4.forward(int(t)), o16.forward(int(t)))


def test_mxfp4_decoder_matches_float64_brute_force():
    cfg = TINYCFG
    w4 = make_weights_mxfp4(cfg, 23, gains="random")
    deq = {k: v.numpy() for k, v in w4.items() if not k.endswith("_scale")}
    for n in FP8_MATRICES:
        deq[n] = _decode_f64(w4[n].numpy(), w4[n + "_scale"].numpy())
    tokens = make_prompt(cfg.vocab, 9, 24).numpy()
    o = oracle.OracleDecoder(cfg, w4, 9)
    got = np.array([o.forward(int(t)) for t in tokens])
    ref = _brute_force_logits(cfg, deq, tokens)
    np.testing.assert_allclose(got, ref, atol=2e-4, rtol=0)
