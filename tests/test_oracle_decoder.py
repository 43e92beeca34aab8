"""Pins of the whole oracle decoder (CPU only): FP64 brute force on tiny
models, structural invariances and decode-call composition."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MODELS, ModelConfig, make_prompt, make_weights

TINYCFG = ModelConfig("t", 2, 16, 4, 2, 4, 24, 50)


def _w(cfg, seed, gains="random"):
    return {k: v.numpy() for k, v in make_weights(cfg, seed, gains=gains).items()}


def _brute_force_logits(cfg, w, tokens, window=None):
    """The decoder written out literally in float64 (K and V rounded to FP16
    on store), one position at a time; returns logits for every position.
    window[l] = W > 0: layer l attends to positions max(0, p-W+1) .. p only."""
    L, d, Hq, Hkv, hd, F = cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim
    f = {k: v.astype(np.float64) for k, v in w.items()}
    Kc = np.zeros((L, Hkv, len(tokens), hd))
    Vc = np.zeros((L, Hkv, len(tokens), hd))

    def norm(x, g):
        return x / math.sqrt(np.mean(x * x) + cfg.rms_eps) * g

    def rope(v, p):
        out = v.copy()
        for i in range(hd // 2):
            a = p * cfg.rope_theta ** (-2.0 * i / hd)
            out[i] = v[i] * math.cos(a) - v[i + hd // 2] * math.sin(a)
            out[i + hd // 2] = v[i + hd // 2] * math.cos(a) + v[i] * math.sin(a)
        return out

    all_logits = []
    for p, t in enumerate(tokens):
        x = f["embed"][t].copy()
        for l in range(L):
            xn = norm(x, f["attn_norm"][l])
            q = f["wq"][l] @ xn
            k = f["wk"][l] @ xn
            v = f["wv"][l] @ xn
            for g in range(Hkv):
                Kc[l, g, p] = rope(k[g * hd:(g + 1) * hd], p).astype(np.float16)
                Vc[l, g, p] = v[g * hd:(g + 1) * hd].astype(np.float16)
            att = np.zeros(Hq * hd)
            for h in range(Hq):
                g = h // (Hq // Hkv)
                qh = rope(q[h * hd:(h + 1) * hd], p)
                j0 = max(0, p + 1 - window[l]) if window is not None and window[l] > 0 else 0
                s = np.array([qh @ Kc[l, g, j] / math.sqrt(hd) for j in range(j0, p + 1)])
                e = np.exp(s - s.max())
                att[h * hd:(h + 1) * hd] = (e / e.sum()) @ Vc[l, g, j0:p + 1]
            x = x + f["wo"][l] @ att
            xn = norm(x, f["ffn_norm"][l])
            if getattr(cfg, "n_experts", 0):
                # mixture of experts: the top-k router logits (ties: lower index), softmax over them
                r = f["w_router"][l] @ xn
                sel = np.argsort(-r, kind="stable")[:cfg.top_k_experts]
                gw = np.exp(r[sel] - r[sel].max())
                gw = gw / gw.sum()
                for j, e in enumerate(sel):
                    gt = f["w_gate"][l, e] @ xn
                    x = x + gw[j] * (f["w_down"][l, e] @ ((gt / (1 + np.exp(-gt))) * (f["w_up"][l, e] @ xn)))
            else:
                gt = f["w_gate"][l] @ xn
                x = x + f["w_down"][l] @ ((gt / (1 + np.exp(-gt))) * (f["w_up"][l] @ xn))
        all_logits.append(f["lm_head"] @ norm(x, f["final_norm"]))
    return np.array(all_logits)


def _oracle_logits(cfg, w, tokens, max_seq=None, window=None):
    o = oracle.OracleDecoder(cfg, w, max_seq or len(tokens), layer_window=window)
    return np.array([o.forward(int(t)) for t in tokens])


@pytest.mark.parametrize("cfg", [TINYCFG, TINYCFG.with_(n_kv_heads=4, n_layers=1, head_dim=8, n_heads=4,
                                                          d_model=24, ffn_dim=40)])
def test_decoder_matches_float64_brute_force(cfg):
    w = _w(cfg, 11)
    # scale the weights up so that attention is far from uniform and RoPE matters
    for k in ("wq", "wk"):
        w[k] = (w[k].astype(np.float32) * 40).astype(np.float16)
    tokens = make_prompt(cfg.vocab, 9, 5).numpy()
    got = _oracle_logits(cfg, w, tokens)
    ref = _brute_force_logits(cfg, w, tokens)
    np.testing.assert_allclose(got, ref, atol=2e-4, rtol=0)


def test_gqa_equals_mha_with_shared_kv_heads():
    """A GQA model (contiguous groups: query head h reads KV head h // group)
    equals the MHA model whose K/V heads are copies of the group's KV head."""
    gqa = TINYCFG.with_(n_heads=4, n_kv_heads=2)
    mha = gqa.with_(n_kv_heads=4)
    w = _w(gqa, 12)
    wm = dict(w)
    hd = gqa.head_dim
    for name in ("wk", "wv"):
        rows = [w[name][:, (h // 2) * hd:(h // 2 + 1) * hd, :] for h in range(4)]
        wm[name] = np.ascontiguousarray(np.concatenate(rows, axis=1))
    tokens = make_prompt(gqa.vocab, 7, 6).numpy()
    np.testing.assert_array_equal(_oracle_logits(gqa, w, tokens), _oracle_logits(mha, wm, tokens))


def test_query_head_permutation_within_group_is_invariant():
    cfg = TINYCFG
    w = _w(cfg, 13)
    hd = cfg.head_dim
    perm = [1, 0, 3, 2]   # swap the two query heads inside each of the two groups
    wp = dict(w)
    wp["wq"] = np.ascontiguousarray(np.concatenate([w["wq"][:, h * hd:(h + 1) * hd, :] for h in perm], axis=1))
    wp["wo"] = np.ascontiguousarray(np.concatenate([w["wo"][:, :, h * hd:(h + 1) * hd] for h in perm], axis=2))
    tokens = make_prompt(cfg.vocab, 6, 7).numpy()
    a, b = _oracle_logits(cfg, w, tokens), _oracle_logits(cfg, wp, tokens)
    np.testing.assert_allclose(a, b, atol=1e-5)
    # swapping a query head across groups is NOT an invariance (it changes which KV head it reads)
    wx = dict(w)
    cross = [2, 1, 0, 3]
    wx["wq"] = np.ascontiguousarray(np.concatenate([w["wq"][:, h * hd:(h + 1) * hd, :] for h in cross], axis=1))
    wx["wo"] = np.ascontiguousarray(np.concatenate([w["wo"][:, :, h * hd:(h + 1) * hd] for h in cross], axis=2))
    assert np.max(np.abs(_oracle_logits(cfg, wx, tokens) - a)) > 1e-4


def test_zero_output_projections_make_every_layer_the_identity():
    cfg = MODELS["tiny"]
    w = _w(cfg, 14)
    w["wo"] = np.zeros_like(w["wo"])
    w["w_down"] = np.zeros_like(w["w_down"])
    tokens = make_prompt(cfg.vocab, 5, 8).numpy()
    got = _oracle_logits(cfg, w, tokens)
    E, H, g = (w[k].astype(np.float64) for k in ("embed", "lm_head", "final_norm"))
    for p, t in enumerate(tokens):
        x = E[t]
        ref = H @ (x / math.sqrt(np.mean(x * x) + cfg.rms_eps) * g)
        np.testing.assert_allclose(got[p], ref, atol=2e-5)


def test_first_position_cache_holds_unrotated_fp16_k_and_v():
    cfg = MODELS["tiny"]
    w = _w(cfg, 15)
    o = oracle.OracleDecoder(cfg, w, 4)
    t = 321
    o.forward(t, want_logits=False)
    K, V = o.kv_cache()
    x = w["embed"][t].astype(np.float64)
    xn = x / math.sqrt(np.mean(x * x) + cfg.rms_eps) * w["attn_norm"][0].astype(np.float64)
    k = (w["wk"][0].astype(np.float64) @ xn).reshape(cfg.n_kv_heads, cfg.head_dim)
    v = (w["wv"][0].astype(np.float64) @ xn).reshape(cfg.n_kv_heads, cfg.head_dim)
    np.testing.assert_allclose(K[0, :, 0].astype(np.float64), k, rtol=1e-3, atol=1e-5)
    np.testing.assert_allclose(V[0, :, 0].astype(np.float64), v, rtol=1e-3, atol=1e-5)
    assert np.all(K[:, :, 1:] == 0) and np.all(V[:, :, 1:] == 0)


@pytest.mark.parametrize("T,k", [(0.0, 0), (0.9, 20), (1.3, 0)])
def test_decode_calls_compose(T, k):
    cfg = MODELS["tiny"]
    w = _w(cfg, 0, gains="ones")
    prompt = make_prompt(cfg.vocab, 16, 1000).numpy()
    a = oracle.OracleDecoder(cfg, w, 64)
    a.prefill(prompt)
    t_all, l_all = a.decode(24, T, k, 555)
    b = oracle.OracleDecoder(cfg, w, 64)
    b.prefill(prompt)
    t1, l1 = b.decode(10, T, k, 555)
    t2, l2 = b.decode(14, T, k, 555)
    assert np.array_equal(t_all, np.concatenate([t1, t2]))
    assert np.array_equal(l_all, np.concatenate([l1, l2]))


def test_prefill_then_forced_decode_equals_step_by_step_forward():
    cfg = MODELS["tiny"]
    w = _w(cfg, 0, gains="ones")
    seq = make_prompt(cfg.vocab, 30, 4).numpy()
    a = oracle.OracleDecoder(cfg, w, 40)
    a.prefill(seq[:10])
    toks, lg = a.decode(20, force_tokens=seq[10:30])
    b = oracle.OracleDecoder(cfg, w, 40)
    ref = np.array([b.forward(int(t)) for t in seq[:30]])
    np.testing.assert_array_equal(lg, ref[9:29])
    np.testing.assert_array_equal(toks, ref[9:29].argmax(axis=1))


def test_capacity_and_argument_errors():
    cfg = MODELS["tiny"]
    w = _w(cfg, 0, gains="ones")
    o = oracle.OracleDecoder(cfg, w, 8)
    with pytest.raises(ValueError):
        o.decode(1)                       # nothing pending
    o.prefill(np.arange(4, dtype=np.int32))
    o.decode(4)                           # positions 3..6
    with pytest.raises(ValueError):
        o.decode(2)                       # would need positions 7..8
    with pytest.raises(ValueError):
        o.prefill(np.arange(9, dtype=np.int32))


def test_synthetic_weights_are_device_independent_and_normal():
    cfg = MODELS["tiny"]
    a = make_weights(cfg, 5)
    b = make_weights(cfg, 5)
    assert all(torch.equal(a[k], b[k]) for k in a)
    assert not torch.equal(a["wq"][0], a["wq"][1])
    x = a["w_up"].float().flatten().numpy()
    assert abs(x.std() - 0.02) < 2e-4 and abs(x.mean()) < 2e-4
    from scipy import stats
    assert stats.kstest(x[::37] / 0.02, "norm").pvalue > 1e-3


# ---- sliding-window attention (shivam2003.com, "Why GQA and sliding windows")

@pytest.mark.parametrize("window", [[3, 0], [1, 4], [2, 2]])
def test_sliding_window_matches_float64_brute_force(window):
    cfg = TINYCFG
    w = _w(cfg, 12)
    for k in ("wq", "wk"):
        w[k] = (w[k].astype(np.float32) * 40).astype(np.float16)
    tokens = make_prompt(cfg.vocab, 10, 6).numpy()
    got = _oracle_logits(cfg, w, tokens, window=window)
    ref = _brute_force_logits(cfg, w, tokens, window=window)
    np.testing.assert_allclose(got, ref, atol=2e-4, rtol=0)
    # and the window does change the result once the context outgrows it
    full = _brute_force_logits(cfg, w, tokens)
    assert np.abs(full[-1] - ref[-1]).max() > 1e-3


def test_window_covering_the_context_changes_nothing():
    cfg = TINYCFG
    w = _w(cfg, 13)
    tokens = make_prompt(cfg.vocab, 8, 7).numpy()
    np.testing.assert_array_equal(_oracle_logits(cfg, w, tokens, window=[8, 100]), _oracle_logits(cfg, w, tokens))


def test_window_of_one_makes_every_position_see_only_itself():
    """With W = 1 everywhere, attention returns the current position's V row
    (one softmax weight of exactly 1), and the query-key rotations cancel, so
    a token's logits no longer depend on its position or on earlier tokens."""
    cfg = TINYCFG
    w = _w(cfg, 14)
    o = oracle.OracleDecoder(cfg, w, 16, layer_window=[1, 1])
    first = o.forward(7)
    for t in (3, 9, 1):
        o.forward(t)
    again = o.forward(7)
    np.testing.assert_array_equal(first, again)


@pytest.mark.parametrize("block", [1, 3, 8, 13, 64])
@pytest.mark.parametrize("window", [None, (5, 0)])
def test_blocked_prefill_equals_position_by_position_prefill(block, window):
    """orc_prefill_blocked only reorders independent positions: its KV cache
    and the logits of the following decode steps equal orc_prefill's bit for
    bit, with a pending token carried over between two prefill calls, a block
    that does not divide the prompt, and sliding windows."""
    cfg = TINYCFG.with_(n_heads=4, n_kv_heads=2, head_dim=8, d_model=32, ffn_dim=48)
    w = _w(cfg, 21)
    for k in ("wq", "wk"):
        w[k] = (w[k].astype(np.float32) * 30).astype(np.float16)
    seq = make_prompt(cfg.vocab, 40, 8).numpy()
    a = oracle.OracleDecoder(cfg, w, 48, layer_window=window)
    b = oracle.OracleDecoder(cfg, w, 48, layer_window=window)
    a.prefill(seq[:11])
    a.prefill(seq[11:30])
    b.prefill_blocked(seq[:11], block)
    b.prefill_blocked(seq[11:30], block)
    assert a.pos == b.pos == 29 and a.pending == b.pending == int(seq[29])
    ka, va = a.kv_cache()
    kb, vb = b.kv_cache()
    assert np.array_equal(ka.view(np.uint16), kb.view(np.uint16))
    assert np.array_equal(va.view(np.uint16), vb.view(np.uint16))
    ta, la = a.decode(6, force_tokens=seq[30:36])
    tb, lb = b.decode(6, force_tokens=seq[30:36])
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))
    assert np.array_equal(ta, tb)


def test_blocked_prefill_rejects_what_it_does_not_cover():
    cfg = MODELS["tiny"]
    w = _w(cfg, 0, gains="ones")
    o = oracle.OracleDecoder(cfg, w, 8)
    with pytest.raises(ValueError):
        o.prefill_blocked(np.arange(9, dtype=np.int32), 4)    # cache too small
    with pytest.raises(ValueError):
        o.prefill_blocked(np.array([1, cfg.vocab], dtype=np.int32), 4)   # bad token id
    with pytest.raises(ValueError):
        o.prefill_blocked(np.arange(4, dtype=np.int32), 0)    # empty block


def test_skip_to_is_a_timing_hook_only():
    """orc_skip_to moves the pending token to a position without running the
    passes before it; at position 0 that is exactly a one-token prefill, and
    positions outside the cache are refused."""
    cfg = MODELS["tiny"]
    w = _w(cfg, 0, gains="ones")
    a = oracle.OracleDecoder(cfg, w, 16)
    a.prefill(np.array([7], dtype=np.int32))
    ta, la = a.decode(3)
    b = oracle.OracleDecoder(cfg, w, 16)
    b.skip_to(0, 7)
    tb, lb = b.decode(3)
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32)) and np.array_equal(ta, tb)
    c = oracle.OracleDecoder(cfg, w, 16)
    c.skip_to(12, 3)
    assert c.pos == 12 and c.pending == 3
    c.decode(4)                            # positions 12 .. 15
    with pytest.raises(ValueError):
        c.skip_to(16, 3)
    with pytest.raises(ValueError):
        c.skip_to(0, cfg.vocab)
