"""Helpers for GPU-vs-oracle parity tests.

Tolerances (from the decode workload definitions): logits max-abs error <= 2e-2
and RMS error <= 2e-3 against the oracle on the same inputs; the chosen token
must equal the oracle's wherever the oracle's decision margin exceeds 0.05,
and otherwise be one of the tokens within 0.05 of the best.
"""
import numpy as np

import oracle

LOGIT_MAX_ABS = 2e-2
LOGIT_RMS = 2e-3
MARGIN = 0.05


def compare_logits(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape
    err = gpu - ref
    max_abs = float(np.max(np.abs(err)))
    rms = float(np.sqrt(np.mean(err * err)))
    assert max_abs <= LOGIT_MAX_ABS, f"logit max-abs error {max_abs:.3g} > {LOGIT_MAX_ABS}"
    assert rms <= LOGIT_RMS, f"logit RMS error {rms:.3g} > {LOGIT_RMS}"
    return max_abs, rms


def decision(ref_logits, temperature, top_k, seed, pos):
    """Oracle's view of one step: (token, margin, acceptable set).

    Greedy: margin = top1 - top2 logit.  Sampled: scores s_i = logit_i/T + g_i
    over the top-k set S; margin = top1 - top2 score in S, set to 0 when a
    logit error of MARGIN could change S in a way that matters (the winner
    near the top-k boundary, or a token just outside S whose score is close
    to the winner's)."""
    lg = np.asarray(ref_logits, dtype=np.float32)
    V = lg.size
    order = np.argsort(-lg.astype(np.float64), kind="stable")
    greedy = not (temperature > 0) or top_k == 1
    if greedy:
        best = int(order[0])
        margin = float(lg[order[0]]) - float(lg[order[1]]) if V > 1 else np.inf
        ok = set(int(i) for i in np.nonzero(lg >= lg[best] - MARGIN)[0])
        return best, margin, ok
    k = V if (top_k <= 0 or top_k >= V) else top_k
    T = np.float32(temperature)
    # candidates: S plus every token within MARGIN of the boundary logit
    lk = lg[order[k - 1]]
    cand = np.nonzero(lg >= lk - MARGIN)[0] if k < V else np.arange(V)
    g = np.array([oracle.gumbel(seed, pos, int(i)) for i in cand], dtype=np.float32)
    sc = lg[cand] / T + g
    in_s = np.isin(cand, order[:k])
    s_scores = np.where(in_s, sc, -np.inf)
    j = int(np.argmax(s_scores))            # argmax picks the first maximum = lowest index (cand is sorted)
    best, best_sc = int(cand[j]), float(sc[j])
    others = np.delete(s_scores, j)
    margin = best_sc - float(np.max(others)) if others.size and np.isfinite(np.max(others)) else np.inf
    if k < V:
        lk1 = lg[order[k]]
        if lg[best] - lk1 <= MARGIN:
            margin = 0.0                     # the winner could drop out of S
        out_near = (~in_s) & (sc >= best_sc - MARGIN)
        if np.any(out_near):
            margin = 0.0                     # an outsider could enter S and win
    # acceptable when ambiguous: a token that can win for some top-k set allowed by
    # logit errors up to MARGIN, i.e. one whose score is within MARGIN of the best
    # score among the members that stay in S under any such error
    sure = in_s & ((lg[cand] - lg[order[k]] > MARGIN) if k < V else True)
    floor = float(np.max(sc[sure])) if np.any(sure) else -np.inf
    ok = set(int(i) for i in cand[sc >= floor - MARGIN])
    ok.add(best)
    return best, margin, ok


def check_tokens(gpu_tokens, ref_logits, temperature, top_k, seed, pos0):
    """Every step: exact where the margin exceeds MARGIN, acceptable otherwise.
    Returns the number of steps checked exactly."""
    exact = 0
    for i, t in enumerate(np.asarray(gpu_tokens)):
        best, margin, ok = decision(ref_logits[i], temperature, top_k, seed, pos0 + i)
        if margin > MARGIN:
            assert int(t) == best, f"step {i}: token {int(t)} != oracle {best} (margin {margin:.3f})"
            exact += 1
        else:
            assert int(t) in ok, f"step {i}: token {int(t)} not within tolerance of the oracle's choice {best}"
    return exact
