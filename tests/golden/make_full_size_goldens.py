"""Write the oracle's logits and tokens for the decode workloads at their full
prompt lengths, for the GPU parity tests (tests/test_gpu_full_size.py).

    python tests/golden/make_full_size_goldens.py [case ...]

Cases (every input seeded and synthetic, see synthetic/):
  2p3b_p512      the ~2.3B decoder, 512-token prompt, 16 greedy steps
  8b_p2048       the 8B-shaped decoder, 2,048-token prompt, 8 steps sampled at
                 temperature 0.8, top-k 50, Philox seed 1234
  attn2l_p32768  two layers with the ~2.3B's attention shape (d_model 2560,
                 20 query / 5 KV heads x 128), a 32,768-token prompt, 16 greedy
                 steps: the long-context attention of the 32k workload (30
                 split-KV pieces of ~1,092 positions per KV head on 152 CTAs)
                 at a size the CPU oracle can follow

Only oracle/ computes anything here; synthetic/ supplies the weights and
prompt ids.  The oracle prefills the prompt with orc_prefill_blocked (the
same forward passes as orc_prefill, bit for bit, visited a block of positions
at a time), then decodes free-running: greedy steps take its own argmax,
sampled steps its own Gumbel-max choice.  Each case is stored as
tests/golden/<case>.npz: the prompt, the oracle's tokens, the logits of every
step (FP32) and the settings.
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from synthetic import MODELS, WORKLOADS, make_prompt, make_weights  # noqa: E402

# name: (model, weight seed, prompt seed, prompt length, decode steps, temperature, top_k, sample seed)
CASES = {
    "2p3b_p512": ("2.3b", WORKLOADS["2.3b"].weight_seed, WORKLOADS["2.3b"].prompt_seed, 512, 16, 0.0, 0, 0),
    "8b_p2048": ("8b", WORKLOADS["8b"].weight_seed, WORKLOADS["8b"].prompt_seed, 2048, 8, 0.8, 50, 1234),
    "attn2l_p32768": ("attn-2l", 5, 1003, 32768, 16, 0.0, 0, 0),
}
BLOCK = 128


def path_of(case: str) -> str:
    return os.path.join(HERE, case + ".npz")


def make(case: str) -> None:
    model, wseed, pseed, n_prompt, n_steps, temp, top_k, sseed = CASES[case]
    cfg = MODELS[model]
    t0 = time.time()
    w = {k: v.numpy() for k, v in make_weights(cfg, wseed, device="cpu").items()}
    prompt = make_prompt(cfg.vocab, n_prompt, pseed).numpy().astype(np.int32)
    orc = oracle.OracleDecoder(cfg, w, n_prompt + n_steps)
    orc.prefill_blocked(prompt, BLOCK)
    t1 = time.time()
    toks, lg = orc.decode(n_steps, temp, top_k, sseed)
    t2 = time.time()
    np.savez(path_of(case), prompt=prompt, tokens=toks.astype(np.int32), logits=lg.astype(np.float32),
             model=model, weight_seed=wseed, prompt_seed=pseed, temperature=np.float32(temp), top_k=top_k,
             sample_seed=np.uint64(sseed), first_pos=n_prompt - 1)
    print(f"{case}: prefill {t1 - t0:.0f} s, {n_steps} steps {t2 - t1:.0f} s, {oracle.num_threads()} threads, "
          f"tokens {toks.tolist()}", flush=True)


if __name__ == "__main__":
    for c in (sys.argv[1:] or list(CASES)):
        make(c)
