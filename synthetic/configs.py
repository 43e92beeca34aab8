"""Workload shapes: Llama-style decoder-only transformers decoded at batch 1.

The five workloads are the decode configurations this library is measured on:
a tiny and a small decoder, a ~2.3B-parameter decoder at short and at 32k
context, and an 8B-shaped decoder sampled at temperature 0.8 / top-k 50.
The ~2.3B size is the one the KOG LaneFormer write-up (shivam2003.com,
"A worked bandwidth ceiling") quotes: 2.3B FP16 parameters, 4.6 GB streamed
per token.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_theta: float = 10000.0
    rms_eps: float = 1e-5
    # mixture of experts: n_experts FFNs of ffn_dim per layer, top_k_experts of
    # them active per token (0: the dense FFN)
    n_experts: int = 0
    top_k_experts: int = 0

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def n_params(self) -> int:
        L, d, F, V = self.n_layers, self.d_model, self.ffn_dim, self.vocab
        ffn = 3 * d * F if not self.n_experts else self.n_experts * (3 * d * F + d)
        per_layer = (self.q_dim + 2 * self.kv_dim) * d + d * self.q_dim + ffn + 2 * d
        return V * d * 2 + L * per_layer + d

    def active_ffn_weights(self) -> int:
        """FFN weights one token uses in one layer: the dense FFN, or the
        router and the top_k_experts active experts."""
        d, F = self.d_model, self.ffn_dim
        if not self.n_experts:
            return 3 * d * F
        return self.n_experts * d + self.top_k_experts * 3 * d * F

    def weight_bytes_per_token(self, weights: str = "fp16") -> int:
        """Bytes every decode step must stream: all layer matrices and norm
        gains, the final norm, the LM head and one embedding row.  FP16
        throughout, or the eight projection matrices as ("fp8") one byte per
        weight plus one FP32 scale per row, or ("mxfp4") half a byte per
        weight plus one scale byte per 32 weights (embedding and gains stay
        FP16)."""
        L, d, F, V = self.n_layers, self.d_model, self.ffn_dim, self.vocab
        Q, KV = self.q_dim, self.kv_dim
        if weights == "fp16":
            per_layer = (Q + 2 * KV) * d + d * Q + self.active_ffn_weights() + 2 * d
            return 2 * (L * per_layer + d + V * d + d)
        if self.n_experts:
            raise ValueError("mixture-of-experts models take FP16 weights")
        rows = L * ((Q + 2 * KV) + d + 2 * F + d) + V
        elems = L * ((Q + 2 * KV) * d + d * Q + 3 * d * F) + V * d
        if weights == "fp8":
            return elems + 4 * rows + 2 * (L * 2 * d + d + d)
        if weights == "mxfp4":
            # half a byte per element plus one E8M0 scale byte per 32 elements
            return elems // 2 + elems // 32 + 2 * (L * 2 * d + d + d)
        raise ValueError(weights)

    def kv_bytes_per_position(self) -> int:
        """FP16 K and V bytes of one cached position over all layers."""
        return 2 * 2 * self.n_layers * self.kv_dim

    def with_(self, **kw) -> "ModelConfig":
        return replace(self, **kw)


@dataclass(frozen=True)
class Workload:
    name: str
    model: ModelConfig
    weight_seed: int
    prompt_seed: int
    prompt_len: int
    decode_steps: int
    temperature: float = 0.0
    top_k: int = 0
    sample_seed: int = 0
    # None, or one attention window per layer in positions (0 = the whole cache)
    layer_window: tuple | None = None
    # projection weights: "fp16", "fp8" (E4M3 codes + FP32 per-row scales) or
    # "mxfp4" (E2M1 codes + E8M0 scales per 32 elements)
    weights: str = "fp16"

    @property
    def max_seq(self) -> int:
        return self.prompt_len + self.decode_steps

    def bytes_per_step(self, pos: int) -> int:
        """Algorithmic HBM bytes of the decode step whose input token sits at
        position `pos`: weights, the KV read of every layer (ctx = pos + 1
        positions, or the layer's window if shorter) and the KV write of one
        position."""
        m = self.model
        per_layer = m.kv_bytes_per_position() // m.n_layers
        ctx = pos + 1
        if self.layer_window is None:
            kv_read = ctx * m.kv_bytes_per_position()
        else:
            kv_read = sum(min(ctx, w) if w > 0 else ctx for w in self.layer_window) * per_layer
        return m.weight_bytes_per_token(self.weights) + kv_read + m.kv_bytes_per_position()

    def decode_bytes(self, first_pos: int, n_steps: int) -> int:
        return sum(self.bytes_per_step(first_pos + i) for i in range(n_steps))


MODELS = {
    "tiny": ModelConfig("tiny", 2, 256, 4, 4, 64, 1024, 4096),
    "small": ModelConfig("small", 16, 1024, 16, 4, 64, 4096, 32000),
    "2.3b": ModelConfig("2.3b", 25, 2560, 20, 5, 128, 8192, 64000),
    "8b": ModelConfig("8b", 32, 4096, 32, 8, 128, 14336, 128256),
    # two layers with the ~2.3B's attention shape: prefill-attention profiling on a small footprint
    "attn-2l": ModelConfig("attn-2l", 2, 2560, 20, 5, 128, 2048, 8000),
    # the ~2.3B decoder's attention with 8 experts of half its FFN width per
    # layer, 2 active: 6.3B parameters, the 2.3B's bytes per token
    "moe-8x": ModelConfig("moe-8x", 25, 2560, 20, 5, 128, 4096, 64000, n_experts=8, top_k_experts=2),
}

WORKLOADS = {
    "tiny": Workload("tiny", MODELS["tiny"], 0, 1000, 64, 32),
    "small": Workload("small", MODELS["small"], 1, 1001, 128, 256),
    "2.3b": Workload("2.3b", MODELS["2.3b"], 2, 1002, 512, 1024),
    "2.3b-32k": Workload("2.3b-32k", MODELS["2.3b"], 2, 1003, 32768, 256),
    # the same at 32k context with sliding-window attention in two of every
    # three layers (the pages' LaneFormer: 10 of 15 layers), window 4,096
    # positions (its stated context length; the pages give no window size)
    "2.3b-32k-swa": Workload("2.3b-32k-swa", MODELS["2.3b"], 2, 1003, 32768, 256,
                             layer_window=tuple(4096 if l % 3 != 2 else 0 for l in range(25))),
    "8b": Workload("8b", MODELS["8b"], 3, 1004, 2048, 512, temperature=0.8, top_k=50, sample_seed=1234),
    # the ~2.3B decoder with weight-only FP8 projections (the pages: FP8 streaming
    # halves the bytes that bound batch-1 decode)
    "2.3b-fp8": Workload("2.3b-fp8", MODELS["2.3b"], 2, 1002, 512, 1024, weights="fp8"),
    # a 4,096-token prompt on the two-layer model: the batched prefill's attention at length
    "prefill-4k": Workload("prefill-4k", MODELS["attn-2l"], 3, 4, 4096, 64),
    # mixture of experts (the pages: only the active experts' weights stream per token)
    "moe-8x": Workload("moe-8x", MODELS["moe-8x"], 4, 1002, 512, 1024),
    # the same with MXFP4 projections (the pages: "FP8/MXFP4" for frontier models)
    "2.3b-mxfp4": Workload("2.3b-mxfp4", MODELS["2.3b"], 2, 1002, 512, 1024, weights="mxfp4"),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]
