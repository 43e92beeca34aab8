"""Seeded FP16 weights and prompt ids, bit-identical on CPU and CUDA.

Every weight is one entry of a fixed table of 65,536 FP16 values: the
quantiles 0.02 * Phi^-1((k + 0.5) / 65536) of N(0, 0.02), each rounded to FP16.
A counter-based integer hash of (seed, tensor, layer, element index) picks the
entry.  Only integer operations and a gather are used, with every intermediate
product below 2**63, so torch gives the same bits on the CPU and on a GPU.  The
weights therefore follow N(0, 0.02) to within FP16 rounding.

Tensor layouts are row-major, nn.Linear style ([out, in]), stacked over layers:
  embed [V, d], attn_norm [L, d], wq [L, Q, d], wk [L, KV, d], wv [L, KV, d],
  wo [L, d, Q], ffn_norm [L, d], w_gate [L, F, d], w_up [L, F, d],
  w_down [L, d, F], final_norm [d], lm_head [V, d].
"""
from __future__ import annotations

from statistics import NormalDist

import torch

from .configs import ModelConfig

MASK32 = 0xFFFFFFFF
# Odd multipliers below 2**31, so that a 32-bit value times one stays below 2**63.
_C1 = 0x7FEB352D
_C2 = 0x2C1B3C6D
_C3 = 0x297A2D39
_C4 = 0x5BD1E995 & 0x7FFFFFFF

WEIGHT_ORDER = ("embed", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "lm_head",
                "attn_norm", "ffn_norm", "final_norm")
_TENSOR_ID = {name: i + 1 for i, name in enumerate(WEIGHT_ORDER)}
_TENSOR_ID["w_router"] = 0x30

_TABLE_CACHE: dict = {}


def normal_table(std: float = 0.02) -> torch.Tensor:
    """FP16 table of the 65,536 mid-quantiles of N(0, std)."""
    key = float(std)
    if key not in _TABLE_CACHE:
        nd = NormalDist(0.0, 1.0)
        vals = [std * nd.inv_cdf((k + 0.5) / 65536.0) for k in range(65536)]
        _TABLE_CACHE[key] = torch.tensor(vals, dtype=torch.float64).to(torch.float16)
    return _TABLE_CACHE[key]


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """Integer avalanche mix of int64 tensors that hold 32-bit values."""
    x = x ^ (x >> 16)
    x = (x * _C1) & MASK32
    x = x ^ (x >> 15)
    x = (x * _C2) & MASK32
    x = x ^ (x >> 16)
    return x


def _mix_scalar(x: int) -> int:
    x &= MASK32
    x ^= x >> 16
    x = (x * _C1) & MASK32
    x ^= x >> 15
    x = (x * _C2) & MASK32
    x ^= x >> 16
    return x


def _stream_key(seed: int, tensor_id: int, layer: int) -> tuple:
    k1 = _mix_scalar((seed * _C3 + tensor_id) & MASK32)
    k1 = _mix_scalar(k1 ^ ((layer * _C4) & MASK32))
    k2 = _mix_scalar(k1 + 0x9E3779B9)
    return k1, k2


def hashed_indices(seed: int, tensor_id: int, layer: int, start: int, n: int, device) -> torch.Tensor:
    """16-bit table indices for elements [start, start + n) of one stream."""
    k1, k2 = _stream_key(seed, tensor_id, layer)
    i = torch.arange(start, start + n, dtype=torch.int64, device=device)
    h = _mix32((i & MASK32) ^ k1)
    h = _mix32((h + k2) & MASK32)
    return (h >> 16) & 0xFFFF


_CHUNK = 1 << 20        # CPU: keeps the int64 temporaries in cache
_CHUNK_CUDA = 1 << 26   # GPU: few launches


def _fill(out: torch.Tensor, table: torch.Tensor, seed: int, tensor_id: int, layer: int) -> None:
    flat = out.view(-1)
    n = flat.numel()
    chunk = _CHUNK_CUDA if flat.is_cuda else _CHUNK
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        idx = hashed_indices(seed, tensor_id, layer, s, m, flat.device)
        flat[s:s + m] = table[idx]


def make_weights(cfg: ModelConfig, seed: int, device="cpu", gains: str = "ones", projections: bool = True) -> dict:
    """All FP16 tensors of one decoder.

    gains="ones" gives RMSNorm gains of exactly 1.0 (the configured
    workloads); gains="random" gives 1 + N(0, 0.1)-distributed gains, used by
    tests to exercise the gain multiply.  projections=False leaves out the
    eight projection matrices (embedding and gains only).
    """
    device = torch.device(device)
    table = normal_table(0.02).to(device)
    L, d, F, V = cfg.n_layers, cfg.d_model, cfg.ffn_dim, cfg.vocab
    Q, KV = cfg.q_dim, cfg.kv_dim
    shapes = {
        "embed": (V, d), "wq": (L, Q, d), "wk": (L, KV, d), "wv": (L, KV, d), "wo": (L, d, Q),
        "w_gate": (L, F, d), "w_up": (L, F, d), "w_down": (L, d, F), "lm_head": (V, d),
    }
    names = WEIGHT_ORDER[:9]
    E = getattr(cfg, "n_experts", 0)
    if E:
        # mixture of experts: E FFNs per layer and the router
        shapes.update({"w_gate": (L, E, F, d), "w_up": (L, E, F, d), "w_down": (L, E, d, F), "w_router": (L, E, d)})
        names = names + ("w_router",)
    w = {}
    for name in names:
        if not projections and name != "embed":
            continue
        shp = shapes[name]
        t = torch.empty(shp, dtype=torch.float16, device=device)
        if len(shp) >= 3:
            for layer in range(shp[0]):
                _fill(t[layer], table, seed, _TENSOR_ID[name], layer)
        else:
            _fill(t, table, seed, _TENSOR_ID[name], 0)
        w[name] = t
    norm_shapes = {"attn_norm": (L, d), "ffn_norm": (L, d), "final_norm": (d,)}
    for name, shp in norm_shapes.items():
        if gains == "ones":
            w[name] = torch.ones(shp, dtype=torch.float16, device=device)
        elif gains == "random":
            t = torch.empty(shp, dtype=torch.float16, device=device)
            _fill(t, table, seed, _TENSOR_ID[name], 0)
            # 1 + 5 * N(0, 0.02) = 1 + N(0, 0.1), rounded to FP16
            w[name] = (1.0 + 5.0 * t.to(torch.float32)).to(torch.float16)
        else:
            raise ValueError(f"gains must be 'ones' or 'random', not {gains!r}")
    return w


# ---- FP8 (E4M3) weights with one FP32 scale per output row

FP8_MATRICES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "lm_head")
_FP8_CODE_STD = 64.0    # the codes' N(0, 64): +-448 (E4M3's largest finite value) is 7 sigma
_FP8_TABLE_CACHE: dict = {}


def fp8_code_table() -> torch.Tensor:
    """uint8 table of 65,536 E4M3 codes: the mid-quantiles of N(0, 64), each
    clipped to +-448 and converted to E4M3 by torch's float8_e4m3fn cast."""
    if "t" not in _FP8_TABLE_CACHE:
        nd = NormalDist(0.0, _FP8_CODE_STD)
        vals = torch.tensor([nd.inv_cdf((k + 0.5) / 65536.0) for k in range(65536)], dtype=torch.float32)
        vals = vals.clamp(-448.0, 448.0)
        _FP8_TABLE_CACHE["t"] = vals.to(torch.float8_e4m3fn).view(torch.uint8)
    return _FP8_TABLE_CACHE["t"]


def _fill_scales(out: torch.Tensor, seed: int, tensor_id: int, layer: int) -> None:
    """Per-row FP32 scales 0.02/64 * u, u uniform on [0.75, 1.25) in 2**-16 steps,
    so that code * scale follows N(0, 0.02) with a row-dependent spread."""
    idx = hashed_indices(seed, 0x100 + tensor_id, layer, 0, out.numel(), out.device)
    u = 0.75 + idx.to(torch.float64) * (0.5 / 65536.0)
    out.copy_((u * (0.02 / _FP8_CODE_STD)).to(torch.float32).view(out.shape))


def make_weights_fp8(cfg: ModelConfig, seed: int, device="cpu", gains: str = "ones") -> dict:
    """A decoder whose eight projection matrices are E4M3 codes (uint8, same
    shapes as the FP16 weights) with FP32 scales per output row (`<name>_scale`,
    [L, rows] or [V]); the embedding and the norm gains stay FP16 (make_weights).
    The matrix a layer applies is diag(scale) . decode(codes)."""
    w = make_weights(cfg, seed, device=device, gains=gains, projections=False)
    device = torch.device(device)
    table = fp8_code_table().to(device)
    L, d, F, V, Q, KV = cfg.n_layers, cfg.d_model, cfg.ffn_dim, cfg.vocab, cfg.q_dim, cfg.kv_dim
    shapes = {"wq": (L, Q, d), "wk": (L, KV, d), "wv": (L, KV, d), "wo": (L, d, Q), "w_gate": (L, F, d),
              "w_up": (L, F, d), "w_down": (L, d, F), "lm_head": (V, d)}
    for name in FP8_MATRICES:
        shp = shapes[name]
        codes = torch.empty(shp, dtype=torch.uint8, device=device)
        scales = torch.empty(shp[:-1], dtype=torch.float32, device=device)
        if len(shp) == 3:
            for layer in range(shp[0]):
                _fill(codes[layer], table, seed, _TENSOR_ID[name], layer)
                _fill_scales(scales[layer], seed, _TENSOR_ID[name], layer)
        else:
            _fill(codes, table, seed, _TENSOR_ID[name], 0)
            _fill_scales(scales, seed, _TENSOR_ID[name], 0)
        w[name] = codes
        w[name + "_scale"] = scales
    return w


# MXFP4 codes: each byte holds two 4-bit codes (sign bit 3, magnitude code
# 0..7 in bits 0-2).  Magnitude codes are drawn with these frequencies (in
# 128ths), a bell-shaped spread over the code range; signs are even.
_MXFP4_MAG_FREQ = (24, 32, 26, 18, 14, 9, 4, 1)
_MXFP4_TABLE_CACHE: dict = {}


def mxfp4_byte_table() -> torch.Tensor:
    """uint8 table of 65,536 bytes: index bits 0-6 pick the low code's
    magnitude bucket, bit 7 its sign, bits 8-14 / 15 the same for the high code."""
    if "t" not in _MXFP4_TABLE_CACHE:
        bucket = []
        for code, f in enumerate(_MXFP4_MAG_FREQ):
            bucket += [code] * f
        assert len(bucket) == 128
        t = torch.empty(65536, dtype=torch.uint8)
        for k in range(65536):
            lo = bucket[k & 127] | (8 if k & 128 else 0)
            hi = bucket[(k >> 8) & 127] | (8 if k & 32768 else 0)
            t[k] = lo | (hi << 4)
        _MXFP4_TABLE_CACHE["t"] = t
    return _MXFP4_TABLE_CACHE["t"]


def _fill_block_scales(out: torch.Tensor, seed: int, tensor_id: int, layer: int) -> None:
    """E8M0 block scales 121 + {-1, 0, +1} (2^-7 .. 2^-5), seeded per element."""
    idx = hashed_indices(seed, 0x200 + tensor_id, layer, 0, out.numel(), out.device)
    out.copy_((120 + idx % 3).to(torch.uint8).view(out.shape))


def make_weights_mxfp4(cfg: ModelConfig, seed: int, device="cpu", gains: str = "ones") -> dict:
    """A decoder whose eight projection matrices are MXFP4: packed 4-bit E2M1
    codes (uint8 [.., rows, cols/2], element 2i in the low nibble of byte i)
    with one E8M0 scale byte per 32 elements of a row (`<name>_scale`, uint8
    [.., rows, cols/32]); the embedding and the norm gains stay FP16."""
    w = make_weights(cfg, seed, device=device, gains=gains, projections=False)
    device = torch.device(device)
    table = mxfp4_byte_table().to(device)
    L, d, F, V, Q, KV = cfg.n_layers, cfg.d_model, cfg.ffn_dim, cfg.vocab, cfg.q_dim, cfg.kv_dim
    shapes = {"wq": (L, Q, d), "wk": (L, KV, d), "wv": (L, KV, d), "wo": (L, d, Q), "w_gate": (L, F, d),
              "w_up": (L, F, d), "w_down": (L, d, F), "lm_head": (V, d)}
    for name in FP8_MATRICES:
        shp = shapes[name]
        codes = torch.empty(shp[:-1] + (shp[-1] // 2,), dtype=torch.uint8, device=device)
        scales = torch.empty(shp[:-1] + (shp[-1] // 32,), dtype=torch.uint8, device=device)
        if len(shp) == 3:
            for layer in range(shp[0]):
                _fill(codes[layer], table, seed, _TENSOR_ID[name], layer)
                _fill_block_scales(scales[layer], seed, _TENSOR_ID[name], layer)
        else:
            _fill(codes, table, seed, _TENSOR_ID[name], 0)
            _fill_block_scales(scales, seed, _TENSOR_ID[name], 0)
        w[name] = codes
        w[name + "_scale"] = scales
    return w


def make_prompt(vocab: int, n: int, seed: int, device="cpu") -> torch.Tensor:
    """n token ids, uniform on [0, vocab) (up to a 2**-32 modulo bias), int32."""
    k1, k2 = _stream_key(seed, 0x50524F4D, 0)  # tensor id "PROM"
    i = torch.arange(n, dtype=torch.int64, device=device)
    h = _mix32((i & MASK32) ^ k1)
    h = _mix32((h + k2) & MASK32)
    return (h % vocab).to(torch.int32)
