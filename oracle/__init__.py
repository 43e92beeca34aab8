"""CPU oracle for batch-1 decoder decode (ctypes wrapper over lf_oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg are the only users.  Nothing in the
persistent_monokernel_gb300 package imports this module, and this module
imports nothing from that package.

Precision: FP32 activations and FP32 sums in index order (the KOG monokernel
write-up, shivam2003.com, "The fused operations, briefly": FP32-accumulated
GEMV partial products), FP16 weights and an FP16 KV cache.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lf_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C11 + OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Config(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("d_model", C.c_int), ("n_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn_dim", C.c_int), ("vocab", C.c_int), ("max_seq", C.c_int),
                ("rope_theta", C.c_float), ("rms_eps", C.c_float)]


_WNAMES = ("embed", "attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down",
           "final_norm", "lm_head")


class _Weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _WNAMES]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            f32p = C.POINTER(C.c_float)
            u16p = C.POINTER(C.c_uint16)
            L.orc_half_to_float.argtypes = [C.c_uint16]
            L.orc_half_to_float.restype = C.c_float
            L.orc_float_to_half.argtypes = [C.c_float]
            L.orc_float_to_half.restype = C.c_uint16
            L.orc_rmsnorm.argtypes = [f32p, u16p, C.c_int, C.c_float, f32p]
            L.orc_matvec.argtypes = [u16p, f32p, C.c_int, C.c_int, f32p]
            L.orc_rope.argtypes = [f32p, C.c_int, C.c_int, C.c_float]
            L.orc_attend_head.argtypes = [f32p, u16p, u16p, C.c_int, C.c_int, C.c_float, f32p, f32p]
            L.orc_silu.argtypes = [C.c_float]
            L.orc_silu.restype = C.c_float
            L.orc_philox4x32_10.argtypes = [C.POINTER(C.c_uint32), C.POINTER(C.c_uint32), C.POINTER(C.c_uint32)]
            L.orc_gumbel.argtypes = [C.c_uint64, C.c_int, C.c_int]
            L.orc_gumbel.restype = C.c_float
            L.orc_sample.argtypes = [f32p, C.c_int, C.c_float, C.c_int, C.c_uint64, C.c_int]
            L.orc_sample.restype = C.c_int
            L.orc_create.argtypes = [C.POINTER(_Config), C.POINTER(_Weights)]
            L.orc_create.restype = C.c_void_p
            L.orc_destroy.argtypes = [C.c_void_p]
            L.orc_reset.argtypes = [C.c_void_p]
            L.orc_set_windows.argtypes = [C.c_void_p, C.POINTER(C.c_int32)]
            L.orc_set_fp8.argtypes = [C.c_void_p, C.POINTER(C.c_void_p)]
            L.orc_e4m3_to_float.argtypes = [C.c_uint8]
            L.orc_e4m3_to_float.restype = C.c_float
            L.orc_matvec_fp8.argtypes = [C.POINTER(C.c_uint8), f32p, f32p, C.c_int, C.c_int, f32p]
            L.orc_set_mxfp4.argtypes = [C.c_void_p, C.POINTER(C.c_void_p)]
            L.orc_set_moe.argtypes = [C.c_void_p, C.c_int, C.c_int, u16p]
            L.orc_route.argtypes = [f32p, C.c_int, C.c_int, C.POINTER(C.c_int32), f32p]
            L.orc_e2m1_to_float.argtypes = [C.c_uint8]
            L.orc_e2m1_to_float.restype = C.c_float
            L.orc_e8m0_to_float.argtypes = [C.c_uint8]
            L.orc_e8m0_to_float.restype = C.c_float
            L.orc_matvec_mxfp4.argtypes = [C.POINTER(C.c_uint8), C.POINTER(C.c_uint8), f32p, C.c_int, C.c_int, f32p]
            L.orc_pos.argtypes = [C.c_void_p]
            L.orc_pending.argtypes = [C.c_void_p]
            L.orc_kcache.argtypes = [C.c_void_p]
            L.orc_kcache.restype = C.c_void_p
            L.orc_vcache.argtypes = [C.c_void_p]
            L.orc_vcache.restype = C.c_void_p
            L.orc_forward.argtypes = [C.c_void_p, C.c_int, f32p]
            L.orc_prefill.argtypes = [C.c_void_p, C.POINTER(C.c_int32), C.c_int]
            L.orc_prefill_blocked.argtypes = [C.c_void_p, C.POINTER(C.c_int32), C.c_int, C.c_int]
            L.orc_skip_to.argtypes = [C.c_void_p, C.c_int, C.c_int]
            L.orc_decode.argtypes = [C.c_void_p, C.c_int, C.c_float, C.c_int, C.c_uint64,
                                     C.POINTER(C.c_int32), C.POINTER(C.c_int32), f32p]
            _lib = L
    return _lib


def _f32(a):
    return a.ctypes.data_as(C.POINTER(C.c_float))


def _u16(a):
    return a.ctypes.data_as(C.POINTER(C.c_uint16))


def _i32(a):
    return a.ctypes.data_as(C.POINTER(C.c_int32))


def _as_np(a) -> np.ndarray:
    if hasattr(a, "numpy"):
        a = a.detach().cpu().contiguous().numpy()
    return np.ascontiguousarray(a)


FP8_MATRICES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "lm_head")


def _as_u16(a) -> np.ndarray:
    """FP16 data (numpy float16 / torch float16 CPU tensor) viewed as uint16, C-contiguous."""
    if hasattr(a, "numpy"):
        a = a.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("expected FP16 data")
    return a


# ---------------------------------------------------------------- op level

def half_to_float(bits: int) -> float:
    return lib().orc_half_to_float(bits)


def float_to_half(x: float) -> int:
    return lib().orc_float_to_half(x)


def rmsnorm(x, g, eps):
    x = np.ascontiguousarray(x, dtype=np.float32)
    g = _as_u16(g)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_f32(x), _u16(g), x.size, eps, _f32(out))
    return out


def matvec(W, x):
    W = _as_u16(W)
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(W.shape[0], dtype=np.float32)
    lib().orc_matvec(_u16(W), _f32(x), W.shape[0], W.shape[1], _f32(y))
    return y


def e4m3_to_float(code: int) -> float:
    return lib().orc_e4m3_to_float(code)


def matvec_fp8(codes, scale, x):
    """y = diag(scale) . decode_e4m3(codes) . x (codes uint8 [rows, cols])."""
    Cc = np.ascontiguousarray(_as_np(codes), dtype=np.uint8)
    sc = np.ascontiguousarray(_as_np(scale), dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(Cc.shape[0], dtype=np.float32)
    lib().orc_matvec_fp8(Cc.ctypes.data_as(C.POINTER(C.c_uint8)), _f32(sc), _f32(x), Cc.shape[0], Cc.shape[1], _f32(y))
    return y


def e2m1_to_float(nibble: int) -> float:
    return lib().orc_e2m1_to_float(nibble)


def e8m0_to_float(code: int) -> float:
    return lib().orc_e8m0_to_float(code)


def matvec_mxfp4(codes, bscale, x):
    """y = decode_mxfp4(codes, bscale) . x (codes uint8 [rows, cols/2], two
    E2M1 elements per byte, low nibble first; bscale uint8 [rows, cols/32])."""
    Cc = np.ascontiguousarray(_as_np(codes), dtype=np.uint8)
    Sc = np.ascontiguousarray(_as_np(bscale), dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(Cc.shape[0], dtype=np.float32)
    u8p = C.POINTER(C.c_uint8)
    lib().orc_matvec_mxfp4(Cc.ctypes.data_as(u8p), Sc.ctypes.data_as(u8p), _f32(x), Cc.shape[0], x.size, _f32(y))
    return y


def route(logits, top_k: int):
    """Top-k expert choice of one token: (experts in decreasing logit order, gates)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    sel = np.empty(top_k, dtype=np.int32)
    gate = np.empty(top_k, dtype=np.float32)
    lib().orc_route(_f32(lg), lg.size, top_k, _i32(sel), _f32(gate))
    return sel, gate


def rope(v, pos, base):
    v = np.array(v, dtype=np.float32, copy=True)
    lib().orc_rope(_f32(v), v.size, pos, base)
    return v


def attend_head(q, K, V, scale):
    q = np.ascontiguousarray(q, dtype=np.float32)
    K = _as_u16(K)
    V = _as_u16(V)
    ctx, hd = K.shape
    scores = np.empty(ctx, dtype=np.float32)
    out = np.empty(hd, dtype=np.float32)
    lib().orc_attend_head(_f32(q), _u16(K), _u16(V), ctx, hd, scale, _f32(scores), _f32(out))
    return out, scores


def silu(z: float) -> float:
    return lib().orc_silu(z)


def philox4x32_10(ctr, key):
    c = (C.c_uint32 * 4)(*[int(v) & 0xFFFFFFFF for v in ctr])
    k = (C.c_uint32 * 2)(*[int(v) & 0xFFFFFFFF for v in key])
    o = (C.c_uint32 * 4)()
    lib().orc_philox4x32_10(c, k, o)
    return [int(v) for v in o]


def gumbel(seed: int, pos: int, i: int) -> float:
    return lib().orc_gumbel(seed, pos, i)


def sample(logits, temperature: float, top_k: int, seed: int, pos: int) -> int:
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    return lib().orc_sample(_f32(lg), lg.size, temperature, top_k, seed, pos)


def num_threads() -> int:
    return lib().orc_num_threads()


# ------------------------------------------------------------- the decoder

class OracleDecoder:
    """The whole decoder on the CPU.  `weights` maps the synthetic tensor
    names to FP16 arrays (numpy float16 or CPU torch.float16).
    `layer_window`: None (every layer attends to the whole cache) or one
    window per layer in positions, 0 = the whole cache."""

    def __init__(self, cfg, weights: dict, max_seq: int, layer_window=None):
        self.cfg = cfg
        self.max_seq = max_seq
        # FP8 weights: the eight projections are uint8 E4M3 codes with FP32
        # per-row scales in weights["<name>_scale"]; MXFP4 weights: packed
        # E2M1 codes [rows, cols/2] with uint8 E8M0 block scales [rows, cols/32]
        quant = _as_np(weights["wq"]).dtype == np.uint8
        self.mxfp4 = quant and _as_np(weights["wq_scale"]).dtype == np.uint8
        self.fp8 = quant and not self.mxfp4
        self._keep = {}
        for n in _WNAMES:
            if quant and n in FP8_MATRICES:
                self._keep[n] = np.ascontiguousarray(_as_np(weights[n]), dtype=np.uint8)
                self._keep[n + "_scale"] = np.ascontiguousarray(_as_np(weights[n + "_scale"]),
                                                                dtype=np.uint8 if self.mxfp4 else np.float32)
            else:
                self._keep[n] = _as_u16(weights[n])
        c = _Config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                    cfg.vocab, max_seq, cfg.rope_theta, cfg.rms_eps)
        w = _Weights(*[self._keep[n].ctypes.data for n in _WNAMES])
        self._h = lib().orc_create(C.byref(c), C.byref(w))
        if not self._h:
            raise ValueError("orc_create rejected the configuration")
        if quant:
            ptrs = (C.c_void_p * 8)(*[self._keep[n + "_scale"].ctypes.data for n in FP8_MATRICES])
            (lib().orc_set_mxfp4 if self.mxfp4 else lib().orc_set_fp8)(self._h, ptrs)
        # mixture-of-experts FFN: w_gate / w_up [L, E, F, d], w_down [L, E, d, F], w_router [L, E, d]
        self.n_experts = int(getattr(cfg, "n_experts", 0) or 0)
        if self.n_experts:
            self._keep["w_router"] = _as_u16(weights["w_router"])
            if lib().orc_set_moe(self._h, self.n_experts, int(cfg.top_k_experts),
                                 _u16(self._keep["w_router"])):
                raise ValueError("orc_set_moe rejected the expert configuration")
        if layer_window is not None:
            win = np.ascontiguousarray(np.asarray(layer_window, dtype=np.int32))
            if win.shape != (cfg.n_layers,):
                raise ValueError("layer_window needs one entry per layer")
            lib().orc_set_windows(self._h, _i32(win))

    def close(self):
        if getattr(self, "_h", None):
            lib().orc_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def reset(self):
        lib().orc_reset(self._h)

    @property
    def pos(self) -> int:
        return lib().orc_pos(self._h)

    @property
    def pending(self) -> int:
        return lib().orc_pending(self._h)

    def kv_cache(self):
        c = self.cfg
        n = c.n_layers * c.n_kv_heads * self.max_seq * c.head_dim
        shape = (c.n_layers, c.n_kv_heads, self.max_seq, c.head_dim)
        k = np.ctypeslib.as_array(C.cast(lib().orc_kcache(self._h), C.POINTER(C.c_uint16)), (n,))
        v = np.ctypeslib.as_array(C.cast(lib().orc_vcache(self._h), C.POINTER(C.c_uint16)), (n,))
        return k.reshape(shape).view(np.float16).copy(), v.reshape(shape).view(np.float16).copy()

    def forward(self, token: int, want_logits: bool = True):
        lg = np.empty(self.cfg.vocab, dtype=np.float32) if want_logits else None
        rc = lib().orc_forward(self._h, int(token), _f32(lg) if want_logits else None)
        if rc:
            raise ValueError("orc_forward failed (cache full or bad token)")
        return lg

    def prefill(self, tokens):
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        if lib().orc_prefill(self._h, _i32(t), t.size):
            raise ValueError("orc_prefill failed (cache full or empty prompt)")

    def prefill_blocked(self, tokens, block: int = 64):
        """The same forward passes as prefill(), visited `block` positions at a
        time (each weight row decoded once per block); the cache and state
        equal prefill()'s bit for bit.  Dense FP16 models only."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        if lib().orc_prefill_blocked(self._h, _i32(t), t.size, int(block)):
            raise ValueError("orc_prefill_blocked failed (cache full, empty prompt or unsupported model)")

    def skip_to(self, pos: int, token: int):
        """Timing hook: `token` becomes the pending token at position `pos`
        without the forward passes before it (their cache rows are left as
        they are).  For timing decode steps at a given context only."""
        if lib().orc_skip_to(self._h, int(pos), int(token)):
            raise ValueError("orc_skip_to: position or token out of range")

    def decode(self, n_steps: int, temperature: float = 0.0, top_k: int = 0, seed: int = 0,
               force_tokens=None, want_logits: bool = True):
        out = np.empty(n_steps, dtype=np.int32)
        lg = np.empty((n_steps, self.cfg.vocab), dtype=np.float32) if want_logits else None
        ft = None
        if force_tokens is not None:
            ft = np.ascontiguousarray(np.asarray(force_tokens, dtype=np.int32))
            assert ft.size >= n_steps
        rc = lib().orc_decode(self._h, n_steps, temperature, top_k, seed,
                              _i32(ft) if ft is not None else None, _i32(out),
                              _f32(lg) if want_logits else None)
        if rc:
            raise ValueError("orc_decode failed (no pending token or cache full)")
        return out, lg
