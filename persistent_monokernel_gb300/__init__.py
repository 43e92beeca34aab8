"""Python binding of liblf.so, the batch-1 decode monokernel (include/lf.h).

The binding marshals arguments only: every step of the decode pass runs in the
CUDA library.  PyTorch provides the device memory and the streams.  Importing
this module loads the in-tree liblf.so and fails loudly if it is missing (build
it with `python -m persistent_monokernel_gb300.build`); there is no CPU path.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblf.so")

LF_OK = 0
STATUS_NAMES = {0: "LF_OK", 1: "LF_ERR_INVALID_ARG", 2: "LF_ERR_OUT_OF_MEMORY", 3: "LF_ERR_CAPACITY",
                4: "LF_ERR_NOT_RESIDENT", 5: "LF_ERR_CUDA", 6: "LF_ERR_TIMEOUT", 7: "LF_ERR_NOT_SUPPORTED",
                8: "LF_ERR_STATE"}
SCHED_FLAGS, SCHED_GRID_BARRIER, SCHED_MULTI_KERNEL = 0, 1, 2
MAX_TOP_K = 64
PREFILL_AUTO = -1   # lf_config.prefill_block: batched prefill, block size chosen by the library (LF_PREFILL_AUTO)
TRACE_STAMPS = 9

# Every symbol include/lf.h declares.
EXPORTS = ("lf_create", "lf_destroy", "lf_prefill", "lf_decode", "lf_generate", "lf_sync", "lf_reset",
           "lf_set_schedule", "lf_get_info", "lf_error_string", "lf_abi_version", "lf_generate_noalloc",
           "lf_enable_trace", "lf_read_trace", "lf_sync_latency")


class LFError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class lf_config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn_dim", C.c_int32), ("vocab", C.c_int32),
                ("max_seq", C.c_int32), ("rope_theta", C.c_float), ("rms_eps", C.c_float),
                ("wait_timeout_ns", C.c_int64), ("n_ctas", C.c_int32), ("fault_step", C.c_int32),
                ("layer_window", C.POINTER(C.c_int32)), ("weight_format", C.c_int32),
                ("prefill_block", C.c_int32), ("n_experts", C.c_int32), ("top_k_experts", C.c_int32)]


WEIGHTS_FP16, WEIGHTS_FP8_E4M3, WEIGHTS_MXFP4 = 0, 1, 2
WEIGHT_FIELDS = ("embed", "attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down",
                 "final_norm", "lm_head")
FP8_MATRICES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "lm_head")
SCALE_FIELDS = tuple(n + "_scale" for n in FP8_MATRICES)


class lf_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in WEIGHT_FIELDS + SCALE_FIELDS + ("w_router",)]


class lf_sampling(C.Structure):
    _fields_ = [("temperature", C.c_float), ("top_k", C.c_int32), ("debug_logits_dev", C.c_void_p),
                ("force_tokens_dev", C.c_void_p)]


class lf_info(C.Structure):
    _fields_ = [("n_ctas", C.c_int32), ("threads_per_cta", C.c_int32), ("smem_bytes", C.c_int32),
                ("ring_bytes", C.c_int32), ("sm_count", C.c_int32), ("position", C.c_int32),
                ("has_pending", C.c_int32), ("schedule", C.c_int32), ("weight_stream_bytes", C.c_int64),
                ("kv_cache_bytes", C.c_int64), ("prefill_block", C.c_int32), ("prefill_bytes", C.c_int64)]


_lib = None


def lib() -> C.CDLL:
    """Load liblf.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with `python -m persistent_monokernel_gb300.build`")
        L = C.CDLL(LIB_PATH)
        vp = C.c_void_p
        L.lf_create.argtypes = [C.POINTER(lf_config), C.POINTER(lf_weights), C.POINTER(vp)]
        L.lf_destroy.argtypes = [vp]
        L.lf_destroy.restype = None
        L.lf_prefill.argtypes = [vp, vp, C.c_int32, vp]
        L.lf_decode.argtypes = [vp, C.c_int32, C.POINTER(lf_sampling), C.c_uint64, vp, vp]
        L.lf_generate.argtypes = [vp, C.POINTER(C.c_int32), C.c_int32, C.c_int32, C.POINTER(lf_sampling),
                                  C.c_uint64, C.POINTER(C.c_int32), vp]
        L.lf_sync.argtypes = [vp]
        L.lf_reset.argtypes = [vp]
        L.lf_set_schedule.argtypes = [vp, C.c_int32]
        L.lf_get_info.argtypes = [vp, C.POINTER(lf_info)]
        L.lf_error_string.argtypes = [C.c_int]
        L.lf_error_string.restype = C.c_char_p
        L.lf_abi_version.restype = C.c_int32
        L.lf_generate_noalloc.argtypes = [C.POINTER(lf_config), C.POINTER(lf_weights), vp, C.c_int32, C.c_int32,
                                          C.POINTER(lf_sampling), C.c_uint64, vp, vp]
        L.lf_generate_noalloc.restype = C.c_int
        L.lf_enable_trace.argtypes = [vp, C.c_int32]
        L.lf_enable_trace.restype = C.c_int
        L.lf_read_trace.argtypes = [vp, vp, C.c_int64, C.POINTER(C.c_int64)]
        L.lf_read_trace.restype = C.c_int
        L.lf_sync_latency.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.POINTER(C.c_double)]
        L.lf_sync_latency.restype = C.c_int
        for name in ("lf_create", "lf_prefill", "lf_decode", "lf_generate", "lf_sync", "lf_reset",
                     "lf_set_schedule", "lf_get_info"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != LF_OK:
        raise LFError(status, where)


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _windows(model, layer_window):
    """lf_config.layer_window: NULL, or a host int32 array of one window per layer."""
    if layer_window is None:
        return None
    vals = [int(v) for v in layer_window]
    if len(vals) != model.n_layers:
        raise ValueError("layer_window needs one entry per layer")
    return (C.c_int32 * len(vals))(*vals)


class Decoder:
    """One decoder on the current CUDA device.

    `model` is any object with the attributes n_layers, d_model, n_heads,
    n_kv_heads, head_dim, ffn_dim, vocab, rope_theta and rms_eps; `weights`
    maps the lf_weights field names to contiguous CUDA float16 tensors.
    """

    def __init__(self, model, weights: dict, max_seq: int, n_ctas: int = 0, wait_timeout_ns: int = 0,
                 fault_step: int = -1, layer_window=None, prefill_block: int = 0):
        import torch
        self.model = model
        self.max_seq = int(max_seq)
        # FP8 weights: the eight projections as uint8 E4M3 codes plus FP32 per-row scales;
        # MXFP4 weights: packed uint8 E2M1 codes plus uint8 E8M0 scales per 32 elements
        quant = weights["wq"].dtype == torch.uint8
        self.mxfp4 = quant and weights["wq_scale"].dtype == torch.uint8
        self.fp8 = quant and not self.mxfp4
        for n in WEIGHT_FIELDS + (SCALE_FIELDS if quant else ()):
            t = weights[n]
            if not quant or n not in FP8_MATRICES + SCALE_FIELDS:
                want = torch.float16
            elif n in FP8_MATRICES or self.mxfp4:
                want = torch.uint8
            else:
                want = torch.float32
            if not (t.is_cuda and t.dtype == want and t.is_contiguous()):
                raise ValueError(f"weight {n} must be a contiguous CUDA {want} tensor")
        fmt = WEIGHTS_MXFP4 if self.mxfp4 else WEIGHTS_FP8_E4M3 if self.fp8 else WEIGHTS_FP16
        # mixture of experts: w_gate / w_up [L, E, F, d], w_down [L, E, d, F] and the router [L, E, d]
        n_exp = int(getattr(model, "n_experts", 0) or 0)
        if n_exp:
            t = weights["w_router"]
            if not (t.is_cuda and t.dtype == torch.float16 and t.is_contiguous()):
                raise ValueError("weight w_router must be a contiguous CUDA torch.float16 tensor")
        # embed, the norm gains and the router are read in place by every step: keep them alive
        self._keep = {n: weights[n] for n in ("embed", "attn_norm", "ffn_norm", "final_norm")
                      + (("w_router",) if n_exp else ())}
        cfg = lf_config(model.n_layers, model.d_model, model.n_heads, model.n_kv_heads, model.head_dim,
                        model.ffn_dim, model.vocab, self.max_seq, model.rope_theta, model.rms_eps,
                        int(wait_timeout_ns), int(n_ctas), int(fault_step), _windows(model, layer_window),
                        fmt, int(prefill_block), n_exp, int(getattr(model, "top_k_experts", 0) or 0) if n_exp else 0)
        w = lf_weights(*[_dptr(weights[n]) for n in WEIGHT_FIELDS],
                       *[_dptr(weights[n]) if quant else None for n in SCALE_FIELDS],
                       _dptr(weights["w_router"]) if n_exp else None)
        h = C.c_void_p()
        _check(lib().lf_create(C.byref(cfg), C.byref(w), C.byref(h)), "lf_create")
        self._h = h

    # ---- lifetime
    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().lf_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # ---- calls
    def prefill(self, tokens, stream=None) -> None:
        import torch
        assert tokens.is_cuda and tokens.dtype == torch.int32 and tokens.is_contiguous()
        _check(lib().lf_prefill(self._h, _dptr(tokens), tokens.numel(), _stream_ptr(stream)), "lf_prefill")

    def decode(self, n_steps: int, temperature: float = 0.0, top_k: int = 0, seed: int = 0, out=None,
               debug_logits=None, force_tokens=None, stream=None):
        import torch
        if out is None:
            out = torch.empty(n_steps, dtype=torch.int32, device="cuda")
        sp = lf_sampling(float(temperature), int(top_k), _dptr(debug_logits), _dptr(force_tokens))
        _check(lib().lf_decode(self._h, int(n_steps), C.byref(sp), int(seed) & (2 ** 64 - 1), _dptr(out),
                               _stream_ptr(stream)), "lf_decode")
        return out

    def generate(self, prompt_host, n_steps: int, temperature: float = 0.0, top_k: int = 0, seed: int = 0,
                 stream=None):
        """Host buffers in and out (lf_generate): returns a numpy int32 array."""
        import numpy as np
        p = np.ascontiguousarray(np.asarray(prompt_host, dtype=np.int32))
        out = np.empty(n_steps, dtype=np.int32)
        sp = lf_sampling(float(temperature), int(top_k), 0, 0)
        _check(lib().lf_generate(self._h, p.ctypes.data_as(C.POINTER(C.c_int32)), p.size, int(n_steps),
                                 C.byref(sp), int(seed) & (2 ** 64 - 1), out.ctypes.data_as(C.POINTER(C.c_int32)),
                                 _stream_ptr(stream)), "lf_generate")
        return out

    def sync(self) -> int:
        """lf_sync: returns the status code (0, or 6 for a device timeout)."""
        return int(lib().lf_sync(self._h))

    def reset(self) -> None:
        _check(lib().lf_reset(self._h), "lf_reset")

    def set_schedule(self, schedule: int) -> None:
        _check(lib().lf_set_schedule(self._h, int(schedule)), "lf_set_schedule")

    def enable_trace(self, max_steps: int) -> None:
        _check(lib().lf_enable_trace(self._h, int(max_steps)), "lf_enable_trace")

    def read_trace(self):
        """Stage trace as a uint64 array [steps, slots, ctas, TRACE_STAMPS] (ns stamps; the last field
        is a count of weight chunks that had not landed when first asked for)."""
        import numpy as np
        n = C.c_int64()
        _check(lib().lf_read_trace(self._h, None, 0, C.byref(n)), "lf_read_trace")
        buf = np.zeros(n.value, dtype=np.uint64)
        _check(lib().lf_read_trace(self._h, buf.ctypes.data, n.value, C.byref(n)), "lf_read_trace")
        slots = 5 * self.model.n_layers + 1
        return buf.reshape(-1, slots, self.info()["n_ctas"], TRACE_STAMPS)

    def info(self) -> dict:
        i = lf_info()
        _check(lib().lf_get_info(self._h, C.byref(i)), "lf_get_info")
        return {f: getattr(i, f) for f, _ in lf_info._fields_}


def sync_latency_ns(mode: int, n_ctas: int, iters: int) -> float:
    """lf_sync_latency: ns per flag hop (mode 0) or per grid barrier (mode 1)."""
    v = C.c_double()
    _check(lib().lf_sync_latency(int(mode), int(n_ctas), int(iters), C.byref(v)), "lf_sync_latency")
    return v.value


def error_string(status: int) -> str:
    return lib().lf_error_string(int(status)).decode()
