"""CPU oracle for the MLA prolog (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this package.  The product library never imports it, and it imports
nothing of the product: the two share only the seeded inputs of
``attention_pre_processing_gb300.workloads``, which the callers pass in.

The arithmetic lives in ``mla_oracle.c`` (plain C, fp64, OpenMP over tokens);
this file only marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmla_oracle.so")
_lib = None

# Bit-exact IEEE arithmetic: no fast-math, no fused multiply-add contraction
# (aarch64 gcc contracts by default), so that x86 and Arm hosts agree.
CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/libmla_oracle.so."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Args(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("T", "He", "Hcq", "N", "D", "Dr", "Hckv", "block_num", "block_size")] + [
        ("eps_cq", ctypes.c_double), ("eps_ckv", ctypes.c_double),
        ("x_int8", ctypes.c_int32), ("uqqr_int8", ctypes.c_int32), ("kv_int8", ctypes.c_int32),
        ("kr_int8", ctypes.c_int32), ("q_int8", ctypes.c_int32), ("num_threads", ctypes.c_int32),
    ] + [(n, ctypes.c_void_p) for n in (
        "x", "w_dq", "w_uqqr", "w_uk", "w_dkvkr", "gamma_cq", "gamma_ckv", "rope_sin", "rope_cos",
        "cache_index", "dequant_scale_x", "dequant_scale_w_dq", "dequant_scale_w_uqqr",
        "dequant_scale_w_dkvkr", "quant_scale_ckv", "quant_scale_ckr", "smooth_scales_cq",
        "kv_cache", "kr_cache", "q_nope", "q_rope", "c_q", "c_kv", "k_r", "q_c",
        "q_nope_i8", "q_nope_scale", "c_q_i8", "c_q_scale")]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        L.mla_oracle_prolog.argtypes = [ctypes.POINTER(_Args)]
        L.mla_oracle_prolog.restype = ctypes.c_int
        L.mla_oracle_bf16_rne.argtypes = [ctypes.c_double]
        L.mla_oracle_bf16_rne.restype = ctypes.c_uint16
        L.mla_oracle_round_i8.argtypes = [ctypes.c_double]
        L.mla_oracle_round_i8.restype = ctypes.c_int8
        dp = ctypes.POINTER(ctypes.c_double)
        L.mla_oracle_rmsnorm.argtypes = [dp, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, dp]
        L.mla_oracle_rope_half.argtypes = [dp, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, dp]
        L.mla_oracle_dynamic_quant.argtypes = [dp, ctypes.c_int64, ctypes.c_void_p]
        L.mla_oracle_dynamic_quant.restype = ctypes.c_double
        L.mla_oracle_row_times_bf16.argtypes = [dp, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                                ctypes.c_int64, ctypes.c_int64, dp]
        L.mla_oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


# ---------------------------------------------------------------- helpers

def _np(t):
    """torch tensor / numpy array -> contiguous numpy array with the same bits (bf16 as uint16)."""
    if t is None:
        return None
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(t)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(lib().mla_oracle_max_threads())


# ------------------------------------------------------------ single steps

def bf16_rne(v) -> np.ndarray:
    """Round doubles to bf16 bit patterns (uint16), nearest-even, one step."""
    v = np.asarray(v, dtype=np.float64)
    f = lib().mla_oracle_bf16_rne
    return np.array([f(float(x)) for x in v.reshape(-1)], dtype=np.uint16).reshape(v.shape)


def round_i8(v) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    f = lib().mla_oracle_round_i8
    return np.array([f(float(x)) for x in v.reshape(-1)], dtype=np.int8).reshape(v.shape)


def rmsnorm(y, gamma_bf16_bits, eps: float) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float64)
    g = np.ascontiguousarray(gamma_bf16_bits, dtype=np.uint16)
    out = np.empty_like(y)
    lib().mla_oracle_rmsnorm(_dptr(y), y.size, _ptr(g), float(eps), _dptr(out))
    return out


def rope_half(v, cos_bf16_bits, sin_bf16_bits) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    c = np.ascontiguousarray(cos_bf16_bits, dtype=np.uint16)
    s = np.ascontiguousarray(sin_bf16_bits, dtype=np.uint16)
    out = np.empty_like(v)
    lib().mla_oracle_rope_half(_dptr(v), v.size, _ptr(c), _ptr(s), _dptr(out))
    return out


def dynamic_quant(v):
    v = np.ascontiguousarray(v, dtype=np.float64)
    codes = np.empty(v.shape, dtype=np.int8)
    scale = lib().mla_oracle_dynamic_quant(_dptr(v), v.size, _ptr(codes))
    return codes, scale


def row_times_bf16(x, w_bf16_bits) -> np.ndarray:
    """out = x . W for one row x (K,) and W (K, n) given as bf16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w_bf16_bits, dtype=np.uint16)
    K, n = w.shape
    out = np.empty(n, dtype=np.float64)
    lib().mla_oracle_row_times_bf16(_dptr(x), K, _ptr(w), n, 0, n, _dptr(out))
    return out


# ------------------------------------------------------------- whole prolog

ERRORS = {1: "bad arguments", 2: "cacheIndex out of range", 3: "duplicate cacheIndex"}


class OracleError(RuntimeError):
    pass


def prolog(inp: Dict, *, dims, eps_cq: float, eps_ckv: float, x_int8=False, uqqr_int8=None,
           kv_int8=False, kr_int8=False, q_int8=False, tokens=None, num_threads: int = 0,
           with_intermediates: bool = True) -> Dict[str, np.ndarray]:
    """Run the oracle on the inputs of ``workloads.make_inputs`` (torch or numpy).

    ``dims`` carries T, He, Hcq, N, D, Dr, Hckv, block_num, block_size.  With
    ``tokens`` (an index list) only those tokens are computed, and only their
    cache rows are written: the prolog is independent across tokens.
    Returns fp64 results before output rounding, the int8 results when asked,
    and copies of both caches with this call's rows written.
    """
    if uqqr_int8 is None:
        uqqr_int8 = x_int8
    T = dims.T
    x = _np(inp["x"])
    sin = _np(inp["rope_sin"])
    cos = _np(inp["rope_cos"])
    idx = _np(inp["cache_index"]).astype(np.int64)
    sx = _np(inp.get("dequant_scale_x"))
    if tokens is not None:
        tok = np.asarray(_np(tokens), dtype=np.int64)
        x, sin, cos, idx = x[tok], sin[tok], cos[tok], idx[tok]
        if sx is not None:
            sx = sx.reshape(-1)[tok]
        T = len(tok)
    x = np.ascontiguousarray(x)
    sin = np.ascontiguousarray(sin)
    cos = np.ascontiguousarray(cos)
    idx = np.ascontiguousarray(idx)
    if sx is not None:
        sx = np.ascontiguousarray(sx.reshape(-1), dtype=np.float32)

    N, D, Dr, Hckv, Hcq = dims.N, dims.D, dims.Dr, dims.Hckv, dims.Hcq
    res = {
        "q_nope": np.zeros((T, N, Hckv)), "q_rope": np.zeros((T, N, Dr)),
        "kv_cache": _np(inp["kv_cache"]).copy(), "kr_cache": _np(inp["kr_cache"]).copy(),
    }
    if with_intermediates:
        res.update(c_q=np.zeros((T, Hcq)), c_kv=np.zeros((T, Hckv)), k_r=np.zeros((T, Dr)),
                   q_c=np.zeros((T, N, D)))
    if q_int8:
        res.update(q_nope_i8=np.zeros((T, N, Hckv), np.int8), q_nope_scale=np.zeros((T, N)))
    if uqqr_int8:
        res.update(c_q_i8=np.zeros((T, Hcq), np.int8), c_q_scale=np.zeros((T,)))

    keep = {}

    def p(name, arr):
        if arr is None:
            return None
        arr = np.ascontiguousarray(arr)
        keep[name] = arr
        return _ptr(arr)

    def f32(name):
        a = _np(inp.get(name))
        return None if a is None else np.ascontiguousarray(a.reshape(-1), dtype=np.float32)

    a = _Args()
    for k in ("He", "Hcq", "N", "D", "Dr", "Hckv", "block_num", "block_size"):
        setattr(a, k, int(getattr(dims, k)))
    a.T = T
    a.eps_cq, a.eps_ckv = float(eps_cq), float(eps_ckv)
    a.x_int8, a.uqqr_int8, a.kv_int8, a.kr_int8, a.q_int8 = map(int, (x_int8, uqqr_int8, kv_int8, kr_int8, q_int8))
    a.num_threads = int(num_threads)
    a.x = p("x", x)
    a.w_dq = p("w_dq", _np(inp["w_dq"]))
    a.w_uqqr = p("w_uqqr", _np(inp["w_uqqr"]))
    a.w_uk = p("w_uk", _np(inp["w_uk"]))
    a.w_dkvkr = p("w_dkvkr", _np(inp["w_dkvkr"]))
    a.gamma_cq = p("gamma_cq", _np(inp["gamma_cq"]))
    a.gamma_ckv = p("gamma_ckv", _np(inp["gamma_ckv"]))
    a.rope_sin = p("sin", sin)
    a.rope_cos = p("cos", cos)
    a.cache_index = p("idx", idx)
    a.dequant_scale_x = p("sx", sx)
    for k in ("dequant_scale_w_dq", "dequant_scale_w_uqqr", "dequant_scale_w_dkvkr", "quant_scale_ckv",
              "quant_scale_ckr", "smooth_scales_cq"):
        setattr(a, k, p(k, f32(k)))
    a.kv_cache = _ptr(res["kv_cache"])
    a.kr_cache = _ptr(res["kr_cache"])
    for k in ("q_nope", "q_rope", "c_q", "c_kv", "k_r", "q_c", "q_nope_i8", "q_nope_scale", "c_q_i8", "c_q_scale"):
        setattr(a, k, _ptr(res.get(k)))
    rc = lib().mla_oracle_prolog(ctypes.byref(a))
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"oracle error {rc}"))
    return res
