"""GB300 (sm_103a) Multi-Head Latent Attention prolog.

Thin Python binding over the C ABI of ``include/mla_prolog.h`` and
``include/mla_preprocess.h``: the functions below
have the C names and only marshal arguments (torch tensors -> ``mla_tensor``
descriptors).  Every step of the prolog runs in the CUDA kernels of
``libmla_prolog.so``; there is no CPU path.  If the library is missing, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

__all__ = [
    "MlaError", "TENSOR_ARGS", "lib", "mla_prolog_workspace_size", "mla_prolog",
    "mla_prolog_device_status", "mla_prolog_status_string", "STATUS", "DEV_CACHE_INDEX_RANGE",
    "DEV_WAIT_TIMEOUT", "library_path", "mla_prolog_timing_enable", "mla_prolog_timing_read",
    "mla_prolog_no_alloc", "mla_prolog_no_alloc_status", "NO_ALLOC_SCRATCH_BYTES", "PP_TENSOR_ARGS", "PP_OUTPUT_ARGS",
    "mla_preprocess_workspace_size", "mla_preprocess", "mla_prolog_debug_wait_probe",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libmla_prolog.so")

STATUS = {0: "MLA_OK", 161001: "MLA_ERR_PARAM_NULLPTR", 161002: "MLA_ERR_PARAM_INVALID",
          361001: "MLA_ERR_RUNTIME", 561002: "MLA_ERR_TILING", 561003: "MLA_ERR_SCRATCH_LIMIT"}
DEV_CACHE_INDEX_RANGE = 0x1
DEV_WAIT_TIMEOUT = 0x2
# Size of the library's fixed scratch buffer behind mla_prolog_no_alloc (MLA_NO_ALLOC_SCRATCH_BYTES).
NO_ALLOC_SCRATCH_BYTES = 16 << 20

# Positional order of the tensor arguments of the C entry points (before the scalars).
TENSOR_ARGS = ("x", "w_dq", "w_uqqr", "w_uk", "w_dkvkr", "gamma_cq", "gamma_ckv", "rope_sin", "rope_cos",
               "cache_index", "kv_cache", "kr_cache", "dequant_scale_x", "dequant_scale_w_dq",
               "dequant_scale_w_uqqr", "dequant_scale_w_dkvkr", "quant_scale_ckv", "quant_scale_ckr",
               "smooth_scales_cq")
OUTPUT_ARGS = ("q_out", "q_rope_out", "dequant_scale_q_nope_out")

# mla_preprocess (the aclnnMlaPreprocess variant): tensor arguments in the header's order.
PP_TENSOR_ARGS = ("input", "gamma0", "beta0", "quant_scale0", "quant_offset0", "wdqkv", "de_scale0", "bias0",
                  "gamma1", "beta1", "quant_scale1", "quant_offset1", "wuq", "de_scale1", "bias1", "gamma2",
                  "cos", "sin", "wuk", "kv_cache", "kv_cache_rope", "slot_mapping", "ctkv_scale", "q_nope_scale")
PP_OUTPUT_ARGS = ("q_out", "kv_cache_out", "q_rope_out", "kr_cache_out")


class MlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)} ({code})")
        self.code = code


class MlaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4)]


class MlaKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("ms", ctypes.c_float)]


_lib = None


def lib():
    """Load libmla_prolog.so (fails loudly when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is missing: build it with attention_pre_processing_gb300.build.build()")
        L = ctypes.CDLL(library_path)
        P = ctypes.POINTER(MlaTensor)
        tens = [P] * len(TENSOR_ARGS)
        scal = [ctypes.c_double, ctypes.c_double, ctypes.c_char_p]
        outs = [P] * len(OUTPUT_ARGS)
        L.mla_prolog_workspace_size.argtypes = tens + scal + outs + [ctypes.POINTER(ctypes.c_uint64)]
        L.mla_prolog_workspace_size.restype = ctypes.c_int
        L.mla_prolog.argtypes = tens + scal + outs + [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
        L.mla_prolog.restype = ctypes.c_int
        L.mla_prolog_no_alloc.argtypes = tens + scal + outs + [ctypes.c_void_p]
        L.mla_prolog_no_alloc.restype = ctypes.c_int
        L.mla_prolog_device_status.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                                               ctypes.POINTER(ctypes.c_uint32)]
        L.mla_prolog_no_alloc_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
        L.mla_prolog_no_alloc_status.restype = ctypes.c_int
        L.mla_prolog_device_status.restype = ctypes.c_int
        L.mla_prolog_debug_wait_probe.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p]
        L.mla_prolog_debug_wait_probe.restype = ctypes.c_int
        L.mla_prolog_timing_enable.argtypes = [ctypes.c_int]
        L.mla_prolog_timing_enable.restype = ctypes.c_int
        L.mla_prolog_timing_read.argtypes = [ctypes.POINTER(MlaKernelTime), ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        L.mla_prolog_timing_read.restype = ctypes.c_int
        L.mla_prolog_status_string.argtypes = [ctypes.c_int]
        L.mla_prolog_status_string.restype = ctypes.c_char_p
        pp_scal = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                   ctypes.c_int64]
        pp_t = [P] * len(PP_TENSOR_ARGS)
        pp_o = [P] * len(PP_OUTPUT_ARGS)
        L.mla_preprocess_workspace_size.argtypes = pp_t + pp_scal + pp_o + [ctypes.POINTER(ctypes.c_uint64)]
        L.mla_preprocess_workspace_size.restype = ctypes.c_int
        L.mla_preprocess.argtypes = pp_t + pp_scal + pp_o + [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
        L.mla_preprocess.restype = ctypes.c_int
        _lib = L
    return _lib


def _dtype_code(t) -> int:
    import torch
    codes = {torch.bfloat16: 0, torch.int8: 1, torch.float32: 2, torch.int64: 3, torch.float16: 4, torch.int32: 5}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def describe(t) -> Optional[MlaTensor]:
    """torch tensor -> mla_tensor descriptor (no copy; the tensor must stay alive)."""
    if t is None:
        return None
    if isinstance(t, MlaTensor):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    if t.dim() < 1 or t.dim() > 4:
        raise ValueError("tensors have 1 to 4 dimensions")
    d = MlaTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _dtype_code(t)
    d.ndim = t.dim()
    for i, s in enumerate(t.shape):
        d.shape[i] = int(s)
    return d


def _marshal(tensors: Dict, eps_cq: float, eps_ckv: float, cache_mode: Optional[str]):
    descs = [describe(tensors.get(k)) for k in TENSOR_ARGS]
    outs = [describe(tensors.get(k)) for k in OUTPUT_ARGS]
    ptrs = [ctypes.byref(d) if d is not None else None for d in descs]
    optrs = [ctypes.byref(d) if d is not None else None for d in outs]
    cm = None if cache_mode is None else cache_mode.encode()
    return ptrs + [float(eps_cq), float(eps_ckv), cm] + optrs, (descs, outs)


def mla_prolog_workspace_size(tensors: Dict, eps_cq: float, eps_ckv: float,
                              cache_mode: Optional[str] = "PA_BSND") -> int:
    """Phase 1: bytes of device workspace for these arguments (raises MlaError on a bad argument)."""
    args, _keep = _marshal(tensors, eps_cq, eps_ckv, cache_mode)
    out = ctypes.c_uint64(0)
    rc = lib().mla_prolog_workspace_size(*args, ctypes.byref(out))
    if rc != 0:
        raise MlaError(rc, "mla_prolog_workspace_size")
    return int(out.value)


def _ptr(x) -> int:
    return x if isinstance(x, int) else x.data_ptr()


def mla_prolog(tensors: Dict, eps_cq: float, eps_ckv: float, workspace, workspace_bytes: Optional[int] = None,
               stream=None, cache_mode: Optional[str] = "PA_BSND", check: bool = True) -> int:
    """Phase 2: enqueue the prolog on ``stream`` (a torch.cuda.Stream, a raw handle, or None for
    torch's current stream).  ``workspace`` is a device tensor or address."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    args, _keep = _marshal(tensors, eps_cq, eps_ckv, cache_mode)
    rc = lib().mla_prolog(*args, ctypes.c_void_p(_ptr(workspace)), ctypes.c_uint64(workspace_bytes),
                          ctypes.c_void_p(stream))
    if check and rc != 0:
        raise MlaError(rc, "mla_prolog")
    return rc


def mla_prolog_no_alloc(tensors: Dict, eps_cq: float, eps_ckv: float, stream=None,
                        cache_mode: Optional[str] = "PA_BSND", check: bool = True) -> int:
    """mla_prolog without a workspace argument, for callers that cannot allocate device memory:
    the library runs the same kernels on its own fixed scratch buffer (NO_ALLOC_SCRATCH_BYTES
    per device).  Calls that overlap on the GPU share that buffer and race; the first call on a
    device looks the buffer up and belongs before any stream capture."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    args, _keep = _marshal(tensors, eps_cq, eps_ckv, cache_mode)
    rc = lib().mla_prolog_no_alloc(*args, ctypes.c_void_p(stream))
    if check and rc != 0:
        raise MlaError(rc, "mla_prolog_no_alloc")
    return rc


def mla_prolog_no_alloc_status(stream=None) -> int:
    """Wait for the stream and return the device status bits of the last mla_prolog_no_alloc
    call on the current device (read from the library's scratch buffer)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    bits = ctypes.c_uint32(0)
    rc = lib().mla_prolog_no_alloc_status(ctypes.c_void_p(stream), ctypes.byref(bits))
    if rc != 0:
        raise MlaError(rc, "mla_prolog_no_alloc_status")
    return int(bits.value)


def mla_prolog_device_status(workspace, workspace_bytes: Optional[int] = None, stream=None) -> int:
    """Wait for the stream and return the device status bits of the last call on ``workspace``."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    bits = ctypes.c_uint32(0)
    rc = lib().mla_prolog_device_status(ctypes.c_void_p(_ptr(workspace)), ctypes.c_uint64(workspace_bytes),
                                        ctypes.c_void_p(stream), ctypes.byref(bits))
    if rc != 0:
        raise MlaError(rc, "mla_prolog_device_status")
    return int(bits.value)


def mla_prolog_debug_wait_probe(workspace, which: int, workspace_bytes: Optional[int] = None, stream=None) -> None:
    """Enqueue the failure-detection probe (a wait nothing satisfies; see mla_prolog.h)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib().mla_prolog_debug_wait_probe(ctypes.c_void_p(_ptr(workspace)), ctypes.c_uint64(workspace_bytes),
                                           int(which), ctypes.c_void_p(stream))
    if rc != 0:
        raise MlaError(rc, "mla_prolog_debug_wait_probe")


def mla_prolog_timing_enable(enable: bool) -> None:
    lib().mla_prolog_timing_enable(1 if enable else 0)


def mla_prolog_timing_read():
    """[(kernel name, ms), ...] of the most recent call made while timing was enabled."""
    buf = (MlaKernelTime * 16)()
    n = ctypes.c_int(0)
    rc = lib().mla_prolog_timing_read(buf, 16, ctypes.byref(n))
    if rc != 0:
        raise MlaError(rc, "mla_prolog_timing_read")
    return [(buf[i].name.decode(), float(buf[i].ms)) for i in range(min(n.value, 16))]


def mla_prolog_status_string(code: int) -> str:
    return lib().mla_prolog_status_string(int(code)).decode()


# ------------------------------------------------------------ the aclnnMlaPreprocess variant

def _pp_marshal(tensors: Dict, epsilon: float, cache_mode: int, do_rmsnorm: bool, wdq_dim: Optional[int],
                q_rope_dim: int, k_rope_dim: int, q_rotary_coeff: int, k_rotary_coeff: int, transpose_wdq: bool,
                transpose_wuq: bool, transpose_wuk: bool, quant_mode: int, wdkv_split_count: int):
    t = dict(tensors)
    t.setdefault("kv_cache_out", t.get("kv_cache"))
    t.setdefault("kr_cache_out", t.get("kv_cache_rope"))
    if wdq_dim is None:
        g1 = t.get("gamma1")
        wdq_dim = 0 if g1 is None else int(g1.shape[g1.ndim - 1] if isinstance(g1, MlaTensor) else g1.shape[-1])
    descs = [describe(t.get(k)) for k in PP_TENSOR_ARGS]
    outs = [describe(t.get(k)) for k in PP_OUTPUT_ARGS]
    ptrs = [ctypes.byref(d) if d is not None else None for d in descs]
    optrs = [ctypes.byref(d) if d is not None else None for d in outs]
    scal = [int(wdq_dim), int(q_rope_dim), int(k_rope_dim), float(epsilon), int(q_rotary_coeff), int(k_rotary_coeff),
            int(bool(transpose_wdq)), int(bool(transpose_wuq)), int(bool(transpose_wuk)), int(cache_mode),
            int(quant_mode), int(bool(do_rmsnorm)), int(wdkv_split_count)]
    return ptrs + scal + optrs, (descs, outs)


def mla_preprocess_workspace_size(tensors: Dict, epsilon: float, cache_mode: int = 0, do_rmsnorm: bool = True,
                                  wdq_dim: Optional[int] = None, q_rope_dim: int = 64, k_rope_dim: int = 64,
                                  q_rotary_coeff: int = 2, k_rotary_coeff: int = 2, transpose_wdq: bool = True,
                                  transpose_wuq: bool = True, transpose_wuk: bool = True, quant_mode: int = 0,
                                  wdkv_split_count: int = 1) -> int:
    """Phase 1 of the aclnnMlaPreprocess variant (raises MlaError on a bad argument).  ``tensors``
    holds PP_TENSOR_ARGS and PP_OUTPUT_ARGS by name; kv_cache_out / kr_cache_out default to
    kv_cache / kv_cache_rope; wdq_dim defaults to gamma1's length."""
    args, _keep = _pp_marshal(tensors, epsilon, cache_mode, do_rmsnorm, wdq_dim, q_rope_dim, k_rope_dim,
                              q_rotary_coeff, k_rotary_coeff, transpose_wdq, transpose_wuq, transpose_wuk,
                              quant_mode, wdkv_split_count)
    out = ctypes.c_uint64(0)
    rc = lib().mla_preprocess_workspace_size(*args, ctypes.byref(out))
    if rc != 0:
        raise MlaError(rc, "mla_preprocess_workspace_size")
    return int(out.value)


def mla_preprocess(tensors: Dict, epsilon: float, workspace, workspace_bytes: Optional[int] = None, stream=None,
                   cache_mode: int = 0, do_rmsnorm: bool = True, check: bool = True, **scalars) -> int:
    """Phase 2: enqueue the variant on ``stream`` (torch.cuda.Stream, raw handle, or None for torch's
    current stream).  Further scalars (wdq_dim, q_rope_dim, ...) as in mla_preprocess_workspace_size."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    kw = dict(wdq_dim=None, q_rope_dim=64, k_rope_dim=64, q_rotary_coeff=2, k_rotary_coeff=2, transpose_wdq=True,
              transpose_wuq=True, transpose_wuk=True, quant_mode=0, wdkv_split_count=1)
    kw.update(scalars)
    args, _keep = _pp_marshal(tensors, epsilon, cache_mode, do_rmsnorm, **kw)
    rc = lib().mla_preprocess(*args, ctypes.c_void_p(_ptr(workspace)), ctypes.c_uint64(workspace_bytes),
                              ctypes.c_void_p(stream))
    if check and rc != 0:
        raise MlaError(rc, "mla_preprocess")
    return rc
