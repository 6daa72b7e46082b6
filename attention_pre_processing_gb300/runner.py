"""Device-side plumbing around the C ABI: places a workload's inputs in device memory,
allocates outputs and the workspace with torch, and enqueues calls.  No arithmetic of the
prolog happens here; every step runs in libmla_prolog.so."""
from __future__ import annotations

import ctypes
from typing import Dict, Optional

import torch

from . import _marshal, _pp_marshal, lib, MlaError, mla_prolog_device_status, mla_prolog_workspace_size
from . import mla_preprocess_workspace_size
from .workloads import MlaConfig, PpConfig

INPUT_KEYS = ("x", "w_dq", "w_uqqr", "w_uk", "w_dkvkr", "gamma_cq", "gamma_ckv", "rope_sin", "rope_cos",
              "cache_index", "kv_cache", "kr_cache", "dequant_scale_x", "dequant_scale_w_dq",
              "dequant_scale_w_uqqr", "dequant_scale_w_dkvkr", "quant_scale_ckv", "quant_scale_ckr",
              "smooth_scales_cq")


class PrologCall:
    """One configured call: device tensors, outputs and workspace, reusable across launches.

    With ``bs = (B, S)`` (B * S = T) the per-token tensors are passed in the page's
    non-concatenated layout: tokenX (B, S, He), ropeSin / ropeCos (B, S, Dr), cacheIndex (B, S),
    queryOut (B, S, N, Hckv), queryRopeOut (B, S, N, Dr) and dequantScaleQNopeOut (B*S, N, 1).

    With ``packed_io`` the per-token inputs (tokenX, ropeSin, ropeCos, cacheIndex) are views of one
    device buffer ``io_in`` and the outputs (queryOut, queryRopeOut and, for int8 q^N, its scales)
    views of one buffer ``io_out`` (each piece 256-byte aligned), so that a step's inputs and
    results cross the host link in one copy each way.
    """

    IO_IN = ("x", "rope_sin", "rope_cos", "cache_index")
    IO_OUT = ("q_out", "q_rope_out", "dequant_scale_q_nope_out")

    def __init__(self, cfg: MlaConfig, inputs: Dict[str, Optional[torch.Tensor]], device="cuda", bs=None,
                 packed_io: bool = False):
        s = cfg.shape
        self.cfg = cfg
        self.t: Dict[str, Optional[torch.Tensor]] = {}
        for k in INPUT_KEYS:
            v = inputs.get(k)
            self.t[k] = None if v is None else v.to(device).contiguous()
        lead = (s.T,)
        if bs is not None:
            B, S = bs
            if B * S != s.T:
                raise ValueError(f"B * S = {B * S} != T = {s.T}")
            lead = (B, S)
            self.t["x"] = self.t["x"].view(B, S, s.He)
            self.t["rope_sin"] = self.t["rope_sin"].view(B, S, s.Dr)
            self.t["rope_cos"] = self.t["rope_cos"].view(B, S, s.Dr)
            self.t["cache_index"] = self.t["cache_index"].view(B, S)
        q_dtype = torch.int8 if cfg.q_int8 else torch.bfloat16
        self.t["q_out"] = torch.empty(lead + (s.N, s.Hckv), dtype=q_dtype, device=device)
        self.t["q_rope_out"] = torch.empty(lead + (s.N, s.Dr), dtype=torch.bfloat16, device=device)
        self.t["dequant_scale_q_nope_out"] = (torch.empty((s.T, s.N, 1), dtype=torch.float32, device=device)
                                              if cfg.q_int8 else None)
        self.io_in = self.io_out = None
        if packed_io:
            self.io_in = self._pack(self.IO_IN, device, copy=True)
            self.io_out = self._pack(self.IO_OUT, device, copy=False)
        self.ws_bytes = mla_prolog_workspace_size(self.t, cfg.eps_cq, cfg.eps_ckv)
        self.workspace = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        # The tensors stay put between calls: their descriptors are marshalled once.
        args, self._keep = _marshal(self.t, cfg.eps_cq, cfg.eps_ckv, "PA_BSND")
        self._args = tuple(args) + (ctypes.c_void_p(self.workspace.data_ptr()), ctypes.c_uint64(self.ws_bytes))
        self._fn = lib().mla_prolog

    def _pack(self, keys, device, copy: bool) -> torch.Tensor:
        """One byte buffer holding the tensors ``keys`` (the present ones) as aligned views."""
        present = [k for k in keys if self.t.get(k) is not None]
        offs, off = [], 0
        for k in present:
            offs.append(off)
            off += (self.t[k].numel() * self.t[k].element_size() + 255) // 256 * 256
        buf = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
        for k, o in zip(present, offs):
            old = self.t[k]
            n = old.numel() * old.element_size()
            view = buf[o:o + n].view(old.dtype).view(old.shape)
            if copy:
                view.copy_(old)
            self.t[k] = view
        return buf

    def __call__(self, stream=None) -> None:
        if stream is None:
            stream = torch.cuda.current_stream()
        h = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
        rc = self._fn(*self._args, ctypes.c_void_p(h))
        if rc != 0:
            raise MlaError(rc, "mla_prolog")

    def status(self, stream=None) -> int:
        return mla_prolog_device_status(self.workspace, self.ws_bytes, stream=stream)

    def outputs(self) -> Dict[str, Optional[torch.Tensor]]:
        return {k: self.t[k] for k in ("q_out", "q_rope_out", "dequant_scale_q_nope_out", "kv_cache", "kr_cache")}


PP_INPUT_KEYS = ("input", "gamma0", "beta0", "quant_scale0", "quant_offset0", "wdqkv", "de_scale0", "bias0",
                 "gamma1", "beta1", "quant_scale1", "quant_offset1", "wuq", "de_scale1", "bias1", "gamma2",
                 "cos", "sin", "wuk", "kv_cache", "kv_cache_rope", "slot_mapping")


class PreprocessCall:
    """One configured call of the aclnnMlaPreprocess variant, reusable across launches."""

    def __init__(self, cfg: PpConfig, inputs: Dict[str, Optional[torch.Tensor]], device="cuda"):
        s = cfg.shape
        self.cfg = cfg
        self.t: Dict[str, Optional[torch.Tensor]] = {}
        for k in PP_INPUT_KEYS:
            v = inputs.get(k)
            self.t[k] = None if v is None else v.to(device).contiguous()
        fdt = self.t["input"].dtype
        qw = s.Hckv + s.Dr if cfg.cache_mode == 0 else s.Hckv
        self.t["q_out"] = torch.empty((s.T, s.N, qw), dtype=fdt, device=device)
        self.t["q_rope_out"] = (torch.empty((s.T, s.N, s.Dr), dtype=fdt, device=device)
                                if cfg.cache_mode == 1 else None)
        self._scal = dict(epsilon=cfg.eps, cache_mode=cfg.cache_mode, do_rmsnorm=cfg.do_rmsnorm, wdq_dim=None,
                          q_rope_dim=64, k_rope_dim=64, q_rotary_coeff=2, k_rotary_coeff=2, transpose_wdq=True,
                          transpose_wuq=True, transpose_wuk=True, quant_mode=0, wdkv_split_count=1)
        self.ws_bytes = mla_preprocess_workspace_size(self.t, **self._scal)
        self.workspace = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        args, self._keep = _pp_marshal(self.t, **self._scal)
        self._args = tuple(args) + (ctypes.c_void_p(self.workspace.data_ptr()), ctypes.c_uint64(self.ws_bytes))
        self._fn = lib().mla_preprocess

    def __call__(self, stream=None) -> None:
        if stream is None:
            stream = torch.cuda.current_stream()
        h = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
        rc = self._fn(*self._args, ctypes.c_void_p(h))
        if rc != 0:
            raise MlaError(rc, "mla_preprocess")

    def status(self, stream=None) -> int:
        return mla_prolog_device_status(self.workspace, self.ws_bytes, stream=stream)
