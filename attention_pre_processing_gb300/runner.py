"""Device-side plumbing around the C ABI: places a workload's inputs in device memory,
allocates outputs and the workspace with torch, and enqueues calls.  No arithmetic of the
prolog happens here; every step runs in libmla_prolog.so."""
from __future__ import annotations

import ctypes
from typing import Dict, Optional

import torch

from . import _marshal, lib, MlaError, mla_prolog_device_status, mla_prolog_workspace_size
from .workloads import MlaConfig

INPUT_KEYS = ("x", "w_dq", "w_uqqr", "w_uk", "w_dkvkr", "gamma_cq", "gamma_ckv", "rope_sin", "rope_cos",
              "cache_index", "kv_cache", "kr_cache", "dequant_scale_x", "dequant_scale_w_dq",
              "dequant_scale_w_uqqr", "dequant_scale_w_dkvkr", "quant_scale_ckv", "quant_scale_ckr",
              "smooth_scales_cq")


class PrologCall:
    """One configured call: device tensors, outputs and workspace, reusable across launches."""

    def __init__(self, cfg: MlaConfig, inputs: Dict[str, Optional[torch.Tensor]], device="cuda"):
        s = cfg.shape
        self.cfg = cfg
        self.t: Dict[str, Optional[torch.Tensor]] = {}
        for k in INPUT_KEYS:
            v = inputs.get(k)
            self.t[k] = None if v is None else v.to(device).contiguous()
        q_dtype = torch.int8 if cfg.q_int8 else torch.bfloat16
        self.t["q_out"] = torch.empty((s.T, s.N, s.Hckv), dtype=q_dtype, device=device)
        self.t["q_rope_out"] = torch.empty((s.T, s.N, s.Dr), dtype=torch.bfloat16, device=device)
        self.t["dequant_scale_q_nope_out"] = (torch.empty((s.T, s.N, 1), dtype=torch.float32, device=device)
                                              if cfg.q_int8 else None)
        self.ws_bytes = mla_prolog_workspace_size(self.t, cfg.eps_cq, cfg.eps_ckv)
        self.workspace = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        # The tensors stay put between calls: their descriptors are marshalled once.
        args, self._keep = _marshal(self.t, cfg.eps_cq, cfg.eps_ckv, "PA_BSND")
        self._args = tuple(args) + (ctypes.c_void_p(self.workspace.data_ptr()), ctypes.c_uint64(self.ws_bytes))
        self._fn = lib().mla_prolog

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
