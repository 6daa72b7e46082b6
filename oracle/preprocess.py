"""CPU oracle for the aclnnMlaPreprocess variant of the MLA prolog (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs import
this module.  The product library never imports it and it imports nothing of
the product; it reads the seeded inputs of
``attention_pre_processing_gb300.workloads.make_pp_inputs`` that the callers
pass in.

The page "aclnnMlaPreprocess" (Function description; Formula) describes the
computation as six paths after one fused down-projection:

  x' = RmsNormQuant(x)                  (gamma0, beta0, quantScale0, quantOffset0)
  y  = x' . W^DQKV                      (int8 x int8, bias0 added, deScale0 applied)
  path 1: y[:Hcq] -> RmsNormQuant (gamma1, beta1, quantScale1, quantOffset1) -> . W^UQ
          (bias1, deScale1) -> z, viewed (N, qNoRopeDim + qRopeDim)
  path 3: q^N = z[:, :D] . W^UK[n]      path 4: q^R = RoPE(z[:, D:])
  path 5: k^N = RmsNorm(y[Hcq:Hcq+512]) (gamma2) -> cache
  path 6: k^R = RoPE(y[Hcq+512:]) -> cache

with RmsNorm(x) = gamma * x_i / sqrt(mean(x^2) + eps) and
RmsNormQuant(x) = (RmsNorm(x) + bias) * scale (same page, Formula).  Everything is
computed in fp64 from the exact input values; nothing is rounded between steps
except the two int8 quantisers the method itself applies, and the outputs and
cache rows, which are rounded to the input's dtype once at the end.

Readings of points the page leaves open (each also stated at the function):
  * quantisation code: q = clamp(round_half_away(v * quantScale) + quantOffset, -128, 127)
    (per-tensor static asymmetric int8, quantMode 0);
  * doRmsNorm = False: the input is only quantised, q = clamp(round_half_away(x * quantScale0)
    + quantOffset0, -128, 127); beta0 belongs to the norm and is not added;
  * the int8 products: y[j] = (sum_k x'[k] * W[j, k] + bias0[j]) * deScale0[j], one scale per
    output column (deScale0 has one entry per column), bias0 absent = 0;
  * one epsilon for all three norms (the page has a single epsilon);
  * RoPE: the half rotation of the page's Constraints (RoPE mode), full-width cos/sin tables.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np


# ---------------------------------------------------------------- exact value conversion

def to_f64(t) -> Optional[np.ndarray]:
    """torch / numpy tensor -> float64 numpy array holding the exact same values."""
    if t is None:
        return None
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                bits = t.view(torch.int16).numpy().view(np.uint16).astype(np.uint32) << 16
                return bits.view(np.float32).astype(np.float64)
            return t.numpy().astype(np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t).astype(np.float64)


def round_half_away(v) -> np.ndarray:
    """Nearest integer, halves away from zero, without the v + 0.5 rounding trap."""
    v = np.asarray(v, dtype=np.float64)
    r = np.trunc(v)
    frac = np.abs(v - r)            # exact: v and its integer part share the exponent range
    return r + np.sign(v) * (frac >= 0.5)


def round_to_dtype(v, dtype: str) -> np.ndarray:
    """fp64 -> the bits of bf16 or fp16, round to nearest even in one step (uint16 array)."""
    v = np.asarray(v, dtype=np.float64)
    if dtype == "fp16":
        return v.astype(np.float16).view(np.uint16)   # numpy rounds double -> half directly
    import oracle
    return oracle.bf16_rne(v)


def bits_to_f64(bits, dtype: str) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- the steps

def rmsnorm(y, gamma, eps: float) -> np.ndarray:
    """gamma * y / sqrt(mean(y^2) + eps) over the last axis ("aclnnMlaPreprocess", Formula:
    RMS(x) and RmsNorm(x); epsilon inside the root)."""
    y = np.asarray(y, dtype=np.float64)
    return gamma * y / np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + eps)


def quant_i8(v, scale: float, offset: int) -> np.ndarray:
    """Static per-tensor asymmetric int8 code: clamp(round_half_away(v * scale) + offset, -128, 127)."""
    q = round_half_away(np.asarray(v, dtype=np.float64) * scale) + offset
    return np.clip(q, -128, 127).astype(np.int64)


def rmsnorm_quant(x, gamma, beta, scale: float, offset: int, eps: float, do_rmsnorm: bool = True) -> np.ndarray:
    """RmsNormQuant(x) = (RmsNorm(x) + beta) * scale, then the int8 code ("aclnnMlaPreprocess",
    Formula: RmsNormQuant).  With do_rmsnorm False (the doRmsNorm parameter) only the
    quantiser is applied to x."""
    v = rmsnorm(x, gamma, eps) + beta if do_rmsnorm else np.asarray(x, dtype=np.float64)
    return quant_i8(v, scale, offset)


def dequant_matmul(a_codes, w_rows, bias, scale) -> np.ndarray:
    """(a . W^T + bias) * scale for int8 codes a (T, K) and a weight stored one row per output
    column, W (ncols, K) ("transposeWdq" / "transposeWuq" true).  Integer sums are exact in fp64
    (|sum| < 2^53); bias (ncols) int32 or None; scale (ncols) one per output column."""
    acc = np.asarray(a_codes, dtype=np.float64) @ np.asarray(w_rows, dtype=np.float64).T
    if bias is not None:
        acc = acc + np.asarray(bias, dtype=np.float64)
    return acc * np.asarray(scale, dtype=np.float64)


def rope_half(v, cos, sin) -> np.ndarray:
    """out = v * cos + rotate_half(v) * sin, rotate_half(v) = [-v[h:], v[:h]] ("aclnnMlaPreprocess",
    Constraints: RoPE half mode, no interleave)."""
    v = np.asarray(v, dtype=np.float64)
    h = v.shape[-1] // 2
    rot = np.concatenate([-v[..., h:], v[..., :h]], axis=-1)
    return v * cos + rot * sin


# ---------------------------------------------------------------- the whole call

def preprocess(inp: Dict, *, dtype: str, cache_mode: int, do_rmsnorm: bool, eps: float,
               tokens=None) -> Dict[str, np.ndarray]:
    """Run the variant on the inputs of ``workloads.make_pp_inputs`` (torch tensors).

    With ``tokens`` (index list) only those tokens are computed and only their cache rows
    written (every step is per token).  Returns the fp64 results before output rounding
    (q_nope (T, N, Hckv), q_rope (T, N, Dr), k_nope (T, Hckv), k_rope (T, Dr)), the int8
    codes of both quantisers (x_codes, cq_codes), y and z, the q output rows as the page lays
    them out for ``cache_mode`` (q_out: (T, N, Hckv + Dr) for 0, (T, N, Hckv) for 1, plus
    q_rope_out for 1), and copies of the caches (uint16 bits) with this call's rows written.
    """
    x = to_f64(inp["input"])
    cos, sin = to_f64(inp["cos"]), to_f64(inp["sin"])
    slots = to_f64(inp["slot_mapping"]).astype(np.int64)
    if tokens is not None:
        tok = np.asarray(tokens, dtype=np.int64)
        x, cos, sin, slots = x[tok], cos[tok], sin[tok], slots[tok]
    T = x.shape[0]
    gamma2 = to_f64(inp["gamma2"])
    Hckv = gamma2.shape[0]
    Dr = cos.shape[1]
    wuk = to_f64(inp["wuk"])
    N, D = wuk.shape[0], wuk.shape[1]
    Hcq = to_f64(inp["gamma1"]).shape[0]
    qs0, qo0 = float(to_f64(inp["quant_scale0"])[0]), int(to_f64(inp["quant_offset0"])[0])
    qs1, qo1 = float(to_f64(inp["quant_scale1"])[0]), int(to_f64(inp["quant_offset1"])[0])

    # first RmsNormQuant and the fused down-projection
    x_codes = rmsnorm_quant(x, to_f64(inp["gamma0"]), to_f64(inp["beta0"]), qs0, qo0, eps, do_rmsnorm)
    y = dequant_matmul(x_codes, to_f64(inp["wdqkv"]), to_f64(inp.get("bias0")), to_f64(inp["de_scale0"]))
    # path 1: second RmsNormQuant, up-projection
    cq_codes = rmsnorm_quant(y[:, :Hcq], to_f64(inp["gamma1"]), to_f64(inp["beta1"]), qs1, qo1, eps, True)
    z = dequant_matmul(cq_codes, to_f64(inp["wuq"]), to_f64(inp.get("bias1")), to_f64(inp["de_scale1"]))
    z = z.reshape(T, N, D + Dr)
    # paths 3 and 4
    q_nope = np.einsum("tnd,ndc->tnc", z[:, :, :D], wuk)
    q_rope = rope_half(z[:, :, D:], cos[:, None, :], sin[:, None, :])
    # paths 5 and 6
    k_nope = rmsnorm(y[:, Hcq:Hcq + Hckv], gamma2, eps)
    k_rope = rope_half(y[:, Hcq + Hckv:Hcq + Hckv + Dr], cos, sin)

    res = {"x_codes": x_codes, "y": y, "cq_codes": cq_codes, "z": z, "q_nope": q_nope, "q_rope": q_rope,
           "k_nope": k_nope, "k_rope": k_rope}

    def cache_bits(t):
        import torch
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()

    kv = cache_bits(inp["kv_cache"])
    nslots = kv.shape[0] * kv.shape[1]
    kv = kv.reshape(nslots, kv.shape[-1])
    if cache_mode == 0:
        res["q_out"] = np.concatenate([q_nope, q_rope], axis=-1)
        rows = np.concatenate([k_nope, k_rope], axis=-1)
        if nslots > 0:
            assert len(set(slots.tolist())) == len(slots), "slotMapping values must be distinct"
            assert slots.min(initial=0) >= 0 and slots.max(initial=0) < nslots, "slotMapping out of range"
            kv[slots] = round_to_dtype(rows, dtype)
        res["kv_cache"] = kv.reshape(cache_bits(inp["kv_cache"]).shape)
    else:
        res["q_out"] = q_nope
        res["q_rope_out"] = q_rope
        kr = cache_bits(inp["kv_cache_rope"])
        kr = kr.reshape(nslots, kr.shape[-1])
        if nslots > 0:
            assert len(set(slots.tolist())) == len(slots), "slotMapping values must be distinct"
            assert slots.min(initial=0) >= 0 and slots.max(initial=0) < nslots, "slotMapping out of range"
            kv[slots] = round_to_dtype(k_nope, dtype)
            kr[slots] = round_to_dtype(k_rope, dtype)
        res["kv_cache"] = kv.reshape(cache_bits(inp["kv_cache"]).shape)
        res["kv_cache_rope"] = kr.reshape(cache_bits(inp["kv_cache_rope"]).shape)
    return res


def for_config(cfg, inp, tokens=None) -> Dict[str, np.ndarray]:
    """``preprocess`` with the switches of a ``workloads.PpConfig``."""
    return preprocess(inp, dtype=cfg.dtype, cache_mode=cfg.cache_mode, do_rmsnorm=cfg.do_rmsnorm, eps=cfg.eps,
                      tokens=tokens)
