"""Seeded synthetic inputs for the MLA prolog.

This module only draws numbers.  It holds none of the prolog's arithmetic:
no projection, norm, rotation or quantiser.  The CPU oracle (under
``oracle/``) and the CUDA library both read the tensors it returns, so both
sides see identical bits.

Shapes follow the parameter table of "aclnnMlaPrologV2WeightNz"
(Parameters; Constraints, shape format field description): tokenX (T, He),
weightDq (He, Hcq), weightUqQr (Hcq, N*(D+Dr)), weightUk (N, D, Hckv),
weightDkvKr (He, Hckv+Dr), ropeSin/ropeCos (T, Dr), cacheIndex (T),
kvCache (BlockNum, BlockSize, 1, Hckv), krCache (BlockNum, BlockSize, 1, Dr).

The RoPE tables are inputs of the operator: the op never sees positions.  The
tables are built here the usual way for the "half" rotation that
"aclnnMlaPreprocess" (Constraints, RoPE mode) names: for j < Dr/2,
cos[t, j] = cos[t, j + Dr/2] = cos(pos_t * theta**(-2j/Dr)) and likewise sin.
That is table construction for synthetic data, not the rotation itself.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

__all__ = ["MlaShape", "MlaConfig", "CONFIGS", "config", "make_inputs", "sample_tokens",
           "PpShape", "PpConfig", "PP_CONFIGS", "pp_config", "make_pp_inputs"]


@dataclasses.dataclass(frozen=True)
class MlaShape:
    T: int
    He: int
    Hcq: int
    N: int
    D: int
    Dr: int
    Hckv: int
    block_num: int
    block_size: int


@dataclasses.dataclass(frozen=True)
class MlaConfig:
    """One synthetic workload: shapes, value distributions and scenario."""
    name: str
    shape: MlaShape
    seed: int
    eps_cq: float = 1e-5
    eps_ckv: float = 1e-5
    x_std: float = 1.0
    w_std: float = 0.05
    gamma_lo: float = 0.5
    gamma_hi: float = 1.5
    pos_hi: int = 512
    theta: float = 1e4
    # scenario switches (aclnnMlaPrologV2WeightNz, Constraints: scenario table)
    x_int8: bool = False          # int8 full quantisation of tokenX and the three weights
    uqqr_int8: bool = False       # partial quantisation: weightUqQr alone is int8
    kv_int8: bool = False         # kv cache quantised with quantScaleCkv
    kr_int8: bool = False         # kr cache quantised with quantScaleCkr (partial quantisation)
    smooth: bool = False          # pass smoothScalesCq ~ U(0.5, 1.5)
    q_int8: bool = False          # q^N dynamically quantised to int8 ("fifth path")
    outlier_frac: float = 0.0     # fraction of x elements multiplied by outlier_mult
    outlier_mult: float = 1.0
    # int8 scale distributions
    sx_lo: float = 0.005
    sx_hi: float = 0.02
    sw_lo: float = 1e-4
    sw_hi: float = 1e-3
    ckv_lo: float = 0.01
    ckv_hi: float = 0.05
    ckv_reciprocal: bool = False  # draw quantScaleCkv as 1/U(lo, hi) instead of U(lo, hi)
    # prefill layout: (num_sequences, seq_len) with positions 0..seq_len-1 and contiguous slots
    sequences: Optional[tuple] = None
    w_uk_std: Optional[float] = None

    @property
    def workload(self) -> str:
        s = self.shape
        q = []
        if self.x_int8:
            q.append("int8-in")
        elif self.uqqr_int8:
            q.append("uqqr-int8")
        if self.kv_int8:
            q.append("kv-int8")
        if self.q_int8:
            q.append("qN-int8")
        tag = ",".join(q) if q else "bf16"
        return (f"{self.name}: T={s.T} He={s.He} Hcq={s.Hcq} N={s.N} D={s.D} Dr={s.Dr} "
                f"Hckv={s.Hckv} cache={s.block_num}x{s.block_size} [{tag}]")


_DSV3 = dict(He=7168, Hcq=1536, N=128, D=128, Dr=64, Hckv=512)

CONFIGS: Dict[str, MlaConfig] = {
    # small case the oracle finishes in well under a second
    "tiny": MlaConfig(
        name="tiny",
        shape=MlaShape(T=8, He=256, Hcq=64, N=4, D=32, Dr=16, Hckv=64, block_num=4, block_size=16),
        seed=1000, eps_cq=1e-5, eps_ckv=1e-5, w_std=0.05, gamma_lo=0.5, gamma_hi=1.5, pos_hi=512),
    # DeepSeek-V3-shaped decode, batch 32, one token each
    "decode_t32": MlaConfig(
        name="decode_t32",
        shape=MlaShape(T=32, block_num=1024, block_size=128, **_DSV3),
        seed=1001, eps_cq=1e-6, eps_ckv=1e-6, w_std=0.02, gamma_lo=0.8, gamma_hi=1.2, pos_hi=32768),
    # T=256 with the int8 q^N output and 1% x outliers at 20x
    "decode_t256_qint8": MlaConfig(
        name="decode_t256_qint8",
        shape=MlaShape(T=256, block_num=1024, block_size=128, **_DSV3),
        seed=1002, eps_cq=1e-6, eps_ckv=1e-6, w_std=0.02, gamma_lo=0.8, gamma_hi=1.2, pos_hi=32768,
        q_int8=True, outlier_frac=0.01, outlier_mult=20.0),
    # int8 full quantisation with an int8 kv cache, T=64
    "int8_t64": MlaConfig(
        name="int8_t64",
        shape=MlaShape(T=64, block_num=1024, block_size=128, **_DSV3),
        seed=1003, eps_cq=1e-6, eps_ckv=1e-6, w_std=0.02, gamma_lo=0.8, gamma_hi=1.2, pos_hi=32768,
        x_int8=True, kv_int8=True, q_int8=True),
    # the same with quantScaleCkv drawn as a reciprocal, so that rounding and saturation are exercised
    "int8_t64_recip": MlaConfig(
        name="int8_t64_recip",
        shape=MlaShape(T=64, block_num=1024, block_size=128, **_DSV3),
        seed=1013, eps_cq=1e-6, eps_ckv=1e-6, w_std=0.02, gamma_lo=0.8, gamma_hi=1.2, pos_hi=32768,
        x_int8=True, kv_int8=True, q_int8=True, ckv_reciprocal=True),
    # prefill: 2 sequences x 4096 tokens, contiguous slots in 2 x 128 blocks of 128
    "prefill_t8192": MlaConfig(
        name="prefill_t8192",
        shape=MlaShape(T=8192, block_num=256, block_size=128, **_DSV3),
        seed=1004, eps_cq=1e-6, eps_ckv=1e-6, w_std=0.02, gamma_lo=0.8, gamma_hi=1.2,
        sequences=(2, 4096)),
}


def config(name: str, **overrides) -> MlaConfig:
    """Return a named config, optionally with shape fields or other fields replaced."""
    cfg = CONFIGS[name]
    shape_keys = {f.name for f in dataclasses.fields(MlaShape)}
    shape_over = {k: v for k, v in overrides.items() if k in shape_keys}
    other = {k: v for k, v in overrides.items() if k not in shape_keys}
    if shape_over:
        other["shape"] = dataclasses.replace(cfg.shape, **shape_over)
    return dataclasses.replace(cfg, **other) if other else cfg


def _uniform(gen, shape, lo, hi):
    return torch.rand(shape, generator=gen, dtype=torch.float64) * (hi - lo) + lo


def _randint8(gen, shape, lo=-127, hi=127):
    return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int16).to(torch.int8)


def _random_bits(gen, shape, dtype):
    if dtype == torch.bfloat16:
        return torch.randint(-32768, 32768, shape, generator=gen, dtype=torch.int16).view(torch.bfloat16)
    return torch.randint(-128, 128, shape, generator=gen, dtype=torch.int16).to(torch.int8)


def make_inputs(cfg: MlaConfig, seed: Optional[int] = None) -> Dict[str, Optional[torch.Tensor]]:
    """Draw every input of one call on the CPU, in a fixed order, from one seed.

    Caches come back pre-filled with random bit patterns; those act as the
    sentinel that shows which slots a call wrote.
    """
    s = cfg.shape
    gen = torch.Generator().manual_seed(cfg.seed if seed is None else seed)
    T, He, Hcq, N, D, Dr, Hckv = s.T, s.He, s.Hcq, s.N, s.D, s.Dr, s.Hckv
    out: Dict[str, Optional[torch.Tensor]] = {}

    # tokenX
    if cfg.x_int8:
        out["x"] = _randint8(gen, (T, He))
    else:
        x = torch.randn((T, He), generator=gen, dtype=torch.float32) * cfg.x_std
        if cfg.outlier_frac > 0:
            mask = torch.rand((T, He), generator=gen) < cfg.outlier_frac
            x = torch.where(mask, x * cfg.outlier_mult, x)
        out["x"] = x.to(torch.bfloat16)

    # weights, (k, n) orientation
    def wmat(shape, std):
        if cfg.x_int8:
            return _randint8(gen, shape)
        return (torch.randn(shape, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)

    out["w_dq"] = wmat((He, Hcq), cfg.w_std)
    if cfg.uqqr_int8 and not cfg.x_int8:
        out["w_uqqr"] = _randint8(gen, (Hcq, N * (D + Dr)))
    else:
        out["w_uqqr"] = wmat((Hcq, N * (D + Dr)), cfg.w_std)
    uk_std = cfg.w_uk_std if cfg.w_uk_std is not None else cfg.w_std
    out["w_uk"] = (torch.randn((N, D, Hckv), generator=gen, dtype=torch.float32) * uk_std).to(torch.bfloat16)
    out["w_dkvkr"] = wmat((He, Hckv + Dr), cfg.w_std)

    out["gamma_cq"] = _uniform(gen, (Hcq,), cfg.gamma_lo, cfg.gamma_hi).to(torch.bfloat16)
    out["gamma_ckv"] = _uniform(gen, (Hckv,), cfg.gamma_lo, cfg.gamma_hi).to(torch.bfloat16)

    # positions -> rope tables
    if cfg.sequences is not None:
        nseq, slen = cfg.sequences
        assert nseq * slen == T
        pos = torch.arange(slen, dtype=torch.int64).repeat(nseq)
    else:
        pos = torch.randint(0, cfg.pos_hi, (T,), generator=gen, dtype=torch.int64)
    out["positions"] = pos
    h = Dr // 2
    inv = cfg.theta ** (-2.0 * torch.arange(h, dtype=torch.float64) / Dr)
    ang = pos.to(torch.float64)[:, None] * inv[None, :]
    out["rope_cos"] = torch.cat([torch.cos(ang), torch.cos(ang)], dim=1).to(torch.bfloat16).contiguous()
    out["rope_sin"] = torch.cat([torch.sin(ang), torch.sin(ang)], dim=1).to(torch.bfloat16).contiguous()

    # cache slots
    nslots = s.block_num * s.block_size
    if cfg.sequences is not None:
        nseq, slen = cfg.sequences
        per_seq = nslots // nseq
        assert slen <= per_seq
        idx = (torch.arange(nseq, dtype=torch.int64)[:, None] * per_seq
               + torch.arange(slen, dtype=torch.int64)[None, :]).reshape(-1)
    elif nslots == 0:
        # Skv = 0: no cache to write; the slot values are never used
        idx = torch.zeros(T, dtype=torch.int64)
    else:
        assert T <= nslots
        idx = torch.randperm(nslots, generator=gen)[:T].to(torch.int64)
    out["cache_index"] = idx.contiguous()

    # caches pre-filled with random bits (the sentinel)
    kv_dtype = torch.int8 if cfg.kv_int8 else torch.bfloat16
    out["kv_cache"] = _random_bits(gen, (s.block_num, s.block_size, 1, Hckv), kv_dtype)
    kr_dtype = torch.int8 if cfg.kr_int8 else torch.bfloat16
    out["kr_cache"] = _random_bits(gen, (s.block_num, s.block_size, 1, Dr), kr_dtype)

    # scales (aclnnMlaPrologV2WeightNz, Constraints: scenario table)
    for k in ("dequant_scale_x", "dequant_scale_w_dq", "dequant_scale_w_uqqr",
              "dequant_scale_w_dkvkr", "quant_scale_ckv", "quant_scale_ckr", "smooth_scales_cq"):
        out[k] = None
    if cfg.x_int8:
        out["dequant_scale_x"] = _uniform(gen, (T, 1), cfg.sx_lo, cfg.sx_hi).to(torch.float32)
        out["dequant_scale_w_dq"] = _uniform(gen, (1, Hcq), cfg.sw_lo, cfg.sw_hi).to(torch.float32)
        out["dequant_scale_w_uqqr"] = _uniform(gen, (1, N * (D + Dr)), cfg.sw_lo, cfg.sw_hi).to(torch.float32)
        out["dequant_scale_w_dkvkr"] = _uniform(gen, (1, Hckv + Dr), cfg.sw_lo, cfg.sw_hi).to(torch.float32)
    elif cfg.uqqr_int8:
        out["dequant_scale_w_uqqr"] = _uniform(gen, (1, N * (D + Dr)), cfg.sw_lo, cfg.sw_hi).to(torch.float32)
    if cfg.kv_int8:
        qs = _uniform(gen, (1, Hckv), cfg.ckv_lo, cfg.ckv_hi)
        if cfg.ckv_reciprocal:
            qs = 1.0 / qs
        out["quant_scale_ckv"] = qs.to(torch.float32)
    if cfg.kr_int8:
        qs = _uniform(gen, (1, Dr), cfg.ckv_lo, cfg.ckv_hi)
        if cfg.ckv_reciprocal:
            qs = 1.0 / qs
        out["quant_scale_ckr"] = qs.to(torch.float32)
    if cfg.smooth and (cfg.x_int8 or cfg.uqqr_int8):
        out["smooth_scales_cq"] = _uniform(gen, (1, Hcq), 0.5, 1.5).to(torch.float32)
    return out


def sample_tokens(T: int, k: int, seed: int = 7) -> torch.Tensor:
    """A sorted, seeded sample of k token indices out of T, always holding the first and last."""
    if k >= T:
        return torch.arange(T, dtype=torch.int64)
    gen = torch.Generator().manual_seed(seed)
    mid = torch.randperm(T - 2, generator=gen)[: max(k - 2, 0)] + 1
    idx = torch.cat([torch.tensor([0, T - 1]), mid]).unique(sorted=True)
    return idx.to(torch.int64)


def nbytes(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def flops_per_token(s: MlaShape) -> int:
    """Multiply-adds x 2 of the three contractions, per token."""
    return 2 * (s.He * (s.Hcq + s.Hckv + s.Dr) + s.Hcq * s.N * (s.D + s.Dr) + s.N * s.D * s.Hckv)


# ------------------------------------------------------------------ the aclnnMlaPreprocess variant
#
# Shapes follow "aclnnMlaPreprocess" (aclnnMlaPreprocessGetWorkspaceSize: parameter table;
# Constraints: shape fields): input (T, He); wdqkv int8 (Hcq + 576, He), one row per output
# column ("transposeWdq" true); wuq int8 (N * (D + 64), Hcq); wuk (N, D, 512); cos/sin (T, 64);
# slotMapping int32 (T); cacheMode 0: kvCache (blockNum, blockSize, 1, 576); cacheMode 1:
# kvCache (..., 512) and kvCacheRope (..., 64).  The page fixes keyTotalDim = 512 + 64 and
# qRopeDim = 64; tokenNum <= 256, blockNum 192 and blockSize 128 in its constraints.


@dataclasses.dataclass(frozen=True)
class PpShape:
    T: int
    He: int
    Hcq: int
    N: int
    D: int            # qNoRopeDim
    block_num: int
    block_size: int
    Hckv: int = 512   # keyTotalDim = Hckv + Dr
    Dr: int = 64      # qRopeDim = kRopeDim


@dataclasses.dataclass(frozen=True)
class PpConfig:
    """One synthetic workload of the aclnnMlaPreprocess variant."""
    name: str
    shape: PpShape
    seed: int
    dtype: str = "bf16"        # "bf16" or "fp16": input, gammas, betas, scales, cos/sin, wuk, caches, outputs
    cache_mode: int = 0        # 0: concatenated 576-wide cache rows and q rows; 1: split
    do_rmsnorm: bool = True    # False: the input is only quantised
    eps: float = 1e-6
    with_bias: bool = True     # bias0 / bias1 passed (int32)
    pos_hi: int = 32768
    theta: float = 1e4

    @property
    def workload(self) -> str:
        s = self.shape
        return (f"{self.name}: T={s.T} He={s.He} Hcq={s.Hcq} N={s.N} D={s.D} Dr={s.Dr} Hckv={s.Hckv} "
                f"cache={s.block_num}x{s.block_size} [int8 wdqkv/wuq, {self.dtype}, cacheMode {self.cache_mode}]")


PP_CONFIGS: Dict[str, PpConfig] = {
    "pp_tiny": PpConfig(name="pp_tiny", shape=PpShape(T=8, He=256, Hcq=64, N=4, D=32, block_num=4, block_size=16),
                        seed=2000),
    # DeepSeek-V3 shapes at the page's fixed blockNum 192 and blockSize 128
    "pp_decode_t32": PpConfig(name="pp_decode_t32",
                              shape=PpShape(T=32, He=7168, Hcq=1536, N=128, D=128, block_num=192, block_size=128),
                              seed=2001),
    "pp_decode_t32_fp16": PpConfig(name="pp_decode_t32_fp16",
                                   shape=PpShape(T=32, He=7168, Hcq=1536, N=128, D=128, block_num=192,
                                                 block_size=128),
                                   seed=2002, dtype="fp16"),
    # the page's largest tokenNum
    "pp_t256": PpConfig(name="pp_t256",
                        shape=PpShape(T=256, He=7168, Hcq=1536, N=128, D=128, block_num=192, block_size=128),
                        seed=2003, cache_mode=1),
}


def pp_config(name: str, **overrides) -> PpConfig:
    """Return a named aclnnMlaPreprocess config, optionally with shape or other fields replaced."""
    cfg = PP_CONFIGS[name]
    shape_keys = {f.name for f in dataclasses.fields(PpShape)}
    shape_over = {k: v for k, v in overrides.items() if k in shape_keys}
    other = {k: v for k, v in overrides.items() if k not in shape_keys}
    if shape_over:
        other["shape"] = dataclasses.replace(cfg.shape, **shape_over)
    return dataclasses.replace(cfg, **other) if other else cfg


def make_pp_inputs(cfg: PpConfig, seed: Optional[int] = None) -> Dict[str, Optional[torch.Tensor]]:
    """Draw every input of one aclnnMlaPreprocess call on the CPU, in a fixed order, from one seed.

    The scale ranges keep the int8 codes of both quantisers mostly inside [-128, 127] (a few
    saturate) and the dequantised products of order one: deScale ~ U(0.5, 1.5) / (sqrt(K) * 25 * 73),
    25 and 73 being the rough rms of the codes and of uniform int8 weights.
    """
    s = cfg.shape
    gen = torch.Generator().manual_seed(cfg.seed if seed is None else seed)
    T, He, Hcq, N, D, Dr, Hckv = s.T, s.He, s.Hcq, s.N, s.D, s.Dr, s.Hckv
    fdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float16
    n1, n2 = Hcq + Hckv + Dr, N * (D + Dr)
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["input"] = torch.randn((T, He), generator=gen, dtype=torch.float32).to(fdt)
    out["gamma0"] = _uniform(gen, (He,), 0.8, 1.2).to(fdt)
    out["beta0"] = _uniform(gen, (He,), -0.1, 0.1).to(fdt)
    out["quant_scale0"] = _uniform(gen, (1,), 20.0, 30.0).to(fdt)
    out["quant_offset0"] = torch.randint(-4, 5, (1,), generator=gen, dtype=torch.int16).to(torch.int8)
    out["wdqkv"] = _randint8(gen, (n1, He))
    out["de_scale0"] = (_uniform(gen, (n1,), 0.5, 1.5) / (He ** 0.5 * 25 * 73)).to(torch.float32)
    b0 = torch.randint(-50000, 50001, (n1,), generator=gen, dtype=torch.int32)
    out["gamma1"] = _uniform(gen, (Hcq,), 0.8, 1.2).to(fdt)
    out["beta1"] = _uniform(gen, (Hcq,), -0.1, 0.1).to(fdt)
    out["quant_scale1"] = _uniform(gen, (1,), 20.0, 30.0).to(fdt)
    out["quant_offset1"] = torch.randint(-4, 5, (1,), generator=gen, dtype=torch.int16).to(torch.int8)
    out["wuq"] = _randint8(gen, (n2, Hcq))
    out["de_scale1"] = (_uniform(gen, (n2,), 0.5, 1.5) / (Hcq ** 0.5 * 25 * 73)).to(torch.float32)
    b1 = torch.randint(-20000, 20001, (n2,), generator=gen, dtype=torch.int32)
    out["bias0"] = b0 if cfg.with_bias else None
    out["bias1"] = b1 if cfg.with_bias else None
    out["gamma2"] = _uniform(gen, (Hckv,), 0.8, 1.2).to(fdt)
    pos = torch.randint(0, cfg.pos_hi, (T,), generator=gen, dtype=torch.int64)
    out["positions"] = pos
    h = Dr // 2
    inv = cfg.theta ** (-2.0 * torch.arange(h, dtype=torch.float64) / Dr)
    ang = pos.to(torch.float64)[:, None] * inv[None, :]
    out["cos"] = torch.cat([torch.cos(ang), torch.cos(ang)], dim=1).to(fdt).contiguous()
    out["sin"] = torch.cat([torch.sin(ang), torch.sin(ang)], dim=1).to(fdt).contiguous()
    out["wuk"] = (torch.randn((N, D, Hckv), generator=gen, dtype=torch.float32) * 0.02).to(fdt)
    nslots = s.block_num * s.block_size
    if nslots == 0:
        slots = torch.zeros(T, dtype=torch.int32)
    else:
        assert T <= nslots
        slots = torch.randperm(nslots, generator=gen)[:T].to(torch.int32)
    out["slot_mapping"] = slots.contiguous()

    def bits(shape):
        return torch.randint(-32768, 32768, shape, generator=gen, dtype=torch.int16).view(fdt)

    if cfg.cache_mode == 0:
        out["kv_cache"] = bits((s.block_num, s.block_size, 1, Hckv + Dr))
        out["kv_cache_rope"] = None
    else:
        out["kv_cache"] = bits((s.block_num, s.block_size, 1, Hckv))
        out["kv_cache_rope"] = bits((s.block_num, s.block_size, 1, Dr))
    return out
