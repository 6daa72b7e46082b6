"""GPU parity: the CUDA library, called through its C ABI, against the CPU oracle.

Tolerances are the ones the task fixes for this operation:
  bf16 outputs (queryOut, queryRopeOut, cache rows): |gpu - ref| <= 1e-2 + 1e-2 * |ref|;
  int8 codes (queryOut, int8 kv cache): within +-1;
  dequantScaleQNope: within 1e-2 relative;
  cache slot placement and every untouched cache row: bit-exact.
Every token of every configuration is compared with the oracle (the 8192-token prefill in
chunks of the oracle's output), plus properties that hold at any size (exactly the rows named by
cacheIndex changed, repeated calls are bit-identical).  The shape-space sweeps compare a seeded
sample of tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_pre_processing_gb300 import workloads, build as _build
from conftest import oracle_for

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="session", autouse=True)
def _built():
    _build.build()


def _runner():
    from attention_pre_processing_gb300.runner import PrologCall
    return PrologCall


def bf16_to_f64(t):
    return t.detach().float().cpu().double().numpy()


def assert_bf16_close(gpu, ref, what):
    g = bf16_to_f64(gpu) if isinstance(gpu, torch.Tensor) else gpu
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements outside |d| <= {ATOL} + {RTOL}|ref|; "
                           f"worst excess {np.max(err - bound):.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def assert_codes_close(gpu_i8, ref_i8, what):
    d = np.abs(gpu_i8.astype(np.int32) - ref_i8.astype(np.int32))
    assert d.max() <= 1, f"{what}: int8 codes differ by up to {d.max()} (> 1 LSB) in {(d > 1).sum()} elements"


def assert_scale_close(gpu, ref, what):
    err = np.abs(gpu - ref)
    bad = err > 1e-2 * np.abs(ref) + 1e-30
    assert not bad.any(), f"{what}: {bad.sum()} scales outside 1e-2 relative"


def _bits(t):
    """Raw bits of a cache tensor (bf16 -> int16), comparable even for NaN patterns."""
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


class Case:
    """Runs one config on the GPU once and the oracle on its tokens (or a seeded sample of them),
    in chunks of at most ``chunk`` tokens so that the oracle's fp64 outputs stay small."""

    def __init__(self, cfg, sample=None, seed=None, chunk=1024, bs=None):
        self.cfg = cfg
        self.inp = workloads.make_inputs(cfg, seed=seed)
        PrologCall = _runner()
        self.call = PrologCall(cfg, self.inp, bs=bs)
        self.kv0 = self.call.t["kv_cache"].clone()
        self.kr0 = self.call.t["kr_cache"].clone()
        self.call()
        torch.cuda.synchronize()
        self.status = self.call.status()
        T = cfg.shape.T
        self.tokens = None if sample is None or sample >= T else workloads.sample_tokens(T, sample).numpy()
        tok = self.tok()
        self.chunks = [tok[i:i + chunk] for i in range(0, len(tok), chunk)]
        self.ref = None
        if len(self.chunks) == 1:
            self.ref = oracle_for(cfg, self.inp, tokens=self.tokens)

    def tok(self):
        return np.arange(self.cfg.shape.T) if self.tokens is None else self.tokens

    def _refs(self):
        """(tokens, oracle result) per chunk."""
        if self.ref is not None:
            yield self.tok(), self.ref
            return
        for c in self.chunks:
            yield c, oracle_for(self.cfg, self.inp, tokens=c)

    def check_all(self):
        cfg, s, out = self.cfg, self.cfg.shape, self.call.outputs()
        assert self.status == 0, f"device status bits {self.status:#x}"
        T = s.T
        q_rope = out["q_rope_out"].reshape(T, s.N, s.Dr).cpu()
        q_out = out["q_out"].reshape(T, s.N, s.Hckv).cpu()
        for tok_np, ref in self._refs():
            tok = torch.as_tensor(tok_np)
            assert_bf16_close(q_rope[tok], ref["q_rope"], "queryRopeOut")
            if cfg.q_int8:
                assert_codes_close(q_out[tok].numpy(), ref["q_nope_i8"], "queryOut int8")
                sc = out["dequant_scale_q_nope_out"].reshape(T, s.N).cpu()[tok].numpy().astype(np.float64)
                assert_scale_close(sc, ref["q_nope_scale"], "dequantScaleQNope")
            else:
                assert_bf16_close(q_out[tok], ref["q_nope"], "queryOut")
            self.check_cache_rows(tok_np, ref)
        self.check_placement()

    def check_placement(self):
        s, out = self.cfg.shape, self.call.outputs()
        nslots = s.block_num * s.block_size
        if nslots == 0:
            return
        idx = self.inp["cache_index"].numpy()
        kv1 = out["kv_cache"].reshape(nslots, s.Hckv)
        kr1 = out["kr_cache"].reshape(nslots, s.Dr)
        # placement: exactly the rows named by cacheIndex changed; every other row is bit-identical
        changed_kv = (_bits(kv1) != _bits(self.kv0.reshape(nslots, s.Hckv))).any(dim=1).nonzero().flatten().cpu()
        changed_kr = (_bits(kr1) != _bits(self.kr0.reshape(nslots, s.Dr))).any(dim=1).nonzero().flatten().cpu()
        assert set(changed_kv.tolist()) == set(idx.tolist())
        assert set(changed_kr.tolist()) == set(idx.tolist())

    def check_cache_rows(self, tok, ref):
        cfg, s, out = self.cfg, self.cfg.shape, self.call.outputs()
        nslots = s.block_num * s.block_size
        if nslots == 0:
            return
        idx = self.inp["cache_index"].numpy()
        kv1 = out["kv_cache"].reshape(nslots, s.Hckv)
        kr1 = out["kr_cache"].reshape(nslots, s.Dr)
        # values of the checked tokens' rows
        slots = torch.as_tensor(idx[tok])
        kv_rows = kv1[slots.to(kv1.device)].cpu()
        kr_rows = kr1[slots.to(kr1.device)].cpu()
        if cfg.kv_int8:
            ref_kv = ref["kv_cache"].reshape(nslots, s.Hckv)[idx[tok]]
            assert_codes_close(kv_rows.numpy(), ref_kv, "kvCache int8")
        else:
            assert_bf16_close(kv_rows, ref["c_kv"], "kvCache")
        if cfg.kr_int8:
            ref_kr = ref["kr_cache"].reshape(nslots, s.Dr)[idx[tok]]
            assert_codes_close(kr_rows.numpy(), ref_kr, "krCache int8")
        else:
            assert_bf16_close(kr_rows, ref["k_r"], "krCache")


_cases = {}


def case(name, sample=None, bs=None, **over):
    key = (name, sample, bs, tuple(sorted(over.items())))
    if key not in _cases:
        _cases[key] = Case(workloads.config(name, **over), sample=sample, bs=bs)
    return _cases[key]


# ------------------------------------------------------------------ configs

def test_tiny_bf16():
    case("tiny").check_all()


def test_decode_t32_bf16():
    case("decode_t32").check_all()


def test_decode_t256_qint8():
    case("decode_t256_qint8").check_all()


def test_int8_full_quant_t64():
    case("int8_t64").check_all()


def test_int8_full_quant_t64_reciprocal_kv_scale():
    c = case("int8_t64_recip")
    c.check_all()
    # the reciprocal draw drives codes into rounding and saturation, not just zero
    kv = c.call.outputs()["kv_cache"].reshape(-1, c.cfg.shape.Hckv)[c.inp["cache_index"].cuda()]
    assert (kv.abs() == 127).any() and (kv != 0).float().mean() > 0.5


def test_prefill_t8192_bf16():
    """Every one of the 8192 tokens against the oracle (32 row tiles of 256 on SM pairs)."""
    c = case("prefill_t8192")
    c.check_all()
    _cases.clear()   # the case holds ~2 GB of device tensors


# ------------------------------------------------------------- shape space
# The pages fix Hcq = 1536, Hckv = 512, D = 128, Dr = 64 and let He take nine values, N seven
# powers of two and BlockSize multiples of 16 from 16 to 1024 (aclnnMlaPrologV2WeightNz, shape
# format fields).  A few tokens of each combination against the oracle, on the persistent
# decode kernel (T <= 64), the split-K decode path (T <= 256) and the prefill path (T > 256).

@pytest.mark.parametrize("He", [1024, 3072, 7680, 8192])
@pytest.mark.parametrize("N", [1, 16, 128])
def test_shape_space_decode(He, N):
    case("decode_t32", T=5, He=He, N=N, block_num=8, block_size=16).check_all()


@pytest.mark.parametrize("He,N,T", [(2048, 8, 100), (5120, 64, 130)])
def test_shape_space_split_k(He, N, T):
    case("decode_t32", sample=16, T=T, He=He, N=N, block_num=4, block_size=1024).check_all()


@pytest.mark.parametrize("He,N", [(1024, 4), (6144, 32), (8192, 2)])
def test_shape_space_prefill(He, N):
    case("decode_t32", sample=16, T=300, He=He, N=N, block_num=3, block_size=112).check_all()


# --------------------------------------------------------------- edge cases

@pytest.mark.parametrize("T", [1, 37, 64, 65, 129, 200])
def test_decode_ragged_token_counts(T):
    """Decode sizes with ragged row counts: the persistent kernel (T <= 64), then the split-K
    kernels with one and two 128-row sub-tiles."""
    case("decode_t32", T=T).check_all()


@pytest.mark.parametrize("T", [257, 300])
def test_tile_path_ragged(T):
    """Whole-tile path with a ragged last row tile, DeepSeek-V3 shapes (fused RoPE epilogue)."""
    case("decode_t32", sample=24, T=T, block_num=8).check_all()


@pytest.mark.parametrize("T", [1, 37, 100, 200])
def test_int8_full_quant_ragged_token_counts(T):
    """int8 inputs at ragged decode sizes: tokenX widened inside the down-projection (T <= 64,
    short activation boxes), widened by its own launch with one 128-row tile (T = 100) and with
    two sub-tiles (T = 200)."""
    case("int8_t64", T=T).check_all()


def test_int8_full_quant_many_tokens():
    """int8 inputs and int8 kv cache / q^N with T above the decode sizes: the warp-per-token
    row pass with its dequant scales, int8 c^Q codes and int8 cache rows."""
    case("int8_t64", sample=24, T=300, block_num=8).check_all()


def test_partial_quant_many_tokens():
    """Partial quantisation (int8 W^UqQr, smooth scales, int8 kv and kr caches) with T above the
    decode sizes."""
    case("decode_t32", sample=24, T=300, block_num=8, uqqr_int8=True, smooth=True, kv_int8=True,
         kr_int8=True, ckv_reciprocal=True).check_all()


def test_tiny_shapes_tile_path():
    """T above the split threshold with small heads: tile GEMMs, fp32 rows, row-wise finalize."""
    case("tiny", T=300, block_num=32).check_all()


def test_tiny_qint8():
    case("tiny", q_int8=True).check_all()


def test_partial_quant_uqqr_int8():
    """Partial quantisation: only weightUqQr is int8; c^Q gets per-token dynamic codes."""
    case("tiny", uqqr_int8=True, smooth=True).check_all()
    case("decode_t32", uqqr_int8=True).check_all()


def test_partial_quant_int8_caches():
    """Partial quantisation with quantised kv and kr caches (reciprocal scales exercise rounding)."""
    case("tiny", uqqr_int8=True, kv_int8=True, kr_int8=True, ckv_reciprocal=True).check_all()


@pytest.mark.parametrize("T", [48, 100])
def test_determinism_bit_identical(T):
    """Every sum is taken in a fixed order (the operation is deterministic by default), so
    repeated calls are bit-identical: T=48 runs the persistent decode kernel (twenty calls, so
    that a race in its cross-CTA hand-offs would show), T=100 the split-K decode path."""
    cfg = workloads.config("decode_t32", T=T)
    inp = workloads.make_inputs(cfg)
    PrologCall = _runner()
    a = PrologCall(cfg, inp)
    b = PrologCall(cfg, inp)
    a()
    for _ in range(20):
        b()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    for k in ("q_out", "q_rope_out", "kv_cache", "kr_cache"):
        assert torch.equal(_bits(a.t[k]), _bits(b.t[k])), k


@pytest.mark.parametrize("T", [300, 8192])
def test_prefill_determinism_bit_identical(T):
    """The prefill path (SM-pair GEMMs, the c^KV | k^R row pass on a second stream) gives
    bit-identical results on repeated calls."""
    cfg = workloads.config("prefill_t8192") if T == 8192 else workloads.config("decode_t32", T=T, block_num=8)
    inp = workloads.make_inputs(cfg)
    PrologCall = _runner()
    a = PrologCall(cfg, inp)
    a()
    torch.cuda.synchronize()
    first = {k: _bits(a.t[k]).clone() for k in ("q_out", "q_rope_out", "kv_cache", "kr_cache")}
    for _ in range(3):
        a()
    torch.cuda.synchronize()
    assert a.status() == 0
    for k, v in first.items():
        assert torch.equal(_bits(a.t[k]), v), k
    del a, first
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,B,S", [("decode_t32", 4, 8), ("decode_t32", 2, 150),
                                       ("decode_t256_qint8", 2, 128)])
def test_batch_seq_layout(name, B, S):
    """The non-concatenated layout of the page: tokenX (B, S, He), ropeSin / ropeCos (B, S, Dr),
    cacheIndex (B, S), queryOut (B, S, N, Hckv), queryRopeOut (B, S, N, Dr) and, with int8
    queryOut, dequantScaleQNopeOut (B*S, N, 1).  Checked against the oracle and bit for bit
    against the same call in the (T, ...) layout."""
    over = {} if B * S == workloads.config(name).shape.T else {"T": B * S, "block_num": 8}
    c = case(name, bs=(B, S), **over)
    assert tuple(c.call.t["q_out"].shape[:2]) == (B, S) and c.call.t["x"].dim() == 3
    c.check_all()
    flat = case(name, **over)
    for k in ("q_out", "q_rope_out", "kv_cache", "kr_cache"):
        assert torch.equal(_bits(c.call.t[k]).reshape(-1), _bits(flat.call.t[k]).reshape(-1)), k


@pytest.mark.parametrize("name", ["decode_t32", "decode_t256_qint8"])
def test_packed_io_matches_separate_tensors(name):
    """PrologCall(packed_io=True) (the per-token inputs and the outputs as views of one buffer
    each way, as the end-to-end bench copies them) gives the same bits as separate tensors."""
    cfg = workloads.config(name)
    inp = workloads.make_inputs(cfg)
    PrologCall = _runner()
    a, b = PrologCall(cfg, inp), PrologCall(cfg, inp, packed_io=True)
    assert b.io_in is not None and b.io_out is not None
    assert b.t["x"].data_ptr() == b.io_in.data_ptr() and b.t["q_out"].data_ptr() == b.io_out.data_ptr()
    a()
    b()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    for k in ("q_out", "q_rope_out", "dequant_scale_q_nope_out", "kv_cache", "kr_cache"):
        if a.t[k] is not None:
            assert torch.equal(_bits(a.t[k]), _bits(b.t[k])), k


def test_empty_tokens_is_a_no_op():
    cfg = workloads.config("tiny", T=0)
    inp = workloads.make_inputs(cfg)
    PrologCall = _runner()
    c = PrologCall(cfg, inp)
    kv0 = c.t["kv_cache"].clone()
    c()
    torch.cuda.synchronize()
    assert torch.equal(_bits(c.t["kv_cache"]), _bits(kv0))


def test_no_cache_blocks_still_computes_queries():
    """Skv = 0: queryOut / queryRopeOut computed, no cache write."""
    case("decode_t32", T=16, block_num=0).check_all()


@pytest.mark.parametrize("name,over", [("tiny", {}), ("decode_t32", {"T": 8})])
def test_out_of_range_slot_sets_status_and_skips_row(name, over):
    """Kernel-per-step path (tiny) and the persistent decode kernel (DeepSeek-V3 shapes, T=8)."""
    cfg = workloads.config(name, **over)
    inp = workloads.make_inputs(cfg)
    bad = int(cfg.shape.block_num * cfg.shape.block_size + 5)
    inp["cache_index"] = inp["cache_index"].clone()
    inp["cache_index"][2] = bad
    PrologCall = _runner()
    c = PrologCall(cfg, inp)
    kv0 = c.t["kv_cache"].clone()
    c()
    torch.cuda.synchronize()
    from attention_pre_processing_gb300 import DEV_CACHE_INDEX_RANGE
    assert c.status() & DEV_CACHE_INDEX_RANGE
    # the other tokens' rows are written, nothing else changes
    s = cfg.shape
    idx = [int(v) for i, v in enumerate(inp["cache_index"].tolist()) if i != 2]
    changed = (_bits(c.t["kv_cache"]) != _bits(kv0)).reshape(-1, s.Hckv).any(1).nonzero().flatten().tolist()
    assert set(changed) == set(idx)
    # queries still match the oracle (run it with the valid slot restored)
    good = dict(inp)
    good["cache_index"] = workloads.make_inputs(cfg)["cache_index"]
    ref = oracle_for(cfg, good)
    assert_bf16_close(c.t["q_out"].cpu(), ref["q_nope"], "queryOut")
