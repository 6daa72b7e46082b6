"""GPU parity of the aclnnMlaPreprocess variant: mla_preprocess (C ABI) against oracle/preprocess.py.

Tolerances as for the prolog: 16-bit outputs and cache rows within 1e-2 + 1e-2 * |ref|; the
rows that change are exactly the slots of slotMapping and every other cache bit is unchanged.
The int8 codes the two quantisers produce are intermediates: the kernels decide them in
fp32, the oracle in fp64, so a value that lands within rounding of a code boundary can differ
by one code; the outputs' tolerance covers that (one code moves a product by under 0.2 %).
"""
import numpy as np
import pytest
import torch

import oracle.preprocess as opp
from attention_pre_processing_gb300 import workloads, build as _build

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="session", autouse=True)
def _built():
    _build.build()


def to_f64(t):
    return t.detach().float().cpu().double().numpy()


def assert_close(gpu, ref, what):
    g = to_f64(gpu) if isinstance(gpu, torch.Tensor) else gpu
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements outside |d| <= {ATOL} + {RTOL}|ref|; "
                           f"worst excess {np.max(err - bound):.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")


class PpCase:
    """Runs one config on the GPU once and the oracle on (a sample of) its tokens."""

    def __init__(self, cfg, sample=None, inputs=None):
        from attention_pre_processing_gb300.runner import PreprocessCall
        self.cfg = cfg
        self.inp = workloads.make_pp_inputs(cfg) if inputs is None else inputs
        self.call = PreprocessCall(cfg, self.inp)
        self.kv0 = self.call.t["kv_cache"].clone()
        self.kr0 = None if self.call.t["kv_cache_rope"] is None else self.call.t["kv_cache_rope"].clone()
        self.call()
        torch.cuda.synchronize()
        self.status = self.call.status()
        T = cfg.shape.T
        self.tokens = None if sample is None or sample >= T else workloads.sample_tokens(T, sample).numpy()
        self.ref = opp.for_config(cfg, self.inp, tokens=self.tokens) if T > 0 else None

    def rows(self, t):
        return t if self.tokens is None else t[torch.as_tensor(self.tokens, device=t.device)]

    def check(self):
        assert self.status == 0, f"device status {self.status:#x}"
        s, c, r = self.cfg.shape, self.call, self.ref
        assert_close(self.rows(c.t["q_out"]), r["q_out"], "qOut")
        if self.cfg.cache_mode == 1:
            assert_close(self.rows(c.t["q_rope_out"]), r["q_rope_out"], "qRopeOut")
        self.check_cache(c.t["kv_cache"], self.kv0, "kvCache",
                         np.concatenate([r["k_nope"], r["k_rope"]], -1) if self.cfg.cache_mode == 0 else r["k_nope"])
        if self.cfg.cache_mode == 1:
            self.check_cache(c.t["kv_cache_rope"], self.kr0, "kvCacheRope", r["k_rope"])

    def check_cache(self, after, before, what, ref_rows):
        s = self.cfg.shape
        nslots = s.block_num * s.block_size
        if nslots == 0:
            return
        a = after.view(torch.int16).reshape(nslots, -1)
        b = before.view(torch.int16).reshape(nslots, -1)
        changed = set(torch.nonzero((a != b).any(dim=1)).flatten().tolist())
        slots = self.inp["slot_mapping"].tolist()
        assert changed == set(slots), f"{what}: the changed rows are not exactly the slots of slotMapping"
        idx = torch.as_tensor([slots[t] for t in (range(s.T) if self.tokens is None else self.tokens)],
                              device=after.device)
        got = after.reshape(nslots, -1)[idx]
        assert_close(got, ref_rows, f"{what} rows")
        untouched = torch.ones(nslots, dtype=torch.bool, device=after.device)
        untouched[torch.as_tensor(slots, device=after.device)] = False
        assert torch.equal(a[untouched], b[untouched]), f"{what}: untouched rows changed"


# ------------------------------------------------------------- small shapes, every switch

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("cache_mode", [0, 1])
def test_tiny_dtypes_and_cache_modes(dtype, cache_mode):
    PpCase(workloads.pp_config("pp_tiny", dtype=dtype, cache_mode=cache_mode)).check()


def test_tiny_quantiser_only_and_no_bias():
    PpCase(workloads.pp_config("pp_tiny", do_rmsnorm=False, with_bias=False)).check()


@pytest.mark.parametrize("T,N,D", [(1, 1, 16), (37, 3, 48), (64, 5, 128), (129, 2, 256), (256, 4, 64)])
def test_ragged_shapes(T, N, D):
    cfg = workloads.pp_config("pp_tiny", T=T, He=512, Hcq=128, N=N, D=D, block_num=8, block_size=64,
                              cache_mode=T % 2)
    PpCase(cfg).check()


def test_empty_cache_still_computes_q():
    PpCase(workloads.pp_config("pp_tiny", block_num=0)).check()


def test_slot_out_of_range_skips_that_row():
    cfg = workloads.pp_config("pp_tiny")
    inp = workloads.make_pp_inputs(cfg)
    nslots = cfg.shape.block_num * cfg.shape.block_size
    bad = inp["slot_mapping"].clone()
    bad[3] = nslots + 5
    inp["slot_mapping"] = bad
    from attention_pre_processing_gb300.runner import PreprocessCall
    call = PreprocessCall(cfg, inp)
    kv0 = call.t["kv_cache"].clone()
    call()
    torch.cuda.synchronize()
    assert call.status() & 0x1
    a = call.t["kv_cache"].view(torch.int16).reshape(nslots, -1)
    b = kv0.view(torch.int16).reshape(nslots, -1)
    changed = set(torch.nonzero((a != b).any(dim=1)).flatten().tolist())
    assert changed == set(bad.tolist()) - {nslots + 5}


# ------------------------------------------------------------- DeepSeek-V3 shapes

@pytest.mark.parametrize("name", ["pp_decode_t32", "pp_decode_t32_fp16"])
def test_decode_full_oracle(name):
    PpCase(workloads.pp_config(name)).check()


@pytest.mark.parametrize("T", [100, 200])
def test_decode_shapes_ragged_token_counts(T):
    """DeepSeek-V3 shapes at ragged token counts, every token: one 128-row tile with the
    down-projection's 128-column tiles and one 512-column W^UK tile per head (T = 100), two
    sub-tiles with 192-column tiles and two W^UK tiles per head (T = 200)."""
    PpCase(workloads.pp_config("pp_decode_t32", T=T, block_num=8)).check()


def test_t256_every_token():
    """The page's largest tokenNum (256), cacheMode 1, every token against the oracle."""
    PpCase(workloads.pp_config("pp_t256")).check()


def test_deterministic_bit_identical():
    cfg = workloads.pp_config("pp_decode_t32")
    from attention_pre_processing_gb300.runner import PreprocessCall
    call = PreprocessCall(cfg, workloads.make_pp_inputs(cfg))
    outs = []
    for _ in range(3):
        call()
        torch.cuda.synchronize()
        outs.append((call.t["q_out"].clone(), call.t["kv_cache"].clone()))
    for q, kv in outs[1:]:
        assert torch.equal(q.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(kv.view(torch.int16), outs[0][1].view(torch.int16))
