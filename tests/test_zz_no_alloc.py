"""The no-allocation entry point, mla_prolog_no_alloc, against mla_prolog.

mla_prolog_no_alloc serves callers that cannot allocate device memory themselves, for
example a plugin whose host process owns the whole device memory budget, or a runtime that
fixes every buffer at start-up.  It runs the same kernels as mla_prolog, with the workspace
in a fixed scratch buffer that the library holds.  These tests call both entry points through
the C ABI on identical inputs and require the same results, within the tolerances of the
parity tests (bf16 |d| <= 1e-2 + 1e-2 |ref|, int8 codes within 1, scales within 1e-2
relative) and bit-identical caches.  Two calls in a row on different inputs show that the
second call does not see the first call's leftovers in the shared scratch buffer.

The file name makes pytest collect it last.
"""
import pytest
import torch

from attention_pre_processing_gb300 import (DEV_CACHE_INDEX_RANGE, NO_ALLOC_SCRATCH_BYTES, MlaError,
                                            build as _build, mla_prolog_no_alloc, mla_prolog_no_alloc_status,
                                            mla_prolog_workspace_size, workloads)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()


def _with_workspace(cfg, seed):
    """Outputs and caches of mla_prolog (caller-supplied workspace) on seeded inputs."""
    from attention_pre_processing_gb300.runner import PrologCall
    call = PrologCall(cfg, workloads.make_inputs(cfg, seed=seed))
    call()
    torch.cuda.synchronize()
    assert call.status() == 0
    return {k: v.clone() for k, v in call.outputs().items() if v is not None}


def _no_alloc(cfg, seed, stream, inp=None):
    """Outputs and caches of mla_prolog_no_alloc on the same seeded inputs.  The tensors are
    allocated here by the test (the caller); the entry point itself allocates nothing."""
    from attention_pre_processing_gb300.runner import INPUT_KEYS
    if inp is None:
        inp = workloads.make_inputs(cfg, seed=seed)
    s = cfg.shape
    t = {k: (None if inp.get(k) is None else inp[k].cuda().contiguous()) for k in INPUT_KEYS}
    t["q_out"] = torch.empty((s.T, s.N, s.Hckv), dtype=torch.int8 if cfg.q_int8 else torch.bfloat16, device="cuda")
    t["q_rope_out"] = torch.empty((s.T, s.N, s.Dr), dtype=torch.bfloat16, device="cuda")
    t["dequant_scale_q_nope_out"] = (torch.empty((s.T, s.N, 1), dtype=torch.float32, device="cuda")
                                     if cfg.q_int8 else None)
    torch.cuda.synchronize()
    mla_prolog_no_alloc(t, cfg.eps_cq, cfg.eps_ckv, stream=stream)
    return t


def _compare(ref, got, cfg, what):
    if cfg.q_int8:
        d = (got["q_out"].int() - ref["q_out"].int()).abs().max().item()
        assert d <= 1, f"{what}: int8 queryOut differs by {d}"
        r, g = ref["dequant_scale_q_nope_out"], got["dequant_scale_q_nope_out"]
        assert torch.all((g - r).abs() <= 1e-2 * r.abs() + 1e-30), f"{what}: dequantScaleQNope"
    else:
        torch.testing.assert_close(got["q_out"].float(), ref["q_out"].float(), atol=ATOL, rtol=RTOL,
                                   msg=lambda m: f"{what}: queryOut: {m}")
    torch.testing.assert_close(got["q_rope_out"].float(), ref["q_rope_out"].float(), atol=ATOL, rtol=RTOL,
                               msg=lambda m: f"{what}: queryRopeOut: {m}")
    for k in ("kv_cache", "kr_cache"):
        a, b = ref[k], got[k]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), f"{what}: {k} differs from the workspace entry point's"


@pytest.mark.parametrize("name", ["tiny", "decode_t32"])
def test_no_alloc_matches_workspace_entry_on_two_calls(name):
    cfg = workloads.config(name)
    stream = torch.cuda.current_stream()
    # two calls in a row on different inputs (different tokens, positions and cache slots)
    seeds = (cfg.seed, cfg.seed + 7919)
    got = []
    for seed in seeds:
        got.append(_no_alloc(cfg, seed, stream))
        assert mla_prolog_no_alloc_status(stream) == 0
    torch.cuda.synchronize()
    for i, seed in enumerate(seeds):
        _compare(_with_workspace(cfg, seed), got[i], cfg, f"{name} call {i + 1}")


def test_no_alloc_q_int8_output():
    cfg = workloads.config("tiny", q_int8=True)
    stream = torch.cuda.current_stream()
    for seed in (cfg.seed, cfg.seed + 1):
        got = _no_alloc(cfg, seed, stream)
        torch.cuda.synchronize()
        _compare(_with_workspace(cfg, seed), got, cfg, f"tiny int8 q^N seed {seed}")


def test_no_alloc_covers_decode_batches_of_128_tokens():
    """The scratch limit covers bf16 decode batches of up to 128 tokens at DeepSeek-V3 shapes."""
    cfg = workloads.config("decode_t32", T=128)
    stream = torch.cuda.current_stream()
    got = _no_alloc(cfg, cfg.seed, stream)
    assert mla_prolog_workspace_size(got, cfg.eps_cq, cfg.eps_ckv) <= NO_ALLOC_SCRATCH_BYTES
    assert mla_prolog_no_alloc_status(stream) == 0
    _compare(_with_workspace(cfg, cfg.seed), got, cfg, "decode T=128")


def test_no_alloc_status_reports_an_out_of_range_slot():
    """The status word in the scratch buffer: an out-of-range cacheIndex row sets its bit; the
    next clean call clears it."""
    cfg = workloads.config("tiny")
    stream = torch.cuda.current_stream()
    inp = workloads.make_inputs(cfg)
    inp["cache_index"] = inp["cache_index"].clone()
    inp["cache_index"][1] = cfg.shape.block_num * cfg.shape.block_size + 3
    _no_alloc(cfg, None, stream, inp=inp)
    assert mla_prolog_no_alloc_status(stream) & DEV_CACHE_INDEX_RANGE
    _no_alloc(cfg, cfg.seed, stream)
    assert mla_prolog_no_alloc_status(stream) == 0


def test_no_alloc_rejects_calls_beyond_the_scratch_limit():
    # 1024 tokens: the q^C hand-off alone (T x N x D bf16) is 32 MiB, twice the limit
    cfg = workloads.config("decode_t32", T=1024, block_num=16)
    from attention_pre_processing_gb300.runner import INPUT_KEYS
    inp = workloads.make_inputs(cfg)
    s = cfg.shape
    t = {k: (None if inp.get(k) is None else inp[k].cuda().contiguous()) for k in INPUT_KEYS}
    t["q_out"] = torch.empty((s.T, s.N, s.Hckv), dtype=torch.bfloat16, device="cuda")
    t["q_rope_out"] = torch.empty((s.T, s.N, s.Dr), dtype=torch.bfloat16, device="cuda")
    t["dequant_scale_q_nope_out"] = None
    assert mla_prolog_workspace_size(t, cfg.eps_cq, cfg.eps_ckv) > NO_ALLOC_SCRATCH_BYTES
    q_before = t["q_out"].clone()
    kv_before = t["kv_cache"].clone()
    with pytest.raises(MlaError) as e:
        mla_prolog_no_alloc(t, cfg.eps_cq, cfg.eps_ckv)
    assert e.value.code == 561003
    torch.cuda.synchronize()
    # bit patterns (the random-bit cache and the unwritten output hold NaN patterns)
    assert torch.equal(t["kv_cache"].view(torch.int16), kv_before.view(torch.int16))
    assert torch.equal(t["q_out"].view(torch.int16), q_before.view(torch.int16))
