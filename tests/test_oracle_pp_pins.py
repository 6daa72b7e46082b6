"""Pins of the aclnnMlaPreprocess oracle (``oracle/preprocess.py``) against what the page and
the mathematics fix.  No GPU.

Each test is chosen so that a plausible slip (rounding halves to even, the offset added
before the scale, beta added without the norm, a transposed weight, the bias added after
the scale, epsilon outside the root, a swapped RoPE half, the wrong cache column order)
fails at least one of them.
"""
import fractions
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.preprocess as pp
from attention_pre_processing_gb300 import workloads
from conftest import read_golden, oracle_for
import naive_preprocess

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


# ------------------------------------------------------------- quantiser

def test_round_half_away_exact():
    v = np.array([2.5, -2.5, 0.5, -0.5, 1.5, 0.49999999999999994, -0.49999999999999994, 126.5, 3.0, -7.2])
    assert pp.round_half_away(v).tolist() == [3, -3, 1, -1, 2, 0, 0, 127, 3, -7]


def test_quant_code_closed_forms():
    # offset added after the scaled value is rounded; asymmetric range [-128, 127]
    assert pp.quant_i8([1.0], 100.4, 3).tolist() == [103]
    assert pp.quant_i8([-1.0], 100.4, 3).tolist() == [-97]
    assert pp.quant_i8([0.5], 5.0, 0).tolist() == [3]          # 2.5 -> 3 (away from zero)
    assert pp.quant_i8([-0.5], 5.0, 2).tolist() == [-1]        # -2.5 -> -3, + 2
    assert pp.quant_i8([10.0, -10.0], 1000.0, 0).tolist() == [127, -128]
    assert pp.quant_i8([0.0], 7.0, -4).tolist() == [-4]


def test_rmsnorm_quant_closed_forms():
    He = 16
    g = np.ones(He)
    b = np.zeros(He)
    # a constant row c normalises to sign(c) when eps = 0
    for c, want in ((2.0, 103), (-0.25, -97)):
        x = np.full((1, He), c)
        assert (pp.rmsnorm_quant(x, g, b, 100.4, 3, 0.0) == want).all()
    # beta is added after the norm and before the scale: a zero row gives round(beta * s) + o
    x = np.zeros((1, He))
    beta = np.full(He, 0.5)
    assert (pp.rmsnorm_quant(x, g, beta, 5.0, 1, 1e-6) == 4).all()      # 2.5 -> 3, + 1
    # epsilon inside the root: tiny rows are scaled by 1 / sqrt(eps), not by 1 / (rms + eps)
    x = np.full((1, He), 1e-4)
    got = pp.rmsnorm_quant(x, g, b, 1000.0, 0, 1e-6)
    want = round(1000.0 * 1e-4 / math.sqrt(1e-8 + 1e-6))
    assert (got == want).all()
    # gamma scales per element
    gam = np.arange(1, He + 1, dtype=np.float64) / He
    got = pp.rmsnorm_quant(np.full((1, He), 3.0), gam, b, 16.0, 0, 0.0)
    assert got.tolist() == [[int(pp.round_half_away(16.0 * gi)) for gi in gam]]


def test_quant_only_ignores_beta_and_norm():
    x = np.array([[0.3, -1.7, 4.0, 0.05]])
    beta = np.full(4, 100.0)
    got = pp.rmsnorm_quant(x, np.full(4, 9.0), beta, 10.0, -2, 1e-6, do_rmsnorm=False)
    assert got.tolist() == [[1, -19, 38, -1]]     # round(3) - 2, round(-17) - 2, 40 - 2, round(0.5) - 2


# ------------------------------------------------------------- int8 products

def test_dequant_matmul_brute_force_and_orientation():
    rng = np.random.default_rng(5)
    T, K, n = 3, 11, 7
    a = rng.integers(-128, 128, (T, K))
    w = rng.integers(-127, 128, (n, K))          # one row per output column
    bias = rng.integers(-1000, 1000, n)
    scale = rng.uniform(1e-4, 1e-3, n)
    got = pp.dequant_matmul(a, w, bias, scale)
    for t in range(T):
        for j in range(n):
            acc = sum(int(a[t, k]) * int(w[j, k]) for k in range(K)) + int(bias[j])
            assert got[t, j] == float(acc) * scale[j]
    # a one-hot code row picks one input column of every output row: W[:, k] * scale
    e = np.zeros((1, K), dtype=np.int64)
    e[0, 4] = 1
    assert np.array_equal(pp.dequant_matmul(e, w, None, scale)[0], w[:, 4] * scale)


# ------------------------------------------------------------- norm, rotation, rounding

def test_rmsnorm_closed_forms():
    y = np.full((1, 8), 3.0)
    assert np.allclose(pp.rmsnorm(y, np.ones(8), 0.0), 1.0, rtol=0, atol=1e-15)
    rng = np.random.default_rng(1)
    y = rng.normal(size=(4, 64))
    out = pp.rmsnorm(y, np.ones(64), 0.0)
    assert np.allclose(np.mean(out * out, axis=1), 1.0, rtol=1e-13)
    assert np.array_equal(pp.rmsnorm(np.zeros((1, 8)), np.ones(8), 1e-6), np.zeros((1, 8)))


def test_rope_golden_dr4():
    g = read_golden("rope_half_dr4.txt")
    out = pp.rope_half(np.array(g["v"]), np.array(g["cos"]), np.array(g["sin"]))
    assert out.tolist() == g["out"]


def test_rope_identity_and_pair_norm():
    rng = np.random.default_rng(2)
    v = rng.normal(size=(3, 64))
    assert np.array_equal(pp.rope_half(v, np.ones(64), np.zeros(64)), v)
    ang = rng.uniform(0, 6.3, 32)
    c = np.concatenate([np.cos(ang), np.cos(ang)])
    s = np.concatenate([np.sin(ang), np.sin(ang)])
    out = pp.rope_half(v, c, s)
    assert np.allclose(out[:, :32] ** 2 + out[:, 32:] ** 2, v[:, :32] ** 2 + v[:, 32:] ** 2, rtol=1e-12)


def _exact_fp16_rne(v: float) -> float:
    """Brute force: the nearest fp16 value by exact rational comparison, ties to even."""
    fv = fractions.Fraction(v)
    a = abs(fv)
    e = math.floor(math.log2(a))
    while fractions.Fraction(2) ** e > a:
        e -= 1
    while fractions.Fraction(2) ** (e + 1) <= a:
        e += 1
    q = fractions.Fraction(2) ** max(e - 10, -24)
    lo = (a // q) * q
    hi = lo + q
    r = lo if a - lo < hi - a else hi if a - lo > hi - a else (lo if (lo / q) % 2 == 0 else hi)
    return float(r) * (1 if fv > 0 else -1)


def test_fp16_output_rounding_single_step():
    rng = np.random.default_rng(3)
    vals = list(rng.normal(size=200) * 10) + [1 + 2 ** -11, 1 + 3 * 2 ** -11, -(2 + 2 ** -10),
                                                1 + 2 ** -11 + 2 ** -40, 3e-6, 6.1e-5]
    bits = pp.round_to_dtype(np.array(vals), "fp16")
    got = pp.bits_to_f64(bits, "fp16")
    assert got.tolist() == [_exact_fp16_rne(v) for v in vals]


# ------------------------------------------------------------- whole call

def _naive_params(inp, t_cos, t_sin):
    f = lambda k: None if inp.get(k) is None else pp.to_f64(inp[k]).tolist()
    wuk = pp.to_f64(inp["wuk"])
    return dict(gamma0=f("gamma0"), beta0=f("beta0"), qs0=f("quant_scale0")[0], qo0=int(f("quant_offset0")[0]),
                wdqkv=[[int(v) for v in r] for r in f("wdqkv")], de0=f("de_scale0"),
                bias0=None if inp.get("bias0") is None else [int(v) for v in f("bias0")],
                gamma1=f("gamma1"), beta1=f("beta1"), qs1=f("quant_scale1")[0], qo1=int(f("quant_offset1")[0]),
                wuq=[[int(v) for v in r] for r in f("wuq")], de1=f("de_scale1"),
                bias1=None if inp.get("bias1") is None else [int(v) for v in f("bias1")],
                gamma2=f("gamma2"), cos=t_cos, sin=t_sin, wuk=wuk.tolist(), N=wuk.shape[0], D=wuk.shape[1],
                Hcq=len(f("gamma1")), Hckv=len(f("gamma2")), Dr=len(t_cos))


@pytest.mark.parametrize("dtype,cache_mode,do_rmsnorm,with_bias", [
    ("bf16", 0, True, True), ("fp16", 1, True, False), ("bf16", 1, False, True)])
def test_whole_call_matches_naive_statement(dtype, cache_mode, do_rmsnorm, with_bias):
    cfg = workloads.pp_config("pp_tiny", T=3, He=64, Hcq=32, N=2, D=16, Hckv=32, Dr=16, dtype=dtype,
                              cache_mode=cache_mode, do_rmsnorm=do_rmsnorm, with_bias=with_bias)
    inp = workloads.make_pp_inputs(cfg)
    r = pp.for_config(cfg, inp)
    x = pp.to_f64(inp["input"])
    cos, sin = pp.to_f64(inp["cos"]), pp.to_f64(inp["sin"])
    for t in range(cfg.shape.T):
        p = _naive_params(inp, cos[t].tolist(), sin[t].tolist())
        qn, qr, kn, kr = naive_preprocess.preprocess_token(x[t].tolist(), p, do_rmsnorm=do_rmsnorm, eps=cfg.eps)
        np.testing.assert_allclose(r["q_nope"][t], np.array(qn), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["q_rope"][t], np.array(qr), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["k_nope"][t], np.array(kn), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["k_rope"][t], np.array(kr), rtol=1e-12, atol=1e-12)


def test_kv_path_reduces_to_the_prolog_oracle():
    """With doRmsNorm off, quantScale0 = 1, quantOffset0 = 0, integer inputs, no bias and
    deScale0 = the prolog's per-column weight scales (per-token scale 1), the variant's
    down-projection, kv RmsNorm and k RoPE are the prolog's int8 path (aclnnMlaPrologV2WeightNz,
    Function: Formula), whose oracle is pinned separately."""
    cfg1 = workloads.config("tiny", x_int8=True)
    s = cfg1.shape
    inp1 = workloads.make_inputs(cfg1)
    inp1["dequant_scale_x"] = torch.ones((s.T, 1), dtype=torch.float32)
    r1 = oracle_for(cfg1, inp1)
    cfg2 = workloads.pp_config("pp_tiny", T=s.T, He=s.He, Hcq=s.Hcq, N=s.N, D=s.D, Hckv=s.Hckv, Dr=s.Dr,
                               block_num=s.block_num, block_size=s.block_size, cache_mode=1, do_rmsnorm=False,
                               with_bias=False, eps=cfg1.eps_ckv)
    inp2 = workloads.make_pp_inputs(cfg2)
    inp2["input"] = inp1["x"].to(torch.bfloat16)
    inp2["quant_scale0"] = torch.ones(1, dtype=torch.bfloat16)
    inp2["quant_offset0"] = torch.zeros(1, dtype=torch.int8)
    inp2["wdqkv"] = torch.cat([inp1["w_dq"], inp1["w_dkvkr"]], dim=1).t().contiguous()
    inp2["de_scale0"] = torch.cat([inp1["dequant_scale_w_dq"].reshape(-1), inp1["dequant_scale_w_dkvkr"].reshape(-1)])
    inp2["gamma2"] = inp1["gamma_ckv"]
    inp2["cos"], inp2["sin"] = inp1["rope_cos"], inp1["rope_sin"]
    inp2["slot_mapping"] = inp1["cache_index"].to(torch.int32)
    inp2["kv_cache"] = inp1["kv_cache"].clone()
    inp2["kv_cache_rope"] = inp1["kr_cache"].clone()
    r2 = pp.for_config(cfg2, inp2)
    np.testing.assert_allclose(r2["k_nope"], r1["c_kv"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r2["k_rope"], r1["k_r"], rtol=1e-12, atol=1e-14)
    assert np.array_equal(r2["kv_cache"], r1["kv_cache"])
    assert np.array_equal(r2["kv_cache_rope"], r1["kr_cache"])


@pytest.mark.parametrize("cache_mode", [0, 1])
def test_cache_rows_written_exactly_at_slots(cache_mode):
    cfg = workloads.pp_config("pp_tiny", cache_mode=cache_mode)
    inp = workloads.make_pp_inputs(cfg)
    r = pp.for_config(cfg, inp)
    s = cfg.shape
    before = inp["kv_cache"].view(torch.int16).numpy().view(np.uint16).reshape(s.block_num * s.block_size, -1)
    after = r["kv_cache"].reshape(s.block_num * s.block_size, -1)
    changed = set(np.nonzero((before != after).any(axis=1))[0].tolist())
    assert changed == set(inp["slot_mapping"].tolist())
    for t, slot in enumerate(inp["slot_mapping"].tolist()):
        row = pp.bits_to_f64(after[slot], cfg.dtype)
        if cache_mode == 0:   # [k^N (512) | k^R (64)] in one 576-wide row
            want = np.concatenate([r["k_nope"][t], r["k_rope"][t]])
        else:
            want = r["k_nope"][t]
            kr = pp.bits_to_f64(r["kv_cache_rope"].reshape(s.block_num * s.block_size, -1)[slot], cfg.dtype)
            assert np.array_equal(kr, pp.bits_to_f64(pp.round_to_dtype(r["k_rope"][t], cfg.dtype), cfg.dtype))
        assert np.array_equal(row, pp.bits_to_f64(pp.round_to_dtype(want, cfg.dtype), cfg.dtype))
    if cache_mode == 0:
        assert r["q_out"].shape == (s.T, s.N, s.Hckv + s.Dr)
        assert np.array_equal(r["q_out"][:, :, :s.Hckv], r["q_nope"])
        assert np.array_equal(r["q_out"][:, :, s.Hckv:], r["q_rope"])


def test_absorbed_weight_invariant():
    """q^N[t, n] = codes1[t] . A_n + b_n with A_n = (W^UQ_n^T diag(deScale1_n)) W^UK[n] and
    b_n = (bias1_n * deScale1_n) W^UK[n], computed the other way round."""
    cfg = workloads.pp_config("pp_tiny")
    inp = workloads.make_pp_inputs(cfg)
    r = pp.for_config(cfg, inp)
    s = cfg.shape
    wuq = pp.to_f64(inp["wuq"]).reshape(s.N, s.D + s.Dr, s.Hcq)
    de1 = pp.to_f64(inp["de_scale1"]).reshape(s.N, s.D + s.Dr)
    b1 = pp.to_f64(inp["bias1"]).reshape(s.N, s.D + s.Dr)
    wuk = pp.to_f64(inp["wuk"])
    for n in range(s.N):
        A = (wuq[n, :s.D].T * de1[n, :s.D]) @ wuk[n]
        b = (b1[n, :s.D] * de1[n, :s.D]) @ wuk[n]
        np.testing.assert_allclose(r["q_nope"][:, n], r["cq_codes"] @ A + b, rtol=1e-10, atol=1e-12)


def test_token_subset_equals_rows_of_full_run():
    cfg = workloads.pp_config("pp_tiny")
    inp = workloads.make_pp_inputs(cfg)
    full = pp.for_config(cfg, inp)
    sub = pp.for_config(cfg, inp, tokens=[1, 5])
    for k in ("q_nope", "q_rope", "k_nope", "k_rope"):
        assert np.array_equal(sub[k], full[k][[1, 5]])
