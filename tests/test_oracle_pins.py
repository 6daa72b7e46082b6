"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU.  Each test is chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand, epsilon outside the root,
rounding halves to even instead of away) fails at least one of them.
"""
import fractions
import math

import numpy as np
import pytest
import torch

import oracle
from attention_pre_processing_gb300 import workloads
from conftest import read_golden, oracle_for
import naive_prolog

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def bf16_bits(values):
    return torch.tensor(values, dtype=torch.float64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits):
    return naive_prolog.bf16_to_f64(bits)


# ------------------------------------------------------------- bf16 rounding

def _exact_bf16_rne(v: float) -> float:
    """Brute force: the nearest bf16 value by exact rational comparison, ties to even."""
    fv = fractions.Fraction(v)
    if fv == 0:
        return 0.0
    a = abs(fv)
    e = math.floor(math.log2(a))
    # guard against float log error
    while fractions.Fraction(2) ** e > a:
        e -= 1
    while fractions.Fraction(2) ** (e + 1) <= a:
        e += 1
    q = fractions.Fraction(2) ** max(e - 7, -133)
    lo = (a // q) * q
    hi = lo + q
    if a - lo < hi - a:
        r = lo
    elif a - lo > hi - a:
        r = hi
    else:
        r = lo if (lo / q) % 2 == 0 else hi
    return float(r) * (1 if fv > 0 else -1)


def test_bf16_rne_single_step_rounding():
    # halfway cases: ties to even
    assert oracle.bf16_rne([1 + 2 ** -8])[0] == 0x3F80
    assert oracle.bf16_rne([1 + 3 * 2 ** -8])[0] == 0x3F82
    # a value just above halfway that float32 would first round onto the halfway
    # point: one-step rounding goes up, two-step rounding would go down to 0x3F80
    assert oracle.bf16_rne([1 + 2 ** -8 + 2 ** -30])[0] == 0x3F81
    assert oracle.bf16_rne([-2.0])[0] == 0xC000
    assert oracle.bf16_rne([float("inf")])[0] == 0x7F80
    assert oracle.bf16_rne([1e39])[0] == 0x7F80


def test_bf16_rne_matches_brute_force():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.normal(size=300) * 10.0 ** rng.integers(-30, 30, size=300),
                           rng.normal(size=50) * 1e-39])
    got = bits_to_f64(oracle.bf16_rne(vals))
    want = np.array([_exact_bf16_rne(float(v)) for v in vals])
    assert np.array_equal(got, want)


# --------------------------------------------------------------- rounding

def test_round_half_away_and_saturation():
    got = oracle.round_i8([2.5, -2.5, 0.5, -0.5, 1.49, 126.7, 200.0, -200.0, 0.0])
    assert got.tolist() == [3, -3, 1, -1, 1, 127, 127, -127, 0]


# ---------------------------------------------------------------- RmsNorm

def test_rmsnorm_golden_eps_inside_root():
    g = read_golden("rmsnorm_row.txt")
    gamma = bf16_bits(g["gamma"])
    out0 = oracle.rmsnorm(g["y"], gamma, g["eps0"][0])
    out1 = oracle.rmsnorm(g["y"], gamma, g["eps1"][0])
    np.testing.assert_allclose(out0, g["out0"], rtol=1e-14)
    np.testing.assert_allclose(out1, g["out1"], rtol=1e-14)


def test_rmsnorm_closed_forms():
    n = 48
    gamma = bf16_bits(np.linspace(0.5, 1.5, n))
    gam = bits_to_f64(gamma)
    # constant row
    c, eps = 1.75, 1e-3
    out = oracle.rmsnorm(np.full(n, c), gamma, eps)
    np.testing.assert_allclose(out, gam * c / math.sqrt(c * c + eps), rtol=1e-14)
    # zero row stays zero; a tiny row is divided by sqrt(eps) (eps inside the root)
    assert np.all(oracle.rmsnorm(np.zeros(n), gamma, 1e-5) == 0.0)
    tiny = np.full(n, 1e-9)
    np.testing.assert_allclose(oracle.rmsnorm(tiny, gamma, 1e-5),
                               gam * 1e-9 / math.sqrt(1e-18 + 1e-5), rtol=1e-14)
    # gamma = 1, eps = 0: mean of squares of the output is exactly 1
    ones = bf16_bits(np.ones(n))
    y = np.random.default_rng(1).normal(size=n)
    o = oracle.rmsnorm(y, ones, 0.0)
    assert abs(np.mean(o * o) - 1.0) < 1e-14
    # scale invariance at eps = 0
    np.testing.assert_allclose(oracle.rmsnorm(37.0 * y, ones, 0.0), o, rtol=1e-13)


# ------------------------------------------------------------------- RoPE

def test_rope_golden_dr4():
    g = read_golden("rope_half_dr4.txt")
    out = oracle.rope_half(g["v"], bf16_bits(g["cos"]), bf16_bits(g["sin"]))
    assert out.tolist() == g["out"]


def test_rope_special_cases_and_invariants():
    rng = np.random.default_rng(2)
    dr, h = 64, 32
    v = rng.normal(size=dr)
    # position 0: identity
    assert np.array_equal(oracle.rope_half(v, bf16_bits(np.ones(dr)), bf16_bits(np.zeros(dr))), v)
    # quarter turn: rotate_half(v) = [-v[h:], v[:h]] exactly
    rq = oracle.rope_half(v, bf16_bits(np.zeros(dr)), bf16_bits(np.ones(dr)))
    assert np.array_equal(rq, np.concatenate([-v[h:], v[:h]]))
    # per-pair norm scales by cos^2 + sin^2 (tables duplicated across halves)
    ang = rng.uniform(0, 6.3, size=h)
    cb = bf16_bits(np.concatenate([np.cos(ang), np.cos(ang)]))
    sb = bf16_bits(np.concatenate([np.sin(ang), np.sin(ang)]))
    c, s = bits_to_f64(cb)[:h], bits_to_f64(sb)[:h]
    out = oracle.rope_half(v, cb, sb)
    np.testing.assert_allclose(out[:h] ** 2 + out[h:] ** 2, (c * c + s * s) * (v[:h] ** 2 + v[h:] ** 2), rtol=1e-12)


def test_rope_relative_position():
    """<RoPE(q, p1), RoPE(k, p2)> depends only on p1 - p2 (up to bf16 table rounding)."""
    cfg = workloads.config("tiny")
    rng = np.random.default_rng(3)
    dr = 64
    q, k = rng.normal(size=dr), rng.normal(size=dr)

    def tables(p):
        inv = 1e4 ** (-2.0 * np.arange(dr // 2) / dr)
        a = p * inv
        return bf16_bits(np.concatenate([np.cos(a), np.cos(a)])), bf16_bits(np.concatenate([np.sin(a), np.sin(a)]))

    def dot(p1, p2):
        c1, s1 = tables(p1)
        c2, s2 = tables(p2)
        return float(np.dot(oracle.rope_half(q, c1, s1), oracle.rope_half(k, c2, s2)))

    ref = dot(10, 3)
    assert abs(dot(107, 100) - ref) < 0.05 * (abs(ref) + 1)
    assert abs(dot(7, 0) - ref) < 0.05 * (abs(ref) + 1)
    del cfg


# ------------------------------------------------------------- quantiser

def test_dynamic_quant_golden():
    g = read_golden("dynamic_quant_row.txt")
    codes, scale = oracle.dynamic_quant(g["v"])
    assert scale == g["scale"][0]
    assert codes.tolist() == [int(c) for c in g["codes"]]


def test_dynamic_quant_invariants():
    rng = np.random.default_rng(4)
    for _ in range(50):
        v = rng.normal(size=512) * rng.uniform(0.01, 100)
        codes, scale = oracle.dynamic_quant(v)
        m = np.max(np.abs(v))
        assert scale == m / 127.0
        assert abs(int(codes[np.argmax(np.abs(v))])) == 127
        assert np.all(np.abs(codes.astype(np.float64) * scale - v) <= scale / 2 * (1 + 1e-12))
    codes, scale = oracle.dynamic_quant(np.zeros(16))
    assert scale == 0.0 and not codes.any()


# ---------------------------------------------------------------- matmul

def test_row_times_matches_numpy_matmul():
    rng = np.random.default_rng(5)
    K, n = 300, 70
    w = bf16_bits(rng.normal(size=(K, n)) * 0.05)
    x = rng.normal(size=K)
    got = oracle.row_times_bf16(x, w)
    np.testing.assert_allclose(got, x @ bits_to_f64(w), rtol=1e-12, atol=1e-14)
    # one-hot x picks out a weight row exactly
    e = np.zeros(K)
    e[17] = 1.0
    assert np.array_equal(oracle.row_times_bf16(e, w), bits_to_f64(w[17]))


# ------------------------------------------------------------ whole prolog

def _tiny(**kw):
    cfg = workloads.config("tiny", **kw)
    return cfg, workloads.make_inputs(cfg)


def _f64(t):
    return oracle._np(t).astype(np.float64) if t.dtype != torch.bfloat16 else bits_to_f64(oracle._np(t))


def test_whole_prolog_matches_naive_statement():
    cfg, inp = _tiny()
    s = cfg.shape
    res = oracle_for(cfg, inp)
    qn, qr, ckv, kr, cq = naive_prolog.prolog(
        _f64(inp["x"]), _f64(inp["w_dq"]), _f64(inp["w_uqqr"]), _f64(inp["w_uk"]), _f64(inp["w_dkvkr"]),
        _f64(inp["gamma_cq"]), _f64(inp["gamma_ckv"]), _f64(inp["rope_sin"]), _f64(inp["rope_cos"]),
        N=s.N, D=s.D, Dr=s.Dr, Hckv=s.Hckv, eps_cq=cfg.eps_cq, eps_ckv=cfg.eps_ckv)
    for got, want in ((res["q_nope"], qn), (res["q_rope"], qr), (res["c_kv"], ckv), (res["k_r"], kr), (res["c_q"], cq)):
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_absorbed_weight_invariant():
    """q^N == c^Q . (W^UQ_n . W^UK_n) per head, with D != Hckv so a transposed W^UK fails."""
    cfg, inp = _tiny(D=24, Hckv=40)
    s = cfg.shape
    res = oracle_for(cfg, inp)
    wuq = _f64(inp["w_uqqr"]).reshape(s.Hcq, s.N, s.D + s.Dr)[:, :, : s.D]
    wuk = _f64(inp["w_uk"])
    for n in range(s.N):
        absorbed = wuq[:, n, :] @ wuk[n]                  # (Hcq, Hckv)
        np.testing.assert_allclose(res["q_nope"][:, n, :], res["c_q"] @ absorbed, rtol=1e-11, atol=1e-13)


def test_cache_rows_written_exactly_at_slots():
    cfg, inp = _tiny()
    s = cfg.shape
    res = oracle_for(cfg, inp)
    kv0 = oracle._np(inp["kv_cache"]).reshape(-1, s.Hckv)
    kr0 = oracle._np(inp["kr_cache"]).reshape(-1, s.Dr)
    kv1 = res["kv_cache"].reshape(-1, s.Hckv)
    kr1 = res["kr_cache"].reshape(-1, s.Dr)
    changed = set(np.nonzero(np.any(kv1 != kv0, axis=1))[0].tolist())
    idx = oracle._np(inp["cache_index"]).tolist()
    assert changed == set(idx)
    assert set(np.nonzero(np.any(kr1 != kr0, axis=1))[0].tolist()) == set(idx)
    for t, slot in enumerate(idx):
        assert np.array_equal(kv1[slot], oracle.bf16_rne(res["c_kv"][t]))
        assert np.array_equal(kr1[slot], oracle.bf16_rne(res["k_r"][t]))
        # block / offset decomposition of the (BlockNum, BlockSize, 1, H) layout
        b, o = divmod(slot, s.block_size)
        assert np.array_equal(res["kv_cache"][b, o, 0], kv1[slot])


def test_slots_checked_before_any_write():
    cfg, inp = _tiny()
    bad = dict(inp)
    idx = inp["cache_index"].clone()
    idx[3] = idx[1]
    bad["cache_index"] = idx
    with pytest.raises(oracle.OracleError, match="duplicate"):
        oracle_for(cfg, bad)
    idx = inp["cache_index"].clone()
    idx[0] = cfg.shape.block_num * cfg.shape.block_size
    bad["cache_index"] = idx
    with pytest.raises(oracle.OracleError, match="range"):
        oracle_for(cfg, bad)


def test_empty_kv_cache_leaves_q_outputs():
    """Skv = 0 (no cache blocks): q outputs computed, nothing written."""
    cfg, inp = _tiny(block_num=0)
    res = oracle_for(cfg, inp)
    full = oracle_for(*_tiny())
    np.testing.assert_array_equal(res["q_nope"], full["q_nope"])
    assert res["kv_cache"].size == 0


def test_token_subset_equals_rows_of_full_run():
    cfg, inp = _tiny()
    full = oracle_for(cfg, inp)
    tok = [1, 5, 6]
    sub = oracle_for(cfg, inp, tokens=tok)
    np.testing.assert_array_equal(sub["q_nope"], full["q_nope"][tok])
    np.testing.assert_array_equal(sub["q_rope"], full["q_rope"][tok])


def test_q_int8_matches_row_quantiser():
    cfg, inp = _tiny(q_int8=True)
    res = oracle_for(cfg, inp)
    for t in range(cfg.shape.T):
        for n in range(cfg.shape.N):
            codes, scale = oracle.dynamic_quant(res["q_nope"][t, n])
            assert res["q_nope_scale"][t, n] == scale
            assert np.array_equal(res["q_nope_i8"][t, n], codes)


def test_int8_chain_exact_against_bf16_chain():
    """Power-of-two scales make the int8 chain's down-projection exact, so it must
    equal the bf16 chain on the dequantised inputs bit for bit."""
    cfg, inp = _tiny(x_int8=True, q_int8=True)
    s = cfg.shape
    inp = dict(inp)
    inp["dequant_scale_x"] = torch.full((s.T, 1), 2.0 ** -4)
    inp["dequant_scale_w_dq"] = torch.full((1, s.Hcq), 2.0 ** -6)
    inp["dequant_scale_w_dkvkr"] = torch.full((1, s.Hckv + s.Dr), 2.0 ** -6)
    inp["dequant_scale_w_uqqr"] = torch.full((1, s.N * (s.D + s.Dr)), 2.0 ** -7)
    res8 = oracle_for(cfg, inp)
    eq = dict(inp)
    eq["x"] = (inp["x"].to(torch.float64) * 2.0 ** -4).to(torch.bfloat16)
    eq["w_dq"] = (inp["w_dq"].to(torch.float64) * 2.0 ** -6).to(torch.bfloat16)
    eq["w_dkvkr"] = (inp["w_dkvkr"].to(torch.float64) * 2.0 ** -6).to(torch.bfloat16)
    cfg_bf = workloads.config("tiny", q_int8=True)
    resb = oracle_for(cfg_bf, eq)
    for k in ("c_q", "c_kv", "k_r"):
        np.testing.assert_array_equal(res8[k], resb[k])
    # the int8 up-projection: codes of c^Q times the int8 weight, dequantised
    z = (res8["c_q_i8"].astype(np.int64) @ oracle._np(inp["w_uqqr"]).astype(np.int64)).astype(np.float64)
    z = z * res8["c_q_scale"][:, None] * 2.0 ** -7
    zc = z.reshape(s.T, s.N, s.D + s.Dr)[:, :, : s.D]
    np.testing.assert_allclose(res8["q_c"], zc, rtol=1e-15, atol=0)
    for t in range(s.T):
        codes, sc = oracle.dynamic_quant(res8["c_q"][t])
        assert np.array_equal(codes, res8["c_q_i8"][t]) and sc == res8["c_q_scale"][t]


def test_kv_int8_cache_quantiser():
    cfg, inp = _tiny(x_int8=True, kv_int8=True, q_int8=True)
    s = cfg.shape
    res = oracle_for(cfg, inp)
    qs = oracle._np(inp["quant_scale_ckv"]).reshape(-1).astype(np.float64)
    kv = res["kv_cache"].reshape(-1, s.Hckv)
    for t, slot in enumerate(oracle._np(inp["cache_index"]).tolist()):
        assert np.array_equal(kv[slot], oracle.round_i8(res["c_kv"][t] * qs))


# ------------------------------------------- partial quantisation: smoothScalesCq

class _HandDims:
    T, He, Hcq, N, D, Dr, Hckv, block_num, block_size = 1, 4, 6, 1, 2, 4, 2, 1, 4


def _hand_inputs(y_q, gamma_cq, y_kvkr, gamma_ckv, cos, sin, kv_int8=False, kr_int8=False):
    """One token whose down-projections are row 0 of the weights: x = (1, 0, 0, 0).

    The other weight rows hold a non-zero filler, so a slip that reads them shows.
    """
    d = _HandDims
    w_dq = np.full((d.He, d.Hcq), 7.0)
    w_dq[0] = y_q
    w_dkvkr = np.full((d.He, d.Hckv + d.Dr), -5.0)
    w_dkvkr[0] = y_kvkr
    bf = lambda a: torch.tensor(np.asarray(a, dtype=np.float64)).to(torch.bfloat16)
    kv_dt = torch.int8 if kv_int8 else torch.bfloat16
    kr_dt = torch.int8 if kr_int8 else torch.bfloat16
    return {
        "x": bf([[1.0, 0.0, 0.0, 0.0]]),
        "w_dq": bf(w_dq),
        "w_uqqr": torch.eye(d.Hcq, d.N * (d.D + d.Dr), dtype=torch.int8),
        "w_uk": bf(np.ones((d.N, d.D, d.Hckv))),
        "w_dkvkr": bf(w_dkvkr),
        "gamma_cq": bf(gamma_cq),
        "gamma_ckv": bf(gamma_ckv),
        "rope_cos": bf([cos]),
        "rope_sin": bf([sin]),
        "cache_index": torch.tensor([2], dtype=torch.int64),
        "kv_cache": torch.zeros((d.block_num, d.block_size, 1, d.Hckv), dtype=kv_dt),
        "kr_cache": torch.zeros((d.block_num, d.block_size, 1, d.Dr), dtype=kr_dt),
        "dequant_scale_w_uqqr": torch.ones((1, d.N * (d.D + d.Dr)), dtype=torch.float32),
    }


def test_smooth_scales_golden_row():
    g = read_golden("smooth_quant_row.txt")
    inp = _hand_inputs(g["y"], g["gamma"], [1, -1, 1, 2, 3, 4], [1, 1], [1, 1, 1, 1], [0, 0, 0, 0])
    inp["smooth_scales_cq"] = torch.tensor([g["smooth"]], dtype=torch.float32)
    res = oracle.prolog(inp, dims=_HandDims, eps_cq=0.0, eps_ckv=0.0, uqqr_int8=True)
    assert res["c_q"][0].tolist() == g["c_q"]
    assert res["c_q_scale"][0] == g["scale"][0]
    assert res["c_q_i8"][0].tolist() == [int(c) for c in g["codes"]]
    assert res["q_c"][0, 0].tolist() == g["q_c"]


def _tiny_partial():
    cfg = workloads.config("tiny", uqqr_int8=True)
    return cfg, dict(workloads.make_inputs(cfg))


def test_smooth_scales_uniform_power_of_two():
    """A uniform smooth of 2^k scales u by 2^k exactly: the codes stay, the per-token scale
    and the dequantised up-projection are multiplied by 2^k exactly."""
    cfg, inp = _tiny_partial()
    base = oracle_for(cfg, inp)
    for k in (3, -2):
        inp["smooth_scales_cq"] = torch.full((1, cfg.shape.Hcq), 2.0 ** k, dtype=torch.float32)
        res = oracle_for(cfg, inp)
        assert np.array_equal(res["c_q_i8"], base["c_q_i8"])
        assert np.array_equal(res["c_q_scale"], base["c_q_scale"] * 2.0 ** k)
        assert np.array_equal(res["q_c"], base["q_c"] * 2.0 ** k)
        assert np.array_equal(res["c_q"], base["c_q"])


def test_smooth_scales_one_hot_moves_the_argmax():
    """smooth = e_j keeps only element j of c^Q: its code is +-127, every other code is 0 and
    the scale is |c^Q_j| / 127, whatever element of c^Q is the largest."""
    cfg, inp = _tiny_partial()
    base = oracle_for(cfg, inp)
    Hcq = cfg.shape.Hcq
    for j in (5, Hcq - 1):
        # j is not the largest element of c^Q in these tokens, so the smooth moves the argmax
        assert sum(int(np.argmax(np.abs(base["c_q"][t]))) != j for t in range(cfg.shape.T)) >= cfg.shape.T - 1
        e = torch.zeros((1, Hcq), dtype=torch.float32)
        e[0, j] = 1.0
        inp["smooth_scales_cq"] = e
        res = oracle_for(cfg, inp)
        for t in range(cfg.shape.T):
            want = np.zeros(Hcq, dtype=np.int8)
            want[j] = 127 if base["c_q"][t, j] > 0 else -127
            assert np.array_equal(res["c_q_i8"][t], want)
            assert res["c_q_scale"][t] == abs(base["c_q"][t, j]) / 127.0


# ----------------------------------------------------- int8 kv and kr caches

def test_int8_cache_rows_golden():
    g = read_golden("int8_cache_rows.txt")
    inp = _hand_inputs([3, -3, 3, -3, 3, -3], [1] * 6, g["ykv"] + g["ykr"], g["gamma_ckv"],
                       g["cos"], g["sin"], kv_int8=True, kr_int8=True)
    inp["quant_scale_ckv"] = torch.tensor([g["qs_ckv"]], dtype=torch.float32)
    inp["quant_scale_ckr"] = torch.tensor([g["qs_ckr"]], dtype=torch.float32)
    res = oracle.prolog(inp, dims=_HandDims, eps_cq=0.0, eps_ckv=0.0, uqqr_int8=True,
                        kv_int8=True, kr_int8=True)
    kv = res["kv_cache"].reshape(-1, _HandDims.Hckv)
    kr = res["kr_cache"].reshape(-1, _HandDims.Dr)
    assert kv[2].tolist() == [int(c) for c in g["kv_codes"]]
    assert kr[2].tolist() == [int(c) for c in g["kr_codes"]]
    # every other slot keeps its (zero) contents
    assert not kv[[0, 1, 3]].any() and not kr[[0, 1, 3]].any()
