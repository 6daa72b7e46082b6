"""A second, independent statement of the aclnnMlaPreprocess variant, for tiny shapes only.

Plain Python scalars and loops (no numpy matrix products), one token, one column at a
time, following "aclnnMlaPreprocess" (Function description: the six paths; Formula:
RMS, RmsNorm, RmsNormQuant; Constraints: RoPE half mode).  Used only to cross-check the
numpy oracle on tiny inputs.  Test-only.
"""
import math


def _round_away(v):
    # halves away from zero, exact for the small magnitudes used here
    f = math.floor(abs(v))
    r = f + (1 if abs(v) - f >= 0.5 else 0)
    return r if v >= 0 else -r


def _code(v, scale, offset):
    q = _round_away(v * scale) + offset
    return max(-128, min(127, q))


def _norm_row(row, gamma, eps):
    ms = sum(v * v for v in row) / len(row)
    r = math.sqrt(ms + eps)
    return [g * v / r for g, v in zip(gamma, row)]


def _rope_row(v, cos, sin):
    h = len(v) // 2
    out = [0.0] * len(v)
    for j in range(h):
        out[j] = v[j] * cos[j] - v[j + h] * sin[j]
        out[j + h] = v[j + h] * cos[j + h] + v[j] * sin[j + h]
    return out


def preprocess_token(x, p, *, do_rmsnorm, eps):
    """One token.  ``x`` a list of floats; ``p`` a dict of Python lists / scalars:
    gamma0, beta0, qs0, qo0, wdqkv (rows = output columns), de0, bias0, gamma1, beta1, qs1, qo1,
    wuq (rows = output columns), de1, bias1, gamma2, cos, sin, wuk [n][d][c], N, D, Hcq, Hckv, Dr.
    Returns (q_nope [n][c], q_rope [n][r], k_nope [c], k_rope [r])."""
    if do_rmsnorm:
        nx = _norm_row(x, p["gamma0"], eps)
        v0 = [a + b for a, b in zip(nx, p["beta0"])]
    else:
        v0 = list(x)
    a0 = [_code(v, p["qs0"], p["qo0"]) for v in v0]
    y = []
    for j, row in enumerate(p["wdqkv"]):
        acc = 0
        for k in range(len(a0)):
            acc += a0[k] * row[k]
        b = p["bias0"][j] if p["bias0"] is not None else 0
        y.append((acc + b) * p["de0"][j])
    Hcq, Hckv, Dr, N, D = p["Hcq"], p["Hckv"], p["Dr"], p["N"], p["D"]
    n1 = _norm_row(y[:Hcq], p["gamma1"], eps)
    a1 = [_code(v + b, p["qs1"], p["qo1"]) for v, b in zip(n1, p["beta1"])]
    z = []
    for j, row in enumerate(p["wuq"]):
        acc = 0
        for k in range(len(a1)):
            acc += a1[k] * row[k]
        b = p["bias1"][j] if p["bias1"] is not None else 0
        z.append((acc + b) * p["de1"][j])
    q_nope, q_rope = [], []
    for n in range(N):
        head = z[n * (D + Dr):(n + 1) * (D + Dr)]
        qn = []
        for c in range(Hckv):
            s = 0.0
            for d in range(D):
                s += head[d] * p["wuk"][n][d][c]
            qn.append(s)
        q_nope.append(qn)
        q_rope.append(_rope_row(head[D:], p["cos"], p["sin"]))
    k_nope = _norm_row(y[Hcq:Hcq + Hckv], p["gamma2"], eps)
    k_rope = _rope_row(y[Hcq + Hckv:Hcq + Hckv + Dr], p["cos"], p["sin"])
    return q_nope, q_rope, k_nope, k_rope
