"""A second, independent statement of the MLA prolog, for tiny shapes only.

Written with numpy fp64 matrix products per head and per branch, in a layout
different from the C oracle's loops, so that a slip in either shows up as a
disagreement.  Follows "aclnnMlaPrologV2WeightNz" (Function: Formula) with the
"half" RoPE of "aclnnMlaPreprocess" (Constraints: RoPE mode).  Test-only.
"""
import numpy as np


def bf16_to_f64(bits):
    bits = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def rms_norm(y, gamma, eps):
    # gamma * y / sqrt(mean(y^2) + eps), over the last axis
    return gamma * y / np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + eps)


def rotate_half(v):
    h = v.shape[-1] // 2
    return np.concatenate([-v[..., h:], v[..., :h]], axis=-1)


def rope(v, cos, sin):
    return v * cos + rotate_half(v) * sin


def prolog(x, w_dq, w_uqqr, w_uk, w_dkvkr, g_cq, g_ckv, sin, cos, *, N, D, Dr, Hckv, eps_cq, eps_ckv):
    """All arguments fp64 arrays. Returns (q_nope (T,N,Hckv), q_rope (T,N,Dr), c_kv (T,Hckv), k_r (T,Dr), c_q)."""
    c_q = rms_norm(x @ w_dq, g_cq, eps_cq)
    y_kvkr = x @ w_dkvkr
    c_kv = rms_norm(y_kvkr[:, :Hckv], g_ckv, eps_ckv)
    k_r = rope(y_kvkr[:, Hckv:], cos, sin)
    T = x.shape[0]
    z = (c_q @ w_uqqr).reshape(T, N, D + Dr)
    q_c = z[:, :, :D]
    q_rope = rope(z[:, :, D:], cos[:, None, :], sin[:, None, :])
    q_nope = np.einsum("tnd,ndc->tnc", q_c, w_uk)
    return q_nope, q_rope, c_kv, k_r, c_q
