"""The committed DRAM-traffic figures (profiles/traffic.json, one ncu capture per kernel) against
the algorithmic bytes of the same launch: every weight byte crosses HBM at least once (nothing
skipped), and the total stays within 1.1x of the algorithmic bytes (no wasted re-reads).  No GPU."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from attention_pre_processing_gb300 import workloads  # noqa: E402


def _traffic():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def _weights_bf16(s):
    return 2 * (s.He * (s.Hcq + s.Hckv + s.Dr) + s.Hcq * s.N * (s.D + s.Dr) + s.N * s.D * s.Hckv)


def test_decode_kernel_traffic_is_its_algorithmic_bytes():
    s = workloads.config("decode_t32").shape
    t = _traffic()["decode_t32"]["decode_persist"]
    assert t >= _weights_bf16(s)
    assert t <= 1.1 * bench.step_bytes(s)


def test_up_projection_traffic_bf16_and_int8_weights():
    s = workloads.config("decode_t256_qint8").shape
    w = s.Hcq * s.N * (s.D + s.Dr)   # W^UqQr elements
    t = _traffic()["decode_t256_qint8"]["k2_up_proj"]
    assert 2 * w <= t <= 1.1 * bench.k2_bytes(s)
    s8 = workloads.config("int8_t64").shape
    t8 = _traffic()["int8_t64"]["k2_up_proj"]
    # int8 weights at one byte, the c^Q codes (fp16) in, q^C and q^R out (bf16)
    alg8 = w + s8.T * s8.Hcq * 2 + s8.T * s8.N * (s8.D + s8.Dr) * 2
    assert w <= t8 <= 1.1 * alg8
