import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden(name):
    """Parse a golden fixture: '#' lines are comments, other lines are 'key v1 v2 ...'."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = [float(v) for v in vals]
    return out


def oracle_for(cfg, inp, tokens=None, num_threads=0, with_intermediates=True):
    """Run the oracle on a workload config's inputs."""
    import oracle
    return oracle.prolog(inp, dims=_Dims(cfg.shape), eps_cq=cfg.eps_cq, eps_ckv=cfg.eps_ckv,
                         x_int8=cfg.x_int8, uqqr_int8=cfg.x_int8 or cfg.uqqr_int8, kv_int8=cfg.kv_int8,
                         kr_int8=cfg.kr_int8, q_int8=cfg.q_int8,
                         tokens=tokens, num_threads=num_threads, with_intermediates=with_intermediates)


class _Dims:
    def __init__(self, s):
        for k in ("T", "He", "Hcq", "N", "D", "Dr", "Hckv", "block_num", "block_size"):
            setattr(self, k, getattr(s, k))
