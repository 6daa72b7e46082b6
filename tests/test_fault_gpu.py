"""Failure detection without a GPU fault: waits that nothing can satisfy give up at their time
limit, set MLA_DEV_WAIT_TIMEOUT in the workspace's status word and return, and the context
stays usable for the next call."""
import pytest
import torch

import attention_pre_processing_gb300 as mla
from attention_pre_processing_gb300 import workloads, build as _build

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()


@pytest.mark.parametrize("which", [0, 1])   # the flag wait (2 s limit), an mbarrier wait (10 ms)
def test_unsatisfiable_wait_sets_status_and_returns(which):
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    mla.mla_prolog_debug_wait_probe(ws, which)
    assert mla.mla_prolog_device_status(ws) & mla.DEV_WAIT_TIMEOUT
    # the context still works: a normal call runs clean afterwards
    from attention_pre_processing_gb300.runner import PrologCall
    cfg = workloads.config("tiny")
    call = PrologCall(cfg, workloads.make_inputs(cfg))
    call()
    torch.cuda.synchronize()
    assert call.status() == 0
