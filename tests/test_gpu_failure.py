"""Failure detection on the GPU without a fault: a bounded device wait that
nothing completes gives up after its limit, reports HLQ_DEV_TIMEOUT through
the status word, and the context stays usable (a later call gives the same
bits as before)."""
import numpy as np
import pytest
import torch

import workloads
import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()


def test_bounded_wait_times_out_and_context_survives():
    inp = workloads.make_inputs(workloads.WORKLOADS[1], T=256)
    gy, w = to_dev(inp, "g_y", "bf16"), to_dev(inp, "w", "bf16")
    before = hlq.hlq_linear_backward_gx(gy, w, seed=2)
    torch.cuda.synchronize()
    assert hlq.hlq_read_device_status(clear=True) == 0
    r = hlq.hlq_debug_wait_timeout(1_000_000)        # 1 ms, nothing arrives
    torch.cuda.synchronize()
    assert int(r.item()) == 0
    assert hlq.hlq_read_device_status(clear=True) == hlq.DEV_TIMEOUT
    after = hlq.hlq_linear_backward_gx(gy, w, seed=2)
    torch.cuda.synchronize()
    assert hlq.hlq_read_device_status(clear=True) == 0
    assert torch.equal(before, after)
