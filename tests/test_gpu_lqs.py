"""Layer-wise quantizer selection (hlq_select_gy_granularity) against the
oracle: the per-tensor and per-token RNE int4 errors (fp64, summed with
atomics: compared to 1e-9 relative) and the choice, on workload-shaped
samples and on constructed cases whose choice is known."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import hadamard_precision_backprop_gb300 as hlq
from hadamard_precision_backprop_gb300 import build as hbuild
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    hbuild.build()
    hlq.lib()
    oracle.build()


def _check(g32, dev_tensor):
    mse, choice = hlq.hlq_select_gy_granularity(dev_tensor)
    torch.cuda.synchronize()
    ref_choice, m_tensor, m_token = oracle.lqs_select(g32)
    got = mse.cpu().numpy()
    np.testing.assert_allclose(got, [m_tensor, m_token], rtol=1e-9, atol=0)
    assert int(choice.item()) == ref_choice
    return ref_choice


@pytest.mark.parametrize("wl_idx,T,dtype", [(0, 256, "f32"), (1, 512, "bf16"),
                                            (3, 256, "bf16"), (4, 512, "bf16")])
def test_lqs_matches_oracle_on_workload_samples(wl_idx, T, dtype):
    wl = workloads.WORKLOADS[wl_idx]
    inp = workloads.make_inputs(wl, T=T)
    _check(inp["g_y"], to_dev(inp, "g_y", dtype))


def test_lqs_known_choices():
    rng = np.random.default_rng(31)
    g = rng.standard_normal((64, 128)).astype(np.float32)
    g[5] *= 4.0                                       # per-tensor scale too coarse
    assert _check(g, torch.from_numpy(g).cuda()) == hlq.PER_TOKEN
    g[5] *= 250.0                                     # the outlier's own error dominates
    assert _check(g, torch.from_numpy(g).cuda()) == hlq.PER_TENSOR
    same = np.tile(rng.standard_normal((1, 128)).astype(np.float32), (32, 1))
    assert _check(same, torch.from_numpy(same).cuda()) == hlq.PER_TENSOR
    z = np.zeros((16, 32), np.float32)
    assert _check(z, torch.from_numpy(z).cuda()) == hlq.PER_TENSOR
