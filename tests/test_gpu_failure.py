"""Failure detection without a fault: a bounded device wait on a phase that
nothing completes runs out, the kernel records MOE_ERR_TIMEOUT in the device
status word (read and cleared by the host) and returns, and the same context
then runs the layer's kernels as before."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from synth import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable(B):
    torch.cuda.synchronize()
    B.moe_device_status()  # read and clear whatever an earlier call left
    B.moe_selftest_wait_timeout(2000)  # 2 ms
    torch.cuda.synchronize()
    assert B.moe_device_status() == B.MOE_ERR_TIMEOUT
    assert B.moe_device_status() == 0  # read and cleared
    # the context still runs work: top-k routing, bit-exact against the oracle
    T, E, k = 300, 64, 4
    logits = gen.random_logits(T, E, tensor=901)
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    g = torch.empty(T, k, dtype=torch.float32, device="cuda")
    B.moe_route_topk(None, None, None, torch.from_numpy(logits).cuda(), T, 0, E, k, None, idx, g, None, 0)
    torch.cuda.synchronize()
    ridx, rg = orc.route_topk(logits, k)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(g.cpu().numpy(), rg, rtol=2e-6, atol=1e-7)
    assert B.moe_device_status() == 0
