"""Full-size GPU parity: every layer configuration of the workload table
(64-expert random and learned/Zipf routing with and without capacity, the
expert-count sweep E in {8, 32, 64, 128} at T=16384, and the d=4096 E=128
layer), forward and backward, in the launch configuration bench.py times.

The oracle is cheap enough in float64 BLAS to run the whole layer at these
sizes on the host, so every output element is compared (not a sample).  The
dense float64 weight copies need up to ~20 GB of host memory (the d=4096
layer); tests whose copy would not fit in the host's available memory are
skipped with the reason."""
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from synth import workloads
from tests.gpu_util import compare_layer, oracle_reference, upload

pytestmark = pytest.mark.gpu

FULL = ["tiny64e_random", "tiny64e_zipf", "tiny64e_zipf_cap125", "scale_E8", "scale_E32", "scale_E64",
        "scale_E128", "large_E128"]


def _avail_bytes():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 1 << 62


@pytest.mark.parametrize("name", FULL)
def test_full_size_layer_parity(name):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding as B
    from top_routing_grouped_moe_gb300.layer import MoELayer

    base = workloads.WORKLOADS[name]
    w = workloads.custom(base.name, T=base.T, d=base.d, E=base.E, k=base.k, H=base.H, Hs=base.Hs,
                         routing=base.routing, zipf_bias=base.zipf_bias, capacity_factor=base.capacity_factor,
                         backward=True)
    f64_weight_bytes = 8 * (3 * w.E * w.d * w.H + 3 * w.d * w.Hs)
    need = 3 * f64_weight_bytes + 24 * w.T * w.k * max(w.d, 2 * w.H) * 8
    if need > _avail_bytes():
        pytest.skip(f"oracle needs ~{need / 2**30:.0f} GiB of host memory")
    inp = workloads.make_inputs(w)
    dev = upload(inp)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity)
    layer.forward(dev["x"], dev, logits_in=dev.get("logits_in"))
    layer.backward(dev["x"], dev["dY"], dev, learned_router=w.routing == "learned")
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    del dev
    _, ref, refb, flips = oracle_reference(w, inp, layer)
    compare_layer(w, inp, layer, ref, refb)
    print(f"{name}: {flips} tokens route differently on the oracle's fp64-router logits (near ties); "
          f"every check ran on the GPU's fp32 logits")


@pytest.mark.parametrize("name", ["large_E128", "tiny64e_zipf_cap125"])
def test_full_size_fused_equals_unfused(name):
    """The fused path (row gathers inside the GEMMs' loads, the combine in the
    shared down projection) at full size, in the configuration the bench
    times: every output and GEMM gradient equal to the unfused path's, which
    the parity test above checks against the oracle; the gate gradient and
    what takes it in within fp32 rounding (its per-row partial sums are split
    differently by single-CTA and CTA-pair tiles)."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding as B
    from top_routing_grouped_moe_gb300.layer import MoELayer

    base = workloads.WORKLOADS[name]
    w = workloads.custom(base.name, T=base.T, d=base.d, E=base.E, k=base.k, H=base.H, Hs=base.Hs,
                         routing=base.routing, zipf_bias=base.zipf_bias, capacity_factor=base.capacity_factor,
                         backward=True)
    dev = upload(workloads.make_inputs(w))
    layers = {}
    for fused in (False, True):
        layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity, fused=fused)
        layer.forward(dev["x"], dev, logits_in=dev.get("logits_in"))
        layer.backward(dev["x"], dev["dY"], dev, learned_router=w.routing == "learned")
        layers[fused] = layer
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    a, b = layers[True], layers[False]
    R = int(b.offsets[-1].item())
    for n in ("y", "h_s", "au_s", "dx_s", "dW_g", "dW_u", "dW_d", "dWs_g", "dWs_u", "dWs_d"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n
    from tests.test_gpu_fused import NEAR, near_close
    for n, rtol, atol in NEAR:
        near_close(n, getattr(a, n), getattr(b, n), rtol, atol)
    for n in ("h", "au", "dx_perm"):
        assert torch.equal(getattr(a, n)[:R], getattr(b, n)[:R]), n
    assert torch.equal(a.o_perm[b.slot_of_row[:R].long()], b.o_perm[:R])
