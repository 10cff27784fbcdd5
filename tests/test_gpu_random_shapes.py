"""Whole-layer parity at seeded random shapes within the C ABI's limits.

Twelve layer configurations drawn from a fixed seed: T in [1, 600], d a
multiple of 64 in [128, 512], E in {8, 16, 24, 40, 64} (E a multiple of 8),
k in [1, min(8, E)], H and Hs multiples of 128 (Hs = 0: no shared expert),
learned or random routing, the Zipf bias on some learned cases, and dropless
or capacity-limited (factors 1.25 and 0.5).  Each uses its own input seed.
Forward and backward, through both call sequences (unfused, and fused: row
gathers in the GEMM loads, the combine in the shared down projection), are
compared with the C++ oracle exactly as the fixed cases are
(tests/gpu_util.py): routing and permutation bit for bit on the GPU's own
fp32 logits, every output and gradient within the layer tolerance."""
import random

import pytest
import torch

from oracle import moe_oracle_cpp as orc_cpp
from synth import gen, workloads
from tests.gpu_util import compare_layer, oracle_reference, upload

pytestmark = pytest.mark.gpu

SEED = 20261203


def random_shapes(n=12, seed=SEED):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        E = rng.choice([8, 16, 24, 40, 64])
        k = rng.randint(1, min(8, E))
        routing = rng.choice(["learned", "learned", "random"])
        w = workloads.custom(f"rand{i}", T=rng.randint(1, 600), d=64 * rng.randint(2, 8), E=E, k=k,
                             H=128 * rng.randint(1, 4), Hs=rng.choice([0, 128, 256]), routing=routing,
                             zipf_bias=routing == "learned" and rng.random() < 0.3,
                             capacity_factor=rng.choice([0.0, 0.0, 1.25, 0.5]), backward=True)
        out.append((w, gen.BASE_SEED + 1000 * (i + 1)))
    return out


CASES = random_shapes()


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
@pytest.mark.parametrize("case", range(len(CASES)), ids=[
    f"{w.name}-T{w.T}-d{w.d}-E{w.E}-k{w.k}-H{w.H}-Hs{w.Hs}-{w.routing}{'-zipf' if w.zipf_bias else ''}"
    f"-cap{w.capacity}" for w, _ in CASES])
def test_random_shape_layer_parity(B, case, fused):
    from top_routing_grouped_moe_gb300.layer import MoELayer
    w, base = CASES[case]
    inp = workloads.make_inputs(w, base=base)
    dev = upload(inp)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity, fused=fused)
    layer.forward(dev["x"], dev, logits_in=dev.get("logits_in"))
    layer.backward(dev["x"], dev["dY"], dev, learned_router=w.routing == "learned")
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    _, ref, refb, _ = oracle_reference(w, inp, layer, impl=orc_cpp)
    compare_layer(w, inp, layer, ref, refb)
