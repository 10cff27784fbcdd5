"""The MoE-layer workloads and their seeded synthetic inputs.

Shapes, routing kinds and value distributions follow the layer configurations
that the Olmo-core DDP MoE pages work at (top-4 routing, one shared expert,
sequences of 8192 tokens; "Production throughput runs" table, random vs learned
routing column; capacity factor named under "Interpreting the eight-layer DDP vs
FSDP comparison"):

  tiny            T=256   d=256  E=8   k=2 H=512  no shared expert, learned router
  tiny64e_random  T=8192  d=2048 E=64  k=4 H=1024 Hs=1024, random routing
  tiny64e_zipf    same shapes, learned router + Zipf-like fixed bias, dropless
  tiny64e_zipf_cap125  same, capacity factor 1.25
  scale_E{8,32,64,128} T=16384 d=2048 k=4 H=768 Hs=768, learned, fwd+bwd
  large_E128      T=8192  d=4096 E=128 k=4 H=1536 Hs=1536, learned, fwd+bwd
  large_E16_slice T=1024  d=4096 E=16  k=4 H=1536 Hs=1536 (large_E128's per-expert
                  shapes with 16 experts: a small case for profiling)

Values: x, dY ~ N(0,1) bf16; every weight ~ N(0, 0.02^2) bf16 (std 0.02).

Storage layouts (row-major, the layout the C ABI takes):
  x [T,d]; W_r [E,d]; W_g, W_u [E,H,d]; W_d [E,d,H]; Ws_g, Ws_u [Hs,d];
  Ws_d [d,Hs]; dY [T,d]; bias [E] f32; logits_in [T,E] f32.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from fractions import Fraction

import numpy as np

from . import gen

WEIGHT_STD = 0.02


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    H: int
    Hs: int
    routing: str          # "learned" | "random"
    zipf_bias: bool = False
    capacity_factor: float = 0.0  # 0 -> dropless
    backward: bool = False

    @property
    def capacity(self) -> int:
        """ceil(cf*T*k/E) computed exactly in integers, cf taken as the
        fraction it denotes (1.25 = 5/4, 0.25 = 1/4); 0 = dropless."""
        if self.capacity_factor == 0.0:
            return 0
        f = Fraction(self.capacity_factor).limit_denominator(1000)
        assert f > 0 and abs(float(f) - self.capacity_factor) < 1e-12
        return (f.numerator * self.T * self.k + f.denominator * self.E - 1) // (f.denominator * self.E)


WORKLOADS = {
    "tiny": Workload("tiny", 256, 256, 8, 2, 512, 0, "learned"),
    "tiny64e_random": Workload("tiny64e_random", 8192, 2048, 64, 4, 1024, 1024, "random"),
    "tiny64e_zipf": Workload("tiny64e_zipf", 8192, 2048, 64, 4, 1024, 1024, "learned", zipf_bias=True),
    "tiny64e_zipf_cap125": Workload("tiny64e_zipf_cap125", 8192, 2048, 64, 4, 1024, 1024, "learned",
                                    zipf_bias=True, capacity_factor=1.25),
    "scale_E8": Workload("scale_E8", 16384, 2048, 8, 4, 768, 768, "learned", backward=True),
    "scale_E32": Workload("scale_E32", 16384, 2048, 32, 4, 768, 768, "learned", backward=True),
    "scale_E64": Workload("scale_E64", 16384, 2048, 64, 4, 768, 768, "learned", backward=True),
    "scale_E128": Workload("scale_E128", 16384, 2048, 128, 4, 768, 768, "learned", backward=True),
    "large_E128": Workload("large_E128", 8192, 4096, 128, 4, 1536, 1536, "learned", backward=True),
    # the per-expert shapes of large_E128 (256 rows per expert, d=4096,
    # H=Hs=1536) with 16 experts and 1024 tokens: a case of a few GB for
    # profiling the same tiles with many counters
    "large_E16_slice": Workload("large_E16_slice", 1024, 4096, 16, 4, 1536, 1536, "learned", backward=True),
}


def custom(name="custom", *, T, d, E, k, H, Hs, routing="learned", zipf_bias=False,
           capacity_factor=0.0, backward=True) -> Workload:
    return Workload(name, T, d, E, k, H, Hs, routing, zipf_bias, capacity_factor, backward)


def expert_weights(w: Workload, e: int, base: int = gen.BASE_SEED):
    """bf16 bits of expert e's (W_g[e] [H,d], W_u[e] [H,d], W_d[e] [d,H]),
    regenerated on their own from the counter-based streams."""
    n = w.H * w.d
    Wg = gen.normal_bf16("W_g", (w.H, w.d), WEIGHT_STD, start=e * n, base=base)
    Wu = gen.normal_bf16("W_u", (w.H, w.d), WEIGHT_STD, start=e * n, base=base)
    Wd = gen.normal_bf16("W_d", (w.d, w.H), WEIGHT_STD, start=e * n, base=base)
    return Wg, Wu, Wd


def make_inputs(w: Workload, base: int = gen.BASE_SEED, weights: bool = True) -> dict:
    """All inputs of one layer call as numpy arrays (bf16 as uint16 bits)."""
    T, d, E, H, Hs = w.T, w.d, w.E, w.H, w.Hs
    inp = {"x": gen.normal_bf16("x", (T, d), 1.0, base=base)}
    if w.routing == "random":
        inp["logits_in"] = gen.random_routing_logits(T, E, w.k, base=base)
    else:
        inp["W_r"] = gen.normal_bf16("W_r", (E, d), WEIGHT_STD, base=base)
        if w.zipf_bias:
            inp["bias"] = gen.zipf_bias(E, base=base)
    if weights:
        inp["W_g"] = gen.normal_bf16("W_g", (E, H, d), WEIGHT_STD, base=base)
        inp["W_u"] = gen.normal_bf16("W_u", (E, H, d), WEIGHT_STD, base=base)
        inp["W_d"] = gen.normal_bf16("W_d", (E, d, H), WEIGHT_STD, base=base)
        if Hs > 0:
            inp["Ws_g"] = gen.normal_bf16("Ws_g", (Hs, d), WEIGHT_STD, base=base)
            inp["Ws_u"] = gen.normal_bf16("Ws_u", (Hs, d), WEIGHT_STD, base=base)
            inp["Ws_d"] = gen.normal_bf16("Ws_d", (d, Hs), WEIGHT_STD, base=base)
    if w.backward:
        inp["dY"] = gen.normal_bf16("dY", (T, d), 1.0, base=base)
    return inp
