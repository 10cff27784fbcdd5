"""The C++ oracle (oracle/moe_oracle.cpp) against the numpy oracle, two
implementations written separately from the same definitions: every routing
and permutation output identical, every float output and gradient equal to
float64 rounding.  Both are pinned on their own by tests/test_oracle_pins.py;
here they must also agree on layers of the workload table's kinds (random
and learned routing, Zipf bias, capacity drops, no shared expert)."""
import numpy as np
import pytest

from oracle import moe_oracle as orc
from oracle import moe_oracle_cpp as orc_cpp
from synth import workloads

CASES = {
    "learned_shared": dict(T=300, d=64, E=8, k=2, H=128, Hs=64, routing="learned"),
    "zipf_capacity": dict(T=513, d=128, E=16, k=4, H=128, Hs=128, routing="learned", zipf_bias=True,
                          capacity_factor=1.25),
    "random_routing": dict(T=256, d=64, E=32, k=4, H=64, Hs=64, routing="random"),
    "no_shared_k1": dict(T=97, d=64, E=8, k=1, H=64, Hs=0, routing="learned"),
}
INT_KEYS = ("idx", "counts_raw", "counts", "offsets", "row_of_slot", "slot_of_row")
FWD_KEYS = ("gates", "x_perm", "a", "u", "h", "o", "y")
BWD_KEYS = ("dgates", "dx_perm", "dW_g", "dW_u", "dW_d", "dlogits", "dx")


@pytest.mark.parametrize("name", list(CASES))
def test_cpp_oracle_agrees_with_numpy_oracle(name):
    w = workloads.custom(name, backward=True, **CASES[name])
    inp = workloads.make_inputs(w)
    a, b = orc.inputs_to_f64(inp), orc_cpp.inputs_to_f64(inp)
    cap = orc.capacity_of(w.T, w.k, w.E) if w.capacity_factor else 0
    fa, fb = orc.layer_forward(a, w.k, cap), orc_cpp.layer_forward(b, w.k, cap)
    ba, bb = orc.layer_backward(a, fa), orc_cpp.layer_backward(b, fb)
    assert np.array_equal(np.asarray(fa["logits"]), np.asarray(fb["logits"]))
    for key in INT_KEYS:
        assert np.array_equal(fa[key], fb[key]), key
    extra_f = ("a_s", "u_s", "h_s", "s") if w.Hs else ()
    extra_b = ("dx_s", "dWs_g", "dWs_u", "dWs_d") if w.Hs else ()
    extra_b += ("dW_r",) if w.routing == "learned" else ()
    for key in FWD_KEYS + extra_f:
        np.testing.assert_allclose(fb[key], fa[key], rtol=1e-12, atol=1e-12, err_msg=key)
    for key in BWD_KEYS + extra_b:
        np.testing.assert_allclose(bb[key], ba[key], rtol=1e-11, atol=1e-12, err_msg=key)


def test_cpp_oracle_results_do_not_depend_on_the_thread_count():
    """Rows and experts are split over the workers; no sum is split, so the
    results are bit-identical for any number of threads."""
    w = workloads.custom("threads", T=200, d=64, E=8, k=2, H=64, Hs=64, backward=True)
    inp = orc_cpp.inputs_to_f64(workloads.make_inputs(w))
    res = []
    for n in (1, 3, 0):
        orc_cpp.set_threads(n)
        f = orc_cpp.layer_forward(inp, w.k, 0)
        res.append((f["y"], orc_cpp.layer_backward(inp, f)["dx"]))
    orc_cpp.set_threads(0)
    for y, dx in res[1:]:
        assert np.array_equal(y, res[0][0]) and np.array_equal(dx, res[0][1])
