"""Host-side accounting of bench.py: the per-kernel algorithmic FLOPs add up
to the step's GEMM FLOPs counted from the layer's shapes, the split-precision
kernels' issued MMA work, and the roofline's choice of the binding roof."""
import pytest

import bench

FWD = ["gemm_gate_up_swiglu", "gemm_down"]
BWD = ["gemm_dgrad_down_swiglu_bwd", "gemm_wgrad_down", "gemm_dgrad_gate_up", "gemm_wgrad_gate_up"]
ROUTER_FWD = ["gemm_router"]
ROUTER_BWD = ["gemm_router_dw", "gemm_router_dx"]


@pytest.mark.parametrize("name", ["tiny", "tiny64e_random", "tiny64e_zipf", "scale_E8", "large_E128"])
def test_kernel_flops_add_up_to_the_step(name):
    w = bench.backward_workload(name)
    R = w.T * w.k
    work = bench.kernel_work(w, R)
    fwd, bwd = bench.gemm_flops(w, R)
    learned = w.routing == "learned"
    f = sum(work[n][0] for n in FWD + (ROUTER_FWD if learned else []))
    b = sum(work[n][0] for n in BWD + (ROUTER_BWD if learned else []))
    assert f == pytest.approx(fwd, rel=1e-12)
    assert b == pytest.approx(bwd, rel=1e-12)


def test_issued_mma_work_of_the_split_kernels():
    w = bench.backward_workload("large_E128")
    R = w.T * w.k
    work = bench.kernel_work(w, R)
    issued = bench.issued_mma_flops(w, R)
    # weight gradients: every K step issued with both halves
    assert issued["gemm_wgrad_gate_up"] == 2 * work["gemm_wgrad_gate_up"][0]
    assert issued["gemm_wgrad_down"] == 2 * work["gemm_wgrad_down"][0]
    # dgrad of gate/up: only the shared expert's rows (T of R + T) twice
    shared = 4.0 * w.d * w.T * w.Hs
    assert issued["gemm_dgrad_gate_up"] == work["gemm_dgrad_gate_up"][0] + shared
    # kernels without a split operand are not listed
    for n in FWD + ["gemm_dgrad_down_swiglu_bwd", "gemm_router"]:
        assert n not in issued


def test_issued_fraction_beside_the_algorithmic_one():
    row = {}
    bench.with_issued(row, "gemm_wgrad_gate_up", {"gemm_wgrad_gate_up": 2e12}, 2.0, 1000.0)
    assert row == {"issued_mma_flops": 2e12, "issued_tensor_frac": 1.0}
    row = {}
    bench.with_issued(row, "combine", {"gemm_wgrad_gate_up": 2e12}, 2.0, 1000.0)
    assert row == {}


def test_roofline_takes_the_binding_roof():
    # 1 TFLOP and 1 GB in 1 ms at 2000 TFLOP/s and 5000 GB/s: the tensor roof
    # takes 0.5 ms, the HBM roof 0.2 ms
    r = bench.kernel_roofline((1e12, 1e9), 1.0, 2000.0, 5000.0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(1000.0) and r["frac"] == pytest.approx(0.5)
    assert r["hbm_frac"] == pytest.approx(0.2)
    # the same bytes with a tenth of the FLOPs: HBM binds
    r = bench.kernel_roofline((1e11, 1e9), 1.0, 2000.0, 5000.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(1000.0) and r["frac"] == pytest.approx(0.2)
    assert r["tensor_frac"] == pytest.approx(0.05)


def test_reference_arm_line_contract():
    """`bench.py --impl reference` (the C++ oracle on the host cores) prints
    one JSON line with the keys of the benchmark contract."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "2", "--warmup", "1", "--cpu-sample-tokens", "16"],
                         capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["workload"] == "tiny" and d["config"]["sample_tokens"] == 16
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
