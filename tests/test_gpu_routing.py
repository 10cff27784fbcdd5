"""GPU parity of the routing, permutation and combine kernels against the CPU
oracle, through the C ABI.  Integer results (top-k indices, counts, offsets,
row maps, permuted rows) must be bit-exact when both sides get the same fp32
logits; floating results meet the layer tolerance."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from synth import gen
from tests.gpu_util import assert_close, dev_bf16, dev_f32, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def adversarial_logits(T, E, seed):
    l = gen.random_logits(T, E, tensor=100 + seed)
    l[0] = 0.0
    if T > 1:
        l[1, ::3] = 5.0
    if T > 2:
        l[2] = -0.0
        l[2, E // 2] = 0.0
    if T > 3:
        l[3, : E // 2] = -np.inf
    if T > 4:
        l[4] = np.round(l[4])
    if T > 6:
        l[6:T:7] = np.round(l[6:T:7] * 2) / 2  # many ties
    return l


def run_topk(B, logits, k):
    T, E = logits.shape
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    g = torch.empty(T, k, dtype=torch.float32, device="cuda")
    B.moe_route_topk(None, None, None, dev_f32(logits), T, 0, E, k, None, idx, g, None, 0)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), g.cpu().numpy()


@pytest.mark.parametrize("T,E,k", [(1, 8, 1), (37, 8, 2), (1000, 64, 4), (777, 128, 4), (300, 256, 8),
                                   (513, 32, 8), (64, 8, 8)])
def test_topk_bit_exact_given_logits(B, T, E, k):
    l = adversarial_logits(T, E, seed=T + E + k)
    idx, g = run_topk(B, l, k)
    ridx, rg = orc.route_topk(l, k)
    assert np.array_equal(idx, ridx)
    np.testing.assert_allclose(g, rg, rtol=2e-6, atol=1e-7)


def run_permute(B, x_bits, idx, E, capacity):
    T, k = idx.shape
    d = x_bits.shape[1]
    ws_bytes = B.moe_workspace_size(T, d, E, k, 128, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    o = {n: torch.full((m,), -7, dtype=torch.int32, device="cuda") for n, m in
         (("counts_raw", E), ("counts", E), ("offsets", E + 1), ("row_of_slot", T * k), ("slot_of_row", T * k))}
    x = dev_bf16(x_bits)
    x_perm = torch.zeros(T * k, d, dtype=torch.bfloat16, device="cuda")
    B.moe_permute(x, torch.from_numpy(idx.astype(np.int32)).cuda(), T, d, E, k, capacity, o["counts_raw"],
                  o["counts"], o["offsets"], o["row_of_slot"], o["slot_of_row"], x_perm, ws, ws_bytes)
    torch.cuda.synchronize()
    out = {n: v.cpu().numpy() for n, v in o.items()}
    out["x_perm"] = x_perm.view(torch.int16).cpu().numpy().view(np.uint16)
    return out


def check_permute(out, ref, x_bits, k):
    for key in ("counts_raw", "counts", "offsets", "row_of_slot"):
        assert np.array_equal(out[key], ref[key]), key
    R = int(ref["offsets"][-1])
    assert np.array_equal(out["slot_of_row"][:R], ref["slot_of_row"])
    assert np.array_equal(out["x_perm"][:R], x_bits[ref["slot_of_row"] // k])


@pytest.mark.parametrize("T,E,k,cap,skew", [
    (1, 8, 1, 0, 0.0), (1, 8, 2, 1, 0.0), (300, 8, 2, 0, 0.0), (300, 8, 2, 40, 2.0),
    (1000, 64, 4, 0, 0.0), (1000, 64, 4, orc.capacity_of(1000, 4, 64), 1.0),
    (4099, 128, 4, 0, 3.0), (700, 256, 8, 0, 0.0), (700, 256, 8, 5, 2.0)])
def test_permute_bit_exact(B, T, E, k, cap, skew):
    d = 128
    l = gen.random_logits(T, E, tensor=200 + T)
    l[:, : max(1, E // 16)] += skew  # skewed load: a few hot experts
    idx, _ = orc.route_topk(l, k)
    x_bits = gen.normal_bf16(300, (T, d))
    out = run_permute(B, x_bits, idx, E, cap)
    check_permute(out, orc.permute(idx, E, cap), x_bits, k)


def test_permute_all_tokens_to_the_same_experts(B):
    T, E, k, d = 2000, 64, 4, 64
    idx = np.tile(np.array([[5, 9, 0, 63]], dtype=np.int32), (T, 1))
    x_bits = gen.normal_bf16(301, (T, d))
    for cap in (0, 1, 300):
        out = run_permute(B, x_bits, idx, E, cap)
        check_permute(out, orc.permute(idx, E, cap), x_bits, k)


def test_permute_is_deterministic(B):
    T, E, k, d = 3000, 64, 4, 256
    idx, _ = orc.route_topk(gen.random_logits(T, E, tensor=302), k)
    x_bits = gen.normal_bf16(303, (T, d))
    a = run_permute(B, x_bits, idx, E, 0)
    for _ in range(2):
        b = run_permute(B, x_bits, idx, E, 0)
        for key in a:
            assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("cap", [0, 30])
def test_identity_expert_combine(B, cap):
    """o_perm = x_perm (identity experts), no shared expert: y = x * sum of kept gates."""
    T, E, k, d = 500, 16, 4, 256
    l = gen.random_logits(T, E, tensor=304)
    idx, g = run_topk(B, l, k)
    x_bits = gen.normal_bf16(305, (T, d))
    p = run_permute(B, x_bits, idx, E, cap)
    x_perm = dev_bf16(p["x_perm"]).half()   # expert outputs are fp16 (bf16 values of this size convert exactly)
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    B.moe_unpermute_combine(x_perm, None, dev_f32(g), torch.from_numpy(p["row_of_slot"]).cuda(), T, d, k, y)
    torch.cuda.synchronize()
    ref = orc.layer_forward({"x": orc.bf16_to_f64(x_bits)}, k, cap, logits=l, expert_fn=lambda e, xr: xr)
    assert_close("y", host_f64(y), ref["y"], atol=1e-2, rtol=1e-2, fro=4e-3)


def test_combine_bwd_gather_and_reduce(B):
    """moe_unpermute_combine_bwd gathers dY into the kept rows (bit copies);
    moe_permute_bwd sums rows back per token."""
    T, E, k, d = 600, 32, 4, 256
    l = gen.random_logits(T, E, tensor=306)
    idx, g = run_topk(B, l, k)
    x_bits = gen.normal_bf16(307, (T, d))
    p = run_permute(B, x_bits, idx, E, 20)
    R = int(p["offsets"][-1])
    o_bits = gen.normal_bf16(308, (T * k, d))
    dY_bits = gen.normal_bf16(309, (T, d))
    row = torch.from_numpy(p["row_of_slot"]).cuda()
    dYp = torch.zeros(T * k, d, dtype=torch.bfloat16, device="cuda")
    B.moe_unpermute_combine_bwd(dev_bf16(dY_bits), row, T, d, k, dYp)
    # reduce: dx = sum_s dx_perm[row] + dx_s, with dx_perm = o, dx_s = dY (fp16 inputs: the bf16 values of
    # this size convert exactly)
    dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    B.moe_permute_bwd(dev_bf16(o_bits).half(), dev_bf16(dY_bits).half(), row, None, None, T, d, E, k, dx, None, 0)
    torch.cuda.synchronize()
    # the oracle routes the same generator logits on its own
    ridx, rg = orc.route_topk(l, k)
    rp = orc.permute(ridx, E, 20)
    assert int(rp["offsets"][-1]) == R
    got = dYp.view(torch.int16).cpu().numpy().view(np.uint16)[:R]
    assert np.array_equal(got, dY_bits[rp["slot_of_row"] // k])
    o = orc.bf16_to_f64(o_bits)
    dY = orc.bf16_to_f64(dY_bits)
    ref_dx = orc.permute_bwd(o[:R], dY, rp["row_of_slot"], T, k)
    assert_close("dx", host_f64(dx), ref_dx)


def test_router_bwd_dlogits(B):
    T, E, k = 700, 64, 4
    l = gen.random_logits(T, E, tensor=310)
    idx, g = run_topk(B, l, k)
    dg = gen.random_logits(T, k, tensor=311)  # N(0,1) upstream gate gradients
    dl = torch.empty(T, E, dtype=torch.float32, device="cuda")
    B.moe_route_topk_bwd(dev_f32(dg), dev_f32(g), torch.from_numpy(idx).cuda(), None, T, 0, E, k, dl, None, None, 0)
    torch.cuda.synchronize()
    ridx, rg = orc.route_topk(l, k)
    ref = orc.topk_bwd(rg, ridx, dg.astype(np.float64), E)
    np.testing.assert_allclose(dl.cpu().numpy(), ref, rtol=1e-5, atol=1e-6)


def test_sum_terms_out_of_fp16_range_are_reported(B):
    """The per-token sums read fp16 terms: a term beyond the fp16 range is
    stored as inf, and the combine and the unpermute reduce then report
    MOE_ERR_RANGE in the device status (an inf planted here on the host); a
    finite sum reports nothing."""
    T, E, k, d = 64, 8, 2, 128
    l = gen.random_logits(T, E, tensor=310)
    idx, g = run_topk(B, l, k)
    x_bits = gen.normal_bf16(311, (T, d))
    p = run_permute(B, x_bits, idx, E, 0)
    row = torch.from_numpy(p["row_of_slot"]).cuda()
    terms = dev_bf16(gen.normal_bf16(312, (T * k, d))).half()
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    assert B.moe_device_status() == 0
    B.moe_unpermute_combine(terms, None, dev_f32(g), row, T, d, k, y)
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    kept_row = int(p["row_of_slot"][0])
    assert kept_row >= 0
    terms[kept_row, 5] = float("inf")
    B.moe_unpermute_combine(terms, None, dev_f32(g), row, T, d, k, y)
    torch.cuda.synchronize()
    assert B.moe_device_status() == B.MOE_ERR_RANGE
    dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    B.moe_permute_bwd(terms, None, row, None, None, T, d, E, k, dx, None, 0)
    torch.cuda.synchronize()
    assert B.moe_device_status() == B.MOE_ERR_RANGE
    assert B.moe_device_status() == 0  # read and cleared
