"""The MXFP8 expert MLP on the GPU against the MXFP8 oracle (oracle/mxfp8.py):
quantized codes and block scales bit-exact (the row quantizer, the packed
gate/up weights, x inside the permutation), routing and the padded row maps
bit-exact, and the expert outputs, the shared expert and the combined layer
output within tolerance of the oracle's MXFP8 expert MLP.

h is quantized on the GPU from fp32 values (fast-math sigmoid) and in the
oracle from float64 ones, so a code of h may differ where h / X falls within
rounding distance of an E4M3 midpoint: such codes must be adjacent values
and rare; everything downstream is compared within tolerance."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from oracle import mxfp8 as mx
from synth import gen, workloads
from tests.gpu_util import assert_close, host_f64, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def unatom(atoms: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """The documented tile-atom scale layout -> [rows, cols/32]."""
    nq, nb = cols // 128, cols // 32
    r = np.arange(rows)[:, None]
    b = np.arange(nb)[None, :]
    off = ((r >> 7) * nq + (b >> 2)) * 512 + 16 * (r & 31) + 4 * ((r & 127) >> 5) + (b & 3)
    return atoms[off]


def u8(n):
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def quantize_gpu(B, bits: np.ndarray):
    rows, cols = bits.shape
    codes = u8(rows * cols)
    scales = u8(B.moe_mxfp8_scales_bytes(rows, cols))
    B.moe_mxfp8_quantize(upload({"x": bits})["x"], rows, cols, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy().reshape(rows, cols), unatom(scales.cpu().numpy(), rows, cols)


def test_quantizer_codes_and_scales_are_bit_exact(B):
    rows, cols = 300, 384
    v = gen.normal_bf16(601, (rows, cols)).astype(np.uint16)
    f = orc.bf16_to_f64(v)
    # edge blocks: all zero, bf16 subnormals, the largest bf16 values, values
    # that land exactly on E4M3 midpoints after scaling (ties to even), mixed
    # magnitudes that flush to zero
    f[0, :32] = 0.0
    f[1, :32] = np.ldexp(np.arange(1, 33), -133)
    f[2, :32] = 3.0e38 * np.sign(np.arange(32) - 15.5)
    f[3, :32] = np.ldexp(np.array([256.0 + 16.0 * (2 * i + 1) for i in range(8)] * 4), -20)
    f[4, :32] = np.ldexp(1.0, -30)
    f[4, 0] = 1.0e4
    f[5, :] *= np.ldexp(1.0, np.repeat(np.arange(-60, 60, 10), 32))[:cols]
    bits = gen.f64_to_bf16_bits(f)
    fb = orc.bf16_to_f64(bits)
    codes, scales = quantize_gpu(B, bits)
    qc, qs = mx.mx_quantize(fb, axis=1)
    assert np.array_equal(scales, qs)
    assert np.array_equal(codes, qc)


def test_packed_gate_up_weights_are_bit_exact(B):
    E, H, d = 3, 256, 256
    Wg = gen.normal_bf16(602, (E, H, d), std=0.02)
    Wu = gen.normal_bf16(603, (E, H, d), std=0.02)
    dev = upload({"W_g": Wg, "W_u": Wu})
    codes = u8(E * 2 * H * d)
    scales = u8(B.moe_mxfp8_scales_bytes(E * 2 * H, d))
    B.moe_mxfp8_quantize_gate_up(dev["W_g"], dev["W_u"], E, H, d, codes, scales)
    torch.cuda.synchronize()
    # packed row 128 j + r of an expert: W_g row 64 j + r (r < 64), else W_u row 64 j + r - 64
    p = np.arange(2 * H)
    src = 64 * (p // 128) + (p % 128) % 64
    from_u = (p % 128) >= 64
    packed = np.where(from_u[None, :, None], orc.bf16_to_f64(Wu)[:, src], orc.bf16_to_f64(Wg)[:, src])
    qc, qs = mx.mx_quantize(packed.reshape(E * 2 * H, d), axis=1)
    assert np.array_equal(codes.cpu().numpy().reshape(E * 2 * H, d), qc)
    assert np.array_equal(unatom(scales.cpu().numpy(), E * 2 * H, d), qs)


CASES = {
    "small_capacity": dict(T=600, d=256, E=8, k=2, H=256, Hs=128, routing="learned", zipf_bias=True,
                           capacity_factor=1.25),
    "large_slice": dict(T=512, d=4096, E=8, k=4, H=1536, Hs=1536, routing="learned"),
}


def _random_cases(n=5, seed=20261203):
    """Seeded random shapes within the MXFP8 path's limits: d a multiple of
    128, E a multiple of 8, k <= min(8, E), H and Hs multiples of 128, a
    shared expert, learned routing (with the Zipf bias or a capacity on some)."""
    import random
    rng = random.Random(seed)
    out = {}
    for i in range(n):
        E = rng.choice([8, 16, 24, 40, 64])
        out[f"random{i}"] = dict(T=rng.randint(1, 600), d=128 * rng.randint(1, 4), E=E, k=rng.randint(1, min(8, E)),
                                 H=128 * rng.randint(1, 4), Hs=128 * rng.randint(1, 2), routing="learned",
                                 zipf_bias=rng.random() < 0.3, capacity_factor=rng.choice([0.0, 1.25, 0.5]))
    return out


CASES.update(_random_cases())


def run_mx_layer(B, w, inp):
    """Routing (bf16 path), the MX permutation, the weights quantized, the MX
    expert MLP and the combine; returns every buffer as numpy."""
    T, d, E, k, H, Hs = w.T, w.d, w.E, w.k, w.H, w.Hs
    dev = upload(inp)
    i32 = lambda n: torch.empty(n, dtype=torch.int32, device="cuda")  # noqa: E731
    f32 = lambda *s: torch.empty(*s, dtype=torch.float32, device="cuda")  # noqa: E731
    ws_bytes = B.moe_workspace_size(T, d, E, k, H, Hs)
    ws = u8(ws_bytes)
    logits, idx, gates = f32(T, E), i32(T * k), f32(T * k)
    B.moe_route_topk(dev["x"], dev["W_r"], dev.get("bias"), None, T, d, E, k, logits, idx, gates, ws, ws_bytes)
    rows = B.moe_mxfp8_rows(T, E, k)
    cap = w.capacity
    counts_raw, counts, offsets, mxoff = i32(E), i32(E), i32(E + 1), i32(E + 1)
    row_of_slot, slot_of_row = i32(T * k), i32(rows)
    x_codes, x_scales = u8(rows * d), u8(B.moe_mxfp8_scales_bytes(rows, d))
    B.moe_permute_mxfp8(dev["x"], idx, T, d, E, k, cap, counts_raw, counts, offsets, mxoff, row_of_slot,
                        slot_of_row, x_codes, x_scales, ws, ws_bytes)
    # weights and the shared expert's input, quantized once
    Wgu_c, Wgu_s = u8(E * 2 * H * d), u8(B.moe_mxfp8_scales_bytes(E * 2 * H, d))
    Wd_c, Wd_s = u8(E * d * H), u8(B.moe_mxfp8_scales_bytes(E * d, H))
    B.moe_mxfp8_quantize_gate_up(dev["W_g"], dev["W_u"], E, H, d, Wgu_c, Wgu_s)
    B.moe_mxfp8_quantize(dev["W_d"], E * d, H, Wd_c, Wd_s)
    Wsgu_c, Wsgu_s = u8(2 * Hs * d), u8(B.moe_mxfp8_scales_bytes(2 * Hs, d))
    Wsd_c, Wsd_s = u8(d * Hs), u8(B.moe_mxfp8_scales_bytes(d, Hs))
    xs_c, xs_s = u8(T * d), u8(B.moe_mxfp8_scales_bytes(T, d))
    B.moe_mxfp8_quantize_gate_up(dev["Ws_g"], dev["Ws_u"], 1, Hs, d, Wsgu_c, Wsgu_s)
    B.moe_mxfp8_quantize(dev["Ws_d"], d, Hs, Wsd_c, Wsd_s)
    B.moe_mxfp8_quantize(dev["x"], T, d, xs_c, xs_s)
    h_c, h_s = u8(rows * H), u8(B.moe_mxfp8_scales_bytes(rows, H))
    hs_c, hs_s = u8(T * Hs), u8(B.moe_mxfp8_scales_bytes(T, Hs))
    # fp16 sum terms; padding rows stay NaN
    o_perm = torch.full((rows, d), float("nan"), dtype=torch.float16, device="cuda")
    s = torch.empty(T, d, dtype=torch.float16, device="cuda")
    B.moe_grouped_swiglu_mxfp8(x_codes, x_scales, mxoff, counts, xs_c, xs_s, T, d, E, k, H, Hs, Wgu_c, Wgu_s,
                               Wd_c, Wd_s, Wsgu_c, Wsgu_s, Wsd_c, Wsd_s, h_c, h_s, hs_c, hs_s, o_perm, s)
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    B.moe_unpermute_combine_mxfp8(o_perm, s, gates, row_of_slot, T, d, E, k, y)
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    g = lambda t: t.cpu().numpy()  # noqa: E731
    return {"logits": g(logits), "idx": g(idx).reshape(T, k), "gates": g(gates).reshape(T, k),
            "counts_raw": g(counts_raw), "counts": g(counts), "offsets": g(offsets), "mx_offsets": g(mxoff),
            "row_of_slot": g(row_of_slot), "slot_of_row": g(slot_of_row), "rows": rows,
            "x_codes": g(x_codes).reshape(rows, d), "x_scales": unatom(g(x_scales), rows, d),
            "h_codes": g(h_c).reshape(rows, H), "h_scales": unatom(g(h_s), rows, H),
            "o_perm": g(o_perm), "s": g(s), "y": host_f64(y)}


@pytest.mark.parametrize("name", list(CASES))
def test_mxfp8_layer_forward_matches_the_mxfp8_oracle(B, name):
    w = workloads.custom(name, backward=False, **CASES[name])
    inp = workloads.make_inputs(w)
    gpu = run_mx_layer(B, w, inp)
    f64 = orc.inputs_to_f64(inp)
    T, k, E, H = w.T, w.k, w.E, w.H
    # routing on the GPU's own fp32 logits: bit-exact permutation
    ref = orc.layer_forward(f64, k, w.capacity, logits=gpu["logits"], expert_fn=lambda e, xr: xr)
    assert np.array_equal(gpu["idx"], ref["idx"])
    for key in ("counts_raw", "counts", "offsets"):
        assert np.array_equal(gpu[key], ref[key]), key
    padded = np.concatenate([[0], np.cumsum((ref["counts"] + 127) // 128 * 128)])
    assert np.array_equal(gpu["mx_offsets"], padded)
    kept = ref["row_of_slot"] >= 0
    e_of = ref["idx"].reshape(-1)
    want_rows = np.where(kept, padded[e_of] + ref["rank"].reshape(-1), -1)
    assert np.array_equal(gpu["row_of_slot"], want_rows)
    prow = want_rows[kept]
    tok = np.nonzero(kept)[0] // k
    assert np.array_equal(gpu["slot_of_row"][prow], np.nonzero(kept)[0])
    # x inside the permutation: every kept row holds its token's codes/scales
    qx, sx = mx.mx_quantize(f64["x"], axis=1)
    assert np.array_equal(gpu["x_codes"][prow], qx[tok])
    assert np.array_equal(gpu["x_scales"][prow], sx[tok])

    # the MXFP8 expert MLP per expert over its kept rows, in token order
    o_ref = np.zeros((len(prow), w.d))
    hq_ref = np.zeros((len(prow), H), dtype=np.uint8)
    order = np.argsort(prow)  # rows grouped by expert, token order within
    for e in range(E):
        sel = order[(e_of[kept][order] == e)]
        if len(sel) == 0:
            continue
        a, u, h, o = mx.mxfp8_swiglu_fwd(f64["x"][tok[sel]], f64["W_g"][e], f64["W_u"][e], f64["W_d"][e])
        o_ref[sel] = o
        hq_ref[sel] = mx.mx_quantize(h, axis=1)[0]
    # h codes: equal except rare flips at E4M3 midpoints, which are adjacent codes
    hg = gpu["h_codes"][prow]
    diff = hg != hq_ref
    assert diff.mean() < 1e-3, diff.mean()
    if diff.any():
        va, vb = mx._TABLE[hg[diff].astype(np.int64)], mx._TABLE[hq_ref[diff].astype(np.int64)]
        step = np.ldexp(1.0, np.maximum(np.frexp(np.maximum(np.abs(va), np.abs(vb)))[1] - 1, -6) - 3)
        assert np.all(np.abs(va - vb) <= step * 1.0000001), "an h code differs by more than one step"
    assert_close("o_perm (MXFP8)", gpu["o_perm"][prow], o_ref, fro=1e-3)
    _, _, _, s_ref = mx.mxfp8_swiglu_fwd(f64["x"], f64["Ws_g"], f64["Ws_u"], f64["Ws_d"])
    assert_close("s (MXFP8)", gpu["s"], s_ref, fro=1e-3)
    # the combined output with the GPU's gates (fp32) and the oracle's MXFP8 experts
    y_ref = s_ref.copy()
    gates = gpu["gates"].astype(np.float64).reshape(-1)
    np.add.at(y_ref, tok, gates[kept][:, None] * o_ref)
    assert_close("y (MXFP8)", gpu["y"], y_ref)
