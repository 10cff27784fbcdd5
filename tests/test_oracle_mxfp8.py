"""Pins of the MXFP8 oracle (oracle/mxfp8.py) to things other than itself:
values the E4M3 format definition fixes, a brute-force nearest-value search
over all 256 codes, the block-scale rule in closed form, the format's
relative error bound, exactness on inputs the format represents without loss,
and agreement with the unquantized expert MLP within the quantization error."""
import numpy as np
import pytest

from oracle import moe_oracle as orc
from oracle import mxfp8 as mx


def test_e4m3_values_fixed_by_the_format():
    t = mx.e4m3_decode_table()
    assert t[0x00] == 0.0
    assert t[0x01] == 2.0 ** -9          # smallest subnormal: 2^-6 * 1/8
    assert t[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x38] == 1.0                # exponent field 7 = bias
    assert t[0x3F] == 1.875
    assert t[0x7E] == 448.0              # largest normal: 1.75 * 2^8
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    assert t[0xB8] == -1.0 and t[0xFE] == -448.0
    finite = t[~np.isnan(t)]
    assert len(np.unique(finite)) == 253  # 254 finite codes, +0 and -0 equal
    # every integer 0..16 is representable (3 mantissa bits), 17 is not
    assert all(float(n) in set(finite) for n in range(17)) and 17.0 not in set(finite)


def brute_force_round(v):
    """Nearest finite E4M3 value by exhaustive search; ties to the code whose
    mantissa is even; beyond +-448 the largest magnitude (saturation)."""
    t = mx.e4m3_decode_table()
    codes = [c for c in range(128) if not np.isnan(t[c])]  # non-negative codes
    out = np.empty_like(v)
    for i, x in enumerate(v):
        a = abs(x)
        if a >= 448.0:
            r = 448.0
        else:
            d = [abs(a - t[c]) for c in codes]
            best = min(d)
            cands = [c for c, dc in zip(codes, d) if dc == best]
            if len(cands) > 1:
                cands = [c for c in cands if (c & 1) == 0]
            r = t[cands[0]]
        out[i] = np.copysign(r, x)
    return out


def test_e4m3_rounding_is_the_nearest_value_ties_to_even():
    rng = np.random.default_rng(7)
    t = mx.e4m3_decode_table()
    pos = np.sort(np.unique(t[(~np.isnan(t)) & (t >= 0)]))
    mids = (pos[:-1] + pos[1:]) / 2                      # exact ties
    logu = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(600.0), 3000))
    vals = np.concatenate([pos, mids, logu, [449.0, 463.9, 464.0, 470.0, 1e6, 0.0, 2.0 ** -11, 2.0 ** -10]])
    vals = np.concatenate([vals, -vals])
    np.testing.assert_array_equal(mx.e4m3_round(vals), brute_force_round(vals))
    # two ties by hand: 1.0625 lies between 1.0 (mantissa 0) and 1.125 (1)
    assert mx.e4m3_round(np.array([1.0625]))[0] == 1.0
    # 1.1875 between 1.125 (mantissa 1) and 1.25 (mantissa 2)
    assert mx.e4m3_round(np.array([1.1875]))[0] == 1.25
    # codes decode back to the rounded values
    r = mx.e4m3_round(vals)
    np.testing.assert_array_equal(t[mx.e4m3_encode(vals).astype(np.int64)], r)


def test_block_scale_rule_and_saturation():
    # amax = m * 2^e with m in [1, 2): shared exponent e - 8
    for e in (-20, -3, 0, 5, 30):
        for m in (1.0, 1.3, 1.75, 1.99):
            v = np.zeros(32)
            v[5] = m * 2.0 ** e
            v[9] = -0.25 * 2.0 ** e
            codes, scales = mx.mx_quantize(v[None, :])
            assert int(scales[0, 0]) == e - 8 + 127
            back = mx.mx_dequantize(codes, scales)[0]
            if m <= 1.75:
                # the largest element is represented within half a step of its binade
                assert abs(back[5] - v[5]) <= 2.0 ** (e - 4)
            else:
                # above 1.75 * 2^e the element saturates at 448 * X = 1.75 * 2^e
                assert back[5] == 1.75 * 2.0 ** e
            assert back[9] == v[9]  # a power of two inside the range is exact
    # all-zero block: smallest scale, zero codes
    codes, scales = mx.mx_quantize(np.zeros((2, 64)))
    assert np.all(codes == 0) and np.all(scales == 0)
    with pytest.raises(ValueError):
        mx.mx_quantize(np.zeros((2, 48)))


def test_roundtrip_error_bound():
    rng = np.random.default_rng(3)
    v = rng.normal(size=(64, 256)) * np.exp(rng.uniform(-8, 8, size=(64, 1)))
    codes, scales = mx.mx_quantize(v, axis=1)
    back = mx.mx_dequantize(codes, scales, axis=1)
    X = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    err = np.abs(back - v)
    normal = np.abs(v) >= X * 2.0 ** -6
    sat = np.abs(v) > 448.0 * X
    # 3 mantissa bits: half a step is 2^-4 of the value's binade
    assert np.all(err[normal & ~sat] <= np.abs(v[normal & ~sat]) * 2.0 ** -4)
    # below the normal range of the block: half the subnormal step 2^-9 X
    assert np.all(err[~normal] <= X[~normal] * 2.0 ** -10)
    assert np.all(np.abs(back[sat]) == 448.0 * X[sat])


def representable_blocks(rng, rows, cols):
    """Values n * 2^p with |n| <= 14 and, in every block of 32 along a row,
    one |n| in 8..14: the block's scale is 2^(p - 5) and every n * 2^5 <= 448
    is an E4M3 value, so quantization loses nothing.  p differs per block."""
    n = rng.integers(-14, 15, size=(rows, cols)).astype(np.float64)
    n[:, ::32] = rng.choice([-14, -11, -8, 8, 9, 12, 14], size=(rows, cols // 32))
    p = rng.integers(-6, 7, size=(rows, cols // 32))
    return n * np.repeat(np.ldexp(1.0, p), 32, axis=1)


def test_mx_matmul_is_exact_on_representable_inputs():
    rng = np.random.default_rng(11)
    a = representable_blocks(rng, 40, 256)
    b = representable_blocks(rng, 24, 256)
    codes, scales = mx.mx_quantize(a, axis=1)
    np.testing.assert_array_equal(mx.mx_dequantize(codes, scales, axis=1), a)
    np.testing.assert_array_equal(mx.mx_matmul_nt(a, b), a @ b.T)
    # blocks run along K, one scale per row and block: two rows 20 binades
    # apart are each exact, while a block across rows (the other axis) puts
    # the small row 15 binades below its scale, under E4M3's range
    blk = np.full((32, 32), 9.0)
    blk[0, :] = 13.0
    blk[1, :] = 13.0 * 2.0 ** 20
    ck, sk = mx.mx_quantize(blk, axis=1)
    np.testing.assert_array_equal(mx.mx_dequantize(ck, sk, axis=1), blk)
    ct, st = mx.mx_quantize(blk, axis=0)
    assert np.all(mx.mx_dequantize(ct, st, axis=0)[0] == 0.0)


def test_mxfp8_expert_agrees_with_the_unquantized_expert_within_the_quantization_error():
    """Each MX operand carries a relative error of at most 2^-4 (about
    2^-4 / sqrt(3) rms for values spread over a binade); a product of two
    such operands summed over K keeps about sqrt(2) of that, and the down
    projection adds its own: well under 10 % relative Frobenius error, and
    far from zero (the operands were quantized)."""
    rng = np.random.default_rng(5)
    n, d, H = 96, 256, 128
    x = orc.bf16_to_f64(rng.normal(size=(n, d)).astype(np.float32).view(np.uint32) >> 16)
    Wg, Wu = (orc.bf16_to_f64((rng.normal(size=(H, d)) * 0.02).astype(np.float32).view(np.uint32) >> 16)
              for _ in range(2))
    Wd = orc.bf16_to_f64((rng.normal(size=(d, H)) * 0.02).astype(np.float32).view(np.uint32) >> 16)
    a, u, h, o = mx.mxfp8_swiglu_fwd(x, Wg, Wu, Wd)
    a0, u0, h0, o0 = orc.swiglu_fwd(x, Wg, Wu, Wd)
    for got, ref in ((a, a0), (u, u0), (o, o0)):
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert 1e-3 < rel < 0.1, rel
    # the grouped form: rows of expert e go through expert e's weights only,
    # and an expert with no rows contributes nothing.  Expert 1 (no rows)
    # doubles every weight; expert 2 is expert 0 with W_d negated, which MX
    # represents exactly (same scales, sign-flipped codes)
    Wg3, Wu3 = (np.stack([W, W * 2.0, W]) for W in (Wg, Wu))
    Wd3 = np.stack([Wd, Wd * 2.0, -Wd])
    offsets = np.array([0, 40, 40, n])
    o_perm = mx.mxfp8_grouped_swiglu_fwd(x, offsets, Wg3, Wu3, Wd3)
    np.testing.assert_array_equal(o_perm[:40], mx.mxfp8_swiglu_fwd(x[:40], Wg, Wu, Wd)[3])
    np.testing.assert_array_equal(o_perm[40:], -mx.mxfp8_swiglu_fwd(x[40:], Wg, Wu, Wd)[3])


def test_vectorized_encoder_equals_the_elementwise_lookup():
    """The vectorized E4M3 encoder returns the element-wise dictionary lookup's
    code for every finite code value, their midpoints, values past 448 and
    random values across the format's range."""
    t = mx.e4m3_decode_table()
    vals = t[~np.isnan(t)]
    mids = (np.sort(np.unique(np.abs(vals)))[1:] + np.sort(np.unique(np.abs(vals)))[:-1]) / 2
    rng = np.random.default_rng(7)
    rand = rng.standard_normal(4000) * np.exp2(rng.integers(-12, 10, 4000))
    v = np.concatenate([vals, mids, -mids, [500.0, -1e6, 0.0, -0.0], rand])
    assert np.array_equal(mx.e4m3_encode(v), mx.e4m3_encode_elementwise(v))


def test_rounding_keeps_the_sign_of_zero():
    """A negative value that rounds to zero encodes as -0 (0x80), a positive
    one and +0 as +0 (0x00), as round-to-nearest does in IEEE arithmetic."""
    v = np.array([-1e-9, -0.0, 0.0, 1e-9, -2.0 ** -11, 2.0 ** -11])
    assert mx.e4m3_encode(v).tolist() == [0x80, 0x80, 0x00, 0x00, 0x80, 0x00]
    assert np.array_equal(mx.e4m3_encode_elementwise(v), mx.e4m3_encode(v))
