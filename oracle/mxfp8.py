"""CPU oracle of the MXFP8 expert MLP (block-scaled FP8 operands).

TEST INFRASTRUCTURE ONLY.  Only the tests, `__graft_entry__.smoke()` and the
bench's CPU-baseline / reference leg may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA path.

The pages name the precision only: the largest runs of the "Olmo-core DDP MoE
examples" README ("Production throughput runs": MXFP8 with per-layer
recompute; "Other experiments in the report": the MXFP8 recipe ablation for
the MLP and the attention projections).  MXFP8 is the OCP Microscaling
format with FP8 E4M3 elements; the plainest reading of it, written out here:

  element   E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; normal
            values 2^(e-7) (1 + m/8) for e = 1..15 except e = 15, m = 7
            (NaN); subnormal 2^-6 (m/8); no infinities; largest 448.
  block     32 consecutive values along the contraction (K) dimension share
            one power-of-two scale X, stored as E8M0 (the biased exponent
            X = 2^(code - 127), codes 0..254; 255 = NaN).
  scale     X = 2^(floor(log2(max |v|)) - 8): 8 is the exponent of E4M3's
            largest normal binade, so the block's largest value lands in
            [256, 512); an all-zero block takes the smallest scale 2^-127.
  convert   code_i = E4M3(v_i / X), rounding to nearest, ties to the even
            mantissa, and saturating to +-448 (v / X can reach up to 512);
            a negative value that rounds to zero gives -0 (code 0x80), as
            rounding keeps the sign of zero in IEEE arithmetic.
  GEMM      C[m, n] = sum_k (A_code[m,k] X_A[m, k/32]) (B_code[n,k] X_B[n, k/32])
            summed exactly (float64 here; the tensor cores sum in fp32).
  expert    a = MX(x) MX(W_g)^T, u = MX(x) MX(W_u)^T, h = silu(a) u,
            o = MX(h) MX(W_d)^T: x and the weights are quantized along d, h
            along H (its quantization is the SwiGLU epilogue's last step);
            a, u, h are not rounded otherwise.

No blocking, fusion or reordering beyond these definitions; the only library
primitive is the matrix product.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import silu

BLOCK = 32
E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest normal binade: 448 = 1.75 * 2^8
E4M3_EMIN = -6         # exponent of the smallest normal: 2^-6
E4M3_MANT_BITS = 3
E8M0_BIAS = 127


def e4m3_decode_table() -> np.ndarray:
    """Value of every E4M3 code 0..255 (float64; NaN for the two NaN codes)."""
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            out[code] = np.nan
        elif e == 0:
            out[code] = s * 2.0 ** E4M3_EMIN * (m / 8.0)
        else:
            out[code] = s * 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return out


_TABLE = e4m3_decode_table()
# magnitude -> code of the non-negative finite values; the sign bit (0x80) is
# added for a negative rounded value, -0 included: rounding to nearest keeps
# the sign of a value that rounds to zero, as in IEEE arithmetic, and E4M3 has
# a negative zero (0x80)
_CODE_OF = {}
for _c in range(0x7F):
    _CODE_OF[float(_TABLE[_c])] = _c


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value of each v (ties to the even mantissa), saturating
    to +-448.  A value's rounding step is 2^(e-3) in its binade 2^e (e =
    floor(log2 |v|), at least -6: the subnormal step 2^-9 below 2^-6)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    mant, ex = np.frexp(a)                   # a = mant * 2^ex, mant in [0.5, 1)
    e = np.maximum(ex - 1, E4M3_EMIN)        # floor(log2 a), clamped to the subnormal binade
    step = np.ldexp(1.0, e - E4M3_MANT_BITS)
    q = np.rint(a / step) * step             # numpy rint: ties to even
    q = np.where(a == 0.0, 0.0, q)
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v)


def e4m3_encode_elementwise(v: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) of the rounded values of v, one element at a time
    through the value -> code dictionary."""
    r = e4m3_round(v)
    flat = r.ravel()
    codes = np.empty(flat.shape, dtype=np.uint8)
    for i, x in enumerate(flat):
        c = _CODE_OF[float(abs(x))]
        codes[i] = c | (0x80 if np.signbit(x) else 0)
    return codes.reshape(r.shape)


# the non-negative finite values in code order (codes 0x00..0x7E increase
# with the value), for the vectorized lookup
_POS_VALUES = _TABLE[:0x7F]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) of the rounded values of v: the same lookup as
    e4m3_encode_elementwise, vectorized (a rounded magnitude is one of the
    table's values exactly, found by binary search)."""
    r = e4m3_round(v)
    c = np.searchsorted(_POS_VALUES, np.abs(r)).astype(np.uint8)
    return np.where(np.signbit(r), c | np.uint8(0x80), c).astype(np.uint8)


def mx_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared exponent floor(log2 amax) - 8 of each block (int64), clamped to
    the E8M0 range [-127, 127]; -127 for an all-zero block."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)
    se = (ex - 1) - E4M3_EMAX
    se = np.where(amax == 0.0, -E8M0_BIAS, se)
    return np.clip(se, -E8M0_BIAS, E8M0_BIAS).astype(np.int64)


def mx_quantize(v: np.ndarray, axis: int = -1):
    """Quantize v along `axis` (its length a multiple of 32) in blocks of 32.

    Returns (codes uint8 of v's shape, scale codes uint8 with `axis` divided by
    32: E8M0 biased exponents)."""
    v = np.asarray(v, dtype=np.float64)
    axis = axis % v.ndim
    n = v.shape[axis]
    if n % BLOCK:
        raise ValueError(f"length {n} along axis {axis} is not a multiple of {BLOCK}")
    vm = np.moveaxis(v, axis, -1)
    blocks = vm.reshape(vm.shape[:-1] + (n // BLOCK, BLOCK))
    se = mx_scale_exponent(np.abs(blocks).max(axis=-1))           # [..., n/32]
    scaled = blocks / np.ldexp(1.0, se)[..., None]
    codes = e4m3_encode(scaled).reshape(vm.shape)
    scales = (se + E8M0_BIAS).astype(np.uint8)
    return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis)


def mx_dequantize(codes: np.ndarray, scales: np.ndarray, axis: int = -1) -> np.ndarray:
    """float64 values code * 2^(scale - 127), blocks of 32 along `axis`."""
    codes = np.asarray(codes, dtype=np.uint8)
    axis = axis % codes.ndim
    cm = np.moveaxis(codes, axis, -1)
    sm = np.moveaxis(np.asarray(scales, dtype=np.uint8), axis, -1)
    vals = _TABLE[cm.astype(np.int64)]
    x = np.ldexp(1.0, sm.astype(np.int64) - E8M0_BIAS)
    out = (vals.reshape(cm.shape[:-1] + (cm.shape[-1] // BLOCK, BLOCK)) * x[..., None]).reshape(cm.shape)
    return np.moveaxis(out, -1, axis)


def mx_matmul_nt(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """C = MX(a) MX(b)^T for a [M, K], b [N, K], both quantized along K."""
    qa, sa = mx_quantize(a, axis=1)
    qb, sb = mx_quantize(b, axis=1)
    return mx_dequantize(qa, sa, axis=1) @ mx_dequantize(qb, sb, axis=1).T


def mxfp8_swiglu_fwd(xr: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray):
    """One expert (or the shared expert) with MXFP8 operands: xr [n, d],
    Wg, Wu [H, d], Wd [d, H] (float64 values of the bf16 inputs).  Returns
    (a, u, h, o) in float64, o [n, d]."""
    a = mx_matmul_nt(xr, Wg)
    u = mx_matmul_nt(xr, Wu)
    h = silu(a) * u
    o = mx_matmul_nt(h, Wd)
    return a, u, h, o


def mxfp8_grouped_swiglu_fwd(x_perm: np.ndarray, offsets: np.ndarray, Wg: np.ndarray, Wu: np.ndarray,
                             Wd: np.ndarray) -> np.ndarray:
    """The routed experts over the permuted rows: rows [offsets[e],
    offsets[e+1]) of x_perm go through expert e.  Returns o_perm [R, d]."""
    R = int(offsets[-1])
    o = np.zeros((R, x_perm.shape[1]), dtype=np.float64)
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            o[r0:r1] = mxfp8_swiglu_fwd(x_perm[r0:r1], Wg[e], Wu[e], Wd[e])[3]
    return o
