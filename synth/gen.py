"""Seeded synthetic inputs for the MoE layer (shared by the CUDA path's tests,
the bench and the oracle).

This module holds no arithmetic of the MoE method itself: it only draws the
numbers that the layer consumes (hidden states, weights, upstream gradients,
random routing choices and the fixed Zipf-like router bias of the learned
routing workload).

Generator (one definition, used everywhere):
  * SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014) read as a counter-based generator: the i-th
    64-bit word of a stream with seed s is mix(s + (i+1)*0x9E3779B97F4A7C15),
    where mix is SplitMix64's finaliser.  Any element can therefore be
    regenerated on its own (the oracle regenerates only the experts it checks).
  * uniform(i) = (word(i) >> 11) * 2**-53, in [0, 1).
  * normal: Box-Muller (1958) on the pair (2j, 2j+1):
    r = sqrt(-2 ln(1 - U_2j)), z_2j = r cos(2 pi U_2j+1), z_2j+1 = r sin(2 pi U_2j+1),
    in float64.
  * bf16 values: float64 -> float32 (round to nearest even) -> bfloat16 (round
    to nearest even on the float32 bits).  Stored as uint16 bit patterns.

Streams: seed(tensor) = BASE_SEED xor (0x9E3779B97F4A7C15 * tensor_id mod 2**64).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BASE_SEED = 20261202
GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids of the streams
TID = {
    "x": 1, "W_r": 2, "W_g": 3, "W_u": 4, "W_d": 5,
    "Ws_g": 6, "Ws_u": 7, "Ws_d": 8, "dY": 9,
    "route_pick": 10, "rank_perm": 11, "route_logit": 12,
    "logits_test": 13,
}

_CHUNK = 1 << 21  # elements per work item


def stream_seed(tensor: str | int, base: int = BASE_SEED) -> np.uint64:
    tid = TID[tensor] if isinstance(tensor, str) else int(tensor)
    return np.uint64((base ^ ((0x9E3779B97F4A7C15 * tid) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def words(seed: np.uint64, start: int, count: int) -> np.ndarray:
    """64-bit words start..start+count-1 of the SplitMix64 stream `seed`."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(seed + ctr * GAMMA)


def uniforms(seed: np.uint64, start: int, count: int) -> np.ndarray:
    w = words(seed, start, count)
    return (w >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normals_chunk(seed: np.uint64, start: int, count: int) -> np.ndarray:
    # pairs covering [start, start+count)
    p0 = start // 2
    p1 = (start + count + 1) // 2
    u = uniforms(seed, 2 * p0, 2 * (p1 - p0))
    u1 = u[0::2]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    th = (2.0 * math.pi) * u2
    z = np.empty(2 * (p1 - p0), dtype=np.float64)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    off = start - 2 * p0
    return z[off:off + count]


def normals(seed: np.uint64, start: int, count: int, threads: int | None = None) -> np.ndarray:
    """Standard normals start..start+count-1 of stream `seed` (float64)."""
    if count <= _CHUNK:
        return _normals_chunk(seed, start, count)
    out = np.empty(count, dtype=np.float64)
    pieces = [(s, min(_CHUNK, count - s)) for s in range(0, count, _CHUNK)]

    def work(p):
        s, n = p
        out[s:s + n] = _normals_chunk(seed, start + s, n)

    with ThreadPoolExecutor(max_workers=threads or min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(work, pieces))
    return out


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 (RNE); returns uint16 bit patterns."""
    f = np.ascontiguousarray(v, dtype=np.float32)
    b = f.view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def normal_bf16(tensor: str | int, shape, std: float = 1.0, start: int = 0,
                base: int = BASE_SEED, threads: int | None = None) -> np.ndarray:
    """bf16 bit patterns of std*N(0,1), elements start.. of the tensor's stream,
    reshaped to `shape`.  Generated in chunks on a thread pool."""
    n = int(np.prod(shape))
    seed = stream_seed(tensor, base)
    out = np.empty(n, dtype=np.uint16)
    pieces = [(s, min(_CHUNK, n - s)) for s in range(0, n, _CHUNK)]

    def work(p):
        s, m = p
        z = _normals_chunk(seed, start + s, m)
        if std != 1.0:
            z *= std
        out[s:s + m] = f64_to_bf16_bits(z)

    if len(pieces) <= 1:
        for p in pieces:
            work(p)
    else:
        with ThreadPoolExecutor(max_workers=threads or min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(work, pieces))
    return out.reshape(shape)


def random_routing_logits(T: int, E: int, k: int, base: int = BASE_SEED) -> np.ndarray:
    """Random-routing input: per token, k distinct experts drawn uniformly
    (partial Fisher-Yates over [0, E) with uniforms t*k+j of stream
    'route_pick'), with N(0,1) logits (normals t*k+j of stream 'route_logit')
    at those experts and -inf elsewhere.  float32 [T, E]."""
    u = uniforms(stream_seed("route_pick", base), 0, T * k).reshape(T, k)
    z = normals(stream_seed("route_logit", base), 0, T * k).reshape(T, k)
    perm = np.tile(np.arange(E, dtype=np.int64), (T, 1))
    rows = np.arange(T)
    for j in range(k):
        r = j + np.floor(u[:, j] * (E - j)).astype(np.int64)
        a = perm[rows, j].copy()
        perm[rows, j] = perm[rows, r]
        perm[rows, r] = a
    logits = np.full((T, E), -np.inf, dtype=np.float32)
    logits[rows[:, None], perm[:, :k]] = z.astype(np.float32)
    return logits


def zipf_bias(E: int, base: int = BASE_SEED) -> np.ndarray:
    """Fixed per-expert logit bias b_e = 0.5*ln(1/rank_e), rank a seeded random
    permutation of 1..E (Fisher-Yates, stream 'rank_perm'); float32 [E]."""
    u = uniforms(stream_seed("rank_perm", base), 0, E)
    rank = np.arange(1, E + 1, dtype=np.int64)
    for i in range(E - 1, 0, -1):
        j = int(math.floor(u[i] * (i + 1)))
        rank[i], rank[j] = rank[j], rank[i]
    return np.array([0.5 * math.log(1.0 / r) for r in rank], dtype=np.float64).astype(np.float32)


def random_logits(T: int, E: int, tensor: str | int = "logits_test", base: int = BASE_SEED) -> np.ndarray:
    """Plain N(0,1) float32 logits [T, E] for routing-only parity cases."""
    return normals(stream_seed(tensor, base), 0, T * E).astype(np.float32).reshape(T, E)
