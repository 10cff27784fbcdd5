// MXFP8 (OCP microscaling: FP8 E4M3 elements, one E8M0 power-of-two scale per
// 32 consecutive values along the contraction dimension) for the expert MLP:
// the row quantizer (weights, the shared expert's input), the packed gate/up
// weight layout, and the permutation that writes x_perm straight in MXFP8.
//
// Scale of a block: X = 2^(floor(log2 max|v|) - 8) (the block's largest value
// lands in [256, 512), the binade of E4M3's largest normal, 448), 2^-127 for
// an all-zero block; codes = E4M3(v / X), round to nearest even, saturating
// at +-448.  v / X is exact in fp32 (a power-of-two scaling of a bf16 value).
//
// Scale layout ("tile atoms"): the scales of rows [128 t, 128 t + 128) and
// blocks [4 q, 4 q + 4) form one 512-byte atom at byte ((t * nq + q) * 512),
// nq = cols / 128; inside it the scale of row 128 t + 32 j + l, block 4 q + b
// is byte 16 l + 4 j + b.  That is the layout the block-scaled tensor-core MMA
// reads from tensor memory after a 32x128b.warpx4 copy, so a GEMM stage of
// 128 rows x 128 K values takes one atom per operand.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarps = 8;

// One warp per destination row; lanes take consecutive 8-value chunks, so
// the 32 values of a block are held by 4 consecutive lanes.
// src_row(p): the bf16 source row of destination row p (packed gate/up:
// 64-row slices of W_g and W_u alternate).
template <bool GATE_UP>
__global__ void mx_quantize_rows_kernel(const uint4* __restrict__ src, const uint4* __restrict__ src2,
                                        long long rows, int cols, int H, uint32_t* __restrict__ codes,
                                        uint8_t* __restrict__ scales) {
  dependency_wait();
  const long long p = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (p >= rows) return;
  const uint4* srow;
  if (GATE_UP) {
    // packed row p of expert e: slice j = (p % 2H) / 128 of 64 h columns,
    // rows [0, 64) of the slice from W_g, [64, 128) from W_u
    const long long e = p / (2LL * H);
    const int q = (int)(p % (2LL * H));
    const int j = q >> 7, r = q & 127;
    const long long srow_idx = e * H + 64LL * j + (r & 63);
    srow = (r < 64 ? src : src2) + srow_idx * (cols / 8);
  } else {
    srow = src + p * (cols / 8);
  }
  const int nq = cols / 128;
  const int vpr = cols / 8;
  // every lane runs every sweep (the block maximum is a 4-lane shuffle);
  // vpr is a multiple of 16, so a block is valid for all of its 4 lanes or none
  for (int c0 = 0; c0 < vpr; c0 += 32) {
    const int c = c0 + lane;
    const bool ok = c < vpr;
    float f[8];
    if (ok) {
      unpack8(__ldg(srow + c), f);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int se = mx_scale_exp(amax);
    const float inv = mx_inv_scale(se);
    if (!ok) continue;
    uint2 w;
    w.x = mx_codes4(f[0], f[1], f[2], f[3], inv);
    w.y = mx_codes4(f[4], f[5], f[6], f[7], inv);
    *reinterpret_cast<uint2*>(codes + (p * cols + 8LL * c) / 4) = w;
    if ((c & 3) == 0) scales[mx_atom_offset(p, c >> 2, nq)] = (uint8_t)(se + 127);
  }
}

// MX permutation scatter: one warp per token; the token's row is quantized
// once (blocks of 32 along d) and its codes go to every kept row in the
// padded row space (expert e's rows start at mx_offsets[e], a multiple of
// 128), its scales to the matching tile atoms.
__global__ void perm_scatter_mx_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ idx,
                                       const int32_t* __restrict__ inrank, const int32_t* __restrict__ tile_base,
                                       const int32_t* __restrict__ mx_offsets, int T, int d, int E, int k,
                                       int capacity, long long max_rows, int32_t* __restrict__ row_of_slot,
                                       int32_t* __restrict__ slot_of_row, uint32_t* __restrict__ codes,
                                       uint8_t* __restrict__ scales, int* status) {
  dependency_wait();
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int row = -1;
  if (lane < k) {
    const long long slot = (long long)t * k + lane;
    const int e = idx[slot];
    const int r = inrank[slot];
    if (e >= 0 && e < E && r >= 0) {
      const int rank = tile_base[(long long)(t / kRouteTile) * E + e] + r;
      if (capacity <= 0 || rank < capacity) row = mx_offsets[e] + rank;
    }
    if (row >= max_rows) {
      record_status(status, MOE_ERR_DEVICE_BOUNDS);
      row = -1;
    }
    row_of_slot[slot] = row;
    if (row >= 0) slot_of_row[row] = (int32_t)slot;
  }
  int rows[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) rows[s] = __shfl_sync(0xffffffffu, row, s < k ? s : 0);
  const int nq = d / 128;
  const int vpr = d / 8;
  const uint4* src = x + (long long)t * vpr;
  for (int c0 = 0; c0 < vpr; c0 += 32) {
    const int c = c0 + lane;
    const bool ok = c < vpr;
    float f[8];
    if (ok) {
      unpack8(__ldg(src + c), f);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int se = mx_scale_exp(amax);
    const float inv = mx_inv_scale(se);
    if (!ok) continue;
    uint2 w;
    w.x = mx_codes4(f[0], f[1], f[2], f[3], inv);
    w.y = mx_codes4(f[4], f[5], f[6], f[7], inv);
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= k) break;
      if (rows[s] < 0) continue;
      *reinterpret_cast<uint2*>(codes + ((long long)rows[s] * d + 8LL * c) / 4) = w;
      if ((c & 3) == 0) scales[mx_atom_offset(rows[s], c >> 2, nq)] = (uint8_t)(se + 127);
    }
  }
}

inline unsigned warp_blocks(long long n) { return (unsigned)((n + kWarps - 1) / kWarps); }

}  // namespace

size_t mx_scales_bytes(long long rows, int cols) {
  return (size_t)((rows + 127) / 128) * (size_t)(cols / 128) * 512;
}

cudaError_t launch_mx_quantize(const void* src, long long rows, int cols, void* codes, void* scales,
                               cudaStream_t s) {
  timing_mark(s, "mx_quantize");
  return launch_pdl(mx_quantize_rows_kernel<false>, dim3(warp_blocks(rows)), dim3(32 * kWarps), 0, s,
      static_cast<const uint4*>(src), nullptr, rows, cols, 0, static_cast<uint32_t*>(codes),
      static_cast<uint8_t*>(scales));
}

cudaError_t launch_mx_quantize_gate_up(const void* W_g, const void* W_u, int E, int H, int d, void* codes,
                                       void* scales, cudaStream_t s) {
  const long long rows = 2LL * E * H;
  timing_mark(s, "mx_quantize_gate_up");
  return launch_pdl(mx_quantize_rows_kernel<true>, dim3(warp_blocks(rows)), dim3(32 * kWarps), 0, s,
      static_cast<const uint4*>(W_g), static_cast<const uint4*>(W_u), rows, d, H, static_cast<uint32_t*>(codes),
      static_cast<uint8_t*>(scales));
}

cudaError_t launch_permute_mx(const void* x, const int32_t* idx, int T, int d, int E, int k, int capacity,
                              int32_t* counts_raw, int32_t* counts, int32_t* offsets, int32_t* mx_offsets,
                              int32_t* row_of_slot, int32_t* slot_of_row, void* codes, void* scales, void* ws,
                              int* status, cudaStream_t s) {
  int32_t* tile_base = nullptr;
  int32_t* inrank = nullptr;
  cudaError_t e = launch_permute_counts(idx, T, E, k, capacity, counts_raw, counts, offsets, mx_offsets, ws,
                                        &tile_base, &inrank, status, s);
  if (e != cudaSuccess) return e;
  timing_mark(s, "perm_scatter_mx");
  return launch_pdl(perm_scatter_mx_kernel, dim3(warp_blocks(T)), dim3(32 * kWarps), 0, s,
      static_cast<const uint4*>(x), idx, inrank, tile_base, mx_offsets, T, d, E, k, capacity,
      mx_rows_max(T, E, k), row_of_slot, slot_of_row, static_cast<uint32_t*>(codes), static_cast<uint8_t*>(scales),
      status);
}

}  // namespace moe
