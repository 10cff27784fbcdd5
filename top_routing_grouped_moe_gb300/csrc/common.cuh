// Shared definitions of the CUDA path (device side and host side).
#pragma once
#include <cstdint>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// Limits (the C ABI's documented shape limits).
constexpr int kMaxE = 256;
constexpr int kMaxK = 8;

// Tokens per routing tile (histogram / in-tile rank granularity).
constexpr int kRouteTile = 128;

// Bounded device waits: a wait that has not completed after this long gives up
// and records MOE_ERR_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Round two fp32 to bf16 (RNE) and pack (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 8 bf16 (one uint4) -> 8 fp32
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}

// fp16 storage of the terms of a per-token sum (expert outputs, the shared
// output, input-gradient terms): four values rounded to nearest even; one
// beyond the fp16 range becomes inf, which the kernel that sums the terms
// finds in its sum and reports.
__device__ __forceinline__ uint2 f16x4(const float4& v) {
  const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}
// 4 fp16 (one uint2) -> fp32
__device__ __forceinline__ float4 unpack_f16x4(const uint2& v) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
// 8 fp16 (one uint4) -> fp32
__device__ __forceinline__ void unpack_f16x8(const uint4& v, float (&f)[8]) {
  const float4 a = unpack_f16x4(make_uint2(v.x, v.y)), b = unpack_f16x4(make_uint2(v.z, v.w));
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// ------------------------------------------------------------ gradient-term scale
// The backward's fp16 sum terms (input-gradient rows) are stored divided by
// 2^e, e = floor(log2 max|dY|): the terms then sit where they sit for
// gradients of order one whatever the gradient's own scale, and the sum is
// multiplied by 2^e again (both exact).  The scale word holds the largest
// bf16 magnitude pattern of dY (an integer maximum, independent of order).

// e of a bf16 magnitude pattern: 0 for zero, inf or NaN (the finite checks
// report the latter two), clamped to [-126, 126].
__device__ __forceinline__ int grad_scale_exp(unsigned word) {
  const int f = (int)((word >> 7) & 0xFFu);
  if (word == 0u || f == 0xFF) return 0;
  return min(max(f - 127, -126), 126);
}
// 2^e as an fp32 normal, e in [-126, 127]
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// ------------------------------------------------------------ MXFP8
// (E4M3 elements, one E8M0 scale 2^(floor(log2 max|v|) - 8) per 32 values along
// K; scales of rows [128 t, 128 t + 128) x blocks [4 q, 4 q + 4) form one
// 512-byte "tile atom", row 128 t + 32 j + l, block 4 q + b at byte
// 16 l + 4 j + b)
// E8M0 exponent of the block scale for the block maximum |v| = amax (fp32):
// floor(log2 amax) - 8, clamped to [-127, 127]; -127 for amax == 0.
__device__ __forceinline__ int mx_scale_exp(float amax) {
  if (!(amax > 0.0f)) return -127;
  const uint32_t b = __float_as_uint(amax);
  const int ef = (int)((b >> 23) & 0xFF);
  int e;
  if (ef != 0) {
    e = ef - 127;
  } else {  // subnormal: amax = m 2^-149, floor(log2) = (31 - clz(m)) - 149
    e = (31 - __clz((int)(b & 0x7FFFFF))) - 149;
  }
  return min(max(e - 8, -127), 127);
}

// 2^-se as an fp32 normal (se in [-127, 126]; bf16 blocks give se <= 120)
__device__ __forceinline__ float mx_inv_scale(int se) { return __uint_as_float((uint32_t)(127 - se) << 23); }

// 4 values -> 4 E4M3 codes (byte i = code of v[i]), each v[i] scaled by
// inv = 2^-se (exact: a power-of-two scaling; a result below fp32's normal
// range is far below E4M3's smallest subnormal and rounds to 0 either way)
__device__ __forceinline__ uint32_t mx_codes4(float v0, float v1, float v2, float v3, float inv) {
  const float a0 = v0 * inv, a1 = v1 * inv, a2 = v2 * inv, a3 = v3 * inv;
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(a2, a3), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ long long mx_atom_offset(long long row, int block, int nq) {
  return ((row >> 7) * nq + (block >> 2)) * 512 + 16 * (row & 31) + 4 * ((row & 127) >> 5) + (block & 3);
}

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialization (launch_pdl below, and the GEMM
// launcher): its CTAs may be scheduled while the kernel before it on the
// stream is still retiring, run a prologue that touches only shared memory,
// tensor memory and kernel parameters, and then wait in dependency_wait()
// until the previous kernel has completed and its memory is visible.  Every
// thread waits before its first global access (read or write), and every CTA
// waits before it exits, so the chain stays ordered however far back a
// kernel's inputs were written.  No kernel signals its dependents early: a
// trigger at kernel entry (dependents resident for the whole kernel) measured
// slower than none.  Launched without the attribute, or after a non-kernel
// operation, the wait is a no-op.
__device__ __forceinline__ void dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kern` on `s` with programmatic stream serialization (see above).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace moe
