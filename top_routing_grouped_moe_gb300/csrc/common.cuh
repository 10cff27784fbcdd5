// Shared definitions of the CUDA path (device side and host side).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
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

// v = hi + lo with hi = bf16(v), lo = bf16(v - hi): about 16 significant bits
// in two bf16 halves (8 values each, packed).
__device__ __forceinline__ void split8(const float (&v)[8], uint4& hi, uint4& lo) {
  float h[8], l[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    h[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
    l[e] = v[e] - h[e];
  }
  hi = pack8(h);
  lo = pack8(l);
}

}  // namespace moe
