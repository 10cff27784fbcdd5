// SIMT kernels of the MoE layer: top-k gating, the deterministic permutation
// (tile histogram + in-tile ranks, column scan, stable scatter), the
// gate-weighted combine and the backward passes of those steps.  All of them
// are bandwidth or latency bound: rows move as 16-byte vectors, one warp per
// token, fp32 accumulation, and nothing depends on the order of atomics.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
  // total order: value descending, then expert index ascending (-0.0 == +0.0)
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

// ------------------------------------------------------------------ top-k
// One warp per token.  Lane l holds logits e = l + 32 j.  k rounds of a
// warp arg-max (butterfly shuffles), ties to the lower expert index.
template <int NJ>
__global__ void topk_gating_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ idx,
                                   float* __restrict__ gates) {
  dependency_wait();
  const int warp = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* row = logits + (long long)warp * E;
  float v[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    int e = lane + 32 * j;
    v[j] = e < E ? __ldg(row + e) : 0.0f;
  }
  uint32_t taken = 0;
  float sel_v[kMaxK];
  int sel_i[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    if (s >= k) break;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      int e = lane + 32 * j;
      if (e < E && !(taken & (1u << j)) && better(v[j], e, bv, bi)) {
        bv = v[j];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    sel_v[s] = bv;
    sel_i[s] = bi;
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
  }
  // gates: softmax over the selected logits (max = the first one)
  const float m = sel_v[0];
  float den = 0.0f;
  float ex[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    if (s >= k) break;
    ex[s] = (sel_v[s] == -INFINITY) ? 0.0f : expf(sel_v[s] - m);
    den += ex[s];
  }
  if (lane < k) {
    float g = 0.0f;
    int id = 0;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s)
      if (s == lane) {
        g = ex[s] / den;
        id = sel_i[s];
      }
    idx[(long long)warp * k + lane] = id;
    gates[(long long)warp * k + lane] = g;
  }
}

// ------------------------------------------------------------------ permutation
// (1) per tile of kRouteTile tokens: a bitmask of the tile's tokens per expert
// in shared memory gives the tile's per-expert counts and each (token, slot)'s
// rank among the tile's tokens that picked the same expert.
__global__ void perm_tile_hist_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                      int32_t* __restrict__ tile_counts, int32_t* __restrict__ inrank,
                                      int* status) {
  dependency_wait();
  __shared__ uint32_t bits[kMaxE][kRouteTile / 32];
  const int tile = blockIdx.x;
  const int t_local = threadIdx.x;  // blockDim.x == kRouteTile
  const int t = tile * kRouteTile + t_local;
  for (int i = threadIdx.x; i < E * (kRouteTile / 32); i += blockDim.x) (&bits[0][0])[i] = 0u;
  __syncthreads();
  int ex[kMaxK];
  if (t < T) {
    for (int s = 0; s < k; ++s) {
      int e = idx[(long long)t * k + s];
      bool bad = e < 0 || e >= E;
      for (int s2 = 0; s2 < s; ++s2) bad |= (ex[s2] == e);
      if (bad) {
        record_status(status, MOE_ERR_DEVICE_BOUNDS);
        e = -1;
      }
      ex[s] = e;
      if (e >= 0) atomicOr(&bits[e][t_local >> 5], 1u << (t_local & 31));
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kRouteTile / 32; ++w) c += __popc(bits[e][w]);
    tile_counts[(long long)tile * E + e] = c;
  }
  if (t < T) {
    const int w0 = t_local >> 5;
    const uint32_t lt = (1u << (t_local & 31)) - 1u;
    for (int s = 0; s < k; ++s) {
      int e = ex[s];
      int r = -1;
      if (e >= 0) {
        r = __popc(bits[e][w0] & lt);
        for (int w = 0; w < w0; ++w) r += __popc(bits[e][w]);
      }
      inrank[(long long)t * k + s] = r;
    }
  }
}

// (2) one block: per expert, exclusive scan of the tile counts over tiles
// (tile_base), totals (counts_raw), capacity clamp (counts) and offsets; with
// mx_offsets, also the offsets of the padded row space in which every
// expert's rows start at a multiple of 128.
__global__ void perm_scan_kernel(const int32_t* __restrict__ tile_counts, int ntile, int E, int capacity,
                                 int32_t* __restrict__ tile_base, int32_t* __restrict__ counts_raw,
                                 int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                 int32_t* __restrict__ mx_offsets) {
  dependency_wait();
  __shared__ int seg[1024];
  __shared__ int cnt[kMaxE];
  const int P = blockDim.x / E;  // segments of tiles per expert
  const int tid = threadIdx.x;
  const int e = tid % E;
  const int p = tid / E;
  const int chunk = (ntile + P - 1) / P;
  int sum = 0;
  if (p < P) {
    const int i0 = p * chunk, i1 = min(ntile, i0 + chunk);
    for (int i = i0; i < i1; ++i) sum += tile_counts[(long long)i * E + e];
  }
  seg[tid] = sum;
  __syncthreads();
  if (p < P) {
    int base = 0;
    for (int q = 0; q < p; ++q) base += seg[q * E + e];
    const int i0 = p * chunk, i1 = min(ntile, i0 + chunk);
    for (int i = i0; i < i1; ++i) {
      tile_base[(long long)i * E + e] = base;
      base += tile_counts[(long long)i * E + e];
    }
    if (p == P - 1) {
      counts_raw[e] = base;
      int c = capacity > 0 ? min(base, capacity) : base;
      counts[e] = c;
      cnt[e] = c;
    }
  }
  __syncthreads();
  // exclusive scan of cnt[0..E) (warp 0) and, with mx_offsets, of the counts
  // rounded up to 128 (warp 1)
  const int w = tid >> 5, lane = tid & 31;
  if (w == 0 || (w == 1 && mx_offsets)) {
    int32_t* out = w == 0 ? offsets : mx_offsets;
    const int round = w == 0 ? 1 : 128;
    int per = (E + 31) / 32;
    int loc = 0;
    for (int j = 0; j < per; ++j) {
      int i = lane * per + j;
      if (i < E) loc += (cnt[i] + round - 1) / round * round;
    }
    int incl = loc;
    for (int s = 1; s < 32; s <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, s);
      if (lane >= s) incl += v;
    }
    int run = incl - loc;
    for (int j = 0; j < per; ++j) {
      int i = lane * per + j;
      if (i < E) {
        out[i] = run;
        run += (cnt[i] + round - 1) / round * round;
      }
    }
    if (lane == 31) out[E] = incl;
  }
}

// (3) one warp per token: rows of its kept slots, row maps, and the copy of
// x[t] into every destination row (the row is read once).
__global__ void perm_scatter_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ idx,
                                    const int32_t* __restrict__ inrank, const int32_t* __restrict__ tile_base,
                                    const int32_t* __restrict__ offsets, int T, int d, int E, int k, int capacity,
                                    int32_t* __restrict__ row_of_slot, int32_t* __restrict__ slot_of_row,
                                    uint4* __restrict__ x_perm) {
  dependency_wait();
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int row = -1;
  if (lane < k) {
    const long long slot = (long long)t * k + lane;
    int e = idx[slot];
    int r = inrank[slot];
    if (e >= 0 && e < E && r >= 0) {
      int rank = tile_base[(long long)(t / kRouteTile) * E + e] + r;
      if (capacity <= 0 || rank < capacity) row = offsets[e] + rank;
    }
    row_of_slot[slot] = row;
    if (row >= 0) slot_of_row[row] = static_cast<int32_t>(slot);
  }
  // maps only (x_perm == NULL: the GEMMs gather the rows themselves)
  if (x_perm == nullptr) return;
  int rows[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) rows[s] = __shfl_sync(0xffffffffu, row, s < k ? s : 0);
  const int vec_per_row = d / 8;  // uint4 = 8 bf16
  const uint4* src = x + (long long)t * vec_per_row;
  for (int c = lane; c < vec_per_row; c += 32 * 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c + 32 * u < vec_per_row) v[u] = __ldg(src + c + 32 * u);
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= k) break;
      if (rows[s] < 0) continue;
      uint4* dst = x_perm + (long long)rows[s] * vec_per_row;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < vec_per_row) dst[c + 32 * u] = v[u];
    }
  }
}

// ------------------------------------------------------------------ combine
// Eight consecutive fp16 terms of a row, as fp32.
__device__ __forceinline__ void load8(const __half* p, float (&f)[8]) {
  unpack_f16x8(__ldg(reinterpret_cast<const uint4*>(p)), f);
}

// Expert / shared outputs (fp16 terms), fp32 accumulation, one bf16 rounding
// of y.  slot_order: the expert outputs are stored by slot (o[t*k+s]) instead
// of by permuted row.
__global__ void combine_kernel(const __half* __restrict__ o_perm, const __half* __restrict__ s_out,
                               const float* __restrict__ gates, const int32_t* __restrict__ row_of_slot, int T, int d,
                               int k, long long max_rows, int slot_order, uint4* __restrict__ y, int* status) {
  dependency_wait();
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int row = -1;
  float g = 0.0f;
  if (lane < k) {
    row = row_of_slot[(long long)t * k + lane];
    g = gates[(long long)t * k + lane];
    if (slot_order && row >= 0) row = t * k + lane;
    if (row >= max_rows) {
      record_status(status, MOE_ERR_DEVICE_BOUNDS);
      row = -1;
    }
  }
  int rows[kMaxK];
  float gs[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    rows[s] = __shfl_sync(0xffffffffu, row, s < k ? s : 0);
    gs[s] = __shfl_sync(0xffffffffu, g, s < k ? s : 0);
  }
  const int vpr = d / 8;  // 8 elements per step, one uint4 out
  for (int c = lane; c < vpr; c += 32) {
    float acc[8];
    if (s_out) {
      load8(s_out + (long long)t * d + 8 * c, acc);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    }
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= k) break;
      if (rows[s] < 0) continue;
      float v[8];
      load8(o_perm + (long long)rows[s] * d + 8 * c, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(gs[s], v[e], acc[e]);
    }
    // an infinite term (an fp16 term beyond its range) or NaN makes the sum
    // non-finite
    bool fin = true;
#pragma unroll
    for (int e = 0; e < 8; ++e) fin &= isfinite(acc[e]);
    if (!fin) record_status(status, MOE_ERR_RANGE);
    y[(long long)t * vpr + c] = pack8(acc);
  }
}

// Backward of the unpermute: the upstream gradient of each token is gathered
// into its kept rows (the gate factor and the gate gradient are applied in the
// expert backward, where they can be formed from fp32 values).
__global__ void gather_rows_kernel(const uint4* __restrict__ dY, const int32_t* __restrict__ row_of_slot, int T,
                                   int d, int k, long long max_rows, uint4* __restrict__ dY_perm, int* status) {
  dependency_wait();
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int row = -1;
  if (lane < k) {
    row = row_of_slot[(long long)t * k + lane];
    if (row >= max_rows) {
      record_status(status, MOE_ERR_DEVICE_BOUNDS);
      row = -1;
    }
  }
  int rows[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) rows[s] = __shfl_sync(0xffffffffu, row, s < k ? s : 0);
  const int vpr = d / 8;
  const uint4* src = dY + (long long)t * vpr;
  for (int c = lane; c < vpr; c += 32 * 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c + 32 * u < vpr) v[u] = __ldg(src + c + 32 * u);
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= k) break;
      if (rows[s] < 0) continue;
      uint4* dst = dY_perm + (long long)rows[s] * vpr;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < vpr) dst[c + 32 * u] = v[u];
    }
  }
}

// dgates[slot] = sum of the per-N-tile partials of its row (0 if dropped)
__global__ void dgates_reduce_kernel(const float* __restrict__ dgp, int P, const int32_t* __restrict__ row_of_slot,
                                     long long n_slots, float* __restrict__ dgates) {
  dependency_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_slots;
       i += (long long)gridDim.x * blockDim.x) {
    const int row = row_of_slot[i];
    float v = 0.0f;
    if (row >= 0)
      for (int p = 0; p < P; ++p) v += dgp[(long long)row * P + p];
    dgates[i] = v;
  }
}

// fp16 terms, fp32 accumulation, one bf16 rounding of dx
// The scale word of the backward's fp16 terms: the largest bf16 magnitude
// pattern of the upstream gradient (grid-stride over 16-byte chunks, four
// independent loads in flight per thread, a warp maximum, one atomicMax per
// warp into the zeroed word).
__device__ __forceinline__ unsigned bf16x8_mag_max(const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  unsigned m = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  return m;
}

__global__ void grad_amax_kernel(const uint4* __restrict__ src, long long n16, unsigned* __restrict__ word) {
  dependency_wait();
  unsigned m = 0u;
  const long long step = (long long)gridDim.x * blockDim.x;
  long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  for (; i + 3 * step < n16; i += 4 * step) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(src + i + u * step);
#pragma unroll
    for (int u = 0; u < 4; ++u) m = max(m, bf16x8_mag_max(v[u]));
  }
  for (; i < n16; i += step) m = max(m, bf16x8_mag_max(__ldg(src + i)));
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m) atomicMax(word, m);
}

__global__ void unpermute_reduce_kernel(const __half* __restrict__ dx_perm, const __half* __restrict__ dx_s,
                                        const __half* __restrict__ dx_r, const int32_t* __restrict__ row_of_slot,
                                        int T, int d, int k, long long max_rows, const unsigned* __restrict__ scale,
                                        uint4* __restrict__ dx, int* status) {
  dependency_wait();
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int row = -1;
  if (lane < k) {
    row = row_of_slot[(long long)t * k + lane];
    if (row >= max_rows) {
      record_status(status, MOE_ERR_DEVICE_BOUNDS);
      row = -1;
    }
  }
  int rows[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) rows[s] = __shfl_sync(0xffffffffu, row, s < k ? s : 0);
  // the terms hold v / 2^e (scale word; none: e = 0)
  const float up = scale ? pow2f(grad_scale_exp(__ldg(scale))) : 1.0f;
  const int vpr = d / 8;
  for (int c = lane; c < vpr; c += 32) {
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    // the per-token terms (shared expert, router), then the kept rows
    const __half* tok_terms[2] = {dx_s, dx_r};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (!tok_terms[i]) continue;
      float v[8];
      load8(tok_terms[i] + (long long)t * d + 8 * c, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += v[e];
    }
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= k) break;
      if (rows[s] < 0) continue;
      float v[8];
      load8(dx_perm + (long long)rows[s] * d + 8 * c, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += v[e];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= up;
    bool fin = true;
#pragma unroll
    for (int e = 0; e < 8; ++e) fin &= isfinite(acc[e]);
    if (!fin) record_status(status, MOE_ERR_RANGE);
    dx[(long long)t * vpr + c] = pack8(acc);
  }
}

// ------------------------------------------------------------------ router backward
// One warp per token: dl_s = g_s (dg_s - sum_j g_j dg_j) scattered into a dense
// [T,E] row (zeros elsewhere), plus optional bf16 hi + lo halves for the GEMMs.
__global__ void router_bwd_dl_kernel(const float* __restrict__ dgates, const float* __restrict__ gates,
                                     const int32_t* __restrict__ idx, int T, int E, int k,
                                     const float* __restrict__ add, float* __restrict__ dl,
                                     uint16_t* __restrict__ dl_hi, uint16_t* __restrict__ dl_lo) {
  dependency_wait();
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float g = 0.0f, dg = 0.0f;
  int e = -1;
  if (lane < k) {
    g = gates[(long long)t * k + lane];
    dg = dgates[(long long)t * k + lane];
    e = idx[(long long)t * k + lane];
  }
  float sgd = g * dg;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sgd += __shfl_xor_sync(0xffffffffu, sgd, off);
  const float mine = g * (dg - sgd);
  int es[kMaxK];
  float vs[kMaxK];
#pragma unroll
  for (int s = 0; s < kMaxK; ++s) {
    es[s] = __shfl_sync(0xffffffffu, e, s < k ? s : 0);
    vs[s] = __shfl_sync(0xffffffffu, mine, s < k ? s : 0);
  }
  for (int c = lane; c < E; c += 32) {
    float v = 0.0f;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s)
      if (s < k && es[s] == c) v = vs[s];
    if (add) v += add[(long long)t * E + c];  // e.g. the balance-loss gradient
    dl[(long long)t * E + c] = v;
    if (dl_hi) {
      __nv_bfloat16 hi = __float2bfloat16_rn(v);
      __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      dl_hi[(long long)t * E + c] = *reinterpret_cast<uint16_t*>(&hi);
      dl_lo[(long long)t * E + c] = *reinterpret_cast<uint16_t*>(&lo);
    }
  }
}

// v -> hi = bf16(v), lo = bf16(v - hi)
__global__ void f32_to_bf16_split_kernel(const float* __restrict__ src, uint16_t* __restrict__ hi,
                                         uint16_t* __restrict__ lo, long long n) {
  dependency_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float v = src[i];
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
    hi[i] = *reinterpret_cast<uint16_t*>(&h);
    lo[i] = *reinterpret_cast<uint16_t*>(&l);
  }
}

__global__ void splitk_reduce_kernel(const float4* __restrict__ part, int S, long long n4, float4* __restrict__ out) {
  dependency_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < S; ++s) {
      float4 b = part[(long long)s * n4 + i];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    out[i] = a;
  }
}

// ------------------------------------------------------------ router balance loss
// Full softmax of one token's logits held by the warp as NJ values per lane
// (expert c = lane + 32 j; -inf where c >= E); a row of -inf gives all zeros.
template <int NJ>
__device__ __forceinline__ void token_softmax(float (&p)[NJ]) {
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < NJ; ++j) m = fmaxf(m, p[j]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    p[j] = (m == -INFINITY || p[j] == -INFINITY) ? 0.0f : expf(p[j] - m);
    sum += p[j];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float inv = sum > 0.0f ? 1.0f / sum : 0.0f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) p[j] *= inv;
}

constexpr int kLblTokensPerWarp = 4;
constexpr int kLblTokensPerBlock = kWarpsPerBlock * kLblTokensPerWarp;

// One pass over the logits.  With f_c = counts_raw[c] / (T k) known up
// front, every warp writes the gradient of its tokens,
//   dl[t,c] = alpha E / T p[t,c] (f_c - sum_e f_e p[t,e]),
// and each block writes the sum of its tokens' probabilities (warps in
// order).  The last block to finish (a ticket counter, zeroed by the host
// before the launch) adds the block partials in block order, so P_mean and
//   loss = alpha E sum_c f_c P_c
// do not depend on which block finishes last.
template <int NJ>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
lbl_kernel(const float* __restrict__ logits, const int32_t* __restrict__ counts_raw, int T, int E, int k, float alpha,
           float* __restrict__ loss, float* __restrict__ P_mean, float* __restrict__ dl, float* __restrict__ partial,
           unsigned* __restrict__ ticket) {
  dependency_wait();
  __shared__ float acc_s[kWarpsPerBlock][32 * NJ];
  __shared__ float red[32 * kWarpsPerBlock];
  __shared__ bool last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float inv_tk = 1.0f / ((float)T * (float)k);
  float fj[NJ], acc[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = lane + 32 * j;
    fj[j] = c < E ? (float)counts_raw[c] * inv_tk : 0.0f;
    acc[j] = 0.0f;
  }
  const int t0 = blockIdx.x * kLblTokensPerBlock + warp * kLblTokensPerWarp;
  float v[kLblTokensPerWarp][NJ];  // all of the warp's rows in flight at once
#pragma unroll
  for (int i = 0; i < kLblTokensPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int c = lane + 32 * j;
      v[i][j] = (t0 + i < T && c < E) ? __ldg(logits + (long long)(t0 + i) * E + c) : -INFINITY;
    }
  const float scale = alpha * (float)E / (float)T;
#pragma unroll
  for (int i = 0; i < kLblTokensPerWarp; ++i) {
    const int t = t0 + i;
    if (t >= T) break;
    token_softmax<NJ>(v[i]);
    float sfp = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      acc[j] += v[i][j];
      sfp += fj[j] * v[i][j];
    }
    if (dl) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sfp += __shfl_xor_sync(0xffffffffu, sfp, off);
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int c = lane + 32 * j;
        if (c < E) dl[(long long)t * E + c] = scale * v[i][j] * (fj[j] - sfp);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NJ; ++j) acc_s[warp][lane + 32 * j] = acc[j];
  __syncthreads();
  for (int c = threadIdx.x; c < E; c += blockDim.x) {
    float s = 0.0f;
    for (int w = 0; w < kWarpsPerBlock; ++w) s += acc_s[w][c];
    partial[(long long)blockIdx.x * E + c] = s;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // E <= blockDim.x (checked on the host)
  const int c = threadIdx.x;
  float term = 0.0f;
  if (c < E) {
    float P = 0.0f;
    for (unsigned b = 0; b < gridDim.x; ++b) P += __ldcg(partial + (long long)b * E + c);
    P /= (float)T;
    if (P_mean) P_mean[c] = P;
    term = (float)counts_raw[c] * inv_tk * P;
  }
  red[c] = term;
  __syncthreads();
  for (int w = blockDim.x >> 1; w > 0; w >>= 1) {
    if (c < w) red[c] += red[c + w];
    __syncthreads();
  }
  if (c == 0) *loss = alpha * (float)E * red[0];
}

inline unsigned warp_blocks(long long n) { return static_cast<unsigned>((n + kWarpsPerBlock - 1) / kWarpsPerBlock); }
inline unsigned flat_blocks(long long n, int per) {
  long long b = (n + per - 1) / per;
  long long cap = 8LL * device_sm_count();
  return static_cast<unsigned>(b < cap ? (b > 0 ? b : 1) : cap);
}

}  // namespace

cudaError_t launch_topk_gating(const float* logits, int T, int E, int k, int32_t* idx, float* gates, int* status,
                               cudaStream_t s) {
  (void)status;
  const unsigned grid = warp_blocks(T);
  const int nj = (E + 31) / 32;
  timing_mark(s, "topk_gating");
  auto kern = nj == 1   ? topk_gating_kernel<1>
              : nj == 2 ? topk_gating_kernel<2>
              : nj <= 4 ? topk_gating_kernel<4>
                        : topk_gating_kernel<8>;
  return launch_pdl(kern, dim3(grid), dim3(32 * kWarpsPerBlock), 0, s, logits, T, E, k, idx, gates);
}

static inline size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

size_t permute_ws_bytes(int T, int E, int k) {
  const size_t ntile = (T + kRouteTile - 1) / kRouteTile;
  return 2 * align256(ntile * E * sizeof(int32_t)) + align256((size_t)T * k * sizeof(int32_t));
}

cudaError_t launch_permute_counts(const int32_t* idx, int T, int E, int k, int capacity, int32_t* counts_raw,
                                  int32_t* counts, int32_t* offsets, int32_t* mx_offsets, void* ws,
                                  int32_t** tile_base_out, int32_t** inrank_out, int* status, cudaStream_t s) {
  const int ntile = (T + kRouteTile - 1) / kRouteTile;
  char* w = static_cast<char*>(ws);
  int32_t* tile_counts = reinterpret_cast<int32_t*>(w);
  int32_t* tile_base = reinterpret_cast<int32_t*>(w + align256((size_t)ntile * E * 4));
  int32_t* inrank = reinterpret_cast<int32_t*>(w + 2 * align256((size_t)ntile * E * 4));
  timing_mark(s, "perm_tile_hist");
  cudaError_t e =
      launch_pdl(perm_tile_hist_kernel, dim3(ntile), dim3(kRouteTile), 0, s, idx, T, E, k, tile_counts, inrank, status);
  if (e != cudaSuccess) return e;
  timing_mark(s, "perm_scan");
  *tile_base_out = tile_base;
  *inrank_out = inrank;
  return launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, s, tile_counts, ntile, E, capacity, tile_base,
                    counts_raw, counts, offsets, mx_offsets);
}

cudaError_t launch_permute(const void* x, const int32_t* idx, int T, int d, int E, int k, int capacity,
                           int32_t* counts_raw, int32_t* counts, int32_t* offsets, int32_t* row_of_slot,
                           int32_t* slot_of_row, void* x_perm, void* ws, int* status, cudaStream_t s) {
  int32_t* tile_base = nullptr;
  int32_t* inrank = nullptr;
  cudaError_t e = launch_permute_counts(idx, T, E, k, capacity, counts_raw, counts, offsets, nullptr, ws,
                                        &tile_base, &inrank, status, s);
  if (e != cudaSuccess) return e;
  timing_mark(s, x_perm ? "perm_scatter" : "perm_maps");
  return launch_pdl(perm_scatter_kernel, dim3(warp_blocks(T)), dim3(32 * kWarpsPerBlock), 0, s,
                    static_cast<const uint4*>(x), idx, inrank, tile_base, offsets, T, d, E, k, capacity, row_of_slot,
                    slot_of_row, static_cast<uint4*>(x_perm));
}

cudaError_t launch_combine_rows(const void* o_perm, const void* s_out, const float* gates,
                                const int32_t* row_of_slot, int T, int d, int k, long long o_rows, void* y,
                                int* status, cudaStream_t s) {
  timing_mark(s, "combine");
  return launch_pdl(combine_kernel, dim3(warp_blocks(T)), dim3(32 * kWarpsPerBlock), 0, s,
      static_cast<const __half*>(o_perm), static_cast<const __half*>(s_out), gates, row_of_slot, T, d, k, o_rows, 0,
      static_cast<uint4*>(y), status);
}

cudaError_t launch_combine_slots(const void* o_slot, const void* s_out, const float* gates,
                                 const int32_t* row_of_slot, int T, int d, int k, void* y, int* status,
                                 cudaStream_t s) {
  timing_mark(s, "combine_slots");
  return launch_pdl(combine_kernel, dim3(warp_blocks(T)), dim3(32 * kWarpsPerBlock), 0, s,
      static_cast<const __half*>(o_slot), static_cast<const __half*>(s_out), gates, row_of_slot, T, d, k,
      (long long)T * k, 1, static_cast<uint4*>(y), status);
}

cudaError_t launch_combine(const void* o_perm, const void* s_out, const float* gates, const int32_t* row_of_slot,
                           int T, int d, int k, void* y, int* status, cudaStream_t s) {
  return launch_combine_rows(o_perm, s_out, gates, row_of_slot, T, d, k, (long long)T * k, y, status, s);
}

cudaError_t launch_gather_rows(const void* dY, const int32_t* row_of_slot, int T, int d, int k, void* dY_perm,
                               int* status, cudaStream_t s) {
  timing_mark(s, "gather_rows");
  return launch_pdl(gather_rows_kernel, dim3(warp_blocks(T)), dim3(32 * kWarpsPerBlock), 0, s,
      static_cast<const uint4*>(dY), row_of_slot, T, d, k, (long long)T * k, static_cast<uint4*>(dY_perm), status);
}

cudaError_t launch_dgates_reduce(const float* dgp, int P, const int32_t* row_of_slot, int T, int k, float* dgates,
                                 cudaStream_t s) {
  const long long n = (long long)T * k;
  timing_mark(s, "dgates_reduce");
  return launch_pdl(dgates_reduce_kernel, dim3(flat_blocks(n, 256)), dim3(256), 0, s, dgp, P, row_of_slot, n, dgates);
}

cudaError_t launch_unpermute_reduce(const void* dx_perm, const void* dx_s, const void* dx_r,
                                    const int32_t* row_of_slot, int T, int d, int k, const uint32_t* scale, void* dx,
                                    int* status, cudaStream_t s) {
  timing_mark(s, "unpermute_reduce");
  return launch_pdl(unpermute_reduce_kernel, dim3(warp_blocks(T)), dim3(32 * kWarpsPerBlock), 0, s,
      static_cast<const __half*>(dx_perm), static_cast<const __half*>(dx_s), static_cast<const __half*>(dx_r),
      row_of_slot, T, d, k, (long long)T * k, scale, static_cast<uint4*>(dx), status);
}

cudaError_t launch_grad_scale(const void* dY, long long n, uint32_t* word, cudaStream_t s) {
  timing_mark(s, "memset_grad_scale");
  cudaError_t e = cudaMemsetAsync(word, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  const long long n16 = n / 8;  // 8 bf16 per 16 bytes (rows are multiples of 64 values)
  timing_mark(s, "grad_amax");
  return launch_pdl(grad_amax_kernel, dim3(flat_blocks(n16, 256)), dim3(256), 0, s, static_cast<const uint4*>(dY),
                    n16, word);
}

cudaError_t launch_router_bwd_dl(const float* dgates, const float* gates, const int32_t* idx, int T, int E, int k,
                                 const float* add, float* dlogits, uint16_t* dl_hi, uint16_t* dl_lo, cudaStream_t s) {
  timing_mark(s, "router_bwd_dl");
  return launch_pdl(router_bwd_dl_kernel, dim3(warp_blocks(T)), dim3(32 * kWarpsPerBlock), 0, s, dgates, gates, idx,
                    T, E, k, add, dlogits, dl_hi, dl_lo);
}

cudaError_t launch_f32_to_bf16_split(const float* src, uint16_t* hi, uint16_t* lo, long long n, cudaStream_t s) {
  timing_mark(s, "f32_to_bf16_split");
  return launch_pdl(f32_to_bf16_split_kernel, dim3(flat_blocks(n, 256)), dim3(256), 0, s, src, hi, lo, n);
}

cudaError_t launch_splitk_reduce(const float* partial, int S, long long n, float* out, cudaStream_t s) {
  const long long n4 = n / 4;
  timing_mark(s, "splitk_reduce");
  return launch_pdl(splitk_reduce_kernel, dim3(flat_blocks(n4, 256)), dim3(256), 0, s,
                    reinterpret_cast<const float4*>(partial), S, n4, reinterpret_cast<float4*>(out));
}

size_t balance_loss_ws_bytes(int T, int E) {
  const size_t nblk = (T + kLblTokensPerBlock - 1) / kLblTokensPerBlock;
  return align256(nblk * E * sizeof(float)) + 256;
}

cudaError_t launch_balance_loss(const float* logits, const int32_t* counts_raw, int T, int E, int k, float alpha,
                                float* loss, float* P_mean, float* dl, void* ws, cudaStream_t s) {
  if (E > 32 * kWarpsPerBlock) return cudaErrorInvalidValue;
  const int nblk = (T + kLblTokensPerBlock - 1) / kLblTokensPerBlock;
  float* partial = static_cast<float*>(ws);
  unsigned* ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + align256((size_t)nblk * E * sizeof(float)));
  timing_mark(s, "memset_ticket");
  cudaError_t e = cudaMemsetAsync(ticket, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const unsigned threads = 32 * kWarpsPerBlock;
  timing_mark(s, "balance_loss");
  const int nj = (E + 31) / 32;
  auto kern = nj == 1 ? lbl_kernel<1> : nj == 2 ? lbl_kernel<2> : nj <= 4 ? lbl_kernel<4> : lbl_kernel<8>;
  return launch_pdl(kern, dim3(nblk), dim3(threads), 0, s, logits, counts_raw, T, E, k, alpha, loss, P_mean, dl,
                    partial, ticket);
}

}  // namespace moe
