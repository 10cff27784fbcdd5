// Host helpers for the grouped GEMM: TMA tensor-map encoding (driver entry
// point fetched through the runtime, so the library needs no link-time
// libcuda) and the generic persistent launch.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "gemm.cuh"
#include "internal.h"

namespace moe {
namespace gemm {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 map over a row-major [outer, inner] tensor with row pitch
// `row_bytes`; box = box_inner x box_outer elements, 128-byte swizzle,
// out-of-bounds elements read as zero.
inline bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                      uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major [rows, cols] bf16 matrix (cols a multiple of 64) seen as 64-column
// blocks: dims (64, rows, cols / 64), the block index outermost although its
// stride (128 bytes) is the smallest.  One box of 64 x box_rows x box_blocks
// lands in shared memory as box_blocks consecutive 64 x box_rows blocks: the
// MN-major operand layout, in one TMA instruction instead of box_blocks.
inline bool encode_blocks(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows,
                          uint32_t box_blocks) {
  EncodeTiledFn f = encode_fn();
  if (!f || cols % 64 != 0) return false;
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_blocks};
  cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 map over a row-major [outer, inner] tensor, no swizzle (rows of a
// box land contiguously), out-of-bounds elements read as zero.
inline bool encode_2d_f32(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                          uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over [d2, d1, d0] (d0 contiguous); box = b0 x b1 x 1.
inline bool encode_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
                      uint32_t b1) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 (one byte per element) maps with 128-byte swizzle, boxes of 128 K
// bytes (one swizzle row) x 128 rows: 2-D over [rows, K], 3-D over [G][N][K].
inline bool encode_u8_2d(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  cuuint64_t dims[2] = {K, rows};
  cuuint64_t strides[1] = {K};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
inline bool encode_u8_3d(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t N, uint64_t G) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  cuuint64_t dims[3] = {K, N, G};
  cuuint64_t strides[2] = {K, K * N};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map for TMA stores of 32 x 32 boxes into [d2][d1][d0] (d0
// contiguous), 64-byte swizzle (the epilogue's staging layout).
inline bool encode_store_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Next free tensor-map slot of P, or -1 when all MAX_MAPS are taken (the
// caller then reports an invalid launch instead of writing past the array).
inline int new_map(Params& P) { return P.num_maps < MAX_MAPS ? P.num_maps++ : -1; }

inline int cdiv_h(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Row gather of problem `pr`'s operand `op` (0 = A, 1 = B) from the bf16
// source [src_rows, cols] by permuted row -> slot (slot / k = source row).
inline bool set_gather(Problem& pr, int op, const void* src, int cols, const int32_t* slot_of_row, int k,
                       int nslots) {
  if (!src || !slot_of_row || k < 1 || (reinterpret_cast<uintptr_t>(src) & 15) || (cols % 64)) return false;
  pr.gather_src = static_cast<const uint8_t*>(src);
  pr.gather_pitch = (long long)cols * 2;
  pr.gather_slot = slot_of_row;
  pr.gather_k = k;
  pr.gather_slots = nslots;
  pr.gather_op = op;
  return true;
}

inline Problem blank_problem() {
  Problem p;
  std::memset(&p, 0, sizeof(p));
  p.map_b2 = -1;
  p.map_a_lo = -1;
  p.map_b_lo = -1;
  p.map_out = -1;
  p.map_out2 = -1;
  p.nsplit = 1;
  return p;
}

// Launch a persistent grid for `tile_bound` tiles at most: one CTA per SM
// (PAIR = 1), or clusters of two CTAs sized by the number of clusters that can
// be resident at once (PAIR = 2), with programmatic stream serialization (the
// kernel waits for its predecessor after its on-chip prologue).  The dynamic
// schedule's tile counter is zeroed by a memset unless the kernel launched
// just before (`counter_ready`) has zeroed it.
template <int AMN, int BMN, int MODE, int EPI, int PAIR, int SPLIT = SPLIT_NONE, int MX = 0, int GATHER = 0>
cudaError_t launch(Params& P, long long tile_bound, cudaStream_t s, const char* name, bool counter_ready = false) {
  auto kern = grouped_gemm_kernel<AMN, BMN, MODE, EPI, PAIR, SPLIT, MX, GATHER>;
  constexpr size_t smem = smem_bytes<MODE, EPI, PAIR, SPLIT, MX>();
  static_assert(smem <= 227 * 1024, "dynamic shared memory above the per-CTA limit");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static unsigned long long configured = 0;  // bit per device
  static int max_clusters[64] = {0};
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!(configured & (1ull << dev))) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      if (PAIR == 2) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * (device_sm_count() / 2), 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        max_clusters[dev] = n > 0 ? n : 1;
      }
      configured |= 1ull << dev;
    }
  }
  if (tile_bound <= 0) return cudaSuccess;
  P.status = device_status_ptr();
  if (P.tile_counter && !counter_ready) {
    timing_mark(s, "memset_tile_counter");
    e = cudaMemsetAsync(P.tile_counter, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
  }
  timing_mark(s, name);
  int grid;
  if (PAIR == 1) {
    grid = device_sm_count();
    if (tile_bound < grid) grid = static_cast<int>(tile_bound);
  } else {
    int clusters = max_clusters[dev];
    if (tile_bound < clusters) clusters = static_cast<int>(tile_bound);
    grid = 2 * clusters;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR == 2 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace gemm
}  // namespace moe
