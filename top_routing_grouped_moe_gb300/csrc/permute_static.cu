// moe_permute_static: the token permutation with its scratch in a fixed,
// library-owned device array instead of a caller workspace.
//
// Some callers cannot allocate device memory for scratch: plug-in hosts that
// hand a library only their own tensors and a stream (no allocator handle),
// and processes whose device memory is entirely owned by a framework pool,
// where an extra cudaMalloc would fail or fragment the pool.  This entry point
// lets them run the permutation with nothing but their inputs and outputs.
//
// The array below lives in every GPU that loads this library, until the
// process exits.  Every call on a device uses the same array, so two calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on it.  The array keeps what the previous call wrote; nothing in
// it needs to start at zero, because each call writes every scratch word it
// reads before reading it (per-tile counts, their scan, in-tile ranks).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// Maximum scratch of one call: permute_ws_bytes(T, E, k) <= 4 MiB, i.e. the
// per-tile counts and bases of ceil(T/128) x E and the T*k in-tile ranks
// (for example T*k up to 512K slots with E = 64 experts).
constexpr size_t kStaticScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of g_permute_scratch on the current device.  The name of the
// array in host code is only a host-side stand-in; the address a kernel can use
// comes from cudaGetSymbolAddress, taken once per device with that device
// current.
cudaError_t scratch_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_permute_static(const void* x, const int32_t* topk_idx, int T, int d, int E, int k, int capacity,
                                  int32_t* counts_raw, int32_t* counts, int32_t* offsets, int32_t* row_of_slot,
                                  int32_t* slot_of_row, void* x_perm, void* stream) {
  // the same checks as moe_permute (one validation path for both)
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  if (!x || !topk_idx || !counts_raw || !counts || !offsets || !row_of_slot || !slot_of_row || !x_perm)
    return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(x_perm)) return MOE_ERR_INVALID_ARG;
  if (permute_ws_bytes(T, E, k) > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch
  void* scratch = nullptr;
  cudaError_t e = scratch_ptr(&scratch);
  if (e == cudaSuccess)
    e = launch_permute(x, topk_idx, T, d, E, k, capacity, counts_raw, counts, offsets, row_of_slot, slot_of_row,
                       x_perm, scratch, device_status_ptr(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
