// C ABI of the MoE layer (include/moe.h): argument validation on the host,
// workspace carving, and the launch sequence of each call.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/moe.h"
#include "common.cuh"
#include "internal.h"

namespace moe {

// Device status word: kernels record the first device-side error here.
__device__ int g_moe_status = 0;
// Where moe_device_status() puts the value it exchanged out of the word.
__device__ int g_moe_status_out = 0;

namespace {
thread_local int t_last_cuda_error = 0;
std::mutex g_dev_mu;
int g_sm_count[64] = {0};
int* g_status_ptr[64] = {nullptr};

// launch timing of the calling thread (moe_timing_begin / _end)
struct LaunchTiming {
  bool on = false;
  void* const* events = nullptr;
  int capacity = 0;
  int n = 0;
  std::vector<const char*> names;
};
thread_local LaunchTiming t_timing;

inline int fail_cuda(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return MOE_ERR_CUDA;
}
inline int check(cudaError_t e) { return e == cudaSuccess ? MOE_OK : fail_cuda(e); }

inline size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// workspace of each call
size_t ws_route_topk_bwd(int T, int d, int E) {
  const int S = router_dw_splits(T, d, E);
  return 2 * align256((size_t)T * E * 2) + (S > 1 ? align256((size_t)S * E * d * 4) : 0);
}
// dlogits as bf16 hi + lo [T,E] x2, the router's fp32 term of dx [T,d]
size_t ws_permute_bwd(int T, int d, int E) { return 2 * align256((size_t)T * E * 2) + align256((size_t)T * d * 2); }

// grouped SwiGLU backward scratch: da|du hi+lo [rows,2H] x2, g*h hi+lo [rows,H] x2,
// gate-gradient partials [rows, ceil(H/256)], for the routed rows (T*k) and the
// shared expert (T rows).
struct SwigluBwdWs {
  size_t dau_hi, dau_lo, gh_hi, gh_lo, dgp, s_dau_hi, s_dau_lo, s_gh_hi, s_gh_lo, tile_counter, group_maps, total;
};
SwigluBwdWs swiglu_bwd_ws(int T, int k, int H, int Hs) {
  SwigluBwdWs w;
  const size_t R = (size_t)T * k;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += align256(bytes); return o; };
  w.dau_hi = take(R * 2 * H * 2);
  w.dau_lo = take(R * 2 * H * 2);
  w.gh_hi = take(R * H * 2);
  w.gh_lo = take(R * H * 2);
  w.dgp = take(R * dgp_slots(H) * 4);
  w.s_dau_hi = take((size_t)T * 2 * Hs * 2);
  w.s_dau_lo = take((size_t)T * 2 * Hs * 2);
  w.s_gh_hi = take((size_t)T * Hs * 2);
  w.s_gh_lo = take((size_t)T * Hs * 2);
  w.tile_counter = take(sizeof(int));  // dynamic tile schedule of the weight-gradient GEMMs
  w.group_maps = take(group_maps_bytes(kMaxE));  // their per-expert tensor maps
  w.total = off;
  return w;
}
size_t ws_swiglu_bwd(int T, int k, int H, int Hs) { return swiglu_bwd_ws(T, k, H, Hs).total; }

// Reads the status word and sets it to zero in one atomic step, so a code
// recorded by a kernel still running cannot fall between the read and the
// clear.
__global__ void status_exchange_kernel(int* status, int* out) { *out = atomicExch(status, 0); }

}  // namespace

int check_dims(int T, int d, int E, int k) {
  if (T < 1 || d < 1 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || k > E || E > kMaxE || (E % 8) != 0 || (d % 64) != 0) return MOE_ERR_UNSUPPORTED;
  if ((long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}
int check_hidden(int H, int Hs) {
  if (H < 128 || (H % 128) != 0) return MOE_ERR_UNSUPPORTED;
  if (Hs < 0 || (Hs % 128) != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

void record_cuda_error(cudaError_t e) { t_last_cuda_error = static_cast<int>(e); }

// An event record on `s`; while `s` is capturing, an event-record node of
// the graph (recorded again at every replay).
cudaError_t record_timing_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, s);
}

void timing_mark(cudaStream_t s, const char* name) {
  LaunchTiming& lt = t_timing;
  if (!lt.on) return;
  if (lt.n < lt.capacity) {
    record_timing_event(static_cast<cudaEvent_t>(lt.events[lt.n]), s);
    lt.names.push_back(name);
  }
  ++lt.n;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_status) == cudaSuccess) g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return (1 << 16) | 0; }

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "shape outside the supported limits";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_TIMEOUT: return "device: bounded wait expired";
    case MOE_ERR_DEVICE_BOUNDS: return "device: index out of range";
    case MOE_ERR_RANGE: return "device: a per-token sum was not finite (an fp16 term beyond its range, or inf / NaN)";
    default: return "unknown status";
  }
}

int moe_last_cuda_error(void) { return t_last_cuda_error; }

int moe_device_status(int* status_out) {
  if (!status_out) return MOE_ERR_INVALID_ARG;
  int* st = device_status_ptr();
  if (!st) return fail_cuda(cudaErrorInvalidSymbol);
  // one thread swaps the word for 0 and leaves the old value in
  // g_moe_status_out, which is copied back once that kernel has run
  int* out = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&out), g_moe_status_out);
  if (e != cudaSuccess) return fail_cuda(e);
  status_exchange_kernel<<<1, 1>>>(st, out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e);
  int v = 0;
  e = cudaMemcpy(&v, out, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  *status_out = v;
  return MOE_OK;
}

int moe_timing_begin(void* const* events, int capacity) {
  if (capacity < 0 || (capacity > 0 && !events)) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < capacity; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  LaunchTiming& lt = t_timing;
  lt.on = true;
  lt.events = events;
  lt.capacity = capacity;
  lt.n = 0;
  lt.names.clear();
  lt.names.reserve(capacity);
  return MOE_OK;
}

int moe_timing_end(int* n_launches) {
  LaunchTiming& lt = t_timing;
  if (!lt.on) return MOE_ERR_INVALID_ARG;
  lt.on = false;
  lt.events = nullptr;
  if (n_launches) *n_launches = lt.n;
  return MOE_OK;
}

int moe_timing_record(void* event, void* stream) {
  if (!event) return MOE_ERR_INVALID_ARG;
  return check(record_timing_event(static_cast<cudaEvent_t>(event), static_cast<cudaStream_t>(stream)));
}

const char* moe_timing_name(int i) {
  const LaunchTiming& lt = t_timing;
  if (i < 0 || i >= static_cast<int>(lt.names.size())) return "";
  return lt.names[i];
}

int moe_workspace_size(int T, int d, int E, int k, int H, int Hs, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  rc = check_hidden(H, Hs);
  if (rc) return rc;
  size_t b = permute_ws_bytes(T, E, k);
  size_t v = ws_route_topk_bwd(T, d, E);
  if (v > b) b = v;
  v = ws_permute_bwd(T, d, E);
  if (v > b) b = v;
  v = ws_swiglu_bwd(T, k, H, Hs);
  if (v > b) b = v;
  v = balance_loss_ws_bytes(T, E);
  if (v > b) b = v;
  *bytes = b;
  return MOE_OK;
}

int moe_route_topk(const void* x, const void* W_r, const float* bias, const float* logits_in, int T, int d, int E,
                   int k, float* logits, int32_t* topk_idx, float* gates, void* ws, size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  if (T < 1 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || k > E || E > kMaxE || (E % 8) != 0) return MOE_ERR_UNSUPPORTED;
  if (!topk_idx || !gates) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float* src = logits_in;
  if (!logits_in) {
    int rc = check_dims(T, d, E, k);
    if (rc) return rc;
    if (!x || !W_r || !logits || !al16(x) || !al16(W_r) || !al16(logits) || (bias && !al16(bias)))
      return MOE_ERR_INVALID_ARG;
    cudaError_t e = gemm_router_fwd(x, W_r, bias, T, d, E, logits, device_status_ptr(), s);
    if (e != cudaSuccess) return fail_cuda(e);
    src = logits;
  }
  return check(launch_topk_gating(src, T, E, k, topk_idx, gates, device_status_ptr(), s));
}

int moe_permute(const void* x, const int32_t* topk_idx, int T, int d, int E, int k, int capacity, int32_t* counts_raw,
                int32_t* counts, int32_t* offsets, int32_t* row_of_slot, int32_t* slot_of_row, void* x_perm, void* ws,
                size_t ws_bytes, void* stream) {
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  if (!topk_idx || !counts_raw || !counts || !offsets || !row_of_slot || !slot_of_row) return MOE_ERR_INVALID_ARG;
  // x_perm == NULL: the maps only (x unused)
  if (x_perm && (!x || !al16(x) || !al16(x_perm))) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < permute_ws_bytes(T, E, k)) return MOE_ERR_WORKSPACE;
  return check(launch_permute(x, topk_idx, T, d, E, k, capacity, counts_raw, counts, offsets, row_of_slot,
                              slot_of_row, x_perm, ws, device_status_ptr(), static_cast<cudaStream_t>(stream)));
}

int moe_grouped_swiglu(const void* x_perm, const int32_t* offsets, const void* x, int T, int d, int E, int k, int H,
                       int Hs, const void* W_g, const void* W_u, const void* W_d, const void* Ws_g, const void* Ws_u,
                       const void* Ws_d, float* au, void* h, void* o_perm, float* au_s, void* h_s, void* s_out,
                       void* ws, size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  rc = check_hidden(H, Hs);
  if (rc) return rc;
  if (!x_perm || !offsets || !W_g || !W_u || !W_d || !h || !o_perm) return MOE_ERR_INVALID_ARG;
  if (!al16(x_perm) || !al16(W_g) || !al16(W_u) || !al16(W_d) || !al16(h) || !al16(o_perm) || (au && !al16(au)))
    return MOE_ERR_INVALID_ARG;
  if (Hs > 0) {
    if (!x || !Ws_g || !Ws_u || !Ws_d || !h_s || !s_out) return MOE_ERR_INVALID_ARG;
    if (!al16(x) || !al16(Ws_g) || !al16(Ws_u) || !al16(Ws_d) || !al16(h_s) || !al16(s_out) ||
        (au_s && !al16(au_s)))
      return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = device_status_ptr();
  SwigluFwdArgs r{x_perm, T * k, offsets, E, d, H, W_g, W_u, au, h};
  SwigluFwdArgs sh{x, T, nullptr, 1, d, Hs, Ws_g, Ws_u, au_s, h_s};
  cudaError_t e = gemm_swiglu_fwd(r, Hs > 0 ? &sh : nullptr, status, st);
  if (e != cudaSuccess) return fail_cuda(e);
  DownFwdArgs rd{h, T * k, offsets, E, d, H, W_d, o_perm};
  DownFwdArgs sd{h_s, T, nullptr, 1, d, Hs, Ws_d, s_out};
  return check(gemm_down_fwd(rd, Hs > 0 ? &sd : nullptr, status, st));
}

int moe_grouped_swiglu_recompute(const void* x_perm, const int32_t* offsets, const void* x, int T, int d, int E,
                                 int k, int H, int Hs, const void* W_g, const void* W_u, const void* Ws_g,
                                 const void* Ws_u, float* au, float* au_s, void* stream) {
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  rc = check_hidden(H, Hs);
  if (rc) return rc;
  if (!x_perm || !offsets || !W_g || !W_u || !au) return MOE_ERR_INVALID_ARG;
  if (!al16(x_perm) || !al16(W_g) || !al16(W_u) || !al16(au)) return MOE_ERR_INVALID_ARG;
  if (Hs > 0) {
    if (!x || !Ws_g || !Ws_u || !au_s) return MOE_ERR_INVALID_ARG;
    if (!al16(x) || !al16(Ws_g) || !al16(Ws_u) || !al16(au_s)) return MOE_ERR_INVALID_ARG;
  }
  SwigluFwdArgs r{x_perm, T * k, offsets, E, d, H, W_g, W_u, au, nullptr};
  SwigluFwdArgs sh{x, T, nullptr, 1, d, Hs, Ws_g, Ws_u, au_s, nullptr};
  return check(gemm_swiglu_fwd(r, Hs > 0 ? &sh : nullptr, device_status_ptr(), static_cast<cudaStream_t>(stream)));
}

int moe_grouped_swiglu_fused(const void* x, const int32_t* slot_of_row, const int32_t* row_of_slot,
                             const float* gates, const int32_t* offsets, int T, int d, int E, int k, int H, int Hs,
                             const void* W_g, const void* W_u, const void* W_d, const void* Ws_g, const void* Ws_u,
                             const void* Ws_d, float* au, void* h, void* o_slot, float* au_s, void* h_s, void* y,
                             void* stream) {
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  rc = check_hidden(H, Hs);
  if (rc) return rc;
  const void* req[] = {x, slot_of_row, row_of_slot, gates, offsets, W_g, W_u, W_d, h, o_slot, y};
  for (const void* p : req)
    if (!p) return MOE_ERR_INVALID_ARG;
  const void* req16[] = {x, W_g, W_u, W_d, h, o_slot, y};
  for (const void* p : req16)
    if (!al16(p)) return MOE_ERR_INVALID_ARG;
  if (au && !al16(au)) return MOE_ERR_INVALID_ARG;
  if (Hs > 0) {
    if (!Ws_g || !Ws_u || !Ws_d || !h_s) return MOE_ERR_INVALID_ARG;
    if (!al16(Ws_g) || !al16(Ws_u) || !al16(Ws_d) || !al16(h_s) || (au_s && !al16(au_s))) return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = device_status_ptr();
  const int R = T * k;
  const RowGather gx{x, T, slot_of_row, k, R};
  // gate/up: routed A rows gathered from x; shared expert on x
  SwigluFwdArgs r{nullptr, R, offsets, E, d, H, W_g, W_u, au, h, gx};
  SwigluFwdArgs sh{x, T, nullptr, 1, d, Hs, Ws_g, Ws_u, au_s, h_s};
  cudaError_t e = gemm_swiglu_fwd(r, Hs > 0 ? &sh : nullptr, status, st);
  if (e != cudaSuccess) return fail_cuda(e);
  // routed down projection: each row's output stored at its slot
  DownFwdArgs rd{h, R, offsets, E, d, H, W_d, o_slot, slot_of_row, R};
  e = gemm_down_fwd(rd, nullptr, status, st);
  if (e != cudaSuccess) return fail_cuda(e);
  if (Hs == 0) return check(launch_combine_slots(o_slot, nullptr, gates, row_of_slot, T, d, k, y, status, st));
  // shared down projection with the combine in its epilogue (after the
  // routed one on the same stream: every o_slot row is written by then)
  DownFwdArgs sd{h_s, T, nullptr, 1, d, Hs, Ws_d, nullptr, nullptr, 0, o_slot, gates, row_of_slot, k, y};
  return check(gemm_down_fwd(sd, nullptr, status, st));
}

int moe_grouped_swiglu_recompute_fused(const void* x, const int32_t* slot_of_row, const int32_t* offsets, int T,
                                       int d, int E, int k, int H, int Hs, const void* W_g, const void* W_u,
                                       const void* Ws_g, const void* Ws_u, float* au, float* au_s, void* stream) {
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  rc = check_hidden(H, Hs);
  if (rc) return rc;
  if (!x || !slot_of_row || !offsets || !W_g || !W_u || !au) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(W_g) || !al16(W_u) || !al16(au)) return MOE_ERR_INVALID_ARG;
  if (Hs > 0) {
    if (!Ws_g || !Ws_u || !au_s) return MOE_ERR_INVALID_ARG;
    if (!al16(Ws_g) || !al16(Ws_u) || !al16(au_s)) return MOE_ERR_INVALID_ARG;
  }
  const int R = T * k;
  SwigluFwdArgs r{nullptr, R, offsets, E, d, H, W_g, W_u, au, nullptr, RowGather{x, T, slot_of_row, k, R}};
  SwigluFwdArgs sh{x, T, nullptr, 1, d, Hs, Ws_g, Ws_u, au_s, nullptr};
  return check(gemm_swiglu_fwd(r, Hs > 0 ? &sh : nullptr, device_status_ptr(), static_cast<cudaStream_t>(stream)));
}

int moe_unpermute_combine(const void* o_perm, const void* s_out, const float* gates, const int32_t* row_of_slot,
                          int T, int d, int k, void* y, void* stream) {
  if (T < 1 || d < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || (d % 64) != 0 || (long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (!o_perm || !gates || !row_of_slot || !y) return MOE_ERR_INVALID_ARG;
  if (!al16(o_perm) || !al16(y) || (s_out && !al16(s_out))) return MOE_ERR_INVALID_ARG;
  return check(launch_combine(o_perm, s_out, gates, row_of_slot, T, d, k, y, device_status_ptr(),
                              static_cast<cudaStream_t>(stream)));
}

int moe_unpermute_combine_bwd(const void* dY, const int32_t* row_of_slot, int T, int d, int k, void* dY_perm,
                              void* stream) {
  if (T < 1 || d < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || (d % 64) != 0 || (long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (!dY || !row_of_slot || !dY_perm) return MOE_ERR_INVALID_ARG;
  if (!al16(dY) || !al16(dY_perm)) return MOE_ERR_INVALID_ARG;
  return check(launch_gather_rows(dY, row_of_slot, T, d, k, dY_perm, device_status_ptr(),
                                  static_cast<cudaStream_t>(stream)));
}

int moe_grouped_swiglu_bwd(const void* dY_perm, const void* dY, const float* gates, const int32_t* row_of_slot,
                           const int32_t* slot_of_row, const int32_t* offsets, const void* x_perm, const void* x,
                           const float* au, const float* au_s, int T, int d, int E, int k, int H, int Hs,
                           const void* W_g, const void* W_u, const void* W_d, const void* Ws_g, const void* Ws_u,
                           const void* Ws_d, void* dx_perm, void* dx_s, void* dW_g, void* dW_u, void* dW_d,
                           void* dWs_g, void* dWs_u, void* dWs_d, float* dgates, uint32_t* dx_scale, void* ws,
                           size_t ws_bytes, void* stream) {
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  rc = check_hidden(H, Hs);
  if (rc) return rc;
  // dY_perm == x_perm == NULL: the GEMMs gather the rows of dY and x
  // themselves (the permutation fused into their loads)
  const bool gather = dY_perm == nullptr;
  if ((x_perm == nullptr) != gather) return MOE_ERR_INVALID_ARG;
  const void* req[] = {gates, row_of_slot, slot_of_row, offsets, au, W_g, W_u, W_d, dx_perm, dW_g, dW_u, dW_d, dgates};
  for (const void* p : req)
    if (!p) return MOE_ERR_INVALID_ARG;
  const void* req16[] = {au, W_g, W_u, W_d, dx_perm, dW_g, dW_u, dW_d};
  for (const void* p : req16)
    if (!al16(p)) return MOE_ERR_INVALID_ARG;
  if (gather ? (!dY || !x || !al16(dY) || !al16(x)) : (!al16(dY_perm) || !al16(x_perm))) return MOE_ERR_INVALID_ARG;
  // the scale of the fp16 input-gradient terms comes from dY
  if (dx_scale && (!dY || !al16(dY))) return MOE_ERR_INVALID_ARG;
  if (Hs > 0) {
    const void* req_s[] = {dY, x, au_s, Ws_g, Ws_u, Ws_d, dx_s, dWs_g, dWs_u, dWs_d};
    for (const void* p : req_s)
      if (!p || !al16(p)) return MOE_ERR_INVALID_ARG;
  }
  const SwigluBwdWs L = swiglu_bwd_ws(T, k, H, Hs);
  if (!ws || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = device_status_ptr();
  char* w = static_cast<char*>(ws);
  const int R = T * k;
  float* dgp = reinterpret_cast<float*>(w + L.dgp);
  const RowGather gdy = gather ? RowGather{dY, T, slot_of_row, k, R} : RowGather{};
  const RowGather gx = gather ? RowGather{x, T, slot_of_row, k, R} : RowGather{};
  cudaError_t e = cudaSuccess;
  if (dx_scale) {
    e = launch_grad_scale(dY, (long long)T * d, dx_scale, st);
    if (e != cudaSuccess) return fail_cuda(e);
  }

  // 1. dgrad of the down projection with the SwiGLU backward epilogue
  DgradDownArgs r1{dY_perm, R, offsets, E, d, H, W_d, au, w + L.dau_hi, w + L.dau_lo, w + L.gh_hi, w + L.gh_lo,
                   gates, slot_of_row, R, dgp, gdy};
  DgradDownArgs s1{dY, T, nullptr, 1, d, Hs, Ws_d, au_s, w + L.s_dau_hi, w + L.s_dau_lo, w + L.s_gh_hi,
                   w + L.s_gh_lo, nullptr, nullptr, 0, nullptr};
  e = gemm_dgrad_down(r1, Hs > 0 ? &s1 : nullptr, status, st);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_dgates_reduce(dgp, dgp_slots(H), row_of_slot, T, k, dgates, st);
  if (e != cudaSuccess) return fail_cuda(e);

  // 2. dW_d = dY_perm^T (g h), g h split into bf16 hi + lo
  WgradArgs r2{dY_perm, nullptr, w + L.gh_hi, w + L.gh_lo, R, offsets, E, d, H, dW_d, nullptr, 0, gdy, 0};
  WgradArgs s2{dY, nullptr, w + L.s_gh_hi, w + L.s_gh_lo, T, nullptr, 1, d, Hs, dWs_d, nullptr, 0};
  int* tile_counter = reinterpret_cast<int*>(w + L.tile_counter);
  void* group_maps = w + L.group_maps;
  e = gemm_wgrad(r2, Hs > 0 ? &s2 : nullptr, tile_counter, group_maps, status, st, "gemm_wgrad_down");
  if (e != cudaSuccess) return fail_cuda(e);

  // 3. dx_perm = [da|du] [W_g; W_u]
  // routed rows carry their gate factor (g < 1), so their bf16 da|du error is
  // small next to the shared expert's; only the shared operand is split
  DgradGuArgs r3{w + L.dau_hi, nullptr, R, offsets, E, d, H, W_g, W_u, dx_perm, dx_scale};
  DgradGuArgs s3{w + L.s_dau_hi, w + L.s_dau_lo, T, nullptr, 1, d, Hs, Ws_g, Ws_u, dx_s, dx_scale};
  e = gemm_dgrad_gu(r3, Hs > 0 ? &s3 : nullptr, status, st);
  if (e != cudaSuccess) return fail_cuda(e);

  // 4. [dW_g; dW_u] = [da|du]^T x_perm, [da|du] split into bf16 hi + lo
  WgradArgs r4{w + L.dau_hi, w + L.dau_lo, x_perm, nullptr, R, offsets, E, 2 * H, d, dW_g, dW_u, H, gx, 1};
  WgradArgs s4{w + L.s_dau_hi, w + L.s_dau_lo, x, nullptr, T, nullptr, 1, 2 * Hs, d, dWs_g, dWs_u, Hs};
  return check(gemm_wgrad(r4, Hs > 0 ? &s4 : nullptr, tile_counter, group_maps, status, st, "gemm_wgrad_gate_up"));
}

int moe_route_topk_bwd(const float* dgates, const float* gates, const int32_t* topk_idx, const void* x, int T, int d,
                       int E, int k, float* dlogits, float* dW_r, const float* dlogits_add, void* ws, size_t ws_bytes,
                       void* stream) {
  if (T < 1 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || k > E || E > kMaxE || (E % 8) != 0) return MOE_ERR_UNSUPPORTED;
  if (!dgates || !gates || !topk_idx || !dlogits) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (dW_r == nullptr)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!x)
    return check(launch_router_bwd_dl(dgates, gates, topk_idx, T, E, k, dlogits_add, dlogits, nullptr, nullptr, st));
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  if (!al16(x) || !al16(dW_r)) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < ws_route_topk_bwd(T, d, E)) return MOE_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  uint16_t* dl_hi = reinterpret_cast<uint16_t*>(w);
  uint16_t* dl_lo = reinterpret_cast<uint16_t*>(w + align256((size_t)T * E * 2));
  cudaError_t e = launch_router_bwd_dl(dgates, gates, topk_idx, T, E, k, dlogits_add, dlogits, dl_hi, dl_lo, st);
  if (e != cudaSuccess) return fail_cuda(e);
  const int S = router_dw_splits(T, d, E);
  float* part = S > 1 ? reinterpret_cast<float*>(w + 2 * align256((size_t)T * E * 2)) : dW_r;
  e = gemm_router_dw(dl_hi, dl_lo, x, T, d, E, S, part, device_status_ptr(), st);
  if (e != cudaSuccess) return fail_cuda(e);
  if (S > 1) return check(launch_splitk_reduce(part, S, (long long)E * d, dW_r, st));
  return MOE_OK;
}

int moe_router_balance_loss(const float* logits, const int32_t* counts_raw, int T, int E, int k, float alpha,
                            float* loss, float* P_mean, float* dlogits_lbl, void* ws, size_t ws_bytes, void* stream) {
  if (T < 1 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || k > E || E > kMaxE || (E % 8) != 0) return MOE_ERR_UNSUPPORTED;
  if (!logits || !counts_raw || !loss) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < balance_loss_ws_bytes(T, E)) return MOE_ERR_WORKSPACE;
  return check(launch_balance_loss(logits, counts_raw, T, E, k, alpha, loss, P_mean, dlogits_lbl, ws,
                                   static_cast<cudaStream_t>(stream)));
}

int moe_mxfp8_rows(int T, int E, int k, long long* rows) {
  if (!rows || T < 1 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || k > E || E > kMaxE || (long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  *rows = mx_rows_max(T, E, k);
  return MOE_OK;
}

int moe_mxfp8_scales_bytes(long long rows, int cols, size_t* bytes) {
  if (!bytes || rows < 1 || cols < 1) return MOE_ERR_INVALID_ARG;
  if (cols % 128) return MOE_ERR_UNSUPPORTED;
  *bytes = mx_scales_bytes(rows, cols);
  return MOE_OK;
}

int moe_mxfp8_quantize(const void* src, long long rows, int cols, void* codes, void* scales, void* stream) {
  if (!src || !codes || !scales || rows < 1 || cols < 1) return MOE_ERR_INVALID_ARG;
  if (cols % 128 || rows * cols >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
  if (!al16(src) || !al16(codes) || !al16(scales)) return MOE_ERR_INVALID_ARG;
  return check(launch_mx_quantize(src, rows, cols, codes, scales, static_cast<cudaStream_t>(stream)));
}

int moe_mxfp8_quantize_gate_up(const void* W_g, const void* W_u, int E, int H, int d, void* codes, void* scales,
                               void* stream) {
  if (!W_g || !W_u || !codes || !scales || E < 1 || H < 1 || d < 1) return MOE_ERR_INVALID_ARG;
  if (d % 128 || H % 128) return MOE_ERR_UNSUPPORTED;
  if (!al16(W_g) || !al16(W_u) || !al16(codes) || !al16(scales)) return MOE_ERR_INVALID_ARG;
  return check(launch_mx_quantize_gate_up(W_g, W_u, E, H, d, codes, scales, static_cast<cudaStream_t>(stream)));
}

int moe_permute_mxfp8(const void* x, const int32_t* topk_idx, int T, int d, int E, int k, int capacity,
                      int32_t* counts_raw, int32_t* counts, int32_t* offsets, int32_t* mx_offsets,
                      int32_t* row_of_slot, int32_t* slot_of_row, void* x_codes, void* x_scales, void* ws,
                      size_t ws_bytes, void* stream) {
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  if (d % 128) return MOE_ERR_UNSUPPORTED;
  if (!x || !topk_idx || !counts_raw || !counts || !offsets || !mx_offsets || !row_of_slot || !slot_of_row ||
      !x_codes || !x_scales)
    return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(x_codes) || !al16(x_scales)) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < permute_ws_bytes(T, E, k)) return MOE_ERR_WORKSPACE;
  return check(launch_permute_mx(x, topk_idx, T, d, E, k, capacity, counts_raw, counts, offsets, mx_offsets,
                                 row_of_slot, slot_of_row, x_codes, x_scales, ws, device_status_ptr(),
                                 static_cast<cudaStream_t>(stream)));
}

int moe_grouped_swiglu_mxfp8(const void* x_codes, const void* x_scales, const int32_t* mx_offsets,
                             const int32_t* counts, const void* xs_codes, const void* xs_scales, int T, int d, int E,
                             int k, int H, int Hs, const void* Wgu_codes, const void* Wgu_scales,
                             const void* Wd_codes, const void* Wd_scales, const void* Wsgu_codes,
                             const void* Wsgu_scales, const void* Wsd_codes, const void* Wsd_scales, void* h_codes,
                             void* h_scales, void* hs_codes, void* hs_scales, void* o_perm, void* s_out,
                             void* stream) {
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  rc = check_hidden(H, Hs);
  if (rc) return rc;
  if (d % 128) return MOE_ERR_UNSUPPORTED;
  const void* req[] = {x_codes, x_scales, mx_offsets, counts, Wgu_codes, Wgu_scales, Wd_codes, Wd_scales,
                       h_codes, h_scales, o_perm};
  for (const void* p : req)
    if (!p) return MOE_ERR_INVALID_ARG;
  const void* req16[] = {x_codes, x_scales, Wgu_codes, Wgu_scales, Wd_codes, Wd_scales, h_codes, h_scales, o_perm};
  for (const void* p : req16)
    if (!al16(p)) return MOE_ERR_INVALID_ARG;
  if (Hs > 0) {
    const void* req_s[] = {xs_codes, xs_scales, Wsgu_codes, Wsgu_scales, Wsd_codes, Wsd_scales, hs_codes,
                           hs_scales, s_out};
    for (const void* p : req_s)
      if (!p || !al16(p)) return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rows = static_cast<int>(mx_rows_max(T, E, k));
  auto U = [](const void* p) { return static_cast<const uint8_t*>(p); };
  MxGemmArgs r1{x_codes, U(x_scales), rows, mx_offsets, counts, E, d, H, Wgu_codes, U(Wgu_scales), h_codes,
                static_cast<uint8_t*>(h_scales)};
  MxGemmArgs s1{xs_codes, U(xs_scales), T, nullptr, nullptr, 1, d, Hs, Wsgu_codes, U(Wsgu_scales), hs_codes,
                static_cast<uint8_t*>(hs_scales)};
  cudaError_t e = gemm_mx_swiglu(r1, Hs > 0 ? &s1 : nullptr, st);
  if (e != cudaSuccess) return fail_cuda(e);
  MxGemmArgs r2{h_codes, U(h_scales), rows, mx_offsets, counts, E, H, d, Wd_codes, U(Wd_scales), o_perm, nullptr};
  MxGemmArgs s2{hs_codes, U(hs_scales), T, nullptr, nullptr, 1, Hs, d, Wsd_codes, U(Wsd_scales), s_out, nullptr};
  return check(gemm_mx_down(r2, Hs > 0 ? &s2 : nullptr, st));
}

int moe_unpermute_combine_mxfp8(const void* o_perm, const void* s_out, const float* gates,
                                const int32_t* row_of_slot, int T, int d, int E, int k, void* y, void* stream) {
  if (T < 1 || d < 1 || k < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || k > E || E > kMaxE || (d % 64) != 0 || (long long)T * k >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED;
  if (!o_perm || !gates || !row_of_slot || !y) return MOE_ERR_INVALID_ARG;
  if (!al16(o_perm) || !al16(y) || (s_out && !al16(s_out))) return MOE_ERR_INVALID_ARG;
  return check(launch_combine_rows(o_perm, s_out, gates, row_of_slot, T, d, k, mx_rows_max(T, E, k), y,
                                   device_status_ptr(), static_cast<cudaStream_t>(stream)));
}

int moe_permute_bwd(const void* dx_perm, const void* dx_s, const int32_t* row_of_slot, const float* dlogits,
                    const void* W_r, int T, int d, int E, int k, void* dx, const uint32_t* dx_scale, void* ws,
                    size_t ws_bytes, void* stream) {
  if (T < 1 || d < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || (d % 64) != 0 || (long long)T * k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (!dx_perm || !row_of_slot || !dx) return MOE_ERR_INVALID_ARG;
  if (!al16(dx_perm) || !al16(dx) || (dx_s && !al16(dx_s))) return MOE_ERR_INVALID_ARG;
  if ((dlogits == nullptr) != (W_r == nullptr)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!W_r)
    return check(
        launch_unpermute_reduce(dx_perm, dx_s, nullptr, row_of_slot, T, d, k, dx_scale, dx, device_status_ptr(), st));
  int rc = check_dims(T, d, E, k);
  if (rc) return rc;
  if (!al16(W_r)) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < ws_permute_bwd(T, d, E)) return MOE_ERR_WORKSPACE;
  uint16_t* dl_hi = static_cast<uint16_t*>(ws);
  uint16_t* dl_lo = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + align256((size_t)T * E * 2));
  cudaError_t e = launch_f32_to_bf16_split(dlogits, dl_hi, dl_lo, (long long)T * E, st);
  if (e != cudaSuccess) return fail_cuda(e);
  void* dx_r = static_cast<char*>(ws) + 2 * align256((size_t)T * E * 2);  // fp16 [T, d]
  e = gemm_router_dx(dl_hi, dl_lo, W_r, T, d, E, dx_r, dx_scale, device_status_ptr(), st);
  if (e != cudaSuccess) return fail_cuda(e);
  return check(
      launch_unpermute_reduce(dx_perm, dx_s, dx_r, row_of_slot, T, d, k, dx_scale, dx, device_status_ptr(), st));
}

}  // extern "C"
