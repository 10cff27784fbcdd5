// Host-side interface between the C ABI (moe_abi.cu) and the kernel files.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// argument checks shared by every entry point (MOE_OK or the ABI's error code)
int check_dims(int T, int d, int E, int k);  // limits of T, d, E, k
int check_hidden(int H, int Hs);             // limits of H and Hs
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// per-device facts and the device status word
int device_sm_count();
int* device_status_ptr();  // device address of the status word of the current device
void record_cuda_error(cudaError_t e);  // what moe_last_cuda_error() reports in this thread
// Launch timing (moe_timing_begin): records the caller's next event on `s`
// and notes `name` (a string literal) when timing is on in this thread; called
// just before every kernel launch or memset the library issues.
void timing_mark(cudaStream_t s, const char* name);

// ------------------------------------------------------------ SIMT kernels
cudaError_t launch_topk_gating(const float* logits, int T, int E, int k, int32_t* idx, float* gates,
                               int* status, cudaStream_t s);
cudaError_t launch_permute(const void* x, const int32_t* idx, int T, int d, int E, int k, int capacity,
                           int32_t* counts_raw, int32_t* counts, int32_t* offsets, int32_t* row_of_slot,
                           int32_t* slot_of_row, void* x_perm, void* ws, int* status, cudaStream_t s);
size_t permute_ws_bytes(int T, int E, int k);
// histogram + scan of the permutation (the scatter's inputs: per-tile bases
// and in-tile ranks, in ws); mx_offsets (nullable) receives the offsets of the
// padded row space of the MXFP8 path (every expert's rows start at a multiple
// of 128)
cudaError_t launch_permute_counts(const int32_t* idx, int T, int E, int k, int capacity, int32_t* counts_raw,
                                  int32_t* counts, int32_t* offsets, int32_t* mx_offsets, void* ws,
                                  int32_t** tile_base_out, int32_t** inrank_out, int* status, cudaStream_t s);

// ------------------------------------------------------------ MXFP8
// rows of the padded row space (each expert's rows rounded up to 128): at most
// T*k + 127*E, rounded up to a whole 128-row tile
inline long long mx_rows_max(int T, int E, int k) {
  return ((long long)T * k + 127LL * E + 127) / 128 * 128;
}
// bytes of the tile-atom scale array of a [rows, cols] MXFP8 matrix
size_t mx_scales_bytes(long long rows, int cols);
cudaError_t launch_mx_quantize(const void* src, long long rows, int cols, void* codes, void* scales, cudaStream_t s);
cudaError_t launch_mx_quantize_gate_up(const void* W_g, const void* W_u, int E, int H, int d, void* codes,
                                       void* scales, cudaStream_t s);
cudaError_t launch_permute_mx(const void* x, const int32_t* idx, int T, int d, int E, int k, int capacity,
                              int32_t* counts_raw, int32_t* counts, int32_t* offsets, int32_t* mx_offsets,
                              int32_t* row_of_slot, int32_t* slot_of_row, void* codes, void* scales, void* ws,
                              int* status, cudaStream_t s);
// o_perm, s_out fp16 (the per-token sum terms); y bf16
cudaError_t launch_combine(const void* o_perm, const void* s_out, const float* gates, const int32_t* row_of_slot,
                           int T, int d, int k, void* y, int* status, cudaStream_t s);
// dY_perm[row_of_slot[t*k+s]] = dY[t] for every kept slot
cudaError_t launch_gather_rows(const void* dY, const int32_t* row_of_slot, int T, int d, int k, void* dY_perm,
                               int* status, cudaStream_t s);
// per-row partials of the gate gradient: two per 256-column tile of H (one
// per accumulator-column half of the tile)
inline int dgp_slots(int H) { return 2 * ((H + 255) / 256); }
// dgates[t,s] = sum_p dgp[row_of_slot[t*k+s], p] (0 for dropped slots)
cudaError_t launch_dgates_reduce(const float* dgp, int P, const int32_t* row_of_slot, int T, int k, float* dgates,
                                 cudaStream_t s);
// dx[t] = 2^e (sum_s dx_perm[row(t,s)] + dx_s[t] + dx_r[t])   (fp16 terms, fp32
// sum; dx_s and dx_r nullable; e from the scale word, NULL: e = 0; dx bf16)
cudaError_t launch_unpermute_reduce(const void* dx_perm, const void* dx_s, const void* dx_r,
                                    const int32_t* row_of_slot, int T, int d, int k, const uint32_t* scale, void* dx,
                                    int* status, cudaStream_t s);
// the scale word of the backward's fp16 terms: zeroed, then the largest bf16
// magnitude pattern of dY[n] (n a multiple of 8)
cudaError_t launch_grad_scale(const void* dY, long long n, uint32_t* word, cudaStream_t s);
// dlogits [T,E] fp32 (dense, + add[T,E] if add != NULL) and, if dl_hi != NULL,
// its bf16 hi + lo halves [T,E]
cudaError_t launch_router_bwd_dl(const float* dgates, const float* gates, const int32_t* idx, int T, int E, int k,
                                 const float* add, float* dlogits, uint16_t* dl_hi, uint16_t* dl_lo, cudaStream_t s);
// router balance loss: loss, P_mean [E] (nullable), dl [T,E] (nullable)
size_t balance_loss_ws_bytes(int T, int E);
cudaError_t launch_balance_loss(const float* logits, const int32_t* counts_raw, int T, int E, int k, float alpha,
                                float* loss, float* P_mean, float* dl, void* ws, cudaStream_t s);
// v -> bf16 hi + lo halves
cudaError_t launch_f32_to_bf16_split(const float* src, uint16_t* hi, uint16_t* lo, long long n, cudaStream_t s);
cudaError_t launch_splitk_reduce(const float* partial, int S, long long n, float* out, cudaStream_t s);

// ------------------------------------------------------------ tensor-core GEMMs
// All return cudaSuccess or an error; tensor-map encoding failures map to
// cudaErrorInvalidValue.
// Row gather (the permutation fused into an operand's TMA loads): permuted
// row r of the operand is row slot_of_row[r] / k of src.  src == NULL: none.
struct RowGather {
  const void* src;             // [src_rows, cols] bf16 (x or dY)
  int src_rows;
  const int32_t* slot_of_row;  // permuted row -> slot t*k+s
  int k;
  int nslots;                  // T*k
};
struct SwigluFwdArgs {
  const void* a;        // [rows, d] bf16 (x_perm or x)
  int rows_total;       // rows of the A buffer
  const int32_t* offsets;  // [G+1] device, or NULL (dense: G = 1 over rows_total)
  int G, d, H;
  const void* Wg;       // [G, H, d]
  const void* Wu;
  float* au;            // [rows, 2H] fp32 (a | u) or NULL
  void* h;              // [rows, H], or NULL (a | u only: the backward's recompute)
  RowGather gather;     // A rows gathered from gather.src (`a` unused)
};
struct DownFwdArgs {
  const void* h;        // [rows, H]
  int rows_total;
  const int32_t* offsets;
  int G, d, H;
  const void* Wd;       // [G, d, H]
  void* o;              // [rows, d] fp16 (unused with comb_y)
  const int32_t* out_row_map;  // row r stored at row out_row_map[r] of o (NULL: r)
  int out_map_rows;            // rows of o with a row map
  // combine fused into this (dense, shared-expert) problem's epilogue:
  // y[t] = bf16(o[t] + sum_{kept j} gates[t,j] comb_o[t*k+j]), o not stored
  const void* comb_o;          // [T*k, d] fp16, slot order
  const float* comb_gates;
  const int32_t* comb_row_of_slot;
  int comb_k;
  void* comb_y;                // [T, d] bf16
};
// routed + (optional) shared in one persistent launch
cudaError_t gemm_swiglu_fwd(const SwigluFwdArgs& routed, const SwigluFwdArgs* shared, int* status, cudaStream_t s);
cudaError_t gemm_down_fwd(const DownFwdArgs& routed, const DownFwdArgs* shared, int* status, cudaStream_t s);
// logits[T,E] = x W_r^T + bias
cudaError_t gemm_router_fwd(const void* x, const void* W_r, const float* bias, int T, int d, int E, float* logits,
                            int* status, cudaStream_t s);

struct DgradDownArgs {    // dau = swiglu_bwd(g * (dY_perm W_d), au), plus g*h and the gate-gradient partials
  const void* dY;         // [rows, d] (gathered upstream gradient, no gate)
  int rows_total;
  const int32_t* offsets;
  int G, d, H;
  const void* Wd;         // [G, d, H]
  const float* au;        // [rows, 2H] fp32
  void* dau_hi;           // [rows, 2H] bf16
  void* dau_lo;
  void* gh_hi;            // [rows, H] bf16
  void* gh_lo;
  const float* gates;     // per-slot gates or NULL (g = 1)
  const int32_t* slot_of_row;
  int gate_slots;
  float* dgp;             // [rows, dgp_slots(H)] or NULL
  RowGather gather;       // dY rows gathered from gather.src (`dY` unused)
};
struct DgradGuArgs {      // dx = (dau_hi + dau_lo) [W_g; W_u]
  const void* dau;        // [rows, 2H] bf16 hi half
  const void* dau_lo;     // lo half (split precision) or NULL
  int rows_total;
  const int32_t* offsets;
  int G, d, H;
  const void* Wg;         // [G, H, d]
  const void* Wu;
  void* dx;               // [rows, d] fp16, divided by 2^e of the scale word
  const uint32_t* scale;  // nullable (e = 0)
};
struct WgradArgs {        // out[g] = A_g^T B_g over rows [off[g], off[g+1])
  const void* A;          // [rows, M] bf16
  const void* A_lo;       // lo half of A (split precision) or NULL
  const void* B;          // [rows, N] bf16
  const void* B_lo;       // lo half of B or NULL
  int rows_total;
  const int32_t* offsets; // or NULL: G = 1 over rows_total
  int G, M, N;
  void* out;              // [G, M, N] (rows < row_split), bf16
  void* out2;             // rows >= row_split go here as [G, M - row_split, N]; NULL = none
  int row_split;
  RowGather gather;       // rows of operand gather_op (0: A, 1: B) gathered (that pointer unused)
  int gather_op;
};
cudaError_t gemm_dgrad_down(const DgradDownArgs& routed, const DgradDownArgs* shared, int* status, cudaStream_t s);
cudaError_t gemm_dgrad_gu(const DgradGuArgs& routed, const DgradGuArgs* shared, int* status, cudaStream_t s);
// `tile_counter`: one device int, zeroed by the launch (dynamic tile schedule);
// `group_maps`: device scratch of group_maps_bytes(G) bytes (128-byte
// aligned) for the per-group tensor maps of a problem with offsets
cudaError_t gemm_wgrad(const WgradArgs& routed, const WgradArgs* shared, int* tile_counter, void* group_maps,
                       int* status, cudaStream_t s, const char* name);
size_t group_maps_bytes(int G);
// Per-group maps: for each group g and operand m, a block view of the whole
// [extent, cols] buffer at base[m] re-based at row off[g] with off[g+1] -
// off[g] rows; out[g * 3 + m] in device memory.  `whole` is encoded with the
// buffer's rows, `whole_1row` with one row (same box).  A non-null
// `tile_counter` is zeroed for the GEMM launched next (in place of a memset,
// which would break the chain of programmatic launches).
cudaError_t launch_group_maps(const CUtensorMap* whole, const CUtensorMap* whole_1row, const void* const* base,
                              const uint64_t* row_bytes, int nmaps, const int32_t* offsets, int G, int extent,
                              CUtensorMap* out, int* tile_counter, cudaStream_t s);
// dW_r partials: part[S, E, d] = split-K pieces of (dl_hi + dl_lo)^T x; dl halves [T, E] bf16
cudaError_t gemm_router_dw(const uint16_t* dl_hi, const uint16_t* dl_lo, const void* x, int T, int d, int E, int S,
                           float* part, int* status, cudaStream_t s);
// dx_r [T, d] fp16 = (dl_hi + dl_lo) W_r / 2^e, the router's term of the input
// gradient (e from the scale word; NULL: e = 0)
cudaError_t gemm_router_dx(const uint16_t* dl_hi, const uint16_t* dl_lo, const void* W_r, int T, int d, int E,
                           void* dx_r, const uint32_t* scale, int* status, cudaStream_t s);

// MXFP8 expert GEMMs (E4M3 operands, tile-atom E8M0 scales).  A: [rows_total,
// K] codes; rows of group g start at offsets[g] (a multiple of 128, or dense
// G = 1 over rows_total when offsets is NULL) and number counts[g] (NULL: up to
// the next offset).  B: [G][Nb][K] codes, Nb = 2N for the packed gate/up
// weights (64 gate rows, then the 64 up rows of the same h columns), N for
// down.  Out: h codes [rows, N] + their scale atoms (SwiGLU), or fp32 [rows, N].
struct MxGemmArgs {
  const void* a_codes;
  const uint8_t* a_scales;
  int rows_total;
  const int32_t* offsets;
  const int32_t* counts;
  int G, K, N;
  const void* b_codes;
  const uint8_t* b_scales;
  void* out;
  uint8_t* out_scales;
};
cudaError_t gemm_mx_swiglu(const MxGemmArgs& routed, const MxGemmArgs* shared, cudaStream_t s);
cudaError_t gemm_mx_down(const MxGemmArgs& routed, const MxGemmArgs* shared, cudaStream_t s);
// o_perm (o_rows rows), s_out fp16; y bf16
cudaError_t launch_combine_rows(const void* o_perm, const void* s_out, const float* gates,
                                const int32_t* row_of_slot, int T, int d, int k, long long o_rows, void* y,
                                int* status, cudaStream_t s);
// the same with the expert outputs stored by slot: y[t] = s[t] + sum_{kept j}
// g[t,j] o_slot[t*k+j]
cudaError_t launch_combine_slots(const void* o_slot, const void* s_out, const float* gates,
                                 const int32_t* row_of_slot, int T, int d, int k, void* y, int* status,
                                 cudaStream_t s);

// split-K factor used for dW_r
int router_dw_splits(int T, int d, int E);

}  // namespace moe
