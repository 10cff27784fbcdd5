/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE layer with top-k routing and one
 * shared expert: router + top-k gating, token permutation into expert-
 * contiguous order, grouped SwiGLU expert MLP (plus the shared expert), and
 * the gate-weighted unpermute/combine, each with its backward.
 *
 * Sources.  The Olmo-core DDP MoE pages describe the layer this computes:
 *   - "Olmo-core DDP MoE examples" README, "Production throughput runs": top-4
 *     routing, one shared expert, sequence length 8192, random vs learned
 *     routing, BF16;
 *   - same README, "Interpreting the eight-layer DDP vs FSDP comparison":
 *     capacity factor, router, shared-branch mixing and sparse kernels;
 *   - "Olmo-core 3 Opens Large MoE Training", "Technical Deep Dive": experts
 *     stay resident in GPU memory while tokens are routed to them;
 *   - "Scaling Trillion-Parameter Models: The Architecture of Olmo-core 3",
 *     "Code Snippet": a per-token expert-selection step (route_input /
 *     select_expert).
 * The pages give no formulas; each call below states the definition it
 * implements.
 *
 * Conventions (all calls):
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     documented otherwise.  The library never allocates or frees device
 *     memory; scratch space comes from a caller workspace of at least
 *     moe_workspace_size() bytes, 256-byte aligned.  Every call uses its
 *     workspace from the start, so calls that share one workspace must be
 *     ordered on the GPU (one stream, or events between streams); calls on
 *     different workspaces and buffers may run concurrently.  The host side
 *     is thread-safe (per-thread error and timing state, per-device caches
 *     under a lock).
 *   - Tensors are dense and row-major.  "bf16" = IEEE bfloat16 bit patterns
 *     (uint16 storage).  Device pointers of bf16/fp32 tensors must be 16-byte
 *     aligned.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = legacy default stream), performs no host synchronisation and
 *     can be captured in a CUDA graph.
 *   - Kernels are launched with programmatic stream serialization: a kernel
 *     may be scheduled while the kernel before it on the stream retires, and
 *     waits (griddepcontrol.wait) for it to complete before any global
 *     memory access.  Stream order with the caller's own work is unchanged.
 *     No kernel of the library signals its dependents early, so a caller's
 *     kernel launched after one of ours with the same attribute still starts
 *     only once ours has finished; it should itself wait (griddepcontrol.wait)
 *     before reading our outputs, as any programmatically launched kernel
 *     must.
 *   - Return value: MOE_OK, or an error code.  Argument errors are detected
 *     on the host before anything is launched.  MOE_ERR_CUDA reports a launch
 *     failure (moe_last_cuda_error() gives the cudaError_t value).  Device-side
 *     problems (a bounded wait that expired, an index out of range) do not
 *     fault: the kernel records a code in a device status word, skips the bad
 *     access and returns; moe_device_status() reads it.
 *   - Shape limits: 1 <= k <= 8, k <= E <= 256, E % 8 == 0 (rows of fp32/bf16
 *     [T,E] tensors must be 16-byte multiples), d % 64 == 0, H % 128 == 0,
 *     Hs % 128 == 0 (0 = no shared expert), T >= 1, T*k < 2^31.
 *
 * Shapes: T tokens, d model width, E experts, k experts per token, H routed
 * expert hidden width, Hs shared expert hidden width, R = number of kept
 * (token, slot) pairs (R = T*k when dropless), C = capacity (<= 0: dropless).
 *
 * Weight layouts (out_features x in_features):
 *   W_r [E,d]; W_g, W_u [E,H,d]; W_d [E,d,H]; Ws_g, Ws_u [Hs,d]; Ws_d [d,Hs].
 * Buffers sized for the dropless maximum R <= T*k (rows >= R are left as
 * they were): x_perm, dY_perm [T*k, d] bf16; o_perm, dx_perm [T*k, d] fp16;
 * au [T*k, 2H] fp32; h [T*k, H] bf16; slot_of_row [T*k].
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer where one is required, bad size */
  MOE_ERR_UNSUPPORTED = 2,  /* shape outside the limits above */
  MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
  MOE_ERR_TIMEOUT = 5,      /* device status: a bounded wait expired */
  MOE_ERR_DEVICE_BOUNDS = 6, /* device status: an index was out of range */
  MOE_ERR_RANGE = 7          /* device status: a per-token sum (combine, input
                                gradient) was not finite: one of its fp16 terms
                                was beyond the fp16 range (|v| > 65504, stored
                                as inf) or a value upstream was inf / NaN */
};

/* Library version, (major << 16) | minor.  No side effects. */
MOE_API int moe_version(void);

/* Static string for a status code; never NULL. */
MOE_API const char* moe_status_string(int status);

/* cudaError_t of the last failed CUDA call made by this library in the calling
 * thread (0 if none). */
MOE_API int moe_last_cuda_error(void);

/* Reads and clears the device status word of the current device (a blocking
 * copy; call it outside stream capture).  *status_out receives MOE_OK or the
 * first device-side error recorded since the last call. */
MOE_API int moe_device_status(int* status_out);

/* Launch timing, for benchmarks and profiling (no counterpart in the pages).
 * moe_timing_begin: from now on, in the calling thread only, every kernel
 * launch or memset that a call of this library issues is preceded by
 * cudaEventRecord(events[i], stream) for its index i = 0, 1, ... on the
 * launch's own stream; launches past `capacity` are counted, not recorded.
 * events: `capacity` cudaEvent_t handles (passed as void*) created by the
 * caller with timing enabled, owned by the caller, not retained after
 * moe_timing_end.  The caller records one more event after its last call, so
 * launch i took elapsed(events[i], events[i+1]) (queue gaps included).
 * moe_timing_end stops recording and returns the number of launches seen;
 * moe_timing_name(i) is the i-th launch's kernel name (a static string, ""
 * out of range), valid until the next moe_timing_begin in this thread.
 * Inside stream capture the records become event-record nodes of the graph
 * (cudaEventRecordExternal): every replay records the events again, so the
 * launches of one replay are timed after it completes.  A record node
 * between two launches orders them plainly (no programmatic overlap).
 * MOE_ERR_INVALID_ARG: NULL events, a negative capacity, or moe_timing_end
 * without a begin.
 * moe_timing_record: records one caller event on `stream` the same way (an
 * event-record node when the stream is capturing): the closing event after
 * the last call.  MOE_ERR_INVALID_ARG: NULL event; MOE_ERR_CUDA: the record
 * failed. */
MOE_API int moe_timing_begin(void* const* events, int capacity);
MOE_API int moe_timing_end(int* n_launches);
MOE_API const char* moe_timing_name(int i);
MOE_API int moe_timing_record(void* event, void* stream);

/* Workspace bytes needed by every call below for this shape (the maximum
 * over the calls; a single buffer can serve all of them in sequence on one
 * stream).  Host only.  Returns MOE_ERR_UNSUPPORTED for shapes outside the
 * limits. */
MOE_API int moe_workspace_size(int T, int d, int E, int k, int H, int Hs, size_t* bytes);

/* ---------------------------------------------------------------- forward */

/* Router logits, softmax and top-k gating ("top-4 routing", README,
 * "Production throughput runs"; the per-token selection step of "Code
 * Snippet").
 *   learned routing (logits_in == NULL):
 *     logits[t,e] = fp32(sum_c x[t,c] * W_r[e,c]) + bias[e]   (bias may be NULL)
 *     x [T,d] bf16, W_r [E,d] bf16, bias [E] fp32 (16-byte aligned); logits [T,E] fp32 is
 *     written (required).  The product runs on the tensor cores with fp32
 *     accumulation.
 *   given logits (logits_in != NULL, e.g. random routing): logits_in [T,E]
 *     fp32 is used as is; x, W_r, bias and logits are ignored (may be NULL).
 *     -inf entries are allowed.
 *   top-k: the k experts first in the order (logit descending, expert index
 *     ascending); -0.0 equals +0.0.  topk_idx [T,k] int32 in that order.
 *   gates [T,k] fp32: exp(l_s - l_0) / sum_j exp(l_j - l_0) over the selected
 *     logits, i.e. the fp32 softmax renormalised over the top-k.
 * NaN logits are not supported. */
MOE_API int moe_route_topk(const void* x, const void* W_r, const float* bias, const float* logits_in,
                   int T, int d, int E, int k,
                   float* logits, int32_t* topk_idx, float* gates,
                   void* ws, size_t ws_bytes, void* stream);

/* Token permutation into expert-contiguous order: per-expert histogram,
 * capacity clamp, exclusive prefix sum, stable scatter (tokens stay resident
 * experts are fed by routing, "Technical Deep Dive"; capacity factor, README
 * "Interpreting the eight-layer DDP vs FSDP comparison").
 *   rank(t,s)      = #{t' < t : topk_idx[t,s] is among t''s experts}
 *   kept(t,s)      = capacity <= 0 || rank(t,s) < capacity
 *   counts_raw[e]  = #{(t,s) : topk_idx[t,s] == e}            [E] int32
 *   counts[e]      = #kept pairs of e = min(counts_raw[e], capacity)  [E]
 *   offsets[e]     = sum_{e' < e} counts[e'];  offsets[E] = R   [E+1] int32
 *   row_of_slot[t*k+s] = offsets[e] + rank(t,s) if kept, else -1   [T*k]
 *   slot_of_row[row]   = t*k+s for every kept pair (rows [0,R))     [T*k]
 *   x_perm[row, :]     = x[t, :]                                  [T*k, d] bf16
 * x_perm == NULL: the maps only (x may be NULL too), for the fused path
 * (moe_grouped_swiglu_fused), whose GEMMs gather the rows of x themselves.
 * Deterministic (no order-dependent atomics): the results are bit-exact. */
MOE_API int moe_permute(const void* x, const int32_t* topk_idx, int T, int d, int E, int k, int capacity,
                int32_t* counts_raw, int32_t* counts, int32_t* offsets,
                int32_t* row_of_slot, int32_t* slot_of_row, void* x_perm,
                void* ws, size_t ws_bytes, void* stream);

/* moe_permute without a workspace (no counterpart in the pages: it exists
 * for callers, not for the method).  Same arguments, results and determinism
 * as moe_permute, minus ws / ws_bytes.
 *
 * Who needs it: callers that cannot allocate device memory for scratch --
 * plug-in hosts that give a library nothing but their own tensors and a
 * stream, and processes whose device memory is entirely held by a framework
 * pool, where one more cudaMalloc would fail or fragment that pool.  Nothing
 * is allocated by this call or by the library on its behalf.
 *
 * Scratch: a fixed 4 MiB array inside the library, present on every GPU that
 * loads the library until the process exits.  Shapes whose scratch
 * (per-tile counts and bases, ceil(T/128) x E ints each, plus T*k in-tile
 * ranks) exceeds 4 MiB are rejected with MOE_ERR_UNSUPPORTED before anything
 * runs -- e.g. T*k up to about 512K slots at E = 64 fits.
 * The first call on a device looks up that array's device address (once per
 * device, with the device current); make that first call outside any stream
 * capture.  All calls on a device share the array: calls whose kernels can
 * overlap on the GPU (different streams without ordering) race and must be
 * serialised by the caller.  The array keeps the previous call's contents;
 * no part of it has to start at zero. */
MOE_API int moe_permute_static(const void* x, const int32_t* topk_idx, int T, int d, int E, int k,
                       int capacity, int32_t* counts_raw, int32_t* counts, int32_t* offsets,
                       int32_t* row_of_slot, int32_t* slot_of_row, void* x_perm, void* stream);

/* Grouped SwiGLU expert MLP over the ragged per-expert row segments plus the
 * shared expert ("one shared expert", README "Production throughput runs";
 * "sparse kernels", "Interpreting the eight-layer ..."):
 *   rows [offsets[e], offsets[e+1]) of x_perm go through expert e:
 *     a = x W_g[e]^T, u = x W_u[e]^T (fp32 accumulate), h = silu(a) * u,
 *     o = h W_d[e]^T;   silu(a) = a / (1 + exp(-a)).
 *   au [T*k, 2H] FP32 receives a in columns [0,H) and u in [H,2H), kept for
 *   the backward pass (may be NULL when no backward follows);
 *   h [T*k, H] bf16 (the down projection's input, required);
 *   o_perm [T*k, d] FP16: the terms of the combine's per-token sum.  fp16
 *   carries 11 significant bits where bf16 carries 8: with bf16 terms the
 *   summed y reaches the edge of the parity bound at d = 4096 (their
 *   rounding adds up where the terms cancel), with fp16 it stays where fp32
 *   terms leave it.  A term beyond the fp16 range (|v| > 65504) is stored
 *   as inf; the combine then records MOE_ERR_RANGE in the device status.
 *   Shared expert (Hs > 0): the same on every token of x [T,d] with Ws_*,
 *   writing au_s [T,2Hs] fp32 (nullable), h_s [T,Hs] bf16 and s [T,d] fp16.
 *   Hs == 0: the shared pointers are ignored.
 * Tensor-core (tcgen05) grouped GEMMs fed by TMA; the per-expert tile
 * schedule is read from `offsets` on the device.  ws is unused (may be NULL). */
MOE_API int moe_grouped_swiglu(const void* x_perm, const int32_t* offsets, const void* x,
                       int T, int d, int E, int k, int H, int Hs,
                       const void* W_g, const void* W_u, const void* W_d,
                       const void* Ws_g, const void* Ws_u, const void* Ws_d,
                       float* au, void* h, void* o_perm,
                       float* au_s, void* h_s, void* s,
                       void* ws, size_t ws_bytes, void* stream);

/* Activation recompute for the backward ("Olmo-core DDP MoE examples"
 * README: the per-layer recompute of the largest "Production throughput
 * runs" and the per-block recompute benchmark of "Other experiments in the
 * report"; the pages name the option only): a forward run with au = au_s =
 * NULL keeps no fp32 a | u, and this call rebuilds them, just before
 * moe_grouped_swiglu_bwd, from the same inputs:
 *   au[r, 0:H]  = x_perm[r] W_g[e]^T,  au[r, H:2H] = x_perm[r] W_u[e]^T
 *   au_s        = the same for x and Ws_g, Ws_u (when Hs > 0)
 * It is the forward's gate/up GEMM with h left unstored, so the values are
 * bit-identical to the ones moe_grouped_swiglu would have saved.  au
 * [T*k, 2H] and au_s [T, 2Hs] fp32 are outputs (scratch that only has to
 * live until the backward call has consumed it); other arguments as for
 * moe_grouped_swiglu.  Rows past offsets[E] are not written. */
MOE_API int moe_grouped_swiglu_recompute(const void* x_perm, const int32_t* offsets, const void* x,
                                 int T, int d, int E, int k, int H, int Hs,
                                 const void* W_g, const void* W_u, const void* Ws_g, const void* Ws_u,
                                 float* au, float* au_s, void* stream);

/* The expert MLP with the permutation and the combine fused into the GEMMs
 * (tokens stay where they are and the experts read them: "Olmo-core 3 Opens
 * Large MoE Training", "Technical Deep Dive"; the combine of "Production
 * throughput runs" of the "Olmo-core DDP MoE examples" README).  Same values
 * as moe_permute (rows) + moe_grouped_swiglu + moe_unpermute_combine, without
 * x_perm, o_perm or s in memory:
 *   - the routed gate/up GEMM loads its A rows straight from x: permuted row
 *     r is token slot_of_row[r] / k, copied 16 bytes per thread (cp.async)
 *     into the tile's swizzled layout; the gathering GEMMs run on single CTAs
 *     (128-row tiles);
 *   - the routed down projection stores row r's output at its slot:
 *     o_slot[slot_of_row[r]] ([T*k, d] fp16; rows of dropped slots are not
 *     written);
 *   - the shared expert's down projection (a second launch on the stream)
 *     adds, in its epilogue, the gate-weighted kept slots of each token in
 *     slot order to its accumulator s[t] (rounded through fp16, as the
 *     unfused path stores s) and writes y[t] in bf16 once:
 *       y[t] = bf16(s[t] + sum_{j kept} gates[t,j] o_slot[t*k+j])
 *     -- the same operations in the same order as moe_unpermute_combine, so y
 *     is bit-identical to the unfused path's.  Hs == 0: a combine pass over
 *     o_slot.
 * slot_of_row, row_of_slot and offsets come from moe_permute (x_perm may be
 * NULL there); au, h, au_s, h_s as for moe_grouped_swiglu (h and au in
 * permuted row order, for the backward).
 * Speed: on GB300 this path is slower than the unfused one -- per-row
 * gathers (cp.async, or TMA tile::gather4) do not reach the rate of the
 * tiled TMA loads that read x_perm -- so the unfused sequence is the fast
 * one; this call exists for callers that cannot hold x_perm / o_perm. */
MOE_API int moe_grouped_swiglu_fused(const void* x, const int32_t* slot_of_row, const int32_t* row_of_slot,
                                     const float* gates, const int32_t* offsets, int T, int d, int E, int k, int H,
                                     int Hs, const void* W_g, const void* W_u, const void* W_d, const void* Ws_g,
                                     const void* Ws_u, const void* Ws_d, float* au, void* h, void* o_slot,
                                     float* au_s, void* h_s, void* y, void* stream);

/* moe_grouped_swiglu_recompute for the fused path: the routed rows are
 * gathered from x by slot_of_row (no x_perm).  Bit-identical to the a | u
 * that moe_grouped_swiglu_fused would have saved. */
MOE_API int moe_grouped_swiglu_recompute_fused(const void* x, const int32_t* slot_of_row, const int32_t* offsets,
                                               int T, int d, int E, int k, int H, int Hs, const void* W_g,
                                               const void* W_u, const void* Ws_g, const void* Ws_u, float* au,
                                               float* au_s, void* stream);

/* Gate-weighted unpermute and combine:
 *   y[t,:] = s[t,:] + sum_{s kept} gates[t,s] * o_perm[row_of_slot[t*k+s], :]
 * o_perm [T*k,d] and s [T,d] fp16 (s may be NULL: no shared expert); fp32
 * accumulation in slot order, one bf16 rounding: y [T,d] bf16.  A
 * non-finite sum records MOE_ERR_RANGE in the device status. */
MOE_API int moe_unpermute_combine(const void* o_perm, const void* s, const float* gates,
                          const int32_t* row_of_slot, int T, int d, int k,
                          void* y, void* stream);

/* Self-check of the device-side tensor-map patching that the weight-gradient
 * GEMMs use (each expert's rows are read through maps re-based on the device
 * from the offsets): builds the per-group maps of two operands for an offsets
 * table with empty, one-row and ragged groups and compares each map byte for
 * byte with the map the CUDA driver's encoder gives for the same sub-matrix.  No
 * tensor copy runs.  Returns MOE_OK, or MOE_ERR_UNSUPPORTED if a map differs.
 * Allocates and frees its own scratch and synchronizes the device. */
MOE_API int moe_selftest_group_maps(void);

/* Self-check of the failure detection: one warp waits, through the bounded
 * wait every GEMM uses, on an mbarrier phase that nothing completes, for
 * limit_us microseconds (1 .. 2,000,000).  The wait then gives up and the
 * kernel records MOE_ERR_TIMEOUT in the device status word (read and cleared
 * by moe_device_status()) and returns: no trap, no fault, the context stays
 * usable.  Asynchronous on `stream`; returns MOE_ERR_INVALID_ARG for a limit
 * out of range. */
MOE_API int moe_selftest_wait_timeout(int limit_us, void* stream);

/* --------------------------------------------------------------- backward */

/* Backward of moe_unpermute_combine, first half: the upstream gradient of
 * every token is gathered into its kept rows,
 *   dY_perm[row_of_slot[t*k+s], :] = dY[t, :]      (bit copies, bf16)
 * The other two factors of the combine backward -- dO_perm = gates * dY_perm
 * and dgates[t,s] = <dY[t], o_perm[row]> -- are formed inside
 * moe_grouped_swiglu_bwd, from fp32 accumulators (dgates = <dY W_d, h>, the
 * same quantity), so that neither the gate factor nor the rounding of o_perm
 * to bf16 limits their precision.  The gradient reaching the shared expert's
 * output is dY itself. */
MOE_API int moe_unpermute_combine_bwd(const void* dY, const int32_t* row_of_slot, int T, int d, int k,
                              void* dY_perm, void* stream);

/* Backward of moe_grouped_swiglu and of the gate factor of the combine.
 * Inputs: dY_perm [T*k,d] (from moe_unpermute_combine_bwd), dY [T,d] (the
 * shared expert's upstream gradient; ignored if Hs == 0), gates [T,k],
 * row_of_slot, slot_of_row, offsets, x_perm, x and the fp32 au (au_s) saved by
 * the forward call.  For each kept row r of expert e, with g = gates of its
 * slot and a, u from au:
 *   dh' = dY_perm[r] W_d[e]          (fp32 accumulate)
 *   dgates[slot] = sum_j dh'_j h_j,  h = silu(a) u   (= <dY, o_perm[r]>)
 *   dh = g dh';  da = dh * u * sig(a) * (1 + a (1 - sig(a)));  du = dh * silu(a)
 *   dx_perm[r] = da W_g[e] + du W_u[e]
 *   dW_d[e] = sum_r dY_perm[r]^T (g h_r);  dW_g[e] = sum_r da_r^T x_perm[r];
 *   dW_u[e] = sum_r du_r^T x_perm[r]
 * and the same for the shared expert over all T tokens with g = 1 (no gate
 * gradient).  The products take their derived operand (g h, da | du) as a
 * bf16 hi + lo pair, so the result keeps ~16 bits over sums of thousands of
 * rows (weight gradients) or of 2H products (input gradients).  Outputs: dx_perm [T*k,d] and dx_s [T,d] in fp16 (the
 * terms of moe_permute_bwd's per-token sum, as o_perm for the combine; a
 * term beyond the fp16 range makes that sum report MOE_ERR_RANGE), dW_g,
 * dW_u [E,H,d],
 * dW_d [E,d,H] (zero for experts with no rows), dWs_g, dWs_u [Hs,d],
 * dWs_d [d,Hs] (all bf16) and dgates [T,k] fp32 (0 for dropped slots).  Each
 * output element is owned by one tile: no atomics, deterministic.
 * Fused path: dY_perm == x_perm == NULL (both or neither) -- the dgrad of
 * the down projection and the two weight gradients then read the rows of dY
 * and x themselves through slot_of_row (16-byte cp.async row copies; the
 * permutation fused into their operand loads, no moe_unpermute_combine_bwd
 * call needed; slower than the permuted copies on GB300);
 * dY and x are required.  Same results as with the permuted copies.
 * dx_scale (nullable; requires dY): a device uint32 scale word.  The call
 * writes into it the largest bf16 magnitude of dY (the bit pattern of
 * max |dY|), whose power of two 2^e (e = floor(log2 max|dY|), 0 for a zero
 * or non-finite dY) then divides dx_perm and dx_s: the fp16 terms sit where
 * they sit for gradients of order one whatever the gradient's own scale (a
 * loss averaged over many tokens gives |dY| far below fp16's normal range),
 * and moe_permute_bwd, given the same word, multiplies the sum by 2^e.
 * Both scalings are exact; NULL: the terms are stored unscaled.
 * ws >= moe_workspace_size() bytes. */
MOE_API int moe_grouped_swiglu_bwd(const void* dY_perm, const void* dY, const float* gates,
                           const int32_t* row_of_slot, const int32_t* slot_of_row,
                           const int32_t* offsets, const void* x_perm, const void* x,
                           const float* au, const float* au_s,
                           int T, int d, int E, int k, int H, int Hs,
                           const void* W_g, const void* W_u, const void* W_d,
                           const void* Ws_g, const void* Ws_u, const void* Ws_d,
                           void* dx_perm, void* dx_s,
                           void* dW_g, void* dW_u, void* dW_d,
                           void* dWs_g, void* dWs_u, void* dWs_d,
                           float* dgates, uint32_t* dx_scale, void* ws, size_t ws_bytes, void* stream);

/* Backward of the top-k softmax gating and of the router product:
 *   dlogits[t,e] = g_s (dgates[t,s] - sum_j g_j dgates[t,j]) if e = topk_idx[t,s],
 *                  0 for experts not selected by t
 *                  + dlogits_add[t,e] if dlogits_add != NULL   [T,E] fp32
 *   dW_r[e,c]    = sum_t dlogits[t,e] x[t,c]                   [E,d] fp32
 * (dropped slots have dgates = 0 but stay in the renormalisation set).  x may
 * be NULL only together with dW_r == NULL (given-logits routing).
 * dlogits_add (nullable, [T,E] fp32, device) is a further gradient of the
 * logits to include, e.g. that of moe_router_balance_loss, so that dW_r and
 * (through moe_permute_bwd) dx carry it.  dW_r uses the tensor cores with
 * dlogits as a bf16 hi + lo pair and fp32 accumulation. */
MOE_API int moe_route_topk_bwd(const float* dgates, const float* gates, const int32_t* topk_idx,
                       const void* x, int T, int d, int E, int k,
                       float* dlogits, float* dW_r, const float* dlogits_add,
                       void* ws, size_t ws_bytes, void* stream);

/* Auxiliary load-balancing loss of the router ("Olmo-core DDP MoE examples"
 * README, "Other experiments in the report": the load-balancing-loss weight
 * runs, weights 0.02 to 0.5; the pages give no formula, the usual loss of
 * top-k routing is taken):
 *   f_e  = counts_raw[e] / (T k)        share of the router assignments of
 *                                       expert e, before any capacity drop
 *   P_e  = (1/T) sum_t softmax(logits[t,:])_e   mean full-softmax probability
 *   loss = alpha E sum_e f_e P_e                device fp32 scalar
 *   dlogits_lbl[t,j] = alpha E / T p[t,j] (f_j - sum_e f_e p[t,e])
 *                      (f is piecewise constant in the logits)  [T,E] fp32
 * logits [T,E] fp32 are the logits the top-k ran on (bias included; -inf
 * allowed); counts_raw [E] int32 from moe_permute.  P_mean [E] and
 * dlogits_lbl may be NULL.  Pass dlogits_lbl to moe_route_topk_bwd as
 * dlogits_add to back-propagate the loss.  One pass over the logits (one
 * kernel after a 4-byte memset); fixed-order reductions: deterministic.
 * ws >= moe_workspace_size() bytes. */
MOE_API int moe_router_balance_loss(const float* logits, const int32_t* counts_raw, int T, int E, int k,
                                    float alpha, float* loss, float* P_mean, float* dlogits_lbl,
                                    void* ws, size_t ws_bytes, void* stream);

/* Backward of the permutation (gather-reduce) plus the router's input
 * gradient:
 *   dx[t,:] = sum_{s kept} dx_perm[row_of_slot[t*k+s], :] + dx_s[t,:]
 *             + sum_e dlogits[t,e] W_r[e,:]
 * dx_perm [T*k,d] and dx_s [T,d] fp16 (from moe_grouped_swiglu_bwd); fp32
 * accumulation, one bf16 rounding: dx [T,d] bf16 (a non-finite sum records
 * MOE_ERR_RANGE).  dx_s may be NULL (no
 * shared expert); dlogits and W_r may both be NULL (given-logits routing).
 * The router term uses the tensor cores with dlogits as a bf16 hi + lo pair
 * and enters the sum as an fp16 term.  dx_scale (nullable): the scale word
 * moe_grouped_swiglu_bwd wrote when it produced dx_perm and dx_s; the router
 * term is stored divided by the same 2^e and the sum multiplied by 2^e
 * (NULL: e = 0, unscaled terms). */
MOE_API int moe_permute_bwd(const void* dx_perm, const void* dx_s, const int32_t* row_of_slot,
                    const float* dlogits, const void* W_r,
                    int T, int d, int E, int k, void* dx, const uint32_t* dx_scale,
                    void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------- MXFP8 */

/* MXFP8 expert MLP ("Olmo-core DDP MoE examples" README: the MXFP8 rows of
 * "Production throughput runs" and the MXFP8 recipe of "Other experiments in
 * the report"; the pages name the precision only).  Format: the OCP
 * microscaling format with FP8 E4M3 elements: every 32 consecutive values
 * along the contraction dimension share one power-of-two scale
 * X = 2^(floor(log2 max|v|) - 8) (E8M0 byte = exponent + 127; 2^-127 for an
 * all-zero block), and code = E4M3(v / X) rounded to nearest (ties to even),
 * saturating at +-448.
 *
 * Layouts.  Codes: one byte per element, row-major.  Scales ("tile atoms"):
 * the scales of rows [128 t, 128 t + 128) and 32-value blocks [4 q, 4 q + 4)
 * of a [rows, cols] matrix form one 512-byte atom at byte (t * cols/128 + q)
 * * 512; in it the scale of row 128 t + 32 j + l, block 4 q + b is byte
 * 16 l + 4 j + b.  moe_mxfp8_scales_bytes gives an array's size (rows rounded
 * up to 128).  Padded row space: the MX permutation places expert e's rows
 * from mx_offsets[e], a multiple of 128 (mx_offsets = exclusive prefix sum of
 * the counts rounded up to 128), in buffers of moe_mxfp8_rows(T, E, k) rows.
 * Shape limits: those of the bf16 path and d % 128 == 0. */

/* *rows = rows of the padded row space: T*k + 127*E rounded up to 128. */
MOE_API int moe_mxfp8_rows(int T, int E, int k, long long* rows);

/* *bytes = size of the tile-atom scale array of a [rows, cols] matrix
 * (cols % 128 == 0). */
MOE_API int moe_mxfp8_scales_bytes(long long rows, int cols, size_t* bytes);

/* Quantize bf16 rows: src [rows, cols] bf16 -> codes [rows, cols] E4M3 and
 * scales (tile atoms), blocks of 32 along each row.  For the weights of the
 * down projection (W_d [E, d, H] as E*d rows of H), of the shared expert and
 * for x (the shared expert's input, T rows of d).  Asynchronous. */
MOE_API int moe_mxfp8_quantize(const void* src, long long rows, int cols, void* codes, void* scales,
                               void* stream);

/* Quantize the gate and up weights W_g, W_u [E, H, d] into one packed matrix
 * [E, 2H, d] of codes (blocks of 32 along d) and its scales: for every 64
 * h-columns j (rows [128 j', 128 j' + 128) of expert e's 2H rows) the 64 rows
 * of W_g, then the 64 rows of W_u of the same h columns, so that one 128-row
 * tile of the packed matrix yields 64 columns of a and of u.  E = 1 with the
 * shared weights [Hs, d] packs those. */
MOE_API int moe_mxfp8_quantize_gate_up(const void* W_g, const void* W_u, int E, int H, int d, void* codes,
                                       void* scales, void* stream);

/* moe_permute with x_perm in MXFP8 and the rows in the padded row space:
 * counts_raw, counts, offsets as moe_permute (bit-exact, unpadded); mx_offsets
 * [E+1] the padded offsets; row_of_slot [T*k] (-1 dropped) and slot_of_row
 * [moe_mxfp8_rows] in padded rows; x_codes [moe_mxfp8_rows, d] and x_scales
 * (tile atoms of that many rows): the codes and scales of x[t], quantized once
 * per token along d, in every kept row of t.  Rows of the padding are not
 * written.  ws as for moe_permute. */
MOE_API int moe_permute_mxfp8(const void* x, const int32_t* topk_idx, int T, int d, int E, int k, int capacity,
                              int32_t* counts_raw, int32_t* counts, int32_t* offsets, int32_t* mx_offsets,
                              int32_t* row_of_slot, int32_t* slot_of_row, void* x_codes, void* x_scales,
                              void* ws, size_t ws_bytes, void* stream);

/* The expert MLP on MXFP8 operands, plus the shared expert: per kept row r of
 * expert e (rows [mx_offsets[e], mx_offsets[e] + counts[e]) of the padded
 * space),
 *   a = MX(x) MX(W_g[e])^T, u = MX(x) MX(W_u[e])^T   (fp32 accumulate)
 *   h = silu(a) u, quantized along H (blocks of 32) into h_codes / h_scales
 *   o = MX(h) MX(W_d[e])^T  -> o_perm [moe_mxfp8_rows, d] fp16
 * and the same on every token with the shared weights (xs = MX(x) from
 * moe_mxfp8_quantize, h_s -> hs_codes [T, Hs] / hs_scales, s [T, d] fp16:
 * o and s are the combine's sum terms, as in moe_grouped_swiglu).
 * Wgu: the packed gate/up codes and scales (moe_mxfp8_quantize_gate_up);
 * Wd: W_d quantized as E*d rows of H.  The products run on the tensor cores
 * as block-scaled E4M3 MMAs (tcgen05 kind::mxf8f6f4, E8M0 scales in tensor
 * memory).  Rows of the padding are not written. */
MOE_API int moe_grouped_swiglu_mxfp8(const void* x_codes, const void* x_scales, const int32_t* mx_offsets,
                                     const int32_t* counts, const void* xs_codes, const void* xs_scales, int T,
                                     int d, int E, int k, int H, int Hs, const void* Wgu_codes,
                                     const void* Wgu_scales, const void* Wd_codes, const void* Wd_scales,
                                     const void* Wsgu_codes, const void* Wsgu_scales, const void* Wsd_codes,
                                     const void* Wsd_scales, void* h_codes, void* h_scales, void* hs_codes,
                                     void* hs_scales, void* o_perm, void* s, void* stream);

/* moe_unpermute_combine for o_perm in the padded row space of the MXFP8
 * path (moe_mxfp8_rows(T, E, k) rows; row_of_slot from moe_permute_mxfp8). */
MOE_API int moe_unpermute_combine_mxfp8(const void* o_perm, const void* s, const float* gates,
                                        const int32_t* row_of_slot, int T, int d, int E, int k, void* y,
                                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
