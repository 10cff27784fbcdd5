// Router GEMMs: logits = x W_r^T + b (forward), dW_r split-K partials and the
// router's input gradient (backward).
#include "gemm_host.cuh"

namespace moe {
using namespace gemm;

cudaError_t gemm_router_fwd(const void* x, const void* W_r, const float* bias, int T, int d, int E, float* logits,
                            int* status, cudaStream_t s) {
  (void)status;
  Params P;
  std::memset(&P, 0, sizeof(P));
  const int nB = (E + 15) / 16 * 16;
  P.num_maps = 2;
  if (!encode_2d(&P.maps[0], x, d, T, (uint64_t)d * 2, 64, BM)) return cudaErrorInvalidValue;
  if (!encode_3d(&P.maps[1], W_r, d, E, 1, 64, nB)) return cudaErrorInvalidValue;
  Problem& pr = P.prob[0];
  pr = blank_problem();
  pr.G = 1;
  pr.extent = T;
  pr.N = E;
  pr.K = d;
  pr.mma_n = nB;
  pr.n_tile = 256;
  pr.map_a = 0;
  pr.map_b = 1;
  pr.tx_bytes = A_BYTES + nB * BK * 2;
  pr.out = logits;
  pr.ldo = E;
  pr.bias = bias;
  P.num_problems = 1;
  return launch<0, 0, MGROUP, EPI_F32, 1>(P, cdiv_h(T, BM), s, "gemm_router");
}

int router_dw_splits(int T, int d, int E) {
  (void)d;
  (void)E;
  int S = T / 512;
  if (S < 1) S = 1;
  if (S > 64) S = 64;
  return S;
}

cudaError_t gemm_router_dw(const uint16_t* dl_hi, const uint16_t* dl_lo, const void* x, int T, int d, int E, int S,
                           float* part, int* status, cudaStream_t s) {
  (void)status;
  Params P;
  std::memset(&P, 0, sizeof(P));
  P.num_maps = 3;
  constexpr int bkk = kg_rows(SPLIT_A);  // K rows (tokens) per stage
  if (!encode_2d(&P.maps[0], dl_hi, E, T, (uint64_t)E * 2, 64, bkk)) return cudaErrorInvalidValue;
  if (!encode_2d(&P.maps[1], x, d, T, (uint64_t)d * 2, 64, bkk)) return cudaErrorInvalidValue;
  if (!encode_2d(&P.maps[2], dl_lo, E, T, (uint64_t)E * 2, 64, bkk)) return cudaErrorInvalidValue;
  Problem& pr = P.prob[0];
  pr = blank_problem();
  pr.map_a_lo = 2;
  pr.nsplit = 2;
  pr.G = S;
  pr.extent = T;
  pr.M = E;
  pr.N = d;
  pr.mma_n = 256;
  pr.n_tile = 256;
  pr.map_a = 0;
  pr.map_b = 1;
  pr.tx_bytes = (2 + 4 + 2) * 64 * bkk * 2;  // A, B, lo half of A
  pr.out = part;
  pr.ldo = d;
  pr.gstride = (long long)E * d;
  P.num_problems = 1;
  return launch<1, 1, KGROUP, EPI_F32, 1, SPLIT_A>(P, (long long)S * cdiv_h(E, BM) * cdiv_h(d, 256), s,
                                                  "gemm_router_dw");
}

cudaError_t gemm_router_dx(const uint16_t* dl_hi, const uint16_t* dl_lo, const void* W_r, int T, int d, int E,
                           void* dx_r, const uint32_t* scale, int* status, cudaStream_t s) {
  (void)status;
  Params P;
  std::memset(&P, 0, sizeof(P));
  P.num_maps = 3;
  if (!encode_2d(&P.maps[0], dl_hi, E, T, (uint64_t)E * 2, 64, BM)) return cudaErrorInvalidValue;
  if (!encode_3d(&P.maps[1], W_r, d, E, 1, 64, 64)) return cudaErrorInvalidValue;
  if (!encode_2d(&P.maps[2], dl_lo, E, T, (uint64_t)E * 2, 64, BM)) return cudaErrorInvalidValue;
  Problem& pr = P.prob[0];
  pr = blank_problem();
  pr.map_a_lo = 2;
  pr.nsplit = 2;
  pr.G = 1;
  pr.extent = T;
  pr.N = d;
  pr.K = E;
  pr.mma_n = 256;
  pr.n_tile = 256;
  pr.map_a = 0;
  pr.map_b = 1;
  pr.tx_bytes = A_BYTES + 4 * MN_BLOCK_BYTES;
  pr.out = dx_r;
  pr.out_f16 = 1;  // fp16 term of the unpermute's sum
  pr.out_scale = scale;
  pr.ldo = d;
  P.num_problems = 1;
  return launch<0, 1, MGROUP, EPI_F32, 1>(P, (long long)cdiv_h(T, BM) * cdiv_h(d, 256), s, "gemm_router_dx");
}

}  // namespace moe
