// MXFP8 expert GEMMs: gate/up with the SwiGLU epilogue that quantizes h, and
// down with fp16 rows out (terms of the combine's sum), on block-scaled E4M3 operands (tcgen05
// kind::mxf8f6f4 with E8M0 scales in tensor memory).
#include "gemm_host.cuh"

namespace moe {
using namespace gemm;

namespace {

bool fill_mx(Params& P, Problem& pr, const MxGemmArgs& a, bool swiglu) {
  const int ia = new_map(P), ib = new_map(P);
  if (ia < 0 || ib < 0) return false;
  const int Nb = swiglu ? 2 * a.N : a.N;  // rows of B per group (packed gate/up: 2H)
  if (!encode_u8_2d(&P.maps[ia], a.a_codes, a.K, a.rows_total)) return false;
  if (!encode_u8_3d(&P.maps[ib], a.b_codes, a.K, Nb, a.G)) return false;
  pr = blank_problem();
  pr.offsets = a.offsets;
  pr.counts = a.counts;
  pr.G = a.G;
  pr.extent = a.rows_total;
  pr.N = a.N;
  pr.K = a.K;
  pr.mma_n = MX_N;
  pr.n_tile = swiglu ? MX_N / 2 : MX_N;  // SwiGLU: 64 gate + 64 up columns -> 64 h columns
  pr.map_a = ia;
  pr.map_b = ib;
  pr.tx_bytes = A_BYTES + MX_B_BYTES + MX_SF_BYTES;
  pr.sfa = a.a_scales;
  pr.sfb = a.b_scales;
  pr.nkq = a.K / 128;
  pr.sfb_gstride = (long long)(Nb / 128) * pr.nkq * 512;
  pr.out = a.out;
  pr.out_f16 = swiglu ? 0 : 1;  // down: fp16 terms of the combine's sum
  pr.ldo = a.N;
  pr.out_sf = a.out_scales;
  pr.out_sf_nq = a.N / 128;
  return true;
}

long long tile_bound(const MxGemmArgs& a, int n_tile) {
  return ((long long)a.rows_total / BM + a.G) * cdiv_h(a.N, n_tile);
}

}  // namespace

cudaError_t gemm_mx_swiglu(const MxGemmArgs& routed, const MxGemmArgs* shared, cudaStream_t s) {
  Params P;
  std::memset(&P, 0, sizeof(P));
  if (!fill_mx(P, P.prob[0], routed, true)) return cudaErrorInvalidValue;
  long long bound = tile_bound(routed, MX_N / 2);
  P.num_problems = 1;
  if (shared) {
    if (!fill_mx(P, P.prob[1], *shared, true)) return cudaErrorInvalidValue;
    bound += tile_bound(*shared, MX_N / 2);
    P.num_problems = 2;
  }
  return launch<0, 0, MGROUP, EPI_SWIGLU_FWD, 1, SPLIT_NONE, 1>(P, bound, s, "gemm_mx_gate_up_swiglu");
}

cudaError_t gemm_mx_down(const MxGemmArgs& routed, const MxGemmArgs* shared, cudaStream_t s) {
  Params P;
  std::memset(&P, 0, sizeof(P));
  if (!fill_mx(P, P.prob[0], routed, false)) return cudaErrorInvalidValue;
  long long bound = tile_bound(routed, MX_N);
  P.num_problems = 1;
  if (shared) {
    if (!fill_mx(P, P.prob[1], *shared, false)) return cudaErrorInvalidValue;
    bound += tile_bound(*shared, MX_N);
    P.num_problems = 2;
  }
  return launch<0, 0, MGROUP, EPI_F32, 1, SPLIT_NONE, 1>(P, bound, s, "gemm_mx_down");
}

}  // namespace moe
