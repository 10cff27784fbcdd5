// Forward expert GEMMs: gate/up with the SwiGLU epilogue, and down.
#include "gemm_host.cuh"

namespace moe {
using namespace gemm;

namespace {

constexpr int kPair = 2;  // expert GEMMs run on CTA pairs

bool fill_swiglu_fwd(Params& P, Problem& pr, const SwigluFwdArgs& a) {
  const int ia = new_map(P), ig = new_map(P), iu = new_map(P);
  if (ia < 0 || ig < 0 || iu < 0) return false;
  if (!encode_2d(&P.maps[ia], a.a, a.d, a.rows_total, (uint64_t)a.d * 2, 64, BM)) return false;
  // 64-row boxes: each 64-column h slice takes 64 rows of W_g and 64 of W_u
  if (!encode_3d(&P.maps[ig], a.Wg, a.d, a.H, a.G, 64, 64)) return false;
  if (!encode_3d(&P.maps[iu], a.Wu, a.d, a.H, a.G, 64, 64)) return false;
  pr = blank_problem();
  pr.offsets = a.offsets;
  pr.G = a.G;
  pr.extent = a.rows_total;
  pr.N = a.H;
  pr.K = a.d;
  pr.mma_n = 256;
  pr.n_tile = 128;  // 128 gate + 128 up accumulator columns -> 128 h columns
  pr.half_ok = 1;
  pr.map_a = ia;
  pr.map_b = ig;
  pr.map_b2 = iu;
  pr.tx_bytes = A_BYTES + PairCfg<kPair>::B_BYTES;
  pr.out = a.h;
  pr.ldo = a.H;
  pr.aux = a.au;  // fp32
  pr.ld_aux = 2LL * a.H;
  pr.H = a.H;
  return true;
}

bool fill_down_fwd(Params& P, Problem& pr, const DownFwdArgs& a) {
  const int ia = new_map(P), ib = new_map(P);
  if (ia < 0 || ib < 0) return false;
  if (!encode_2d(&P.maps[ia], a.h, a.H, a.rows_total, (uint64_t)a.H * 2, 64, BM)) return false;
  if (!encode_3d(&P.maps[ib], a.Wd, a.H, a.d, a.G, 64, 256 / kPair)) return false;
  pr = blank_problem();
  pr.offsets = a.offsets;
  pr.G = a.G;
  pr.extent = a.rows_total;
  pr.N = a.d;
  pr.K = a.H;
  pr.mma_n = 256;
  pr.n_tile = 256;
  pr.half_ok = 1;
  pr.map_a = ia;
  pr.map_b = ib;
  pr.tx_bytes = A_BYTES + PairCfg<kPair>::B_BYTES;
  pr.out = a.o;
  pr.ldo = a.d;
  return true;
}

long long mgroup_tile_bound(int rows_total, int G, int N, int n_tile) {
  return ((long long)rows_total / PairCfg<kPair>::TILE_M + G) * cdiv_h(N, n_tile);
}

}  // namespace

cudaError_t gemm_swiglu_fwd(const SwigluFwdArgs& routed, const SwigluFwdArgs* shared, int* status, cudaStream_t s) {
  (void)status;
  Params P;
  std::memset(&P, 0, sizeof(P));
  if (!fill_swiglu_fwd(P, P.prob[0], routed)) return cudaErrorInvalidValue;
  long long bound = mgroup_tile_bound(routed.rows_total, routed.G, routed.H, 128);
  P.num_problems = 1;
  if (shared) {
    if (!fill_swiglu_fwd(P, P.prob[1], *shared)) return cudaErrorInvalidValue;
    bound += mgroup_tile_bound(shared->rows_total, shared->G, shared->H, 128);
    P.num_problems = 2;
  }
  return launch<0, 0, MGROUP, EPI_SWIGLU_FWD, kPair>(P, bound, s,
                                                    routed.h ? "gemm_gate_up_swiglu" : "gemm_gate_up_recompute");
}

cudaError_t gemm_down_fwd(const DownFwdArgs& routed, const DownFwdArgs* shared, int* status, cudaStream_t s) {
  (void)status;
  Params P;
  std::memset(&P, 0, sizeof(P));
  if (!fill_down_fwd(P, P.prob[0], routed)) return cudaErrorInvalidValue;
  long long bound = mgroup_tile_bound(routed.rows_total, routed.G, routed.d, 256);
  P.num_problems = 1;
  if (shared) {
    if (!fill_down_fwd(P, P.prob[1], *shared)) return cudaErrorInvalidValue;
    bound += mgroup_tile_bound(shared->rows_total, shared->G, shared->d, 256);
    P.num_problems = 2;
  }
  return launch<0, 0, MGROUP, EPI_F32, kPair>(P, bound, s, "gemm_down");
}

}  // namespace moe
