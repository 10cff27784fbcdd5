// Forward expert GEMMs: gate/up with the SwiGLU epilogue, and down.
#include "gemm_host.cuh"

namespace moe {
using namespace gemm;

namespace {

constexpr int kPair = 2;  // expert GEMMs run on CTA pairs (single CTAs when a row gather feeds A)

// B bytes per CTA and stage, rows per tile
int b_bytes(int pair) { return pair == 2 ? PairCfg<2>::B_BYTES : PairCfg<1>::B_BYTES; }

bool fill_swiglu_fwd(Params& P, Problem& pr, const SwigluFwdArgs& a, int pair) {
  const int ia = new_map(P), ig = new_map(P), iu = new_map(P);
  if (ia < 0 || ig < 0 || iu < 0) return false;
  const bool gat = a.gather.src != nullptr;
  // with a row gather the tiled A map (not loaded from) covers the source
  if (!encode_2d(&P.maps[ia], gat ? a.gather.src : a.a, a.d, gat ? a.gather.src_rows : a.rows_total,
                 (uint64_t)a.d * 2, 64, BM))
    return false;
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
  pr.tx_bytes = (gat ? 0 : A_BYTES) + b_bytes(pair);  // gathered A rows arrive by cp.async
  pr.out = a.h;
  pr.ldo = a.H;
  pr.aux = a.au;  // fp32
  pr.ld_aux = 2LL * a.H;
  pr.H = a.H;
  if (gat && !set_gather(pr, 0, a.gather.src, a.d, a.gather.slot_of_row, a.gather.k, a.gather.nslots)) return false;
  return true;
}

bool fill_down_fwd(Params& P, Problem& pr, const DownFwdArgs& a) {
  const int pair = kPair;
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
  pr.tx_bytes = A_BYTES + b_bytes(pair);
  pr.out = a.o;
  pr.out_f16 = 1;  // expert / shared outputs: fp16 terms of the combine's sum
  pr.ldo = a.d;
  pr.out_row_map = a.out_row_map;
  pr.out_map_rows = a.out_map_rows;
  pr.comb_o = a.comb_o;
  pr.comb_gates = a.comb_gates;
  pr.comb_row_of_slot = a.comb_row_of_slot;
  pr.comb_k = a.comb_k;
  pr.comb_y = a.comb_y;
  return true;
}

long long mgroup_tile_bound(int rows_total, int G, int N, int n_tile, int pair = kPair) {
  return ((long long)rows_total / (BM * pair) + G) * cdiv_h(N, n_tile);
}

}  // namespace

cudaError_t gemm_swiglu_fwd(const SwigluFwdArgs& routed, const SwigluFwdArgs* shared, int* status, cudaStream_t s) {
  (void)status;
  Params P;
  std::memset(&P, 0, sizeof(P));
  const int pair = routed.gather.src ? 1 : kPair;
  if (shared && shared->gather.src) return cudaErrorInvalidValue;
  if (!fill_swiglu_fwd(P, P.prob[0], routed, pair)) return cudaErrorInvalidValue;
  long long bound = mgroup_tile_bound(routed.rows_total, routed.G, routed.H, 128, pair);
  P.num_problems = 1;
  if (shared) {
    if (!fill_swiglu_fwd(P, P.prob[1], *shared, pair)) return cudaErrorInvalidValue;
    bound += mgroup_tile_bound(shared->rows_total, shared->G, shared->H, 128, pair);
    P.num_problems = 2;
  }
  if (routed.gather.src)
    return launch<0, 0, MGROUP, EPI_SWIGLU_FWD, 1, SPLIT_NONE, 0, 1>(
        P, bound, s, routed.h ? "gemm_gate_up_swiglu_gather" : "gemm_gate_up_recompute_gather");
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
  const char* name = routed.comb_y ? "gemm_down_shared_combine" : routed.out_row_map ? "gemm_down_slots" : "gemm_down";
  return launch<0, 0, MGROUP, EPI_F32, kPair>(P, bound, s, name);
}

}  // namespace moe
