// Backward expert GEMMs: dgrad of the down projection with the SwiGLU
// backward epilogue, dgrad of gate/up, and the ragged-K weight gradients.
#include "gemm_host.cuh"

namespace moe {
using namespace gemm;

namespace {

constexpr int kPair = 2;  // expert GEMMs run on CTA pairs (single CTAs when a row gather feeds A)

long long mgroup_tile_bound(int rows_total, int G, int N, int n_tile, int pair = kPair) {
  return ((long long)rows_total / (BM * pair) + G) * cdiv_h(N, n_tile);
}
int b_bytes(int pair) { return pair == 2 ? PairCfg<2>::B_BYTES : PairCfg<1>::B_BYTES; }

bool fill_dgrad_down(Params& P, Problem& pr, const DgradDownArgs& a, int pair) {
  const int ia = new_map(P), ib = new_map(P);
  if (ia < 0 || ib < 0) return false;
  const bool gat = a.gather.src != nullptr;
  // with a row gather the tiled A map (not loaded from) covers the source
  if (!encode_2d(&P.maps[ia], gat ? a.gather.src : a.dY, a.d, gat ? a.gather.src_rows : a.rows_total,
                 (uint64_t)a.d * 2, 64, BM))
    return false;
  // B[n = j in H, k = c in d] = W_d[g][c][j]: MN-major, stored [G][K=d][N=H]
  if (!encode_3d(&P.maps[ib], a.Wd, a.H, a.d, a.G, 64, 64)) return false;
  pr = blank_problem();
  pr.offsets = a.offsets;
  pr.G = a.G;
  pr.extent = a.rows_total;
  pr.N = a.H;
  pr.K = a.d;
  pr.mma_n = 256;
  pr.n_tile = 256;
  pr.half_ok = 1;
  pr.map_a = ia;
  pr.map_b = ib;
  pr.tx_bytes = (gat ? 0 : A_BYTES) + b_bytes(pair);  // gathered A rows arrive by cp.async
  pr.out = a.dau_hi;
  pr.out_lo = a.dau_lo;
  pr.ldo = 2LL * a.H;
  pr.aux = const_cast<float*>(a.au);
  pr.ld_aux = 2LL * a.H;
  pr.H = a.H;
  pr.gh_hi = a.gh_hi;
  pr.gh_lo = a.gh_lo;
  pr.gates = a.gates;
  pr.slot_of_row = a.slot_of_row;
  pr.gate_slots = a.gate_slots;
  pr.dgp = a.dgp;
  pr.ld_dgp = dgp_slots(a.H);
  // a | u come into shared memory by TMA, one 32-row x 32-column box each
  pr.map_aux = new_map(P);
  if (pr.map_aux < 0) return false;
  if (!encode_2d_f32(&P.maps[pr.map_aux], a.au, 2 * (uint64_t)a.H, a.rows_total, 2 * (uint64_t)a.H * 4, 32, 32))
    return false;
  if (gat && !set_gather(pr, 0, a.gather.src, a.d, a.gather.slot_of_row, a.gather.k, a.gather.nslots)) return false;
  return true;
}

bool fill_dgrad_gu(Params& P, Problem& pr, const DgradGuArgs& a) {
  const int ia = new_map(P), ig = new_map(P), iu = new_map(P);
  if (ia < 0 || ig < 0 || iu < 0) return false;
  if (!encode_2d(&P.maps[ia], a.dau, 2 * a.H, a.rows_total, (uint64_t)a.H * 4, 64, BM)) return false;
  // B[n = c in d, k = j in 2H]: W_g[g][j][c] for j < H, W_u[g][j-H][c] after
  if (!encode_3d(&P.maps[ig], a.Wg, a.d, a.H, a.G, 64, 64)) return false;
  if (!encode_3d(&P.maps[iu], a.Wu, a.d, a.H, a.G, 64, 64)) return false;
  pr = blank_problem();
  if (a.dau_lo) {
    pr.map_a_lo = new_map(P);
    if (pr.map_a_lo < 0) return false;
    if (!encode_2d(&P.maps[pr.map_a_lo], a.dau_lo, 2 * a.H, a.rows_total, (uint64_t)a.H * 4, 64, BM)) return false;
    pr.nsplit = 2;
  }
  pr.offsets = a.offsets;
  pr.G = a.G;
  pr.extent = a.rows_total;
  pr.N = a.d;
  pr.K = 2 * a.H;
  pr.mma_n = 256;
  pr.n_tile = 256;
  pr.half_ok = 1;
  pr.map_a = ia;
  pr.map_b = ig;
  pr.map_b2 = iu;
  pr.ksplit = a.H;
  pr.tx_bytes = A_BYTES + PairCfg<kPair>::B_BYTES;
  pr.out = a.dx;
  pr.out_f16 = 1;  // input-gradient rows: fp16 terms of the unpermute's sum
  pr.out_scale = a.scale;
  pr.ldo = a.d;
  return true;
}

// The block view that stands for operand m (0 = A, 1 = B) of a weight
// gradient: a gathered operand is never loaded through its map, so its map
// (and its per-group maps) are views of the other operand.
struct WgOperand {
  const void* ptr;
  uint64_t cols;
  uint32_t nblk;
};
WgOperand wg_operand(const WgradArgs& a, int m) {
  const bool gathered = a.gather.src != nullptr && a.gather_op == m;
  const int use = gathered ? 1 - m : m;
  return use == 0 ? WgOperand{a.A, (uint64_t)a.M, 2u} : WgOperand{a.B, (uint64_t)a.N, 4u};
}

bool fill_wgrad(Params& P, Problem& pr, const WgradArgs& a) {
  const int ia = new_map(P), ib = new_map(P);
  if (ia < 0 || ib < 0) return false;
  // 64-column block views: one TMA box per operand and stage (A: 2 blocks, B: 4)
  const int bkk = kg_rows(a.A_lo ? SPLIT_A : a.B_lo ? SPLIT_B : SPLIT_NONE);
  const WgOperand oa = wg_operand(a, 0), ob = wg_operand(a, 1);
  if (!encode_blocks(&P.maps[ia], oa.ptr, oa.cols, a.rows_total, bkk, oa.nblk)) return false;
  if (!encode_blocks(&P.maps[ib], ob.ptr, ob.cols, a.rows_total, bkk, ob.nblk)) return false;
  pr = blank_problem();
  if (a.A_lo) {
    pr.map_a_lo = new_map(P);
    if (pr.map_a_lo < 0) return false;
    if (!encode_blocks(&P.maps[pr.map_a_lo], a.A_lo, a.M, a.rows_total, bkk, 2)) return false;
  }
  if (a.B_lo) {
    pr.map_b_lo = new_map(P);
    if (pr.map_b_lo < 0) return false;
    if (!encode_blocks(&P.maps[pr.map_b_lo], a.B_lo, a.N, a.rows_total, bkk, 4)) return false;
  }
  pr.nsplit = (a.A_lo || a.B_lo) ? 2 : 1;
  pr.blk3d = 1;
  pr.offsets = a.offsets;
  pr.G = a.G;
  pr.extent = a.rows_total;
  pr.M = a.M;
  pr.N = a.N;
  pr.mma_n = 256;
  pr.n_tile = 256;
  pr.map_a = ia;
  pr.map_b = ib;
  // one ragged-K stage: A (2 blocks), B (4), and the lo half of A (2) or of B (4)
  // (a gathered operand's blocks arrive by cp.async)
  const int gathered_blocks = a.gather.src ? (a.gather_op == 0 ? 2 : 4) : 0;
  pr.tx_bytes = (2 + 4 + (a.A_lo ? 2 : a.B_lo ? 4 : 0) - gathered_blocks) * 64 * bkk * 2;
  pr.out = a.out;
  pr.out2 = a.out2;
  pr.row_split = a.out2 ? a.row_split : 0;
  pr.ldo = a.N;
  pr.gstride = (long long)(a.out2 ? a.row_split : a.M) * a.N;
  // the epilogue's TMA stores: out [G][rows < row_split][N], out2 [G][the rest][N]
  const int rows1 = a.out2 ? a.row_split : a.M;
  pr.map_out = new_map(P);
  if (pr.map_out < 0) return false;
  if (!encode_store_3d(&P.maps[pr.map_out], a.out, a.N, rows1, a.G)) return false;
  if (a.out2) {
    pr.map_out2 = new_map(P);
    if (pr.map_out2 < 0) return false;
    if (!encode_store_3d(&P.maps[pr.map_out2], a.out2, a.N, a.M - a.row_split, a.G)) return false;
  }
  if (a.gather.src && !set_gather(pr, a.gather_op, a.gather.src, a.gather_op == 0 ? a.M : a.N, a.gather.slot_of_row,
                                  a.gather.k, a.gather.nslots))
    return false;
  return true;
}

}  // namespace

cudaError_t gemm_dgrad_down(const DgradDownArgs& routed, const DgradDownArgs* shared, int* status, cudaStream_t s) {
  (void)status;
  Params P;
  std::memset(&P, 0, sizeof(P));
  const int pair = routed.gather.src ? 1 : kPair;
  if (shared && shared->gather.src) return cudaErrorInvalidValue;
  if (!fill_dgrad_down(P, P.prob[0], routed, pair)) return cudaErrorInvalidValue;
  long long bound = mgroup_tile_bound(routed.rows_total, routed.G, routed.H, 256, pair);
  P.num_problems = 1;
  if (shared) {
    if (!fill_dgrad_down(P, P.prob[1], *shared, pair)) return cudaErrorInvalidValue;
    bound += mgroup_tile_bound(shared->rows_total, shared->G, shared->H, 256, pair);
    P.num_problems = 2;
  }
  if (routed.gather.src)
    return launch<0, 1, MGROUP, EPI_SWIGLU_BWD, 1, SPLIT_NONE, 0, 1>(P, bound, s,
                                                                       "gemm_dgrad_down_swiglu_bwd_gather");
  return launch<0, 1, MGROUP, EPI_SWIGLU_BWD, kPair>(P, bound, s, "gemm_dgrad_down_swiglu_bwd");
}

cudaError_t gemm_dgrad_gu(const DgradGuArgs& routed, const DgradGuArgs* shared, int* status, cudaStream_t s) {
  (void)status;
  Params P;
  std::memset(&P, 0, sizeof(P));
  if (!fill_dgrad_gu(P, P.prob[0], routed)) return cudaErrorInvalidValue;
  long long bound = mgroup_tile_bound(routed.rows_total, routed.G, routed.d, 256);
  P.num_problems = 1;
  if (shared) {
    if (!fill_dgrad_gu(P, P.prob[1], *shared)) return cudaErrorInvalidValue;
    bound += mgroup_tile_bound(shared->rows_total, shared->G, shared->d, 256);
    P.num_problems = 2;
  }
  return launch<0, 1, MGROUP, EPI_F32, kPair>(P, bound, s, "gemm_dgrad_gate_up");
}

size_t group_maps_bytes(int G) { return (size_t)G * KG_MAPS_PER_GROUP * sizeof(CUtensorMap); }

cudaError_t gemm_wgrad(const WgradArgs& routed, const WgradArgs* shared, int* tile_counter, void* group_maps,
                       int* status, cudaStream_t s, const char* name) {
  (void)status;
  Params P;
  std::memset(&P, 0, sizeof(P));
  // the shared expert's tiles (K = all tokens) are numbered first, so the
  // dynamic schedule starts the heaviest tiles first
  const WgradArgs* order[2] = {shared ? shared : &routed, shared ? &routed : nullptr};
  long long bound = 0;
  int with_offsets = 0;
  bool counter_zeroed = false;  // by the group-maps kernel
  for (int i = 0; i < 2 && order[i]; ++i) {
    const WgradArgs& a = *order[i];
    Problem& pr = P.prob[i];
    if (!fill_wgrad(P, pr, a)) return cudaErrorInvalidValue;
    bound += (long long)a.G * cdiv_h(a.M, BM) * cdiv_h(a.N, 256);
    P.num_problems = i + 1;
    if (a.offsets) {
      // per-group maps of A, B and the lo half, built on the device before
      // the GEMM (one scratch area: at most one problem has offsets)
      if (!group_maps || with_offsets++ > 0) return cudaErrorInvalidValue;
      const void* lo = a.A_lo ? a.A_lo : a.B_lo;
      const int nmaps = lo ? 3 : 2;
      CUtensorMap whole[KG_MAPS_PER_GROUP] = {P.maps[pr.map_a], P.maps[pr.map_b]};
      if (lo) whole[2] = P.maps[a.A_lo ? pr.map_a_lo : pr.map_b_lo];
      const WgOperand oa = wg_operand(a, 0), ob = wg_operand(a, 1);
      const void* base[KG_MAPS_PER_GROUP] = {oa.ptr, ob.ptr, lo};
      const uint64_t cols[KG_MAPS_PER_GROUP] = {oa.cols, ob.cols, (uint64_t)(a.A_lo ? a.M : a.N)};
      const uint32_t nblk[KG_MAPS_PER_GROUP] = {oa.nblk, ob.nblk, a.A_lo ? 2u : 4u};
      CUtensorMap whole_1row[KG_MAPS_PER_GROUP];
      uint64_t rb[KG_MAPS_PER_GROUP];
      const int bkk = kg_rows(a.A_lo ? SPLIT_A : a.B_lo ? SPLIT_B : SPLIT_NONE);
      for (int m = 0; m < nmaps; ++m) {
        rb[m] = cols[m] * 2;
        if (!encode_blocks(&whole_1row[m], base[m], cols[m], 1, bkk, nblk[m])) return cudaErrorInvalidValue;
      }
      CUtensorMap* gm = static_cast<CUtensorMap*>(group_maps);
      cudaError_t e = launch_group_maps(whole, whole_1row, base, rb, nmaps, a.offsets, a.G, a.rows_total, gm,
                                        tile_counter, s);
      if (e != cudaSuccess) return e;
      pr.gmaps = gm;
      counter_zeroed = tile_counter != nullptr;
    }
  }
  P.tile_counter = tile_counter;
  // ragged K: single CTAs; both problems split the same operand
  if (shared && (!shared->A_lo != !routed.A_lo || !shared->B_lo != !routed.B_lo)) return cudaErrorInvalidValue;
  if (routed.A_lo && routed.B_lo) return cudaErrorInvalidValue;
  // the shared expert's problem reads its operands directly; a row gather is
  // the routed problem's
  if (shared && shared->gather.src) return cudaErrorInvalidValue;
  if (routed.gather.src) {
    if (routed.A_lo) return launch<1, 1, KGROUP, EPI_BF16, 1, SPLIT_A, 0, 1>(P, bound, s, name, counter_zeroed);
    if (routed.B_lo) return launch<1, 1, KGROUP, EPI_BF16, 1, SPLIT_B, 0, 1>(P, bound, s, name, counter_zeroed);
    return cudaErrorInvalidValue;
  }
  if (routed.A_lo) return launch<1, 1, KGROUP, EPI_BF16, 1, SPLIT_A>(P, bound, s, name, counter_zeroed);
  if (routed.B_lo) return launch<1, 1, KGROUP, EPI_BF16, 1, SPLIT_B>(P, bound, s, name, counter_zeroed);
  return launch<1, 1, KGROUP, EPI_BF16, 1, SPLIT_NONE>(P, bound, s, name, counter_zeroed);
}

}  // namespace moe
