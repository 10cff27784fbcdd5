// Persistent, warp-specialised grouped GEMM on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM, operands staged by TMA with 128-byte
// swizzle).  One CTA per SM; each CTA walks a device-side tile schedule built
// from per-group row offsets that never leave the GPU.
//
//   warp 0      TMA producer (one lane): A and B tiles into a STAGES-deep ring
//   warp 1      TMEM allocator + MMA issuer (one lane)
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator (one TMEM lane
//               = one output row per thread), fused elementwise work, stores
//
// Two fp32 accumulators of 128 x 256 (all 512 TMEM columns) let the epilogue
// of tile i overlap the main loop of tile i+1.
//
// Grouping modes:
//   MGROUP  ragged M: group g owns rows [off[g], off[g+1]) of A and of the
//           output, and its own B (3-D tensor map, group = 3rd coordinate).
//           Forward expert GEMMs and activation-gradient (dgrad) GEMMs.
//   KGROUP  ragged K: group g contracts over rows [off[g], off[g+1]) of A and
//           B (both stored with K as the row index) into its own output slab.
//           Weight-gradient (wgrad) GEMMs.  Each group is read through its
//           own tensor maps (built on the device from the offsets), so the
//           rows of its last K step past its end arrive as zeros.
//
// Split precision (nsplit = 2): one operand is given as a pair of bf16
// tensors hi + lo (hi = bf16(v), lo = bf16(v - hi), together ~16 mantissa
// bits); every K step is issued with each half into the same fp32
// accumulator.  Used where a derived operand feeds a long reduction (weight
// gradients), so that bf16 rounding of that operand does not grow with the
// number of rows summed.  Ragged-M problems load the halves in consecutive
// stages; ragged-K problems load both halves and the other operand in one
// stage (32 K rows), so the unsplit operand is read once.
//
// Tile schedule: static round-robin (tile t to CTA t mod grid), or, when the
// launch passes a zeroed tile counter (ragged K), dynamic: each CTA's first
// tile is its index, later ones come from an atomic counter; the producer
// publishes each tile index to the MMA and epilogue warps through a small
// ring in shared memory.  Tiles are numbered heaviest problem first.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace gemm {

constexpr int BM = 128;
constexpr int BN = 256;  // accumulator columns per tile
constexpr int BK = 64;   // K per pipeline stage: 128 bytes of bf16 (one swizzle row)
constexpr int UMMA_K = 16;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB: this CTA's A tile per stage
constexpr int NUM_THREADS = 192;
constexpr int MAX_PROBLEMS = 2;
constexpr int MAX_MAPS = 12;
constexpr int MAX_G = kMaxE + 1;
constexpr int TMEM_COLS = 2 * BN;
constexpr int MN_BLOCK_BYTES = 64 * BK * 2;  // one 64(MN) x 64(K) MN-major box: 8 KB

constexpr int RING = 4;  // tile indices in flight from the producer to the other roles
constexpr int KG_MAPS_PER_GROUP = 3;  // ragged K, per-group maps: A, B, lo half

enum Mode : int { MGROUP = 0, KGROUP = 1 };
// Ragged K: which operand comes as hi + lo halves (a compile-time choice, so
// that each kernel issues its MMAs from one straight-line sequence)
enum Split : int { SPLIT_NONE = 0, SPLIT_A = 1, SPLIT_B = 2 };

// K rows per ragged-K stage: 64 (four 16-row MMA sub-steps) when A or
// nothing is split, 32 when B (256 columns) is split, so that a stage stays
// small enough for several of them to be in flight.  Host code sizes the TMA
// boxes with the same function.
__host__ __device__ constexpr int kg_rows(int split) { return split == SPLIT_B ? 32 : 64; }

// Ragged-K stage: BKK K rows of A (2 MN-major blocks of 64 columns) | B (4
// blocks) | the lo half of the split operand (A's 2 blocks or B's 4), as many
// stages as fit in ~200 KB: 48 KB x 4 (no split), 64 KB x 3 (A split),
// 40 KB x 5 (B split, 32 rows).
template <int SPLIT>
struct KgCfg {
  static constexpr int BKK = kg_rows(SPLIT);
  static constexpr int BLOCK_BYTES = 64 * BKK * 2;  // one 64 (MN) x BKK (K) block
  static constexpr int A_BYTES = 2 * BLOCK_BYTES;
  static constexpr int B_BYTES = 4 * BLOCK_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + (SPLIT == SPLIT_A ? A_BYTES : SPLIT == SPLIT_B ? B_BYTES : 0);
  static constexpr int STAGES = (200 * 1024) / STAGE_BYTES;
};
enum Epi : int { EPI_BF16 = 0, EPI_F32 = 1, EPI_SWIGLU_FWD = 2, EPI_SWIGLU_BWD = 3 };

struct Problem {
  const int* offsets;  // [G+1] device; NULL: `extent` split evenly into G chunks
  int G;
  int extent;          // rows (MGROUP) or K (KGROUP) covered when offsets == NULL; also an upper clamp
  int M, N, K;         // MGROUP uses N, K (M per group); KGROUP uses M, N (K per group)
  int mma_n;           // instruction N (multiple of 16, <= 256)
  int half_ok;         // CTA pair, ragged M: a group's last tile with <= 128 rows
                       // runs as an M = 128 pair MMA (n_tile == mma_n == 256, or
                       // the SwiGLU forward's interleaved gate/up tile)
  int n_tile;          // output columns per tile (256; 128 h columns for EPI_SWIGLU_FWD)
  int map_a, map_b, map_b2;  // tensor-map indices; map_b2 = second B map or -1
  int ksplit;          // MN-major B: k >= ksplit reads map_b2 at k - ksplit (0 = off)
  int map_a_lo, map_b_lo;  // lo halves of a split operand (-1 = none)
  int nsplit;          // 1, or 2 = every K step issued with the hi and the lo half
  int blk3d;           // ragged K: A, B (and lo) maps are 64-column block views, one box per operand
  // ragged K with offsets: per-group block-view maps [G][KG_MAPS_PER_GROUP]
  // (A, B, lo half) on the device, each over its group's rows only, so that
  // reads past a group's end come back as zeros; K coordinates are then
  // relative to the group's first row
  const CUtensorMap* gmaps;
  uint32_t tx_bytes;   // bytes landing per stage
  // epilogue
  void* out;
  long long ldo;       // elements
  long long gstride;   // elements between groups' output slabs (KGROUP)
  void* out2;          // rows >= row_split go to out2 (KGROUP; 0 = off)
  int row_split;
  int map_out, map_out2;   // EPI_BF16 (ragged K): TMA-store maps of out / out2, [G][rows][N], 32 x 32 boxes
  // MXFP8 operands (MX launches): tile-atom scale arrays of A (rows of the A
  // buffer) and B (per group, sfb_gstride bytes apart), K / 128 atoms per row
  // tile; `counts` (nullable) ends group g's rows at off[g] + counts[g]
  // (the offsets then mark padded segments)
  const uint8_t* sfa;
  const uint8_t* sfb;
  long long sfb_gstride;
  int nkq;
  const int* counts;
  uint8_t* out_sf;         // SwiGLU (MX): tile-atom scales of the quantized h
  int out_sf_nq;           // ... H / 128
  void* aux;           // SWIGLU_FWD: au out; SWIGLU_BWD: au in
  long long ld_aux;
  const float* bias;   // EPI_F32 (nullable)
  int out_f16;         // EPI_F32: out holds fp16 (a value beyond its range records MOE_ERR_RANGE)
  const uint32_t* out_scale;  // out_f16: values stored divided by 2^e of this gradient scale word (NULL: e = 0)
  int H;               // SWIGLU: column offset of u within au
  // EPI_SWIGLU_BWD
  const float* gates;      // per-slot gate (nullable: g = 1)
  const int* slot_of_row;  // row -> slot (with gates)
  int gate_slots;          // number of valid slots (bounds check)
  void* out_lo;            // lo half of da | du
  void* gh_hi;             // g*h, hi / lo halves, [rows, H]
  void* gh_lo;
  float* dgp;              // per-row partials of the gate gradient, [rows, ld_dgp] (nullable)
  int ld_dgp;
  int map_aux;             // tensor map of au (fp32, 32 x 32 boxes): a | u staged by TMA
  // Row gather (the permutation fused into the operand loads; GATHER
  // launches, single CTAs): one operand is read row by row from a
  // token-indexed source [src rows, cols] (gather_src, gather_pitch bytes per
  // row) by 16-byte cp.async copies into the stage's 128-byte-swizzled
  // layout; the stage's barrier expects one more arrival per producer lane.
  // Permuted row r stands for source row gather_slot[r] / gather_k.  Ragged
  // M: A row r of the tile.  Ragged K: K row r of the group (the operand
  // gather_op, 0 = A, 1 = B).  Rows past the group's end read source row 0:
  // ragged-M rows there are never stored, and on ragged-K rows there the
  // other operand is zero.
  const int* gather_slot;  // NULL: no gather
  const uint8_t* gather_src;
  long long gather_pitch;
  int gather_k;
  int gather_slots;        // valid slot values are [0, gather_slots)
  int gather_op;
  // EPI_F32, ragged M: row r of the problem is stored at output row
  // out_row_map[r] (NULL: row r), which must lie in [0, out_map_rows)
  const int* out_row_map;
  int out_map_rows;
  // EPI_F32, the shared expert's down projection with the combine fused in
  // (comb_y != NULL): instead of s, y[t] = bf16(s[t] + sum over kept slots
  // (t,j) of gates[t,j] o_slot[t*k+j]), the sum taken in slot order
  const void* comb_o;           // [T*k, ldo] fp16 expert outputs in slot order
  const float* comb_gates;      // [T*k]
  const int* comb_row_of_slot;  // [T*k]: slot kept iff >= 0
  int comb_k;
  void* comb_y;                 // [T, ldo] bf16
};

struct Params {
  CUtensorMap maps[MAX_MAPS];
  Problem prob[MAX_PROBLEMS];
  int num_problems;
  int num_maps;
  int* status;
  int* tile_counter;  // zeroed device int: dynamic schedule (ragged K); NULL: static
};

struct Sched {
  int tile_start[MAX_PROBLEMS + 1];
  int off[MAX_PROBLEMS][MAX_G];
  int tpre[MAX_PROBLEMS][MAX_G];  // MGROUP: exclusive prefix of tiles per group
  int end[MAX_PROBLEMS][MAX_G];   // MGROUP: first row past group g's rows
};

// PAIR = 1: one CTA computes a 128 x 256 tile.  PAIR = 2: a cluster of two
// CTAs computes a 256 x 256 tile with pair MMAs (tcgen05 cta_group::2): each
// CTA holds 128 rows of A and 128 of the 256 columns of B, so a stage is
// 32 KB instead of 48 KB and six stages fit where four did.
template <int PAIR>
struct PairCfg {
  static constexpr int STAGES = PAIR == 2 ? 6 : 4;
  static constexpr int B_BYTES = BN * BK * 2 / PAIR;  // this CTA's share of the B tile per stage
  static constexpr int TILE_M = BM * PAIR;
};

template <int STG>
struct SmemTailT {
  float tbuf[4][32 * 36];  // per epilogue warp: 32x32 fp32 staging chunk, rows padded to 36
  uint64_t full[STG];      // the stage's data landed (PAIR = 2: the leader's counts both CTAs)
  uint64_t empty[STG];     // stage consumed by the MMAs (both CTAs, PAIR = 2)
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t au_full[4][2];     // SwiGLU backward: a | u chunk landed (per epilogue warp, 2 buffers)
  uint64_t ring_full[RING];   // dynamic schedule: tile index published
  uint64_t ring_empty[RING];  // ... and read by the MMA warp and the four epilogue warps
  int ring[RING];
  alignas(16) int gsrc[2][128];  // row gather: source rows of the rows being loaded (two buffers)
  uint32_t tmem_base;
  int abort_flag;
  Sched sched;
};

// SwiGLU backward: per epilogue warp, two buffers of one 32-row x 32-column
// chunk of a and of u (fp32), filled by TMA; the main loop gives up two
// stages for them (it is not what bounds that launch)
constexpr int AU_CHUNK_BYTES = 2 * 32 * 32 * 4;

// MXFP8 (MX = 1, ragged M, single CTA): a stage holds 128 K values (128 bytes
// of E4M3 per row: one 128-byte swizzle row) of A (128 rows) and B (128 rows)
// and one 512-byte scale atom of each; 6 stages.  The scale atoms go to a
// ring of tensor-memory columns (MX_SF_COL + 8 * stage) between the two
// 128-column accumulators.
constexpr int MX_BK = 128;
constexpr int MX_B_BYTES = 128 * MX_BK;
constexpr int MX_SF_BYTES = 1024;
constexpr int MX_STAGES = 6;
constexpr int MX_N = 128;      // MMA N of the MX launches
constexpr int MX_SF_COL = 128;  // first tensor-memory column of the scale ring

template <int MODE, int EPI, int PAIR, int SPLIT, int MX = 0>
struct StageCfg {
  static constexpr int STAGES =
      MX ? MX_STAGES
         : (MODE == KGROUP ? KgCfg<SPLIT>::STAGES
                           : (EPI == EPI_SWIGLU_BWD ? (PAIR == 2 ? 4 : 2) : PairCfg<PAIR>::STAGES));
  static constexpr int BYTES = MX ? A_BYTES + MX_B_BYTES + MX_SF_BYTES
                                  : (MODE == KGROUP ? KgCfg<SPLIT>::STAGE_BYTES : A_BYTES + PairCfg<PAIR>::B_BYTES);
  static constexpr int EPI_BYTES = EPI == EPI_SWIGLU_BWD ? 4 * 2 * AU_CHUNK_BYTES : 0;
};

template <int MODE, int EPI, int PAIR, int SPLIT, int MX = 0>
constexpr size_t smem_bytes() {
  using C = StageCfg<MODE, EPI, PAIR, SPLIT, MX>;
  return 1024 + C::STAGES * C::BYTES + C::EPI_BYTES + sizeof(SmemTailT<C::STAGES>);
}

// Source row of permuted row `row` of a gathered operand (0 for rows at or
// past `end`, and for an out-of-range slot, which is recorded as a device
// bounds error).
__device__ __forceinline__ int gather_source(const int* slot_of_row, int div, int nslots, int row, int end,
                                             int* status) {
  if (row >= end) return 0;
  const int slot = __ldg(slot_of_row + row);
  if (slot < 0 || slot >= nslots) {
    record_status(status, MOE_ERR_DEVICE_BOUNDS);
    return 0;
  }
  return slot / div;
}

struct TileInfo {
  int p, g, m0, n0, rows_end, k0, k1, nk;
  // CTA pair, last tile of a group with at most 128 rows left: an M = 128
  // pair MMA (64 rows from each CTA) at half the MMA work of a 256-row tile.
  // Its accumulator is folded over the lanes: in each CTA, TMEM lanes 0-63
  // hold the CTA's 64 rows for accumulator columns [0, N/2) and lanes 64-127
  // the same rows for columns [N/2, N), both at TMEM columns [0, N/2).
  bool half;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

template <int MODE, int TILE_M, int KBK, int MBK>
__device__ __forceinline__ TileInfo decode(const Params& P, const Sched& S, int t) {
  TileInfo ti;
  int p = (P.num_problems > 1 && t >= S.tile_start[1]) ? 1 : 0;
  const Problem& pr = P.prob[p];
  int local = t - S.tile_start[p];
  int nt = cdiv(pr.N, pr.n_tile);
  ti.p = p;
  if (MODE == MGROUP) {
    int lo = 0, hi = pr.G - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (S.tpre[p][mid] <= local) lo = mid; else hi = mid - 1;
    }
    int g = lo;
    int within = local - S.tpre[p][g];
    int r0 = S.off[p][g], r1 = S.off[p][g + 1];
    // n fastest: tiles that run at the same time share one slab of A rows and
    // walk the group's weights, which stay in L2 across slabs
    int m_idx = within / nt, n_idx = within - m_idx * nt;
    ti.g = g;
    ti.m0 = r0 + m_idx * TILE_M;
    ti.rows_end = S.end[p][g];
    (void)r1;
    ti.n0 = n_idx * pr.n_tile;
    ti.k0 = 0;
    ti.k1 = pr.K;
    ti.nk = cdiv(pr.K, MBK) * pr.nsplit;
    ti.half = TILE_M == 2 * BM && pr.half_ok && ti.rows_end - ti.m0 <= BM;
  } else {
    int mt = cdiv(pr.M, TILE_M);
    int per = mt * nt;
    int g = local / per;
    int within = local - g * per;
    int m_idx = within / nt, n_idx = within - m_idx * nt;
    ti.g = g;
    ti.m0 = m_idx * TILE_M;
    ti.rows_end = pr.M;
    ti.n0 = n_idx * pr.n_tile;
    ti.k0 = S.off[p][g];
    ti.k1 = S.off[p][g + 1];
    ti.nk = cdiv(ti.k1 - ti.k0, KBK);
    ti.half = false;
  }
  return ti;
}

// Schedule set-up, run by every thread of the CTA before the roles start.
template <int MODE, int TILE_M>
__device__ void build_schedule(const Params& P, Sched& S) {
  const int tid = threadIdx.x;
  for (int p = 0; p < P.num_problems; ++p) {
    const Problem& pr = P.prob[p];
    int chunk = pr.offsets ? 0 : cdiv(cdiv(pr.extent, pr.G), BK) * BK;
    for (int i = tid; i <= pr.G; i += blockDim.x) {
      int v = pr.offsets ? __ldg(pr.offsets + i) : min(i * chunk, pr.extent);
      S.off[p][i] = v;
    }
  }
  __syncthreads();
  // clamp to a monotone sequence inside [0, extent]; count out-of-range
  // offsets as a device error (they would index outside the caller buffers)
  if (threadIdx.x < 32 * P.num_problems && (threadIdx.x & 31) == 0) {
    int p = threadIdx.x >> 5;
    const Problem& pr = P.prob[p];
    int prev = 0;
    bool bad = false;
    for (int i = 0; i <= pr.G; ++i) {
      int v = S.off[p][i];
      if (v < prev || v > pr.extent || (i == 0 && v != 0)) bad = true;
      v = min(max(v, prev), pr.extent);
      if (i == 0) v = 0;
      S.off[p][i] = v;
      prev = v;
    }
    if (bad) record_status(P.status, MOE_ERR_DEVICE_BOUNDS);
  }
  __syncthreads();
  for (int p = 0; p < P.num_problems; ++p) {
    const Problem& pr = P.prob[p];
    for (int g = threadIdx.x; g < pr.G; g += blockDim.x) {
      const int r0 = S.off[p][g], r1 = S.off[p][g + 1];
      S.end[p][g] = pr.counts ? r0 + min(max(__ldg(pr.counts + g), 0), r1 - r0) : r1;
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int base = 0;
    for (int p = 0; p < P.num_problems; ++p) {
      const Problem& pr = P.prob[p];
      int nt = cdiv(pr.N, pr.n_tile);
      int total;
      if (MODE == MGROUP) {
        // warp scan of per-group tile counts
        int per_lane = cdiv(pr.G, 32);
        int g0 = lane * per_lane;
        int local = 0;
        for (int j = 0; j < per_lane; ++j) {
          int g = g0 + j;
          if (g < pr.G) local += cdiv(S.off[p][g + 1] - S.off[p][g], TILE_M) * nt;
        }
        int incl = local;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
          int v = __shfl_up_sync(0xffffffffu, incl, s);
          if (lane >= s) incl += v;
        }
        int run = incl - local;
        for (int j = 0; j < per_lane; ++j) {
          int g = g0 + j;
          if (g < pr.G) {
            S.tpre[p][g] = run;
            run += cdiv(S.off[p][g + 1] - S.off[p][g], TILE_M) * nt;
          }
        }
        total = __shfl_sync(0xffffffffu, incl, 31);
        if (lane == 0) S.tpre[p][pr.G] = total;
      } else {
        total = pr.G * cdiv(pr.M, TILE_M) * nt;
      }
      if (lane == 0) S.tile_start[p] = base;
      base += total;
    }
    if (lane == 0) S.tile_start[P.num_problems] = base;
  }
  __syncthreads();
}

// sigmoid with CUDA's fast exponential and fast division (about 2 ulp; an
// IEEE-exact division here was most of the SwiGLU epilogues' time).  For
// a < -87 the denominator overflows and the result is 0, the right limit.
__device__ __forceinline__ float sigmoidf_(float a) { return __fdividef(1.0f, 1.0f + __expf(-a)); }

// Epilogue register layout ("quad layout"): for a warp's 32 rows x 32
// columns, lane l holds, for j = 0..7, the four consecutive columns
// 4*(l%8) .. 4*(l%8)+3 of row 4*j + l/8.  Eight lanes cover one row, so every
// global access of an instruction is four rows x 128 contiguous bytes (fp32)
// or 64 bytes (bf16).
constexpr int TB_STRIDE = 36;  // floats per row of the staging buffer (16-byte aligned, conflict-free)

// 32 accumulator columns at `taddr` (row-per-thread in TMEM) -> quad layout,
// through the warp's 32 x 36 shared-memory buffer (float4 writes and reads,
// free of bank conflicts).
__device__ __forceinline__ void tmem_chunk_quad(uint32_t taddr, float* tb, int lane, float4 (&v)[8]) {
  uint32_t r[32];
  ptx::tmem_ld32(taddr, r);
  ptx::tmem_ld_wait(r);
  __syncwarp();
#pragma unroll
  for (int m = 0; m < 8; ++m)
    *reinterpret_cast<float4*>(tb + lane * TB_STRIDE + 4 * m) =
        make_float4(__uint_as_float(r[4 * m]), __uint_as_float(r[4 * m + 1]), __uint_as_float(r[4 * m + 2]),
                    __uint_as_float(r[4 * m + 3]));
  __syncwarp();
  const int rs = lane >> 3, cq = (lane & 7) * 4;
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const float4*>(tb + (4 * j + rs) * TB_STRIDE + cq);
}

__device__ __forceinline__ void zero_quad(float4 (&v)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
}
// v = hi + lo, hi = bf16(v), lo = bf16(v - hi), four values
__device__ __forceinline__ void split_store4(__nv_bfloat16* hi, __nv_bfloat16* lo, float4 v) {
  const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y), h23 = __floats2bfloat162_rn(v.z, v.w);
  const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
  *reinterpret_cast<uint2*>(hi) = make_uint2(*reinterpret_cast<const uint32_t*>(&h01),
                                             *reinterpret_cast<const uint32_t*>(&h23));
  *reinterpret_cast<uint2*>(lo) = make_uint2(pack_bf16(v.x - f01.x, v.y - f01.y), pack_bf16(v.z - f23.x, v.w - f23.y));
}

// TMA load into this CTA's shared memory.  PAIR = 1: bytes counted on this
// CTA's barrier.  PAIR = 2: bytes counted on the leader CTA's barrier (so the
// leader's single wait covers both halves of the stage).
template <int PAIR>
__device__ __forceinline__ void load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, uint32_t bar_leader, int c0,
                                        int c1) {
  if (PAIR == 1) ptx::tma_load_2d(dst, m, bar, c0, c1);
  else ptx::tma_load_2d_pair(dst, m, bar_leader, c0, c1);
}
template <int PAIR>
__device__ __forceinline__ void load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, uint32_t bar_leader, int c0,
                                        int c1, int c2) {
  if (PAIR == 1) ptx::tma_load_3d(dst, m, bar, c0, c1, c2);
  else ptx::tma_load_3d_pair(dst, m, bar_leader, c0, c1, c2);
}

template <int AMN, int BMN, int MODE, int EPI, int PAIR, int SPLIT, int MX = 0, int GATHER = 0>
__global__ void __launch_bounds__(NUM_THREADS, 1) grouped_gemm_kernel(const __grid_constant__ Params P) {
  static_assert(!GATHER || (!MX && PAIR == 1 && (MODE == KGROUP || AMN == 0)),
                "row gather: single CTAs, K-major A (ragged M) or ragged K");
  static_assert(!(MODE == KGROUP && PAIR == 2), "ragged-K GEMMs run on single CTAs");
  static_assert(!MX || (MODE == MGROUP && PAIR == 1 && AMN == 0 && BMN == 0 && SPLIT == SPLIT_NONE &&
                        (EPI == EPI_SWIGLU_FWD || EPI == EPI_F32)),
                "MXFP8: ragged-M, single-CTA, K-major operands, SwiGLU or fp32 epilogue");
  static_assert(MODE == MGROUP || (AMN == 1 && BMN == 1), "ragged-K operands are MN-major");
  static_assert(MODE == KGROUP || SPLIT == SPLIT_NONE, "ragged-M split operands use consecutive stages");
  using Cfg = PairCfg<PAIR>;
  using SC = StageCfg<MODE, EPI, PAIR, SPLIT, MX>;
  constexpr int STAGES = SC::STAGES;
  constexpr int B_BYTES = MX ? MX_B_BYTES : Cfg::B_BYTES;
  constexpr int MBK = MX ? MX_BK : BK;  // K per ragged-M stage
  constexpr int TILE_M = Cfg::TILE_M;
  // ragged K: rows per stage and the stage's blocks
  constexpr int KBK = KgCfg<SPLIT>::BKK;
  constexpr int KG_BLOCK_BYTES = KgCfg<SPLIT>::BLOCK_BYTES;
  constexpr int KG_A_BYTES = KgCfg<SPLIT>::A_BYTES;
  constexpr int KG_B_BYTES = KgCfg<SPLIT>::B_BYTES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // ragged M: A ring then B ring; ragged K: stage s at smem + s * SC::BYTES
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sSF = sB + STAGES * B_BYTES;  // MX: the stages' scale atoms (A at +0, B at +512)
  using Tail = SmemTailT<STAGES>;
  uint8_t* au_buf = smem + STAGES * SC::BYTES;  // SwiGLU backward only
  Tail* tail = reinterpret_cast<Tail*>(au_buf + SC::EPI_BYTES);
  Sched& S = tail->sched;
  volatile int* abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // PAIR = 2: rank 0 (leader) issues the pair MMAs; rank 1 loads the other
  // halves of A and B, whose bytes are counted on the leader's barriers.
  const int rank = PAIR == 2 ? static_cast<int>(ptx::cluster_ctarank()) : 0;
  const int tile0 = blockIdx.x / PAIR;
  const int tile_step = gridDim.x / PAIR;

  // programmatic launch: this prologue touches shared memory, tensor memory
  // and the kernel parameters only; the wait below (every thread, before the
  // schedule reads the offsets) orders all global accesses after the
  // previous kernel
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // GATHER: the lead's expect-tx arrival and one cp.async arrival per lane
      ptx::mbar_init(&tail->full[s], GATHER ? 33 : 1);
      ptx::mbar_init(&tail->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tail->tmem_full[a], 1);
      ptx::mbar_init(&tail->tmem_empty[a], 4 * PAIR);  // one arrival per epilogue warp of each CTA
    }
    for (int w = 0; w < 4; ++w) {
      ptx::mbar_init(&tail->au_full[w][0], 1);
      ptx::mbar_init(&tail->au_full[w][1], 1);
    }
    for (int r = 0; r < RING; ++r) {
      ptx::mbar_init(&tail->ring_full[r], 1);
      ptx::mbar_init(&tail->ring_empty[r], 5);  // the MMA thread and the four epilogue warps
    }
    tail->abort_flag = 0;
    ptx::fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < P.num_maps; ++i) ptx::prefetch_tmap(&P.maps[i]);
  }
  if (warp == 1) {
    ptx::tmem_alloc<PAIR>(&tail->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish<PAIR>();
    ptx::tc_fence_before();
  }
  dependency_wait();
  build_schedule<MODE, TILE_M>(P, S);  // contains __syncthreads
  if (PAIR == 2) ptx::cluster_sync();  // the peer's barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;
  const int total = S.tile_start[P.num_problems];
  const int row_half = rank * BM;  // this CTA's first row (or M column) within a tile
  const bool dyn = MODE == KGROUP && P.tile_counter != nullptr;

  // The i-th tile of this CTA, for the MMA and epilogue warps (whole warp):
  // static, or read from the ring the producer fills.  False on timeout.
  auto take_tile = [&](int i, int& t) -> bool {
    if (!dyn) {
      t = tile0 + i * tile_step;
      return true;
    }
    const int slot = i & (RING - 1);
    if (!ptx::mbar_wait_bounded(&tail->ring_full[slot], (i / RING) & 1, abort_flag, kWaitLimitNs)) return false;
    t = *reinterpret_cast<volatile int*>(&tail->ring[slot]);
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&tail->ring_empty[slot]);
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // One thread waits on the barriers and issues the loads.  GATHER: the
    // whole warp runs the loop; lane 0 waits and issues the tiled loads, and
    // every lane issues gathers of four rows of the gathered operand.
    if (GATHER || lane == 0) {
      const bool lead = lane == 0;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase_mask = 0;  // bit s: parity of the last load issued into stage s
      uint32_t issued_any = 0;
      bool ok = true;
      int fetched = 0;   // raw value of the last tile-counter atomic
      int acquired = -1;  // (problem, group) whose per-group maps this thread last acquired
      for (int i = 0; ok; ++i) {
        int t = 0;
        if (dyn) {
          // publish this tile's index, then fetch the next one (its latency
          // is hidden behind this tile's loads)
          const int slot = i & (RING - 1);
          bool got = true;
          if (lead) {
            got = ptx::mbar_wait_bounded(&tail->ring_empty[slot], ((i / RING) & 1) ^ 1, abort_flag, kWaitLimitNs);
            if (got) {
              t = i == 0 ? tile0 : fetched + tile_step;
              *reinterpret_cast<volatile int*>(&tail->ring[slot]) = t;
              ptx::mbar_arrive(&tail->ring_full[slot]);
              // used at the next tile only: no instruction here waits for the
              // atomic's round trip
              if (t < total) fetched = atomicAdd(P.tile_counter, 1);
            }
          }
          if (GATHER) {
            got = __shfl_sync(0xffffffffu, got, 0);
            t = __shfl_sync(0xffffffffu, t, 0);
          }
          if (!got) {
            ok = false;
            break;
          }
          if (t >= total) break;
        } else {
          t = tile0 + i * tile_step;
          if (t >= total) break;
        }
        TileInfo ti = decode<MODE, TILE_M, KBK, MBK>(P, S, t);
        // Everything the stage loop needs, read once per tile: a parameter
        // read inside the loop would be repeated after every asm statement
        // (they all clobber memory), which cost as much as the MMAs.
        const Problem& pr = P.prob[ti.p];
        const uint32_t tx = pr.tx_bytes * PAIR;
        const int nsplit = pr.nsplit, ksplit = pr.ksplit, blk3d = pr.blk3d;
        const int nblk = pr.n_tile / 64 / PAIR;
        const CUtensorMap* mA = &P.maps[pr.map_a];
        const CUtensorMap* mB = &P.maps[pr.map_b];
        const CUtensorMap* mB2 = &P.maps[pr.map_b2 >= 0 ? pr.map_b2 : pr.map_b];
        const CUtensorMap* mAlo = pr.map_a_lo >= 0 ? &P.maps[pr.map_a_lo] : nullptr;
        const CUtensorMap* mBlo = pr.map_b_lo >= 0 ? &P.maps[pr.map_b_lo] : nullptr;
        // a half tile takes 64 rows from each CTA: the peer's start 64 rows on
        const int am = ti.m0 + (ti.half ? rank * (BM / 2) : row_half), bn = ti.n0 + row_half;
        const uint8_t* mx_sfa = pr.sfa;
        const uint8_t* mx_sfb = pr.sfb + (long long)ti.g * pr.sfb_gstride;
        const int mx_nkq = pr.nkq;
        int k0 = ti.k0;
        const int g = ti.g, nk = ti.nk;
        // Row gather: ragged M gathers this CTA's 128 A rows (this lane's four
        // rows am + 4 lane + 0..3, fixed for the tile); ragged K gathers, per
        // stage, the quad kq of the stage's K rows into every block of the
        // gathered operand (lanes past the last (quad, block) pair idle)
        // Row gather: the lanes look the source rows up (slot_of_row / k)
        // into shared memory, then copy them 16 bytes at a time (lane: chunk
        // lane & 7 of rows lane >> 3, +4, +8, ...: four whole 128-byte rows
        // per instruction).  These copies go through the L1's miss queue, so
        // fewer bytes are in flight than with a tiled TMA load (TMA's own
        // four-row gathers take about 60 cycles per instruction): a gathering
        // GEMM runs at a fraction of the tiled one's rate.
        const bool gat = GATHER && pr.gather_slot != nullptr;
        const uint8_t* g_src = pr.gather_src;
        const long long g_pitch = pr.gather_pitch;
        const int g_chunk = lane & 7, g_rg = lane >> 3;
        const int* g_slot = pr.gather_slot;
        const int g_div = pr.gather_k, g_nslots = pr.gather_slots, g_op = pr.gather_op;
        constexpr int KNQ = KBK / 4;  // ragged K: row quads per stage (<= 16)
        int gnext[4] = {0, 0, 0, 0};  // ragged K: source rows of lane's quad of the next stage
        if (gat) {
          if (MODE == MGROUP) {
            // rows am .. am + 127 of this tile, fixed for its stages (the
            // last tile's gathers were issued before lane 0 reaches this sync)
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              tail->gsrc[0][4 * lane + q] =
                  gather_source(g_slot, g_div, g_nslots, am + 4 * lane + q, ti.rows_end, P.status);
            __syncwarp();
          } else if (nk > 0 && lane < KNQ) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              gnext[q] = gather_source(g_slot, g_div, g_nslots, ti.k0 + 4 * lane + q, ti.k1, P.status);
          }
        }
        if (MODE == KGROUP && pr.gmaps != nullptr && nk > 0) {
          // this group's own maps (written by an earlier launch: acquired for
          // the tensor-map proxy once per group by the thread that loads from
          // them); K rows counted from the group's start
          const CUtensorMap* gm = pr.gmaps + (long long)g * KG_MAPS_PER_GROUP;
          mA = gm;
          mB = gm + 1;
          if (SPLIT == SPLIT_A) mAlo = gm + 2;
          if (SPLIT == SPLIT_B) mBlo = gm + 2;
          const int key = ti.p * MAX_G + g;
          if (lead && key != acquired) {
            ptx::tmap_acquire(mA);
            ptx::tmap_acquire(mB);
            if (SPLIT != SPLIT_NONE) ptx::tmap_acquire(gm + 2);
            acquired = key;
          }
          k0 = 0;
        }
        for (int kb = 0; kb < nk; ++kb) {
          if (MODE == KGROUP && gat) {
            // this stage's source rows into buffer kb & 1 (lane 0 reads the
            // other buffer for the previous stage until this sync); the next
            // stage's lookups are issued now and complete behind this stage's
            // wait
            if (lane < KNQ) {
#pragma unroll
              for (int q = 0; q < 4; ++q) tail->gsrc[kb & 1][4 * lane + q] = gnext[q];
              if (kb + 1 < nk) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  gnext[q] = gather_source(g_slot, g_div, g_nslots, ti.k0 + (kb + 1) * KBK + 4 * lane + q, ti.k1,
                                           P.status);
              }
            }
            __syncwarp();
          }
          bool got = true;
          if (lead) got = ptx::mbar_wait_bounded(&tail->empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs);
          if (GATHER) got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) {
            ok = false;
            break;
          }
          uint64_t* fb = &tail->full[stage];
          const uint32_t fbl = PAIR == 2 ? ptx::mapa(ptx::smem_u32(fb), 0) : 0u;
          if (lead && rank == 0) ptx::mbar_arrive_expect_tx(fb, tx);
          issued_any |= 1u << stage;
          issued_phase_mask = (issued_phase_mask & ~(1u << stage)) | (phase << stage);
          if (MODE == KGROUP) {
            // A (2 blocks) | B (nblk blocks) | lo half of A or of B
            const int k = k0 + kb * KBK;
            uint8_t* st = smem + stage * SC::BYTES;
            uint8_t* lo = st + KG_A_BYTES + KG_B_BYTES;
            if (blk3d) {
              // one instruction per operand (a TMA load's issue cost barely
              // depends on its size)
              if (lead) {
                if (!(gat && g_op == 0)) ptx::tma_load_3d(st, mA, fb, 0, k, am / 64);
                if (!(gat && g_op == 1)) ptx::tma_load_3d(st + KG_A_BYTES, mB, fb, 0, k, bn / 64);
                if (SPLIT == SPLIT_A) ptx::tma_load_3d(lo, mAlo, fb, 0, k, am / 64);
                if (SPLIT == SPLIT_B) ptx::tma_load_3d(lo, mBlo, fb, 0, k, bn / 64);
              }
              if (gat) {
                // the gathered operand's blocks (A: 2, B: 4) of 64 columns
                // x KBK rows
                const int nbg = g_op == 0 ? 2 : 4;
                uint8_t* gdst = st + (g_op == 0 ? 0 : KG_A_BYTES);
                const uint8_t* gsrc0 = g_src + (long long)(g_op == 0 ? am : bn) * 2 + g_chunk * 16;
                const int* rows = tail->gsrc[kb & 1];
                for (int i = 0; i < KBK / 4; ++i) {
                  const int r = 4 * i + g_rg;
                  const uint8_t* src = gsrc0 + (long long)rows[r] * g_pitch;
                  uint8_t* dst = gdst + r * 128 + ((g_chunk ^ (r & 7)) << 4);
                  for (int j = 0; j < nbg; ++j) ptx::cp_async_16(dst + j * KG_BLOCK_BYTES, src + j * 128);
                }
              }
            } else if (lead) {
              ptx::tma_load_2d(st, mA, fb, am, k);
              ptx::tma_load_2d(st + KG_BLOCK_BYTES, mA, fb, am + 64, k);
              for (int j = 0; j < nblk; ++j) ptx::tma_load_2d(st + KG_A_BYTES + j * KG_BLOCK_BYTES, mB, fb, bn + 64 * j, k);
              if (SPLIT == SPLIT_A) {
                ptx::tma_load_2d(lo, mAlo, fb, am, k);
                ptx::tma_load_2d(lo + KG_BLOCK_BYTES, mAlo, fb, am + 64, k);
              } else if (SPLIT == SPLIT_B) {
                for (int j = 0; j < nblk; ++j) ptx::tma_load_2d(lo + j * KG_BLOCK_BYTES, mBlo, fb, bn + 64 * j, k);
              }
            }
          } else if constexpr (MX) {
            // E4M3 A and B tiles (128 K values = 128 bytes per row) and the
            // two scale atoms of this 128-row x 128-K stage.  B rows: the
            // packed gate/up matrix holds 64 gate and 64 up rows per 64 h
            // columns, so the tile of h columns [n0, n0 + 64) starts at row 2 n0
            const int k = kb * MX_BK;
            const int brow = EPI == EPI_SWIGLU_FWD ? 2 * ti.n0 : ti.n0;
            uint8_t* sf = sSF + stage * MX_SF_BYTES;
            ptx::tma_load_2d(sA + stage * A_BYTES, mA, fb, k, am);
            ptx::tma_load_3d(sB + stage * B_BYTES, mB, fb, k, brow, g);
            ptx::bulk_load(sf, mx_sfa + ((long long)(am >> 7) * mx_nkq + kb) * 512, 512, fb);
            ptx::bulk_load(sf + 512, mx_sfb + ((long long)(brow >> 7) * mx_nkq + kb) * 512, 512, fb);
          } else {
            const int part = nsplit == 2 ? (kb & 1) : 0;
            const int k = k0 + (nsplit == 2 ? (kb >> 1) : kb) * BK;
            uint8_t* a_dst = sA + stage * A_BYTES;
            uint8_t* b_dst = sB + stage * B_BYTES;
            const CUtensorMap* mAk = (part && mAlo) ? mAlo : mA;
            if (gat) {
              // the tile's 128 A rows, K columns [k, k + 64)
              const uint8_t* gsrc0 = g_src + (long long)k * 2 + g_chunk * 16;
              const int* rows = tail->gsrc[0];
#pragma unroll 8
              for (int i = 0; i < 32; ++i) {
                const int r = 4 * i + g_rg;
                ptx::cp_async_16(a_dst + r * 128 + ((g_chunk ^ (r & 7)) << 4), gsrc0 + (long long)rows[r] * g_pitch);
              }
            } else if (lead) {
              if (AMN == 0) {
                load_2d<PAIR>(a_dst, mAk, fb, fbl, k, am);
              } else {
                load_2d<PAIR>(a_dst, mAk, fb, fbl, am, k);
                load_2d<PAIR>(a_dst + MN_BLOCK_BYTES, mAk, fb, fbl, am + 64, k);
              }
            }
            if (lead) {
              if (EPI == EPI_SWIGLU_FWD) {
                // B tile = 128 h columns as two 64-column slices, each [64 rows
                // of W_g ; 64 rows of W_u] (accumulator columns: a | u | a | u,
                // 64 each); with a CTA pair each CTA holds one slice, so that a
                // and u of an h column stay in the same lanes of a folded
                // (half-tile) accumulator too
#pragma unroll
                for (int j = 0; j < 2 / PAIR; ++j) {
                  const int slice = PAIR == 1 ? j : rank;
                  uint8_t* dst = b_dst + j * (2 * MN_BLOCK_BYTES);
                  load_3d<PAIR>(dst, mB, fb, fbl, k, ti.n0 + 64 * slice, g);
                  load_3d<PAIR>(dst + MN_BLOCK_BYTES, mB2, fb, fbl, k, ti.n0 + 64 * slice, g);
                }
              } else if (BMN == 0) {
                load_3d<PAIR>(b_dst, mB, fb, fbl, k, bn, g);
              } else {
                const bool second = ksplit > 0 && k >= ksplit;
                const CUtensorMap* mBk = second ? mB2 : mB;
                const int kk = second ? k - ksplit : k;
                for (int j = 0; j < nblk; ++j) load_3d<PAIR>(b_dst + j * MN_BLOCK_BYTES, mBk, fb, fbl, bn + 64 * j, kk, g);
              }
            }
          }
          // GATHER: each lane's arrival fires once its copies have landed
          // (every stage, gathered or not: the barrier counts 32 of them)
          if (GATHER) ptx::cp_async_mbar_arrive(fb);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // copies still in flight land before the CTA's shared memory goes away
      if (GATHER) asm volatile("cp.async.wait_all;" ::: "memory");
      if (!ok && lead) {
        *abort_flag = 1;
        record_status(P.status, MOE_ERR_TIMEOUT);
        // let copies already in flight land before the CTA's shared memory goes
        // away (the leader's barriers count the peer's copies too)
        for (int s = 0; s < STAGES; ++s)
          if (rank == 0 && (issued_any & (1u << s))) {
            volatile int never = 0;
            ptx::mbar_wait_bounded(&tail->full[s], (issued_phase_mask >> s) & 1u, &never, 100000000ull);
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues everything: lane 0 of the CTA (PAIR = 2: of the
    // leader, whose full barriers count both CTAs' bytes and whose commits
    // arrive on the barriers of both CTAs).  The other lanes take part in the
    // TMEM allocation only: a warp-wide wait or sync inside this loop makes the
    // warp reconverge, which costs hundreds of cycles between MMA groups.
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        int t;
        if (dyn) {
          const int slot = it & (RING - 1);
          if (!ptx::mbar_wait_bounded(&tail->ring_full[slot], (it / RING) & 1, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          t = *reinterpret_cast<volatile int*>(&tail->ring[slot]);
          ptx::mbar_arrive(&tail->ring_empty[slot]);
        } else {
          t = tile0 + it * tile_step;
        }
        if (t >= total) break;
        TileInfo ti = decode<MODE, TILE_M, KBK, MBK>(P, S, t);
        const Problem& pr = P.prob[ti.p];
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!ptx::mbar_wait_cluster_bounded(&tail->tmem_empty[acc], acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        // per-tile values in registers (see the producer)
        const uint32_t idesc = ptx::idesc_bf16(ti.half ? BM : TILE_M, pr.mma_n, AMN, BMN);
        const int nk = ti.nk, k_left = ti.k1 - ti.k0;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait_bounded(&tail->full[stage], phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          // rows copied by cp.async (generic proxy) are read by the MMAs
          // (async proxy)
          if (GATHER) ptx::fence_proxy_async_smem();
          // Ragged K: the rows of a group's last step past its end are zeros
          // (per-group maps, or TMA's fill past `extent`), and a 16-row
          // sub-step entirely past the end is not issued.
          const bool tail_step = MODE == KGROUP && (kb + 1) * KBK > k_left;
          ptx::tc_fence_after();
          if (MODE == MGROUP && MX) {
            // the stage's scale atoms into this stage's tensor-memory columns,
            // then four K = 32 block-scaled MMAs (scale byte = K block)
            const uint32_t a_addr = ptx::smem_u32(sA + stage * A_BYTES);
            const uint32_t b_addr = ptx::smem_u32(sB + stage * B_BYTES);
            const uint32_t sf_t = tmem_base + MX_SF_COL + stage * 8;
            const uint32_t sf_s = ptx::smem_u32(sSF + stage * MX_SF_BYTES);
            ptx::tmem_cp_scales(sf_t, ptx::smem_desc_plain(sf_s, 128, 128));
            ptx::tmem_cp_scales(sf_t + 4, ptx::smem_desc_plain(sf_s + 512, 128, 128));
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const uint64_t ad = ptx::smem_desc(a_addr + s * 32, 16, 1024);
              const uint64_t bd = ptx::smem_desc(b_addr + s * 32, 16, 1024);
              ptx::mma_mxf8(d_tmem, ad, bd, ptx::idesc_mxf8(BM, MX_N, s), sf_t, sf_t + 4, (kb | s) != 0 ? 1u : 0u);
            }
            ptx::mma_commit(&tail->empty[stage]);
          } else if (MODE == MGROUP) {
            const uint32_t a_addr = ptx::smem_u32(sA + stage * A_BYTES);
            const uint32_t b_addr = ptx::smem_u32(sB + stage * B_BYTES);
#pragma unroll
            for (int s = 0; s < BK / UMMA_K; ++s) {
              const uint64_t ad = AMN ? ptx::smem_desc(a_addr + s * 2048, MN_BLOCK_BYTES, 1024)
                                      : ptx::smem_desc(a_addr + s * 32, 16, 1024);
              const uint64_t bd = BMN ? ptx::smem_desc(b_addr + s * 2048, MN_BLOCK_BYTES, 1024)
                                      : ptx::smem_desc(b_addr + s * 32, 16, 1024);
              if (PAIR == 1) ptx::mma_bf16(d_tmem, ad, bd, idesc, (kb | s) != 0 ? 1u : 0u);
              else ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | s) != 0 ? 1u : 0u);
            }
            if (PAIR == 1) ptx::mma_commit(&tail->empty[stage]);
            else ptx::mma_commit_pair(&tail->empty[stage], 0x3);
          } else {
            // KBK K rows: per 16-row sub-step one MMA, plus one with the lo half
            // of the split operand; a full step is one straight-line sequence
            const uint32_t sa = ptx::smem_u32(smem + stage * SC::BYTES), sb = sa + KG_A_BYTES,
                           sl = sb + KG_B_BYTES;
            constexpr int NSUB = KBK / UMMA_K;
            const int nsub = tail_step ? (k_left - kb * KBK + UMMA_K - 1) / UMMA_K : NSUB;
            auto sub_step = [&](int s) {
              const uint64_t as = ptx::smem_desc(sa + s * 2048, KG_BLOCK_BYTES, 1024);
              const uint64_t bs = ptx::smem_desc(sb + s * 2048, KG_BLOCK_BYTES, 1024);
              const uint32_t acc0 = (kb | s) != 0 ? 1u : 0u;
              ptx::mma_bf16(d_tmem, as, bs, idesc, acc0);
              if (SPLIT == SPLIT_A) ptx::mma_bf16(d_tmem, ptx::smem_desc(sl + s * 2048, KG_BLOCK_BYTES, 1024), bs, idesc, 1u);
              if (SPLIT == SPLIT_B) ptx::mma_bf16(d_tmem, as, ptx::smem_desc(sl + s * 2048, KG_BLOCK_BYTES, 1024), idesc, 1u);
            };
            if (nsub == NSUB) {
#pragma unroll
              for (int s = 0; s < NSUB; ++s) sub_step(s);
            } else {
              for (int s = 0; s < nsub; ++s) sub_step(s);
            }
            ptx::mma_commit(&tail->empty[stage]);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (nk > 0) {
          if (PAIR == 1) ptx::mma_commit(&tail->tmem_full[acc]);
          else ptx::mma_commit_pair(&tail->tmem_full[acc], 0x3);
        } else {
          ptx::mbar_arrive(&tail->tmem_full[acc]);
          if (PAIR == 2) ptx::mbar_arrive_remote(ptx::mapa(ptx::smem_u32(&tail->tmem_full[acc]), 1));
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(P.status, MOE_ERR_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w owns TMEM lanes [32q, 32q+32) (q = w % 4) = rows
    // [32q, 32q+32) of this CTA's 128 rows of the tile.  Each 32-column
    // accumulator chunk goes TMEM -> registers (row per thread) -> shared
    // memory -> quad layout (tmem_chunk_quad), so that all global traffic is
    // vectorised and coalesced.
    const int q = warp & 3;
    float* tb = &tail->tbuf[q][0];
    const unsigned FULL = 0xffffffffu;
    const int rs = lane >> 3;         // row within each group of four
    const int cq = (lane & 7) * 4;    // first of this lane's four columns
    // SwiGLU backward: a | u chunks of this warp's 32 rows arrive by TMA in a
    // two-buffer ring; au_next counts chunks issued, au_done chunks consumed
    uint32_t au_next = 0, au_done = 0;
    uint32_t n_stores = 0;  // EPI_BF16: TMA stores issued by this warp (staging boxes alternate)
    uint8_t* au_mine = au_buf + q * 2 * AU_CHUNK_BYTES;
    for (int it = 0;; ++it) {
      int t;
      if (!take_tile(it, t)) {
        *abort_flag = 1;
        record_status(P.status, MOE_ERR_TIMEOUT);
        break;
      }
      if (t >= total) break;
      TileInfo ti = decode<MODE, TILE_M, KBK, MBK>(P, S, t);
      const Problem& pr = P.prob[ti.p];
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      // first row (KGROUP: first M index) of this CTA.  A half tile's
      // accumulator is folded: warps 0-1 take the CTA's 64 rows for the
      // accumulator columns [0, N/2), warps 2-3 the same rows for [N/2, N),
      // which sit at TMEM columns [0, N/2) of lanes 64-127.
      const int m_cta = ti.m0 + (ti.half ? rank * (BM / 2) : row_half);
      const int ch = ti.half ? (q >> 1) : 0;
      const int row0 = m_cta + (ti.half ? (q & 1) : q) * 32;
      const int col_shift = ch * (pr.mma_n / 2);  // accumulator column at this warp's TMEM column 0
      // SwiGLU backward: chunk c of a | u (columns n0 + 32c of a and of u)
      const CUtensorMap* m_au = EPI == EPI_SWIGLU_BWD ? &P.maps[pr.map_aux] : nullptr;
      const int au_H = pr.H;
      // this warp's chunks [au_c0, au_c1) (a half tile's warp: its half of them)
      const int au_all = EPI == EPI_SWIGLU_BWD ? min(pr.n_tile, pr.N - ti.n0) / 32 : 0;
      const int au_c0 = ti.half ? min(au_all, col_shift / 32) : 0;
      const int au_c1 = ti.half ? min(au_all, au_c0 + pr.mma_n / 64) : au_all;
      auto au_issue = [&](int c) {
        const int buf = au_next & 1;
        if (lane == 0) {
          uint64_t* bar = &tail->au_full[q][buf];
          uint8_t* dst = au_mine + buf * AU_CHUNK_BYTES;
          ptx::mbar_arrive_expect_tx(bar, AU_CHUNK_BYTES);
          ptx::tma_load_2d(dst, m_au, bar, ti.n0 + 32 * c, row0);
          ptx::tma_load_2d(dst + AU_CHUNK_BYTES / 2, m_au, bar, au_H + ti.n0 + 32 * c, row0);
        }
        ++au_next;
      };
      if (EPI == EPI_SWIGLU_BWD) {
        // the first two chunks load while the main loop still runs
        for (int c = au_c0; c < au_c0 + 2 && c < au_c1; ++c) au_issue(c);
      }
      if (!ptx::mbar_wait_cluster_bounded(&tail->tmem_full[acc], acc_phase, abort_flag, kWaitLimitNs)) {
        *abort_flag = 1;
        record_status(P.status, MOE_ERR_TIMEOUT);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
      const int nrows = max(0, min(32, ti.rows_end - row0));
      const bool has_acc = ti.nk > 0;

      if (EPI == EPI_BF16) {
        // Ragged K, bf16 out: each 32-column chunk goes TMEM -> registers (one
        // row per thread) -> bf16 -> this warp's staging box in shared memory
        // (64-byte swizzle, two boxes in turn) -> TMA store of the 32 x 32 box.
        // The next chunk's TMEM load is in flight while a chunk is stored.
        static_assert(EPI != EPI_BF16 || MODE == KGROUP, "bf16 output: ragged-K GEMMs");
        const bool second = pr.row_split > 0 && m_cta >= pr.row_split;
        const CUtensorMap* mo = &P.maps[second ? pr.map_out2 : pr.map_out];
        const int orow = row0 - (second ? pr.row_split : 0);
        const int nch = min(pr.n_tile, pr.N - ti.n0) / 32;
        uint8_t* stage_box = reinterpret_cast<uint8_t*>(tb);
        if (row0 < ti.rows_end) {
          uint32_t r[2][32];
          if (has_acc) {
            ptx::tmem_ld32(taddr, r[0]);
            ptx::tmem_ld_wait(r[0]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[0][e] = 0u;
          }
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            if (c >= nch) break;
            uint32_t(&cur)[32] = r[c & 1];
            uint32_t(&nxt)[32] = r[(c + 1) & 1];
            if (c + 1 < nch) {
              if (has_acc) {
                ptx::tmem_ld32(taddr + 32 * (c + 1), nxt);
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) nxt[e] = 0u;
              }
            }
            // the box written two stores ago has been read by its TMA store
            uint8_t* box = stage_box + (n_stores & 1) * 2048;
            if (n_stores >= 2) {
              if (lane == 0) ptx::bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 v = make_uint4(
                  pack_bf16(__uint_as_float(cur[8 * j]), __uint_as_float(cur[8 * j + 1])),
                  pack_bf16(__uint_as_float(cur[8 * j + 2]), __uint_as_float(cur[8 * j + 3])),
                  pack_bf16(__uint_as_float(cur[8 * j + 4]), __uint_as_float(cur[8 * j + 5])),
                  pack_bf16(__uint_as_float(cur[8 * j + 6]), __uint_as_float(cur[8 * j + 7])));
              // row `lane` of the box, 16-byte piece j at its 64-byte-swizzle slot
              *reinterpret_cast<uint4*>(box + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = v;
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_3d(mo, box, ti.n0 + 32 * c, orow, ti.g);
              ptx::bulk_commit();
            }
            ++n_stores;
            if (has_acc && c + 1 < nch) ptx::tmem_ld_wait(nxt);
          }
        }
      } else if (EPI == EPI_F32) {
        long long base;  // element offset of (row0, 0)
        void* outv;
        if (MODE == KGROUP && pr.row_split > 0 && m_cta >= pr.row_split) {
          outv = pr.out2;
          base = ti.g * pr.gstride + (long long)(row0 - pr.row_split) * pr.ldo;
        } else {
          outv = pr.out;
          base = (MODE == KGROUP ? ti.g * pr.gstride : 0) + (long long)row0 * pr.ldo;
        }
        // out: fp32, or (out_f16) fp16 terms of a per-token sum
        // element offset of each of this thread's eight rows 4 j + rs (-1: not
        // stored): row base + r, or with a row map (ragged M) out_row_map[r]
        const bool mapped = MODE == MGROUP && pr.out_row_map != nullptr;
        long long roff[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = 4 * j + rs;
          roff[j] = -1;
          if (r < nrows) {
            if (mapped) {
              const int v = __ldg(pr.out_row_map + row0 + r);
              if (v < 0 || v >= pr.out_map_rows) record_status(P.status, MOE_ERR_DEVICE_BOUNDS);
              else roff[j] = (long long)v * pr.ldo;
            } else {
              roff[j] = base + (long long)r * pr.ldo;
            }
          }
        }
        const bool comb = MODE == MGROUP && pr.comb_y != nullptr;
        const float down = pr.out_scale ? pow2f(-grad_scale_exp(__ldg(pr.out_scale))) : 1.0f;
        const int ck = pr.comb_k;
        const __half* comb_o = reinterpret_cast<const __half*>(pr.comb_o);
        const int c_end = ti.half ? col_shift + pr.mma_n / 2 : pr.n_tile;
        for (int c0 = col_shift; c0 < c_end; c0 += 32) {
          if (ti.n0 + c0 >= pr.N) break;
          float4 v[8];
          if (has_acc) tmem_chunk_quad(taddr + c0 - col_shift, tb, lane, v);
          else zero_quad(v);
          const int col = ti.n0 + c0 + cq;
          if (col >= pr.N) continue;  // N is a multiple of 4
          if (EPI == EPI_F32 && pr.bias) {
            const float4 b = __ldg(reinterpret_cast<const float4*>(pr.bias + col));
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = make_float4(v[j].x + b.x, v[j].y + b.y, v[j].z + b.z, v[j].w + b.w);
          }
          if (comb) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 4 * j + rs;
              if (r >= nrows) continue;
              // token t = row0 + r: s rounded through fp16 (as the unfused
              // path stores it), then its kept slots' expert outputs, gate-
              // weighted, added in slot order (the combine's own order); a
              // non-finite sum (a term beyond the fp16 range) is reported
              float4 a = unpack_f16x4(f16x4(v[j]));
              const long long slot0 = (long long)(row0 + r) * ck;
              float4 o[kMaxK];
#pragma unroll
              for (int q = 0; q < kMaxK; ++q)
                if (q < ck) o[q] = unpack_f16x4(__ldg(reinterpret_cast<const uint2*>(comb_o + (slot0 + q) * pr.ldo + col)));
#pragma unroll
              for (int q = 0; q < kMaxK; ++q) {
                if (q >= ck) break;
                if (__ldg(pr.comb_row_of_slot + slot0 + q) < 0) continue;
                const float gq = __ldg(pr.comb_gates + slot0 + q);
                a = make_float4(fmaf(gq, o[q].x, a.x), fmaf(gq, o[q].y, a.y), fmaf(gq, o[q].z, a.z),
                                fmaf(gq, o[q].w, a.w));
              }
              if (!(isfinite(a.x) && isfinite(a.y) && isfinite(a.z) && isfinite(a.w)))
                record_status(P.status, MOE_ERR_RANGE);
              store4(reinterpret_cast<__nv_bfloat16*>(pr.comb_y) + (long long)(row0 + r) * pr.ldo + col, a);
            }
          } else if (pr.out_f16) {
            // fp16 terms of a per-token sum (gradient terms: divided by 2^e)
            __half* outp = reinterpret_cast<__half*>(outv) + col;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (roff[j] >= 0)
                *reinterpret_cast<uint2*>(outp + roff[j]) =
                    f16x4(make_float4(v[j].x * down, v[j].y * down, v[j].z * down, v[j].w * down));
          } else {
            float* outp = reinterpret_cast<float*>(outv) + col;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (roff[j] >= 0) store4(outp + roff[j], v[j]);
          }
        }
      } else if (EPI == EPI_SWIGLU_FWD && MX) {
        // MXFP8: accumulator columns [0,64) = a (the tile's 64 gate rows),
        // [64,128) = u; h = silu(a) u in fp32, quantized per row in blocks of
        // 32 h columns (one chunk: the row's 8 lanes reduce the block maximum
        // by shuffles) into E4M3 codes [rows, H] and the scale tile atoms
        uint8_t* hc = reinterpret_cast<uint8_t*>(pr.out);
        for (int c0 = 0; c0 < 64; c0 += 32) {
          float4 va[8], vu[8];
          tmem_chunk_quad(taddr + c0, tb, lane, va);
          tmem_chunk_quad(taddr + 64 + c0, tb, lane, vu);
          const int col = ti.n0 + c0 + cq;
          const int block = (ti.n0 + c0) >> 5;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = 4 * j + rs;
            const float4 a = va[j], u = vu[j];
            const float h0 = a.x * sigmoidf_(a.x) * u.x, h1 = a.y * sigmoidf_(a.y) * u.y;
            const float h2 = a.z * sigmoidf_(a.z) * u.z, h3 = a.w * sigmoidf_(a.w) * u.w;
            float amax = fmaxf(fmaxf(fabsf(h0), fabsf(h1)), fmaxf(fabsf(h2), fabsf(h3)));
            amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 4));
            const int se = mx_scale_exp(amax);
            const uint32_t codes = mx_codes4(h0, h1, h2, h3, mx_inv_scale(se));
            if (r < nrows) {
              const long long row = row0 + r;
              *reinterpret_cast<uint32_t*>(hc + row * pr.ldo + col) = codes;
              if (cq == 0) pr.out_sf[mx_atom_offset(row, block, pr.out_sf_nq)] = (uint8_t)(se + 127);
            }
          }
        }
      } else if (EPI == EPI_SWIGLU_FWD) {
        // accumulator columns a | u | a | u, 64 each: h columns [n0, n0+64)
        // then [n0+64, n0+128) (a half tile's warp: one of the two slices).
        // h goes out in bf16 (down-projection input; not stored when `out` is
        // NULL, the recompute of a and u for the backward), a and u in fp32
        __nv_bfloat16* hp = pr.out ? reinterpret_cast<__nv_bfloat16*>(pr.out) + (long long)row0 * pr.ldo + ti.n0
                                   : nullptr;
        float* ap = pr.aux ? reinterpret_cast<float*>(pr.aux) + (long long)row0 * pr.ld_aux + ti.n0 : nullptr;
        const int cc0 = ti.half ? 2 * ch : 0, cc1 = ti.half ? 2 * ch + 2 : 4;
        for (int cc = cc0; cc < cc1; ++cc) {
          // 32 h columns [32 cc, 32 cc + 32) of the tile: a at accumulator
          // column la, u at la + 64
          const int la = 128 * (cc >> 1) + 32 * (cc & 1);
          float4 va[8], vu[8];
          tmem_chunk_quad(taddr + la - col_shift, tb, lane, va);
          tmem_chunk_quad(taddr + la + 64 - col_shift, tb, lane, vu);
          const int c = 32 * cc + cq;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = 4 * j + rs;
            if (r < nrows) {
              const float4 a = va[j], u = vu[j];
              const float4 h = make_float4(a.x * sigmoidf_(a.x) * u.x, a.y * sigmoidf_(a.y) * u.y,
                                           a.z * sigmoidf_(a.z) * u.z, a.w * sigmoidf_(a.w) * u.w);
              if (hp) store4(hp + (long long)r * pr.ldo + c, h);
              if (ap) {
                store4(ap + (long long)r * pr.ld_aux + c, a);
                store4(ap + (long long)r * pr.ld_aux + pr.H + c, u);
              }
            }
          }
        }
      } else if (EPI == EPI_SWIGLU_BWD) {
        // accumulator = dY_perm W_d for H columns [n0, n0+256) (no gate yet);
        // au = fp32 a | u of the forward.  Per element:
        //   h = silu(a) u;  dg += acc * h;  dh = g acc;
        //   da = dh u sig(a) (1 + a (1 - sig(a)));  du = dh silu(a)
        // da | du go out as bf16 hi + lo, g*h as bf16 hi + lo (operands of the
        // weight-gradient GEMMs), and the gate-gradient partial per row.
        float g_mine = 1.0f;  // gate of row row0 + lane
        if (pr.gates && lane < nrows) {
          const int slot = __ldg(pr.slot_of_row + row0 + lane);
          if (slot < 0 || slot >= pr.gate_slots) {
            record_status(P.status, MOE_ERR_DEVICE_BOUNDS);
            g_mine = 0.0f;
          } else {
            g_mine = __ldg(pr.gates + slot);
          }
        }
        float gj[8], part[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          gj[j] = __shfl_sync(FULL, g_mine, 4 * j + rs);
          part[j] = 0.0f;
        }
        const int H = au_H;
        const long long ldo = pr.ldo;
        const long long ro = (long long)row0 * ldo + ti.n0;  // into [rows, 2H]
        const long long rh = (long long)row0 * H + ti.n0;    // into [rows, H]
        __nv_bfloat16* dhi = reinterpret_cast<__nv_bfloat16*>(pr.out) + ro;
        __nv_bfloat16* dlo = reinterpret_cast<__nv_bfloat16*>(pr.out_lo) + ro;
        __nv_bfloat16* ghh = reinterpret_cast<__nv_bfloat16*>(pr.gh_hi) + rh;
        __nv_bfloat16* ghl = reinterpret_cast<__nv_bfloat16*>(pr.gh_lo) + rh;
        bool au_ok = true;
        for (int c = au_c0; c < au_c1; ++c) {
          const int buf = au_done & 1;
          if (!ptx::mbar_wait_bounded(&tail->au_full[q][buf], (au_done >> 1) & 1, abort_flag, kWaitLimitNs)) {
            au_ok = false;
            break;
          }
          ++au_done;
          // a, u of this chunk: [32 rows][32 columns] fp32 each, quad layout
          const float* sa = reinterpret_cast<const float*>(au_mine + buf * AU_CHUNK_BYTES);
          const float* su = sa + 32 * 32;
          float4 ca[8], cu[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            ca[j] = *reinterpret_cast<const float4*>(sa + (4 * j + rs) * 32 + cq);
            cu[j] = *reinterpret_cast<const float4*>(su + (4 * j + rs) * 32 + cq);
          }
          // the buffer is read: chunk c + 2 may overwrite it
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (c + 2 < au_c1) au_issue(c + 2);
          float4 vd[8];
          tmem_chunk_quad(taddr + 32 * c - col_shift, tb, lane, vd);
          const int col = 32 * c + cq;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = 4 * j + rs;
            if (r < nrows) {
              const float a[4] = {ca[j].x, ca[j].y, ca[j].z, ca[j].w}, u[4] = {cu[j].x, cu[j].y, cu[j].z, cu[j].w};
              const float dv[4] = {vd[j].x, vd[j].y, vd[j].z, vd[j].w};
              float da[4], du[4], gh[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float sg = sigmoidf_(a[e]);
                const float si = a[e] * sg;
                const float h = si * u[e];
                part[j] = fmaf(dv[e], h, part[j]);
                const float dh = gj[j] * dv[e];
                da[e] = dh * u[e] * sg * (1.0f + a[e] * (1.0f - sg));
                du[e] = dh * si;
                gh[e] = gj[j] * h;
              }
              const long long o2 = (long long)r * ldo + col;
              const long long o1 = (long long)r * H + col;
              split_store4(dhi + o2, dlo + o2, make_float4(da[0], da[1], da[2], da[3]));
              split_store4(dhi + o2 + H, dlo + o2 + H, make_float4(du[0], du[1], du[2], du[3]));
              split_store4(ghh + o1, ghl + o1, make_float4(gh[0], gh[1], gh[2], gh[3]));
            }
          }
        }
        if (!au_ok) {
          *abort_flag = 1;
          record_status(P.status, MOE_ERR_TIMEOUT);
          break;
        }
        if (pr.dgp) {
          // sum each row's partials over its eight lanes; two slots per
          // column tile, one per accumulator-column half (a full tile puts
          // its whole sum in the first and 0 in the second)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float v = part[j];
            v += __shfl_xor_sync(FULL, v, 1);
            v += __shfl_xor_sync(FULL, v, 2);
            v += __shfl_xor_sync(FULL, v, 4);
            const int r = 4 * j + rs;
            if ((lane & 7) == 0 && r < nrows) {
              float* slot = pr.dgp + (long long)(row0 + r) * pr.ld_dgp + 2 * (ti.n0 / pr.n_tile);
              if (ti.half) {
                slot[ch] = v;
              } else {
                slot[0] = v;
                slot[1] = 0.0f;
              }
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR == 1 || rank == 0) ptx::mbar_arrive(&tail->tmem_empty[acc]);
        else ptx::mbar_arrive_remote(ptx::mapa(ptx::smem_u32(&tail->tmem_empty[acc]), 0));
      }
    }
    // TMA stores still reading their staging box (or in flight) complete
    // before the CTA's shared memory goes away
    if (EPI == EPI_BF16 && lane == 0) ptx::bulk_wait_all();
    // after an abort: let a | u copies still in flight land before the CTA's
    // shared memory goes away
    if (EPI == EPI_SWIGLU_BWD) {
      volatile int never = 0;
      for (; au_done < au_next; ++au_done)
        ptx::mbar_wait_bounded(&tail->au_full[q][au_done & 1], (au_done >> 1) & 1, &never, 100000000ull);
    }
  }

  __syncthreads();
  if (PAIR == 2) ptx::cluster_sync();  // no remote arrive is still in flight to a CTA that exits
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<PAIR>(tmem_base, TMEM_COLS);
  }
}

}  // namespace gemm
}  // namespace moe
