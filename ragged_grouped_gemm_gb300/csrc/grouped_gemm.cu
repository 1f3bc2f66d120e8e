// Persistent, warp-specialised tcgen05 grouped GEMM for sm_103a.
//
// Roles (320 threads, one CTA per SM):
//   warp 0      TMA producer: one lane streams A/B k-blocks into a ring of
//               shared-memory stages (128-byte swizzle), signalled by
//               mbarriers with transaction counts.
//   warp 1      TMEM owner and MMA issuer: one lane issues
//               tcgen05.mma.cta_group::1.kind::f16 (M=128, N=BN, K=16) into a
//               double-buffered fp32 accumulator in tensor memory and commits
//               stage releases and accumulator hand-offs to mbarriers.
//   warps 2..9  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31 = tile rows, and half (w-2)/4 of the columns),
//               apply the fused epilogue and store.
// The accumulator is double-buffered, so the epilogue of tile i overlaps the
// main loop of tile i+1.  Tiles are walked in a persistent loop; for the
// ragged-M form the tile list is derived on the device from the group
// offsets (prefix of per-group tile counts), so a launch needs no host-side
// knowledge of the group sizes.
//
// CTA-pair form (PAIR, bf16 operands): a cluster of two CTAs on two SMs
// shares one 256 x BN tile through tcgen05.mma.cta_group::2 (M = 256).  Each
// CTA loads its own 128 rows of the output's A operand and half of the B tile
// (B columns 0..BN/2-1 in rank 0, the rest in rank 1), so each SM streams
// half of the B bytes it would need alone.  Rank 0's MMA lane issues for the
// pair and its commits arrive on both CTAs' stage-release and
// accumulator-ready barriers (multicast).  Both CTAs' TMA loads complete on
// rank 0's stage barrier, except (ragged K) a k-block whose group ends off a
// 16-row boundary: that one lands on each CTA's own barrier, and the peer's
// idle MMA warp zeroes its rows past the group's end and forwards the stage
// to rank 0.  Each CTA's epilogue reads its own 128 TMEM lanes and signals
// rank 0's accumulator-free barrier.  TMEM is allocated and freed by both
// CTAs together, between cluster barriers.
//
// fp32 outputs of the ragged-M forms leave through TMA tensor stores: each
// epilogue warp stages 16 rows x 32 columns (whole 128-byte rows) at a time
// in 2 KB of shared memory, or 32 x 16 when a tile's column halves are 16
// wide.  The weight gradients (ragged K) have 4 KB per warp: the one-SM form
// double-buffers its 16 x 32 boxes; the CTA-pair form stages 32 x 32 and
// writes it with plain coalesced stores, which leaves the TMA unit to the
// operand loads.
//
// Shared-memory operand layouts (both 1024-byte aligned per stage):
//   K-major : rows of 64 bf16 (128 B), 8-row swizzle atoms of 1024 B;
//             descriptor SBO = 1024, advance 32 B per K=16 step.
//   MN-major: per 64-wide MN atom a region of kb K-rows x 128 B (kb = 64,
//             or 128 for the weight gradients on CTA pairs: eight K=16 MMAs
//             per stage barrier, 5-9% faster than four on one expert's dW);
//             descriptor LBO = kb x 128 (next MN atom), SBO = 1024 (next 8
//             K-rows), advance 2048 B per K=16 step.
#include "grouped_gemm.cuh"
#include "sm100_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BKR = 128;   // k-block rows of the bf16 weight gradients on CTA pairs
constexpr int kThreads = 320;        // producer, MMA, 8 epilogue warps
constexpr int kThreadsQ = 448;       // + 4 scale-factor warps (MXFP8 operands)
constexpr int kThreadsW8 = 576;      // + 8 converter warps (FP8 weights)
constexpr int kConvWarps = 8;
constexpr int kEpiThreads = 256;
constexpr int kSfWarps = 4;

constexpr int kMaxGroups = 1024;
constexpr int kABytes = BM * BK * 2;   // 16 KB

struct KParams {
  CUtensorMap tmA[2];    // A per contraction source (MXFP8: codes)
  CUtensorMap tmB[2];    // B per source, or the W1 | W3 halves of a dual-N tile (MXFP8: codes)
  CUtensorMap tmAs[2];   // MXFP8: A scales per source
  CUtensorMap tmBs[2];   // MXFP8: B scales (per source or per half)
  CUtensorMap tmC;       // fp32 output map {n, m, group}, used when c_tma != 0
  int32_t c_tma;
  int32_t c_rows;        // rows of the output map (ragged M, one group)
  const int32_t* offsets;
  int32_t num_groups;
  int32_t m_size;
  int32_t n_size;
  int32_t kb0, kb1;
  int32_t kblk;          // contraction elements per k-block (64 bf16, 128 MXFP8)
  int32_t ksplit;        // ragged M, one group: contraction slices (tile-minor); 0 or 1 = none
  int32_t b_dual_n;
  int32_t tile_n;
  void* out0;
  void* out1;
  void* out2;
  void* out3;
  void* out4;
  int64_t s_ld;
  const void* in0;
  const void* in1;
  int64_t ld_out;
  int64_t group_stride_out;
  int32_t* status;
  // FP8 weights: fp32 scale per 128 x 128 tile of each weight matrix
  // [rows][cols] (K-major B: rows = n; MN-major B: rows = k), per source or
  // per dual-N half, [groups][ceil(rows/128)][ceil(cols/128)]
  const float* wscale[2];
  int32_t ws_cols;       // column tiles per matrix
  int64_t ws_gstride;    // tiles per matrix
  // GATHER: A row r of the ragged-M problem is row a_gather[r] / gather_k of
  // the token matrix behind tmA[0] (a 2-D map with one-row boxes)
  const int32_t* a_gather;
  int32_t gather_k;
  // Ragged K (bf16), several groups: per-group copies of tmA[0] / tmB[0]
  // whose rows are exactly the group's rows ([0, G) for A, [G, 2G) for B),
  // written by build_group_maps_kernel before the launch; null with one group
  // (the whole-tensor maps end at the group's end already)
  const CUtensorMap* gmaps;
};

// The per-group maps of a ragged-K launch: thread g writes group g's copy of
// the A and B maps, rebased to the group's first row with a row extent of
// the group's row count (at least 1; an empty group is never loaded).
__global__ void build_group_maps_kernel(CUtensorMap* out, const __grid_constant__ CUtensorMap ta,
                                        const __grid_constant__ CUtensorMap tb, const int32_t* __restrict__ offsets,
                                        int G, const char* a_ptr, int64_t a_ld_bytes, const char* b_ptr,
                                        int64_t b_ld_bytes) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= G) return;
  const int r0 = offsets[g];
  const uint32_t rows = static_cast<uint32_t>(max(offsets[g + 1] - r0, 1));
  tensormap_rebase_rows(out + g, &ta, reinterpret_cast<uint64_t>(a_ptr + static_cast<int64_t>(r0) * a_ld_bytes),
                        rows);
  tensormap_rebase_rows(out + G + g, &tb, reinterpret_cast<uint64_t>(b_ptr + static_cast<int64_t>(r0) * b_ld_bytes),
                        rows);
}

// STG: the kernel stages fp32 output blocks for TMA stores (weight gradients)
// MAXG / MAXS: the most groups the shared-memory tables hold and the most
// ring stages.  MAXG = 0: no tables (the bf16 ragged-K form reads the group
// offsets from global memory), and the room goes to 4 KB of fp32 staging per
// epilogue warp: two 2 KB TMA-store buffers (one-SM form) or one 32 x 32 box
// for plain stores (CTA-pair form)
template <int BN, bool QUANT = false, bool PAIR = false, bool W8 = false, bool STG = false, int MAXG = kMaxGroups,
          int MAXS = 6>
struct Cfg {
  // FP8 weights (W8): the B codes of a k-block (BN x 64 bytes) land in a
  // two-slot staging ring; converters write the bf16 B tile into the stage
  static constexpr int kW8Slots = W8 ? 2 : 0;
  static constexpr int kW8SlotBytes = BN * 64;
  // MXFP8 (QUANT) stage, one k-block of 128 E4M3 elements = 4 scale blocks:
  //   A codes [128][128] | B codes [BN][128] (both 128-byte swizzled) |
  //   A scale rows [4][144] (from a 16-aligned row) | B scale rows [4][BN] |
  //   scale atoms for tcgen05.cp: A 512 B, B 2 x 512 B
  // (CTA pair, ragged M: this CTA holds half of the B tile's codes, all of
  // its scale rows)
  static constexpr int kQBRows = PAIR ? BN / 2 : BN;
  static constexpr int kQBCodes = BM * 128;
  static constexpr int kQARaw = kQBCodes + kQBRows * 128;
  static constexpr int kQBRaw = kQARaw + 640;
  static constexpr int kQAtoms = kQBRaw + 4 * BN;
  static constexpr uint32_t kQTxBytes = BM * 128 + kQBRows * 128 + 4 * 144 + 4 * BN;    // ragged M
  static constexpr uint32_t kQTxBytesK = BM * 128 + BN * 128 + 4 * 128 + 4 * BN;   // ragged K
  // bf16: PAIR = this CTA holds half of the B tile (the pair shares a 256-row tile)
  // k-block length: 128 rows for the bf16 ragged-K form on CTA pairs (eight
  // K=16 MMAs per stage barrier instead of four), 64 elsewhere
  static constexpr int kKb = (MAXG == 0 && PAIR && !QUANT && !W8) ? BKR : BK;
  static constexpr int kABytesC = BM * kKb * 2;   // A bytes of a bf16 stage
  static constexpr int kStageBytes =
      QUANT ? (kQAtoms + 1536 + 1023) / 1024 * 1024 : (BM + (PAIR ? BN / 2 : BN)) * kKb * 2;
  // shared memory left for the stages: 227 KB less the alignment slack, the
  // staging buffers, the barriers (at most MAXS stages) and the group tables
  static constexpr bool kWideStaging = STG && MAXG == 0;
  static constexpr int kEpiWarpBytes = kWideStaging ? 4096 : 2048;
  static constexpr int kEpiBytes = STG ? 8 * kEpiWarpBytes : 0;
  static constexpr int kTableBytes = MAXG > 0 ? 2 * 4 * (MAXG + 1) : 0;
  static constexpr int kStageBudget = 232448 - 1024 - kEpiBytes - (3 * MAXS + 2 * 2 + 5) * 8 - 16 -
                                      kTableBytes - kW8Slots * kW8SlotBytes;
  static constexpr int kStagesRaw = kStageBudget / kStageBytes;
  static constexpr int kStages = kStagesRaw > MAXS ? MAXS : kStagesRaw;
  // accumulators (2 x BN columns) and, for MXFP8, one 16-column scale buffer per stage
  static constexpr uint32_t kTmemCols = QUANT ? 512 : ((2 * BN < 32) ? 32 : 2 * BN);
  static constexpr uint32_t kSfCol = 2 * BN;
  // stages | W8 code slots | fp32 staging (8 warps x kEpiWarpBytes, STG only) |
  // barriers (2S, + S scale-ready for MXFP8, + 5) | tmem base, abort | offsets[G+1] | prefix[G+1]
  static constexpr int kW8Off = kStages * kStageBytes;
  static constexpr int kEpiOff = kW8Off + kW8Slots * kW8SlotBytes;
  static constexpr int kBarOff = kEpiOff + kEpiBytes;
  static constexpr int kMiscOff = kBarOff + ((QUANT ? 3 : 2) * kStages + 2 * kW8Slots + 5) * 8;
  static constexpr int kOffOff = kMiscOff + 16;
  static constexpr int kMaxG = MAXG;
  static constexpr size_t smem_bytes(int groups) {
    return 1024 + kOffOff + (MAXG > 0 ? 2 * 4 * (groups + 1) : 0);
  }
  static_assert(kStages >= 2, "shared memory holds fewer than two stages");
  static_assert(smem_bytes(MAXG) <= 232448, "shared memory above 227 KB");
  static_assert(!QUANT || 2 * BN + 16 * kStages <= 512, "accumulators and scale buffers exceed tensor memory");
};

// The configuration of each kernel form: the bf16 ragged-K (weight-gradient)
// form keeps no group tables and has 4 KB of fp32 staging per epilogue warp.
template <int BN, bool A_MN, int EPI, bool QUANT, bool PAIR, bool W8>
using KernelCfg = Cfg<BN, QUANT, PAIR, W8, EPI == EPI_F32, (A_MN && !QUANT && !W8) ? 0 : kMaxGroups>;

struct Tile {
  int g, mt, nt;
  int row0;        // ragged M: first permuted row of the tile; ragged K: first row of the group
  int m0;          // ragged K: first output row of this CTA's 128 rows
  int rows_valid;  // valid output rows of this CTA's 128 (may be <= 0 in a CTA pair)
  int k_rows;      // ragged K: rows of the group (contraction length)
  int num_kb;
  int kbeg;        // ragged M: first k-block of this tile's contraction slice
  int split;       // ragged M: contraction slice (partial-output index)
};

// Ragged K: the group of a tile (tiles of a group are consecutive: its M
// tiles times its N tiles) and the tile from the group's first and
// one-past-last rows.
template <int BN, bool PAIR>
__device__ __forceinline__ int rk_group(int tile, const KParams& p) {
  constexpr int UR = PAIR ? 2 * BM : BM;
  return tile / (((p.m_size + UR - 1) / UR) * ((p.n_size + BN - 1) / BN));
}

template <int BN, bool PAIR>
__device__ __forceinline__ Tile decode_tile_rk(int tile, const KParams& p, int off0, int off1, int rank) {
  Tile t;
  constexpr int UR = PAIR ? 2 * BM : BM;
  const int prank = rank & 1;
  const int ntiles = (p.n_size + BN - 1) / BN;
  const int per_g = ((p.m_size + UR - 1) / UR) * ntiles;
  t.kbeg = 0;
  t.split = 0;
  t.g = tile / per_g;
  const int rem = tile - t.g * per_g;
  t.mt = rem / ntiles;
  t.nt = rem - t.mt * ntiles;
  t.row0 = off0;
  t.m0 = t.mt * UR + prank * BM;
  t.k_rows = off1 - off0;
  t.rows_valid = min(BM, p.m_size - t.m0);
  t.num_kb = (t.k_rows + p.kblk - 1) / p.kblk;
  return t;
}

// rank: the CTA's rank in its cluster; bit 0 picks its 128 rows of a pair
// tile.
template <bool RAGGED_K, int BN, bool PAIR = false>
__device__ __forceinline__ Tile decode_tile(int tile, const KParams& p, const int* s_off, const int* s_pre,
                                            int rank = 0) {
  Tile t;
  constexpr int UR = PAIR ? 2 * BM : BM;   // rows of one M unit (a CTA pair covers 256)
  const int prank = rank & 1;
  t.kbeg = 0;
  t.split = 0;
  if (!RAGGED_K) {
    if (p.ksplit > 1) {   // the slices of one output tile are adjacent in the tile order
      t.split = tile % p.ksplit;
      tile /= p.ksplit;
    }
    // Expert-major raster: expert, then N tile, then M tile (innermost), so the
    // CTAs running at once share one expert's rows of A (L2-resident) and each
    // weight block is streamed from HBM once.  s_pre holds the prefix of
    // per-expert tile counts mtiles_g * ntiles.
    int lo = 0, hi = p.num_groups;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pre[mid] <= tile) lo = mid; else hi = mid;
    }
    t.g = lo;
    const int mtiles = max(0, s_off[lo + 1] - s_off[lo] + UR - 1) / UR;
    const int rem = tile - s_pre[lo];
    t.nt = rem / mtiles;
    t.mt = rem - t.nt * mtiles;
    t.row0 = s_off[lo] + t.mt * UR + prank * BM;
    t.rows_valid = min(BM, s_off[lo + 1] - t.row0);
    t.m0 = 0;
    t.k_rows = 0;
    t.num_kb = p.kb0 + p.kb1;
    if (p.ksplit > 1) {   // slices of ceil(kb / ksplit) k-blocks; the host makes none empty
      const int kbs = (t.num_kb + p.ksplit - 1) / p.ksplit;
      t.kbeg = t.split * kbs;
      t.num_kb = max(0, min(kbs, t.num_kb - t.kbeg));
    }
  } else {
    t = decode_tile_rk<BN, PAIR>(tile, p, s_off[rk_group<BN, PAIR>(tile, p)], s_off[rk_group<BN, PAIR>(tile, p) + 1],
                                 rank);
  }
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float sigmoidf_fast(float a) { return 1.0f / (1.0f + __expf(-a)); }

// 16 E4M3 codes (little-endian in a uint4) times an fp32 tile scale ->
// 8 bf16x2 words: each decoded value (exact in fp32) times the scale, the
// fp32 product rounded to bf16 (round to nearest even).
__device__ __forceinline__ void dequant16_scaled(const uint4 c, float sc, uint32_t (&w)[8]) {
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const __half2_raw hr =
          __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(cw[i] >> (16 * hh)), __NV_E4M3);
      __half2 h2;
      *reinterpret_cast<__half2_raw*>(&h2) = hr;
      const float2 f = __half22float2(h2);
      w[2 * i + hh] = pack_bf16x2(f.x * sc, f.y * sc);
    }
  }
}

__device__ __forceinline__ int mx_exponent_of(float amax) {
  if (!(amax > 0.0f)) return -127;
  const uint32_t b = __float_as_uint(amax);
  const int ex = static_cast<int>(b >> 23);
  const int fl = ex ? ex - 127 : -149 + (31 - __clz(static_cast<int>(b)));
  return max(-127, min(127, fl - 8));
}

// GATHER (ragged M, bf16, one contraction source): A rows are gathered from
// the token matrix through p.a_gather by TMA tile::gather4, four rows per
// instruction, every lane of the producer warp taking four of the tile's
// 128 rows; no permuted copy of the tokens is read.
template <int BN, bool A_MN, bool B_MN, int EPI, bool QUANT, bool PAIR, bool W8 = false, bool GATHER = false>
__global__ void __launch_bounds__(QUANT ? kThreadsQ : (W8 ? kThreadsW8 : kThreads), 1)
    grouped_gemm_kernel(const __grid_constant__ KParams p) {
  static_assert(!GATHER || (!A_MN && !B_MN && !QUANT && !W8), "GATHER: K-major bf16 ragged-M forms");
  using C = KernelCfg<BN, A_MN, EPI, QUANT, PAIR, W8>;
  // bf16: the MN-major-A form is the ragged-K (weight-gradient) form.  MXFP8
  // operands are always K-major; A_MN then only selects the ragged-K form.
  constexpr bool RAGGED_K = A_MN;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + S;
  uint64_t* sready = empty + S;           // MXFP8: scale atoms of the stage built
  uint64_t* wfull = sready + (QUANT ? S : 0);   // FP8 weights: code slot loaded
  uint64_t* wempty = wfull + C::kW8Slots;       // FP8 weights: code slot consumed
  uint64_t* tfull = wempty + C::kW8Slots;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
  // group offsets: a shared copy, or (no tables) the caller's array itself
  int* s_tab = reinterpret_cast<int*>(smem + C::kOffOff);
  const int* s_off = C::kMaxG > 0 ? s_tab : p.offsets;
  int* s_pre = s_tab + (p.num_groups + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.num_groups;
  // CTA pair (2-SM MMA): the even CTA of the pair issues the MMAs for both
  constexpr int CN = PAIR ? 2 : 1;   // CTAs per cluster
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = (rank & 1) == 0;
  const uint32_t lead = static_cast<uint32_t>(rank & ~1);   // cluster rank of the pair's leader
  const int unit0 = static_cast<int>(blockIdx.x) / CN;
  const int ustride = static_cast<int>(gridDim.x) / CN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // TMA (tx bytes), the converter threads, or (ragged-K pair, rank 0) this
      // CTA's TMA plus the peer's forwarded arrival
      // (FP8 weights: A's TMA bytes plus one arrival per converter warp)
      mbar_init(&full[s], W8 ? 1 + kConvWarps : 1);
      mbar_init(&empty[s], 1);
    }
    // the scale warp that builds the stage (CTA pair: that of each CTA, on the leader's barrier)
    for (int s = 0; s < (QUANT ? S : 0); ++s) mbar_init(&sready[s], PAIR ? 2 : 1);
    for (int s = 0; s < C::kW8Slots; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], kConvWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], (PAIR ? 2 : 1) * (kEpiThreads / 32));   // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA[0]);
    tma_prefetch_desc(&p.tmB[0]);
    if (QUANT) {
      tma_prefetch_desc(&p.tmAs[0]);
      tma_prefetch_desc(&p.tmBs[0]);
    }
  }
  if (warp == 1) {
    if (PAIR) {   // collective: one warp of each CTA of the pair
      tmem_alloc_pair(s_tmem, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(s_tmem, C::kTmemCols);
      tmem_relinquish();
    }
  }
  // group offsets and (ragged M) the prefix of per-group tile counts
  // (128-row M tiles times N tiles)
  if (C::kMaxG > 0)
    for (int i = threadIdx.x; i <= G; i += blockDim.x) s_tab[i] = p.offsets[i];
  __syncthreads();
  if (!RAGGED_K && warp == 0) {
    const int ntiles = (p.n_size + p.tile_n - 1) / p.tile_n;
    const int per = (G + 31) / 32;
    const int lo = lane * per;
    const int hi = min(G, lo + per);
    int sum = 0;
    constexpr int UR = PAIR ? 2 * BM : BM;
    for (int g = lo; g < hi; ++g) sum += max(0, s_off[g + 1] - s_off[g] + UR - 1) / UR * ntiles;
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - sum;
    for (int g = lo; g < hi; ++g) {
      s_pre[g] = run;
      run += max(0, s_off[g + 1] - s_off[g] + UR - 1) / UR * ntiles;
    }
    if (lane == 31) s_pre[G] = incl;
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();   // the peer's barriers are initialised and its TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  int total_tiles;
  if (!RAGGED_K) {
    total_tiles = s_pre[G] * (p.ksplit > 1 ? p.ksplit : 1);
  } else {
    constexpr int UR = PAIR ? 2 * BM : BM;
    const int mtiles = (p.m_size + UR - 1) / UR;
    total_tiles = G * mtiles * ((p.n_size + BN - 1) / BN);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (QUANT && lane == 0) {
      // MXFP8 operands: E4M3 codes (128-byte swizzled, straight to the MMA) and
      // the raw scale rows of each 128-element k-block
      uint32_t it = 0;
      bool ok = true;
      for (int tile = unit0; ok && tile < total_tiles; tile += ustride) {
        const Tile t = decode_tile<RAGGED_K, BN, PAIR>(tile, p, s_off, s_pre, rank);
        for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, s_abort, p.status, 100 + s)) { ok = false; break; }
          uint8_t* st = smem + s * C::kStageBytes;
          if (RAGGED_K) {
            // weight gradient: A [M][tokens] and B [N][tokens] codes (tokens of
            // each group padded to 128 with zero codes), scales [tokens/32][M or N]
            mbar_arrive_expect_tx(&full[s], C::kQTxBytesK);
            const int k0 = t.row0 + kb * 128;
            tma_load_2d(st, &p.tmA[0], &full[s], k0, t.m0);
            tma_load_2d(st + C::kQARaw, &p.tmAs[0], &full[s], t.m0, k0 / 32);
            tma_load_2d(st + C::kQBCodes, &p.tmB[0], &full[s], k0, t.nt * BN);
            tma_load_2d(st + C::kQBRaw, &p.tmBs[0], &full[s], t.nt * BN, k0 / 32);
            continue;
          }
          mbar_arrive_expect_tx(&full[s], C::kQTxBytes);
          const int src = (kb < p.kb0) ? 0 : 1;
          const int k0 = (src == 0 ? kb : kb - p.kb0) * 128;
          tma_load_2d(st, &p.tmA[src], &full[s], k0, t.row0);
          tma_load_2d(st + C::kQARaw, &p.tmAs[src], &full[s], t.row0 & ~15, k0 / 32);   // 16-byte aligned x
          // CTA pair: this CTA's half of the B codes (W1 or W3 for the dual-N
          // tile), and every B scale row (each CTA's tensor memory needs them all)
          if (p.b_dual_n) {
            const int f0 = t.nt * (BN / 2);
            if (PAIR) {
              tma_load_3d(st + C::kQBCodes, &p.tmB[rank & 1], &full[s], k0, f0, t.g);
            } else {
              tma_load_3d(st + C::kQBCodes, &p.tmB[0], &full[s], k0, f0, t.g);
              tma_load_3d(st + C::kQBCodes + (BN / 2) * 128, &p.tmB[1], &full[s], k0, f0, t.g);
            }
            tma_load_3d(st + C::kQBRaw, &p.tmBs[0], &full[s], f0, k0 / 32, t.g);
            tma_load_3d(st + C::kQBRaw + 2 * BN, &p.tmBs[1], &full[s], f0, k0 / 32, t.g);
          } else {
            tma_load_3d(st + C::kQBCodes, &p.tmB[src], &full[s], k0, t.nt * BN + (PAIR ? (rank & 1) * (BN / 2) : 0),
                        t.g);
            tma_load_3d(st + C::kQBRaw, &p.tmBs[src], &full[s], t.nt * BN, k0 / 32, t.g);
          }
        }
      }
      for (int s = 0; s < S; ++s) {
        if (it > static_cast<uint32_t>(s)) {
          const uint32_t last = s + S * ((it - 1 - s) / S);
          mbar_wait_drain(&full[s], (last / S) & 1u);
        }
      }
    } else if (GATHER) {
      // Gathered A: lane l loads the tile's rows 4l..4l+3 (token row
      // a_gather[r] / gather_k; a row past the group's end loads token row 0,
      // whose products the epilogue never stores) by one gather4 into its
      // 512-byte quarter-atom of the stage; lane 0 waits for the stage, arms
      // the barrier and loads B.
      uint32_t it = 0;
      bool ok = true;
      for (int tile = unit0; ok && tile < total_tiles; tile += ustride) {
        const Tile t = decode_tile<false, BN, PAIR>(tile, p, s_off, s_pre, rank);
        const int gend = s_off[t.g + 1];
        int rr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = t.row0 + 4 * lane + j;
          rr[j] = r < gend ? __ldg(p.a_gather + r) / p.gather_k : 0;
        }
        for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1u;
          int okl = 1;
          if (lane == 0) okl = mbar_wait_bounded(&empty[s], ph ^ 1u, s_abort, p.status, 100 + s) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, okl, 0)) {
            ok = false;
            break;
          }
          uint8_t* sA = smem + s * C::kStageBytes;
          uint8_t* sB = sA + (RAGGED_K ? C::kABytesC : kABytes);
          const int k0 = kb * BK;
          if (PAIR) {
            if (leader && lane == 0) mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
            const uint32_t bar = mapa_shared(smem_u32(&full[s]), lead);
            __syncwarp();
            tma_gather4_pair(sA + lane * 512, &p.tmA[0], bar, k0, rr[0], rr[1], rr[2], rr[3]);
            if (lane == 0) {
              if (p.b_dual_n) tma_load_3d_pair(sB, &p.tmB[rank], bar, k0, t.nt * (BN / 2), t.g);
              else tma_load_3d_pair(sB, &p.tmB[0], bar, k0, t.nt * BN + rank * (BN / 2), t.g);
            }
          } else {
            if (lane == 0) mbar_arrive_expect_tx(&full[s], C::kStageBytes);
            __syncwarp();
            tma_gather4(sA + lane * 512, &p.tmA[0], &full[s], k0, rr[0], rr[1], rr[2], rr[3]);
            if (lane == 0) {
              if (p.b_dual_n) {
                const int f0 = t.nt * (BN / 2);
                tma_load_3d(sB, &p.tmB[0], &full[s], k0, f0, t.g);
                tma_load_3d(sB + (BN / 2) * 128, &p.tmB[1], &full[s], k0, f0, t.g);
              } else {
                tma_load_3d(sB, &p.tmB[0], &full[s], k0, t.nt * BN, t.g);
              }
            }
          }
        }
      }
      // every stage's last armed load has landed before the CTA exits (for a
      // pair the leader's barriers count both CTAs' copies)
      if (lane == 0 && (!PAIR || leader)) {
        for (int s = 0; s < S; ++s) {
          if (it > static_cast<uint32_t>(s)) {
            const uint32_t last = s + S * ((it - 1 - s) / S);
            mbar_wait_drain(&full[s], (last / S) & 1u);
          }
        }
      }
      __syncwarp();
    } else if (!QUANT && lane == 0) {
      uint32_t it = 0;
      int map_g = -1;   // ragged K: the group whose maps this thread last acquired
      bool ok = true;
      for (int tile = unit0; ok && tile < total_tiles; tile += ustride) {
        const Tile t = decode_tile<RAGGED_K, BN, PAIR>(tile, p, s_off, s_pre, rank);
        for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, s_abort, p.status, 100 + s)) { ok = false; break; }
          uint8_t* sA = smem + s * C::kStageBytes;
          uint8_t* sB = sA + (RAGGED_K ? C::kABytesC : kABytes);
          if (W8) {
            // FP8 weights: A (bf16) straight into the stage; the B codes of the
            // k-block into a staging slot for the converters
            const int src = (kb < p.kb0) ? 0 : 1;
            const int k0 = (src == 0 ? kb : kb - p.kb0) * BK;
            mbar_arrive_expect_tx(&full[s], kABytes);
            tma_load_2d(sA, &p.tmA[src], &full[s], k0, t.row0);
            const uint32_t wit = it;   // one code slot use per k-block
            const int ws_ = wit % C::kW8Slots;
            if (!mbar_wait_bounded(&wempty[ws_], ((wit / C::kW8Slots) & 1u) ^ 1u, s_abort, p.status, 130 + ws_)) {
              ok = false;
              break;
            }
            uint8_t* q = smem + C::kW8Off + ws_ * C::kW8SlotBytes;
            mbar_arrive_expect_tx(&wfull[ws_], C::kW8SlotBytes);
            if (!B_MN) {
              if (p.b_dual_n) {
                const int f0 = t.nt * (BN / 2);
                tma_load_3d(q, &p.tmB[0], &wfull[ws_], k0, f0, t.g);
                tma_load_3d(q + (BN / 2) * 64, &p.tmB[1], &wfull[ws_], k0, f0, t.g);
              } else {
                tma_load_3d(q, &p.tmB[src], &wfull[ws_], k0, t.nt * BN, t.g);
              }
            } else {
#pragma unroll
              for (int a = 0; a < BN / 64; ++a)
                tma_load_3d(q + a * 4096, &p.tmB[src], &wfull[ws_], t.nt * BN + 64 * a, k0, t.g);
            }
            continue;
          }
          if (RAGGED_K) {
            // The group's own maps end at its last row, so its last k-block
            // reads zeros past the group's end (TMA fill) instead of the next
            // group's rows.  One group: the whole-tensor maps do the same.
            const bool gm = p.gmaps != nullptr;
            const CUtensorMap* mA = gm ? p.gmaps + t.g : &p.tmA[0];
            const CUtensorMap* mB = gm ? p.gmaps + G + t.g : &p.tmB[0];
            if (gm && t.g != map_g) {
              tensormap_acquire(mA);
              tensormap_acquire(mB);
              map_g = t.g;
            }
            const int r = gm ? kb * C::kKb : t.row0 + kb * C::kKb;   // rows of the group's map
            if (PAIR) {
              // both CTAs' loads complete on the leader's barrier, armed by the leader
              const int n0 = t.nt * BN + (rank & 1) * (BN / 2);
              if (leader) mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
              const uint32_t bar = mapa_shared(smem_u32(&full[s]), lead);
              tma_load_2d_pair(sA, mA, bar, t.m0, r);
              tma_load_2d_pair(sA + C::kKb * 128, mA, bar, t.m0 + 64, r);
#pragma unroll
              for (int a = 0; a < BN / 128; ++a) tma_load_2d_pair(sB + a * C::kKb * 128, mB, bar, n0 + 64 * a, r);
            } else {
              mbar_arrive_expect_tx(&full[s], C::kStageBytes);
              tma_load_2d(sA, mA, &full[s], t.m0, r);
              tma_load_2d(sA + 8192, mA, &full[s], t.m0 + 64, r);
#pragma unroll
              for (int a = 0; a < BN / 64; ++a) tma_load_2d(sB + a * 8192, mB, &full[s], t.nt * BN + 64 * a, r);
            }
            continue;
          }
          if (PAIR && !RAGGED_K) {
            // both CTAs' loads complete on the leader's barrier, armed by the leader
            if (leader) mbar_arrive_expect_tx(&full[s], 2 * C::kStageBytes);
            const uint32_t bar = mapa_shared(smem_u32(&full[s]), lead);
            const int src = (kb < p.kb0) ? 0 : 1;
            const int k0 = (src == 0 ? kb : kb - p.kb0) * BK;
            tma_load_2d_pair(sA, &p.tmA[src], bar, k0, t.row0);
            if (!B_MN) {
              if (p.b_dual_n) tma_load_3d_pair(sB, &p.tmB[rank], bar, k0, t.nt * (BN / 2), t.g);  // W1 | W3 half
              else tma_load_3d_pair(sB, &p.tmB[src], bar, k0, t.nt * BN + rank * (BN / 2), t.g);
            } else {
#pragma unroll
              for (int a = 0; a < BN / 128; ++a)
                tma_load_3d_pair(sB + a * 8192, &p.tmB[src], bar, t.nt * BN + rank * (BN / 2) + 64 * a, k0, t.g);
            }
            continue;
          }
          mbar_arrive_expect_tx(&full[s], C::kStageBytes);
          if (!RAGGED_K) {
            const int kbg = t.kbeg + kb;   // k-block within the whole contraction
            const int src = (kbg < p.kb0) ? 0 : 1;
            const int k0 = (src == 0 ? kbg : kbg - p.kb0) * BK;
            tma_load_2d(sA, &p.tmA[src], &full[s], k0, t.row0);
            // B maps of the ragged-M form are always 3-D: {cols, rows, group}
            if (!B_MN) {
              if (p.b_dual_n) {
                const int f0 = t.nt * (BN / 2);
                tma_load_3d(sB, &p.tmB[0], &full[s], k0, f0, t.g);
                tma_load_3d(sB + (BN / 2) * 128, &p.tmB[1], &full[s], k0, f0, t.g);
              } else {
                tma_load_3d(sB, &p.tmB[src], &full[s], k0, t.nt * BN, t.g);
              }
            } else {
#pragma unroll
              for (int a = 0; a < BN / 64; ++a)
                tma_load_3d(sB + a * 8192, &p.tmB[src], &full[s], t.nt * BN + 64 * a, k0, t.g);
            }
          }
        }
      }
      // Wait (bounded) for every stage's last armed load so that no copy is
      // still landing in shared memory when the CTA exits (for a pair the
      // leader's barriers count both CTAs' copies).
      for (int s = 0; s < S && (!PAIR || leader); ++s) {
        if (it > static_cast<uint32_t>(s)) {
          const uint32_t last = s + S * ((it - 1 - s) / S);
          mbar_wait_drain(&full[s], (last / S) & 1u);
        }
      }
      for (int s = 0; s < C::kW8Slots; ++s) {
        if (it > static_cast<uint32_t>(s)) {
          const uint32_t last = s + C::kW8Slots * ((it - 1 - s) / C::kW8Slots);
          mbar_wait_drain(&wfull[s], (last / C::kW8Slots) & 1u);
        }
      }
    }
  } else if (PAIR && warp == 1 && !leader) {
    // the leader CTA issues the pair's MMAs; this warp has nothing to do
  } else if (warp == 1 && QUANT) {
    // ------------------------------------------------------------ MMA issuer (MXFP8)
    // Per k-block: the scale atoms go to tensor memory by tcgen05.cp, then four
    // block-scaled MMAs (K = 32 each) select scale byte 0..3.  Both are issued
    // by the same thread, so the copies are ordered before the MMAs.
    uint32_t it = 0, tcount = 0;
    bool ok = true;
    for (int tile = unit0; ok && tile < total_tiles; tile += ustride, ++tcount) {
      const Tile t = decode_tile<RAGGED_K, BN, PAIR>(tile, p, s_off, s_pre, rank);
      const uint32_t buf = tcount & 1u;
      const uint32_t aph = (tcount >> 1) & 1u;
      if (!mbar_wait_bounded(&tempty[buf], aph ^ 1u, s_abort, p.status, 200)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1u;
        if (!mbar_wait_bounded(&sready[s], ph, s_abort, p.status, 320 + s)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint8_t* st = smem + s * C::kStageBytes;
          // one 16-column scale buffer per stage (A: +0..3, B: +4..11): a buffer is
          // rewritten only after the MMAs that read it have completed (stage release)
          const uint32_t sf = tmem_base + C::kSfCol + s * 16;
          const uint32_t atoms = smem_u32(st + C::kQAtoms);
          if (PAIR) {   // each CTA's atoms to its own tensor memory
            tc_cp_32x128b_warpx4_pair(sf, atoms);
            tc_cp_32x128b_warpx4_pair(sf + 4, atoms + 512);
            if (BN > 128) tc_cp_32x128b_warpx4_pair(sf + 8, atoms + 1024);
          } else {
            tc_cp_32x128b_warpx4(sf, atoms);
            tc_cp_32x128b_warpx4(sf + 4, atoms + 512);
            if (BN > 128) tc_cp_32x128b_warpx4(sf + 8, atoms + 1024);
          }
          const uint32_t a_base = smem_u32(st);
          const uint32_t b_base = smem_u32(st + C::kQBCodes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b_base + kk * 32, 16, 1024);
            if (PAIR)
              tc_mma_mxf8_pair(d_tmem, ad, bd, idesc_mxf8(2 * BM, BN, kk), sf, sf + 4, (kb > 0 || kk > 0) ? 1u : 0u);
            else
              tc_mma_mxf8(d_tmem, ad, bd, idesc_mxf8(BM, BN, kk), sf, sf + 4, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          if (PAIR) tc_commit_pair_mc(&empty[s], 3);
          else tc_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {
        if (PAIR) tc_commit_pair_mc(&tfull[buf], static_cast<uint16_t>(3u << lead));
        else if (t.num_kb > 0) tc_commit(&tfull[buf]);
        else mbar_arrive(&tfull[buf]);
      }
      __syncwarp();
    }
    if (lane == 0) {
      if (PAIR) tc_commit_pair_mc(mma_done, static_cast<uint16_t>(1u << lead));
      else tc_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * BM : BM, BN, A_MN, B_MN);
    uint32_t it = 0, tcount = 0;
    bool ok = true;
    // ragged K: the next tile's group offsets (global memory) are loaded
    // before this tile's k-blocks are issued and used only after them, so
    // their latency falls while the MMAs run instead of between tiles
    int nx0 = 0, nx1 = 0;
    if (RAGGED_K && unit0 < total_tiles) {
      const int g = rk_group<BN, PAIR>(unit0, p);
      nx0 = s_off[g];
      nx1 = s_off[g + 1];
    }
    for (int tile = unit0; ok && tile < total_tiles; tile += ustride, ++tcount) {
      const Tile t = RAGGED_K ? decode_tile_rk<BN, PAIR>(tile, p, nx0, nx1, rank)
                              : decode_tile<RAGGED_K, BN, PAIR>(tile, p, s_off, s_pre, rank);
      if (RAGGED_K && tile + ustride < total_tiles) {
        const int g = rk_group<BN, PAIR>(tile + ustride, p);
        nx0 = s_off[g];
        nx1 = s_off[g + 1];
      }
      const uint32_t buf = tcount & 1u;
      const uint32_t aph = (tcount >> 1) & 1u;
      if (!mbar_wait_bounded(&tempty[buf], aph ^ 1u, s_abort, p.status, 200)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * BN;
      for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1u;
        if (!mbar_wait_bounded(&full[s], ph, s_abort, p.status, 300 + s)) { ok = false; break; }
        tc_fence_after();
        uint8_t* sA = smem + s * C::kStageBytes;
        uint8_t* sB = sA + (RAGGED_K ? C::kABytesC : kABytes);
        // Ragged K: rows past the group's end arrive as zeros (the per-group
        // maps end at the group's last row); K=16 steps holding none of the
        // group's rows are skipped.
        constexpr int KB = RAGGED_K ? C::kKb : BK;
        const int rv = t.k_rows - kb * KB;
        const int nkk = (RAGGED_K && rv < KB) ? (rv + 15) / 16 : KB / 16;
        if (lane == 0) {
          const uint32_t a_base = smem_u32(sA);
          const uint32_t b_base = smem_u32(sB);
          for (int kk = 0; kk < nkk; ++kk) {
            const uint64_t ad = A_MN ? smem_desc_sw128(a_base + kk * 2048, KB * 128, 1024)
                                     : smem_desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(b_base + kk * 2048, KB * 128, 1024)
                                     : smem_desc_sw128(b_base + kk * 32, 16, 1024);
            if (PAIR) tc_mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            else tc_mma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          if (PAIR) tc_commit_pair_mc(&empty[s], 3);
          else tc_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {
        if (PAIR) tc_commit_pair_mc(&tfull[buf], static_cast<uint16_t>(3u << lead));
        else if (t.num_kb > 0) tc_commit(&tfull[buf]);
        else mbar_arrive(&tfull[buf]);
      }
      __syncwarp();
    }
    // every MMA issued by this CTA has completed before TMEM is released
    if (lane == 0) {
      if (PAIR) tc_commit_pair_mc(mma_done, static_cast<uint16_t>(1u << lead));
      else tc_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
    __syncwarp();
  } else if (warp >= 10) {
    // ------------------------------------------------------------ scale atoms (MXFP8)
    // Rearrange the stage's raw scale rows ([block][row]) into the 512-byte
    // atoms tcgen05.cp expects: for row r, byte j (scale block) of 32-bit word
    // (r/32)%4 of 16-byte row r%32; one atom per 128 rows of A or of B.
    // Warp w of the kSfWarps builds the whole of every stage s with
    // s % kSfWarps == w, so consecutive stages are built at once; lane l
    // writes 16-byte row l of each atom (rows l, l+32, l+64, l+96).  A warp
    // owns whole stages and meets each of their fills in order: a parity
    // wait must never skip a phase of its barrier.
    if (QUANT) {
      const int sfw = warp - 10;
      uint32_t it = 0;
      bool ok = true;
      for (int tile = unit0; ok && tile < total_tiles; tile += ustride) {
        const Tile t = decode_tile<RAGGED_K, BN, PAIR>(tile, p, s_off, s_pre, rank);
        // A scale rows: ragged M [4][144] from a 16-aligned row; ragged K [4][128]
        const int a_rem = RAGGED_K ? 0 : (t.row0 & 15);
        constexpr int AS = RAGGED_K ? 128 : 144;
        for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
          const int s = it % S;
          if (s % kSfWarps != sfw) continue;
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait_bounded(&full[s], ph, s_abort, p.status, 500 + s)) { ok = false; break; }
          uint8_t* st = smem + s * C::kStageBytes;
          const uint8_t* ra = st + C::kQARaw;
          const uint8_t* rb = st + C::kQBRaw;
          const uint32_t atoms = smem_u32(st + C::kQAtoms);
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = a_rem + lane + 32 * i;
            w[i] = static_cast<uint32_t>(ra[r]) | (static_cast<uint32_t>(ra[AS + r]) << 8) |
                   (static_cast<uint32_t>(ra[2 * AS + r]) << 16) | (static_cast<uint32_t>(ra[3 * AS + r]) << 24);
          }
          st_shared_v4(atoms + lane * 16, w[0], w[1], w[2], w[3]);
          // dual N: rows [0, BN/2) from the W1 scale rows, the rest from W3's
          const int w_ = p.b_dual_n ? BN / 2 : BN;
#pragma unroll
          for (int a = 0; a < (BN + 127) / 128; ++a) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = 128 * a + lane + 32 * i;
              const int half = p.b_dual_n ? (r >= BN / 2 ? 1 : 0) : 0;
              const uint8_t* src = rb + half * 2 * BN + (r - half * (BN / 2));
              w[i] = r < BN ? (static_cast<uint32_t>(src[0]) | (static_cast<uint32_t>(src[w_]) << 8) |
                               (static_cast<uint32_t>(src[2 * w_]) << 16) | (static_cast<uint32_t>(src[3 * w_]) << 24))
                            : 0u;
            }
            st_shared_v4(atoms + 512 + a * 512 + lane * 16, w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // CTA pair: the leader copies both CTAs' atoms; the peer's arrival
            // releases its atom writes at cluster scope
            if (PAIR && !leader) mbar_arrive_remote_release(mapa_shared(smem_u32(&sready[s]), lead));
            else mbar_arrive(&sready[s]);
          }
        }
      }
    }
    if (W8) {
      // ---------------------------------------------------------- converters (FP8 weights)
      // Each k-block: wait for its code slot and for the stage to be free,
      // write the bf16 B tile (dequantised value = E4M3 code x its 128 x 128
      // tile scale, rounded to bf16) in the 128-byte-swizzled layout of the
      // MMA, release the slot and arrive on the stage.
      const int ct = threadIdx.x - 10 * 32;   // 0..255
      uint32_t it = 0;
      bool ok = true;
      for (int tile = unit0; ok && tile < total_tiles; tile += ustride) {
        const Tile t = decode_tile<RAGGED_K, BN, PAIR>(tile, p, s_off, s_pre, rank);
        for (int kb = 0; kb < t.num_kb; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1u;
          const int ws_ = it % C::kW8Slots;
          if (!mbar_wait_bounded(&wfull[ws_], (it / C::kW8Slots) & 1u, s_abort, p.status, 540 + ws_)) {
            ok = false;
            break;
          }
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, s_abort, p.status, 560 + s)) { ok = false; break; }
          const int src = (kb < p.kb0) ? 0 : 1;
          const int k0 = (src == 0 ? kb : kb - p.kb0) * BK;
          const uint8_t* q = smem + C::kW8Off + ws_ * C::kW8SlotBytes;
          uint8_t* sB = smem + s * C::kStageBytes + kABytes;
          const int64_t gbase = static_cast<int64_t>(t.g) * p.ws_gstride;
          // rows / columns past the weight matrix hold zero codes (TMA fill):
          // clamp their tile index into this matrix's tile grid
          const int rtiles = static_cast<int>(p.ws_gstride / p.ws_cols);
          // BN rows (K-major) or 4 MN atoms x 64 k-rows (MN-major), 4 chunks of 16 codes each
          for (int task = ct; task < BN * 4; task += kConvWarps * 32) {
            const int j = task & 3;
            const int row = task >> 2;   // K-major: tile row n; MN-major: atom * 64 + k
            uint4 codes;
            float sc;
            uint8_t* rowp;
            int sw;
            if (!B_MN) {
              codes = *reinterpret_cast<const uint4*>(q + row * 64 + j * 16);
              const int half = p.b_dual_n ? row / (BN / 2) : 0;
              const int wrow = p.b_dual_n ? t.nt * (BN / 2) + (row - half * (BN / 2)) : t.nt * BN + row;
              const float* ss = p.wscale[p.b_dual_n ? half : src];
              sc = ss[gbase + static_cast<int64_t>(min(wrow / 128, rtiles - 1)) * p.ws_cols + min(k0 / 128, p.ws_cols - 1)];
              rowp = sB + row * 128;
              sw = row & 7;
            } else {
              const int a = row >> 6, k = row & 63;
              codes = *reinterpret_cast<const uint4*>(q + a * 4096 + k * 64 + j * 16);
              const int ncol = t.nt * BN + a * 64 + j * 16;
              sc = p.wscale[src][gbase + static_cast<int64_t>(min((k0 + k) / 128, rtiles - 1)) * p.ws_cols +
                                 min(ncol / 128, p.ws_cols - 1)];
              rowp = sB + a * 8192 + k * 128;
              sw = k & 7;
            }
            uint32_t w[8];
            dequant16_scaled(codes, sc, w);
            *reinterpret_cast<uint4*>(rowp + (((2 * j) ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(rowp + (((2 * j + 1) ^ sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&wempty[ws_]);
            mbar_arrive(&full[s]);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quarter = tile rows 32q..32q+31
    const int hf = (warp - 2) >> 2;   // column half of the tile
    const int r = q * 32 + lane;
    uint32_t tcount = 0;
    uint32_t nstore = 0;   // TMA stores this warp has issued (fp32 staging)
    for (int tile = unit0; tile < total_tiles; tile += ustride, ++tcount) {
      const Tile t = decode_tile<RAGGED_K, BN, PAIR>(tile, p, s_off, s_pre, rank);
      const uint32_t buf = tcount & 1u;
      const uint32_t aph = (tcount >> 1) & 1u;
      if (!mbar_wait_bounded(&tfull[buf], aph, s_abort, p.status, 400)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + buf * BN + (static_cast<uint32_t>(q * 32) << 16);
      const bool row_ok = r < t.rows_valid;
      if (EPI == EPI_BF16 || EPI == EPI_F32) {
        int64_t grow;
        char* obase = static_cast<char*>(p.out0);
        if (!RAGGED_K) {
          grow = t.row0 + r;
        } else {
          grow = static_cast<int64_t>(t.m0) + r;
          obase += static_cast<int64_t>(t.g) * p.group_stride_out * (EPI == EPI_F32 ? 4 : 2);
        }
        const bool zero = t.num_kb == 0;
        const int c_begin = hf * (BN / 2);
        if (EPI == EPI_F32 && C::kWideStaging && PAIR && p.c_tma && (BN / 2) % 32 == 0) {
          // Weight gradients on CTA pairs: the warp's 32 rows x 32 columns go to a 4 KB
          // shared buffer (one row per lane, 128-byte swizzle: 16-byte chunk j
          // of row r at chunk j ^ (r & 7)) and leave by plain 16-byte stores,
          // lane l writing chunk l % 8 of rows l / 8 + 4j, so each store
          // instruction covers four whole 128-byte lines (L2 evict-first: the
          // fp32 output is written once).  The TMA unit then carries only the
          // operand loads: the output is a quarter of the bytes a tile moves,
          // and as TMA stores it delayed the loads behind them (this form is
          // tensor-bound; the one-SM form, bound by its output stores, keeps
          // the TMA stores below).  The TMEM
          // load of the next 32 columns is in flight meanwhile.  (c_tma: the
          // output's rows start 16-byte aligned.)
          constexpr int NCH = BN / 64;
          const uint32_t stg = smem_u32(smem + C::kEpiOff + (warp - 2) * C::kEpiWarpBytes);
          const uint64_t pol = policy_evict_first();
          const int rows = RAGGED_K ? p.m_size : p.c_rows;
          float* gbase = reinterpret_cast<float*>(obase);
          const int c8 = lane & 7;
          uint32_t va[16], vb[16], vc[16], vd[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) va[j] = vb[j] = vc[j] = vd[j] = 0u;
          if (!zero) {
            tmem_ld_32x32b_x16(tb + c_begin, va);
            tmem_ld_32x32b_x16(tb + c_begin + 16, vb);
            tmem_wait_ld(va);
            reg_fence(vb);
          }
#pragma unroll
          for (int i = 0; i < NCH; ++i) {
            if (!zero && i + 1 < NCH) {
              tmem_ld_32x32b_x16(tb + c_begin + 32 * (i + 1), vc);
              tmem_ld_32x32b_x16(tb + c_begin + 32 * (i + 1) + 16, vd);
            }
            const int col = t.nt * BN + c_begin + 32 * i;
            const int row = (RAGGED_K ? t.m0 : t.row0) + q * 32;
            if (col < p.n_size && row < rows) {   // uniform across the warp
#pragma unroll
              for (int j = 0; j < 4; ++j)
                st_shared_v4(stg + lane * 128 + ((j ^ (lane & 7)) << 4), va[4 * j], va[4 * j + 1], va[4 * j + 2],
                             va[4 * j + 3]);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                st_shared_v4(stg + lane * 128 + (((j + 4) ^ (lane & 7)) << 4), vb[4 * j], vb[4 * j + 1],
                             vb[4 * j + 2], vb[4 * j + 3]);
              __syncwarp();
              const int gc = col + 4 * c8;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int r2 = (lane >> 3) + 4 * j;
                uint32_t x0, x1, x2, x3;
                ld_shared_v4(stg + r2 * 128 + ((c8 ^ (r2 & 7)) << 4), x0, x1, x2, x3);
                if (row + r2 < rows && gc < p.n_size) {
                  float* dst = gbase + static_cast<int64_t>(row + r2) * p.ld_out + gc;
                  if (gc + 4 <= p.n_size) {
                    st_global_v4_hint(dst, x0, x1, x2, x3, pol);
                  } else {   // the output's last columns
                    dst[0] = __uint_as_float(x0);
                    if (gc + 1 < p.n_size) dst[1] = __uint_as_float(x1);
                    if (gc + 2 < p.n_size) dst[2] = __uint_as_float(x2);
                  }
                }
              }
              __syncwarp();
            }
            if (i + 1 < NCH) {
              if (!zero) {
                tmem_wait_ld(vc);
                reg_fence(vd);
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                va[j] = vc[j];
                vb[j] = vd[j];
              }
            }
          }
        } else if (EPI == EPI_F32 && p.c_tma && (BN / 2) % 32 == 0) {
          // Stage this warp's 32 rows x 32 columns as two 16-row halves in a
          // 2 KB shared-memory buffer (128-byte swizzle: 16-byte chunk j of
          // row r at chunk j ^ (r & 7)) and write each half with a TMA tensor
          // store of 16 full 128-byte rows, which clips rows and columns
          // outside the output (evict-first in L2: the fp32 output is written
          // once and not read back).  The TMEM load of the next 32 columns is
          // in flight while these are staged.  With two buffers (4 KB of
          // staging) a warp waits only for the store before the last to have
          // read its buffer; a box that starts past the output is neither
          // staged nor stored, so the buffers alternate over the stores
          // actually issued.
          constexpr int NCH = BN / 64;
          constexpr int NB = C::kWideStaging ? 2 : 1;
          uint8_t* stg0 = smem + C::kEpiOff + (warp - 2) * C::kEpiWarpBytes;
          uint32_t va[16], vb[16], vc[16], vd[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) va[j] = vb[j] = vc[j] = vd[j] = 0u;
          if (!zero) {
            tmem_ld_32x32b_x16(tb + c_begin, va);
            tmem_ld_32x32b_x16(tb + c_begin + 16, vb);
            tmem_wait_ld(va);
            reg_fence(vb);
          }
          const int rr = lane & 15;
#pragma unroll
          for (int i = 0; i < NCH; ++i) {
            if (!zero && i + 1 < NCH) {
              tmem_ld_32x32b_x16(tb + c_begin + 32 * (i + 1), vc);
              tmem_ld_32x32b_x16(tb + c_begin + 32 * (i + 1) + 16, vd);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // boxes that start past the output's last column or row hold nothing to write
              const int col = t.nt * BN + c_begin + 32 * i;
              const int row = (RAGGED_K ? t.m0 : t.row0) + q * 32 + 16 * h;
              const int rows = RAGGED_K ? p.m_size : p.c_rows;
              if (!(col < p.n_size && row < rows)) continue;   // uniform across the warp
              uint8_t* stg = stg0 + (NB == 2 ? (nstore & 1u) * 2048 : 0);
              const uint32_t stg_addr = smem_u32(stg);
              if (lane == 0) {   // the store that last used this buffer has read it
                if (NB == 2) bulk_wait_group_read1();
                else bulk_wait_group_read0();
              }
              __syncwarp();
              if ((lane >> 4) == h) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  st_shared_v4(stg_addr + rr * 128 + ((j ^ (rr & 7)) << 4), va[4 * j], va[4 * j + 1],
                               va[4 * j + 2], va[4 * j + 3]);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  st_shared_v4(stg_addr + rr * 128 + (((j + 4) ^ (rr & 7)) << 4), vb[4 * j], vb[4 * j + 1],
                               vb[4 * j + 2], vb[4 * j + 3]);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d_hint(&p.tmC, stg, col, row, RAGGED_K ? t.g : t.split, policy_evict_first());
                bulk_commit_group();
              }
              ++nstore;
            }
            if (i + 1 < NCH) {
              if (!zero) {
                tmem_wait_ld(vc);
                reg_fence(vd);
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                va[j] = vc[j];
                vb[j] = vd[j];
              }
            }
          }
        } else if (EPI == EPI_F32 && p.c_tma) {
          // 16-column form of the above for tiles whose column halves are not
          // a multiple of 32 wide: 32 rows x 16 columns per 2 KB buffer
          // (64-byte swizzle: chunk j of row r at chunk j ^ ((r >> 1) & 3)).
          constexpr int NCH = BN / 32;
          uint8_t* stg = smem + C::kEpiOff + (warp - 2) * C::kEpiWarpBytes;
          const uint32_t stg_addr = smem_u32(stg);
          uint32_t va[16], vb[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) va[j] = vb[j] = 0u;
          if (!zero) {
            tmem_ld_32x32b_x16(tb + c_begin, va);
            tmem_wait_ld(va);
          }
#pragma unroll
          for (int i = 0; i < NCH; ++i) {
            if (!zero && i + 1 < NCH) tmem_ld_32x32b_x16(tb + c_begin + 16 * (i + 1), vb);
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j)
              st_shared_v4(stg_addr + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), va[4 * j], va[4 * j + 1],
                           va[4 * j + 2], va[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int col = t.nt * BN + c_begin + 16 * i;
              const int row = RAGGED_K ? t.m0 + q * 32 : t.row0 + q * 32;
              const int rows = RAGGED_K ? p.m_size : p.c_rows;
              if (col < p.n_size && row < rows) {
                tma_store_3d_hint(&p.tmC, stg, col, row, RAGGED_K ? t.g : t.split, policy_evict_first());
                bulk_commit_group();
              }
            }
            if (i + 1 < NCH) {
              if (!zero) tmem_wait_ld(vb);
#pragma unroll
              for (int j = 0; j < 16; ++j) va[j] = vb[j];
            }
          }
        } else {
#pragma unroll 1
          for (int c = c_begin; c < c_begin + BN / 2; c += 16) {
            uint32_t v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0u;
            if (!zero) {
              tmem_ld_32x32b_x16(tb + c, v);
              tmem_wait_ld(v);
            }
            const int col = t.nt * BN + c;
            if (row_ok && col < p.n_size) {
              const int nvalid = min(16, p.n_size - col);
              if (EPI == EPI_F32) {
                float* dst = reinterpret_cast<float*>(obase) + grow * p.ld_out + col;
                if (nvalid == 16 && (p.ld_out & 3) == 0) {
#pragma unroll
                  for (int j = 0; j < 4; ++j)
                    reinterpret_cast<uint4*>(dst)[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                } else {
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    if (j < nvalid) dst[j] = __uint_as_float(v[j]);
                }
              } else {
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(obase) + grow * p.ld_out + col;
                uint32_t w[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                if (nvalid == 16) {
                  reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                  reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                } else {
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    if (j < nvalid) dst[j] = __float2bfloat16_rn(__uint_as_float(v[j]));
                }
              }
            }
          }
        }
      } else if (EPI == EPI_SWIGLU_FWD) {
        const int64_t grow = t.row0 + r;
        const int f0 = t.nt * (BN / 2);
#pragma unroll 1
        for (int c = hf * (BN / 4); c < (hf + 1) * (BN / 4); c += 16) {
          uint32_t u[16], v[16];
          tmem_ld_32x32b_x16(tb + c, u);
          tmem_ld_32x32b_x16(tb + BN / 2 + c, v);
          tmem_wait_ld(u);
          reg_fence(v);
          const int col = f0 + c;
          if (row_ok && col < p.n_size) {
            uint32_t hw[8], aw[8], bw[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float a0 = __uint_as_float(u[2 * j]), a1 = __uint_as_float(u[2 * j + 1]);
              const float b0 = __uint_as_float(v[2 * j]), b1 = __uint_as_float(v[2 * j + 1]);
              hw[j] = pack_bf16x2(a0 * sigmoidf_fast(a0) * b0, a1 * sigmoidf_fast(a1) * b1);
              aw[j] = pack_bf16x2(a0, a1);
              bw[j] = pack_bf16x2(b0, b1);
            }
            const int64_t off = grow * p.ld_out + col;
            uint4* h = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out0) + off);
            h[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            h[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
            if (p.out1) {
              uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out1) + off);
              d[0] = make_uint4(aw[0], aw[1], aw[2], aw[3]);
              d[1] = make_uint4(aw[4], aw[5], aw[6], aw[7]);
            }
            if (p.out2) {
              uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out2) + off);
              d[0] = make_uint4(bw[0], bw[1], bw[2], bw[3]);
              d[1] = make_uint4(bw[4], bw[5], bw[6], bw[7]);
            }
          }
        }
      } else if (EPI == EPI_SWIGLU_FWD_Q) {
        // h = silu(a1) * a3 per row, quantised to MXFP8 in 32-column blocks
        // (each thread owns a row, so a block's amax is thread-local)
        const int64_t grow = t.row0 + r;
        const int f0 = t.nt * (BN / 2);
        // 32-column quantisation blocks of the BN/2 f columns, alternating between
        // the two warps of this lane quarter
#pragma unroll 1
        for (int c = 32 * hf; c < BN / 2; c += 64) {
          const int col = f0 + c;
          const bool ok = row_ok && col < p.n_size;
          const int64_t off = grow * p.ld_out + col;
          float h[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t u[16], v[16];
            tmem_ld_32x32b_x16(tb + c + 16 * half, u);
            tmem_ld_32x32b_x16(tb + BN / 2 + c + 16 * half, v);
            tmem_wait_ld(u);
            reg_fence(v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float a = __uint_as_float(u[j]), b = __uint_as_float(v[j]);
              h[16 * half + j] = a * sigmoidf_fast(a) * b;
            }
            if (ok && p.out3) {
              uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out3) + off + 16 * half);
              d[0] = make_uint4(pack_bf16x2(__uint_as_float(u[0]), __uint_as_float(u[1])),
                                pack_bf16x2(__uint_as_float(u[2]), __uint_as_float(u[3])),
                                pack_bf16x2(__uint_as_float(u[4]), __uint_as_float(u[5])),
                                pack_bf16x2(__uint_as_float(u[6]), __uint_as_float(u[7])));
              d[1] = make_uint4(pack_bf16x2(__uint_as_float(u[8]), __uint_as_float(u[9])),
                                pack_bf16x2(__uint_as_float(u[10]), __uint_as_float(u[11])),
                                pack_bf16x2(__uint_as_float(u[12]), __uint_as_float(u[13])),
                                pack_bf16x2(__uint_as_float(u[14]), __uint_as_float(u[15])));
            }
            if (ok && p.out4) {
              uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out4) + off + 16 * half);
              d[0] = make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                                pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                                pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                                pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
              d[1] = make_uint4(pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9])),
                                pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11])),
                                pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13])),
                                pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15])));
            }
          }
          if (ok) {
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(h[j]));
            const int e = mx_exponent_of(amax);
            const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
            uint32_t cw[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const __nv_fp8x2_storage_t lo =
                  __nv_cvt_float2_to_fp8x2(make_float2(h[4 * i] * inv, h[4 * i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
              const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                  make_float2(h[4 * i + 2] * inv, h[4 * i + 3] * inv), __NV_SATFINITE, __NV_E4M3);
              cw[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            uint4* cd = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out0) + off);
            cd[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            cd[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
            static_cast<uint8_t*>(p.out1)[static_cast<int64_t>(col / 32) * p.s_ld + grow] = static_cast<uint8_t>(e + 127);
            if (p.out2) {
              uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out2) + off);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                d[j] = make_uint4(pack_bf16x2(h[8 * j], h[8 * j + 1]), pack_bf16x2(h[8 * j + 2], h[8 * j + 3]),
                                  pack_bf16x2(h[8 * j + 4], h[8 * j + 5]), pack_bf16x2(h[8 * j + 6], h[8 * j + 7]));
            }
          }
        }
      } else {  // EPI_SWIGLU_BWD
        const int64_t grow = t.row0 + r;
#pragma unroll 1
        for (int c = hf * (BN / 2); c < (hf + 1) * (BN / 2); c += 16) {
          uint32_t u[16];
          tmem_ld_32x32b_x16(tb + c, u);
          tmem_wait_ld(u);
          const int col = t.nt * BN + c;
          if (row_ok && col < p.n_size) {
            const int64_t off = grow * p.ld_out + col;
            const uint4* pa = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.in0) + off);
            const uint4* pb = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.in1) + off);
            const uint4 a01 = pa[0], a23 = pa[1], b01 = pb[0], b23 = pb[1];
            const uint32_t aw[8] = {a01.x, a01.y, a01.z, a01.w, a23.x, a23.y, a23.z, a23.w};
            const uint32_t bw[8] = {b01.x, b01.y, b01.z, b01.w, b23.x, b23.y, b23.z, b23.w};
            uint32_t d1[8], d3[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float o1[2], o3[2];
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const float dh = __uint_as_float(u[2 * j + hh]);
                const float a1 = hh ? bf16hi(aw[j]) : bf16lo(aw[j]);
                const float a3 = hh ? bf16hi(bw[j]) : bf16lo(bw[j]);
                const float sg = sigmoidf_fast(a1);
                o3[hh] = dh * a1 * sg;
                o1[hh] = dh * a3 * sg * (1.0f + a1 * (1.0f - sg));
              }
              d1[j] = pack_bf16x2(o1[0], o1[1]);
              d3[j] = pack_bf16x2(o3[0], o3[1]);
            }
            uint4* q1 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out0) + off);
            uint4* q3 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out1) + off);
            q1[0] = make_uint4(d1[0], d1[1], d1[2], d1[3]);
            q1[1] = make_uint4(d1[4], d1[5], d1[6], d1[7]);
            q3[0] = make_uint4(d3[0], d3[1], d3[2], d3[3]);
            q3[1] = make_uint4(d3[4], d3[5], d3[6], d3[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR) mbar_arrive_remote(mapa_shared(smem_u32(&tempty[buf]), lead));
        else mbar_arrive(&tempty[buf]);
      }
    }
    if (EPI == EPI_F32 && lane == 0) bulk_wait_group0();   // every TMA store of this warp has landed
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();   // the leader's MMAs into the peer's TMEM and all cross-CTA arrivals are done
  tc_fence_after();
  if (warp == 1) {
    if (PAIR) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ host
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  });
  return fn;
}

// bf16 tensor map with 128-byte swizzle and zero fill out of bounds.
// rank3 == false: 2-D {cols, rows} (op.groups must be 1);
// rank3 == true : 3-D {cols, rows, groups} (also for a single group).
bool make_map(CUtensorMap* map, const Operand& op, uint32_t box_cols, uint32_t box_rows, bool rank3) {
  EncodeFn enc = get_encode_fn();
  if (!enc || !op.ptr) return false;
  if ((reinterpret_cast<uintptr_t>(op.ptr) & 15u) != 0 || (op.ld * 2) % 16 != 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(op.cols), static_cast<cuuint64_t>(op.rows),
                        static_cast<cuuint64_t>(op.groups)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(op.ld) * 2, static_cast<cuuint64_t>(op.group_stride) * 2};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (!rank3 && op.groups != 1) return false;
  const cuuint32_t rank = rank3 ? 3 : 2;
  if (rank == 3 && ((op.group_stride * 2) % 16 != 0 || op.group_stride < op.rows * op.ld)) return false;
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(op.ptr), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 output map {n, m, groups} for the TMA-store epilogue (box shape and
// swizzle below).  False when the layout is not TMA-compatible.
bool make_out_map_f32(CUtensorMap* map, void* base, int64_t n, int64_t m, int64_t groups, int64_t ld,
                      int64_t group_stride, bool wide) {
  EncodeFn enc = get_encode_fn();
  if (!enc || !base || (reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
  if ((ld * 4) % 16 != 0 || (group_stride * 4) % 16 != 0 || group_stride < m * ld) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(m), static_cast<cuuint64_t>(groups)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 4, static_cast<cuuint64_t>(group_stride) * 4};
  // wide: 32 columns x 16 rows, 128-byte swizzle; else 16 columns x 32 rows, 64-byte swizzle
  cuuint32_t box[3] = {wide ? 32u : 16u, wide ? 16u : 32u, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// uint8 tensor map (MXFP8 codes, 128-byte swizzled for the MMA, or scales,
// unswizzled), zero fill.
bool make_map_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                 const uint32_t* box, bool swizzle128 = false) {
  EncodeFn enc = get_encode_fn();
  if (!enc || !base || (reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
  cuuint64_t d[3];
  cuuint64_t st[2];
  cuuint32_t b[3];
  cuuint32_t e[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    if (i + 1 < rank) {
      if (strides[i] % 16 != 0) return false;
      st[i] = strides[i];
    }
  }
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), d, st, b, e,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool A_MN, bool B_MN, int EPI, bool QUANT = false, bool PAIR = false, bool W8 = false,
          bool GATHER = false>
cudaError_t launch_impl(const KParams& kp, int64_t units_ub, cudaStream_t stream) {
  using C = KernelCfg<BN, A_MN, EPI, QUANT, PAIR, W8>;
  constexpr int CN = 2;   // CTAs per cluster (PAIR)
  const size_t smem = C::smem_bytes(kp.num_groups);
  auto kern = grouped_gemm_kernel<BN, A_MN, B_MN, EPI, QUANT, PAIR, W8, GATHER>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_units = 0;   // co-resident CTAs (or CTA pairs)
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(C::smem_bytes(C::kMaxG)));
    max_units = PAIR ? num_sms() / CN : num_sms();
    if (attr_err == cudaSuccess && PAIR) {
      cudaLaunchConfig_t cfg{};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = CN;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(CN * max_units);
      cfg.blockDim = dim3(QUANT ? kThreadsQ : (W8 ? kThreadsW8 : kThreads));
      cfg.dynamicSmemBytes = C::smem_bytes(C::kMaxG);
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) max_units = n;
      cudaGetLastError();
    }
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int units = static_cast<int>(units_ub < max_units ? units_ub : max_units);
  if (!PAIR) {
    kern<<<units, QUANT ? kThreadsQ : (W8 ? kThreadsW8 : kThreads), smem, stream>>>(kp);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CN;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(CN * units);
  cfg.blockDim = dim3(QUANT ? kThreadsQ : (W8 ? kThreadsW8 : kThreads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, kp);
}

// 2-SM MMA (CTA pairs) is chosen when the groups average at least 512 rows:
// a pair tile spans 256 rows (ragged M), so smaller groups leave tiles half
// empty, and short contractions (ragged K) are bound by the fp32 output
// writes, where the pair gains nothing.  MOE_GEMM_CTA_PAIR=0 or =1 forces the
// one-SM or the pair form (read at every launch).
bool use_cta_pair(int64_t rows, int groups) {
  const char* e = std::getenv("MOE_GEMM_CTA_PAIR");
  if (e && e[0] == '0') return false;
  if (e && e[0] == '1') return true;
  return rows >= 512LL * groups;
}

}  // namespace

int gemm_ksplit(int64_t k, int requested) {
  const int64_t kb = (k + BK - 1) / BK;
  if (requested <= 1 || kb <= 1) return 1;
  const int64_t per = (kb + requested - 1) / requested;   // k-blocks per slice
  return static_cast<int>((kb + per - 1) / per);           // slices, none empty
}

int num_sms() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  });
  return n;
}

cudaError_t launch_grouped_gemm(const GemmArgs& a, cudaStream_t stream) {
  if (a.num_groups < 1 || a.num_groups > kMaxGroups || !a.offsets || !a.out0 || a.n_size <= 0)
    return cudaErrorInvalidValue;
  if (a.block_n != 256 && !(a.block_n == 32 && !a.b_mn && !a.a_mn && a.epi == EPI_F32))
    return cudaErrorInvalidValue;
  // bf16: ragged K comes with MN-major A (the two forms this kernel implements)
  if (!a.quant && a.ragged_k != a.a_mn) return cudaErrorInvalidValue;
  const int BN = a.block_n;
  KParams kp{};
  kp.offsets = a.offsets;
  kp.num_groups = a.num_groups;
  kp.m_size = a.m_size;
  kp.n_size = a.n_size;
  kp.b_dual_n = a.b_dual_n ? 1 : 0;
  kp.tile_n = a.b_dual_n ? BN / 2 : BN;
  kp.out0 = a.out0;
  kp.out1 = a.out1;
  kp.out2 = a.out2;
  kp.out3 = a.out3;
  kp.out4 = a.out4;
  kp.s_ld = a.s_ld;
  kp.in0 = a.in0;
  kp.in1 = a.in1;
  kp.ld_out = a.ld_out;
  kp.group_stride_out = a.group_stride_out;
  kp.status = a.status;

  int64_t tiles_ub = 0;
  if (a.quant) {
    // MXFP8 operands (block-scaled MMA), K-major A and B, 128 x 192 tiles,
    // k-blocks of 128 elements (4 scale blocks); a partial last k-block of a
    // source reads zero codes past its K.
    constexpr int QBN = 192;
    kp.kblk = 128;
    if (a.a_mn || a.b_mn) return cudaErrorInvalidValue;
    if (!a.ragged_k) {
      if (a.epi != EPI_SWIGLU_FWD_Q && a.epi != EPI_BF16 && a.epi != EPI_SWIGLU_BWD) return cudaErrorInvalidValue;
      if (a.max_rows <= 0) return cudaSuccess;
      const int nsrc = a.k1 > 0 ? 2 : 1;
      if (a.b_dual_n && nsrc != 1) return cudaErrorInvalidValue;
      kp.kb0 = static_cast<int>((a.k0 + 127) / 128);
      kp.kb1 = static_cast<int>((a.k1 + 127) / 128);
      if (kp.kb0 <= 0) return cudaErrorInvalidValue;
      kp.tile_n = a.b_dual_n ? QBN / 2 : QBN;
      // CTA pairs (256-row tiles, each CTA half of B): only when forced with
      // MOE_GEMM_CTA_PAIR=1.  Measured on the Mixtral shape they tie the
      // one-SM form at best, and the peer's cluster-scope release of its scale
      // atoms on every stage makes them 15% slower
      const char* pe = std::getenv("MOE_GEMM_CTA_PAIR");
      const bool qpair = pe && pe[0] == '1';
      const uint32_t brows = a.b_dual_n ? QBN / 2 : QBN;
      const uint32_t bcode_rows = (a.b_dual_n || qpair) ? QBN / 2 : QBN;
      for (int src = 0; src < nsrc; ++src) {
        const int64_t K = src == 0 ? a.k0 : a.k1;
        const MxOperand& q = a.qa[src];
        if (K <= 0 || K % 32 || q.cols != K) return cudaErrorInvalidValue;
        const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(q.rows)};
        const uint64_t str[1] = {static_cast<uint64_t>(K)};
        const uint32_t box[2] = {128, BM};
        if (!make_map_u8(&kp.tmA[src], q.codes, 2, dims, str, box, true)) return cudaErrorInvalidValue;
        const uint64_t sd[2] = {static_cast<uint64_t>(q.rows), static_cast<uint64_t>(K / 32)};
        const uint64_t ss[1] = {static_cast<uint64_t>(q.scale_ld)};
        const uint32_t sbox[2] = {144, 4};
        if (!make_map_u8(&kp.tmAs[src], q.scales, 2, sd, ss, sbox)) return cudaErrorInvalidValue;
      }
      const int nb = a.b_dual_n ? 2 : nsrc;
      for (int i = 0; i < nb; ++i) {
        const int64_t K = (a.b_dual_n || i == 0) ? a.k0 : a.k1;
        const MxOperand& b = a.qb[i];
        if (b.cols != K) return cudaErrorInvalidValue;
        const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(b.rows), static_cast<uint64_t>(b.groups)};
        const uint64_t str[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(b.rows * K)};
        const uint32_t box[3] = {128, bcode_rows, 1};
        if (!make_map_u8(&kp.tmB[i], b.codes, 3, dims, str, box, true)) return cudaErrorInvalidValue;
        const uint64_t sd[3] = {static_cast<uint64_t>(b.rows), static_cast<uint64_t>(K / 32), static_cast<uint64_t>(b.groups)};
        const uint64_t ss[2] = {static_cast<uint64_t>(b.scale_ld), static_cast<uint64_t>(b.scale_ld * (K / 32))};
        const uint32_t sbox[3] = {brows, 4, 1};
        if (!make_map_u8(&kp.tmBs[i], b.scales, 3, sd, ss, sbox)) return cudaErrorInvalidValue;
      }
      const int64_t ntiles = (a.n_size + kp.tile_n - 1) / kp.tile_n;
      const int64_t ur = qpair ? 2 * BM : BM;
      tiles_ub = ntiles * ((a.max_rows + ur - 1) / ur + a.num_groups);
      switch (a.epi) {
        case EPI_SWIGLU_FWD_Q:
          return qpair ? launch_impl<QBN, false, false, EPI_SWIGLU_FWD_Q, true, true>(kp, tiles_ub, stream)
                       : launch_impl<QBN, false, false, EPI_SWIGLU_FWD_Q, true>(kp, tiles_ub, stream);
        case EPI_SWIGLU_BWD:
          return qpair ? launch_impl<QBN, false, false, EPI_SWIGLU_BWD, true, true>(kp, tiles_ub, stream)
                       : launch_impl<QBN, false, false, EPI_SWIGLU_BWD, true>(kp, tiles_ub, stream);
        default:
          return qpair ? launch_impl<QBN, false, false, EPI_BF16, true, true>(kp, tiles_ub, stream)
                       : launch_impl<QBN, false, false, EPI_BF16, true>(kp, tiles_ub, stream);
      }
    }
    // ragged K (weight gradients): offsets are the padded group starts, every
    // group a multiple of 128 tokens; A [m_size][K_padded], B [n_size][K_padded]
    if (a.epi != EPI_F32 || a.m_size <= 0) return a.m_size <= 0 ? cudaSuccess : cudaErrorInvalidValue;
    const MxOperand& qa = a.qa[0];
    const MxOperand& qb = a.qb[0];
    const int64_t Kp = qa.cols;
    if (Kp <= 0 || Kp % 128 || qb.cols != Kp || qa.rows < a.m_size || qb.rows < a.n_size) return cudaErrorInvalidValue;
    {
      const uint64_t dims[2] = {static_cast<uint64_t>(Kp), static_cast<uint64_t>(qa.rows)};
      const uint64_t str[1] = {static_cast<uint64_t>(Kp)};
      const uint32_t box[2] = {128, BM};
      if (!make_map_u8(&kp.tmA[0], qa.codes, 2, dims, str, box, true)) return cudaErrorInvalidValue;
      const uint64_t sd[2] = {static_cast<uint64_t>(qa.rows), static_cast<uint64_t>(Kp / 32)};
      const uint64_t ss[1] = {static_cast<uint64_t>(qa.scale_ld)};
      const uint32_t sbox[2] = {BM, 4};
      if (!make_map_u8(&kp.tmAs[0], qa.scales, 2, sd, ss, sbox)) return cudaErrorInvalidValue;
    }
    {
      const uint64_t dims[2] = {static_cast<uint64_t>(Kp), static_cast<uint64_t>(qb.rows)};
      const uint64_t str[1] = {static_cast<uint64_t>(Kp)};
      const uint32_t box[2] = {128, QBN};
      if (!make_map_u8(&kp.tmB[0], qb.codes, 2, dims, str, box, true)) return cudaErrorInvalidValue;
      const uint64_t sd[2] = {static_cast<uint64_t>(qb.rows), static_cast<uint64_t>(Kp / 32)};
      const uint64_t ss[1] = {static_cast<uint64_t>(qb.scale_ld)};
      const uint32_t sbox[2] = {QBN, 4};
      if (!make_map_u8(&kp.tmBs[0], qb.scales, 2, sd, ss, sbox)) return cudaErrorInvalidValue;
    }
    kp.c_tma = make_out_map_f32(&kp.tmC, a.out0, a.n_size, a.m_size, a.num_groups, a.ld_out, a.group_stride_out,
                                (QBN / 2) % 32 == 0) ? 1 : 0;
    kp.c_rows = a.m_size;
    tiles_ub = static_cast<int64_t>(a.num_groups) * ((a.m_size + BM - 1) / BM) * ((a.n_size + QBN - 1) / QBN);
    return launch_impl<QBN, true, true, EPI_F32, true>(kp, tiles_ub, stream);
  }
  if (a.w8) {
    // FP8 weights: bf16 A (K-major), E4M3 B codes dequantised by converter
    // warps; ragged M, one-SM tiles 128 x 256
    if (a.ragged_k || a.a_mn || BN != 256 || a.max_rows <= 0) return a.max_rows <= 0 ? cudaSuccess : cudaErrorInvalidValue;
    if (a.epi != EPI_SWIGLU_FWD && a.epi != EPI_BF16 && a.epi != EPI_SWIGLU_BWD) return cudaErrorInvalidValue;
    kp.kblk = BK;
    kp.kb0 = (a.k0 + BK - 1) / BK;
    kp.kb1 = (a.k1 + BK - 1) / BK;
    if (kp.kb0 <= 0) return cudaErrorInvalidValue;
    const int nsrc = kp.kb1 > 0 ? 2 : 1;
    if (a.b_dual_n && (a.b_mn || nsrc != 1)) return cudaErrorInvalidValue;
    for (int s2 = 0; s2 < nsrc; ++s2)
      if (!make_map(&kp.tmA[s2], a.a[s2], 64, BM, false)) return cudaErrorInvalidValue;
    if (nsrc == 1) kp.tmA[1] = kp.tmA[0];
    const int nb = a.b_dual_n ? 2 : nsrc;
    for (int i = 0; i < nb; ++i) {
      const Operand& b = a.b[i];
      if (!a.w8_scale[i] || (b.ld % 16) || (b.group_stride % 16)) return cudaErrorInvalidValue;
      const uint64_t dims[3] = {static_cast<uint64_t>(b.cols), static_cast<uint64_t>(b.rows),
                                static_cast<uint64_t>(b.groups)};
      const uint64_t str[2] = {static_cast<uint64_t>(b.ld), static_cast<uint64_t>(b.group_stride)};
      const uint32_t box[3] = {64, a.b_mn ? 64u : static_cast<uint32_t>(a.b_dual_n ? BN / 2 : BN), 1};
      if (!make_map_u8(&kp.tmB[i], b.ptr, 3, dims, str, box)) return cudaErrorInvalidValue;
      kp.wscale[i] = a.w8_scale[i];
    }
    if (nb == 1) {
      kp.tmB[1] = kp.tmB[0];
      kp.wscale[1] = kp.wscale[0];
    }
    kp.ws_cols = static_cast<int32_t>((a.b[0].cols + 127) / 128);
    kp.ws_gstride = static_cast<int64_t>((a.b[0].rows + 127) / 128) * kp.ws_cols;
    const int64_t ntiles = (a.n_size + kp.tile_n - 1) / kp.tile_n;
    tiles_ub = ntiles * ((a.max_rows + BM - 1) / BM + a.num_groups);
    if (!a.b_mn) {
      if (a.epi == EPI_SWIGLU_FWD) return launch_impl<256, false, false, EPI_SWIGLU_FWD, false, false, true>(kp, tiles_ub, stream);
      if (a.epi == EPI_BF16) return launch_impl<256, false, false, EPI_BF16, false, false, true>(kp, tiles_ub, stream);
      return cudaErrorInvalidValue;
    }
    if (a.epi == EPI_SWIGLU_BWD) return launch_impl<256, false, true, EPI_SWIGLU_BWD, false, false, true>(kp, tiles_ub, stream);
    if (a.epi == EPI_BF16) return launch_impl<256, false, true, EPI_BF16, false, false, true>(kp, tiles_ub, stream);
    return cudaErrorInvalidValue;
  }
  if (a.a_gather) {
    // gathered A rows (ragged M, K-major bf16, one contraction source): a 2-D
    // map of the token matrix with one-row boxes for tile::gather4
    if (a.ragged_k || a.a_mn || a.b_mn || a.k1 > 0 || BN != 256 || a.gather_k <= 0 ||
        (a.epi != EPI_SWIGLU_FWD && a.epi != EPI_BF16) || a.max_rows <= 0)
      return a.max_rows <= 0 ? cudaSuccess : cudaErrorInvalidValue;
    const bool pair = use_cta_pair(a.max_rows, a.num_groups);
    kp.kblk = BK;
    kp.kb0 = (a.k0 + BK - 1) / BK;
    kp.kb1 = 0;
    if (kp.kb0 <= 0) return cudaErrorInvalidValue;
    if (!make_map(&kp.tmA[0], a.a[0], 64, 1, false)) return cudaErrorInvalidValue;
    kp.tmA[1] = kp.tmA[0];
    const int box_rows = (a.b_dual_n || pair) ? BN / 2 : BN;
    if (!make_map(&kp.tmB[0], a.b[0], 64, box_rows, true)) return cudaErrorInvalidValue;
    if (a.b_dual_n) {
      if (!make_map(&kp.tmB[1], a.b[1], 64, BN / 2, true)) return cudaErrorInvalidValue;
    } else {
      kp.tmB[1] = kp.tmB[0];
    }
    kp.a_gather = a.a_gather;
    kp.gather_k = a.gather_k;
    const int64_t ntiles = (a.n_size + kp.tile_n - 1) / kp.tile_n;
    const int64_t ur = pair ? 2 * BM : BM;
    const int64_t u = ntiles * ((a.max_rows + ur - 1) / ur + a.num_groups);
    if (a.epi == EPI_SWIGLU_FWD)
      return pair ? launch_impl<256, false, false, EPI_SWIGLU_FWD, false, true, false, true>(kp, u, stream)
                  : launch_impl<256, false, false, EPI_SWIGLU_FWD, false, false, false, true>(kp, u, stream);
    return pair ? launch_impl<256, false, false, EPI_BF16, false, true, false, true>(kp, u, stream)
                : launch_impl<256, false, false, EPI_BF16, false, false, false, true>(kp, u, stream);
  }
  // CTA pairs: each CTA loads its own 128 rows of A and half of the B tile
  const bool pair = BN == 256 && use_cta_pair(a.max_rows, a.num_groups) &&
                    (a.ragged_k ? a.epi == EPI_F32
                                : (a.epi == EPI_BF16 || a.epi == EPI_SWIGLU_FWD || a.epi == EPI_SWIGLU_BWD));
  kp.kblk = BK;
  if (!a.ragged_k) {
    if (a.max_rows <= 0) return cudaSuccess;
    kp.kb0 = (a.k0 + BK - 1) / BK;
    kp.kb1 = (a.k1 + BK - 1) / BK;
    if (kp.kb0 <= 0) return cudaErrorInvalidValue;
    const int nsrc = kp.kb1 > 0 ? 2 : 1;
    for (int s = 0; s < nsrc; ++s) {
      if (!make_map(&kp.tmA[s], a.a[s], 64, BM, false)) return cudaErrorInvalidValue;
      if (!a.b_mn) {
        const int box_rows = (a.b_dual_n || pair) ? BN / 2 : BN;
        if (!make_map(&kp.tmB[s], a.b[s], 64, box_rows, true)) return cudaErrorInvalidValue;
      } else {
        if (!make_map(&kp.tmB[s], a.b[s], 64, 64, true)) return cudaErrorInvalidValue;
      }
    }
    if (a.b_dual_n) {
      if (a.b_mn || nsrc != 1 || !make_map(&kp.tmB[1], a.b[1], 64, BN / 2, true)) return cudaErrorInvalidValue;
    }
    if (nsrc == 1) {
      kp.tmA[1] = kp.tmA[0];
      if (!a.b_dual_n) kp.tmB[1] = kp.tmB[0];
    }
    const int64_t ntiles = (a.n_size + kp.tile_n - 1) / kp.tile_n;
    const int64_t ur = pair ? 2 * BM : BM;
    tiles_ub = ntiles * ((a.max_rows + ur - 1) / ur + a.num_groups);
    kp.ksplit = gemm_ksplit(a.k0, a.ksplit);
    if (kp.ksplit > 1) {
      if (a.epi != EPI_F32 || a.num_groups != 1 || pair || a.b_dual_n || kp.kb1 > 0) return cudaErrorInvalidValue;
      tiles_ub *= kp.ksplit;
    }
  } else {
    if (a.m_size <= 0) return cudaSuccess;
    // k-blocks of BKR rows on CTA pairs (the kernel form's k-block length)
    const int kbr = pair ? BKR : BK;
    kp.kblk = kbr;
    if (!make_map(&kp.tmA[0], a.a[0], 64, kbr, false) || !make_map(&kp.tmB[0], a.b[0], 64, kbr, false))
      return cudaErrorInvalidValue;
    kp.tmA[1] = kp.tmA[0];
    kp.tmB[1] = kp.tmB[0];
    if (a.num_groups > 1) {
      // every group's own maps (copies of these two, rebased), written just before the GEMM
      if (!a.map_ws || (reinterpret_cast<uintptr_t>(a.map_ws) & 127u) != 0 ||
          2 * static_cast<size_t>(a.num_groups) * sizeof(CUtensorMap) > kGemmMapScratchBytes)
        return cudaErrorInvalidValue;
      CUtensorMap* maps = static_cast<CUtensorMap*>(a.map_ws);
      build_group_maps_kernel<<<(a.num_groups + 127) / 128, 128, 0, stream>>>(
          maps, kp.tmA[0], kp.tmB[0], a.offsets, a.num_groups, static_cast<const char*>(a.a[0].ptr), a.a[0].ld * 2,
          static_cast<const char*>(a.b[0].ptr), a.b[0].ld * 2);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      kp.gmaps = maps;
    }
    const int64_t ur = pair ? 2 * BM : BM;
    tiles_ub = static_cast<int64_t>(a.num_groups) * ((a.m_size + ur - 1) / ur) * ((a.n_size + BN - 1) / BN);
  }
  if (tiles_ub <= 0) return cudaSuccess;
  // fp32 outputs go through TMA stores when every tile's rows either belong to
  // its own output matrix (weight gradients) or end at the tensor's end (one group)
  if (a.epi == EPI_F32 && (a.ragged_k || a.num_groups == 1)) {
    const int64_t m = a.ragged_k ? a.m_size : a.max_rows;
    const int64_t gs = a.ragged_k ? a.group_stride_out : m * a.ld_out;
    kp.c_tma = make_out_map_f32(&kp.tmC, a.out0, a.n_size, m, a.ragged_k ? a.num_groups : std::max(1, kp.ksplit),
                                a.ld_out, gs, (BN / 2) % 32 == 0) ? 1 : 0;
    kp.c_rows = static_cast<int32_t>(m);
  }
  if (kp.ksplit > 1 && !kp.c_tma) return cudaErrorInvalidValue;   // partials leave through the TMA stores
  const int64_t u = tiles_ub;

  if (BN == 32) return launch_impl<32, false, false, EPI_F32>(kp, u, stream);
  if (!a.a_mn && !a.b_mn) {
    switch (a.epi) {
      case EPI_BF16:
        return pair ? launch_impl<256, false, false, EPI_BF16, false, true>(kp, u, stream)
                    : launch_impl<256, false, false, EPI_BF16>(kp, u, stream);
      case EPI_F32: return launch_impl<256, false, false, EPI_F32>(kp, u, stream);
      case EPI_SWIGLU_FWD:
        return pair ? launch_impl<256, false, false, EPI_SWIGLU_FWD, false, true>(kp, u, stream)
                    : launch_impl<256, false, false, EPI_SWIGLU_FWD>(kp, u, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (!a.a_mn && a.b_mn) {
    switch (a.epi) {
      case EPI_BF16:
        return pair ? launch_impl<256, false, true, EPI_BF16, false, true>(kp, u, stream)
                    : launch_impl<256, false, true, EPI_BF16>(kp, u, stream);
      case EPI_SWIGLU_BWD:
        return pair ? launch_impl<256, false, true, EPI_SWIGLU_BWD, false, true>(kp, u, stream)
                    : launch_impl<256, false, true, EPI_SWIGLU_BWD>(kp, u, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (a.a_mn && a.b_mn && a.epi == EPI_F32) {
    return pair ? launch_impl<256, true, true, EPI_F32, false, true>(kp, u, stream)
                : launch_impl<256, true, true, EPI_F32>(kp, u, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
