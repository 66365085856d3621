// Token-batched linear layers of the mixed step on the tcgen05 tensor cores.
//
// Prefill-chunk rows and decode rows are rows of one GEMM, so every weight
// tile is read once for all of them (ConfluxServe summary, "Why can linear
// layers be batched but attention cannot?"; pofe.ai "Chunked prefill": decodes
// "are 64 more rows in a 4,160-row matrix multiply").
//
// D[M][N] = A[M][K] B[N][K]^T, bf16 in, fp32 accumulate in TMEM.
//   tiles     by token count M (K step 64: one 128-byte swizzle atom):
//             * M <= 128: 128 x 256 per CTA, 4 stages of 48 KB, two
//               256-column accumulators (the epilogue of one tile overlaps
//               the next tile's main loop);
//             * otherwise 256 x 256 over a CTA pair (tcgen05 cta_group::2):
//               each CTA stages its 128 rows of A and one 128-row half of B
//               (32 KB a stage, 6 stages), rank 0 issues M = 256 MMAs that
//               read both CTAs' stages, each CTA's TMEM holds its 128 rows in
//               two 256-column accumulators;
//             * below 1,024 tokens, where 128-row tiles pad M less (M mod 256
//               in 1..128), 128 x 256 per CTA as for M <= 128.
//             The main loop is bound by load latency: a stage takes ~1,700-
//             2,900 cycles from its slot freeing to the MMA seeing it full,
//             so throughput is stages x stage bytes in flight over that time;
//             the pair's 32 KB stage per 512 MMA cycles (against 48 KB)
//             is what lets 6 stages cover it.
//   warps     0: TMA producer, 1: MMA issuer (+ TMEM owner), 2-5: epilogue
//             (warp w reads TMEM lane quarter w % 4); the 256-row-per-CTA
//             configuration (NH = 2, not used by the dispatcher) adds warps 6-9
//   TMEM      all 512 columns
//   schedule  persistent; whole tiles data-parallel while there are several
//             waves, the rest split along K evenly over all CTAs (stream-K:
//             the last one to two waves below 192 K steps, the last partial
//             wave from there on).  A split tile's later pieces go to fp32
//             partial slots (the rows of A only); the CTA that holds the
//             tile's first piece waits (bounded) for them, adds them in rank
//             order (deterministic) and runs the epilogue.  That wait needs every CTA of the grid resident at
//             once: the grid never exceeds the SM count, or the number of
//             clusters the occupancy query says fit.
//   epilogues store | + residual | SwiGLU (B rows [gate F; up F]: a tile loads
//             128 gate rows and the matching 128 up rows and writes
//             silu(g) * u for 128 output features)
//
// The partial tile quantisation the pofe.ai page warns about (chunk 257 vs
// 256, "Tile quantisation") is what the stream-K tail removes along N x K; a
// ragged M tail still costs a full 128-row MMA.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <atomic>
#include <cstdio>
#include <mutex>

#include "mb.h"
#include "mb_internal.h"
#include "mb_kernels.h"
#include "mb_launch.cuh"
#include "mb_ptx.cuh"

namespace mb {
namespace {

using namespace dev;

constexpr int HM = 128;                // rows of a half (the MMA's M)
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int A_HALF = HM * BK * 2;    // 16 KB
constexpr int B_STAGE = BN * BK * 2;   // 32 KB
constexpr int CHUNK = 128 * 32 * 4;    // one fp32 partial chunk: 128 rows x 32 columns
constexpr uint32_t IDESC = idesc_bf16(HM, BN, false);
constexpr uint32_t IDESC_PAIR = idesc_bf16(2 * HM, BN, false);   // M = 256 over a CTA pair
constexpr int kMaxHalves = 2;
constexpr int kMaxGroupedTilesM = 8;   // grouped schedule up to 8 M-tiles
constexpr int kWideMinRows = 1024;     // from this many tokens on, tiles have two halves
#ifndef MB_GEMM_PAIRS
#define MB_GEMM_PAIRS 1                // 0: no CTA pairs (128- and 256-row tiles per CTA); 2: pairs from 129 tokens
#endif
#ifndef MB_GEMM_PAIR_STAGES
#define MB_GEMM_PAIR_STAGES 6
#endif
constexpr int kLongKSteps = 192;       // stream-K over the last partial wave only from here on

// Tile configurations: NH halves of 128 rows per tile.
//  NH = 1: 128 x 256 tiles, 4 stages of 48 KB, two TMEM accumulators, so the
//          epilogue of one tile overlaps the main loop of the next;
//  NH = 2: 256 x 256 tiles, 3 stages of 64 KB (1.5x the MMA work per staged
//          byte), one accumulator pair that fills TMEM.
//  PAIR:   256 x 256 tiles over a CTA pair (2 SMs, one pair MMA of M = 256):
//          each CTA stages its 128 rows of A and one 128-row half of B, so
//          a 32 KB stage feeds 512 tensor cycles on each SM (64 B/cycle, as
//          for NH = 2) while each SM keeps two 256-column accumulators;
//          6 stages.
// Measured on GB300 (standalone, L2 flushed): pairs beat NH = 2 at every
// shape from 2,048 tokens (e.g. 2,144 x 5,120 x 17,408: 484 -> 322 us) and
// NH = 1 where their padding is no larger; at 576 tokens (768 padded rows
// against 640) NH = 1 stays faster.
template <int NH, bool PAIR = false>
struct TileCfg {
  static_assert(!PAIR || NH == 1, "a pair CTA holds one 128-row half");
  static constexpr int BM = PAIR ? 2 * HM : HM * NH;   // rows of a tile
  static constexpr int B_STG = PAIR ? B_STAGE / 2 : B_STAGE;
  static constexpr int STAGES = PAIR ? MB_GEMM_PAIR_STAGES : NH == 1 ? 4 : 3;
  static constexpr int A_STAGE = NH * A_HALF;
  static constexpr int SMEM_TILES = STAGES * (A_STAGE + B_STG);
  static constexpr int SMEM_BYTES = SMEM_TILES + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr int EPI_THREADS = 128 * NH;
  static constexpr int THREADS = 64 + EPI_THREADS;     // TMA, MMA, 4 epilogue warps per half
  static constexpr int NACC = NH == 1 ? 2 : 1;          // accumulator buffers in TMEM
  static constexpr int FIX_CHUNKS = NH == 1 ? 8 : 4;    // partial chunks staged per fix-up round
  static_assert(NACC * NH * BN <= 512, "TMEM holds 512 columns");
  static_assert(NH * FIX_CHUNKS * CHUNK <= SMEM_TILES, "fix-up staging lives in the idle stage buffers");
};
// Weight k-blocks warmed into L2 behind the ring's first STAGES, before the
// grid-dependency wait (while the previous kernel of the stream finishes).
// Only there: prefetching ahead of the ring inside the main loop as well was
// slower on GB300 at every shape measured (L2 flushed clean before each
// call): at 2,144 tokens (Qwen3-14B shapes) QKV 108.5 -> 98.3 us, O 90.1 ->
// 81.9, gate/up 432 -> 406 and down 287 -> 262 without it; at 16 tokens
// gate/up 73.7 -> 63.5 and down 55.3 -> 51.2.  A read-only TMA stream of the
// same boxes, no MMA, shows the same: 59.4 us for 356 MB without prefetch,
// 67.6 with it 4 blocks ahead.
#ifndef MB_GEMM_PREFETCH
#define MB_GEMM_PREFETCH 8
#endif
constexpr int kPrefetchAhead = MB_GEMM_PREFETCH;
// Grouped schedule: split an N-tile along K over several groups only if that
// takes at least this many K steps off each CTA; below it the stream-K fix-up
// (partials out, the head piece waiting, partials back in) costs more than the
// split saves.  Llama-3-8B shapes at 576 tokens on GB300: QKV 41.6 -> 37.6 us
// and O 39.6 -> 35.5 us unsplit (64 K steps against 51 and 34 split), down
// 72.3 us split (120 K steps) against 90.8 us unsplit (224).
constexpr int kSplitMinSaving = 32;
// Up to this many rows of A (a few decode rows) a split tile's head stages
// every other piece at once (the partial layout keeps a piece's rows of A
// contiguous: one bulk copy each) and adds them up with all four epilogue
// warps before one pass over TMEM, instead of one round trip per piece.
// Measured on GB300, 16 rows (Qwen3-14B shapes, L2 flushed clean): QKV 30.7
// -> 26.6 us, O 32.8 -> 26.6, down 51.2 -> 45.1.  At 64 rows the batched
// code was slower (O 34.8 -> 36.9 us), hence a kernel of its own.
constexpr int kFoldBatchRows = 32;

struct Params {
  int M, N, K;          // N: output width (F for SwiGLU)
  int k_iters;
  int tiles_m, tiles_n;
  int grouped;          // 1: CTA (g, m) streams weight tiles of group g for M-tile m
  int n_groups;         // grouped: CTA groups (grid = n_groups * tiles_m)
  int cluster;          // 2: CTA pairs (cluster of two SMs); 1 otherwise
  int dp_tiles, sk_tiles;
  int grid;
  __nv_bfloat16 *D;
  int ldd;
  const __nv_bfloat16 *R;
  int ldr;
  int F;                // SwiGLU: row offset of the up half in B
  float *partials;      // [2 grid][NH halves][8 / FIX groups][128 rows][FIX x 32] fp32 (part_row)
  int *tickets;
  int *err;
  uint64_t split_wait_ns;   // limit of the head piece's wait for the other pieces of its tile
  int split_phantom;        // pieces the head also waits for that no CTA writes (failure-path tests; 0)
  int b_const;              // 1: no kernel of the stream writes B (a layer's weights): loaded before the wait
  // First (unit, k) iteration of each rank; rlo[ranks] = all iterations.
  // Filled on the host (fill_rank_bounds) so that no CTA divides 64-bit
  // numbers before its first load.
  int rlo[kMaxGemmGrid + 1];
};

// Work decomposition.  Two schedules share one iteration space of (unit, k)
// pairs, split into contiguous ranges over "ranks":
//  * grouped (few M-tiles): a unit is an N-tile, a rank is a group of
//    tiles_m CTAs, one per M-tile, that walk the same weight tiles at the
//    same time (each weight tile then streams from HBM once);
//  * default: whole tiles round-robin over the grid, then the tail tiles'
//    (tile, k) space split over all CTAs (stream-K); a unit is a tail tile.
// A unit covered by several ranks is summed from fp32 partial tiles by the
// rank that arrives last (deterministic order: rank order).
struct Seg {
  int tile, k0, k1;
  int partial;  // 0: whole K range; 1: a piece of a split tile
  int slot;     // partial slot of this piece
  int unit;     // unit index of a split piece
};

__host__ __device__ __forceinline__ int sk_ranks(const Params &p) { return p.grouped ? p.n_groups : p.grid; }
__device__ __forceinline__ int rank_lo(const Params &p, int rank) { return p.rlo[rank]; }

// The split fix-up's wait (mb_gemm_set_split_wait), read at launch: its time
// limit and the phantom pieces that make it run out in failure-path tests.
std::atomic<uint64_t> g_split_wait_ns{kWaitLimitNs};
std::atomic<int> g_split_phantom{0};

// Rank boundaries: rank r covers iterations [total r / R, total (r + 1) / R)
// of the (unit, k) space.  False if the space does not fit 32-bit indices.
bool fill_rank_bounds(Params &p) {
  const long long total = static_cast<long long>(p.grouped ? p.tiles_n : p.sk_tiles) * p.k_iters;
  const int R = sk_ranks(p);
  if (total >= (1ll << 31) || R < 1 || R > kMaxGemmGrid) return false;
  for (int r = 0; r <= R; ++r) p.rlo[r] = static_cast<int>(total * r / R);
  return true;
}

struct SegIter {
  const Params &p;
  int b, rank, mi;
  int dp_next;
  int it, it_end, first_unit;
  // b: this CTA's place in the schedule (a pair's two CTAs share one);
  // slot_cta: the CTA index that owns its partial slots
  int slot_cta;
  __device__ SegIter(const Params &pp, int bb, int sc) : p(pp), b(bb), slot_cta(sc) {
    rank = p.grouped ? b / p.tiles_m : b;
    mi = p.grouped ? b % p.tiles_m : 0;
    dp_next = p.grouped ? p.dp_tiles : b;
    it = rank_lo(p, rank);
    it_end = rank_lo(p, rank + 1);
    first_unit = it / p.k_iters;
  }
  __device__ bool next(Seg &s) {
    if (dp_next < p.dp_tiles) {
      s.tile = dp_next;
      s.k0 = 0;
      s.k1 = p.k_iters;
      s.partial = 0;
      s.slot = 0;
      s.unit = -1;
      dp_next += p.grid;
      return true;
    }
    if (it >= it_end) return false;
    const int u = it / p.k_iters;
    const int k0 = it - u * p.k_iters;
    const int k1 = min(p.k_iters, k0 + (it_end - it));
    s.tile = p.grouped ? u * p.tiles_m + mi : p.dp_tiles + u;
    s.k0 = k0;
    s.k1 = k1;
    s.partial = !(k0 == 0 && k1 == p.k_iters);
    s.slot = 2 * slot_cta + (u == first_unit ? 0 : 1);
    s.unit = u;
    it += k1 - k0;
    return true;
  }
};

// Ranks whose ranges overlap unit u: [r_first, r_last].
__device__ void unit_ranks(const Params &p, int u, int &r_first, int &r_last) {
  const int R = sk_ranks(p);
  auto owner = [&](int x) {   // the last rank whose range starts at or before x
    int lo = 0, hi = R - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.rlo[mid] <= x)
        lo = mid;
      else
        hi = mid - 1;
    }
    return lo;
  };
  const int lo = u * p.k_iters;
  r_first = owner(lo);
  r_last = owner(lo + p.k_iters - 1);
}

// Schedule index of rank `rank`'s CTA (or pair) for M-tile mi.
__device__ __forceinline__ int sched_cta(const Params &p, int rank, int mi) {
  return p.grouped ? rank * p.tiles_m + mi : rank;
}
// Partial slot that the CTA of `rank` (same M-tile; for pairs the CTA of the
// same rank in the pair, `crank`) used for unit u.
template <bool PAIR>
__device__ __forceinline__ int slot_of(const Params &p, int rank, int mi, int crank, int u) {
  const int c = sched_cta(p, rank, mi);
  return 2 * (PAIR ? 2 * c + crank : c) + (u == rank_lo(p, rank) / p.k_iters ? 0 : 1);
}

// silu(x) = x / (1 + e^-x), with the fast exponential and division (relative
// error ~1e-6, far below the bf16 rounding of the result; for x < -87 the
// denominator overflows and the result is 0, as it rounds to in bf16 anyway).
// A correctly rounded reciprocal has a special-case branch per element that
// serialises the epilogue's 4 warps (measured: ~8 us per 128 x 128 tile).
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// Partial tiles: per slot and half, 8 / FIX row groups, each [128 rows][FIX
// chunks x 32] fp32 (FIX = the chunks a fix-up round stages per half), so
// that the rows of A in a group are one contiguous block: one bulk copy
// stages them, however few.
template <int NH>
__device__ __forceinline__ float *part_row(const Params &p, int slot, int h, int g, int r) {
  constexpr int FIX = NH == 1 ? 8 : 4;
  return p.partials + ((((static_cast<size_t>(slot) * NH + h) * (8 / FIX) + g) * 128 + r) * (FIX * 32));
}
// Halves of the tile at m0 that hold rows of A.
template <int NH>
__device__ __forceinline__ int halves_of(const Params &p, int m0) { return (NH == 2 && m0 + HM < p.M) ? 2 : 1; }
// Within a partial row of 32 floats, 16-byte group q is stored at q ^ (row % 8)
// so that the finisher's shared-memory reads of 128 rows spread over banks.
__device__ __forceinline__ int part_swz(int q, int r) { return q ^ (r & 7); }

// Residual for 4 chunks (128 columns) of one row, issued early.
__device__ __forceinline__ void load_resid4(const Params &p, int row, int col, uint4 (&rb)[16]) {
  if (row >= p.M) return;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool in = col + 32 * j < p.N;
    const uint4 *rp = reinterpret_cast<const uint4 *>(p.R + static_cast<size_t>(row) * p.ldr + col + 32 * j);
#pragma unroll
    for (int q = 0; q < 4; ++q) rb[4 * j + q] = in ? rp[q] : make_uint4(0, 0, 0, 0);
  }
}

// Epilogue of one 32-column chunk: v (and u for SwiGLU) -> bf16 -> D.
template <int EPI>
__device__ __forceinline__ void store_chunk(const Params &p, int row, int col, const float (&v)[32],
                                            const float *u, const uint4 *rb) {
  if (row >= p.M || col >= p.N) return;
  uint32_t packed[16];
  if (EPI == kEpiSwiGLU) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      packed[i] = pack_bf16x2(silu(v[2 * i]) * u[2 * i], silu(v[2 * i + 1]) * u[2 * i + 1]);
  } else if (EPI == kEpiResidual) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t rr[4] = {rb[q].x, rb[q].y, rb[q].z, rb[q].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = q * 4 + j;
        packed[i] = pack_bf16x2(v[2 * i] + bf16lo(rr[j]), v[2 * i + 1] + bf16hi(rr[j]));
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) packed[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  }
  uint4 *dp = reinterpret_cast<uint4 *>(p.D + static_cast<size_t>(row) * p.ldd + col);
#pragma unroll
  for (int q = 0; q < 4; ++q) dp[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
}

// PAIR: the grid is p.grid pairs (2 p.grid CTAs, clusters of 2).  Rank 0 of
// a pair issues the pair MMAs, owns the stage-full and accumulator-empty
// barriers both CTAs' copies and epilogues report to; each CTA loads, drains
// and fixes up its own 128 rows.
// FOLDB: a split tile's head stages all other pieces at once and adds them
// up with every epilogue thread before one pass over TMEM (tiles of at most
// kFoldBatchRows rows of A); otherwise it folds one piece per round.
template <int EPI, int NH, bool PAIR, bool FOLDB = false>
__global__ void __launch_bounds__(TileCfg<NH, PAIR>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p) {
  using C = TileCfg<NH, PAIR>;
  constexpr int BM = C::BM, STAGES = C::STAGES, A_STAGE = C::A_STAGE, EPI_THREADS = C::EPI_THREADS;
  constexpr int B_STG = C::B_STG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_STAGE;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::SMEM_TILES);   // [STAGES] (a pair: rank 0's)
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;   // [NACC]
  uint64_t *tempty = tfull + C::NACC; // [NACC]
  uint64_t *fixbar = tempty + C::NACC;   // [NH], one per half
  uint64_t *fin = fixbar + 2;            // a pair: all pair MMAs done (rank 0)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      // one MMA commit releases the stage (a pair's releases both CTAs' stages)
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < C::NACC; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], (PAIR ? 2 : 1) * EPI_THREADS);   // a pair: both CTAs' epilogues
    }
    for (int h = 0; h < NH; ++h) mbar_init(&fixbar[h], 1);
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // a pair's peer arrives on this CTA's barriers and its MMAs write this
  // CTA's TMEM: both must be set up first
  if (p.cluster > 1) cluster_sync();
  const uint32_t crank = p.cluster > 1 ? cluster_ctarank() : 0;
  const int sched_b = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  // a pair's stage-full barriers live in rank 0 (cluster addresses)
  const uint32_t full_r0 = PAIR ? mapa_shared(smem_u32(full), 0) : 0u;
  // bytes that land for one stage (a pair: both CTAs'; a pair CTA whose rows
  // all lie past M loads no A)
  auto stage_bytes = [&](int m0, int nh) -> uint32_t {
    if (PAIR) return (m0 + HM < p.M ? 2 : 1) * A_HALF + 2 * B_STG;
    return nh * A_HALF + B_STG;
  };

  // A layer's weights are read-only for the whole stream: while earlier
  // kernels finish, arm the first stages and load their weight tiles (and
  // warm L2 with the next ones); only the activation tiles wait for those
  // kernels.  Other B operands (standalone calls) may come from the kernel
  // just before: they wait like A.
  int pre = 0;   // stages whose weight tiles are already on their way
  if (warp == 0 && lane == 0 && p.b_const) {
    SegIter first(p, sched_b, blockIdx.x);
    Seg s0;
    if (first.next(s0)) {
      const int m0f = (s0.tile % p.tiles_m) * BM;
      const int nh = halves_of<NH>(p, m0f);
      const int nt = s0.tile / p.tiles_m;
      const int rows0 = EPI == kEpiSwiGLU ? nt * 128 : nt * BN;
      const int rows1 = EPI == kEpiSwiGLU ? p.F + nt * 128 : nt * BN + 128;
      const bool prefetcher = (p.grouped ? (sched_b % p.tiles_m) == 0 : true) && crank == 0;
      for (int kb = s0.k0; kb < s0.k1 && pre < STAGES; ++kb, ++pre) {
        if (PAIR) {
          if (crank == 0) mbar_arrive_expect_tx(&full[pre], stage_bytes(m0f, nh));
          tma_load_2d_pair(sB + pre * B_STG, &tmB, full_r0 + 8 * pre, kb * BK, crank ? rows1 : rows0);
          continue;
        }
        mbar_arrive_expect_tx(&full[pre], stage_bytes(m0f, nh));
        tma_load_2d(sB + pre * B_STG, &tmB, &full[pre], kb * BK, rows0);
        tma_load_2d(sB + pre * B_STG + B_STAGE / 2, &tmB, &full[pre], kb * BK, rows1);
      }
      // then warm L2 with the next k-blocks (a TMA instruction costs ~90
      // cycles to issue: the stage loads go first)
      if (prefetcher)
        for (int kb = s0.k0 + STAGES; kb < s0.k1 && kb < s0.k0 + STAGES + kPrefetchAhead; ++kb) {
          tma_prefetch_2d(&tmB, kb * BK, rows0);
          tma_prefetch_2d(&tmB, kb * BK, rows1);
        }
    }
  }
  pdl_wait();   // A, R, D, the tickets and partials belong to earlier kernels of the stream
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------- TMA producer
      SegIter segs(p, sched_b, blockIdx.x);
      Seg sg;
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued_mask = 0, issued_ph = 0;
      int n_issued = 0;   // k steps issued so far (the first `pre` have their weights in flight)
      bool ok = true;
      while (ok && segs.next(sg)) {
        const int m0 = (sg.tile % p.tiles_m) * BM;
        const int nh = halves_of<NH>(p, m0);
        const int nt = sg.tile / p.tiles_m;
        const int rows0 = EPI == kEpiSwiGLU ? nt * 128 : nt * BN;
        const int rows1 = EPI == kEpiSwiGLU ? p.F + nt * 128 : nt * BN + 128;
        for (int kb = sg.k0; kb < sg.k1; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.err, kErrWaitProducer)) {
            ok = false;
            break;
          }
          const bool b_sent = n_issued++ < pre;
          if (PAIR) {
            // rank 0 arms its barrier for both CTAs' bytes; each CTA loads its
            // rows of A and its half of B and reports to rank 0
            if (crank == 0 && !b_sent) mbar_arrive_expect_tx(&full[s], stage_bytes(m0, nh));
            const uint32_t fb = full_r0 + 8 * s;
            if (m0 + static_cast<int>(crank) * HM < p.M)
              tma_load_2d_pair(sA + s * A_STAGE, &tmA, fb, kb * BK, m0 + crank * HM);
            if (!b_sent) tma_load_2d_pair(sB + s * B_STG, &tmB, fb, kb * BK, crank ? rows1 : rows0);
            issued_mask |= 1u << s;
            issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
            if (++s == STAGES) {
              s = 0;
              ph ^= 1;
            }
            continue;
          }
          if (!b_sent) mbar_arrive_expect_tx(&full[s], stage_bytes(m0, nh));
          tma_load_2d(sA + s * A_STAGE, &tmA, &full[s], kb * BK, m0);
          if (nh == 2) tma_load_2d(sA + s * A_STAGE + A_HALF, &tmA, &full[s], kb * BK, m0 + HM);
          if (!b_sent) {
            tma_load_2d(sB + s * B_STG, &tmB, &full[s], kb * BK, rows0);
            tma_load_2d(sB + s * B_STG + B_STAGE / 2, &tmB, &full[s], kb * BK, rows1);
          }
          issued_mask |= 1u << s;
          issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok) {
        // let copies already in flight land before the CTA exits (rank 1 of a
        // pair reports its copies to rank 0's barriers, which it cannot poll:
        // it gives them a millisecond, far beyond a copy's latency)
        if (PAIR && crank != 0) {
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 1000000ull) {
          }
          issued_mask = 0;
        }
        for (int i = 0; i < STAGES; ++i)
          if (issued_mask & (1u << i)) {
            const uint32_t a = smem_u32(&full[i]);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(a, (issued_ph >> i) & 1u) && globaltimer() - t0 < kWaitLimitNs) {
            }
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      // (a pair: rank 0 only; the pair MMA writes both CTAs' TMEM)
      SegIter segs(p, sched_b, blockIdx.x);
      Seg sg;
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = !(PAIR && crank != 0);
      while (ok && segs.next(sg)) {
        const int nh = halves_of<NH>(p, (sg.tile % p.tiles_m) * BM);
        // the epilogue has drained this accumulator buffer's previous tile
        if (!mbar_wait(&tempty[acc], acc_ph ^ 1, abort_flag, p.err, kErrWaitMma)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * NH * BN;
        for (int kb = sg.k0; kb < sg.k1; ++kb) {
          if (!mbar_wait(&full[s], ph, abort_flag, p.err, kErrWaitMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * A_STAGE);
          const uint32_t b0 = smem_u32(sB + s * B_STG);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = sdesc_sw128(b0 + kk * 32, 16, 1024);
            const uint32_t accum = (kb > sg.k0 || kk > 0) ? 1u : 0u;
            if (PAIR) {
              mma_bf16_pair(d, sdesc_sw128(a0 + kk * 32, 16, 1024), bd, IDESC_PAIR, accum);
              continue;
            }
            mma_bf16(d, sdesc_sw128(a0 + kk * 32, 16, 1024), bd, IDESC, accum);
            if (nh == 2) mma_bf16(d + BN, sdesc_sw128(a0 + A_HALF + kk * 32, 16, 1024), bd, IDESC, accum);
          }
          if (PAIR)
            mma_commit_pair(&empty[s], 3);
          else
            mma_commit(&empty[s]);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        if (PAIR)
          mma_commit_pair(&tfull[acc], 3);
        else
          mma_commit(&tfull[acc]);
        if (++acc == C::NACC) {
          acc = 0;
          acc_ph ^= 1;
        }
      }
      if (PAIR && crank == 0) {
        // no pair MMA may still write either CTA's TMEM when they free it
        mma_commit_pair(fin, 1);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(fin), 0) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Every branch below that contains a named barrier is taken by all 256
    // epilogue threads or by none (decisions go through barrier ORs).
    const int q = warp & 3;            // TMEM lane quarter this warp may read
    const int h = (warp - 2) >> 2;     // half of the tile (TMEM columns h*256 ..)
    const int r = q * 32 + lane;       // row within the half
    const int ep = threadIdx.x - 64;   // 0 .. EPI_THREADS-1
    // a drained accumulator goes back to the MMA issuer (a pair: rank 0's barrier)
    const uint32_t tempty_r0 = PAIR ? mapa_shared(smem_u32(tempty), 0) : 0u;
    auto release_acc = [&](int a) {
      tc_fence_before();
      if (PAIR && crank != 0)
        mbar_arrive_remote(tempty_r0 + 8 * a);
      else
        mbar_arrive(&tempty[a]);
    };
    SegIter segs(p, sched_b, blockIdx.x);
    Seg sg;
    int acc = 0;
    uint32_t acc_ph = 0;
    uint32_t fix_ph = 0;
    bool ok = true;
    while (ok && segs.next(sg)) {
      const int mi = sg.tile % p.tiles_m;
      const int m0 = mi * BM;
      // this half (a pair: this CTA's 128 rows) holds rows of A
      const bool mine = PAIR ? m0 + static_cast<int>(crank) * HM < p.M : h < halves_of<NH>(p, m0);
      const int nt = sg.tile / p.tiles_m;
      const int hrow0 = m0 + (PAIR ? static_cast<int>(crank) : h) * HM;   // first row of this half
      const int row = hrow0 + r;
      // rows of A in this half: only these go through the split fix-up and the
      // stores (a few decode rows then move a few KB of partials, not 128 KB)
      const int rv = mine ? min(HM, p.M - hrow0) : 0;
      const bool wrows = q * 32 < rv;   // this warp's lane quarter holds some (warp-uniform)
      const int col0 = EPI == kEpiSwiGLU ? nt * 128 : nt * BN;
      uint4 rb[16];
      // the residual does not depend on the accumulator: fetch it while the
      // MMAs run (a split tile fetches it after its fix-up instead)
      if (EPI == kEpiResidual && mine && !sg.partial) load_resid4(p, row, col0, rb);
      const bool got = mbar_wait(&tfull[acc], acc_ph, abort_flag, p.err, kErrWaitEpilogue);
      if (named_bar_or(1, EPI_THREADS, !got)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + (acc * NH + h) * BN + (static_cast<uint32_t>(q * 32) << 16);
      bool finish = !sg.partial;
      if (sg.partial) {
        int r_first, r_last;
        unit_ranks(p, sg.unit, r_first, r_last);
        const int my_rank = p.grouped ? sched_b / p.tiles_m : sched_b;
        // A split unit is identified by its first rank (no other split unit
        // starts there), so flags stay below the grid size.  The CTAs of a
        // pair fix up their own rows: one flag each.
        const int fidx = sched_cta(p, r_first, mi);
        int *flag = p.tickets + (PAIR ? 2 * fidx + static_cast<int>(crank) : fidx);
        if (my_rank != r_first) {
          // a later piece: hand the fp32 partial to the rank that covers the
          // unit's head (for which this unit is its last segment)
          if (wrows) {
#pragma unroll 1
            for (int j = 0; j < BN / 32; ++j) {
              float v[32];
              tmem_ld32(tbase + 32 * j, v);
              float4 *w4 = reinterpret_cast<float4 *>(part_row<NH>(p, sg.slot, h, j / C::FIX_CHUNKS, r) +
                                                      (j % C::FIX_CHUNKS) * 32);
              if (r < rv) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  w4[part_swz(i, r)] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
              }
            }
          }
          release_acc(acc);
          __threadfence();
          named_bar_sync(1, EPI_THREADS);
          if (ep == 0) atomicAdd(flag, 1);
        } else {
          // the head piece: wait for the other pieces (written early in their
          // ranks' timelines), fold them into the accumulator in TMEM
          if (ep == 0) {
            const int want = r_last - r_first + p.split_phantom;
            const uint64_t t0 = globaltimer();
            int spins = 0;
            while (ld_acquire_gpu(flag) < want) {
              if ((++spins & 255) == 0 && globaltimer() - t0 > p.split_wait_ns) {
                *abort_flag = 1;
                atomicExch(p.err, kErrWaitEpilogue);
                break;
              }
            }
            *flag = 0;
            fence_proxy_async_global();
          }
          if (named_bar_or(1, EPI_THREADS, *abort_flag != 0)) {
            ok = false;
          } else {
            // this unit is the rank's last segment: the stage buffers are idle.
            // Each half stages the other pieces' row groups (their rows of A,
            // one bulk copy each) in its own area, as many per round as fit:
            // 128 / rv of them, so with a few rows of A every piece lands in
            // one round.  Item i is group i % G of piece r_first + 1 + i / G;
            // every element adds, in rank order, the round's pieces to each
            // other and then their sum to the accumulator.  Both halves of a
            // 256-row tile size their rounds by half 0's rows, so that they
            // take the same number of rounds (the named barrier is shared).
            constexpr int G = 8 / C::FIX_CHUNKS;
            constexpr uint32_t rbytes = C::FIX_CHUNKS * 128u;   // one row of a group
            uint8_t *stage = smem + h * C::FIX_CHUNKS * CHUNK;
            const int rv0 = PAIR ? rv : min(HM, p.M - m0);
            const int per_round = FOLDB && rv0 > 0 ? HM / rv0 : 1;
            const uint32_t gbytes = static_cast<uint32_t>(rv) * rbytes;
            const int n_items = (r_last - r_first) * G;
#pragma unroll 1
            for (int i0 = 0; i0 < n_items && ok; i0 += per_round) {
              const int i1 = min(n_items, i0 + per_round);
              bool fine = true;
              if (mine) {
                if (q == 0 && lane == 0) {
                  mbar_arrive_expect_tx(&fixbar[h], static_cast<uint32_t>(i1 - i0) * gbytes);
                  for (int i = i0; i < i1; ++i) {
                    const int slot = slot_of<PAIR>(p, r_first + 1 + i / G, mi, static_cast<int>(crank), sg.unit);
                    bulk_load(stage + (i - i0) * gbytes, part_row<NH>(p, slot, h, i % G, 0), gbytes, &fixbar[h]);
                  }
                }
                fine = __all_sync(0xffffffffu, mbar_wait(&fixbar[h], fix_ph, abort_flag, p.err, kErrWaitEpilogue));
                fix_ph ^= 1;
              }
              // leave together: the barrier at the end of each round is shared
              if (named_bar_or(1, EPI_THREADS, !fine)) {
                ok = false;
                break;
              }
              // all threads of the half first add each group's later items into
              // its first one (consecutive float4 per thread: no bank conflicts),
              // then the warps that own rows of A add that sum into TMEM
              if (FOLDB && mine) {
#pragma unroll 1
                for (int g = 0; g < G; ++g) {
                  const int ig = i0 + (g - i0 % G + G) % G;   // first item of group g staged now
                  if (ig + G >= i1) continue;                 // at most one item of group g
                  float4 *dst = reinterpret_cast<float4 *>(stage + (ig - i0) * gbytes);
                  const int n4 = static_cast<int>(gbytes / 16);
                  auto item4 = [&](int i, int e) {
                    return reinterpret_cast<const float4 *>(stage + (i - i0) * gbytes)[e];
                  };
                  auto add4 = [](float4 &a, const float4 &t) {
                    a.x += t.x;
                    a.y += t.y;
                    a.z += t.z;
                    a.w += t.w;
                  };
#pragma unroll 2
                  for (int e = r; e < n4; e += HM) {
                    float4 a = dst[e];
                    int i = ig + G;
                    // four items' loads in flight at a time, added in rank order
#pragma unroll 1
                    for (; i + 3 * G < i1; i += 4 * G) {
                      const float4 t0 = item4(i, e), t1 = item4(i + G, e), t2 = item4(i + 2 * G, e),
                                   t3 = item4(i + 3 * G, e);
                      add4(a, t0);
                      add4(a, t1);
                      add4(a, t2);
                      add4(a, t3);
                    }
#pragma unroll 1
                    for (; i < i1; i += G) add4(a, item4(i, e));
                    dst[e] = a;
                  }
                }
              }
              if (FOLDB) named_bar_sync(1, EPI_THREADS);
              if (wrows) {
                const int rs = r < rv ? r : 0;   // the staged row this lane adds
#pragma unroll 1
                for (int g = 0; g < G; ++g) {
                  const int ig = i0 + (g - i0 % G + G) % G;
                  if (ig >= i1) continue;
#pragma unroll 1
                  for (int jj = 0; jj < C::FIX_CHUNKS; ++jj) {
                    float v[32];
                    tmem_ld32(tbase + 32 * (g * C::FIX_CHUNKS + jj), v);   // the warp's whole lane quarter
                    // rows past A's have nothing staged and are never stored: they
                    // add row 0 (no lane may branch off before the aligned tcgen05.st)
                    const float4 *src =
                        reinterpret_cast<const float4 *>(stage + (ig - i0) * gbytes + rs * rbytes + jj * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                      const float4 t = src[part_swz(c, rs)];
                      v[4 * c] += t.x;
                      v[4 * c + 1] += t.y;
                      v[4 * c + 2] += t.z;
                      v[4 * c + 3] += t.w;
                    }
                    tmem_st32(tbase + 32 * (g * C::FIX_CHUNKS + jj), v);
                  }
                }
              }
              named_bar_sync(1, EPI_THREADS);   // the next round overwrites the staging
            }
            finish = ok;
          }
          if (!finish) release_acc(acc);
        }
      }
      if (finish) {
        if (wrows) {
          if (EPI == kEpiSwiGLU) {
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
              float g[32], u[32];
              tmem_ld32(tbase + 32 * j, g);
              tmem_ld32(tbase + 128 + 32 * j, u);
              store_chunk<EPI>(p, row, col0 + 32 * j, g, u, nullptr);
            }
          } else if (EPI == kEpiResidual) {
            if (sg.partial) load_resid4(p, row, col0, rb);
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
              if (hc == 1) load_resid4(p, row, col0 + 128, rb);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                float v[32];
                tmem_ld32(tbase + 128 * hc + 32 * j, v);
                store_chunk<EPI>(p, row, col0 + 128 * hc + 32 * j, v, nullptr, rb + 4 * j);
              }
            }
          } else {
#pragma unroll 1
            for (int j = 0; j < BN / 32; ++j) {
              float v[32];
              tmem_ld32(tbase + 32 * j, v);
              store_chunk<EPI>(p, row, col0 + 32 * j, v, nullptr, nullptr);
            }
          }
        }
        release_acc(acc);
      }
      if (++acc == C::NACC) {
        acc = 0;
        acc_ph ^= 1;
      }
    }
  }

  __syncthreads();
  // no CTA of a pair leaves while its peer may still arrive on it (rank 0's
  // MMA issuer saw its last MMA complete before this)
  if (p.cluster > 1) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem, 512);
    else
      tmem_dealloc(tmem, 512);
  }
}

template <int EPI, int NH, bool PAIR = false, bool FOLDB = false>
cudaError_t launch(const CUtensorMap &tmA, const CUtensorMap &tmB, const Params &p, cudaStream_t st) {
  using C = TileCfg<NH, PAIR>;
  const cudaError_t attr_err =
      ensure_max_smem(reinterpret_cast<const void *>(gemm_kernel<EPI, NH, PAIR, FOLDB>), C::SMEM_BYTES);
  if (attr_err != cudaSuccess) return attr_err;
  // a pair schedule's p.grid counts pairs
  return launch_pdl(gemm_kernel<EPI, NH, PAIR, FOLDB>, dim3(PAIR ? 2 * p.grid : p.grid), dim3(C::THREADS), C::SMEM_BYTES,
                    st, p.cluster, tmA, tmB, p);
}

// mode: 1 = 128-row tiles, 2 = 256-row tiles, kModePair = 256-row tiles over CTA pairs,
// kModeFew = 128-row tiles holding at most kFoldBatchRows rows of A (batched fix-up)
constexpr int kModePair = 3;
constexpr int kModeFew = 4;

cudaError_t launch_for(int epi, int nh, const CUtensorMap &tmA, const CUtensorMap &tmB, const Params &p,
                       cudaStream_t st) {
  if (nh == kModePair) {
    switch (epi) {
      case kEpiStore: return launch<kEpiStore, 1, true>(tmA, tmB, p, st);
      case kEpiResidual: return launch<kEpiResidual, 1, true>(tmA, tmB, p, st);
      case kEpiSwiGLU: return launch<kEpiSwiGLU, 1, true>(tmA, tmB, p, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (nh == 2) {
    switch (epi) {
      case kEpiStore: return launch<kEpiStore, 2>(tmA, tmB, p, st);
      case kEpiResidual: return launch<kEpiResidual, 2>(tmA, tmB, p, st);
      case kEpiSwiGLU: return launch<kEpiSwiGLU, 2>(tmA, tmB, p, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (nh == kModeFew) {
    switch (epi) {
      case kEpiStore: return launch<kEpiStore, 1, false, true>(tmA, tmB, p, st);
      case kEpiResidual: return launch<kEpiResidual, 1, false, true>(tmA, tmB, p, st);
      case kEpiSwiGLU: return launch<kEpiSwiGLU, 1, false, true>(tmA, tmB, p, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (epi) {
    case kEpiStore: return launch<kEpiStore, 1>(tmA, tmB, p, st);
    case kEpiResidual: return launch<kEpiResidual, 1>(tmA, tmB, p, st);
    case kEpiSwiGLU: return launch<kEpiSwiGLU, 1>(tmA, tmB, p, st);
    default: return cudaErrorInvalidValue;
  }
}

// Clusters of `size` CTAs of this kernel that can be resident at once (the
// split fix-up waits on other CTAs, so the whole grid must be co-resident).
template <int EPI, int NH, bool PAIR = false>
int max_clusters(int size) {
  using C = TileCfg<NH, PAIR>;
  static std::mutex mu;
  static int cache[9] = {0};
  std::lock_guard<std::mutex> lk(mu);
  if (size < 1 || size > 8) return 0;
  if (cache[size] == 0) {
    ensure_max_smem(reinterpret_cast<const void *>(gemm_kernel<EPI, NH, PAIR>), C::SMEM_BYTES);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(size * 64);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<EPI, NH, PAIR>, &cfg) != cudaSuccess || n <= 0) n = -1;
    cache[size] = n;
  }
  return cache[size];
}

// CTA pairs of the pair kernel that can be resident at once.
int max_pairs_for(int epi) {
  switch (epi) {
    case kEpiStore: return max_clusters<kEpiStore, 1, true>(2);
    case kEpiResidual: return max_clusters<kEpiResidual, 1, true>(2);
    default: return max_clusters<kEpiSwiGLU, 1, true>(2);
  }
}

}  // namespace

constexpr size_t kPartialSlotBytes = static_cast<size_t>(kMaxHalves) * HM * BN * sizeof(float);

size_t gemm_workspace_bytes() {
  return static_cast<size_t>(2 * kMaxGemmGrid) * kPartialSlotBytes + 2 * kMaxGemmGrid * sizeof(int);
}

GemmWorkspace gemm_workspace_carve(void *base) {
  GemmWorkspace w;
  w.partials = static_cast<float *>(base);
  w.tickets = reinterpret_cast<int *>(static_cast<char *>(base) + static_cast<size_t>(2 * kMaxGemmGrid) * kPartialSlotBytes);
  return w;
}

// SMs a GEMM may use: the device's, at most kMaxGemmGrid, at most max_ctas.
static int gemm_sms(int max_ctas) {
  int sms = device_sm_count() < kMaxGemmGrid ? device_sm_count() : kMaxGemmGrid;
  if (max_ctas > 0 && max_ctas < sms) sms = max_ctas;
  return sms;
}

int gemm_launches(int M, int, int, int, int) { return M > 0 ? 1 : 0; }

cudaError_t gemm_run(const void *A, const void *B, const CUtensorMap *tmB_pre, void *D, const void *R, int M, int N,
                     int K, int epi, const GemmWorkspace &ws, int *err, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const int b_rows = epi == kEpiSwiGLU ? 2 * N : N;
  CUtensorMap tmA, tmB;
  cudaError_t e = encode_tmap_2d(&tmA, A, K, M, static_cast<uint64_t>(K) * 2, BK, HM);
  if (e != cudaSuccess) return e;
  if (tmB_pre) {
    tmB = *tmB_pre;
  } else {
    e = encode_tmap_2d(&tmB, B, K, b_rows, static_cast<uint64_t>(K) * 2, BK, 128);
    if (e != cudaSuccess) return e;
  }
  Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.k_iters = K / BK;
  const int sm_count = gemm_sms(ws.max_ctas);
  // Tile shape.  Up to 128 tokens: one 128-row tile per CTA.  From
  // kWideMinRows tokens on: 256-row tiles over CTA pairs.  In between, pairs
  // where they pad M no more than 128-row tiles do (M mod 256 = 0 or > 128):
  // at 576 tokens, 768 padded rows against 640 cost more than the pairs'
  // faster main loop saves (measured on GB300).
  const auto round_up = [](int x, int t) { return (x + t - 1) / t * t; };
  const bool want_pairs = MB_GEMM_PAIRS && M > HM &&
                          (MB_GEMM_PAIRS == 2 || M >= kWideMinRows || round_up(M, 2 * HM) == round_up(M, HM));
  const int pairs = want_pairs ? std::min(sm_count / 2, max_pairs_for(epi)) : 0;
  const int nh = pairs > 0 ? kModePair : M >= kWideMinRows ? 2 : 1;
  const int tile_rows = nh == 1 ? HM : 2 * HM;
  p.tiles_m = (M + tile_rows - 1) / tile_rows;
  p.tiles_n = epi == kEpiSwiGLU ? N / 128 : (N + BN - 1) / BN;
  const int tiles = p.tiles_m * p.tiles_n;
  // schedule units: CTAs, or CTA pairs
  const int sms = pairs > 0 ? pairs : sm_count;
  const int base_cluster = pairs > 0 ? 2 : 1;
  if (p.tiles_m <= kMaxGroupedTilesM && p.tiles_m <= sms) {
    // Few token tiles: every weight tile is consumed by tiles_m CTAs running
    // side by side, and the (N-tile, k) space is split evenly over the groups
    // (one whole N-tile per group where a split would save too little).
    long long groups = sms / p.tiles_m;
    if (groups > p.tiles_n) {
      const long long split_iters = (static_cast<long long>(p.tiles_n) * p.k_iters + groups - 1) / groups;
      if (p.k_iters - split_iters < kSplitMinSaving) groups = p.tiles_n;   // one whole N-tile per group
    }
    p.cluster = base_cluster;
    const long long iters = static_cast<long long>(p.tiles_n) * p.k_iters;
    if (iters < 2 * groups) groups = iters / 2 > 0 ? iters / 2 : 1;  // at least two K steps per CTA
    p.grouped = 1;
    p.n_groups = static_cast<int>(groups);
    p.grid = p.n_groups * p.tiles_m;
    p.dp_tiles = 0;
    p.sk_tiles = 0;
  } else if (tiles % sms == 0) {
    p.cluster = base_cluster;
    p.dp_tiles = tiles;
    p.sk_tiles = 0;
    p.grid = sms;
  } else {
    p.cluster = base_cluster;
    // Whole waves run data-parallel; the rest is spread along K over every SM
    // (stream-K).  Short K: the last one to two waves.  Long K: only the last
    // partial wave.  A rank's stream-K range starts at its own K offset in
    // its tile, so ranks that share a weight tile read it at different times;
    // with long K that is more than L2 holds, and the weights come from HBM
    // once per rank.  Measured on GB300 (down projection, 272 K steps, 5,120
    // wide): 2,304 tokens (180 pair tiles for 76 pairs) 315 -> 236 us, 2,216
    // 309 -> 236, 4,100 490 -> 416; at 80 K steps (QKV, O, gate/up at 2,144
    // tokens) one extra wave of stream-K stays faster (100 against 104 us,
    // 82 / 86, 412 / 428).  With this, a long-K GEMM whose last pair tiles
    // are mostly padding (2,144 = 8 x 256 + 96) also needs no second launch
    // for those rows: 234 us in one launch against 266 with the 96 rows as a
    // 128-row-tile launch of their own.
    const int waves = tiles / sms;
    const int sk_waves = p.k_iters >= kLongKSteps ? 0 : 1;
    p.dp_tiles = waves >= 1 + sk_waves ? (waves - sk_waves) * sms : 0;
    p.sk_tiles = tiles - p.dp_tiles;
    const long long sk_iters = static_cast<long long>(p.sk_tiles) * p.k_iters;
    long long g = sms;
    if (sk_iters < 2LL * g) g = sk_iters / 2 > 0 ? sk_iters / 2 : 1;
    if (p.dp_tiles > 0 && g < sms) g = sms;
    p.grid = static_cast<int>(g);
    if (p.dp_tiles > 0 && p.grid != sms) return cudaErrorInvalidValue;
  }
  p.D = static_cast<__nv_bfloat16 *>(D);
  p.ldd = N;
  p.R = static_cast<const __nv_bfloat16 *>(R);
  p.ldr = N;
  p.F = epi == kEpiSwiGLU ? N : 0;
  p.partials = ws.partials;
  p.tickets = ws.tickets;
  p.err = err;
  p.split_wait_ns = g_split_wait_ns.load(std::memory_order_relaxed);
  p.split_phantom = g_split_phantom.load(std::memory_order_relaxed);
  p.b_const = tmB_pre != nullptr;   // the layers' pre-encoded weight maps
  if (!fill_rank_bounds(p)) return cudaErrorInvalidValue;
  return launch_for(epi, nh == 1 && M <= kFoldBatchRows ? kModeFew : nh, tmA, tmB, p, st);
}

}  // namespace mb

// ---------------------------------------------------------------------------
// Allocation-free variant of the GEMM entry point.
//
// Some callers cannot call cudaMalloc: code running under an allocator that
// must not be re-entered (a memory pool's own hooks, an out-of-memory
// handler), processes whose device memory is fully handed out up front, or
// plugins that may only touch buffers their host gives them.  For them,
// mb_gemm_noalloc keeps the stream-K scratch (fp32 partial tiles, tile tickets
// and the error word) in the file-scope device array below instead of a
// cudaMalloc'ed workspace.  Every GPU that loads this library holds the array
// (16 MiB + 4 KiB) until the process exits.  All calls on a device share it:
// calls that overlap on the GPU (different streams without ordering) race.
// The tickets are cleared on the call's stream before every launch; the
// partial tiles need no clearing (every slot is written before it is read).
// The error word is cleared once, when the array's address is first looked
// up on a device, and after that only by mb_device_status(NULL, stream),
// which reports it; so a bounded wait that gave up in one call stays
// visible after later calls.  The stream-K part runs on at most kNoAllocGrid
// CTAs so that its partial tiles fit; problems with at least one tile per SM
// run without any split.

static __device__ __align__(256) uint8_t g_gemm_noalloc_scratch[(2u * 64u * 128u * 256u * 4u) + 4096u];

namespace mb {
namespace {

constexpr int kNoAllocGrid = 64;
constexpr size_t kNoAllocPartialBytes = static_cast<size_t>(2 * kNoAllocGrid) * TileCfg<1>::BM * BN * sizeof(float);
constexpr size_t kNoAllocTailBytes = 4096;  // tickets, then the error word in the last 16 bytes
constexpr size_t kNoAllocTicketBytes = kNoAllocTailBytes - 16;
static_assert(sizeof(g_gemm_noalloc_scratch) == kNoAllocPartialBytes + kNoAllocTailBytes, "scratch layout");

std::mutex g_noalloc_mu;
void *g_noalloc_addr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device (host code only has a stand-in for the symbol).  The first
// lookup also clears the tail (tickets and error word), synchronously.
cudaError_t noalloc_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gemm_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemset(static_cast<uint8_t *>(p) + kNoAllocPartialBytes, 0, kNoAllocTailBytes);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return cudaSuccess;
}

}  // namespace

// Error code the allocation-free GEMM recorded on the current device since
// the last call (0: none, or the array was never used here); a non-zero code
// is cleared together with the tickets a kernel that gave up may have left
// raised.  The caller has synchronised the streams that used it.
cudaError_t gemm_noalloc_take_error(int *code) {
  *code = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  uint8_t *base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    base = static_cast<uint8_t *>(g_noalloc_addr[dev]);
  }
  if (!base) return cudaSuccess;
  int word = 0;
  e = cudaMemcpy(&word, base + kNoAllocPartialBytes + kNoAllocTicketBytes, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  if (word != 0) {
    e = cudaMemset(base + kNoAllocPartialBytes, 0, kNoAllocTailBytes);
    if (e != cudaSuccess) return e;
  }
  *code = word;
  return cudaSuccess;
}

}  // namespace mb

extern "C" mb_status mb_gemm_noalloc(const void *A, const void *B, void *D, const void *R, int32_t M, int32_t N,
                                     int32_t K, int32_t epilogue, void *stream) {
  using namespace mb;
  if (!A || !B || !D || M < 0 || N <= 0 || K <= 0) return fail(MB_EINVAL, "mb_gemm_noalloc: bad argument");
  if (epilogue < 0 || epilogue > 2) return fail(MB_EINVAL, "mb_gemm_noalloc: epilogue must be 0, 1 or 2");
  if (epilogue == 1 && (!R || R == D)) return fail(MB_EINVAL, "mb_gemm_noalloc: residual epilogue needs R != D");
  if (K % 64) return fail(MB_EUNSUPPORTED, "mb_gemm_noalloc: K must be a multiple of 64");
  if (epilogue == 2 && N % 128) return fail(MB_EUNSUPPORTED, "mb_gemm_noalloc: SwiGLU needs F = N %% 128 == 0");
  if (N % 32) return fail(MB_EUNSUPPORTED, "mb_gemm_noalloc: N must be a multiple of 32");
  for (const void *p : {A, B, static_cast<const void *>(D), R})
    if (p && reinterpret_cast<uintptr_t>(p) % 16)
      return fail(MB_EINVAL, "mb_gemm_noalloc: pointers must be 16-byte aligned");
  if (M == 0) return MB_OK;
  int dev = 0, sms = 0, major = 0, minor = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return fail(MB_ECUDA, "mb_gemm_noalloc: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return fail(MB_EUNSUPPORTED, "mb_gemm_noalloc: device is sm_%d%d; these kernels are built for sm_103a", major,
                minor);
  if (sms > kMaxGemmGrid) sms = kMaxGemmGrid;

  Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.k_iters = K / BK;
  p.tiles_m = (M + TileCfg<1>::BM - 1) / TileCfg<1>::BM;
  p.tiles_n = epilogue == kEpiSwiGLU ? N / 128 : (N + BN - 1) / BN;
  const long long tiles = static_cast<long long>(p.tiles_m) * p.tiles_n;
  p.cluster = 1;
  if (tiles >= sms) {
    p.dp_tiles = static_cast<int>(tiles);
    p.sk_tiles = 0;
    p.grid = sms;
  } else {
    p.dp_tiles = 0;
    p.sk_tiles = static_cast<int>(tiles);
    const long long sk_iters = tiles * p.k_iters;
    long long g = kNoAllocGrid;
    if (sk_iters < 2LL * g) g = sk_iters / 2 > 0 ? sk_iters / 2 : 1;
    p.grid = static_cast<int>(g);
  }
  const size_t need_partials = p.sk_tiles ? static_cast<size_t>(2 * p.grid) * TileCfg<1>::BM * BN * sizeof(float) : 0;
  const size_t need_tickets = static_cast<size_t>(p.sk_tiles) * sizeof(int);
  if (need_partials > kNoAllocPartialBytes || need_tickets > kNoAllocTicketBytes)
    return fail(MB_EUNSUPPORTED,
                "mb_gemm_noalloc: this shape needs %zu bytes of partial tiles and %zu of tickets; the static "
                "scratch holds %zu and %zu",
                need_partials, need_tickets, kNoAllocPartialBytes, kNoAllocTicketBytes);

  void *scratch = nullptr;
  e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return fail(MB_ECUDA, "mb_gemm_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
  uint8_t *base = static_cast<uint8_t *>(scratch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the tickets only: the error word keeps an earlier call's code until it is read
  e = cudaMemsetAsync(base + kNoAllocPartialBytes, 0, kNoAllocTicketBytes, st);
  if (e != cudaSuccess) return fail(MB_ECUDA, "mb_gemm_noalloc: cudaMemsetAsync: %s", cudaGetErrorString(e));

  const int b_rows = epilogue == kEpiSwiGLU ? 2 * N : N;
  CUtensorMap tmA, tmB;
  e = encode_tmap_2d(&tmA, A, K, M, static_cast<uint64_t>(K) * 2, BK, HM);
  if (e == cudaSuccess) e = encode_tmap_2d(&tmB, B, K, b_rows, static_cast<uint64_t>(K) * 2, BK, 128);
  if (e != cudaSuccess) return fail(MB_ECUDA, "mb_gemm_noalloc: tensor map encoding failed");
  p.D = static_cast<__nv_bfloat16 *>(D);
  p.ldd = N;
  p.R = static_cast<const __nv_bfloat16 *>(R);
  p.ldr = N;
  p.F = epilogue == kEpiSwiGLU ? N : 0;
  p.partials = reinterpret_cast<float *>(base);
  p.tickets = reinterpret_cast<int *>(base + kNoAllocPartialBytes);
  p.err = reinterpret_cast<int *>(base + kNoAllocPartialBytes + kNoAllocTicketBytes);
  p.split_wait_ns = g_split_wait_ns.load(std::memory_order_relaxed);
  p.split_phantom = g_split_phantom.load(std::memory_order_relaxed);
  if (!fill_rank_bounds(p)) return fail(MB_EUNSUPPORTED, "mb_gemm_noalloc: too many (tile, K step) pairs");
  e = launch_for(epilogue, 1, tmA, tmB, p, st);   // 128-row tiles: their partials fit the array
  if (e != cudaSuccess) return fail(MB_ECUDA, "mb_gemm_noalloc: launch: %s", cudaGetErrorString(e));
  return MB_OK;
}

extern "C" mb_status mb_gemm_set_split_wait(int64_t limit_ns, int32_t phantom_pieces) {
  if (phantom_pieces < 0 || phantom_pieces > 1024)
    return mb::fail(MB_EINVAL, "mb_gemm_set_split_wait: phantom_pieces must be in [0, 1024]");
  mb::g_split_wait_ns.store(limit_ns > 0 ? static_cast<uint64_t>(limit_ns) : mb::dev::kWaitLimitNs,
                            std::memory_order_relaxed);
  mb::g_split_phantom.store(phantom_pieces, std::memory_order_relaxed);
  return MB_OK;
}
