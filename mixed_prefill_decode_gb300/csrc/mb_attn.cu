// Ragged paged attention of the mixed step.
//
// After the token-batched linear layers the batch splits (ConfluxServe
// summary, "Why can linear layers be batched but attention cannot?"; Perplexity
// "Disaggregated Prefill and Decode": prefill rows have large qo_len, decode
// rows qo_len = 1 against long kv_len):
//
//  * chunk tiles: 128 query rows x one q-head of a prefill chunk.  A query at
//    position c + i sees keys 0 .. c + i (llm-stack-book 7.8, "Attention on
//    Partial KV Caches"); keys and values are read page by page through the
//    block table with TMA (one 16 x 64 box per page, head and 64-wide half,
//    from the HND pool), S = Q K^T and O_blk = P V run on tcgen05 with fp32
//    accumulators in TMEM, the online softmax runs in registers (one thread
//    per query row).  S is double-buffered in TMEM so the next block's Q K^T
//    overlaps this block's softmax.
//  * decode rows: split-KV.  One warp per (request, KV head, page range)
//    serves all q-heads of the GQA group from one read of K and V (16-byte
//    loads, 8 bf16 per lane), keeps (m, l, o) per head, and either writes the
//    normalised output (single split) or a partial that the merge pass
//    combines by log-sum-exp.
//
// GQA: q head h reads KV head h / (Hq / Hkv) (llm-stack-book 7.8, exercise 5).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "mb_kernels.h"
#include "mb_launch.cuh"
#include "mb_ptx.cuh"

namespace mb {
namespace {

using namespace dev;

constexpr float kLog2e = 1.4426950408889634f;
// decode partial row: o[hd], m, l, padding to a 16-byte multiple
template <int HD>
__host__ __device__ constexpr int part_stride() { return HD + 4; }

// ============================================================ chunk tiles
// A chunk tile is 256 query rows of one q-head of a prefill chunk, as two
// 128-row query tiles t = 0, 1 that share every staged block of keys and
// values.  Keys and values come through the block table in 128-key blocks
// (8 pages, one TMA copy per page and K or V).  Per block j and tile t:
//
//   S_t = Q_t K^T     tcgen05, M = 128 rows, N = 128 keys, K = hd (TMEM)
//   softmax           four warps per tile, one thread per query row, so a
//                     row's maximum and sum need no exchange between threads
//   O_t += P_t V      P_t (bf16) written over S_t in TMEM is the A operand,
//                     V the MN-major B operand straight from its stage
//
// The MMA issuer alternates the tiles, PV_0(j), S_0(j+1), PV_1(j), S_1(j+1),
// so the tensor cores run one tile's products while the other tile's softmax
// runs (the FA4-style ping-pong).  O_t accumulates in TMEM; a row is rescaled
// only when its maximum grows by more than 2^8 over the reference it uses,
// so probabilities stay <= 256 and most blocks never wait for the previous PV.
template <int HD>
struct ChunkCfg {
  static constexpr int NH = HD / 64;               // 64-wide swizzle chunks along hd
  static constexpr int TILE_BYTES = 128 * 128;     // [128 rows][64 bf16]
  static constexpr int QT_BYTES = NH * TILE_BYTES; // one query tile
  static constexpr int KV_BYTES = NH * TILE_BYTES; // a block of K or of V
  // A K or V stage holds 128 keys as [8-key group][hd half][8 keys][128 B]
  // (what one copy per page delivers): atoms of a half are ATOM_STRIDE apart.
  static constexpr int ATOM_STRIDE = NH * 1024;
  static constexpr int PAGE_BYTES = 2 * ATOM_STRIDE;
  // Separate K and V rings: a K block is free once both tiles' S products
  // are done, a V block only after both PV products, a block period later.
  // With 3 K and 2 V stages each load gets about two block periods of lead
  // (two query tiles take the room a third V stage would need).
  static constexpr int NK = HD == 128 ? 3 : 4;
  static constexpr int NV = HD == 128 ? 2 : 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * QT_BYTES;
  static constexpr int OFF_V = OFF_K + NK * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + NV * KV_BYTES;
  // The kernel checks that the dynamic shared memory starts 1024-aligned, so
  // no alignment slack is reserved.
  static constexpr int SMEM = OFF_BAR + 256;
  static constexpr int THREADS = 320;              // TMA, MMA, 2 x 4 softmax warps
  static constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, HD, true);
  static constexpr uint32_t TMEM_COLS = 512;       // S_0 [0,128), S_1 [128,256), O_0, O_1 from 256
  static constexpr uint32_t O_COL = 256;
};

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Probabilities of 64 logits against the reference m (log2 domain, scale
// folded in): p = 2^(s scale - m) in pairs, packed as bf16 pairs, summed into
// `sum` (pairwise, packed fp32).
__device__ __forceinline__ void probs64(const float (&sv)[64], float2 sc2, float m, uint32_t (&pk)[32],
                                        float2 &sum) {
  const float2 negm = make_float2(-m, -m);
#pragma unroll
  for (int c = 0; c < 64; c += 2) {
    const float2 x = __ffma2_rn(make_float2(sv[c], sv[c + 1]), sc2, negm);
    const float p0 = ex2_approx(x.x);
    const float p1 = ex2_approx(x.y);
    sum = __fadd2_rn(sum, make_float2(p0, p1));
    pk[c / 2] = pack_bf16x2(p0, p1);
  }
}

struct ChunkParams {
  __nv_bfloat16 *o;
  const int32_t *qo_indptr, *kv_len, *bt_indptr, *bt, *tiles;
  int Hq, Hkv, num_pages;
  float scale_log2;
  int *err;
  float *part;   // partials of split tiles: [slot][256 rows][hd + 4] (o, m, l, pad)
  int *ctr;      // one counter per split tile: pieces finished (the merger resets it)
};

// One chunk tile (up to 256 query rows x one q-head); needs
// ChunkCfg<HD>::THREADS threads and ChunkCfg<HD>::SMEM bytes of shared memory.
template <int HD>
__device__ __forceinline__ void chunk_tile(const CUtensorMap &tmQ, const CUtensorMap &tmKV, const ChunkParams &p,
                                           int tile, uint8_t *smem_raw) {
  using C = ChunkCfg<HD>;
  uint8_t *smem = align1024(smem_raw);
  uint8_t *sQ = smem + C::OFF_Q;
  uint8_t *sK = smem + C::OFF_K;
  uint8_t *sV = smem + C::OFF_V;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *q_full = bars + 0;
  uint64_t *k_full = bars + 1;             // [NK]
  uint64_t *k_empty = k_full + C::NK;      // [NK]
  uint64_t *v_full = k_empty + C::NK;      // [NV]
  uint64_t *v_empty = v_full + C::NV;      // [NV]
  uint64_t *s_full = v_empty + C::NV;      // [2 tiles]
  uint64_t *p_full = s_full + 2;           // [2 tiles]
  uint64_t *o_full = p_full + 2;           // [2 tiles]: PV_t(j) done, j < n_kb_t - 1
  uint64_t *o_last = o_full + 2;           // every MMA of the tile done (committed once)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(o_last + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *merge_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);
  static_assert((1 + 2 * C::NK + 2 * C::NV + 7) * 8 + 12 <= 256, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // work unit {req, row0, head, j0, j1, piece, n_pieces, slot}: key blocks
  // [j0, j1) of the tile (all of them when n_pieces == 1)
  const int32_t *unit = p.tiles + tile * 8;
  const int req = unit[0];
  const int i0 = unit[1];
  const int h = unit[2];
  const int j0 = unit[3];
  const int n_pieces = unit[6];
  const int slot = unit[7];
  const int t0 = p.qo_indptr[req];
  const int qo = p.qo_indptr[req + 1] - t0;
  const int kv = p.kv_len[req];
  const int cached = kv - qo;
  const int rows_valid = min(256, qo - i0);
  const int last_pos = cached + i0 + rows_valid - 1;
  const int n_kb = (last_pos + 1 + 127) / 128;   // the tile's blocks (all pieces)
  const int j_end = min(unit[4], n_kb);          // this unit's blocks: [j0, j_end)
  const int nb = j_end - j0;
  // blocks each query tile needs (0: the tile has no rows), and where this
  // unit's part of them ends (every row of a tile sees every key of a piece
  // that is not the tile's last: only the last piece holds the diagonal)
  int nkb_t[2], jt_end[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int rows = min(128, rows_valid - 128 * t);
    nkb_t[t] = rows > 0 ? (cached + i0 + 128 * t + rows - 1 + 1 + 127) / 128 : 0;
    jt_end[t] = min(nkb_t[t], j_end);
  }
  const int hk = h / (p.Hq / p.Hkv);
  const int32_t *table = p.bt + p.bt_indptr[req];

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&o_full[t], 1);
    }
    mbar_init(o_last, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmKV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // q, the KV pool and o belong to earlier kernels of the stream
  pdl_trigger();

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    // Lane 0 waits and arms each stage; the block's 8 pages go out as one
    // TMA per lane (one thread issuing them all would pace the rings at ~90
    // cycles a copy).  K runs NK - NV blocks ahead of V, the order in which
    // their slots free up.  Page ids: one per lane, loaded a block ahead.
    if (lane == 0) {
      const int nq = jt_end[1] > j0 ? 2 : 1;
      mbar_arrive_expect_tx(q_full, nq * C::QT_BYTES);
      for (int t = 0; t < nq; ++t)
        for (int c = 0; c < C::NH; ++c)
          tma_load_2d(sQ + t * C::QT_BYTES + c * C::TILE_BYTES, &tmQ, q_full, h * HD + c * 64, t0 + i0 + 128 * t);
    }
    constexpr int AHEAD = C::NK - C::NV;
    const int n_pages = (last_pos + 1 + 15) / 16;
    auto page_of = [&](int blk) { return lane < 8 && 8 * blk + lane < n_pages ? table[8 * blk + lane] : 0; };
    // one ring: wait for the slot, arm it, 8 copies (lanes 0-7)
    // blk: the block's index in the tile; rings count from the unit's first
    auto load_block = [&](bool is_v, int blk, int pg) -> bool {
      const int ns = is_v ? C::NV : C::NK;
      const int lb = blk - j0;
      const int st = lb % ns;
      uint64_t *full = (is_v ? v_full : k_full) + st;
      uint64_t *empty = (is_v ? v_empty : k_empty) + st;
      const int key0 = 128 * blk;
      const int np = (min(key0 + 128, last_pos + 1) - key0 + 15) / 16;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(empty, ((lb / ns) & 1) ^ 1, abort_flag, p.err, kErrWaitProducer);
        if (ok) mbar_arrive_expect_tx(full, np * C::NH * 2048);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return false;
      if (lane < np) {
        if (pg < 0 || pg >= p.num_pages) {
          atomicExch(p.err, kErrBounds);
          pg = 0;
        }
        const int z = (pg * 2 + (is_v ? 1 : 0)) * p.Hkv + hk;
        tma_load_5d((is_v ? sV : sK) + st * C::KV_BYTES + lane * C::PAGE_BYTES, &tmKV, full, 0, 0, 0, 0, z);
      }
      return true;
    };
    bool ok = true;
    // each ring keeps its own page ids for its current and next block
    int pk = page_of(j0), pk_next = page_of(j0 + 1), pv = pk, pv_next = pk_next;
    int kb = j0, vb = j0;   // next K and V block to load
    while (ok && vb < j_end) {
      if (kb < j_end && kb <= vb + AHEAD) {
        ok = load_block(false, kb, pk);
        ++kb;
        pk = pk_next;
        pk_next = page_of(kb + 1);
      } else {
        ok = load_block(true, vb, pv);
        ++vb;
        pv = pv_next;
        pv_next = page_of(vb + 1);
      }
    }
    if (lane == 0) {
      // let copies in flight land before the CTA exits (bounded), and the Q load
      const uint64_t t_start = globaltimer();
      if (!ok) {
        for (int b = max(0, kb - j0 - C::NK); b < kb - j0; ++b)
          while (!mbar_try_wait(smem_u32(&k_full[b % C::NK]), (b / C::NK) & 1) && globaltimer() - t_start < kWaitLimitNs) {
          }
        for (int b = max(0, vb - j0 - C::NV); b < vb - j0; ++b)
          while (!mbar_try_wait(smem_u32(&v_full[b % C::NV]), (b / C::NV) & 1) && globaltimer() - t_start < kWaitLimitNs) {
          }
      }
      while (!mbar_try_wait(smem_u32(q_full), 0) && globaltimer() - t_start < kWaitLimitNs) {
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      // j: the block's index in the tile; stages and phases count from j0
      // Matrix descriptors of the stage bases, built once; an operand at byte
      // offset `off` from a base is the base descriptor plus off / 16 (the
      // start-address field; shared-memory addresses stay below 2^18, so the
      // sum never carries out of it).
      const uint64_t qd0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t kd0 = sdesc_sw128(smem_u32(sK), 16, C::ATOM_STRIDE);
      const uint64_t vd0 = sdesc_sw128(smem_u32(sV), 1024, C::ATOM_STRIDE);
      auto issue_s = [&](int t, int j) {
        const uint32_t d = tmem + 128 * t;
        const uint64_t qd = qd0 + static_cast<uint64_t>((t * C::QT_BYTES) >> 4);
        const uint64_t kd = kd0 + static_cast<uint64_t>((((j - j0) % C::NK) * C::KV_BYTES) >> 4);
#pragma unroll
        for (int c = 0; c < C::NH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(d, qd + ((c * C::TILE_BYTES + kk * 32) >> 4), kd + ((c * 1024 + kk * 32) >> 4), C::IDESC_S,
                     (c > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&s_full[t]);
      };
      auto issue_pv = [&](int t, int j) {
        const uint64_t vd = vd0 + static_cast<uint64_t>((((j - j0) % C::NV) * C::KV_BYTES) >> 4);
        // P_t(j) sits in TMEM over S_t(j): 128 keys as 64 columns of bf16 pairs
        const uint32_t pcol = tmem + 128 * t;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)   // 16 keys (two atoms) per MMA; hd halves 1 KB apart
          mma_bf16_ts(tmem + C::O_COL + HD * t, pcol + ks * 8, vd + ((ks * 2 * C::ATOM_STRIDE) >> 4), C::IDESC_PV,
                      (j > j0 || ks > 0) ? 1u : 0u);
        // the last PV of a tile is covered by the o_last commit after the loop
        if (j + 1 < jt_end[t]) mma_commit(&o_full[t]);
      };
      auto wait = [&](uint64_t *bar, uint32_t par) { return mbar_wait(bar, par, abort_flag, p.err, kErrWaitMma); };
      // the last tile that reads block j (tile 1 reads every block it needs,
      // and needs at least the blocks of tile 0 when it has rows)
      auto last_tile = [&](int j) { return j < jt_end[1] ? 1 : 0; };
      bool ok = wait(q_full, 0) && wait(&k_full[0], 0);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (jt_end[t] > j0) issue_s(t, j0);
        if (C::NK < nb) mma_commit(&k_empty[0]);
      }
      // Block j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1); a tile that needs no
      // more blocks drops out.  A K block is released after the last S that
      // reads it, a V block after the last PV.
      for (int j = j0; j < j_end && ok; ++j) {
        const int lj = j - j0;
        ok = wait(&v_full[lj % C::NV], (lj / C::NV) & 1);
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= jt_end[t]) continue;
          ok = wait(&p_full[t], lj & 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(t, j);
          if (t == last_tile(j) && lj + C::NV < nb) mma_commit(&v_empty[lj % C::NV]);
          if (j + 1 < jt_end[t]) {
            ok = wait(&k_full[(lj + 1) % C::NK], ((lj + 1) / C::NK) & 1);
            if (!ok) break;
            tc_fence_after();
            issue_s(t, j + 1);
            if (t == last_tile(j + 1) && lj + 1 + C::NK < nb) mma_commit(&k_empty[(lj + 1) % C::NK]);
          }
        }
      }
      // One commit for all MMAs issued above (on every path), waited on here
      // too, so no MMA is in flight when the tile frees its TMEM.
      mma_commit(o_last);
      const uint64_t t_end = globaltimer();
      while (!mbar_try_wait(smem_u32(o_last), 0) && globaltimer() - t_end < kWaitLimitNs) {
      }
    }
  } else {
    // ------------------------------------------------- softmax / epilogue
    const int t = (warp - 2) >> 2;          // query tile of this warp group
    const int q = warp & 3;                 // TMEM lane quarter
    const int r = q * 32 + lane;            // row within the tile
    const int i = i0 + 128 * t + r;         // row within the chunk
    const int q_pos = cached + i;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t s_col = tmem + lane_base + 128 * t;
    const uint32_t o_col = tmem + lane_base + C::O_COL + HD * t;
    constexpr float kRescaleAbove = 8.f;     // log2 units
    const float scale = p.scale_log2;
    const int zero_t = nkb_t[0] == n_kb ? 0 : 1;   // the tile whose WG zeroes stale V rows
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = j0; j < jt_end[t]; ++j) {
      const int lj = j - j0;   // phases and stages count from the unit's first block
      bool bad = !ok || !mbar_wait(&s_full[t], lj & 1, abort_flag, p.err, kErrWaitSoftmax);
      bad = __any_sync(0xffffffffu, bad);   // tcgen05.ld below is warp-collective
      if (bad) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key0 = 128 * j;
      const bool full = key0 + 127 <= q_pos;   // every key of the block is visible to this row
      const int vis = q_pos - key0;            // else keys key0 .. key0 + vis are (vis < 127)
      // One pass over S while the reference holds: each half of the block's
      // 128 logits is loaded once, masked, and its probabilities
      // P = 2^(s scale - m_ref) are kept packed (bf16 pairs) in registers
      // beside the row's raw maximum.  If a row of the warp rose more than
      // 2^8 above its reference (always at the unit's first block, where
      // m_ref = -inf), the warp moves the reference, rescales O and takes the
      // probabilities again from S, which stays intact in TMEM until P is
      // stored at the end.  Pairs of logits go through the packed fp32 FMA and
      // add, and the maximum through 3-input max.
      uint32_t pk_lo[32], pk_hi[32];
      float2 lsum = make_float2(0.f, 0.f);
      float mq0 = -INFINITY, mq1 = -INFINITY, mq2 = -INFINITY, mq3 = -INFINITY;
      const float2 sc2 = make_float2(scale, scale);
      const bool have_ref = m_ref != -INFINITY;   // the same for every row of the warp
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float sv[64];
        tmem_ld64(s_col + 64 * hh, sv);
        if (!full)
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (64 * hh + c > vis) sv[c] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          mq0 = max3f(mq0, sv[c], sv[c + 1]);
          mq1 = max3f(mq1, sv[c + 2], sv[c + 3]);
          mq2 = max3f(mq2, sv[c + 4], sv[c + 5]);
          mq3 = max3f(mq3, sv[c + 6], sv[c + 7]);
        }
        if (have_ref) probs64(sv, sc2, m_ref, hh ? pk_hi : pk_lo, lsum);
      }
      const float mx = fmaxf(fmaxf(mq0, mq1), fmaxf(mq2, mq3)) * scale;
      const bool grow = !have_ref || (mx > m_ref + kRescaleAbove);
      if (__any_sync(0xffffffffu, grow)) {
        if (j > j0) {
          // O_t holds blocks < j relative to m_ref: finish PV_t(j-1), then rescale
          bad = !mbar_wait(&o_full[t], (lj - 1) & 1, abort_flag, p.err, kErrWaitSoftmax);
          bad = __any_sync(0xffffffffu, bad);
          if (bad) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = grow ? ex2_approx(m_ref - mx) : 1.f;
#pragma unroll
          for (int cc = 0; cc < HD / 32; ++cc) {
            float v[32];
            tmem_ld32(o_col + cc * 32, v);
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] *= alpha;
            tmem_st32(o_col + cc * 32, v);
          }
          if (grow) l *= alpha;
        }
        if (grow) m_ref = mx;
        lsum = make_float2(0.f, 0.f);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float sv[64];
          tmem_ld64(s_col + 64 * hh, sv);
          if (!full)
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (64 * hh + c > vis) sv[c] = -INFINITY;
          probs64(sv, sc2, m_ref, hh ? pk_hi : pk_lo, lsum);
        }
      }
      l += lsum.x + lsum.y;
      // P over S_t in TMEM: keys 0-63 in columns 0-31, keys 64-127 in 32-63
      tmem_st32u(s_col, pk_lo);
      tmem_st32u(s_col + 32, pk_hi);
      if (j == n_kb - 1 && t == zero_t) {
        // the block's V copies must have landed before they are patched
        bad = !mbar_wait(&v_full[lj % C::NV], (lj / C::NV) & 1, abort_flag, p.err, kErrWaitSoftmax);
        if (__any_sync(0xffffffffu, bad)) {
          ok = false;
          break;
        }
      }
      if (j == n_kb - 1 && t == zero_t && key0 + r > last_pos) {
        // keys past the tile's last position may be stale or non-finite in the
        // stage: zero their V rows so that P = 0 contributes exactly nothing.
        // One warp group does it (tile 0 if it reads this block), before its
        // P is ready; the other tile's PV is issued after this one's.
        uint8_t *vrow = sV + (lj % C::NV) * C::KV_BYTES + (r >> 3) * C::ATOM_STRIDE + (r & 7) * 128;
#pragma unroll
        for (int c = 0; c < C::NH; ++c)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4 *>(vrow + c * 1024 + k * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }
    const bool have = jt_end[t] > j0;   // this query tile has rows and blocks in this unit
    bool fin = ok;
    if (have && fin) fin = mbar_wait(o_last, 0, abort_flag, p.err, kErrWaitSoftmax) && !*abort_flag;
    fin = __all_sync(0xffffffffu, fin);   // tcgen05.ld below is warp-collective
    if (n_pieces == 1) {
      if (have && fin) {
        tc_fence_after();
        const bool valid = i < qo;
        const float inv = 1.f / l;
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + static_cast<size_t>(t0 + i) * (p.Hq * HD) + h * HD);
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
          float v[32];
          tmem_ld32(o_col + cc * 32, v);
          if (valid)
#pragma unroll
            for (int v8 = 0; v8 < 4; ++v8)
              dst[cc * 4 + v8] = make_uint4(pack_bf16x2(v[8 * v8] * inv, v[8 * v8 + 1] * inv),
                                            pack_bf16x2(v[8 * v8 + 2] * inv, v[8 * v8 + 3] * inv),
                                            pack_bf16x2(v[8 * v8 + 4] * inv, v[8 * v8 + 5] * inv),
                                            pack_bf16x2(v[8 * v8 + 6] * inv, v[8 * v8 + 7] * inv));
        }
      }
    } else if (!named_bar_or(2, 256, !fin)) {
      // A piece of a split tile: its unnormalised o with the row's reference
      // maximum m and sum l go to its partial slot; the last piece of the tile
      // to finish merges every piece by log-sum-exp,
      //   o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s.
      // All eight softmax warps take part (a tile without rows writes nothing).
      const int first = slot - unit[5];   // the tile's first partial slot
      if (have) {
        tc_fence_after();
        float *row = p.part + (static_cast<size_t>(slot) * 256 + 128 * t + r) * (HD + 4);
#pragma unroll
        for (int cc = 0; cc < HD / 32; ++cc) {
          float v[32];
          tmem_ld32(o_col + cc * 32, v);
          float4 *w4 = reinterpret_cast<float4 *>(row + cc * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k) w4[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
        row[HD] = m_ref;
        row[HD + 1] = l;
      }
      __threadfence();
      named_bar_sync(2, 256);
      if (threadIdx.x == 64) *merge_flag = atomicAdd(&p.ctr[first], 1) == n_pieces - 1;
      named_bar_sync(2, 256);
      if (*merge_flag) {
        __threadfence();
        // warp w takes rows w, w + 8, ...; lane s holds piece s's (m, l) (at
        // most 32 pieces) and the hd row is spread over the lanes
        const int w = warp - 2;
        constexpr int PER = HD / 32;
        for (int rr = w; rr < rows_valid; rr += 8) {
          const float *base = p.part + (static_cast<size_t>(first) * 256 + rr) * (HD + 4);
          const size_t pstride = static_cast<size_t>(256) * (HD + 4);
          float mv = -INFINITY, lv = 0.f;
          if (lane < n_pieces) {
            mv = base[lane * pstride + HD];
            lv = base[lane * pstride + HD + 1];
          }
          float M = mv;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
          const float wgt = lane < n_pieces ? exp2f(mv - M) : 0.f;
          float L = wgt * lv;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
          float acc[PER];
#pragma unroll
          for (int k = 0; k < PER; ++k) acc[k] = 0.f;
#pragma unroll 4
          for (int sp = 0; sp < n_pieces; ++sp) {
            const float ws = __shfl_sync(0xffffffffu, wgt, sp);
            const float *src = base + sp * pstride;
#pragma unroll
            for (int k = 0; k < PER; ++k) acc[k] = fmaf(ws, src[lane + 32 * k], acc[k]);
          }
          const float inv = 1.f / L;
          __nv_bfloat16 *dst = p.o + static_cast<size_t>(t0 + i0 + rr) * (p.Hq * HD) + h * HD;
#pragma unroll
          for (int k = 0; k < PER; ++k) dst[lane + 32 * k] = __float2bfloat16_rn(acc[k] * inv);
        }
        if (threadIdx.x == 64) p.ctr[first] = 0;   // ready for the next launch
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ============================================================ decode rows
// Persistent decode workers on the tensor cores.  A work item is {request,
// KV head, page range}; a worker CTA takes items from an atomic counter until
// none are left, so workers that start late (behind chunk tiles) simply take
// fewer.  For each 128-key block (8 pages) of an item:
//
//   S^T = K Q^T      M = 128 keys, N = 16 (the G q-heads of the group,
//                    padded), K = hd: K is staged by TMA page by page exactly
//                    as for the chunk tiles, Q^T is a 16-row tile of q
//   softmax          one thread per key; each head's block maximum and sum
//                    are reduced over the 128 threads, the running (m, l)
//                    per head is updated online (exp2 domain)
//   O^T_blk = V^T P^T  M = hd, N = 16, K = 128 keys: V is read as an
//                    MN-major A operand straight from its TMA stage, P^T is
//                    written by the softmax threads to shared memory
//   o = o alpha + O_blk  per thread = one hd row, in registers
//
// A block moves 64 KB of KV (hd 128) through a 3-stage ring; the producer
// runs on into the next item while the current one finishes, and the MMAs of
// the next block's S overlap the softmax of this one.  The work per KV byte
// on the CUDA cores is a few instructions per key, not G FMAs per element, so
// the stream runs at HBM speed.  Keys past kv_len in the last block are
// masked (their V rows are zeroed in shared memory so that P = 0 adds 0).
// The items' results go straight to o (single split) or to a partial row
// {o, m, l} for the merge pass.
struct DecodeParams {
  __nv_bfloat16 *o;
  float *part;
  const int32_t *qo_indptr, *kv_len, *bt_indptr, *bt, *items;
  int n_items, Hq, Hkv, num_pages, n_workers;
  float scale_log2;
  int *err;
  int *ctr;   // [0]: next item, [1]: workers done (the last one resets both)
  int *mctr;  // per split (request, KV head): splits finished (the merger resets it)
};

template <int HD>
struct DecCfg {
  static constexpr int NH = HD / 64;
  static constexpr int TILE = 128 * 128;                 // 128 keys x 64 bf16
  static constexpr int KV_STAGE = 2 * NH * TILE;         // K then V
  // K and V each as [8-key group][hd half][8 keys][128 B] (one copy per page)
  static constexpr int ATOM_STRIDE = NH * 1024;
  static constexpr int PAGE_BYTES = 2 * ATOM_STRIDE;
  static constexpr int STAGES = 3;
  static constexpr int QT = NH * 16 * 128;               // Q^T: [NH][16 rows][128 B]
  static constexpr int PT = 2 * 16 * 128;                // P^T: [2 key chunks][16 rows][128 B]
  static constexpr int OFF_Q = STAGES * KV_STAGE;
  static constexpr int OFF_P = OFF_Q + 2 * QT;
  static constexpr int OFF_HDR = OFF_P + 2 * PT;
  static constexpr int OFF_RED = OFF_HDR + STAGES * 32;
  static constexpr int OFF_FLAG = OFF_RED + 2 * 4 * 16 * 4;   // merge decision broadcast
  static constexpr int OFF_BAR = OFF_FLAG + 16;
  static constexpr int SMEM = OFF_BAR + 256;
  static constexpr uint32_t IDESC_S = idesc_bf16_ab(128, 16, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_ab(128, 16, true, false);
};

// Stage header written by the producer before it arms the stage.
struct DecHdr {
  int item;     // -1: no more items
  int nvalid;   // keys of the block below kv_len
  int flags;    // 1: first block of the item, 2: last block
  int qb;       // Q^T buffer of the item
};

template <int HD, int G>
__device__ __forceinline__ void decode_worker(const CUtensorMap &tmKV, const CUtensorMap &tmQd, const DecodeParams &p,
                                              uint8_t *smem) {
  using C = DecCfg<HD>;
  static_assert(G >= 1 && G <= 16, "a GQA group fills at most the 16 columns");
  uint8_t *sKV = smem;
  uint8_t *sQ = smem + C::OFF_Q;
  uint8_t *sP = smem + C::OFF_P;
  DecHdr *hdr = reinterpret_cast<DecHdr *>(smem + C::OFF_HDR);
  float *red = reinterpret_cast<float *>(smem + C::OFF_RED);     // [max | sum][4 warps][16]
  volatile int *merge_flag = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *k_full = bars;                   // [STAGES]: the block's K landed (and its header is set)
  uint64_t *v_full = bars + C::STAGES;       // [STAGES]: the block's V landed
  uint64_t *kv_empty = bars + 2 * C::STAGES; // [STAGES]
  uint64_t *q_full = bars + 3 * C::STAGES;   // [2]
  uint64_t *q_empty = q_full + 2;            // [2]
  uint64_t *s_full = q_full + 4;             // [2]
  uint64_t *s_empty = q_full + 6;            // [2]
  uint64_t *p_full = q_full + 8;             // [2]
  uint64_t *o_full = q_full + 10;            // [2]
  uint64_t *o_empty = q_full + 12;           // [2]
  uint64_t *mma_done = q_full + 14;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(q_full + 15);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], 128);
      mbar_init(&p_full[b], 128);
      mbar_init(&o_full[b], 1);
      mbar_init(&o_empty[b], 128);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmKV);
    prefetch_tmap(&tmQd);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 64);   // S^T x 2 (cols 0-31), O^T_blk x 2 (cols 32-63)
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // q, the KV pool, o and the work counter belong to earlier kernels
  pdl_trigger();

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    // The whole warp: lane 0 waits, fetches work and arms each stage, then
    // the block's 8 pages x (K, V) x hd chunks go out as one TMA per lane
    // (a single thread needs ~90 cycles per copy, which would pace the ring):
    // the K copies first (lanes 0-7), on a barrier of their own, so that the
    // block's S can start while its V is still arriving.  Global loads the
    // producer depends on (the next item, the next block's page ids, one per
    // lane) are issued a block ahead.
    const int my_pg = lane & 7, my_kv = lane >> 3;   // one copy per (page, K or V): lanes 0-15
    int seq = 0, k_local = 0;
    bool ok = true;
    int next_item = lane == 0 ? atomicAdd(&p.ctr[0], 1) : 0;
    while (ok) {
      const int item = __shfl_sync(0xffffffffu, next_item, 0);
      if (item >= p.n_items) {
        if (lane == 0) {
          const int s = seq % C::STAGES;
          if (mbar_wait(&kv_empty[s], ((seq / C::STAGES) & 1) ^ 1, abort_flag, p.err, kErrWaitProducer)) {
            hdr[s].item = -1;
            mbar_arrive(&k_full[s]);
          }
        }
        break;
      }
      if (lane == 0) next_item = atomicAdd(&p.ctr[0], 1);   // used at the next item
      const int32_t *it = p.items + item * 8;
      const int req = it[0], hk = it[1], pb = it[2], pe = it[3];
      const int t = p.qo_indptr[req];
      const int kv = p.kv_len[req];
      const int32_t *table = p.bt + p.bt_indptr[req];
      const int nblk = (pe - pb + 7) / 8;
      int nxt = lane < 8 && pb + lane < pe ? table[pb + lane] : 0;
      const int qb = k_local & 1;
      if (lane == 0) {
        ok = mbar_wait(&q_empty[qb], ((k_local >> 1) & 1) ^ 1, abort_flag, p.err, kErrWaitProducer);
        if (ok) {
          mbar_arrive_expect_tx(&q_full[qb], C::QT);
          for (int c = 0; c < C::NH; ++c)
            tma_load_2d(sQ + qb * C::QT + c * 2048, &tmQd, &q_full[qb], c * 64, t * p.Hq + hk * G);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (int b = 0; b < nblk && ok; ++b) {
        const int pg0 = pb + 8 * b;
        const int npg = min(8, pe - pg0);
        const int cur = nxt;
        if (b + 1 < nblk) nxt = lane < 8 && pg0 + 8 + lane < pe ? table[pg0 + 8 + lane] : 0;
        const int s = seq % C::STAGES;
        if (lane == 0) {
          ok = mbar_wait(&kv_empty[s], ((seq / C::STAGES) & 1) ^ 1, abort_flag, p.err, kErrWaitProducer);
          if (ok) {
            hdr[s].item = item;
            hdr[s].nvalid = min(npg * 16, kv - pg0 * 16);
            hdr[s].flags = (b == 0 ? 1 : 0) | (b == nblk - 1 ? 2 : 0);
            hdr[s].qb = qb;
            mbar_arrive_expect_tx(&k_full[s], npg * C::NH * 2048);
            mbar_arrive_expect_tx(&v_full[s], npg * C::NH * 2048);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        int page = __shfl_sync(0xffffffffu, cur, my_pg & 7);
        if (lane < 16 && my_pg < npg) {
          if (page < 0 || page >= p.num_pages) {
            atomicExch(p.err, kErrBounds);
            page = 0;
          }
          const int z = (page * 2 + my_kv) * p.Hkv + hk;
          tma_load_5d(sKV + s * C::KV_STAGE + my_kv * C::NH * C::TILE + my_pg * C::PAGE_BYTES, &tmKV,
                      my_kv ? &v_full[s] : &k_full[s], 0, 0, 0, 0, z);
        }
        ++seq;
      }
      ++k_local;
    }
    // on an abort, let copies in flight land before the CTA exits
    if (lane == 0 && (!ok || *abort_flag)) {
      for (int i = max(0, seq - C::STAGES); i < seq; ++i) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&k_full[i % C::STAGES]), (i / C::STAGES) & 1) &&
               globaltimer() - t0 < kWaitLimitNs) {
        }
        while (!mbar_try_wait(smem_u32(&v_full[i % C::STAGES]), (i / C::STAGES) & 1) &&
               globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      // Block j: S(j+1) as soon as its K (and Q) landed and S buffer (j+1)&1
      // is free; PV(j) as soon as P(j) is written and O_blk buffer j&1 is free.
      auto issue_s = [&](int j, int s, int qb) {
        const uint32_t d = tmem + (j & 1) * 16;
        const uint32_t k0 = smem_u32(sKV + s * C::KV_STAGE);
        const uint32_t q0 = smem_u32(sQ + qb * C::QT);
#pragma unroll
        for (int c = 0; c < C::NH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(d, sdesc_sw128(k0 + c * 1024 + kk * 32, 16, C::ATOM_STRIDE),
                     sdesc_sw128(q0 + c * 2048 + kk * 32, 16, 1024), C::IDESC_S, (c > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&s_full[j & 1]);
      };
      auto issue_pv = [&](int j, int s) {
        const uint32_t d = tmem + 32 + (j & 1) * 16;
        const uint32_t v0 = smem_u32(sKV + s * C::KV_STAGE + C::NH * C::TILE);
        const uint32_t p0 = smem_u32(sP + (j & 1) * C::PT);
#pragma unroll
        // 16 keys (two atoms) per MMA; the hd halves are 1 KB apart (hd 64: the
        // ignored upper 64 rows are read 16 KB on)
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16(d, sdesc_sw128(v0 + ks * 2 * C::ATOM_STRIDE, C::NH == 2 ? 1024 : C::TILE, C::ATOM_STRIDE),
                   sdesc_sw128(p0 + (ks >> 2) * 2048 + (ks & 3) * 32, 16, 1024), C::IDESC_PV, ks > 0 ? 1u : 0u);
        mma_commit(&o_full[j & 1]);
        mma_commit(&kv_empty[s]);
      };
      // S and PV advance independently: S(ns) goes out as soon as its K (and
      // the item's Q) landed and S buffer ns&1 is free, PV(np) as soon as P(np)
      // is written and O_blk buffer np&1 is free.
      int ns = 0, npv = 0, qcount = 0;   // qcount: items whose Q^T the S MMAs are done with
      bool s_end = false, ok = true;
      uint64_t t_idle = globaltimer();
      for (uint32_t spin = 0;; ++spin) {
        bool progress = false;
        if (!s_end) {
          const int s = ns % C::STAGES;
          if (mbar_test_wait(smem_u32(&k_full[s]), (ns / C::STAGES) & 1)) {
            if (hdr[s].item < 0) {
              s_end = progress = true;
            } else {
              const int qb = hdr[s].qb;
              const bool need_q = hdr[s].flags & 1;
              if ((!need_q || mbar_test_wait(smem_u32(&q_full[qb]), (qcount >> 1) & 1)) &&
                  mbar_test_wait(smem_u32(&s_empty[ns & 1]), ((ns >> 1) & 1) ^ 1)) {
                tc_fence_after();
                issue_s(ns, s, qb);
                if (hdr[s].flags & 2) {
                  mma_commit(&q_empty[qb]);
                  ++qcount;
                }
                ++ns;
                progress = true;
              }
            }
          }
        }
        if (npv < ns && mbar_test_wait(smem_u32(&p_full[npv & 1]), (npv >> 1) & 1) &&
            mbar_test_wait(smem_u32(&o_empty[npv & 1]), ((npv >> 1) & 1) ^ 1) &&
            mbar_test_wait(smem_u32(&v_full[npv % C::STAGES]), (npv / C::STAGES) & 1)) {
          tc_fence_after();
          issue_pv(npv, npv % C::STAGES);
          ++npv;
          progress = true;
        }
        if (s_end && npv == ns) break;
        if (progress) {
          t_idle = globaltimer();
        } else if ((spin & 15u) == 15u) {
          if (*abort_flag) {
            ok = false;
            break;
          }
          if (globaltimer() - t_idle > kWaitLimitNs) {
            *abort_flag = 1;
            atomicExch(p.err, kErrWaitMma);
            ok = false;
            break;
          }
        }
      }
      (void)ok;
      // every MMA issued above has completed before TMEM is freed
      mma_commit(mma_done);
      const uint64_t t_end = globaltimer();
      while (!mbar_try_wait(smem_u32(mma_done), 0) && globaltimer() - t_end < kWaitLimitNs) {
      }
    }
  } else if (warp < 6) {
    // ---------------------------------------------- softmax / accumulation
    // Per block, one barrier-OR asks whether any logit rose more than 2^8
    // above its head's reference m; only then do the warps exchange the block
    // maxima and move m (O and the sums rescaled by alpha).  Softmax does not
    // depend on the reference, and every exponent stays <= 8, so P < 2^8.
    // Each thread keeps its own partial sum of P; the 128 partials of a head
    // are added once, when the item ends.
    constexpr float kRescaleAbove = 8.f;     // log2 units
    const int q = warp & 3;
    const int t = q * 32 + lane;             // key of the block (S^T lane) and hd row (O^T lane)
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    float m[G], l[G], o[G], alpha_prev[G];   // l: this thread's partial sum
    bool ok = true;
    for (int j = 0;; ++j) {
      const int s = j % C::STAGES;
      bool bad = !ok || !mbar_wait(&k_full[s], (j / C::STAGES) & 1, abort_flag, p.err, kErrWaitSoftmax);
      const DecHdr h = hdr[s];
      if (named_bar_or(1, 128, bad) || h.item < 0) break;
      bad = !mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, p.err, kErrWaitSoftmax);
      bad = __any_sync(0xffffffffu, bad);
      float sv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) sv[i] = 0.f;
      if (!bad) {
        tc_fence_after();
        tmem_ld16(tmem + lane_base + (j & 1) * 16, sv);
      }
      tc_fence_before();
      mbar_arrive(&s_empty[j & 1]);
      if (h.flags & 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          m[g] = -INFINITY;
          l[g] = 0.f;
          o[g] = 0.f;
        }
      }
      const bool valid = t < h.nvalid;
      float sc[G], alpha[G];
      bool grow = false;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        sc[g] = valid ? sv[g] * p.scale_log2 : -INFINITY;
        grow |= sc[g] > m[g] + kRescaleAbove;   // always at an item's first block
        alpha[g] = 1.f;
      }
      if (named_bar_or(1, 128, bad || grow)) {
        if (named_bar_or(1, 128, bad)) {
          ok = false;
          break;
        }
        float mx[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          mx[g] = sc[g];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], off));
        }
        if (lane == 0)
#pragma unroll
          for (int g = 0; g < G; ++g) red[q * 16 + g] = mx[g];
        named_bar_sync(1, 128);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float bm = fmaxf(fmaxf(red[g], red[16 + g]), fmaxf(red[32 + g], red[48 + g]));
          const float mn = fmaxf(m[g], bm);
          alpha[g] = (m[g] == -INFINITY) ? 0.f : ex2_approx(m[g] - mn);
          m[g] = mn;
        }
      }
      float pr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) pr[g] = ex2_approx(sc[g] - m[g]);   // 0 for masked keys
      // P^T[g][t] into the K-major 128-byte-swizzled B tile (two 64-key chunks)
      uint8_t *pt = sP + (j & 1) * C::PT + (t >> 6) * 2048;
#pragma unroll
      for (int g = 0; g < G; ++g)
        *reinterpret_cast<__nv_bfloat16 *>(pt + sw128_offset(g, t & 63)) = __float2bfloat16_rn(pr[g]);
      if (h.nvalid < 128 && !mbar_wait(&v_full[s], (j / C::STAGES) & 1, abort_flag, p.err, kErrWaitSoftmax))
        ok = false;   // the V rows below must have landed before they are patched
      if (!valid && ok) {
        // a key past kv_len: its V row may hold anything; make it exactly 0
        uint8_t *vrow = sKV + s * C::KV_STAGE + C::NH * C::TILE + (t >> 3) * C::ATOM_STRIDE + (t & 7) * 128;
#pragma unroll
        for (int c = 0; c < C::NH; ++c)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4 *>(vrow + c * 1024 + k * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      mbar_arrive(&p_full[j & 1]);
#pragma unroll
      for (int g = 0; g < G; ++g) l[g] = fmaf(l[g], alpha[g], pr[g]);
      // O^T_blk(i): row t = hd element t, column g = head.  Block j-1 is
      // folded in here, after this block's softmax, so that PV(j-1) ran
      // meanwhile; an item's last block is folded at once.
      auto fold = [&](int i, const float (&al)[G]) -> bool {
        const bool b = __any_sync(0xffffffffu, !mbar_wait(&o_full[i & 1], (i >> 1) & 1, abort_flag, p.err,
                                                          kErrWaitSoftmax));
        float ob[16];
        if (!b) {
          tc_fence_after();
          tmem_ld16(tmem + lane_base + 32 + (i & 1) * 16, ob);
        }
        tc_fence_before();
        mbar_arrive(&o_empty[i & 1]);
        if (!b)
#pragma unroll
          for (int g = 0; g < G; ++g) o[g] = fmaf(o[g], al[g], ob[g]);
        return !b;
      };
      // a failed wait leaves via the next block's first barrier-OR
      if (!(h.flags & 1) && !fold(j - 1, alpha_prev)) ok = false;
#pragma unroll
      for (int g = 0; g < G; ++g) alpha_prev[g] = alpha[g];
      if (!(h.flags & 2)) continue;
      if (ok && !fold(j, alpha)) ok = false;
      // the item's sums: the partials of the 128 threads, per head
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float sw = l[g];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, off);
        if (lane == 0) red[64 + q * 16 + g] = sw;
      }
      // all or none enter the barriers below; the barrier also publishes the sums
      if (named_bar_or(1, 128, !ok)) break;
      float lsum[G];
#pragma unroll
      for (int g = 0; g < G; ++g) lsum[g] = (red[64 + g] + red[80 + g]) + (red[96 + g] + red[112 + g]);
      // ---- the item is done: its output, or its split's partial
      const int32_t *it = p.items + h.item * 8;
      const int req = it[0], hk = it[1], sidx = it[4], n_splits = it[5], grp = it[6], pbase = it[7];
      const size_t tok = static_cast<size_t>(p.qo_indptr[req]);
      if (n_splits == 1) {
        if (t < HD)
#pragma unroll
          for (int g = 0; g < G; ++g)
            p.o[(tok * p.Hq + hk * G + g) * HD + t] = __float2bfloat16_rn(o[g] / lsum[g]);
        continue;
      }
      if (t < HD)
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float *dst = p.part + (static_cast<size_t>(pbase + sidx) * G + g) * part_stride<HD>();
          dst[t] = o[g];
          if (t == 0) {
            dst[HD] = m[g];
            dst[HD + 1] = lsum[g];
          }
        }
      // The last split of the (request, KV head) to finish merges all of its
      // partials by log-sum-exp: o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
      __threadfence();
      named_bar_sync(1, 128);
      if (t == 0) *merge_flag = atomicAdd(&p.mctr[grp], 1) == n_splits - 1;
      named_bar_sync(1, 128);
      if (*merge_flag) {
        // warp q takes heads q, q + 4, ...; lane s holds split s's (m, l)
        // (at most 32 splits), the hd row is spread over the lanes, and the
        // loads of consecutive splits are independent, so a merge costs a few
        // L2 round trips rather than one per split
        __threadfence();
        const float *first = p.part + static_cast<size_t>(pbase) * G * part_stride<HD>();
        constexpr int PER = HD / 32;
        for (int g = q; g < G; g += 4) {
          float mv = -INFINITY, lv = 0.f;
          if (lane < n_splits) {
            const float *src = first + (static_cast<size_t>(lane) * G + g) * part_stride<HD>();
            mv = src[HD];
            lv = src[HD + 1];
          }
          float M = mv;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
          const float w = lane < n_splits ? exp2f(mv - M) : 0.f;
          float L = w * lv;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
          float acc[PER];
#pragma unroll
          for (int k = 0; k < PER; ++k) acc[k] = 0.f;
#pragma unroll 4
          for (int sp = 0; sp < n_splits; ++sp) {
            const float ws = __shfl_sync(0xffffffffu, w, sp);
            const float *src = first + (static_cast<size_t>(sp) * G + g) * part_stride<HD>();
#pragma unroll
            for (int k = 0; k < PER; ++k) acc[k] = fmaf(ws, src[lane + 32 * k], acc[k]);
          }
          const float inv = 1.f / L;
#pragma unroll
          for (int k = 0; k < PER; ++k)
            p.o[(tok * p.Hq + hk * G + g) * HD + lane + 32 * k] = __float2bfloat16_rn(acc[k] * inv);
        }
        if (t == 0) p.mctr[grp] = 0;   // ready for the next launch
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
  if (threadIdx.x == 0) {
    // the last worker out resets the counter for the next launch
    __threadfence();
    if (atomicAdd(&p.ctr[1], 1) == p.n_workers - 1) {
      p.ctr[0] = 0;
      p.ctr[1] = 0;
      __threadfence();
    }
  }
}

// ============================================================ one grid
// The ragged attention of a step is ONE launch: blocks [0, n_tiles) run a
// prefill-chunk tile (tensor cores, compute-heavy), the rest are persistent
// decode workers (tensor cores, HBM stream) that take decode items until none
// are left, so the two kinds share the GPU instead of running back to back.
// Tiles come first, heaviest first; workers fill SMs as they free up.
template <int HD>
struct FusedCfg {
  static constexpr int THREADS = ChunkCfg<HD>::THREADS;   // 10 warps
  static constexpr int SMEM = ChunkCfg<HD>::SMEM > DecCfg<HD>::SMEM ? ChunkCfg<HD>::SMEM : DecCfg<HD>::SMEM;
  using D = DecCfg<HD>;
  // the decode worker's V^T operand reads 128 hd rows; for hd 64 the upper 64
  // (ignored) rows of the last stage lie past it and must stay in this CTA
  static_assert((D::STAGES - 1) * D::KV_STAGE + D::NH * D::TILE + 2 * D::TILE <= SMEM, "V^T over-read");
  static_assert(THREADS >= 6 * 32, "the decode worker uses warps 0-5");
};

template <int HD, int G>
__global__ void __launch_bounds__(FusedCfg<HD>::THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                     const __grid_constant__ CUtensorMap tmQd, const ChunkParams cp, const DecodeParams dp,
                     int n_tiles) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    // the layouts above need a 1024-aligned base and reserve no slack
    pdl_wait();
    if (threadIdx.x == 0) atomicExch(cp.err, kErrBounds);
    return;
  }
  if (static_cast<int>(blockIdx.x) < n_tiles)
    chunk_tile<HD>(tmQ, tmKV, cp, blockIdx.x, smem_raw);   // waits for earlier kernels after its set-up
  else
    decode_worker<HD, G>(tmKV, tmQd, dp, smem_raw);       // likewise
}

template <int HD, int G>
cudaError_t launch_attention(const CUtensorMap &tq, const CUtensorMap &tkv, const CUtensorMap &tqd,
                             const ChunkParams &cp, const DecodeParams &dp, int n_tiles, cudaStream_t st) {
  const cudaError_t attr_err =
      ensure_max_smem(reinterpret_cast<const void *>(attention_kernel<HD, G>), FusedCfg<HD>::SMEM);
  if (attr_err != cudaSuccess) return attr_err;
  return launch_pdl(attention_kernel<HD, G>, dim3(n_tiles + dp.n_workers), dim3(FusedCfg<HD>::THREADS),
                    FusedCfg<HD>::SMEM, st, 1, tq, tkv, tqd, cp, dp, n_tiles);
}

template <int HD>
cudaError_t launch_attention_g(const CUtensorMap &tq, const CUtensorMap &tkv, const CUtensorMap &tqd,
                               const ChunkParams &cp, const DecodeParams &dp, int n_tiles, int G, cudaStream_t st) {
  switch (G) {
    case 1: return launch_attention<HD, 1>(tq, tkv, tqd, cp, dp, n_tiles, st);
    case 2: return launch_attention<HD, 2>(tq, tkv, tqd, cp, dp, n_tiles, st);
    case 3: return launch_attention<HD, 3>(tq, tkv, tqd, cp, dp, n_tiles, st);
    case 4: return launch_attention<HD, 4>(tq, tkv, tqd, cp, dp, n_tiles, st);
    case 5: return launch_attention<HD, 5>(tq, tkv, tqd, cp, dp, n_tiles, st);
    case 6: return launch_attention<HD, 6>(tq, tkv, tqd, cp, dp, n_tiles, st);
    case 7: return launch_attention<HD, 7>(tq, tkv, tqd, cp, dp, n_tiles, st);
    case 8: return launch_attention<HD, 8>(tq, tkv, tqd, cp, dp, n_tiles, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t attention_run(const AttnArgs &a, cudaStream_t st) {
  if (a.n_tiles + a.n_items <= 0) return cudaSuccess;
  const float scale_log2 = kLog2e / sqrtf(static_cast<float>(a.hd));
  ChunkParams cp;
  cp.o = static_cast<__nv_bfloat16 *>(a.o);
  cp.qo_indptr = a.qo_indptr;
  cp.kv_len = a.kv_len;
  cp.bt_indptr = a.bt_indptr;
  cp.bt = a.bt;
  cp.tiles = a.tiles;
  cp.Hq = a.Hq;
  cp.Hkv = a.Hkv;
  cp.num_pages = a.num_pages;
  cp.scale_log2 = scale_log2;
  cp.err = a.err;
  cp.part = a.chunk_part;
  cp.ctr = a.chunk_ctr;
  DecodeParams dp;
  dp.o = static_cast<__nv_bfloat16 *>(a.o);
  dp.part = a.part;
  dp.qo_indptr = a.qo_indptr;
  dp.kv_len = a.kv_len;
  dp.bt_indptr = a.bt_indptr;
  dp.bt = a.bt;
  dp.items = a.items;
  dp.n_items = a.n_items;
  dp.Hq = a.Hq;
  dp.Hkv = a.Hkv;
  dp.num_pages = a.num_pages;
  dp.scale_log2 = scale_log2;
  dp.err = a.err;
  dp.ctr = a.dec_ctr;
  dp.mctr = a.merge_ctr;
  const int sms = device_sm_count();
  const int cap = a.max_workers > 0 && a.max_workers < sms ? a.max_workers : sms;
  dp.n_workers = a.n_items < cap ? a.n_items : cap;
  const int G = a.Hq / a.Hkv;
  return a.hd == 128 ? launch_attention_g<128>(*a.tm_q, *a.tm_kv, *a.tm_qd, cp, dp, a.n_tiles, G, st)
                     : launch_attention_g<64>(*a.tm_q, *a.tm_kv, *a.tm_qd, cp, dp, a.n_tiles, G, st);
}

}  // namespace mb
