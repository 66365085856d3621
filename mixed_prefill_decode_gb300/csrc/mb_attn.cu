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
template <int HD>
struct ChunkCfg {
  static constexpr int NH = HD / 64;              // 64-wide swizzle chunks along hd
  static constexpr int TILE_BYTES = 128 * 128;    // [128 rows][64 bf16]
  static constexpr int Q_BYTES = NH * TILE_BYTES;
  static constexpr int KV_BYTES = NH * TILE_BYTES;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int NKV = 3;                   // K/V stages
  static constexpr int OFF_V = OFF_K + NKV * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + NKV * KV_BYTES;
  static constexpr int OFF_RED = OFF_BAR + 128;   // softmax row max / sum exchange
  // The kernel checks that the dynamic shared memory starts 1024-aligned, so
  // no alignment slack is reserved (it would not fit beside three stages).
  static constexpr int SMEM = OFF_RED + 4 * 128 * 4;
  static constexpr int THREADS = 320;             // TMA, MMA, 8 softmax warps
  static constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, HD, true);
  static constexpr uint32_t TMEM_COLS = 512;      // S0 [0,128), S1 [128,256), O [256, 256+HD)
};

struct ChunkParams {
  __nv_bfloat16 *o;
  const int32_t *qo_indptr, *kv_len, *bt_indptr, *bt, *tiles;
  int Hq, Hkv, num_pages;
  float scale_log2;
  int *err;
};

// One prefill-chunk tile (128 query rows x one q-head); needs
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
  uint64_t *kv_full = bars + 1;   // [NKV]
  uint64_t *kv_empty = bars + 4;  // [NKV]
  uint64_t *s_full = bars + 7;    // [2]
  uint64_t *p_full = bars + 9;    // [2]
  uint64_t *o_full = bars + 11;   // PV(j) done, j < n_kb - 1
  uint64_t *o_last = bars + 12;   // every MMA of the tile done (committed once)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 13);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int req = p.tiles[tile * 4 + 0];
  const int i0 = p.tiles[tile * 4 + 1];
  const int h = p.tiles[tile * 4 + 2];
  const int t0 = p.qo_indptr[req];
  const int qo = p.qo_indptr[req + 1] - t0;
  const int kv = p.kv_len[req];
  const int cached = kv - qo;
  const int rows_valid = min(128, qo - i0);
  const int last_pos = cached + i0 + rows_valid - 1;
  const int n_kb = (last_pos + 1 + 127) / 128;
  const int hk = h / (p.Hq / p.Hkv);
  const int32_t *table = p.bt + p.bt_indptr[req];

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NKV; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full[0], 256);
    mbar_init(&p_full[1], 256);
    mbar_init(o_full, 1);
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

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      for (int c = 0; c < C::NH; ++c) tma_load_2d(sQ + c * C::TILE_BYTES, &tmQ, q_full, h * HD + c * 64, t0 + i0);
      uint32_t issued = 0, issued_ph = 0;
      bool ok = true;
      for (int j = 0; j < n_kb && ok; ++j) {
        const int s = j % C::NKV;
        const uint32_t ph = (j / C::NKV) & 1;
        if (!mbar_wait(&kv_empty[s], ph ^ 1, abort_flag, p.err, kErrWaitProducer)) {
          ok = false;
          break;
        }
        const int key0 = 128 * j;
        const int key_end = min(key0 + 128, last_pos + 1);
        const int np = (key_end - key0 + 15) / 16;
        mbar_arrive_expect_tx(&kv_full[s], np * 2 * C::NH * 2048);
        for (int pg = 0; pg < np; ++pg) {
          int page = table[key0 / 16 + pg];
          if (page < 0 || page >= p.num_pages) {
            atomicExch(p.err, kErrBounds);
            page = 0;
          }
          const int zk = (page * 2 + 0) * p.Hkv + hk;
          const int zv = (page * 2 + 1) * p.Hkv + hk;
          for (int c = 0; c < C::NH; ++c) {
            tma_load_3d(sK + s * C::KV_BYTES + c * C::TILE_BYTES + pg * 2048, &tmKV, &kv_full[s], c * 64, 0, zk);
            tma_load_3d(sV + s * C::KV_BYTES + c * C::TILE_BYTES + pg * 2048, &tmKV, &kv_full[s], c * 64, 0, zv);
          }
        }
        issued |= 1u << s;
        issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
      }
      if (!ok) {
        for (int s = 0; s < C::NKV; ++s)
          if (issued & (1u << s)) {
            const uint64_t t_start = globaltimer();
            while (!mbar_try_wait(smem_u32(&kv_full[s]), (issued_ph >> s) & 1u) &&
                   globaltimer() - t_start < kWaitLimitNs) {
            }
          }
      }
      // the Q load is always in flight once issued; make sure it landed
      {
        const uint64_t t_start = globaltimer();
        while (!mbar_try_wait(smem_u32(q_full), 0) && globaltimer() - t_start < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      auto issue_s = [&](int j) {
        const int b = j & 1;                 // S buffer in TMEM
        const int s = j % C::NKV;            // K/V stage
        const uint32_t d = tmem + b * 128;
        const uint32_t q0 = smem_u32(sQ);
        const uint32_t k0 = smem_u32(sK + s * C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::NH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sdesc_sw128(q0 + c * C::TILE_BYTES + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(k0 + c * C::TILE_BYTES + kk * 32, 16, 1024);
            mma_bf16(d, ad, bd, C::IDESC_S, (c > 0 || kk > 0) ? 1u : 0u);
          }
        mma_commit(&s_full[b]);
      };
      auto issue_pv = [&](int j) {
        const int b = j & 1;
        const int s = j % C::NKV;
        const uint32_t vbase = smem_u32(sV + s * C::KV_BYTES);
        // P(j) sits in TMEM over S(j): 128 keys as 64 columns of bf16 pairs
        const uint32_t pcol = tmem + b * 128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // 16 keys per MMA
          const uint64_t bd = sdesc_sw128(vbase + ks * 2048, C::TILE_BYTES, 1024);
          mma_bf16_ts(tmem + 256, pcol + ks * 8, bd, C::IDESC_PV, (j > 0 || ks > 0) ? 1u : 0u);
        }
        // the last PV is covered by the o_last commit after the loop; stages
        // the producer will not refill get no release (nothing waits on it)
        if (j + 1 < n_kb) mma_commit(o_full);
        if (j + C::NKV < n_kb) mma_commit(&kv_empty[s]);
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, p.err, kErrWaitMma);
      if (ok) ok = mbar_wait(&kv_full[0], 0, abort_flag, p.err, kErrWaitMma);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      // Block j: S(j+1) as soon as its K/V landed, PV(j) as soon as P(j) is
      // ready, in whichever order they come (neither waits on the other).
      for (int j = 0; j < n_kb && ok; ++j) {
        bool s_done = j + 1 >= n_kb, pv_done = false;
        const uint32_t kv_bar = smem_u32(&kv_full[(j + 1) % C::NKV]);
        const uint32_t kv_par = ((j + 1) / C::NKV) & 1;
        const uint32_t p_bar = smem_u32(&p_full[j & 1]);
        const uint32_t p_par = (j >> 1) & 1;
        const uint64_t t_start = globaltimer();
        for (uint32_t spin = 0; !(s_done && pv_done); ++spin) {
          if (!s_done && mbar_test_wait(kv_bar, kv_par)) {
            tc_fence_after();
            issue_s(j + 1);
            s_done = true;
          }
          if (!pv_done && mbar_test_wait(p_bar, p_par)) {
            tc_fence_after();
            issue_pv(j);
            pv_done = true;
          }
          if ((spin & 63u) == 63u) {
            if (*abort_flag) {
              ok = false;
              break;
            }
            if (globaltimer() - t_start > kWaitLimitNs) {
              *abort_flag = 1;
              atomicExch(p.err, kErrWaitMma);
              ok = false;
              break;
            }
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
    // 8 warps: two per TMEM lane quarter, splitting the 128 key columns of S
    // (and the hd columns of O) in halves; a row's max and sum are combined
    // through shared memory once per key block.  O accumulates in TMEM (the
    // PV MMA adds each block); a row is rescaled only when its maximum grows
    // by more than 2^8 over the reference it uses, so probabilities stay
    // <= 256 and most blocks never wait for the previous PV.
    const int q = warp & 3;
    const int hh = (warp - 2) >> 2;          // column half
    const int r = q * 32 + lane;
    const int q_pos = cached + i0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    constexpr int OH = HD / 2;               // O columns per half
    constexpr float kRescaleAbove = 8.f;     // log2 units
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);  // [2 bufs][2 halves][128]
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    bool bad = false;
    for (int j = 0; j < n_kb; ++j) {
      const int b = j & 1;
      bad = !ok || !mbar_wait(&s_full[b], (j >> 1) & 1, abort_flag, p.err, kErrWaitSoftmax);
      bad = __any_sync(0xffffffffu, bad);   // tcgen05.ld below is warp-collective
      tc_fence_after();
      const int key0 = 128 * j + hh * 64;   // first key of this thread's half
      const bool full = (key0 + 63 <= q_pos) && (key0 + 63 < kv);
      const uint32_t scol = tmem + lane_base + b * 128 + hh * 64;
      // pass 1: this half row of S into registers, and its visible maximum
      float sv[64];
      float mx = -INFINITY;
      if (!bad) {
        tmem_ld64(scol, sv);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          sv[i] *= p.scale_log2;
          if (!full) {
            const int key = key0 + i;
            if (!(key <= q_pos && key < kv)) sv[i] = -INFINITY;
          }
          mx = fmaxf(mx, sv[i]);
        }
      }
      red[(b * 2 + hh) * 128 + r] = mx;
      // every thread is past its reads of S(j) here, so P(j) may overwrite it
      if (named_bar_or(2, 256, bad)) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, red[(b * 2 + (hh ^ 1)) * 128 + r]);
      const bool grow = (m_ref == -INFINITY) || (mx > m_ref + kRescaleAbove);
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O holds blocks < j relative to m_ref: finish PV(j-1), then rescale
        bad = !mbar_wait(o_full, (j - 1) & 1, abort_flag, p.err, kErrWaitSoftmax);
        bad = __any_sync(0xffffffffu, bad);
        if (bad) {
          ok = false;
          continue;
        }
        tc_fence_after();
        const float alpha = grow ? exp2f(m_ref - mx) : 1.f;
#pragma unroll
        for (int cc = 0; cc < OH / 32; ++cc) {
          float v[32];
          tmem_ld32(tmem + lane_base + 256 + hh * OH + cc * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= alpha;
          tmem_st32(tmem + lane_base + 256 + hh * OH + cc * 32, v);
        }
        if (grow) l *= alpha;
      }
      if (grow) m_ref = mx;
      // pass 2: probabilities relative to m_ref -> bf16 pairs into TMEM over S(j)
      float pk[32];
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float p0 = exp2f(sv[i] - m_ref);
        const float p1 = exp2f(sv[i + 1] - m_ref);
        l += p0 + p1;
        pk[i / 2] = __uint_as_float(pack_bf16x2(p0, p1));
      }
      tmem_st32(tmem + lane_base + b * 128 + hh * 32, pk);
      if (j == n_kb - 1 && 128 * j + r > last_pos) {
        // rows past the last visible key may hold stale or non-finite data:
        // zero them so that P = 0 rows contribute exactly nothing
        uint8_t *vrow = sV + (j % C::NKV) * C::KV_BYTES + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int c = 0; c < C::NH; ++c)
          if ((c & 1) == hh)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<uint4 *>(vrow + c * C::TILE_BYTES + k * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    // row sum over both halves (reuses the exchange buffer of the parity the
    // last block did not use, so no reader of the last maxima is overtaken)
    float *lsum = red + (((n_kb - 1) & 1) ^ 1) * 256;
    lsum[hh * 128 + r] = l;
    named_bar_sync(2, 256);
    l += lsum[(hh ^ 1) * 128 + r];
    if (ok && mbar_wait(o_last, 0, abort_flag, p.err, kErrWaitSoftmax) && !*abort_flag) {
      tc_fence_after();
      float o_acc[OH];
#pragma unroll
      for (int cc = 0; cc < OH / 32; ++cc)
        tmem_ld32(tmem + lane_base + 256 + hh * OH + cc * 32, *reinterpret_cast<float(*)[32]>(&o_acc[cc * 32]));
      if (i0 + r < qo) {
        const float inv = 1.f / l;
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + static_cast<size_t>(t0 + i0 + r) * (p.Hq * HD) + h * HD + hh * OH);
#pragma unroll
        for (int v8 = 0; v8 < OH / 8; ++v8)
          dst[v8] = make_uint4(pack_bf16x2(o_acc[8 * v8] * inv, o_acc[8 * v8 + 1] * inv),
                               pack_bf16x2(o_acc[8 * v8 + 2] * inv, o_acc[8 * v8 + 3] * inv),
                               pack_bf16x2(o_acc[8 * v8 + 4] * inv, o_acc[8 * v8 + 5] * inv),
                               pack_bf16x2(o_acc[8 * v8 + 6] * inv, o_acc[8 * v8 + 7] * inv));
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
struct DecodeParams {
  const __nv_bfloat16 *q;
  const __nv_bfloat16 *pool;
  __nv_bfloat16 *o;
  float *part;
  const int32_t *qo_indptr, *kv_len, *bt_indptr, *bt, *items;
  int n_items, Hq, Hkv, num_pages;
  float scale_log2;
  int *err;
};

// One CTA per work item {request, KV head, page range}.  Warp 4 streams the
// K and V blocks of each (page, head) -- contiguous 16 x hd bf16 in the HND
// pool -- into a ring of shared-memory slots with bulk copies; warps 0-3 take
// every fourth page.  A warp serves all G q-heads of the GQA group: HD/8
// lanes share a key (8 bf16 = one 16-byte shared load each), scores are
// reduced across those lanes with a transposed butterfly (each lane ends with
// the score of one key), and each key costs one exp2 per head.  The warps'
// (m, l, o) are merged in shared memory at the end.
template <int HD>
struct DecCfg {
  static constexpr int PAGE_BYTES = 16 * HD * 2;
  static constexpr int SLOT_BYTES = 2 * PAGE_BYTES;
  static constexpr int LPK = HD / 8;            // lanes per key
  static constexpr int KPS = 32 / LPK;          // keys per step
  static constexpr int STEPS = 16 / KPS;
};

__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

__device__ __forceinline__ float2 bf2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

// NW consumer warps (warps 0 .. NW-1) and one producer warp (warp NW);
// further warps of the CTA idle.  `dsm` holds NSLOT ring slots, then the
// barriers.
template <int HD, int G, int NW, int NSLOT>
__device__ __forceinline__ void decode_item(const DecodeParams &p, int item, uint8_t *dsm, int warp_base,
                                            int bar_id) {
  using C = DecCfg<HD>;
  constexpr int RING = NSLOT * C::SLOT_BYTES;
  uint8_t *ring = dsm;
  uint64_t *full = reinterpret_cast<uint64_t *>(dsm + RING);
  uint64_t *empty = full + NSLOT;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + NSLOT);

  const int warp = (threadIdx.x >> 5) - warp_base, lane = threadIdx.x & 31;
  const int tid = threadIdx.x - warp_base * 32;   // 0 .. (NW + 1) * 32 - 1
  const int32_t *it = p.items + item * 8;
  const int req = it[0], hk = it[1], pb = it[2], pe = it[3], n_splits = it[5];
  const int np = pe - pb;
  const int t = p.qo_indptr[req];
  const int kv = p.kv_len[req];
  const int32_t *table = p.bt + p.bt_indptr[req];

  if (tid == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  named_bar_sync(bar_id, (NW + 1) * 32);

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const size_t head_stride = static_cast<size_t>(16) * HD;
      int last_slot_issued = -1;
      for (int i = 0; i < np; ++i) {
        const int slot = i % NSLOT;
        if (i >= NSLOT &&
            !mbar_wait(&empty[slot], ((i / NSLOT) - 1) & 1, abort_flag, p.err, kErrWaitProducer))
          break;
        int page = table[pb + i];
        if (page < 0 || page >= p.num_pages) {
          atomicExch(p.err, kErrBounds);
          page = 0;
        }
        const __nv_bfloat16 *kb = p.pool + ((static_cast<size_t>(page) * 2 + 0) * p.Hkv + hk) * head_stride;
        const __nv_bfloat16 *vb = kb + static_cast<size_t>(p.Hkv) * head_stride;
        mbar_arrive_expect_tx(&full[slot], 2 * C::PAGE_BYTES);
        bulk_load(ring + slot * C::SLOT_BYTES, kb, C::PAGE_BYTES, &full[slot]);
        bulk_load(ring + slot * C::SLOT_BYTES + C::PAGE_BYTES, vb, C::PAGE_BYTES, &full[slot]);
        last_slot_issued = i;
      }
      // every issued copy is waited on by a consumer; if consumers gave up,
      // wait here (bounded) for the last copies to land
      if (*abort_flag) {
        for (int i = (last_slot_issued - NSLOT + 1 > 0 ? last_slot_issued - NSLOT + 1 : 0);
             i <= last_slot_issued; ++i) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(smem_u32(&full[i % NSLOT]), (i / NSLOT) & 1) &&
                 globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    const int sub = lane % C::LPK;   // 8-element slice of hd
    const int kk = lane / C::LPK;    // key within a step
    const int my_st = sub >> 1;      // step whose score this lane ends up holding
    float2 qf[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(p.q + (static_cast<size_t>(t) * p.Hq + hk * G + g) * HD + sub * 8);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = bf2(w[e]);
        qf[g][e] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
      }
    }
    float m[G], l[G];
    float2 acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[g][e] = make_float2(0.f, 0.f);
    }
    for (int i = warp; i < np; i += NW) {
      const int slot = i % NSLOT;
      if (!mbar_wait(&full[slot], (i / NSLOT) & 1, abort_flag, p.err, kErrWaitSoftmax)) break;
      const uint8_t *ks = ring + slot * C::SLOT_BYTES;
      const uint8_t *vs = ks + C::PAGE_BYTES;
      const int key_base = (pb + i) * 16;
      // partial dot products of this lane's 8 dims with each step's key
      float part[G][C::STEPS];
#pragma unroll
      for (int st = 0; st < C::STEPS; ++st) {
        const uint4 kr = lds128(ks + (st * C::KPS + kk) * HD * 2 + sub * 16);
        const float2 k0 = bf2(kr.x), k1 = bf2(kr.y), k2 = bf2(kr.z), k3 = bf2(kr.w);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float2 a = __fmul2_rn(qf[g][0], k0);
          a = __ffma2_rn(qf[g][1], k1, a);
          a = __ffma2_rn(qf[g][2], k2, a);
          a = __ffma2_rn(qf[g][3], k3, a);
          part[g][st] = a.x + a.y;
        }
      }
      // transposed butterfly: each lane ends with the full score of step my_st
      float s[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float v[C::STEPS];
#pragma unroll
        for (int st = 0; st < C::STEPS; ++st) v[st] = part[g][st];
        int n = C::STEPS;
#pragma unroll
        for (int o = C::LPK / 2; o >= 2; o >>= 1) {
          const bool upper = (lane & o) != 0;
          const int half = n / 2;
#pragma unroll
          for (int i2 = 0; i2 < C::STEPS / 2; ++i2) {
            if (i2 < half) {
              const float send = upper ? v[i2] : v[i2 + half];
              const float keep = upper ? v[i2 + half] : v[i2];
              v[i2] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
          }
          n = half;
        }
        s[g] = v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
      }
      const int my_key = key_base + my_st * C::KPS + kk;
      const bool my_valid = my_key < kv;
      float pv[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mx = my_valid ? s[g] : -INFINITY;
#pragma unroll
        for (int o = 16; o >= 2; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m[g], mx);
        const float alpha = (m[g] == -INFINITY) ? 0.f : exp2f(m[g] - m_new);
        m[g] = m_new;
        pv[g] = my_valid ? exp2f(s[g] - m_new) : 0.f;
        l[g] = l[g] * alpha + ((sub & 1) ? 0.f : pv[g]);
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][e] = __fmul2_rn(acc[g][e], a2);
      }
      // o += p v over this lane's keys (step st, key st*KPS + kk)
#pragma unroll
      for (int st = 0; st < C::STEPS; ++st) {
        const int src = kk * C::LPK + 2 * st;
        const bool valid = key_base + st * C::KPS + kk < kv;
        uint4 vr = lds128(vs + (st * C::KPS + kk) * HD * 2 + sub * 16);
        if (!valid) vr = make_uint4(0, 0, 0, 0);
        const float2 v0 = bf2(vr.x), v1 = bf2(vr.y), v2 = bf2(vr.z), v3 = bf2(vr.w);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pr = __shfl_sync(0xffffffffu, pv[g], src);
          const float2 p2 = make_float2(pr, pr);
          acc[g][0] = __ffma2_rn(p2, v0, acc[g][0]);
          acc[g][1] = __ffma2_rn(p2, v1, acc[g][1]);
          acc[g][2] = __ffma2_rn(p2, v2, acc[g][2]);
          acc[g][3] = __ffma2_rn(p2, v3, acc[g][3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    // fold the KPS key lanes that share an hd slice, and the l partials
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int o = C::LPK; o < 32; o <<= 1)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[g][e].x += __shfl_xor_sync(0xffffffffu, acc[g][e].x, o);
          acc[g][e].y += __shfl_xor_sync(0xffffffffu, acc[g][e].y, o);
        }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) l[g] += __shfl_xor_sync(0xffffffffu, l[g], o);
    }
    // stash this warp's (m, l, o) for the CTA merge; the ring is free once
    // every consumer is past its last page (barrier below)
    named_bar_sync(bar_id + 1, NW * 32);
    float *stash = reinterpret_cast<float *>(ring) + warp * G * (HD + 2);
    if (kk == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          stash[g * (HD + 2) + sub * 8 + 2 * e] = acc[g][e].x;
          stash[g * (HD + 2) + sub * 8 + 2 * e + 1] = acc[g][e].y;
        }
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        stash[g * (HD + 2) + HD] = m[g];
        stash[g * (HD + 2) + HD + 1] = l[g];
      }
    }
    named_bar_sync(bar_id + 1, NW * 32);
    const float *all = reinterpret_cast<const float *>(ring);
    for (int idx = tid; idx < G * HD; idx += NW * 32) {
      const int g = idx / HD, d = idx % HD;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, all[(w * G + g) * (HD + 2) + HD]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float* base = all + (w * G + g) * (HD + 2);
        const float wt = base[HD] == -INFINITY ? 0.f : exp2f(base[HD] - M);
        L += wt * base[HD + 1];
        O += wt * base[d];
      }
      if (n_splits == 1) {
        p.o[(static_cast<size_t>(t) * p.Hq + hk * G + g) * HD + d] = __float2bfloat16_rn(O / L);
      } else {
        float *dst = p.part + (static_cast<size_t>(item) * G + g) * part_stride<HD>();
        dst[d] = O;
        if (d == 0) {
          dst[HD] = M;
          dst[HD + 1] = L;
        }
      }
    }
  }
}

// ============================================================ merge pass
// One warp per (request, q head) with several splits: o = sum_s w_s o_s /
// sum_s w_s l_s with w_s = 2^(m_s - max m).
template <int HD>
__global__ void __launch_bounds__(128) merge_kernel(const float *part, const int32_t *list, int n, __nv_bfloat16 *o,
                                                    const int32_t *qo_indptr, int Hq, int G) {
  pdl_wait();
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (w >= n * G) return;
  const int lane = threadIdx.x & 31;
  const int idx = w / G, g = w % G;
  const int req = list[idx * 4 + 0], hk = list[idx * 4 + 1], first = list[idx * 4 + 2], ns = list[idx * 4 + 3];
  float mmax = -INFINITY;
  for (int s = 0; s < ns; ++s) mmax = fmaxf(mmax, part[(static_cast<size_t>(first + s) * G + g) * part_stride<HD>() + HD]);
  constexpr int PER = HD / 32;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float *src = part + (static_cast<size_t>(first + s) * G + g) * part_stride<HD>();
    const float ms = src[HD];
    const float wgt = (ms == -INFINITY) ? 0.f : exp2f(ms - mmax);
    L += wgt * src[HD + 1];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += wgt * src[lane * PER + e];
  }
  const float inv = 1.f / L;
  const int t = qo_indptr[req];
  __nv_bfloat16 *dst = o + (static_cast<size_t>(t) * Hq + hk * G + g) * HD + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; ++e) dst[e] = __float2bfloat16_rn(acc[e] * inv);
}

// ============================================================ one grid
// The ragged attention of a step is ONE launch: blocks [0, n_tiles) run a
// prefill-chunk tile (tensor cores), the rest run a decode item (HBM stream),
// so the two kinds share the GPU instead of running back to back.  Tiles come
// first, heaviest first; decode items fill SMs as they free up.  A decode CTA
// runs two items side by side, each with 4 consumer warps, a producer warp and
// a ring in its half of the tile's shared memory.
template <int HD>
struct FusedCfg {
  static constexpr int THREADS = ChunkCfg<HD>::THREADS;          // 10 warps
  static constexpr int DEC_NW = 4;                                // consumers per decode item
  static constexpr int SMEM = ChunkCfg<HD>::SMEM;
  // two decode items per CTA, each with half of the shared memory
  static constexpr int HALF = (SMEM / 2) & ~1023;
  // Page i lives in slot i % NSLOT and is consumed by warp i % DEC_NW; with
  // NSLOT a multiple of DEC_NW every slot has a single consumer warp, which
  // takes its pages in order, so a parity wait on a slot can never match a
  // phase two copies ahead.
  static constexpr int FIT = (HALF - 256) / DecCfg<HD>::SLOT_BYTES;
  static constexpr int NSLOT = ((FIT < 16 ? FIT : 16) / DEC_NW) * DEC_NW;
  static_assert(2 * (DEC_NW + 1) * 32 == THREADS, "two decode items fill the CTA");
  static_assert(NSLOT >= DEC_NW && NSLOT % DEC_NW == 0, "one consumer warp per ring slot");
  // ring, full/empty barriers and the abort word of one item fit its half
  static_assert(NSLOT * DecCfg<HD>::SLOT_BYTES + 16 * NSLOT + 4 <= HALF, "decode item exceeds its half");
  // the end-of-item merge stash (8 q-heads at most) reuses the ring
  static_assert(DEC_NW * 8 * (HD + 2) * 4 <= NSLOT * DecCfg<HD>::SLOT_BYTES, "merge stash exceeds the ring");
};

template <int HD, int G>
__global__ void __launch_bounds__(FusedCfg<HD>::THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                     const ChunkParams cp, const DecodeParams dp, int n_tiles) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    // the layouts above need a 1024-aligned base and reserve no slack
    pdl_wait();
    if (threadIdx.x == 0) atomicExch(cp.err, kErrBounds);
    return;
  }
  if (static_cast<int>(blockIdx.x) < n_tiles) {
    chunk_tile<HD>(tmQ, tmKV, cp, blockIdx.x, smem_raw);   // waits after its set-up
  } else {
    pdl_wait();
    // warps 0-4 take item 2k, warps 5-9 item 2k + 1 (if it exists)
    using F = FusedCfg<HD>;
    const int half = threadIdx.x >= (F::DEC_NW + 1) * 32;
    const int item = 2 * (blockIdx.x - n_tiles) + half;
    if (item < dp.n_items)
      decode_item<HD, G, F::DEC_NW, F::NSLOT>(dp, item, align1024(smem_raw) + half * F::HALF,
                                              half * (F::DEC_NW + 1), 1 + 2 * half);
  }
}

template <int HD, int G>
cudaError_t launch_attention(const CUtensorMap &tq, const CUtensorMap &tkv, const ChunkParams &cp,
                             const DecodeParams &dp, int n_tiles, int n_items, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attention_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    FusedCfg<HD>::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  return launch_pdl(attention_kernel<HD, G>, dim3(n_tiles + (n_items + 1) / 2), dim3(FusedCfg<HD>::THREADS),
                    FusedCfg<HD>::SMEM, st, 1, tq, tkv, cp, dp, n_tiles);
}

template <int HD>
cudaError_t launch_attention_g(const CUtensorMap &tq, const CUtensorMap &tkv, const ChunkParams &cp,
                               const DecodeParams &dp, int n_tiles, int n_items, int G, cudaStream_t st) {
  switch (G) {
    case 1: return launch_attention<HD, 1>(tq, tkv, cp, dp, n_tiles, n_items, st);
    case 2: return launch_attention<HD, 2>(tq, tkv, cp, dp, n_tiles, n_items, st);
    case 3: return launch_attention<HD, 3>(tq, tkv, cp, dp, n_tiles, n_items, st);
    case 4: return launch_attention<HD, 4>(tq, tkv, cp, dp, n_tiles, n_items, st);
    case 5: return launch_attention<HD, 5>(tq, tkv, cp, dp, n_tiles, n_items, st);
    case 6: return launch_attention<HD, 6>(tq, tkv, cp, dp, n_tiles, n_items, st);
    case 7: return launch_attention<HD, 7>(tq, tkv, cp, dp, n_tiles, n_items, st);
    case 8: return launch_attention<HD, 8>(tq, tkv, cp, dp, n_tiles, n_items, st);
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
  DecodeParams dp;
  dp.q = static_cast<const __nv_bfloat16 *>(a.q);
  dp.pool = static_cast<const __nv_bfloat16 *>(a.pool);
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
  const int G = a.Hq / a.Hkv;
  return a.hd == 128 ? launch_attention_g<128>(*a.tm_q, *a.tm_kv, cp, dp, a.n_tiles, a.n_items, G, st)
                     : launch_attention_g<64>(*a.tm_q, *a.tm_kv, cp, dp, a.n_tiles, a.n_items, G, st);
}

cudaError_t attn_merge_run(const MergeArgs &m, cudaStream_t st) {
  if (m.n_merge <= 0) return cudaSuccess;
  const int G = m.Hq / m.Hkv;
  const int warps = m.n_merge * G;
  const int blocks = (warps + 3) / 4;
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(m.o);
  if (m.hd == 128)
    return launch_pdl(merge_kernel<128>, dim3(blocks), dim3(128), 0, st, 1, m.part, m.merge_list, m.n_merge, o,
                      m.qo_indptr, m.Hq, G);
  return launch_pdl(merge_kernel<64>, dim3(blocks), dim3(128), 0, st, 1, m.part, m.merge_list, m.n_merge, o,
                    m.qo_indptr, m.Hq, G);
}

}  // namespace mb
