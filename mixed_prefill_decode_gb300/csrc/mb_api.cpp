// C-ABI of the mixed prefill+decode layer step: argument and descriptor
// validation, work-list construction, descriptor upload and the launch
// sequence.  See include/mb.h for the contract of every entry point.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <queue>
#include <string>
#include <vector>

#include "mb.h"
#include "mb_internal.h"
#include "mb_kernels.h"


namespace mb {

static thread_local std::string g_last_error;

mb_status fail(mb_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

static mb_status cuda_fail(cudaError_t e, const char *where) {
  return fail(e == cudaErrorMemoryAllocation ? MB_ENOMEM : MB_ECUDA, "%s: %s (%s)", where, cudaGetErrorName(e),
              cudaGetErrorString(e));
}

// ------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

cudaError_t encode_tmap_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                           uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_tmap_5d(CUtensorMap *map, const void *base, const uint64_t dims[5], const uint64_t strides_bytes[4],
                           const uint32_t box[5]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], estr[5] = {1, 1, 1, 1, 1};
  for (int i = 0; i < 5; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < 4; ++i) st[i] = strides_bytes[i];
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), d, st, b, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// ------------------------------------------------------ per-device context
struct DeviceCtx {
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  void *gemm_ws = nullptr;  // shared GEMM partial workspace
  int *err = nullptr;       // error word for standalone calls
};
static std::mutex g_dev_mu;
static DeviceCtx g_dev[64];

static mb_status device_ctx(DeviceCtx **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(MB_EUNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceCtx &c = g_dev[dev];
  if (c.sms == 0) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
      return fail(MB_EUNSUPPORTED, "device %d is sm_%d%d; these kernels are built for sm_103a only", dev,
                  prop.major, prop.minor);
    c.cc_major = prop.major;
    c.cc_minor = prop.minor;
    c.sms = prop.multiProcessorCount;
  }
  if (!c.gemm_ws) {
    e = cudaMalloc(&c.gemm_ws, gemm_workspace_bytes());
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(gemm workspace)");
    e = cudaMemset(c.gemm_ws, 0, gemm_workspace_bytes());
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(gemm workspace)");
    e = cudaMalloc(&c.err, 16);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
    e = cudaMemset(c.err, 0, 16);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
  }
  *out = &c;
  return MB_OK;
}

// The current device's context if an entry point has set it up already
// (nullptr otherwise); allocates nothing.
static DeviceCtx *device_ctx_if_ready() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  return g_dev[dev].gemm_ws ? &g_dev[dev] : nullptr;
}

// SM count of the current device; every entry point has set up its context
// (device_ctx) before launching, so the fallback is never taken there.
int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  return g_dev[dev].sms > 0 ? g_dev[dev].sms : 152;
}

}  // namespace mb

using mb::fail;

// ===================================================================== layer
namespace {

constexpr int kNumTimed = 9;
constexpr int kRing = 4;

struct EventSet {
  cudaEvent_t ev[kNumTimed + 1];
};

struct StagingSlot {
  int32_t *host = nullptr;
  size_t cap = 0;  // int32 elements
  cudaEvent_t done = nullptr;
  bool used = false;
};

int32_t pages_for(int64_t n) { return static_cast<int32_t>((n + MB_PAGE_TOKENS - 1) / MB_PAGE_TOKENS); }

}  // namespace

struct mb_kv {
  mb_layer *layer = nullptr;
  void *base = nullptr;
  bool owned = false;
  int32_t num_pages = 0;
  CUtensorMap tmap;
  std::vector<uint32_t> stamp;  // page -> last step that referenced it (duplicate check)
  uint32_t stamp_gen = 0;
};

struct mb_layer {
  mb_layer_desc d;
  mb_layer_weights w;
  int device = 0;
  int qkv_dim = 0;
  // workspaces (bf16)
  void *xn = nullptr, *qkv = nullptr, *q = nullptr, *o = nullptr, *h = nullptr, *hn = nullptr, *a = nullptr;
  size_t bytes_x = 0, bytes_qkv = 0, bytes_q = 0, bytes_a = 0;
  int *err = nullptr;
  mb::GemmWorkspace gws{};
  CUtensorMap tm_wqkv, tm_wo, tm_wgu, tm_wd;
  // descriptor upload
  StagingSlot ring[kRing];
  int ring_next = 0;
  int32_t *dblob = nullptr;
  size_t dblob_cap = 0;
  // Attention scratch: counters first (decode split groups, then split chunk
  // tiles; every one is zero between launches, since the kernel that raises
  // a counter lowers it), then the decode and chunk partials.  The counter
  // region keeps its place and size until it must grow, so no step's
  // counters ever land on an earlier step's partials.
  float *part = nullptr;
  size_t part_cap = 0;  // floats, counters included
  size_t ctr_cap = 0;   // 4-byte words of counters at the start
  // last step
  int32_t last_T = 0;
  int32_t last_launches = 0;
  int64_t last_upload = 0;
  // timing
  bool timing = false;
  int32_t dec_sms = 0;   // decode worker CTAs at most (mb_layer_set_decode_sms; 0: one per SM)
  std::vector<EventSet> ev_pool;
  size_t ev_used = 0;
  double ms[kNumTimed] = {0};
  int64_t steps_timed = 0;
  cudaStream_t last_stream = nullptr;
  // host scratch
  std::vector<int32_t> hbuf;
};


// A stack of layers that share one batch descriptor per step.
// Everything a captured step's launches take from the batch: the sizes, the
// descriptor's section offsets (kernel arguments point into the blob) and the
// buffers.  Batches with equal keys replay one graph; the graph reads the
// descriptor's contents from the blob at run time.
struct GraphKey {
  int64_t T;
  int n_reqs, n_tiles, n_items, n_merge, n_chunk_slots, gemm_ctas, dec_workers;
  size_t ctr_cap;
  const void *gws;
  size_t offs[8];
  const void *db, *part, *x_in, *x_out, *kv0;
  int dec_sms;
  bool operator==(const GraphKey &o) const {
    return T == o.T && n_reqs == o.n_reqs && n_tiles == o.n_tiles && n_items == o.n_items &&
           n_merge == o.n_merge && n_chunk_slots == o.n_chunk_slots && gemm_ctas == o.gemm_ctas &&
           dec_workers == o.dec_workers &&
           ctr_cap == o.ctr_cap && gws == o.gws &&
           std::equal(offs, offs + 8, o.offs) && db == o.db && part == o.part &&
           x_in == o.x_in && x_out == o.x_out && kv0 == o.kv0 && dec_sms == o.dec_sms;
  }
};

struct mb_stack {
  std::vector<mb_layer *> layers;
  void *act[2] = {nullptr, nullptr};  // ping-pong activations between layers
  std::vector<uint32_t> stamp;
  uint32_t stamp_gen = 0;
  bool use_graphs = true;
  struct Entry {
    GraphKey key;
    cudaGraphExec_t exec;
    int launches;
  };
  std::vector<Entry> graphs;
  std::vector<mb_kv *> graph_kvs;
  cudaStream_t cap_stream = nullptr;
  int32_t last_launches = 0;
  int32_t last_T = 0;
  void drop_graphs() {
    for (auto &g : graphs) cudaGraphExecDestroy(g.exec);
    graphs.clear();
    graph_kvs.clear();
  }
};

namespace {

mb_status alloc_dev(void **p, size_t bytes, const char *what) {
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) return mb::fail(e == cudaErrorMemoryAllocation ? MB_ENOMEM : MB_ECUDA, "cudaMalloc(%s, %zu bytes): %s", what, bytes, cudaGetErrorString(e));
  return MB_OK;
}

void free_layer_mem(mb_layer *L) {
  void *ptrs[] = {L->xn, L->qkv, L->q, L->o, L->h, L->hn, L->a, L->err, L->dblob, L->part};
  for (void *p : ptrs)
    if (p) cudaFree(p);
  for (auto &s : L->ring) {
    if (s.host) cudaFreeHost(s.host);
    if (s.done) cudaEventDestroy(s.done);
  }
  for (auto &es : L->ev_pool)
    for (auto &e : es.ev) cudaEventDestroy(e);
}

mb_status flush_timing(mb_layer *L) {
  if (L->ev_used == 0) return MB_OK;
  for (size_t i = 0; i < L->ev_used; ++i) {
    EventSet &es = L->ev_pool[i];
    cudaError_t e = cudaEventSynchronize(es.ev[kNumTimed]);
    if (e != cudaSuccess) return mb::fail(MB_ECUDA, "cudaEventSynchronize: %s", cudaGetErrorString(e));
    for (int k = 0; k < kNumTimed; ++k) {
      float t = 0.f;
      e = cudaEventElapsedTime(&t, es.ev[k], es.ev[k + 1]);
      if (e != cudaSuccess) return mb::fail(MB_ECUDA, "cudaEventElapsedTime: %s", cudaGetErrorString(e));
      L->ms[k] += t;
    }
    L->steps_timed += 1;
  }
  L->ev_used = 0;
  return MB_OK;
}


// Descriptor rules of include/mb.h; `stamp` (num_pages entries) marks pages
// already seen with `gen` to catch a page used twice.
mb_status validate_batch(const mb_batch *b, int32_t num_pages, int32_t max_tokens, uint32_t *stamp, uint32_t gen,
                         int64_t *T_out) {
  const int n = b->num_reqs;
  if (n < 0) return mb::fail(MB_EINVAL, "batch: num_reqs < 0");
  if (n == 0) {
    *T_out = 0;
    return MB_OK;
  }
  if (!b->qo_indptr || !b->kv_len || !b->bt_indptr || !b->bt) return mb::fail(MB_EINVAL, "batch: null descriptor array");
  if (b->qo_indptr[0] != 0) return mb::fail(MB_EINVAL, "batch: qo_indptr[0] must be 0");
  int64_t T = 0;
  for (int r = 0; r < n; ++r) {
    const int64_t qo = static_cast<int64_t>(b->qo_indptr[r + 1]) - b->qo_indptr[r];
    const int64_t kvl = b->kv_len[r];
    if (qo < 1) return mb::fail(MB_EINVAL, "batch: request %d has qo_len %lld < 1", r, (long long)qo);
    if (kvl < qo)
      return mb::fail(MB_EINVAL, "batch: request %d has kv_len %lld < qo_len %lld", r, (long long)kvl, (long long)qo);
    if (kvl > (1 << 24)) return mb::fail(MB_EUNSUPPORTED, "batch: request %d kv_len > 2^24", r);
    const int64_t tl = static_cast<int64_t>(b->bt_indptr[r + 1]) - b->bt_indptr[r];
    if (b->bt_indptr[r] < 0 || tl < pages_for(kvl))
      return mb::fail(MB_EINVAL, "batch: request %d block table has %lld pages, needs %d", r, (long long)tl,
                      pages_for(kvl));
    for (int64_t i = 0; i < pages_for(kvl); ++i) {
      const int32_t pg = b->bt[b->bt_indptr[r] + i];
      if (pg < 0 || pg >= num_pages)
        return mb::fail(MB_EINVAL, "batch: request %d page id %d outside [0, %d)", r, pg, num_pages);
      if (stamp[pg] == gen) return mb::fail(MB_EINVAL, "batch: page %d referenced twice in one batch", pg);
      stamp[pg] = gen;
    }
    T += qo;
  }
  if (T > max_tokens) return mb::fail(MB_EINVAL, "batch: T = %lld exceeds max_tokens %d", (long long)T, max_tokens);
  *T_out = T;
  return MB_OK;
}


// A chunk tile: 256 query rows (qt = 1 or 2 query tiles of 128 rows with
// rows in them) of one q-head, over nkb key blocks of 128.
struct ChunkTile {
  int32_t r, i0, h, nkb, qt;
};
// A unit of the attention launch's chunk work: key blocks [j0, j1) of a tile.
struct ChunkUnit {
  int32_t r, i0, h, j0, j1, piece, n_pieces, slot;
  int64_t cost;
};

constexpr int32_t kMinPieceBlocks = 8;   // a piece covers at least 1,024 keys
constexpr int64_t kUnitRamp = 2;         // a CTA's set-up, first loads and epilogue, in key blocks
constexpr int64_t kPieceExtra = 2;       // a piece's partial round trip and share of the merge
constexpr int64_t kItemRamp = 3;         // a decode item's Q load, first blocks and output or partial
constexpr double kDecodeSatFrac = 0.85;  // share of the SMs whose decode workers saturate HBM

// Makespan of list scheduling: each unit, in order, to the processor that
// frees first.  That is how CTAs launched in that order spread over the SMs
// (one chunk CTA per SM).
int64_t list_makespan(const std::vector<int64_t> &costs, int m) {
  std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> q;
  for (int i = 0; i < m; ++i) q.push(0);
  int64_t span = 0;
  for (int64_t c : costs) {
    const int64_t t = q.top() + c;
    q.pop();
    q.push(t);
    span = std::max(span, t);
  }
  return span;
}

// Chunk tiles cover the GPU in waves of one CTA per SM; when their count is
// just past a multiple of the SM count, the last wave runs a few tiles on an
// otherwise idle GPU (320 tiles of a 2,048-row chunk over 40 heads on 152
// SMs: 2.1 waves).  A tile can be split along its keys into pieces whose
// partial softmax states are merged by log-sum-exp (every piece but the last
// covers keys that all of the tile's rows see; the last holds the diagonal).
// Candidate plans: no split; the tiles of the last partial wave split so that
// their pieces cover every SM; every tile in 2, 3 or 4 pieces.  The plan with
// the shortest list-scheduling makespan (in key blocks, with a fixed cost per
// CTA and per piece) wins; ties keep the plan with fewer units.  Units come
// out heaviest first; the pieces of a split tile get consecutive partial
// slots.  Returns the number of slots.
int plan_chunk_units(std::vector<ChunkTile> tiles, int sms, std::vector<ChunkUnit> *out) {
  out->clear();
  if (tiles.empty()) return 0;
  std::stable_sort(tiles.begin(), tiles.end(),
                   [](const ChunkTile &x, const ChunkTile &y) { return x.nkb * x.qt > y.nkb * y.qt; });
  const int n = static_cast<int>(tiles.size());
  const int m = std::max(1, sms);
  auto max_pieces = [](const ChunkTile &t) { return std::max(1, std::min(32, t.nkb / kMinPieceBlocks)); };
  auto piece_lo = [](const ChunkTile &t, int p, int ns) {
    return static_cast<int32_t>(static_cast<int64_t>(p) * t.nkb / ns);
  };
  auto build = [&](const std::vector<int> &ns, std::vector<ChunkUnit> *units) {
    units->clear();
    int slot = 0;
    for (int i = 0; i < n; ++i) {
      const ChunkTile &t = tiles[i];
      if (ns[i] == 1) {
        units->push_back({t.r, t.i0, t.h, 0, t.nkb, 0, 1, 0, static_cast<int64_t>(t.nkb) * t.qt + kUnitRamp});
        continue;
      }
      for (int p = 0; p < ns[i]; ++p) {
        const int32_t lo = piece_lo(t, p, ns[i]), hi = piece_lo(t, p + 1, ns[i]);
        units->push_back({t.r, t.i0, t.h, lo, hi, p, ns[i], slot + p,
                          static_cast<int64_t>(hi - lo) * t.qt + kUnitRamp + kPieceExtra});
      }
      slot += ns[i];
    }
    std::stable_sort(units->begin(), units->end(),
                     [](const ChunkUnit &x, const ChunkUnit &y) { return x.cost > y.cost; });
    return slot;
  };
  auto span_of = [&](const std::vector<int> &ns, size_t *count) {
    std::vector<ChunkUnit> u;
    build(ns, &u);
    std::vector<int64_t> costs(u.size());
    for (size_t i = 0; i < u.size(); ++i) costs[i] = u[i].cost;
    *count = u.size();
    return list_makespan(costs, m);
  };
  std::vector<std::vector<int>> plans;
  plans.push_back(std::vector<int>(n, 1));
  const int first_tail = (n / m) * m;
  if (first_tail < n) {
    std::vector<int> ns(n, 1);
    const int s = (m + (n - first_tail) - 1) / (n - first_tail);
    for (int i = first_tail; i < n; ++i) ns[i] = std::min(s, max_pieces(tiles[i]));
    plans.push_back(ns);
  }
  for (int k = 2; k <= 4; ++k) {
    std::vector<int> ns(n);
    for (int i = 0; i < n; ++i) ns[i] = std::min(k, max_pieces(tiles[i]));
    plans.push_back(ns);
  }
  size_t best = 0, best_count = 0;
  int64_t best_span = span_of(plans[0], &best_count);
  for (size_t k = 1; k < plans.size(); ++k) {
    size_t count = 0;
    const int64_t sp = span_of(plans[k], &count);
    if (sp < best_span || (sp == best_span && count < best_count)) {
      best = k;
      best_span = sp;
      best_count = count;
    }
  }
  return build(plans[best], out);
}

// Device-side plan of one step: where the descriptor, per-token tables and
// work lists live in the uploaded blob, and their sizes.
struct StepPlan {
  int64_t T = 0;
  size_t o_qo = 0, o_kv = 0, o_bti = 0, o_bt = 0, o_treq = 0, o_tpos = 0, o_tiles = 0, o_items = 0;
  int n_tiles = 0, n_items = 0, n_merge = 0;   // n_tiles: chunk units; n_merge: decode split groups
  int n_chunk_slots = 0;                       // partial slots of split chunk tiles
  int dec_workers = 0;                         // decode worker CTAs the plan is for
  const int32_t *db = nullptr;
  int64_t upload_bytes = 0;
};

// Host part of a step: per-token tables, attention work lists (chunk tiles,
// decode splits, merge list), one upload through `L`'s pinned ring into its
// device blob.  The batch has been validated.
mb_status prepare_step(mb_layer *L, const mb_batch *b, int64_t T, cudaStream_t s, StepPlan *plan) {
  mb::DeviceCtx *ctx = nullptr;
  mb_status st = mb::device_ctx(&ctx);
  if (st != MB_OK) return st;
  const mb_layer_desc &d = L->d;
  const int n = b->num_reqs;
  const int Hq = d.n_q_heads, Hkv = d.n_kv_heads, hd = d.head_dim, G = Hq / Hkv;
  const int64_t nb = b->bt_indptr[n];
  std::vector<int32_t> &hb = L->hbuf;
  hb.clear();
  auto sec = [&](size_t count) {
    size_t off = hb.size();
    hb.resize(off + ((count + 3) & ~size_t(3)), 0);
    return off;
  };
  StepPlan &P = *plan;
  P.T = T;
  // Section order: everything whose size depends only on (n, T, tiles,
  // items) first, the block tables (whose length changes with every prefix)
  // last, so that batches of one geometry share every offset and a captured
  // graph's kernel arguments stay valid for all of them.
  P.o_qo = sec(n + 1);
  P.o_kv = sec(n);
  P.o_bti = sec(n + 1);
  P.o_treq = sec(T);
  P.o_tpos = sec(T);
  std::copy(b->qo_indptr, b->qo_indptr + n + 1, hb.begin() + P.o_qo);
  std::copy(b->kv_len, b->kv_len + n, hb.begin() + P.o_kv);
  std::copy(b->bt_indptr, b->bt_indptr + n + 1, hb.begin() + P.o_bti);
  for (int r = 0; r < n; ++r) {
    const int32_t t0 = b->qo_indptr[r], t1 = b->qo_indptr[r + 1];
    const int32_t c = b->kv_len[r] - (t1 - t0);
    for (int32_t t = t0; t1 > t; ++t) {
      hb[P.o_treq + t] = r;
      hb[P.o_tpos + t] = c + (t - t0);
    }
  }
  // chunk tiles: 256 query rows (two 128-row tiles) of one q-head each
  std::vector<ChunkTile> tiles;
  for (int r = 0; r < n; ++r) {
    const int32_t qo = b->qo_indptr[r + 1] - b->qo_indptr[r];
    if (qo > 1) {
      const int32_t c = b->kv_len[r] - qo;
      for (int32_t i0 = 0; i0 < qo; i0 += 256) {
        const int32_t rows = std::min(256, qo - i0);
        const int32_t nkb = (c + i0 + rows - 1 + 128) / 128;
        for (int32_t hh = 0; hh < Hq; ++hh) tiles.push_back({r, i0, hh, nkb, rows > 128 ? 2 : 1});
      }
    }
  }
  std::vector<ChunkUnit> units;
  P.n_chunk_slots = plan_chunk_units(tiles, ctx->sms, &units);
  P.o_tiles = sec(units.size() * 8);
  for (size_t i = 0; i < units.size(); ++i) {
    const ChunkUnit &u = units[i];
    const int32_t rec[8] = {u.r, u.i0, u.h, u.j0, u.j1, u.piece, u.n_pieces, u.slot};
    std::copy(rec, rec + 8, hb.begin() + P.o_tiles + 8 * i);
  }
  // Decode splits.  A request's 128-key blocks (8 pages) are divided evenly
  // among its splits, so only its last block can be partial; the splits of
  // one (request, KV head) hold consecutive partial slots and the last one to
  // finish merges them (group = its counter).  Workers take items from a
  // counter in list order, so the list runs heaviest first (list
  // scheduling); the split size is the candidate (about 2 to 8 items per
  // decode worker) whose list-scheduling makespan, at kItemRamp blocks per
  // item of overhead, is shortest (ties: fewer items).  Measured on GB300
  // (attention launch): 16 decodes at 8,192 keys 0.132 ms with one block of
  // overhead per item (7 splits each), 0.118 ms with three (2 splits), 0.125
  // ms with the earlier fixed 4 items per SM in request order; 64 decodes at
  // 1,126 keys beside a 512-row chunk 0.091, 0.079 and 0.080 ms.
  std::vector<std::pair<int32_t, int32_t>> decs;   // (request, 128-key blocks)
  int64_t dec_blocks = 0;
  for (int r = 0; r < n; ++r) {
    if (b->qo_indptr[r + 1] - b->qo_indptr[r] != 1) continue;
    const int32_t nblk = (pages_for(b->kv_len[r]) + 7) / 8;
    decs.push_back({r, nblk});
    dec_blocks += static_cast<int64_t>(nblk) * Hkv;
  }
  // The worker count is planned too (one per SM at most), whatever the
  // decode SM cap, so that a cap changes only which worker takes an item,
  // not what the items compute.  The stream saturates HBM before every SM
  // takes part (measured: 16 decodes at 8,192 keys, 4.68 TB/s on 128 workers
  // against 4.50 on 152), so a plan's time is modelled as its makespan in
  // blocks times W / min(W, kDecodeSatFrac * SMs) for W workers.
  auto splits_of = [](int32_t nblk, int64_t bps) {
    // at most 32 splits: the merge holds one split per lane
    return static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>({nblk, (nblk + bps / 2) / bps, 32})));
  };
  auto decode_span = [&](int64_t bps, int workers, size_t *count) {
    std::vector<int64_t> costs;
    for (const auto &d : decs) {
      const int32_t ns = splits_of(d.second, bps);
      for (int32_t sidx = 0; sidx < ns; ++sidx) {
        const int64_t nb_item = static_cast<int64_t>(d.second) * (sidx + 1) / ns - static_cast<int64_t>(d.second) * sidx / ns;
        for (int32_t hk = 0; hk < Hkv; ++hk) costs.push_back(nb_item + kItemRamp);
      }
    }
    std::stable_sort(costs.begin(), costs.end(), std::greater<int64_t>());
    *count = costs.size();
    return list_makespan(costs, workers);
  };
  int64_t bps = 1;
  P.dec_workers = std::max(1, ctx->sms);
  if (!decs.empty()) {
    const double sat = kDecodeSatFrac * ctx->sms;
    double best_t = -1.0;
    size_t best_count = 0;
    for (int w : {ctx->sms, ctx->sms * 7 / 8, ctx->sms * 3 / 4}) {
      if (w < 1) continue;
      for (int k : {1, 2, 3, 4, 6, 8}) {
        const int64_t cand = std::max<int64_t>(1, (dec_blocks + static_cast<int64_t>(w) * k - 1) /
                                                      (static_cast<int64_t>(w) * k));
        size_t count = 0;
        const double t = static_cast<double>(decode_span(cand, w, &count)) * w / std::min<double>(w, sat);
        if (best_t < 0 || t < best_t - 1e-9 || (std::fabs(t - best_t) <= 1e-9 && count < best_count)) {
          best_t = t;
          best_count = count;
          bps = cand;
          P.dec_workers = w;
        }
      }
    }
  }
  struct DecItem {
    int32_t f[8];
    int32_t blocks;
  };
  std::vector<DecItem> ditems;
  int32_t n_groups = 0, n_slots = 0;
  for (const auto &d : decs) {
    const int32_t r = d.first, nblk = d.second;
    const int32_t np = pages_for(b->kv_len[r]);
    const int32_t ns = splits_of(nblk, bps);
    for (int32_t hk = 0; hk < Hkv; ++hk) {
      const int32_t grp = ns > 1 ? n_groups++ : -1;
      const int32_t slot0 = ns > 1 ? n_slots : 0;
      if (ns > 1) n_slots += ns;
      for (int32_t sidx = 0; sidx < ns; ++sidx) {
        const int32_t b0 = static_cast<int32_t>(static_cast<int64_t>(nblk) * sidx / ns);
        const int32_t b1 = static_cast<int32_t>(static_cast<int64_t>(nblk) * (sidx + 1) / ns);
        const int32_t pb = 8 * b0;
        const int32_t pe = std::min(np, 8 * b1);
        ditems.push_back({{r, hk, pb, pe, sidx, ns, grp, slot0}, b1 - b0});
      }
    }
  }
  std::stable_sort(ditems.begin(), ditems.end(),
                   [](const DecItem &x, const DecItem &y) { return x.blocks > y.blocks; });
  std::vector<int32_t> items;
  items.reserve(ditems.size() * 8);
  for (const DecItem &it : ditems) items.insert(items.end(), it.f, it.f + 8);
  P.o_items = sec(items.size());
  std::copy(items.begin(), items.end(), hb.begin() + P.o_items);
  P.o_bt = sec(static_cast<size_t>(nb));
  std::copy(b->bt, b->bt + nb, hb.begin() + P.o_bt);
  P.n_tiles = static_cast<int>(units.size());
  P.n_items = static_cast<int>(items.size() / 8);
  P.n_merge = n_groups;

  // ---- upload through a pinned ring slot
  StagingSlot &slot = L->ring[L->ring_next];
  L->ring_next = (L->ring_next + 1) % kRing;
  cudaError_t e;
  if (slot.used) {
    e = cudaEventSynchronize(slot.done);
    if (e != cudaSuccess) return mb::fail(MB_ECUDA, "step: %s", cudaGetErrorString(e));
  }
  if (slot.cap < hb.size()) {
    if (slot.host) cudaFreeHost(slot.host);
    slot.host = nullptr;
    size_t cap = std::max<size_t>(hb.size() * 2, 4096);
    e = cudaHostAlloc(reinterpret_cast<void **>(&slot.host), cap * 4, cudaHostAllocDefault);
    if (e != cudaSuccess) {
      slot.cap = 0;
      return mb::fail(MB_ENOMEM, "step: cudaHostAlloc: %s", cudaGetErrorString(e));
    }
    slot.cap = cap;
  }
  if (L->dblob_cap < hb.size()) {
    cudaStreamSynchronize(s);
    if (L->dblob) cudaFree(L->dblob);
    L->dblob = nullptr;
    size_t cap = std::max<size_t>(hb.size() * 2, 4096);
    st = alloc_dev(reinterpret_cast<void **>(&L->dblob), cap * 4, "descriptor");
    if (st != MB_OK) {
      L->dblob_cap = 0;
      return st;
    }
    L->dblob_cap = cap;
  }
  // attention scratch: counters (decode split groups, then split chunk
  // tiles' slots), then decode split partials and chunk tile partials (rows
  // of hd + 4 floats: o, m, l, pad); counters must start at zero
  const size_t ctr_need = static_cast<size_t>(P.n_merge) + static_cast<size_t>(P.n_chunk_slots);
  const size_t part_need = static_cast<size_t>(P.n_items) * G * (hd + 4) +
                           static_cast<size_t>(P.n_chunk_slots) * 256 * (hd + 4);
  if (L->ctr_cap < ctr_need || L->part_cap < L->ctr_cap + part_need) {
    cudaStreamSynchronize(s);
    if (L->part) cudaFree(L->part);
    L->part = nullptr;
    const size_t ctr_cap = std::max<size_t>(std::max(L->ctr_cap, (ctr_need * 2 + 3) & ~size_t(3)), 64);
    const size_t cap = ctr_cap + std::max(part_need * 2, L->part_cap > L->ctr_cap ? L->part_cap - L->ctr_cap : 0);
    st = alloc_dev(reinterpret_cast<void **>(&L->part), cap * 4, "attention partials");
    if (st == MB_OK && cudaMemset(L->part, 0, cap * 4) != cudaSuccess) st = fail(MB_ECUDA, "cudaMemset(partials)");
    if (st != MB_OK) {
      L->part_cap = L->ctr_cap = 0;
      return st;
    }
    L->part_cap = cap;
    L->ctr_cap = ctr_cap;
  }
  std::memcpy(slot.host, hb.data(), hb.size() * 4);
  e = cudaMemcpyAsync(L->dblob, slot.host, hb.size() * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return mb::fail(MB_ECUDA, "step: descriptor upload: %s", cudaGetErrorString(e));
  e = cudaEventRecord(slot.done, s);
  if (e != cudaSuccess) return mb::fail(MB_ECUDA, "step: %s", cudaGetErrorString(e));
  slot.used = true;
  P.db = L->dblob;
  P.upload_bytes = static_cast<int64_t>(hb.size()) * 4;
  return MB_OK;
}

// The launches of one layer: weights and tensor maps of `L`, workspaces of
// `W` (the layer itself, or the first layer of a stack), KV pool `kv`.
mb_status launch_layer(mb_layer *L, mb_layer *W, mb_kv *kv, const StepPlan &P, const void *x_in, void *x_out,
                       cudaStream_t s, EventSet *es, int *launches) {
  const mb_layer_desc &d = L->d;
  const int Hq = d.n_q_heads, Hkv = d.n_kv_heads, hd = d.head_dim;
  const int Ti = static_cast<int>(P.T);
  const int hqd = Hq * hd;
  const int32_t *db = P.db;
  auto mark = [&](int k) {
    if (es) cudaEventRecord(es->ev[k], s);
  };
  auto chk = [&](cudaError_t err, const char *what) -> mb_status {
    if (err != cudaSuccess) return mb::fail(MB_ECUDA, "step: %s: %s", what, cudaGetErrorString(err));
    return MB_OK;
  };
  mb_status st;
  mark(0);
  if ((st = chk(mb::rmsnorm_run(x_in, L->w.g_attn, W->xn, Ti, d.d_model, d.rms_eps, s), "rmsnorm")) != MB_OK) return st;
  ++*launches;
  mark(1);
  if ((st = chk(mb::gemm_run(W->xn, L->w.w_qkv, &L->tm_wqkv, W->qkv, nullptr, Ti, L->qkv_dim, d.d_model,
                             mb::kEpiStore, W->gws, W->err, s), "gemm qkv")) != MB_OK)
    return st;
  *launches += mb::gemm_launches(Ti, L->qkv_dim, d.d_model, mb::kEpiStore, W->gws.max_ctas);
  mark(2);
  mb::RopeArgs ra;
  ra.qkv = W->qkv;
  ra.q_out = W->q;
  ra.pool = kv->base;
  ra.tok_req = db + P.o_treq;
  ra.tok_pos = db + P.o_tpos;
  ra.bt_indptr = db + P.o_bti;
  ra.bt = db + P.o_bt;
  ra.g_q = L->w.g_q;
  ra.g_k = L->w.g_k;
  ra.T = Ti;
  ra.Hq = Hq;
  ra.Hkv = Hkv;
  ra.hd = hd;
  ra.qk_norm = d.qk_norm;
  ra.num_pages = kv->num_pages;
  ra.eps = d.rms_eps;
  ra.theta = d.rope_theta;
  ra.err = W->err;
  if ((st = chk(mb::rope_append_run(ra, s), "rope/append")) != MB_OK) return st;
  ++*launches;
  mark(3);
  CUtensorMap tm_q, tm_qd;
  cudaError_t e = mb::encode_tmap_2d(&tm_q, W->q, hqd, Ti, hqd * 2ull, 64, 128);
  if (e == cudaSuccess) e = mb::encode_tmap_2d(&tm_qd, W->q, hd, static_cast<uint64_t>(Ti) * Hq, hd * 2ull, 64, 16);
  if (e != cudaSuccess) return mb::fail(MB_ECUDA, "step: Q tensor map");
  mb::AttnArgs aa;
  aa.q = W->q;
  aa.pool = kv->base;
  aa.o = W->o;
  aa.qo_indptr = db + P.o_qo;
  aa.kv_len = db + P.o_kv;
  aa.bt_indptr = db + P.o_bti;
  aa.bt = db + P.o_bt;
  aa.tiles = db + P.o_tiles;
  aa.items = db + P.o_items;
  aa.n_tiles = P.n_tiles;
  aa.n_items = P.n_items;
  aa.max_workers = L->dec_sms > 0 ? std::min(L->dec_sms, P.dec_workers) : P.dec_workers;
  aa.T = Ti;
  aa.Hq = Hq;
  aa.Hkv = Hkv;
  aa.hd = hd;
  aa.num_pages = kv->num_pages;
  aa.err = W->err;
  aa.tm_q = &tm_q;
  aa.tm_qd = &tm_qd;
  aa.tm_kv = &kv->tmap;
  aa.dec_ctr = W->err + 2;   // words 2-3 of the layer's error block
  aa.merge_ctr = reinterpret_cast<int *>(W->part);
  aa.chunk_ctr = aa.merge_ctr + P.n_merge;
  aa.part = W->part + W->ctr_cap;
  aa.chunk_part = aa.part + static_cast<size_t>(P.n_items) * (Hq / Hkv) * (hd + 4);
  if ((st = chk(mb::attention_run(aa, s), "attention")) != MB_OK) return st;
  *launches += (aa.n_tiles + aa.n_items) > 0;
  mark(4);
  // (split merging happens inside the attention launch)
  mark(5);
  if ((st = chk(mb::gemm_run(W->o, L->w.w_o, &L->tm_wo, W->h, x_in, Ti, d.d_model, hqd, mb::kEpiResidual, W->gws,
                             W->err, s), "gemm o")) != MB_OK)
    return st;
  *launches += mb::gemm_launches(Ti, d.d_model, hqd, mb::kEpiResidual, W->gws.max_ctas);
  mark(6);
  if ((st = chk(mb::rmsnorm_run(W->h, L->w.g_ffn, W->hn, Ti, d.d_model, d.rms_eps, s), "rmsnorm ffn")) != MB_OK)
    return st;
  ++*launches;
  mark(7);
  if ((st = chk(mb::gemm_run(W->hn, L->w.w_gate_up, &L->tm_wgu, W->a, nullptr, Ti, d.d_ff, d.d_model,
                             mb::kEpiSwiGLU, W->gws, W->err, s), "gemm gate/up")) != MB_OK)
    return st;
  *launches += mb::gemm_launches(Ti, d.d_ff, d.d_model, mb::kEpiSwiGLU, W->gws.max_ctas);
  mark(8);
  if ((st = chk(mb::gemm_run(W->a, L->w.w_down, &L->tm_wd, x_out, W->h, Ti, d.d_model, d.d_ff, mb::kEpiResidual,
                             W->gws, W->err, s), "gemm down")) != MB_OK)
    return st;
  *launches += mb::gemm_launches(Ti, d.d_model, d.d_ff, mb::kEpiResidual, W->gws.max_ctas);
  mark(9);
  return MB_OK;
}


}  // namespace

extern "C" {

mb_status mb_batch_validate(const mb_batch *b, int32_t num_pages, int32_t max_tokens) {
  if (!b || num_pages < 0) return mb::fail(MB_EINVAL, "mb_batch_validate: null batch or negative num_pages");
  std::vector<uint32_t> stamp(static_cast<size_t>(num_pages), 0u);
  int64_t T = 0;
  return validate_batch(b, num_pages, max_tokens, stamp.data(), 1u, &T);
}

const char *mb_last_error(void) { return mb::g_last_error.c_str(); }

int64_t mb_gemm_workspace_bytes(void) { return static_cast<int64_t>(mb::gemm_workspace_bytes()); }

mb_status mb_layer_create(const mb_layer_desc *desc, const mb_layer_weights *w, mb_layer **out) {
  if (!desc || !w || !out) return fail(MB_EINVAL, "mb_layer_create: null argument");
  const mb_layer_desc &d = *desc;
  if (d.d_model <= 0 || d.n_q_heads <= 0 || d.n_kv_heads <= 0 || d.head_dim <= 0 || d.d_ff <= 0 ||
      d.max_tokens <= 0 || !(d.rms_eps >= 0.f) || !(d.rope_theta > 0.f))
    return fail(MB_EINVAL, "mb_layer_create: sizes must be positive, eps >= 0, theta > 0");
  if (d.n_q_heads % d.n_kv_heads != 0)
    return fail(MB_EINVAL, "mb_layer_create: n_q_heads must be a multiple of n_kv_heads");
  if (d.head_dim != 64 && d.head_dim != 128)
    return fail(MB_EUNSUPPORTED, "mb_layer_create: head_dim %d (supported: 64, 128)", d.head_dim);
  if (d.n_q_heads / d.n_kv_heads > 8)
    return fail(MB_EUNSUPPORTED, "mb_layer_create: GQA group %d > 8", d.n_q_heads / d.n_kv_heads);
  if (d.d_model % 128 || (d.n_q_heads * d.head_dim) % 128 || d.d_ff % 128)
    return fail(MB_EUNSUPPORTED, "mb_layer_create: d_model, n_q_heads*head_dim and d_ff must be multiples of 128");
  if (d.d_model > 8192) return fail(MB_EUNSUPPORTED, "mb_layer_create: d_model > 8192");
  if (!w->g_attn || !w->w_qkv || !w->w_o || !w->g_ffn || !w->w_gate_up || !w->w_down ||
      (d.qk_norm && (!w->g_q || !w->g_k)))
    return fail(MB_EINVAL, "mb_layer_create: missing weight pointer");
  const void *wp[] = {w->g_attn, w->w_qkv, w->w_o, w->g_ffn, w->w_gate_up, w->w_down};
  for (const void *p : wp)
    if (reinterpret_cast<uintptr_t>(p) % 16)
      return fail(MB_EINVAL, "mb_layer_create: weight pointers must be 16-byte aligned");

  mb::DeviceCtx *ctx = nullptr;
  mb_status st = mb::device_ctx(&ctx);
  if (st != MB_OK) return st;

  mb_layer *L = new (std::nothrow) mb_layer();
  if (!L) return fail(MB_ENOMEM, "mb_layer_create: out of host memory");
  L->d = d;
  L->w = *w;
  cudaGetDevice(&L->device);
  L->qkv_dim = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
  const size_t T = static_cast<size_t>(d.max_tokens);
  L->bytes_x = T * d.d_model * 2;
  L->bytes_qkv = T * L->qkv_dim * 2;
  L->bytes_q = T * d.n_q_heads * d.head_dim * 2;
  L->bytes_a = T * d.d_ff * 2;
  struct {
    void **p;
    size_t n;
    const char *what;
  } allocs[] = {{&L->xn, L->bytes_x, "xn"}, {&L->qkv, L->bytes_qkv, "qkv"}, {&L->q, L->bytes_q, "q"},
                {&L->o, L->bytes_q, "o"},   {&L->h, L->bytes_x, "h"},       {&L->hn, L->bytes_x, "hn"},
                {&L->a, L->bytes_a, "a"}};
  for (auto &al : allocs) {
    st = alloc_dev(al.p, al.n, al.what);
    if (st != MB_OK) {
      free_layer_mem(L);
      delete L;
      return st;
    }
  }
  st = alloc_dev(reinterpret_cast<void **>(&L->err), 16, "error word");
  if (st == MB_OK && cudaMemset(L->err, 0, 16) != cudaSuccess) st = fail(MB_ECUDA, "cudaMemset(error word)");
  if (st != MB_OK) {
    free_layer_mem(L);
    delete L;
    return st;
  }
  L->gws = mb::gemm_workspace_carve(ctx->gemm_ws);
  const int hq = d.n_q_heads * d.head_dim;
  cudaError_t e = mb::encode_tmap_2d(&L->tm_wqkv, w->w_qkv, d.d_model, L->qkv_dim, d.d_model * 2ull, 64, 128);
  if (e == cudaSuccess) e = mb::encode_tmap_2d(&L->tm_wo, w->w_o, hq, d.d_model, hq * 2ull, 64, 128);
  if (e == cudaSuccess) e = mb::encode_tmap_2d(&L->tm_wgu, w->w_gate_up, d.d_model, 2ull * d.d_ff, d.d_model * 2ull, 64, 128);
  if (e == cudaSuccess) e = mb::encode_tmap_2d(&L->tm_wd, w->w_down, d.d_ff, d.d_model, d.d_ff * 2ull, 64, 128);
  if (e != cudaSuccess) {
    free_layer_mem(L);
    delete L;
    return fail(MB_ECUDA, "mb_layer_create: tensor map encoding failed (%s)", cudaGetErrorString(e));
  }
  for (auto &s : L->ring) {
    if (cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess) {
      free_layer_mem(L);
      delete L;
      return fail(MB_ECUDA, "mb_layer_create: cudaEventCreate failed");
    }
  }
  *out = L;
  return MB_OK;
}

mb_status mb_destroy(mb_layer *L) {
  if (!L) return MB_OK;
  cudaDeviceSynchronize();
  free_layer_mem(L);
  delete L;
  return MB_OK;
}

mb_status mb_kv_alloc(mb_layer *L, int32_t num_pages, void *dev_buf, mb_kv **out) {
  if (!L || !out || num_pages <= 0) return fail(MB_EINVAL, "mb_kv_alloc: null layer/out or num_pages <= 0");
  if (dev_buf && reinterpret_cast<uintptr_t>(dev_buf) % 128)
    return fail(MB_EINVAL, "mb_kv_alloc: dev_buf must be 128-byte aligned");
  const int64_t Hkv = L->d.n_kv_heads, hd = L->d.head_dim;
  const int64_t z = static_cast<int64_t>(num_pages) * 2 * Hkv;
  if (z > INT32_MAX) return fail(MB_EUNSUPPORTED, "mb_kv_alloc: pool too large for 32-bit TMA coordinates");
  mb_kv *kv = new (std::nothrow) mb_kv();
  if (!kv) return fail(MB_ENOMEM, "mb_kv_alloc: out of host memory");
  kv->layer = L;
  kv->num_pages = num_pages;
  const size_t bytes = static_cast<size_t>(z) * MB_PAGE_TOKENS * hd * 2;
  if (dev_buf) {
    kv->base = dev_buf;
  } else {
    mb_status st = alloc_dev(&kv->base, bytes, "kv pool");
    if (st != MB_OK) {
      delete kv;
      return st;
    }
    kv->owned = true;
  }
  // The attention kernels fetch one (page, K or V, head) block of 16 x hd per
  // copy, as a 5-D view: (64 hd elements, 8 slots, hd/64 halves, 2 slot
  // groups, page*2*Hkv + kv*Hkv + head).  In shared memory that lands as
  // [slot group][hd half][8 slots][128 B], 128-byte swizzled: every 8 keys of
  // one hd half form a swizzle atom, and consecutive atoms of a half sit
  // hd/64 KB apart, which the tensor-core descriptors step over uniformly.
  const uint64_t nh = static_cast<uint64_t>(hd) / 64;
  const uint64_t dims5[5] = {64, 8, nh, MB_PAGE_TOKENS / 8, static_cast<uint64_t>(z)};
  const uint64_t strides5[4] = {static_cast<uint64_t>(hd) * 2, 128, 8ull * hd * 2, MB_PAGE_TOKENS * hd * 2ull};
  const uint32_t box5[5] = {64, 8, static_cast<uint32_t>(nh), MB_PAGE_TOKENS / 8, 1};
  cudaError_t e = mb::encode_tmap_5d(&kv->tmap, kv->base, dims5, strides5, box5);
  if (e != cudaSuccess) {
    if (kv->owned) cudaFree(kv->base);
    delete kv;
    return fail(MB_ECUDA, "mb_kv_alloc: tensor map encoding failed");
  }
  kv->stamp.assign(static_cast<size_t>(num_pages), 0);
  *out = kv;
  return MB_OK;
}

mb_status mb_kv_layout(const mb_kv *kv, int64_t strides[5], void **base) {
  if (!kv || !strides || !base) return fail(MB_EINVAL, "mb_kv_layout: null argument");
  const int64_t Hkv = kv->layer->d.n_kv_heads, hd = kv->layer->d.head_dim;
  strides[4] = 1;
  strides[3] = hd;
  strides[2] = MB_PAGE_TOKENS * hd;
  strides[1] = Hkv * MB_PAGE_TOKENS * hd;
  strides[0] = 2 * Hkv * MB_PAGE_TOKENS * hd;
  *base = kv->base;
  return MB_OK;
}

mb_status mb_kv_free(mb_kv *kv) {
  if (!kv) return MB_OK;
  if (kv->owned) {
    cudaDeviceSynchronize();
    cudaFree(kv->base);
  }
  delete kv;
  return MB_OK;
}

mb_status mb_layer_buffer(const mb_layer *L, int32_t which, void **ptr, int64_t *bytes) {
  if (!L || !ptr || !bytes) return fail(MB_EINVAL, "mb_layer_buffer: null argument");
  const int64_t T = L->last_T;
  const int64_t d = L->d.d_model, hq = L->d.n_q_heads * L->d.head_dim;
  switch (which) {
    case 0: *ptr = L->xn; *bytes = T * d * 2; break;
    case 1: *ptr = L->qkv; *bytes = T * L->qkv_dim * 2; break;
    case 2: *ptr = L->q; *bytes = T * hq * 2; break;
    case 3: *ptr = L->o; *bytes = T * hq * 2; break;
    case 4: *ptr = L->h; *bytes = T * d * 2; break;
    case 5: *ptr = L->hn; *bytes = T * d * 2; break;
    case 6: *ptr = L->a; *bytes = T * L->d.d_ff * 2; break;
    default: return fail(MB_EINVAL, "mb_layer_buffer: unknown buffer %d", which);
  }
  return MB_OK;
}

mb_status mb_layer_set_gemm_sms(mb_layer *L, int32_t n) {
  if (!L) return fail(MB_EINVAL, "mb_layer_set_gemm_sms: null layer");
  if (n < 0) return fail(MB_EINVAL, "mb_layer_set_gemm_sms: n must be >= 0");
  L->gws.max_ctas = n;
  return MB_OK;
}

mb_status mb_layer_set_gemm_workspace(mb_layer *L, void *workspace) {
  if (!L) return fail(MB_EINVAL, "mb_layer_set_gemm_workspace: null layer");
  if (reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(MB_EINVAL, "mb_layer_set_gemm_workspace: workspace must be 256-byte aligned");
  mb::DeviceCtx *ctx = nullptr;
  mb_status st = mb::device_ctx(&ctx);
  if (st != MB_OK) return st;
  const int cap = L->gws.max_ctas;
  L->gws = mb::gemm_workspace_carve(workspace ? workspace : ctx->gemm_ws);
  L->gws.max_ctas = cap;
  return MB_OK;
}

mb_status mb_layer_set_decode_sms(mb_layer *L, int32_t n) {
  if (!L) return fail(MB_EINVAL, "mb_layer_set_decode_sms: null layer");
  if (n < 0) return fail(MB_EINVAL, "mb_layer_set_decode_sms: n must be >= 0");
  L->dec_sms = n;
  return MB_OK;
}

mb_status mb_layer_set_timing(mb_layer *L, int32_t enable) {
  if (!L) return fail(MB_EINVAL, "mb_layer_set_timing: null layer");
  mb_status st = flush_timing(L);
  if (st != MB_OK) return st;
  L->timing = enable != 0;
  std::fill(L->ms, L->ms + kNumTimed, 0.0);
  L->steps_timed = 0;
  return MB_OK;
}

mb_status mb_layer_timing(mb_layer *L, double *ms, int32_t n, int64_t *steps) {
  if (!L || (n > 0 && !ms)) return fail(MB_EINVAL, "mb_layer_timing: null argument");
  mb_status st = flush_timing(L);
  if (st != MB_OK) return st;
  for (int i = 0; i < n && i < kNumTimed; ++i) ms[i] = L->ms[i];
  if (steps) *steps = L->steps_timed;
  return MB_OK;
}

int32_t mb_layer_last_launches(const mb_layer *L) { return L ? L->last_launches : 0; }

int64_t mb_layer_last_upload_bytes(const mb_layer *L) { return L ? L->last_upload : 0; }

mb_status mb_device_status(mb_layer *L, void *stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(MB_ECUDA, "mb_device_status: %s", cudaGetErrorString(e));
  // A layer's context exists (its creation set it up).  Without a layer the
  // call allocates nothing: it reads the context's word only if some entry
  // point has set the context up, then the allocation-free GEMM's word.
  mb::DeviceCtx *ctx = nullptr;
  if (L) {
    mb_status st = mb::device_ctx(&ctx);
    if (st != MB_OK) return st;
  } else {
    ctx = mb::device_ctx_if_ready();
  }
  int code = 0;
  if (ctx) {
    int *errp = L ? L->err : ctx->err;
    e = cudaMemcpy(&code, errp, sizeof code, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(MB_ECUDA, "mb_device_status: %s", cudaGetErrorString(e));
    if (code != 0) {
      cudaMemset(errp, 0, 16);
      // a decode worker that gave up may leave split-merge counters raised
      if (L && L->part) cudaMemset(L->part, 0, L->part_cap * 4);
      // a kernel that unwound early may leave stream-K tickets raised (in the
      // device's workspace, and in the layer's own if it has one)
      cudaMemset(ctx->gemm_ws, 0, mb::gemm_workspace_bytes());
      if (L && static_cast<void *>(L->gws.partials) != ctx->gemm_ws)
        cudaMemset(L->gws.partials, 0, mb::gemm_workspace_bytes());
    }
  }
  if (!L) {
    int nc = 0;
    e = mb::gemm_noalloc_take_error(&nc);
    if (e != cudaSuccess) return fail(MB_ECUDA, "mb_device_status: %s", cudaGetErrorString(e));
    if (code == 0) code = nc;
  }
  if (code != 0) return fail(MB_EDEVICE, "mb_device_status: kernel error code %d", code);
  return MB_OK;
}

// ------------------------------------------------------------------ GEMM
mb_status mb_gemm(const void *A, const void *B, void *D, const void *R, int32_t M, int32_t N, int32_t K,
                  int32_t epilogue, void *workspace, void *stream) {
  if (!A || !B || !D || M < 0 || N <= 0 || K <= 0) return fail(MB_EINVAL, "mb_gemm: bad argument");
  if (epilogue < 0 || epilogue > 2) return fail(MB_EINVAL, "mb_gemm: epilogue must be 0, 1 or 2");
  if (epilogue == 1 && (!R || R == D)) return fail(MB_EINVAL, "mb_gemm: residual epilogue needs R != D");
  if (K % 64) return fail(MB_EUNSUPPORTED, "mb_gemm: K must be a multiple of 64");
  if (epilogue == 2 && N % 128) return fail(MB_EUNSUPPORTED, "mb_gemm: SwiGLU needs F = N %% 128 == 0");
  if (N % 32) return fail(MB_EUNSUPPORTED, "mb_gemm: N must be a multiple of 32");
  for (const void *p : {A, B, static_cast<const void *>(D), R})
    if (p && reinterpret_cast<uintptr_t>(p) % 16) return fail(MB_EINVAL, "mb_gemm: pointers must be 16-byte aligned");
  if (M == 0) return MB_OK;
  mb::DeviceCtx *ctx = nullptr;
  mb_status st = mb::device_ctx(&ctx);
  if (st != MB_OK) return st;
  mb::GemmWorkspace ws = mb::gemm_workspace_carve(workspace ? workspace : ctx->gemm_ws);
  cudaError_t e = mb::gemm_run(A, B, nullptr, D, R, M, N, K, epilogue, ws, ctx->err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return mb::cuda_fail(e, "mb_gemm");
  return MB_OK;
}

// ------------------------------------------------------- next tokens
mb_status mb_sample_greedy(const void *x, int32_t T, const int32_t *rows, int32_t n_rows, int32_t d, float eps,
                           const void *g_final, const void *w_lm, int32_t vocab, void *y_work, void *logits,
                           int32_t *ids, void *stream) {
  if (!x || !rows || !g_final || !w_lm || !y_work || !logits || !ids || T < 0 || n_rows < 0 || d <= 0 || vocab <= 0)
    return fail(MB_EINVAL, "mb_sample_greedy: bad argument");
  if (d % 64) return fail(MB_EUNSUPPORTED, "mb_sample_greedy: d must be a multiple of 64");
  if (vocab % 32) return fail(MB_EUNSUPPORTED, "mb_sample_greedy: vocab must be a multiple of 32");
  if (d > 8192) return fail(MB_EUNSUPPORTED, "mb_sample_greedy: d must be at most 8192");
  for (const void *p : {x, g_final, w_lm, static_cast<const void *>(y_work), static_cast<const void *>(logits)})
    if (reinterpret_cast<uintptr_t>(p) % 16) return fail(MB_EINVAL, "mb_sample_greedy: pointers must be 16-byte aligned");
  if (n_rows == 0) return MB_OK;
  mb::DeviceCtx *ctx = nullptr;
  mb_status st = mb::device_ctx(&ctx);
  if (st != MB_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = mb::rmsnorm_rows_run(x, T, rows, n_rows, g_final, y_work, d, eps, ctx->err, s);
  if (e != cudaSuccess) return mb::cuda_fail(e, "mb_sample_greedy: final norm");
  e = mb::gemm_run(y_work, w_lm, nullptr, logits, nullptr, n_rows, vocab, d, mb::kEpiStore,
                   mb::gemm_workspace_carve(ctx->gemm_ws), ctx->err, s);
  if (e != cudaSuccess) return mb::cuda_fail(e, "mb_sample_greedy: LM head");
  e = mb::argmax_rows_run(logits, n_rows, vocab, ids, s);
  if (e != cudaSuccess) return mb::cuda_fail(e, "mb_sample_greedy: argmax");
  return MB_OK;
}

mb_status mb_embed(const void *table, int32_t vocab, int32_t d, const int32_t *ids, int32_t n, void *out,
                   void *stream) {
  if (!table || !ids || !out || vocab <= 0 || d <= 0 || n < 0) return fail(MB_EINVAL, "mb_embed: bad argument");
  if (d % 8) return fail(MB_EUNSUPPORTED, "mb_embed: d must be a multiple of 8");
  if (reinterpret_cast<uintptr_t>(table) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(MB_EINVAL, "mb_embed: table and out must be 16-byte aligned");
  if (n == 0) return MB_OK;
  mb::DeviceCtx *ctx = nullptr;
  mb_status st = mb::device_ctx(&ctx);
  if (st != MB_OK) return st;
  cudaError_t e = mb::embed_rows_run(table, vocab, d, ids, n, out, ctx->err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return mb::cuda_fail(e, "mb_embed");
  return MB_OK;
}

// ------------------------------------------------------------------ step
mb_status mb_step(mb_layer *L, mb_kv *kv, const mb_batch *b, const void *x_in, void *x_out, void *stream) {
  if (!L || !kv || !b || !x_in || !x_out) return fail(MB_EINVAL, "mb_step: null argument");
  if (kv->layer != L) return fail(MB_EINVAL, "mb_step: kv pool belongs to another layer");
  if (x_in == x_out) return fail(MB_EINVAL, "mb_step: x_out must not alias x_in");
  if (reinterpret_cast<uintptr_t>(x_in) % 16 || reinterpret_cast<uintptr_t>(x_out) % 16)
    return fail(MB_EINVAL, "mb_step: x_in and x_out must be 16-byte aligned");
  if (b->num_reqs < 0) return fail(MB_EINVAL, "mb_step: num_reqs < 0");
  L->last_launches = 0;
  if (b->num_reqs == 0) {
    L->last_T = 0;
    return MB_OK;
  }
  if (++kv->stamp_gen == 0) {
    std::fill(kv->stamp.begin(), kv->stamp.end(), 0u);
    kv->stamp_gen = 1;
  }
  int64_t T = 0;
  mb_status st = validate_batch(b, kv->num_pages, L->d.max_tokens, kv->stamp.data(), kv->stamp_gen, &T);
  if (st != MB_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StepPlan plan;
  if ((st = prepare_step(L, b, T, s, &plan)) != MB_OK) return st;
  EventSet *es = nullptr;
  if (L->timing) {
    if (L->ev_used == 4096 && (st = flush_timing(L)) != MB_OK) return st;
    if (L->ev_used == L->ev_pool.size()) {
      EventSet ns;
      for (auto &ev : ns.ev) cudaEventCreate(&ev);
      L->ev_pool.push_back(ns);
    }
    es = &L->ev_pool[L->ev_used++];
  }
  int launches = 0;
  if ((st = launch_layer(L, L, kv, plan, x_in, x_out, s, es, &launches)) != MB_OK) return st;
  L->last_T = static_cast<int32_t>(T);
  L->last_launches = launches;
  L->last_upload = plan.upload_bytes;
  L->last_stream = s;
  return MB_OK;
}

// ------------------------------------------------------------------ stack
mb_status mb_stack_create(mb_layer *const *layers, int32_t n_layers, int32_t use_graphs, mb_stack **out) {
  if (!layers || n_layers <= 0 || !out) return fail(MB_EINVAL, "mb_stack_create: need layers and n_layers > 0");
  const mb_layer_desc &d0 = layers[0]->d;
  for (int i = 0; i < n_layers; ++i) {
    const mb_layer *L = layers[i];
    if (!L) return fail(MB_EINVAL, "mb_stack_create: layer %d is null", i);
    const mb_layer_desc &d = L->d;
    if (d.d_model != d0.d_model || d.n_q_heads != d0.n_q_heads || d.n_kv_heads != d0.n_kv_heads ||
        d.head_dim != d0.head_dim || d.d_ff != d0.d_ff || d.max_tokens != d0.max_tokens ||
        d.qk_norm != d0.qk_norm || L->device != layers[0]->device)
      return fail(MB_EINVAL, "mb_stack_create: layer %d differs in shape, max_tokens or device from layer 0", i);
  }
  mb_stack *S = new (std::nothrow) mb_stack();
  if (!S) return fail(MB_ENOMEM, "mb_stack_create: out of host memory");
  S->layers.assign(layers, layers + n_layers);
  S->use_graphs = use_graphs != 0;
  if (cudaStreamCreateWithFlags(&S->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
    delete S;
    return fail(MB_ECUDA, "mb_stack_create: cudaStreamCreate failed");
  }
  const size_t bytes = static_cast<size_t>(d0.max_tokens) * d0.d_model * 2;
  for (int i = 0; i < 2; ++i) {
    mb_status st = alloc_dev(&S->act[i], bytes, "stack activations");
    if (st != MB_OK) {
      mb_stack_destroy(S);
      return st;
    }
  }
  *out = S;
  return MB_OK;
}

mb_status mb_stack_step(mb_stack *S, mb_kv *const *kvs, const mb_batch *b, const void *x_in, void *x_out,
                        void *stream) {
  if (!S || !kvs || !b || !x_in || !x_out) return fail(MB_EINVAL, "mb_stack_step: null argument");
  if (x_in == x_out) return fail(MB_EINVAL, "mb_stack_step: x_out must not alias x_in");
  if (reinterpret_cast<uintptr_t>(x_in) % 16 || reinterpret_cast<uintptr_t>(x_out) % 16)
    return fail(MB_EINVAL, "mb_stack_step: x_in and x_out must be 16-byte aligned");
  const int nl = static_cast<int>(S->layers.size());
  int32_t min_pages = INT32_MAX;
  for (int i = 0; i < nl; ++i) {
    if (!kvs[i] || kvs[i]->layer != S->layers[i])
      return fail(MB_EINVAL, "mb_stack_step: kv pool %d is missing or belongs to another layer", i);
    min_pages = std::min(min_pages, kvs[i]->num_pages);
  }
  if (b->num_reqs < 0) return fail(MB_EINVAL, "mb_stack_step: num_reqs < 0");
  S->last_launches = 0;
  if (b->num_reqs == 0) return MB_OK;
  mb_layer *L0 = S->layers[0];
  if (S->stamp.size() < static_cast<size_t>(min_pages)) S->stamp.assign(static_cast<size_t>(min_pages), 0u);
  if (++S->stamp_gen == 0) {
    std::fill(S->stamp.begin(), S->stamp.end(), 0u);
    S->stamp_gen = 1;
  }
  int64_t T = 0;
  mb_status st = validate_batch(b, min_pages, L0->d.max_tokens, S->stamp.data(), S->stamp_gen, &T);
  if (st != MB_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StepPlan plan;
  if ((st = prepare_step(L0, b, T, s, &plan)) != MB_OK) return st;

  // Every launch of the L layers depends on the batch only through the
  // plan's sizes and the (fixed) buffers, so one captured graph serves every
  // step with the same geometry.
  uint32_t dec_sms_key = 0;   // every layer's decode SM cap (a change re-captures)
  for (mb_layer *Li : S->layers) dec_sms_key = dec_sms_key * 31u + static_cast<uint32_t>(Li->dec_sms);
  GraphKey key{};
  key.T = T;
  key.n_reqs = b->num_reqs;
  key.n_tiles = plan.n_tiles;
  key.n_items = plan.n_items;
  key.n_merge = plan.n_merge;
  key.n_chunk_slots = plan.n_chunk_slots;
  key.ctr_cap = L0->ctr_cap;
  key.gemm_ctas = L0->gws.max_ctas;   // every layer's GEMMs run on layer 0's workspace
  key.dec_workers = plan.dec_workers;
  key.gws = L0->gws.partials;
  const size_t offs[8] = {plan.o_qo, plan.o_kv, plan.o_bti, plan.o_bt, plan.o_treq, plan.o_tpos, plan.o_tiles,
                          plan.o_items};
  std::copy(offs, offs + 8, key.offs);
  key.db = plan.db;
  key.part = L0->part;
  key.x_in = x_in;
  key.x_out = x_out;
  key.kv0 = kvs[0];
  key.dec_sms = static_cast<int>(dec_sms_key);
  auto enqueue = [&](int *launches) -> mb_status {
    for (int i = 0; i < nl; ++i) {
      const void *in = i == 0 ? x_in : S->act[(i - 1) & 1];
      void *outp = i == nl - 1 ? x_out : S->act[i & 1];
      mb_status st2 = launch_layer(S->layers[i], L0, kvs[i], plan, in, outp, s, nullptr, launches);
      if (st2 != MB_OK) return st2;
    }
    return MB_OK;
  };
  int launches = 0;
  if (!S->use_graphs) {
    if ((st = enqueue(&launches)) != MB_OK) return st;
  } else {
    // graphs hold every layer's pool: a different set of pools invalidates them
    if (!S->graph_kvs.empty() && !std::equal(kvs, kvs + nl, S->graph_kvs.begin())) S->drop_graphs();
    cudaGraphExec_t exec = nullptr;
    for (auto &g : S->graphs)
      if (g.key == key) exec = g.exec;
    if (!exec) {
      // capture on the stack's own stream (capturing the legacy default
      // stream is not allowed); the graph is then launched on `s`
      cudaStream_t cs = S->cap_stream;
      s = cs;
      cudaGraph_t graph = nullptr;
      cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
      if (e != cudaSuccess) return mb::fail(MB_ECUDA, "mb_stack_step: begin capture: %s", cudaGetErrorString(e));
      st = enqueue(&launches);
      e = cudaStreamEndCapture(cs, &graph);
      s = static_cast<cudaStream_t>(stream);
      if (st != MB_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
      }
      if (e != cudaSuccess) return mb::fail(MB_ECUDA, "mb_stack_step: end capture: %s", cudaGetErrorString(e));
      e = cudaGraphInstantiate(&exec, graph, 0);
      cudaGraphDestroy(graph);
      if (e != cudaSuccess) return mb::fail(MB_ECUDA, "mb_stack_step: instantiate: %s", cudaGetErrorString(e));
      if (S->graphs.size() == 8) S->drop_graphs();
      S->graphs.push_back({key, exec, launches});
      S->graph_kvs.assign(kvs, kvs + nl);
    } else {
      for (auto &g : S->graphs)
        if (g.key == key) launches = g.launches;
    }
    cudaError_t e = cudaGraphLaunch(exec, s);
    if (e != cudaSuccess) return mb::fail(MB_ECUDA, "mb_stack_step: graph launch: %s", cudaGetErrorString(e));
  }
  S->last_launches = launches;
  S->last_T = static_cast<int32_t>(T);
  L0->last_upload = plan.upload_bytes;   // the stack's one descriptor upload goes through layer 0
  return MB_OK;
}

int32_t mb_stack_last_launches(const mb_stack *S) { return S ? S->last_launches : 0; }

mb_status mb_stack_destroy(mb_stack *S) {
  if (!S) return MB_OK;
  cudaDeviceSynchronize();
  S->drop_graphs();
  for (void *p : S->act)
    if (p) cudaFree(p);
  if (S->cap_stream) cudaStreamDestroy(S->cap_stream);
  delete S;
  return MB_OK;
}

}  // extern "C"
