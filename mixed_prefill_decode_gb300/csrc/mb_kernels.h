// Host-side launchers of the device kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace mb {

constexpr int kPage = 16;

// ---- tensor maps (driver entry point fetched at run time; the library does
// not link libcuda, so it loads on machines without a driver) ----
cudaError_t encode_tmap_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                           uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
cudaError_t encode_tmap_5d(CUtensorMap *map, const void *base, const uint64_t dims[5], const uint64_t strides_bytes[4],
                           const uint32_t box[5]);
int device_sm_count();

// ---- token-batched GEMM on tcgen05 ----
enum GemmEpilogue : int { kEpiStore = 0, kEpiResidual = 1, kEpiSwiGLU = 2 };

struct GemmWorkspace {
  float *partials;  // [2 * kMaxGemmGrid][256][256] fp32
  int *tickets;     // [2 * kMaxGemmGrid]
  int max_ctas = 0; // the GEMMs' CTAs at most (0: one per SM)
};
constexpr int kMaxGemmGrid = 256;
size_t gemm_workspace_bytes();
GemmWorkspace gemm_workspace_carve(void *base);

// D = A B^T (+ R) or SwiGLU; A [M][K], B [Nb][K] (Nb = N, or 2F for SwiGLU
// where N = F is the output width).  tmB may be a pre-encoded map of B (box
// 64 x 128) or nullptr.  A pre-encoded map marks B as a layer's weights, which
// no kernel of the stream writes: the kernel loads its first weight tiles
// before its grid-dependency wait.  With nullptr, B waits like A.
cudaError_t gemm_run(const void *A, const void *B, const CUtensorMap *tmB, void *D, const void *R, int M, int N,
                     int K, int epi, const GemmWorkspace &ws, int *err, cudaStream_t st);
// Kernel launches gemm_run issues for an M x N x K GEMM with epilogue epi
// (one, or none for M = 0).
int gemm_launches(int M, int N, int K, int epi, int max_ctas);

// Error code recorded by the allocation-free GEMM on the current device since
// the last call (0 if none); a non-zero code is cleared.  Allocates nothing.
cudaError_t gemm_noalloc_take_error(int *code);

// ---- element-wise kernels ----
cudaError_t rmsnorm_run(const void *x, const void *g, void *y, int rows, int d, float eps, cudaStream_t st);
// y[i] = RMSNorm(x[rows[i]]) g for i < n_rows (rows: device int32, each in [0, n_src))
cudaError_t rmsnorm_rows_run(const void *x, int n_src, const int32_t *rows, int n_rows, const void *g, void *y, int d,
                             float eps, int *err, cudaStream_t st);
// ids[i] = argmax of bf16 row i of logits [n_rows][vocab] (lowest index among equal maxima)
cudaError_t argmax_rows_run(const void *logits, int n_rows, int vocab, int32_t *ids, cudaStream_t st);
// out[i] = table[ids[i]] (bf16 [vocab][d] -> [n][d])
cudaError_t embed_rows_run(const void *table, int vocab, int d, const int32_t *ids, int n, void *out, int *err,
                           cudaStream_t st);

struct RopeArgs {
  const void *qkv;          // [T][(Hq + 2 Hkv) hd] bf16
  void *q_out;              // [T][Hq][hd] bf16
  void *pool;               // [P][2][Hkv][16][hd] bf16
  const int32_t *tok_req;   // [T] request of each token
  const int32_t *tok_pos;   // [T] absolute position of each token
  const int32_t *bt_indptr; // [n+1]
  const int32_t *bt;        // block tables
  const void *g_q, *g_k;    // [hd] bf16 or null
  int T, Hq, Hkv, hd, qk_norm, num_pages;
  float eps, theta;
  int *err;
};
cudaError_t rope_append_run(const RopeArgs &a, cudaStream_t st);

// ---- attention ----
// Work lists (device int32, built on the host per step):
//   chunk units:   {req, q_row0, q_head, j0, j1, piece, n_pieces, slot} x n_tiles: key blocks [j0, j1)
//                  of a 256-row tile (n_pieces == 1: the whole tile; otherwise piece `piece`, whose
//                  partial goes to slot `slot`, the tile's pieces holding consecutive slots)
//   decode items:  {req, kv_head, page_begin, page_end, split, n_splits, group, slot0} x n_items: a split
//                  item writes its partial to slot slot0 + split (the group's splits hold consecutive slots)
struct AttnArgs {
  const void *q;            // [T][Hq][hd] bf16 (rotated)
  const void *pool;         // [P][2][Hkv][16][hd]
  void *o;                  // [T][Hq hd] bf16
  const int32_t *qo_indptr, *kv_len, *bt_indptr, *bt;
  const int32_t *tiles;     // chunk tile list
  const int32_t *items;     // decode item list
  float *part;              // decode split partials [n_items][Hq/Hkv group][hd + 4]: o, m, l, pad (merged in-kernel)
  int n_tiles, n_items;
  int max_workers;          // decode worker CTAs at most (0: one per SM)
  int T, Hq, Hkv, hd, num_pages;
  int *err;
  const CUtensorMap *tm_q;  // Q map [T][Hq hd], box 64 x 128 (host pointer; copied into launch)
  const CUtensorMap *tm_qd; // Q map [T Hq][hd], box 64 x 16: the G q-heads of one decode row (and padding)
  const CUtensorMap *tm_kv; // pool map, 5-D view of [P*2*Hkv][16][hd]: one (page, K/V, head) block per copy
  int *dec_ctr;             // two ints, zero between launches: decode work counter
  int *merge_ctr;           // one int per split group, zero between launches
  float *chunk_part;        // split chunk tiles' partials [slots][256][hd + 4] (o, m, l, pad)
  int *chunk_ctr;           // one int per slot (the tile's first slot counts its pieces), zero between launches
};
// Prefill-chunk tiles and persistent decode workers (both tcgen05) in one launch.
cudaError_t attention_run(const AttnArgs &a, cudaStream_t st);

}  // namespace mb
