// Bandwidth-bound kernels of the step: RMSNorm, and the fused
// (q/k RMSNorm) + RoPE + KV-append that writes this step's keys and values
// into their 16-token pages before attention reads them (pofe.ai "Chunked
// prefill", "How it works, step by step", step 4: chunks write their K/V into
// the cache, then attend).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "mb_kernels.h"
#include "mb_launch.cuh"
#include "mb_ptx.cuh"

namespace mb {
namespace {

using namespace dev;

// ------------------------------------------------------------------ RMSNorm
// y = x / sqrt(mean(x^2) + eps) * g, one CTA per row, 16-byte vectors.
constexpr int kNormThreads = 128;
constexpr int kNormMaxVec = 8;  // d <= 128 * 8 * 8 = 8192

// rows (optional): output row i normalises input row rows[i] (each in
// [0, n_src); an id out of range records kErrBounds and gives a zero row).
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const __nv_bfloat16 *__restrict__ x,
                                                               const __nv_bfloat16 *__restrict__ g,
                                                               __nv_bfloat16 *__restrict__ y, int d, float eps,
                                                               const int32_t *__restrict__ rows, int n_src, int *err) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const int nv = d / 8;
  int src = row;
  if (rows) {
    src = rows[row];
    if (src < 0 || src >= n_src) {
      if (threadIdx.x == 0) atomicExch(err, kErrBounds);
      uint4 *yr = reinterpret_cast<uint4 *>(y + static_cast<size_t>(row) * d);
      for (int v = threadIdx.x; v < nv; v += kNormThreads) yr[v] = make_uint4(0, 0, 0, 0);
      return;
    }
  }
  const uint4 *xr = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(src) * d);
  const uint4 *gr = reinterpret_cast<const uint4 *>(g);
  uint4 buf[kNormMaxVec], gbuf[kNormMaxVec];
  float ss = 0.f;
  // the gains are requested with the row, not after the reduction
#pragma unroll
  for (int i = 0; i < kNormMaxVec; ++i) {
    const int v = threadIdx.x + i * kNormThreads;
    if (v < nv) {
      buf[i] = xr[v];
      gbuf[i] = gr[v];
    }
  }
#pragma unroll
  for (int i = 0; i < kNormMaxVec; ++i) {
    const int v = threadIdx.x + i * kNormThreads;
    if (v < nv) {
      const uint32_t w[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = bf16lo(w[e]), b = bf16hi(w[e]);
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  __shared__ float red[kNormThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += red[i];
  const float inv = rsqrtf(tot / static_cast<float>(d) + eps);
  uint4 *yr = reinterpret_cast<uint4 *>(y + static_cast<size_t>(row) * d);
#pragma unroll
  for (int i = 0; i < kNormMaxVec; ++i) {
    const int v = threadIdx.x + i * kNormThreads;
    if (v < nv) {
      const uint4 gv = gbuf[i];
      const uint32_t w[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o[e] = pack_bf16x2(bf16lo(w[e]) * inv * bf16lo(gw[e]), bf16hi(w[e]) * inv * bf16hi(gw[e]));
      yr[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// ------------------------------------------------------- RoPE + KV append
// One CTA per token; warp w handles heads w, w + 8, ... of
// [Q heads | K heads | V heads].  Rotate-half pairing (i, i + hd/2) with
// frequency theta^(-2i/hd) at the token's absolute position.  The angle is
// pos * f with f split into a float head and tail (pos is exact in fp32), and
// reduced modulo 2 pi with a two-constant Cody-Waite step (W. J. Cody and
// W. Waite, "Software Manual for the Elementary Functions", 1980: 2 pi split
// into its fp32 value and the remainder) before sincosf is called, so it
// keeps ~1e-6 rad accuracy at positions in the tens of thousands.
constexpr int kRopeThreads = 256;
constexpr float kTwoPiHi = 6.28318548202514648f;         // fp32(2 pi)
constexpr float kTwoPiLo = -1.7484556000744893e-07f;     // 2 pi - kTwoPiHi

struct RopeParams {
  const __nv_bfloat16 *qkv;
  __nv_bfloat16 *q_out;
  __nv_bfloat16 *pool;
  const int32_t *tok_req, *tok_pos, *bt_indptr, *bt;
  const __nv_bfloat16 *g_q, *g_k;
  int Hq, Hkv, qk_norm, num_pages;
  float eps;
  int *err;
  float f_hi[64], f_lo[64];
};

// Element pairs of a head row, by lane: PAIRS consecutive elements of each
// half (bf16x2 loads and stores for hd 128, single elements for hd 64).
template <int PAIRS>
struct HalfVec;
template <>
struct HalfVec<1> {
  using T = uint16_t;
  static __device__ __forceinline__ void unpack(T v, float (&x)[1]) { x[0] = __uint_as_float(static_cast<uint32_t>(v) << 16); }
  static __device__ __forceinline__ T pack(const float (&x)[1]) {
    return static_cast<uint16_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x[0])));
  }
};
template <>
struct HalfVec<2> {
  using T = uint32_t;
  static __device__ __forceinline__ void unpack(T v, float (&x)[2]) {
    x[0] = bf16lo(v);
    x[1] = bf16hi(v);
  }
  static __device__ __forceinline__ T pack(const float (&x)[2]) { return pack_bf16x2(x[0], x[1]); }
};

template <int HD>
__global__ void __launch_bounds__(kRopeThreads) rope_append_kernel(const RopeParams p) {
  constexpr int HALF = HD / 2;
  constexpr int PAIRS = HALF / 32;          // elements of each half per lane
  constexpr int NW = kRopeThreads / 32;
  constexpr int MAXH = 8;                   // heads a warp holds in registers per round
  using V = HalfVec<PAIRS>;
  using VT = typename V::T;
  __shared__ float cs[HALF], sn[HALF];
  __shared__ int s_page;
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads = p.Hq + 2 * p.Hkv;
  const int row_len = heads * HD;
  const VT *src_row = reinterpret_cast<const VT *>(p.qkv + static_cast<size_t>(t) * row_len);
  // Every load below is independent of the position and the page, so the
  // first round's head rows are requested before the position, the sines and
  // the page lookup (three dependent loads) are worked out.
  VT a1[MAXH], a2[MAXH];
  auto load_round = [&](int base) {
#pragma unroll
    for (int k = 0; k < MAXH; ++k) {
      const int hh = base + warp + k * NW;
      if (hh < heads) {
        a1[k] = src_row[(hh * HD) / PAIRS + lane];
        a2[k] = src_row[(hh * HD + HALF) / PAIRS + lane];
      }
    }
  };
  load_round(0);
  const int pos = p.tok_pos[t];
  for (int i = threadIdx.x; i < HALF; i += kRopeThreads) {
    const float fp = static_cast<float>(pos);
    const float hi = fp * p.f_hi[i];
    const float lo = fmaf(fp, p.f_hi[i], -hi) + fp * p.f_lo[i];
    const float k = rintf(hi * 0.15915494309189535f);
    float r = fmaf(-k, kTwoPiHi, hi);
    r = fmaf(-k, kTwoPiLo, r) + lo;
    float sv, cv;
    sincosf(r, &sv, &cv);
    cs[i] = cv;
    sn[i] = sv;
  }
  if (threadIdx.x == kRopeThreads - 32) {   // the last warp looks the page up
    const int req = p.tok_req[t];
    const int page = p.bt[p.bt_indptr[req] + pos / kPage];
    s_page = (page < 0 || page >= p.num_pages) ? -1 : page;
  }
  __syncthreads();
  const int page = s_page;
  if (page < 0) {
    if (threadIdx.x == 0) atomicExch(p.err, kErrBounds);
    return;
  }
  const int slot = pos % kPage;
  for (int base = 0; base < heads; base += NW * MAXH) {
    if (base > 0) load_round(base);
#pragma unroll
    for (int k = 0; k < MAXH; ++k) {
      const int hh = base + warp + k * NW;
      if (hh >= heads) break;
      float x1[PAIRS], x2[PAIRS];
      V::unpack(a1[k], x1);
      V::unpack(a2[k], x2);
      const bool is_q = hh < p.Hq;
      const bool is_k = !is_q && hh < p.Hq + p.Hkv;
      if (is_q || is_k) {
        if (p.qk_norm) {
          float ss = 0.f;
#pragma unroll
          for (int j = 0; j < PAIRS; ++j) ss += x1[j] * x1[j] + x2[j] * x2[j];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
          const float inv = rsqrtf(ss / static_cast<float>(HD) + p.eps);
          const __nv_bfloat16 *g = is_q ? p.g_q : p.g_k;
#pragma unroll
          for (int j = 0; j < PAIRS; ++j) {
            const int i = lane * PAIRS + j;
            x1[j] = x1[j] * inv * __bfloat162float(g[i]);
            x2[j] = x2[j] * inv * __bfloat162float(g[i + HALF]);
          }
        }
#pragma unroll
        for (int j = 0; j < PAIRS; ++j) {
          const int i = lane * PAIRS + j;
          const float a = x1[j], b = x2[j];
          x1[j] = a * cs[i] - b * sn[i];
          x2[j] = b * cs[i] + a * sn[i];
        }
      }
      VT *dst;
      if (is_q) {
        dst = reinterpret_cast<VT *>(p.q_out + (static_cast<size_t>(t) * p.Hq + hh) * HD);
      } else {
        const int kvsel = is_k ? 0 : 1;
        const int hk = is_k ? hh - p.Hq : hh - p.Hq - p.Hkv;
        dst = reinterpret_cast<VT *>(p.pool + (((static_cast<size_t>(page) * 2 + kvsel) * p.Hkv + hk) * kPage + slot) * HD);
      }
      dst[lane] = V::pack(x1);
      dst[HALF / PAIRS + lane] = V::pack(x2);
    }
  }
}

// ------------------------------------------------------- greedy sampling
// One CTA per row: the largest logit and its index, the lowest index among
// equal maxima (a NaN never wins).  16-byte loads of 8 bf16.
constexpr int kArgmaxThreads = 256;

__device__ __forceinline__ bool argmax_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kArgmaxThreads) argmax_kernel(const __nv_bfloat16 *__restrict__ logits, int vocab,
                                                                int32_t *__restrict__ ids) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const uint4 *lr = reinterpret_cast<const uint4 *>(logits + static_cast<size_t>(row) * vocab);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int v = threadIdx.x; v < vocab / 8; v += kArgmaxThreads) {
    const uint4 q = lr[v];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = bf16lo(w[e]), b = bf16hi(w[e]);
      const int i = 8 * v + 2 * e;
      if (argmax_better(a, i, bv, bi)) { bv = a; bi = i; }
      if (argmax_better(b, i + 1, bv, bi)) { bv = b; bi = i + 1; }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
    if (argmax_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  __shared__ float sv[kArgmaxThreads / 32];
  __shared__ int si[kArgmaxThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kArgmaxThreads / 32; ++w)
      if (argmax_better(sv[w], si[w], bv, bi)) { bv = sv[w]; bi = si[w]; }
    ids[row] = bi == 0x7fffffff ? 0 : bi;   // all NaN: token 0
  }
}

// ------------------------------------------------------------ embeddings
constexpr int kEmbedThreads = 128;

__global__ void __launch_bounds__(kEmbedThreads) embed_kernel(const __nv_bfloat16 *__restrict__ table, int vocab, int d,
                                                              const int32_t *__restrict__ ids,
                                                              __nv_bfloat16 *__restrict__ out, int *err) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const int id = ids[row];
  uint4 *o = reinterpret_cast<uint4 *>(out + static_cast<size_t>(row) * d);
  if (id < 0 || id >= vocab) {
    if (threadIdx.x == 0) atomicExch(err, kErrBounds);
    for (int v = threadIdx.x; v < d / 8; v += kEmbedThreads) o[v] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4 *t = reinterpret_cast<const uint4 *>(table + static_cast<size_t>(id) * d);
  for (int v = threadIdx.x; v < d / 8; v += kEmbedThreads) o[v] = t[v];
}

}  // namespace

cudaError_t rmsnorm_run(const void *x, const void *g, void *y, int rows, int d, float eps, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (d % 8 != 0 || d > kNormThreads * kNormMaxVec * 8) return cudaErrorInvalidValue;
  return launch_pdl(rmsnorm_kernel, dim3(rows), dim3(kNormThreads), 0, st, 1, static_cast<const __nv_bfloat16 *>(x),
                    static_cast<const __nv_bfloat16 *>(g), static_cast<__nv_bfloat16 *>(y), d, eps,
                    static_cast<const int32_t *>(nullptr), 0, static_cast<int *>(nullptr));
}

cudaError_t rmsnorm_rows_run(const void *x, int n_src, const int32_t *rows, int n_rows, const void *g, void *y, int d,
                             float eps, int *err, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  if (d % 8 != 0 || d > kNormThreads * kNormMaxVec * 8) return cudaErrorInvalidValue;
  return launch_pdl(rmsnorm_kernel, dim3(n_rows), dim3(kNormThreads), 0, st, 1, static_cast<const __nv_bfloat16 *>(x),
                    static_cast<const __nv_bfloat16 *>(g), static_cast<__nv_bfloat16 *>(y), d, eps, rows, n_src, err);
}

cudaError_t argmax_rows_run(const void *logits, int n_rows, int vocab, int32_t *ids, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  if (vocab <= 0 || vocab % 8 != 0) return cudaErrorInvalidValue;
  return launch_pdl(argmax_kernel, dim3(n_rows), dim3(kArgmaxThreads), 0, st, 1,
                    static_cast<const __nv_bfloat16 *>(logits), vocab, ids);
}

cudaError_t embed_rows_run(const void *table, int vocab, int d, const int32_t *ids, int n, void *out, int *err,
                           cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (d % 8 != 0) return cudaErrorInvalidValue;
  return launch_pdl(embed_kernel, dim3(n), dim3(kEmbedThreads), 0, st, 1, static_cast<const __nv_bfloat16 *>(table),
                    vocab, d, ids, static_cast<__nv_bfloat16 *>(out), err);
}

cudaError_t rope_append_run(const RopeArgs &a, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  RopeParams p;
  p.qkv = static_cast<const __nv_bfloat16 *>(a.qkv);
  p.q_out = static_cast<__nv_bfloat16 *>(a.q_out);
  p.pool = static_cast<__nv_bfloat16 *>(a.pool);
  p.tok_req = a.tok_req;
  p.tok_pos = a.tok_pos;
  p.bt_indptr = a.bt_indptr;
  p.bt = a.bt;
  p.g_q = static_cast<const __nv_bfloat16 *>(a.g_q);
  p.g_k = static_cast<const __nv_bfloat16 *>(a.g_k);
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.qk_norm = a.qk_norm;
  p.num_pages = a.num_pages;
  p.eps = a.eps;
  p.err = a.err;
  const int half = a.hd / 2;
  for (int i = 0; i < 64; ++i) {
    double f = i < half ? std::pow(static_cast<double>(a.theta), -2.0 * i / a.hd) : 0.0;
    p.f_hi[i] = static_cast<float>(f);
    p.f_lo[i] = static_cast<float>(f - static_cast<double>(p.f_hi[i]));
  }
  if (a.hd == 128) return launch_pdl(rope_append_kernel<128>, dim3(a.T), dim3(kRopeThreads), 0, st, 1, p);
  if (a.hd == 64) return launch_pdl(rope_append_kernel<64>, dim3(a.T), dim3(kRopeThreads), 0, st, 1, p);
  return cudaErrorInvalidValue;
}

}  // namespace mb
