/*
 * mb.h -- one transformer-layer step over a mixed prefill+decode batch, on one
 * GB300 (sm_103a).  C ABI: plain pointers and sizes only.
 *
 * The operation.  A mixed batch holds, per request r, qo_len[r] new tokens and
 * a KV cache that holds kv_len[r] = cached prefix + qo_len[r] tokens once this
 * step has appended its own.  Prefill chunks (qo_len > 1) and decodes
 * (qo_len = 1) share one token-batched pass through the linear layers, then
 * split into a ragged attention over a 16-token paged KV cache:
 *   - ConfluxServe summary (paper-daily.com), "Why can linear layers be batched
 *     but attention cannot?": tokens of both phases form one matrix multiply,
 *     weights are read once; attention splits per request.
 *   - pofe.ai "Chunked prefill", "How it works, step by step", step 4: one
 *     forward pass over the flattened tokens; prompt chunks write their K/V into
 *     the cache and attend causally to everything cached so far; decodes append
 *     one token.
 *   - llm-stack-book 7.8, "Attention on Partial KV Caches": a query at position
 *     T_past + i sees keys 0 .. T_past + i.
 *   - Perplexity "Disaggregated Prefill and Decode", "Prefill versus
 *     Decode-prestaties": qo_len / kv_len framing of prefill and decode rows.
 *
 * The layer (pre-norm, no biases; the pages never write one out, this is the
 * plainest Llama-3 / Qwen3 reading):
 *   xn = RMSNorm(x) g_attn;  [q k v] = xn W_qkv^T;  (Qwen3) q,k = RMSNorm_hd(.) g_q,g_k
 *   q,k = RoPE(rotate-half, pos = cached + i, theta);  append k,v;  o = attention
 *   h = x + o W_o^T;  a = silu(RMSNorm(h) g_ffn W_gate^T) * (RMSNorm(h) g_ffn W_up^T)
 *   y = h + a W_down^T
 *
 * Conventions for every call:
 *   - Return value is an mb_status; on failure mb_last_error() gives a message
 *     (thread-local, valid until the next failing call on that thread).
 *   - "device" pointers are CUDA device addresses on the current device; "host"
 *     pointers are ordinary CPU memory.  Nothing here takes ownership of a
 *     caller pointer unless stated.
 *   - Asynchronous calls run on the given stream (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  Argument and descriptor
 *     errors are returned before anything is launched.  A device-side check
 *     that fails records an error word that mb_device_status() reports.
 *   - There is no CPU fallback: without a usable sm_103a device every compute
 *     call returns MB_ECUDA or MB_EUNSUPPORTED.
 */
#ifndef MB_H_
#define MB_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MB_OK = 0,
  MB_EINVAL = -1,        /* bad argument or malformed batch descriptor */
  MB_ENOMEM = -2,        /* device or pinned-host allocation failed */
  MB_ENOSPACE = -3,      /* KV pages exhausted (scheduler) */
  MB_ECUDA = -4,         /* a CUDA runtime / driver call failed */
  MB_EUNSUPPORTED = -5,  /* shape or device the kernels do not handle */
  MB_EDEVICE = -6        /* a kernel recorded an error (bounds, wait limit) */
} mb_status;

#define MB_PAGE_TOKENS 16

/* Model shape of one layer.  Supported: head_dim in {64, 128}; n_q_heads a
 * multiple of n_kv_heads (GQA group = n_q_heads / n_kv_heads, any value up to
 * 8); d_model, n_q_heads*head_dim and d_ff multiples of 128; max_tokens >= 1. */
typedef struct {
  int32_t d_model;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t d_ff;
  float rms_eps;
  float rope_theta;
  int32_t qk_norm;      /* 1: per-head RMSNorm on q and k before RoPE (Qwen3) */
  int32_t max_tokens;   /* largest T = sum(qo_len) any step will pass */
} mb_layer_desc;

/* Device bf16 weights, caller-owned, must outlive the layer.  Linear weights
 * are row-major [N][K] (y = x W^T), rows 16-byte aligned:
 *   w_qkv     [(Hq + 2 Hkv) hd][d]   rows: Q heads, then K heads, then V heads
 *   w_o       [d][Hq hd]
 *   w_gate_up [2 F][d]               rows: gate (F), then up (F)
 *   w_down    [d][F]
 *   g_attn, g_ffn [d];  g_q, g_k [hd] (may be NULL when qk_norm == 0). */
typedef struct {
  const void *g_attn, *w_qkv, *g_q, *g_k, *w_o, *g_ffn, *w_gate_up, *w_down;
} mb_layer_weights;

/* Batch descriptor, HOST int32 arrays (CSR).  Request r owns step tokens
 * [qo_indptr[r], qo_indptr[r+1]) (so T = qo_indptr[num_reqs]), holds
 * kv_len[r] keys once this step's tokens are appended, and its KV pages are
 * bt[bt_indptr[r] .. bt_indptr[r+1]).  Token p of request r lives in page
 * bt[bt_indptr[r] + p / 16], slot p % 16.  Rules, checked on the host:
 * qo_indptr[0] = 0; 1 <= qo_len <= kv_len; table length >= ceil(kv_len / 16);
 * page ids in [0, num_pages) and distinct across the whole batch;
 * T <= max_tokens.  A request with qo_len = 1 is a decode row. */
typedef struct {
  int32_t num_reqs;
  const int32_t *qo_indptr;
  const int32_t *kv_len;
  const int32_t *bt_indptr;
  const int32_t *bt;
} mb_batch;

typedef struct mb_layer mb_layer;
typedef struct mb_kv mb_kv;

/* Create a layer: validates the shape, keeps the weight pointers, allocates
 * the library-owned workspaces for max_tokens tokens on the current device.
 * Errors: MB_EINVAL (shape), MB_EUNSUPPORTED (shape or device not sm_103),
 * MB_ENOMEM, MB_ECUDA. */
mb_status mb_layer_create(const mb_layer_desc *desc, const mb_layer_weights *w, mb_layer **out);

/* Free a layer and its workspaces (synchronises the device first). */
mb_status mb_destroy(mb_layer *layer);

/* A paged KV pool for this layer: num_pages pages of
 * [2 (K, V)][n_kv_heads][16 slots][head_dim] bf16 (the HND layout of the
 * Perplexity page, "Gesharcde KV Cache Transfers": each head of a page is one
 * contiguous 16 x hd block).  dev_buf: caller device memory of
 * num_pages * 2 * Hkv * 16 * hd * 2 bytes, 128-byte aligned, or NULL to let
 * the library allocate (contents then undefined).  Errors: MB_EINVAL,
 * MB_ENOMEM, MB_ECUDA. */
mb_status mb_kv_alloc(mb_layer *layer, int32_t num_pages, void *dev_buf, mb_kv **out);

/* Element strides of the pool as [page][kv][head][slot][dim] and its base. */
mb_status mb_kv_layout(const mb_kv *kv, int64_t strides[5], void **base);

/* Release a pool (frees the memory only if the library allocated it). */
mb_status mb_kv_free(mb_kv *kv);

/* One layer step, asynchronous on `stream`.
 *   x_in  device bf16 [T][d_model], read only
 *   x_out device bf16 [T][d_model], written; must not alias x_in
 * K/V of every new token are written into `kv` before attention reads it.
 * The descriptor is copied during the call; the caller may reuse its arrays
 * on return.  Workspaces are shared by successive steps of one layer, so
 * steps of one layer must be issued on one stream (or otherwise ordered).
 * T = 0 is a no-op.  Errors: MB_EINVAL (descriptor), MB_ECUDA. */
mb_status mb_step(mb_layer *layer, mb_kv *kv, const mb_batch *batch, const void *x_in,
                  void *x_out, void *stream);

/* ---------------- stacks (several layers, one descriptor per step) ---------
 * A model is L layers applied in turn to the same mixed batch; every layer
 * has its own weights and KV pool, and the batch descriptor is the same for
 * all of them.  A stack uploads the descriptor and builds the work lists once
 * per step and runs the L layers back to back on `stream`, with activations
 * ping-ponging between two library-owned buffers.  All layers must share the
 * model shape, max_tokens and device; they also share the first layer's
 * workspaces, so the layers of a stack must not be stepped concurrently on
 * their own.  With use_graphs != 0 the L layers' launches are captured once
 * into a CUDA graph per batch geometry (T, work-list sizes, buffers) and
 * replayed (the same geometry recurs across steps of a fixed batch shape; the
 * descriptor's contents may change).  Capture happens inside mb_stack_step,
 * so `stream` must not already be capturing.  layers: host array of n_layers
 * handles (not owned).  Errors: MB_EINVAL, MB_ENOMEM, MB_ECUDA. */
typedef struct mb_stack mb_stack;
mb_status mb_stack_create(mb_layer *const *layers, int32_t n_layers, int32_t use_graphs, mb_stack **out);
/* One step of all layers: kvs is a host array of the n_layers pools (pool i
 * belongs to layer i); x_in / x_out device bf16 [T][d_model], not aliased.
 * The descriptor is checked against the smallest pool. */
mb_status mb_stack_step(mb_stack *stack, mb_kv *const *kvs, const mb_batch *batch, const void *x_in,
                        void *x_out, void *stream);
int32_t mb_stack_last_launches(const mb_stack *stack);
mb_status mb_stack_destroy(mb_stack *stack);

/* Check a batch descriptor against the rules above, on the host only (no
 * device work; usable without a GPU).  num_pages: pool size; max_tokens: the
 * layer's limit on T.  Errors: MB_EINVAL with a message naming the first
 * violated rule. */
mb_status mb_batch_validate(const mb_batch *batch, int32_t num_pages, int32_t max_tokens);

/* Synchronise `stream` and report any error word the kernels recorded since
 * the last call (then clears it).  MB_EDEVICE if one was set.  layer: that
 * layer's steps; NULL: the standalone calls on the current device (mb_gemm,
 * mb_sample_greedy, mb_embed and mb_gemm_noalloc).  With NULL it allocates
 * nothing, so callers of mb_gemm_noalloc can use it too. */
mb_status mb_device_status(mb_layer *layer, void *stream);

/* Device pointer and byte size of an intermediate of the last step, for
 * inspection: valid once the step's stream has completed and until the next
 * mb_step.  which: 0 xn, 1 qkv, 2 q (rotated, [T][Hq][hd]), 3 o, 4 h, 5 hn,
 * 6 a.  Errors: MB_EINVAL. */
mb_status mb_layer_buffer(const mb_layer *layer, int32_t which, void **ptr, int64_t *bytes);

/* Per-kernel timing of subsequent steps (CUDA events on the step's stream).
 * mb_layer_timing returns the accumulated milliseconds of each launch kind
 * since enable, in the order: rmsnorm_attn, gemm_qkv, rope_append,
 * attention (prefill-chunk tiles and decode rows, one grid), attn_merge,
 * gemm_o, rmsnorm_ffn, gemm_gate_up, gemm_down (n <= 9), and the number of
 * steps timed.  It synchronises on the
 * recorded events. */
mb_status mb_layer_set_timing(mb_layer *layer, int32_t enable);
/* SM partition for decode attention: the attention launch runs at most n
 * persistent decode-worker CTAs (one per SM), the prefill-chunk tiles and
 * the rest of the GPU around them; 0 (the default) allows one per SM, so
 * workers fill every SM the chunk tiles leave (ConfluxServe gives decode "just
 * enough SMs" for most of its bandwidth; this is the knob that measures it).
 * Takes effect at the next step (stacks re-capture their graphs).  Errors:
 * MB_EINVAL for n < 0. */
mb_status mb_layer_set_decode_sms(mb_layer *layer, int32_t n);
/* The other half of the SM partition: the layer's GEMM launches run at most
 * n CTAs (one per SM; 0, the default, allows one per SM).  With two layers
 * stepping concurrently on two streams (two micro-batches, the decode
 * attention of one beside the GEMMs of the other, as ConfluxServe overlaps
 * them), the caps of the kernels that run at the same time must add up to at
 * most the SM count: a GEMM's K-split waits on CTAs of its own grid, which
 * must all be resident.  A stack uses its first layer's setting.  Errors:
 * MB_EINVAL for n < 0. */
mb_status mb_layer_set_gemm_sms(mb_layer *layer, int32_t n);
/* The layer's GEMM workspace (fp32 partial tiles and tile tickets): device
 * memory of mb_gemm_workspace_bytes() bytes, 256-byte aligned, zero-filled,
 * owned by the caller; NULL returns to the device's shared one.  Layers that
 * step concurrently on different streams need workspaces of their own.
 * Errors: MB_EINVAL, MB_ECUDA, MB_EUNSUPPORTED. */
mb_status mb_layer_set_gemm_workspace(mb_layer *layer, void *workspace);
mb_status mb_layer_timing(mb_layer *layer, double *ms, int32_t n, int64_t *steps);

/* Number of kernel launches the last mb_step issued, and the bytes it copied
 * host to device (the descriptor and its work lists; for a stack, whose one
 * upload per step goes through its first layer, the last mb_stack_step's). */
int32_t mb_layer_last_launches(const mb_layer *layer);
int64_t mb_layer_last_upload_bytes(const mb_layer *layer);

/* Standalone token-batched GEMM D = A B^T on the tcgen05 tensor cores (the
 * linear layers of the step; ConfluxServe summary, "Why can linear layers be
 * batched"). A device bf16 [M][K], B device bf16 [N][K], both row-major with
 * K % 64 == 0 and 16-byte aligned rows.  epilogue:
 *   0  D[M][N] = A B^T                          (bf16)
 *   1  D[M][N] = A B^T + R[M][N]                (bf16 residual R, may not alias D)
 *   2  N = 2F, B rows = [gate F; up F], F % 128 == 0:
 *      D[M][F] = silu(A Bg^T) * (A Bu^T)        (bf16)
 * Accumulation is fp32.  workspace: device memory of mb_gemm_workspace_bytes()
 * bytes (fp32 partial tiles and tile tickets), or NULL to use the library's
 * own (allocated once per device on first use).  Errors: MB_EINVAL,
 * MB_EUNSUPPORTED, MB_ECUDA. */
mb_status mb_gemm(const void *A, const void *B, void *D, const void *R, int32_t M, int32_t N,
                  int32_t K, int32_t epilogue, void *workspace, void *stream);
int64_t mb_gemm_workspace_bytes(void);

/* The GEMM's bounded wait in a K-split tile, for failure-path tests: the CTA
 * holding the tile's first piece waits for the other pieces, at most
 * limit_ns (<= 0: the default, 2 s).  phantom_pieces > 0 makes it also wait
 * for that many pieces that no CTA writes, so the wait runs out every time
 * (0, the default, for normal use).  When the limit runs out the kernel
 * records an error and unwinds instead of waiting on; mb_device_status
 * reports it as MB_EDEVICE and resets the tile tickets, and the next call
 * computes normally.  Applies to GEMM launches issued after the call,
 * process-wide (a stack's CUDA graph keeps what it was captured with).
 * Errors: MB_EINVAL for phantom_pieces outside [0, 1024]. */
mb_status mb_gemm_set_split_wait(int64_t limit_ns, int32_t phantom_pieces);

/* The same GEMM for callers that cannot allocate device memory (code inside
 * an allocator's own hooks or out-of-memory path, processes whose device
 * memory is all handed out in advance, plugins limited to the buffers their
 * host passes in).  The pages have no counterpart: this is a deployment
 * convenience, not part of the method.  Arguments, layouts and epilogues are
 * those of mb_gemm; there is no workspace argument.  It calls no cudaMalloc,
 * cudaFree or allocating library routine: its scratch (stream-K partial
 * tiles, tile tickets, error word) is a file-scope device array of
 * 16 MiB + 4 KiB that every GPU loading the library holds until exit.  The
 * first call on a device looks the array's address up (once per device, with
 * that device current); make that first call before any stream capture.
 * Every call shares the array and clears its tickets on `stream` first, so
 * calls that overlap on the GPU (unordered streams) race.  Shapes whose split
 * would need more scratch than the array holds are rejected with
 * MB_EUNSUPPORTED and a message giving both sizes.  Errors: as mb_gemm for
 * the arguments (sm_103 only); a device-side error (a bounded wait that gave
 * up) stays in the array until mb_device_status(NULL, stream) reports it as
 * MB_EDEVICE, clearing it and the tickets, without allocating. */
mb_status mb_gemm_noalloc(const void *A, const void *B, void *D, const void *R, int32_t M, int32_t N,
                          int32_t K, int32_t epilogue, void *stream);

/* ---------------- scheduler side (host only, no device work) ---------------
 * The token-budget packer of the pofe.ai "Chunked prefill" page, "How it works,
 * step by step" (steps 1-3) and its schedule() sketch: every step takes one
 * token per running decode, then continues partial prefills min(C_left,
 * p - p_done), then admits waiting prompts in arrival order while budget,
 * sequence slots and KV pages remain, each with as many tokens as fit.
 * Readings where the pages differ or are silent: decodes never drive the
 * budget below zero (llm-stack-book 7.8 scheduler, budget >= 1); chunk_cap > 0
 * caps every prefill chunk (pofe.ai, head-of-line blocking); admission stops
 * at the first prompt refused for sequence slots or pages; pages are handed
 * out FIFO from free_order at pack time, exactly ceil(kv_len / 16) per
 * request; a decode that needs a page when none is free is skipped this
 * step; a partial chunk shrinks to what its pages plus free pages hold;
 * finishing a request appends its pages to the free list in table order. */
typedef struct {
  int32_t budget;     /* token budget C per step, >= 1 */
  int32_t max_seqs;   /* running + partially prefilled requests, >= 1 */
  int32_t chunk_cap;  /* per-request prefill chunk cap, 0 = none */
} mb_pack_cfg;

typedef struct {
  mb_batch batch;          /* host arrays owned by the scheduler */
  const int64_t *req_ids;  /* request id of each row */
} mb_sched_batch;

typedef struct mb_sched mb_sched;

/* free_order: host int32[num_pages], a permutation of 0..num_pages-1 giving
 * the initial free-list order (copied). */
mb_status mb_sched_create(const mb_pack_cfg *cfg, int32_t num_pages, const int32_t *free_order,
                          mb_sched **out);
/* Add a request.  computed = tokens already in the cache: 0 for a new
 * prompt, 0 < computed < prompt_len for a partial prefill, computed >=
 * prompt_len for a running decode.  Pages for `computed` tokens are taken at
 * once.  Errors: MB_EINVAL (duplicate id, bad lengths), MB_ENOSPACE. */
mb_status mb_sched_add(mb_sched *s, int64_t req_id, int32_t prompt_len, int32_t computed);
/* Build the next step's batch and advance the state as if it ran.  The
 * output arrays stay valid until the next mb_sched_* call on `s`. */
mb_status mb_sched_pack(mb_sched *s, mb_sched_batch *out);
/* Remove a request and return its pages.  Errors: MB_EINVAL (unknown id). */
mb_status mb_sched_finish(mb_sched *s, int64_t req_id);
/* Next tokens of a pass, greedy (pofe.ai "Chunked prefill", "How it works,
 * step by step", step 5: every decode row, and the last row of a prompt
 * whose last chunk ran in the pass, samples a token in that same pass; the
 * pages leave the sampling rule open, this is the greedy one):
 *   y_i      = RMSNorm(x[rows[i]]) * g_final                    (eps)
 *   logits_i = y_i W_lm^T                    bf16, fp32 accumulation
 *   ids[i]   = argmax_j logits_i[j], the lowest j among equal maxima
 * x: device bf16 [T][d] (the last layer's output); rows: device int32
 * [n_rows], each in [0, T); g_final: device bf16 [d]; w_lm: device bf16
 * [vocab][d]; y_work: device bf16 [n_rows][d] and logits: device bf16
 * [n_rows][vocab], caller-owned workspaces (logits holds the row logits
 * afterwards); ids: device int32 [n_rows].  d % 64 == 0, d <= 8192, vocab %
 * 32 == 0, pointers 16-byte aligned.  Asynchronous on `stream`; a row id out
 * of range records MB_EDEVICE (mb_device_status with layer NULL). */
mb_status mb_sample_greedy(const void *x, int32_t T, const int32_t *rows, int32_t n_rows, int32_t d, float eps,
                           const void *g_final, const void *w_lm, int32_t vocab, void *y_work, void *logits,
                           int32_t *ids, void *stream);
/* Token embeddings for the next pass: out[i] = table[ids[i]] (device bf16
 * [vocab][d] -> [n][d]; ids device int32 [n]).  An id out of range records
 * MB_EDEVICE and gives a zero row.  d % 8 == 0. */
mb_status mb_embed(const void *table, int32_t vocab, int32_t d, const int32_t *ids, int32_t n, void *out,
                   void *stream);

/* Adaptive chunk size (llm-stack-book 7.8, "Priority and Preemption Policies",
 * adaptive_chunk_size, and its exercise 4, which applies it in schedule()):
 * from the next mb_sched_pack on, every prefill chunk of a step is capped at
 *   max_chunk                                    with no running decode,
 *   min_chunk                                    with >= decode_pressure,
 *   trunc(base - (d / pressure) (base - min))    with d running decodes between,
 * clamped to [min_chunk, base_chunk], and at chunk_cap too if that is set
 * (the fixed per-request cap against head-of-line blocking, pofe.ai "Failure
 * modes and how to spot them").  The ratio is computed in double precision.
 * min_chunk = 0 turns it off.  Errors: MB_EINVAL unless 1 <= min <= base <=
 * max and decode_pressure >= 1. */
mb_status mb_sched_set_adaptive(mb_sched *s, int32_t min_chunk, int32_t base_chunk, int32_t max_chunk,
                                int32_t decode_pressure);
/* Counts: free pages, running, partial, waiting. */
mb_status mb_sched_counts(const mb_sched *s, int32_t counts[4]);
mb_status mb_sched_destroy(mb_sched *s);

/* Checkpoint and resume of the packer.  Chunked prefill adds one piece of
 * state per request: how many of its prompt tokens are already in the KV
 * cache (pofe.ai "Chunked prefill", "How it works, step by step"; the
 * num_computed field of the minimal scheduler in llm-stack-book 7.8, "A
 * Minimal End-to-End Chunked Prefill Scheduler").  With each request's block
 * table and the order of the queues and of the free list, that is all the
 * later batches depend on.
 *
 * mb_sched_save writes the state of `s` as int64 words into `buf` (host,
 * caller-owned, `cap` words) and sets *len to the number of words it needs;
 * with buf == NULL and cap == 0 it only sets *len.  Layout (version 1):
 *   0x4D4253434844 (magic), 1 (version), budget, max_seqs, chunk_cap,
 *   num_pages, adaptive min, base, max and pressure (all 0 when off),
 *   n_free, the free pages in hand-out order; then the running, partially
 *   prefilled and waiting queues in turn: the queue's length and, per
 *   request in queue order, id, prompt_len, computed, n_pages and its pages
 *   in block-table order.
 * The output arrays of the last mb_sched_pack are not part of the state.
 * Errors: MB_EINVAL (null argument), MB_ENOSPACE (cap < *len; nothing written).
 *
 * mb_sched_load builds a new scheduler in *out (free it with
 * mb_sched_destroy) from such words; it packs the same batches as the saved
 * one would from the same calls on.  The state is checked whole: magic and
 * version, a valid configuration, every page id in [0, num_pages) exactly
 * once over the free list and the block tables, unique request ids, each
 * request holding ceil(computed / 16) pages in the queue its progress implies
 * (waiting: computed 0; partial: 0 < computed < prompt_len; running: computed
 * >= prompt_len), and no words left over.  Errors: MB_EINVAL (a check fails;
 * nothing is built), MB_ENOMEM. */
mb_status mb_sched_save(const mb_sched *s, int64_t *buf, int64_t cap, int64_t *len);
mb_status mb_sched_load(const int64_t *buf, int64_t len, mb_sched **out);

const char *mb_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MB_H_ */
