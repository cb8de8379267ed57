/*
 * gva.h -- C ABI of the Grouped Value Attention (GVA) decode hot path for NVIDIA B300
 * (sm_103a).
 *
 * GVA keeps, per token and layer, only the G grouped value heads V_g and ONE small
 * positional key k_r of width d_r, stored already RoPE-rotated and shared by every query
 * head; there is no content-key cache.  Each query head h scores the cache through the
 * absorbed query q'_h = M_h q_c,h (the content key K_h = V_g(h) M_h is never built), adds
 * the decoupled positional score q~_r,h . k_r,j, and returns o_h = sum_j softmax(s)_j v_j.
 *   - "Grouped Value Attention: Efficient KV Caching via On-Demand Key Reconstruction"
 *     (abstract): grouped values, learned linear key map absorbed into the query, shared
 *     decoupled RoPE channel with a separately cached positional key.
 *   - ai-feeds.com summary "Grouped Value Attention:通过按需 key 重建实现高效 KV 缓存",
 *     section 方法: K_h = V_g(h) M_h, Q' = Q M^T, output is the value-weighted sum.
 *   - review "[논문리뷰] Grouped Value Attention ...", section 3, Decoupled RoPE: query and
 *     key split into an unrotated content slice (d_n) and a rotated positional slice (d_r);
 *     RoPE on the positional slice only; positional key shared across heads.
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless a parameter says otherwise; they must be
 *     16-byte aligned.  All tensors are dense, row-major, in the shapes given.
 *   - The caller owns every buffer (inputs, outputs, cache pools, block table, workspace).
 *     The library allocates device memory only in gva_create (its error word and RoPE
 *     table) and frees it in gva_destroy; nothing is allocated on the decode path.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).  GVA_OK means
 *     the work was enqueued.  Host-side argument errors return a status and enqueue
 *     nothing.  Index errors that only the device can see (a position past the block
 *     table, a block id outside the pool, a bad context length) make the kernel skip that
 *     access and set a bit in the context's device error word; gva_get_device_error
 *     reads it.  No kernel traps.
 *   - Cache layout, 64-token blocks (GVA_BLOCK_TOKENS), NB blocks in a pool:
 *       V pool   [NB][G][64][d_v]   element (blk, g, o, i) at ((blk*G + g)*64 + o)*d_v + i
 *       k_r pool [NB][64][d_r]      element (blk, o, c)    at (blk*64 + o)*d_r + c
 *     Position p of sequence b lives in block block_table[b*max_blocks + p/64], slot p%64.
 *     The fp8 value cache (GVA_FP8_E4M3) stores in the V pool NB*G*64*d_v one-byte E4M3 codes
 *     in the layout above, followed by NB*G*64 int8 scale exponents, exponent (blk, g, o) at
 *     byte NB*G*64*d_v + (blk*G + g)*64 + o: value = code * 2^exponent.  Its k_r pool is bf16.
 *   - Head h reads value group g(h) = h / (H/G) (contiguous head blocks, as in grouped-
 *     query attention).  RoPE turns pair (2i, 2i+1) by p * base^(-2i/d_r).  The softmax
 *     scale defaults to 1/sqrt(d_n + d_r).
 */
#ifndef GVA_H_
#define GVA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GVA_BLOCK_TOKENS 64

/* Same type as cudaStream_t, so callers need no CUDA header. */
typedef struct CUstream_st* gva_stream_t;

typedef enum {
  GVA_OK = 0,
  GVA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent shape */
  GVA_ERR_UNSUPPORTED = 2,  /* valid, but a shape or dtype no kernel here was built for */
  GVA_ERR_WORKSPACE = 3,    /* workspace null or smaller than gva_decode_workspace_size() */
  GVA_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, attribute, copy) */
  GVA_ERR_DEVICE_INDEX = 5  /* gva_get_device_error found a device-side error bit set */
} gva_status;

/* Cache dtypes.  GVA_FP8_E4M3 is a low-precision value cache of this library (the paper
 * stores values in the model's precision): each (token, group) value row is kept as E4M3
 * codes (OCP FP8: 4 exponent bits with bias 7, 3 mantissa bits, largest finite 448) times
 * one power-of-two scale 2^e, e the smallest integer with max|v| <= 448 * 2^e (clamped to
 * [-126, 120]); each code is v * 2^-e rounded to nearest even, saturating at 448.  The
 * positional keys stay bf16; new values and keys are given in bf16.  G*d_v + G + 2*d_r
 * bytes per token (292 at G = 4, d_v = 64, d_r = 16, against 544 for bf16).  Tensor-core
 * path only: d_v 64 or 128, one query per sequence (gva_decode_attention, _partial,
 * _combine, _noalloc, gva_decode_step and its parts), no gqa_decode_attention. */
typedef enum { GVA_F32 = 0, GVA_BF16 = 1, GVA_FP8_E4M3 = 2 } gva_dtype;

/* Bits of the device error word. */
#define GVA_DEVERR_POSITION 1u /* position < 0, or position/64 >= max_blocks */
#define GVA_DEVERR_BLOCK_ID 2u /* block-table entry outside [0, num_blocks) */
#define GVA_DEVERR_SEQ_LEN 4u  /* seq_lens[b] <= 0 or > max_seq_len (that row's output is 0) */
#define GVA_DEVERR_TIMEOUT 8u  /* a bounded wait for an async copy gave up (tile skipped) */

/* Decode kernel family for gva_set_decode_path. */
typedef enum {
  GVA_PATH_AUTO = 0, /* tensor-core path where it applies, else the CUDA-core path */
  GVA_PATH_FMA = 1,  /* CUDA-core fp32 FMA path (every dtype) */
  GVA_PATH_MMA = 2   /* tensor-core path (bf16 cache only; GVA_ERR_UNSUPPORTED otherwise) */
} gva_decode_path;

typedef struct {
  int H;                 /* query heads */
  int G;                 /* value heads (groups); H % G == 0 */
  int d_v;               /* value width; multiple of 32 */
  int d_n;               /* content query width (absorbed query input); multiple of 4 */
  int d_r;               /* positional width; even, 0 <= d_r <= 32 (0 = no positional slice) */
  int block_size;        /* tokens per cache block; must be 64 */
  gva_dtype cache_dtype; /* GVA_F32, GVA_BF16 or GVA_FP8_E4M3 */
  double rope_base;      /* <= 0 selects 10000 */
  float scale;           /* softmax scale; <= 0 selects 1/sqrt(d_n + d_r) */
} gva_dims;

typedef struct gva_ctx gva_ctx;

/* Validates dims and creates a context bound to the CURRENT device: it holds the dims, the
 * decode options, a device error word and the RoPE digit tables (cos and sin of every 8-bit
 * digit of a position times each pair's frequency, computed in fp64 on the host, kept in fp64 and fp32; 12*d_r KB
 * of cudaMalloc in all).  Returns
 * GVA_ERR_INVALID_ARG / GVA_ERR_UNSUPPORTED for bad dims, GVA_ERR_CUDA if the allocation
 * fails.  *out is set only on success. */
gva_status gva_create(const gva_dims* dims, gva_ctx** out);

/* Frees the context (synchronises nothing; call after the context's work has finished). */
void gva_destroy(gva_ctx* ctx);

/* gva_absorb_query -- per-step query preparation.
 * Folds the key map into the query, q'_{b,h} = M_h q_c,{b,h} (column form of Q' = Q M^T,
 * ai-feeds.com summary section 方法; m.szthrk.cn explainer section "GVA 的正式方案"), and
 * rotates the positional query q~_r,{b,h} = RoPE(q_r,{b,h}, pos_q[b]) (review section 3,
 * Decoupled RoPE).
 *   q_c   [B,H,d_n] f32      content query
 *   q_r   [B,H,d_r] f32      positional query, unrotated (may be NULL when d_r == 0)
 *   pos_q [B] int32          query position (normally seq_len - 1)
 *   M     [H,d_v,d_n] f32    key maps, M[h][i][k]
 *   q_abs [B,H,d_v] f32 out  absorbed query (no scale folded in)
 *   q_rot [B,H,d_r] f32 out  rotated positional query (may be NULL when d_r == 0)
 * fp32 accumulation.  The rotation for position p is the product of the table rotations of
 * p's four bytes, composed in fp32 (relative error a few units of 2^-24).  B == 0 is a
 * no-op. */
gva_status gva_absorb_query(gva_ctx* ctx, int B, const float* q_c, const float* q_r,
                            const int32_t* pos_q, const float* M, float* q_abs, float* q_rot,
                            gva_stream_t stream);

/* gva_cache_append -- write n new tokens per sequence into the compact cache (the
 * "append the new token's state, then read through the current position" step of the
 * decode lifecycle, GQA explainer section "与位置编码和 KV Cache 的关系"; cache content per
 * the abstract and the review's section 3: grouped values plus one rotated positional key).
 *   v_new  [B,n,G,d_v] cache dtype   new values, copied bit for bit (fp8 cache: bf16
 *                                    values, quantised row by row as GVA_FP8_E4M3 states)
 *   kr_new [B,n,d_r]   cache dtype   new positional keys, UNROTATED; each is rotated to its
 *                                    own position (fp64 for fp32 caches, fp32 for bf16 and
 *                                    fp8 caches) and rounded once to nearest even (fp8
 *                                    cache: bf16 keys)
 *   pos    [B] int32                 position of the first new token of each sequence
 *   block_table [B,max_blocks] int32, pools as in the layout above (NB = num_blocks)
 * Token t of sequence b goes to position pos[b]+t.  A position beyond the table or a block
 * id outside [0,num_blocks) skips that token and sets a device error bit.  seq_lens is not
 * touched (the caller advances it), so a call can be repeated.  n == 0 or B == 0 is a
 * no-op. */
gva_status gva_cache_append(gva_ctx* ctx, int B, int n, const void* v_new, const void* kr_new,
                            const int32_t* pos, const int32_t* block_table, int max_blocks,
                            int num_blocks, void* v_pool, void* kr_pool, gva_stream_t stream);

/* Bytes of workspace gva_decode_attention needs for this batch (partial softmax states of
 * the split-T plan).  max_seq_len is the host's upper bound on seq_lens.  Depends on the
 * context's split option, so query it after gva_set_split_tokens. */
size_t gva_decode_workspace_size(const gva_ctx* ctx, int B, int max_seq_len);

/* gva_decode_attention -- decode attention over the compact cache.
 * For each b and head h with g = g(h) and T = seq_lens[b]:
 *   s_j = scale * (q_abs[b,h,:] . V[g] at position j  +  q_rot[b,h,:] . k_r at position j)
 *   out[b,h,:] = sum_{j<T} softmax(s)_j  V[g] at position j
 * (summary section 方法: content score as one inner product with the stored value, output
 * the value-weighted sum; review section 3: positional score from the shared rotated key.)
 * Split-T flash decoding: the batch's (sequence, value group, 64-token block) units are
 * shared out evenly over the warps of one wave of CTAs; each warp yields a partial (max,
 * sum, weighted sum) per (sequence, group) it covers, in the workspace, and a combine pass
 * merges them.  B <= 8192.
 *   q_abs [B,H,d_v] f32, q_rot [B,H,d_r] f32 (NULL when d_r == 0)
 *   seq_lens [B] int32 (device), each in [1, max_seq_len]
 *   out [B,H,d_v] f32
 *   workspace: device scratch of at least gva_decode_workspace_size(ctx, B, max_seq_len)
 *   bytes, 16-byte aligned; its contents are not needed between calls.
 * fp32 accumulation for every cache dtype. */
gva_status gva_decode_attention(gva_ctx* ctx, int B, const float* q_abs, const float* q_rot,
                                const void* v_pool, const void* kr_pool,
                                const int32_t* block_table, int max_blocks, int num_blocks,
                                const int32_t* seq_lens, int max_seq_len, float* out,
                                void* workspace, size_t ws_bytes, gva_stream_t stream);

/* The two passes of gva_decode_attention as separate calls, for callers that schedule them
 * apart (or time them apart).  gva_decode_attention(...) is exactly gva_decode_partial
 * followed by gva_decode_combine on the same stream.
 *   gva_decode_partial: the split-T pass (the split-T flash-decoding kernel);
 *     arguments as gva_decode_attention without `out`.  Its results (partial maxima, sums
 *     and weighted value sums, plus the batch's tile prefix sums) stay in the workspace.
 *   gva_decode_combine: merges them into out [B,H,d_v] f32.  It must follow the partial pass
 *     of the same context, B, max_seq_len and workspace on the same stream, with no change
 *     to the context's decode options in between (both passes derive the same split plan
 *     from them); the workspace is read, not written. */
gva_status gva_decode_partial(gva_ctx* ctx, int B, const float* q_abs, const float* q_rot,
                              const void* v_pool, const void* kr_pool,
                              const int32_t* block_table, int max_blocks, int num_blocks,
                              const int32_t* seq_lens, int max_seq_len, void* workspace,
                              size_t ws_bytes, gva_stream_t stream);
gva_status gva_decode_combine(gva_ctx* ctx, int B, int max_seq_len, float* out, void* workspace,
                              size_t ws_bytes, gva_stream_t stream);

/* gva_decode_attention_multi -- decode attention for n_q query tokens per sequence, the last
 * n_q positions of its context (tokens just appended, e.g. drafts to verify in speculative
 * decoding).  Query i of sequence b sits at position p = seq_lens[b] - n_q + i and reads the
 * cache up to and including its own position (the decode lifecycle of the GQA explainer,
 * section "与位置编码和 KV Cache 的关系": a query reads the cache through the current position),
 * with the same scores and softmax as gva_decode_attention:
 *   q_abs [B,n_q,H,d_v] f32 and q_rot [B,n_q,H,d_r] f32 (gva_absorb_query over B*n_q rows,
 *   pos_q = p), out [B,n_q,H,d_v] f32; seq_lens[b] in [n_q, max_seq_len] (a shorter length
 *   sets GVA_DEVERR_SEQ_LEN and zeroes that sequence's rows).
 * Tensor-core path only (bf16 caches; GVA_ERR_UNSUPPORTED otherwise when n_q > 1).  The
 * kernel packs R*nqp (query, head) pairs into its MMA columns, nqp = up to 4 queries per
 * pass with R*nqp <= 16 (R = H/G); more queries take more passes, each reading the cache.
 * n_q == 1 is gva_decode_attention.  Workspace: gva_decode_workspace_size_multi bytes. */
gva_status gva_decode_attention_multi(gva_ctx* ctx, int B, int n_q, const float* q_abs,
                                      const float* q_rot, const void* v_pool, const void* kr_pool,
                                      const int32_t* block_table, int max_blocks, int num_blocks,
                                      const int32_t* seq_lens, int max_seq_len, float* out,
                                      void* workspace, size_t ws_bytes, gva_stream_t stream);
size_t gva_decode_workspace_size_multi(const gva_ctx* ctx, int B, int n_q, int max_seq_len);

/* Step mode for gva_set_step_mode. */
typedef enum {
  GVA_STEP_AUTO = 0,     /* fused where it applies, the key maps of a group are small
                            (R*d_v*d_n*4 <= 64 KB) and the batch has at most 8 (group,
                            sequence) segments per unit range; else the separate kernels */
  GVA_STEP_FUSED = 1,    /* fused kernel (GVA_ERR_UNSUPPORTED where it does not apply) */
  GVA_STEP_SEPARATE = 2  /* append, absorb and decode as separate kernels */
} gva_step_mode;

/* gva_decode_step -- one whole decode step of a layer: append each sequence's new token,
 * absorb and rotate its query, and attend over the context including the new token.
 * Sequence b's context length T = seq_lens[b] ALREADY COUNTS the new token, which goes to
 * position p = T - 1, and its query sits at p (the decode lifecycle of the GQA explainer,
 * section "与位置编码和 KV Cache 的关系": append the new token's state, then read the cache
 * through the current position).  The result equals
 *   gva_cache_append(ctx, B, 1, v_new, kr_new, pos = T - 1, ...);
 *   gva_absorb_query(ctx, B, q_c, q_r, pos_q = T - 1, M, q_abs, q_rot, ...);
 *   gva_decode_attention(ctx, B, q_abs, q_rot, ...);
 * bit for bit, and the cache holds the new token afterwards in both forms.
 *   q_c [B,H,d_n] f32, q_r [B,H,d_r] f32 (NULL when d_r == 0), M [H,d_v,d_n] f32
 *   v_new [B,G,d_v] and kr_new [B,d_r] cache dtype (kr_new unrotated; 4-byte aligned)
 *   v_pool, kr_pool, block_table, seq_lens, out: as gva_cache_append and gva_decode_attention
 *   workspace: at least gva_decode_step_workspace_size(ctx, B, max_seq_len) bytes.
 * q_c, q_r, v_new, kr_new and out may also point to page-locked host memory that the device
 * can address (cudaHostAlloc, or cudaHostRegister with the mapped flag; under unified virtual
 * addressing the host pointer itself): the kernels then read the step's inputs and write its
 * output across the bus directly, with no copy before or after the step.  Any other host
 * memory (pageable: malloc, the stack) is rejected with GVA_ERR_INVALID_ARG before anything
 * is enqueued, as it is by gva_decode_step_multi and gva_decode_step_partial.
 * The fused form (tensor-core path, d_n == d_v) is one partial kernel plus the combine: the
 * partial kernel forms the absorbed queries in its prologue (the "extra query-side compute"
 * of absorption, summary section 方法, done where the queries are used) and appends the new
 * token while it streams the sequence's last block.  The separate form is the three calls
 * above on `stream`.  gva_set_step_mode picks one; the default decides from the batch shape.
 * A sequence whose length is outside [1, max_seq_len] sets GVA_DEVERR_SEQ_LEN, gets a zero
 * output row, and its new slot's contents are unspecified. */
gva_status gva_decode_step(gva_ctx* ctx, int B, const float* q_c, const float* q_r, const float* M,
                           const void* v_new, const void* kr_new, void* v_pool, void* kr_pool,
                           const int32_t* block_table, int max_blocks, int num_blocks,
                           const int32_t* seq_lens, int max_seq_len, float* out, void* workspace,
                           size_t ws_bytes, gva_stream_t stream);
size_t gva_decode_step_workspace_size(const gva_ctx* ctx, int B, int max_seq_len);
gva_status gva_set_step_mode(gva_ctx* ctx, gva_step_mode mode);

/* gva_decode_step_multi -- a decode step of n_q tokens per sequence (drafts to verify in
 * speculative decoding): the n_q new tokens go to the last n_q positions of each context,
 * seq_lens[b] - n_q + i (the lengths already count them), their queries are absorbed and
 * rotated at the same positions, and query i reads the cache through its own position (the
 * decode lifecycle of the GQA explainer, section "与位置编码和 KV Cache 的关系").  Equals
 *   gva_cache_append(ctx, B, n_q, v_new, kr_new, pos = T - n_q, ...);
 *   gva_absorb_query(ctx, B*n_q, q_c, q_r, pos_q = T - n_q + i, M, q_abs, q_rot, ...);
 *   gva_decode_attention_multi(ctx, B, n_q, q_abs, q_rot, ...);
 * bit for bit.
 *   q_c [B,n_q,H,d_n] f32, q_r [B,n_q,H,d_r] f32, M [H,d_v,d_n] f32
 *   v_new [B,n_q,G,d_v] and kr_new [B,n_q,d_r] cache dtype (kr_new unrotated)
 *   out [B,n_q,H,d_v] f32; seq_lens[b] in [n_q, max_seq_len]
 *   workspace: at least gva_decode_step_workspace_size_multi(ctx, B, n_q, max_seq_len) bytes.
 * The kernels run separately (append and absorb side by side, then the multi-query decode);
 * q_c, q_r, v_new, kr_new and out may be pinned host memory as for gva_decode_step.  n_q == 1
 * is gva_decode_step (whose fused form then applies). */
gva_status gva_decode_step_multi(gva_ctx* ctx, int B, int n_q, const float* q_c, const float* q_r,
                                 const float* M, const void* v_new, const void* kr_new, void* v_pool,
                                 void* kr_pool, const int32_t* block_table, int max_blocks, int num_blocks,
                                 const int32_t* seq_lens, int max_seq_len, float* out, void* workspace,
                                 size_t ws_bytes, gva_stream_t stream);
size_t gva_decode_step_workspace_size_multi(const gva_ctx* ctx, int B, int n_q, int max_seq_len);

/* Which form gva_decode_step takes for this batch shape under the context's mode: 1 the fused
 * kernel, 0 the separate kernels, -1 none (bad arguments, or fused mode where it does not
 * apply). */
int gva_step_is_fused(const gva_ctx* ctx, int B, int max_seq_len);

/* The fused step's first pass alone (the split-T partial kernel with the absorption in its
 * prologue and the append), for callers that schedule or time the passes apart:
 * gva_decode_step in its fused form is exactly gva_decode_step_partial followed by
 * gva_decode_combine (same context, B, max_seq_len and workspace, same stream).  Arguments as
 * gva_decode_step without `out`; GVA_ERR_UNSUPPORTED where the fused form does not apply,
 * whatever the step mode. */
gva_status gva_decode_step_partial(gva_ctx* ctx, int B, const float* q_c, const float* q_r, const float* M,
                                   const void* v_new, const void* kr_new, void* v_pool, void* kr_pool,
                                   const int32_t* block_table, int max_blocks, int num_blocks,
                                   const int32_t* seq_lens, int max_seq_len, void* workspace, size_t ws_bytes,
                                   gva_stream_t stream);

/* gqa_decode_attention -- the matching grouped-query attention decode, built with the same
 * tiling and pools so that the cost of a key cache can be timed beside GVA (GQA explainer,
 * section "一次 GQA 计算如何展开": grouped keys and values, head h reads group g(h)).
 * Uses the context's H, G, d_v (= head width d), cache dtype and scale; the context must
 * have d_r == 0 (so the default scale is 1/sqrt(d_n)).
 *   q [B,H,d] f32 (already rotated), k_pool and v_pool [NB][G][64][d] cache dtype.
 * Workspace as for gva_decode_attention. */
gva_status gqa_decode_attention(gva_ctx* ctx, int B, const float* q, const void* k_pool,
                                const void* v_pool, const int32_t* block_table, int max_blocks,
                                int num_blocks, const int32_t* seq_lens, int max_seq_len,
                                float* out, void* workspace, size_t ws_bytes,
                                gva_stream_t stream);

/* Decode options.  split_tokens: about how many context tokens each warp of the split-T
 * partial kernel covers when every sequence is at max_seq_len, a multiple of 64 (0 =
 * automatic: one wave of CTAs over the GPU, every warp an equal share of the batch's tiles).
 * path: kernel family. */
gva_status gva_set_split_tokens(gva_ctx* ctx, int split_tokens);
gva_status gva_set_decode_path(gva_ctx* ctx, gva_decode_path path);

/* The split the next decode call uses for this batch shape: *split_tokens = context tokens
 * per warp when every sequence is at max_seq_len, *max_splits = warps of the partial kernel
 * (each writes one partial record per (sequence, group) its range touches). */
gva_status gva_decode_plan(const gva_ctx* ctx, int B, int max_seq_len, int* split_tokens,
                           int* max_splits);

/* Bytes of device scratch that gva_decode_attention_noalloc holds on every GPU that loads
 * this library (4 MiB). */
#define GVA_NOALLOC_SCRATCH_BYTES (4u << 20)

/* gva_decode_attention_noalloc -- gva_decode_attention for callers that cannot allocate
 * device memory: an operator inside a host framework that hands it only its inputs and
 * outputs, an engine that has already given all device memory to its own pools, or a
 * latency-critical loop that must not call the CUDA allocator (it may synchronise the device
 * and takes an unbounded time).  The paper has no counterpart to this call: it is a
 * convenience of this library.
 * Same arguments, computation and results as gva_decode_attention, without the workspace:
 * the scratch is a fixed GVA_NOALLOC_SCRATCH_BYTES array that is part of the library's
 * device image, so it exists on every GPU that loads the library until the process exits.
 * Nothing is allocated.
 *   - Batches whose gva_decode_workspace_size() exceeds GVA_NOALLOC_SCRATCH_BYTES are
 *     rejected with GVA_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on each device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.  The address is kept for
 *     the life of the process: after cudaDeviceReset (or anything else that destroys the
 *     device's primary context) it no longer names the array, so do not call this entry
 *     point on that device again in the same process.
 *   - Every call on a device shares the one array, and it keeps the previous call's
 *     contents.  Calls whose work can overlap on the GPU (different streams without
 *     ordering between them) race on it and give wrong results; order them on one stream. */
gva_status gva_decode_attention_noalloc(gva_ctx* ctx, int B, const float* q_abs,
                                        const float* q_rot, const void* v_pool,
                                        const void* kr_pool, const int32_t* block_table,
                                        int max_blocks, int num_blocks, const int32_t* seq_lens,
                                        int max_seq_len, float* out, gva_stream_t stream);

/* Synchronises the device, reads the device error word into *bits and clears it.
 * Returns GVA_ERR_DEVICE_INDEX if any bit was set, GVA_OK if none, GVA_ERR_CUDA if the
 * copy failed. */
gva_status gva_get_device_error(gva_ctx* ctx, unsigned* bits);

/* Static description of a status code. */
const char* gva_status_string(gva_status status);

/* Library version, major*10000 + minor*100 + patch. */
int gva_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GVA_H_ */
