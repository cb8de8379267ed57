// gva_internal.h -- host-side structures shared by the GVA translation units (not part of
// the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gva.h"

struct gva_ctx {
  gva_dims dims;
  float scale;          // resolved softmax scale
  double rope_base;     // resolved RoPE base
  int device;           // device the context was created on
  int num_sms;          // SM count of that device
  unsigned* d_err;      // device error word
  double2* d_rope;      // RoPE digit table [4][256][d_r/2] in fp64 (nullptr when d_r == 0)
  float2* d_rope32;     // the same table rounded to fp32
  int split_tokens;     // 0 = automatic
  gva_decode_path path;
  gva_step_mode step_mode;
};

namespace gva {

constexpr int kMaxDevicesHost = 64;  // per-device host caches (function attributes, addresses)

// Arguments of the decode partial kernels (GVA and the matching GQA form).
struct DecodeArgs {
  const float* q_abs;        // [B,H,d_v] absorbed query (GQA: the plain query)
  const float* q_rot;        // [B,H,d_r] rotated positional query (nullptr when d_r == 0)
  const void* v_pool;        // [NB][G][64][d_v] (fp8 cache: the E4M3 codes)
  const signed char* v_exp;  // fp8 cache: the scale exponents [NB][G][64], after the codes
  const void* k_pool;        // GQA only: [NB][G][64][d_v]
  const void* kr_pool;       // [NB][64][d_r]
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* out;                // [B,H,d_v]
  float* part;               // workspace: header (prefix sums) + partial records
  unsigned* err;
  int B, H, G, d_v, d_r;
  // Query tokens per sequence (the last nq positions; 1 for plain decode).  A pass of the
  // tensor-core kernel handles queries [q0, q0 + nqp): queries are rows (b*nq + q)*H + h of
  // q_abs / q_rot / out, and a partial record holds R*nqp (query, head) sub-records.
  int nq, q0, nqp;
  int max_blocks, num_blocks, max_seq_len;
  int n_warps;               // warps of the partial grid that stream units
  // The batch's units are cut into n_groups equal contiguous ranges; the group_warps warps
  // of a range share it round-robin (unit k of the range goes to warp k % group_warps).
  // Warp w of range c writes its partial record of segment f at index (c + f)*group_warps + w.
  int n_groups, group_warps;
  int n_stages;              // tensor-core kernel: ring depth of each warp pair (tiles)
  float scale_log2;          // softmax scale * log2(e)
  // Fused decode step (tensor-core kernel, one query per sequence, d_n == d_v): the partial
  // kernel absorbs and rotates the queries itself and appends the new token of every
  // sequence, at position seq_lens[b] - 1, to the cache.  q_abs and q_rot are then unused.
  int fused;
  const float* q_c;          // [B,H,d_n] content query
  const float* q_r;          // [B,H,d_r] positional query, unrotated
  const float* M;            // [H,d_v,d_n] key maps
  const void* v_new;         // [B,G,d_v] new values (bf16)
  const void* kr_new;        // [B,d_r] new positional keys, unrotated (bf16)
  void* v_pool_w;            // v_pool and kr_pool again, written at the new token's slot
  signed char* v_exp_w;      // (fp8 cache: and the exponents)
  void* kr_pool_w;
  const float2* rope32;      // fp32 RoPE digit table
  // Per (range c, segment f) at index c + f: step_stage_floats(R, d_v, d_r) floats holding
  // the R absorbed queries [d_v] each followed by its rotated positional query [d_r], then the
  // new token's rotated positional key as d_r/2 packed bf16 pairs.  A CTA keeps its stages in
  // the shared memory the ring leaves over (spare_smem bytes) when they fit, here otherwise.
  float* qstage;
  int spare_smem;
  // Combine pass launched right after this call's partial pass (its programmatic dependent):
  // every write that preceded the partial pass, the lengths included, is complete when the
  // combine starts, so it may form its prefix sums from seq_lens before its own wait instead of
  // reading the header after it (set for batches of up to 256 sequences: each combine CTA
  // reads all B lengths).
  int combine_after_partial;
  // combine: one CTA per (group, sequence) fits on the SMs at once, so each may stage its
  // records in the large rounds (kBigStageBytes) instead of the small ones
  int combine_big;
};

// Floats of one fused-step query stage (a multiple of 4, so every stage is 16-byte aligned).
__host__ __device__ constexpr int step_stage_floats(int R, int d_v, int d_r) {
  return (R * (d_v + d_r) + d_r / 2 + 3) / 4 * 4;
}

// Record layout of one partial: m (log2 domain), l, two pad words, then d_v weighted sums.
__host__ __device__ inline size_t partial_stride_floats(int d_v) { return static_cast<size_t>(d_v) + 4; }

constexpr int kMaxBatch = 8192;  // sequences per decode call (prefix sums live in shared memory)

struct Plan {
  int path;         // GVA_PATH_FMA or GVA_PATH_MMA
  int nqp;          // queries per pass (records hold R*nqp sub-records)
  int grid;         // CTAs of the partial kernel
  int n_warps;      // warps that stream units (grid * unit warps per CTA)
  int n_groups;     // unit ranges (FMA: one per warp; MMA: one per CTA)
  int group_warps;  // warps sharing one range
  int n_stages;     // MMA ring depth per warp pair
  size_t ws_bytes;
};

// Launchers (return cudaSuccess or the launch error).
// With pos_q (pos) null, the positions come from the lengths: the n new tokens of sequence b
// are its last n positions, seq_lens[b] - n + t, and query row b*n + i (rows_per_seq = n)
// sits at seq_lens[b] - n + i (one decode step, or a step of n tokens).  after_own_append:
// the absorb is launched right after launch_append of the same step, on the same stream, and
// overlaps it (its inputs are not the append's outputs).
cudaError_t launch_absorb(const gva_ctx* ctx, int B, const float* q_c, const float* q_r,
                          const int32_t* pos_q, const float* M, float* q_abs, float* q_rot,
                          cudaStream_t stream, const int32_t* seq_lens = nullptr,
                          bool after_own_append = false, int rows_per_seq = 1);
cudaError_t launch_append(const gva_ctx* ctx, int B, int n, const void* v_new,
                          const void* kr_new, const int32_t* pos, const int32_t* block_table,
                          int max_blocks, int num_blocks, void* v_pool, void* kr_pool,
                          cudaStream_t stream, const int32_t* seq_lens = nullptr);
// Decode: partial kernel + combine.  sep_k selects the GQA form (k_pool used, d_r == 0).
// Partial kernels: one CTA = 4 warps, each warp a balanced range of (b, g, tile) units.
bool fma_supported(const gva_dims& d, bool sep_k);
int fma_ctas_per_sm(const gva_dims& d, bool sep_k, int B);
cudaError_t launch_decode_fma(const DecodeArgs& a, int cache_dtype, bool sep_k, int grid,
                              cudaStream_t stream);
bool mma_supported(const gva_dims& d, bool sep_k);
// Tensor-core kernel: one CTA per range, made of P warp pairs (a copy warp filling a private
// ring of D tiles, and the consumer warp that computes on it); P consumer warps share the
// range.  mma_shape picks P and D for the dims (0 if no ring fits).
constexpr int kMmaMaxPairs = 6;
bool mma_shape(const gva_dims& d, bool sep_k, int B, int nqp, int* pairs, int* stages);
// Queries per pass of the tensor-core kernel (its (query, head) column pairs: R*nqp <= 16 at
// d_v = 64, 8 at d_v = 128; at most 4).
int mma_max_queries_per_pass(int R, int d_v);
cudaError_t launch_decode_mma(const DecodeArgs& a, bool sep_k, int grid, cudaStream_t stream);
// The same kernel over the fp8 value cache (single query per sequence, plain or fused step).
cudaError_t launch_decode_mma_fp8(const DecodeArgs& a, int grid, cudaStream_t stream);
// Merges the partial records of each (b, g) into out; launched as a programmatic dependent
// of the partial kernel.
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t stream);

}  // namespace gva
