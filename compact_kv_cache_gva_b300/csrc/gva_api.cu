// gva_api.cu -- the C ABI (include/gva.h): argument checks, the split-T plan and launches.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include "gva_internal.h"
#include "gva_sched.cuh"

namespace {

constexpr int kVersion = 200;  // 0.2.0
// Automatic step mode: fuse while the batch has at most this many (group, sequence) segments
// per unit range and a CTA's key maps (R*d_v*d_n fp32) are at most kStepAutoMapBytes.
// Measured on B300 (one-call step, fused against separate kernels): d_v = d_n = 64, R = 4
// (64 KB of maps) wins up to 7 segments per range (68.3 us against 73.6 us) and ties at 14;
// d_v = d_n = 128 (256 KB) loses already at 1.8 (104.8 us against 102.9 us).
constexpr long long kStepAutoSegmentsPerRange = 8;
constexpr long long kStepAutoMapBytes = 64 * 1024;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether the kernels may read or write p: device or managed memory, or page-locked host
// memory mapped into the device's address space at the same address (cudaHostAlloc, or
// cudaHostRegister with the mapped flag, under unified addressing).  Pageable host memory
// (malloc, the stack) is not: a kernel touching it would fault.  Null passes (the caller
// checks required pointers itself).
bool device_addressable(const void* p) {
  if (!p) return true;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();  // clear the error the query left behind
    return false;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

// The step's per-call inputs and output, which may be pinned host memory.
bool step_buffers_addressable(const void* q_c, const void* q_r, const void* v_new, const void* kr_new,
                              const void* out) {
  return device_addressable(q_c) && device_addressable(q_r) && device_addressable(v_new) &&
         device_addressable(kr_new) && device_addressable(out);
}

bool on_ctx_device(const gva_ctx* ctx) {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && dev == ctx->device;
}

gva_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GVA_OK : GVA_ERR_CUDA; }

// RoPE digit tables: entry (k, dgt, i) holds cos and sin of dgt * 256^k * theta_i,
// theta_i = base^(-2i/d_r), in fp64 (pairs (2i, 2i+1) turned by position * theta_i), and
// the same values rounded to fp32.
bool build_rope_table(gva_ctx* ctx) {
  const int pairs = ctx->dims.d_r / 2;
  if (pairs == 0) return true;
  const size_t n = static_cast<size_t>(4) * 256 * pairs;
  double2* host = static_cast<double2*>(malloc(n * sizeof(double2)));
  float2* host32 = static_cast<float2*>(malloc(n * sizeof(float2)));
  bool ok = host && host32;
  if (ok) {
    for (int k = 0; k < 4; ++k)
      for (int dgt = 0; dgt < 256; ++dgt)
        for (int i = 0; i < pairs; ++i) {
          const double theta = pow(ctx->rope_base, -2.0 * i / static_cast<double>(ctx->dims.d_r));
          const double a = ldexp(static_cast<double>(dgt), 8 * k) * theta;
          const size_t e = (static_cast<size_t>(k) * 256 + dgt) * pairs + i;
          host[e] = make_double2(cos(a), sin(a));
          host32[e] = make_float2(static_cast<float>(host[e].x), static_cast<float>(host[e].y));
        }
    ok = cudaMalloc(reinterpret_cast<void**>(&ctx->d_rope), n * sizeof(double2)) == cudaSuccess &&
         cudaMemcpy(ctx->d_rope, host, n * sizeof(double2), cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMalloc(reinterpret_cast<void**>(&ctx->d_rope32), n * sizeof(float2)) == cudaSuccess &&
         cudaMemcpy(ctx->d_rope32, host32, n * sizeof(float2), cudaMemcpyHostToDevice) == cudaSuccess;
  }
  free(host);
  free(host32);
  return ok;
}

// Which decode kernel family runs for these dims.
int choose_path(const gva_ctx* ctx, bool sep_k) {
  const bool mma_ok = gva::mma_supported(ctx->dims, sep_k);
  if (ctx->path == GVA_PATH_MMA) return mma_ok ? GVA_PATH_MMA : -1;
  if (ctx->path == GVA_PATH_FMA) return gva::fma_supported(ctx->dims, sep_k) ? GVA_PATH_FMA : -1;
  if (mma_ok) return GVA_PATH_MMA;
  return gva::fma_supported(ctx->dims, sep_k) ? GVA_PATH_FMA : -1;
}

// Split-T plan.  The batch's (sequence, group, 64-token tile) units are cut into equal
// contiguous ranges (gva_sched.cuh).  Tensor-core path: one range per CTA, one CTA per SM;
// its P consumer warps share the range, each fed by its own copy warp (mma_shape picks P).
// CUDA-core path: one range per warp, 4 warps per CTA, as many CTAs as fit on the SMs.
// Automatic plans launch one wave, fewer CTAs when the batch has fewer units than that; a
// caller-set split length asks for about split_tokens tokens per warp at max_seq_len.
bool make_plan(const gva_ctx* ctx, int B, int max_seq_len, bool sep_k, gva::Plan* plan, int nq = 1) {
  const int path = choose_path(ctx, sep_k);
  if (path < 0 || B > gva::kMaxBatch || nq < 1) return false;
  if (nq > 1 && (path != GVA_PATH_MMA || sep_k)) return false;  // several queries: tensor-core path
  const int R = ctx->dims.H / ctx->dims.G;
  int nqp = 1;  // queries per pass: powers of two up to the kernel's limit
  while (2 * nqp <= nq && 2 * nqp <= gva::mma_max_queries_per_pass(R, ctx->dims.d_v)) nqp *= 2;
  const long long nt_max = (max_seq_len + GVA_BLOCK_TOKENS - 1) / GVA_BLOCK_TOKENS;
  const long long units_max = static_cast<long long>(B) * ctx->dims.G * nt_max;
  const bool mma = path == GVA_PATH_MMA;
  int pairs = 0, stages = 0;
  if (mma && !gva::mma_shape(ctx->dims, sep_k, B, nqp, &pairs, &stages)) return false;
  const int warps_per_cta = mma ? pairs : 4;  // warps that stream units
  long long grid;
  if (ctx->split_tokens > 0) {
    const long long per_warp = ctx->split_tokens / GVA_BLOCK_TOKENS;
    const long long W = (units_max + per_warp - 1) / per_warp;
    grid = (W + warps_per_cta - 1) / warps_per_cta;
  } else {
    const int per_sm = mma ? 1 : gva::fma_ctas_per_sm(ctx->dims, sep_k, B);
    grid = static_cast<long long>(ctx->num_sms) * per_sm;
    // G*Q ranges: the G ranges of slice q read the same blocks together (gva_sched.cuh),
    // so each block's positional-key tile is read from HBM once
    if (mma && grid >= ctx->dims.G) grid -= grid % ctx->dims.G;
    const long long useful = (units_max + warps_per_cta - 1) / warps_per_cta;
    if (grid > useful) grid = useful;
  }
  if (grid < 1) grid = 1;
  if (grid > (1LL << 20)) return false;
  plan->path = path;
  plan->nqp = nqp;
  plan->grid = static_cast<int>(grid);
  plan->n_warps = static_cast<int>(warps_per_cta * grid);
  plan->n_groups = mma ? plan->grid : plan->n_warps;
  plan->group_warps = mma ? pairs : 1;
  plan->n_stages = mma ? stages : 0;
  plan->ws_bytes = gva::header_bytes(B) +
                   sizeof(float) * (static_cast<size_t>(plan->n_groups) + static_cast<size_t>(B) * ctx->dims.G) *
                       plan->group_warps * R * nqp * gva::partial_stride_floats(ctx->dims.d_v);
  return true;
}

// Phases of a decode call: the split-T partial pass and the combine pass.
constexpr int kPhasePartial = 1;
constexpr int kPhaseCombine = 2;

// Inputs of the fused decode step that the plain decode call does not take.
struct StepInputs {
  const float* q_c;
  const float* q_r;
  const float* M;
  const void* v_new;
  const void* kr_new;
  void* v_pool;
  void* kr_pool;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bytes of E4M3 codes in an fp8 value pool of num_blocks blocks (its exponents follow them).
size_t fp8_code_bytes(int num_blocks, const gva_dims& d) {
  return static_cast<size_t>(num_blocks) * d.G * GVA_BLOCK_TOKENS * d.d_v;
}

// Bytes of the fused step's query stages for a plan: one per (range, segment) pair.
size_t step_stage_bytes(const gva_ctx* ctx, int B, const gva::Plan& plan) {
  const gva_dims& d = ctx->dims;
  return sizeof(float) * (static_cast<size_t>(plan.n_groups) + static_cast<size_t>(B) * d.G) *
         gva::step_stage_floats(d.H / d.G, d.d_v, d.d_r);
}

// Whether the fused step can run for this context (tensor-core path, d_n == d_v).
bool step_fusable(const gva_ctx* ctx, const gva::Plan& plan) {
  return plan.path == GVA_PATH_MMA && plan.nqp == 1 && ctx->dims.d_n == ctx->dims.d_v;
}

// Form gva_decode_step takes for this batch shape: 1 fused, 0 separate kernels, -1 the
// context's mode asks for the fused form where it does not apply.
int step_form(const gva_ctx* ctx, int B, const gva::Plan& plan) {
  switch (ctx->step_mode) {
    case GVA_STEP_FUSED: return step_fusable(ctx, plan) ? 1 : -1;
    case GVA_STEP_SEPARATE: return 0;
    default: {
      // The prologue streams the group's key maps and forms the queries of every segment a
      // CTA's range meets: with large maps or many segments per range the separate absorb
      // kernel does that work faster.
      const gva_dims& d = ctx->dims;
      const long long map_bytes = 4ll * (d.H / d.G) * d.d_v * d.d_n;
      return step_fusable(ctx, plan) && map_bytes <= kStepAutoMapBytes &&
                     static_cast<long long>(B) * d.G <= kStepAutoSegmentsPerRange * plan.n_groups
                 ? 1
                 : 0;
    }
  }
}

gva_status decode_common(gva_ctx* ctx, bool sep_k, int phases, int B, const float* q_abs,
                         const float* q_rot, const void* k_pool, const void* v_pool,
                         const void* kr_pool, const int32_t* block_table, int max_blocks,
                         int num_blocks, const int32_t* seq_lens, int max_seq_len, float* out,
                         void* workspace, size_t ws_bytes, cudaStream_t stream, int nq = 1,
                         const StepInputs* step = nullptr) {
  const bool partial = phases & kPhasePartial, combine = phases & kPhaseCombine;
  if (!ctx || B < 0 || max_seq_len < 1) return GVA_ERR_INVALID_ARG;
  if (partial && (max_blocks < 1 || num_blocks < 1)) return GVA_ERR_INVALID_ARG;
  if (B == 0) return GVA_OK;
  if (B > gva::kMaxBatch) return GVA_ERR_UNSUPPORTED;  // prefix sums live in shared memory
  const gva_dims& d = ctx->dims;
  if (partial) {
    if ((!q_abs && !step) || !v_pool || !block_table || !seq_lens) return GVA_ERR_INVALID_ARG;
    if (sep_k && !k_pool) return GVA_ERR_INVALID_ARG;
    if (!sep_k && d.d_r > 0 && ((!q_rot && !step) || !kr_pool)) return GVA_ERR_INVALID_ARG;
    if (static_cast<long long>(max_blocks) * GVA_BLOCK_TOKENS < max_seq_len) return GVA_ERR_INVALID_ARG;
    if ((q_abs && !aligned16(q_abs)) || !aligned16(v_pool) || (k_pool && !aligned16(k_pool)) ||
        (kr_pool && !aligned16(kr_pool)) || (q_rot && !aligned16(q_rot)))
      return GVA_ERR_INVALID_ARG;
  }
  if (combine && (!out || !aligned16(out))) return GVA_ERR_INVALID_ARG;
  if (!on_ctx_device(ctx)) return GVA_ERR_INVALID_ARG;
  if (nq < 1) return GVA_ERR_INVALID_ARG;
  gva::Plan plan;
  if (!make_plan(ctx, B, max_seq_len, sep_k, &plan, nq)) return GVA_ERR_UNSUPPORTED;
  if (partial && plan.path == GVA_PATH_MMA &&
      static_cast<long long>(num_blocks) * d.G * GVA_BLOCK_TOKENS >= (1LL << 31))
    return GVA_ERR_UNSUPPORTED;  // token rows are int32 tensor-copy coordinates
  if (step && (!step_fusable(ctx, plan) || sep_k || nq != 1)) return GVA_ERR_UNSUPPORTED;
  const size_t stage_off = round_up(plan.ws_bytes, 256);
  const size_t need = step ? stage_off + step_stage_bytes(ctx, B, plan) : plan.ws_bytes;
  if (!workspace || ws_bytes < need || !aligned16(workspace)) return GVA_ERR_WORKSPACE;

  gva::DecodeArgs a{};
  a.q_abs = q_abs;
  a.q_rot = sep_k ? nullptr : q_rot;
  a.v_pool = v_pool;
  if (d.cache_dtype == GVA_FP8_E4M3 && v_pool)  // the exponents follow the codes
    a.v_exp = static_cast<const signed char*>(v_pool) + fp8_code_bytes(num_blocks, d);
  a.k_pool = k_pool;
  a.kr_pool = sep_k ? nullptr : kr_pool;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.part = static_cast<float*>(workspace);
  a.err = ctx->d_err;
  a.B = B;
  a.H = d.H;
  a.G = d.G;
  a.d_v = d.d_v;
  a.d_r = sep_k ? 0 : d.d_r;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.max_seq_len = max_seq_len;
  a.n_warps = plan.n_warps;
  a.n_groups = plan.n_groups;
  a.group_warps = plan.group_warps;
  a.n_stages = plan.n_stages;
  a.scale_log2 = static_cast<float>(static_cast<double>(ctx->scale) * 1.4426950408889634);
  a.nq = nq;
  if (step) {
    a.fused = 1;
    a.q_c = step->q_c;
    a.q_r = step->q_r;
    a.M = step->M;
    a.v_new = step->v_new;
    a.kr_new = step->kr_new;
    a.v_pool_w = step->v_pool;
    if (d.cache_dtype == GVA_FP8_E4M3)
      a.v_exp_w = static_cast<signed char*>(step->v_pool) + fp8_code_bytes(num_blocks, d);
    a.kr_pool_w = step->kr_pool;
    a.rope32 = ctx->d_rope32;
    a.qstage = reinterpret_cast<float*>(static_cast<char*>(workspace) + stage_off);
  }
  // passes over the queries, each a partial pass and a combine: the largest power of two
  // that fits, then smaller ones for the rest (each pass reads the cache once more)
  for (a.q0 = 0; a.q0 < nq; a.q0 += a.nqp) {
    a.nqp = plan.nqp;
    while (a.nqp > nq - a.q0) a.nqp /= 2;
    if (partial) {
      const cudaError_t e = plan.path == GVA_PATH_MMA
                                ? gva::launch_decode_mma(a, sep_k, plan.grid, stream)
                                : gva::launch_decode_fma(a, d.cache_dtype, sep_k, plan.grid, stream);
      if (e != cudaSuccess) return GVA_ERR_CUDA;
    }
    if (combine) {
      // each combine CTA then reads all B lengths: only for batches of up to 256 sequences
      a.combine_after_partial = partial && a.seq_lens && B <= 256 ? 1 : 0;
      a.combine_big = static_cast<long long>(B) * d.G <= ctx->num_sms ? 1 : 0;
      const cudaError_t e = gva::launch_combine(a, stream);
      if (e != cudaSuccess) return GVA_ERR_CUDA;
    }
  }
  return GVA_OK;
}

}  // namespace

extern "C" {

gva_status gva_create(const gva_dims* dims, gva_ctx** out) {
  if (!dims || !out) return GVA_ERR_INVALID_ARG;
  const gva_dims& d = *dims;
  if (d.H <= 0 || d.G <= 0 || d.H % d.G != 0 || d.d_v <= 0 || d.d_n <= 0 || d.d_r < 0 ||
      (d.d_r & 1) || d.d_v % 32 != 0 || d.d_n % 4 != 0 || d.block_size != GVA_BLOCK_TOKENS)
    return GVA_ERR_INVALID_ARG;
  if (d.cache_dtype != GVA_F32 && d.cache_dtype != GVA_BF16 && d.cache_dtype != GVA_FP8_E4M3)
    return GVA_ERR_INVALID_ARG;
  if (d.d_r > 32) return GVA_ERR_UNSUPPORTED;
  if (!gva::fma_supported(d, false) && !gva::mma_supported(d, false) &&
      !(d.d_r == 0 && (gva::fma_supported(d, true) || gva::mma_supported(d, true))))
    return GVA_ERR_UNSUPPORTED;
  gva_ctx* ctx = static_cast<gva_ctx*>(calloc(1, sizeof(gva_ctx)));
  if (!ctx) return GVA_ERR_CUDA;
  ctx->dims = d;
  ctx->scale = d.scale > 0.f ? d.scale : static_cast<float>(1.0 / sqrt(static_cast<double>(d.d_n + d.d_r)));
  ctx->rope_base = d.rope_base > 0.0 ? d.rope_base : 10000.0;
  ctx->split_tokens = 0;
  ctx->path = GVA_PATH_AUTO;
  ctx->step_mode = GVA_STEP_AUTO;
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess ||
      cudaMalloc(reinterpret_cast<void**>(&ctx->d_err), sizeof(unsigned)) != cudaSuccess) {
    gva_destroy(ctx);
    return GVA_ERR_CUDA;
  }
  if (cudaMemset(ctx->d_err, 0, sizeof(unsigned)) != cudaSuccess || !build_rope_table(ctx)) {
    gva_destroy(ctx);
    return GVA_ERR_CUDA;
  }
  *out = ctx;
  return GVA_OK;
}

void gva_destroy(gva_ctx* ctx) {
  if (!ctx) return;
  if (ctx->d_err) cudaFree(ctx->d_err);
  if (ctx->d_rope) cudaFree(ctx->d_rope);
  if (ctx->d_rope32) cudaFree(ctx->d_rope32);
  free(ctx);
}

gva_status gva_absorb_query(gva_ctx* ctx, int B, const float* q_c, const float* q_r,
                            const int32_t* pos_q, const float* M, float* q_abs, float* q_rot,
                            gva_stream_t stream) {
  if (!ctx || B < 0) return GVA_ERR_INVALID_ARG;
  if (B == 0) return GVA_OK;
  if (!q_c || !pos_q || !M || !q_abs) return GVA_ERR_INVALID_ARG;
  if (ctx->dims.d_r > 0 && (!q_r || !q_rot)) return GVA_ERR_INVALID_ARG;
  if (!aligned16(q_c) || !aligned16(M) || !aligned16(q_abs) || (q_r && !aligned16(q_r)) ||
      (q_rot && !aligned16(q_rot)))
    return GVA_ERR_INVALID_ARG;
  if (!on_ctx_device(ctx)) return GVA_ERR_INVALID_ARG;
  return from_cuda(gva::launch_absorb(ctx, B, q_c, q_r, pos_q, M, q_abs, q_rot,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

gva_status gva_cache_append(gva_ctx* ctx, int B, int n, const void* v_new, const void* kr_new,
                            const int32_t* pos, const int32_t* block_table, int max_blocks,
                            int num_blocks, void* v_pool, void* kr_pool, gva_stream_t stream) {
  if (!ctx || B < 0 || n < 0) return GVA_ERR_INVALID_ARG;
  if (B == 0 || n == 0) return GVA_OK;
  if (!v_new || !pos || !block_table || !v_pool || max_blocks < 1 || num_blocks < 1)
    return GVA_ERR_INVALID_ARG;
  if (ctx->dims.d_r > 0 && (!kr_new || !kr_pool)) return GVA_ERR_INVALID_ARG;
  if (!aligned16(v_new) || !aligned16(v_pool)) return GVA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * n > (1LL << 40)) return GVA_ERR_INVALID_ARG;
  if (!on_ctx_device(ctx)) return GVA_ERR_INVALID_ARG;
  return from_cuda(gva::launch_append(ctx, B, n, v_new, kr_new, pos, block_table, max_blocks,
                                      num_blocks, v_pool, kr_pool,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t gva_decode_workspace_size(const gva_ctx* ctx, int B, int max_seq_len) {
  if (!ctx || B <= 0 || max_seq_len < 1) return 0;
  gva::Plan plan;
  const bool sep_k = false;
  if (!make_plan(ctx, B, max_seq_len, sep_k, &plan)) {
    if (!make_plan(ctx, B, max_seq_len, true, &plan)) return 0;
  }
  // The GQA form of a d_r == 0 context may plan differently; cover both.
  gva::Plan other;
  if (ctx->dims.d_r == 0 && make_plan(ctx, B, max_seq_len, true, &other) &&
      other.ws_bytes > plan.ws_bytes)
    plan = other;
  return plan.ws_bytes;
}

gva_status gva_decode_attention(gva_ctx* ctx, int B, const float* q_abs, const float* q_rot,
                                const void* v_pool, const void* kr_pool,
                                const int32_t* block_table, int max_blocks, int num_blocks,
                                const int32_t* seq_lens, int max_seq_len, float* out,
                                void* workspace, size_t ws_bytes, gva_stream_t stream) {
  return decode_common(ctx, false, kPhasePartial | kPhaseCombine, B, q_abs, q_rot, nullptr, v_pool,
                       kr_pool, block_table, max_blocks, num_blocks, seq_lens, max_seq_len, out,
                       workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

gva_status gva_decode_partial(gva_ctx* ctx, int B, const float* q_abs, const float* q_rot,
                              const void* v_pool, const void* kr_pool, const int32_t* block_table,
                              int max_blocks, int num_blocks, const int32_t* seq_lens,
                              int max_seq_len, void* workspace, size_t ws_bytes,
                              gva_stream_t stream) {
  return decode_common(ctx, false, kPhasePartial, B, q_abs, q_rot, nullptr, v_pool, kr_pool,
                       block_table, max_blocks, num_blocks, seq_lens, max_seq_len, nullptr,
                       workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

gva_status gva_decode_combine(gva_ctx* ctx, int B, int max_seq_len, float* out, void* workspace,
                              size_t ws_bytes, gva_stream_t stream) {
  return decode_common(ctx, false, kPhaseCombine, B, nullptr, nullptr, nullptr, nullptr, nullptr,
                       nullptr, 0, 0, nullptr, max_seq_len, out, workspace, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

gva_status gva_decode_attention_multi(gva_ctx* ctx, int B, int n_q, const float* q_abs,
                                      const float* q_rot, const void* v_pool, const void* kr_pool,
                                      const int32_t* block_table, int max_blocks, int num_blocks,
                                      const int32_t* seq_lens, int max_seq_len, float* out,
                                      void* workspace, size_t ws_bytes, gva_stream_t stream) {
  if (n_q < 1) return GVA_ERR_INVALID_ARG;
  if (n_q > max_seq_len) return GVA_ERR_INVALID_ARG;
  return decode_common(ctx, false, kPhasePartial | kPhaseCombine, B, q_abs, q_rot, nullptr, v_pool,
                       kr_pool, block_table, max_blocks, num_blocks, seq_lens, max_seq_len, out,
                       workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream), n_q);
}

size_t gva_decode_workspace_size_multi(const gva_ctx* ctx, int B, int n_q, int max_seq_len) {
  if (!ctx || B <= 0 || n_q < 1 || max_seq_len < 1) return 0;
  gva::Plan plan;
  if (!make_plan(ctx, B, max_seq_len, false, &plan, n_q)) return 0;
  return plan.ws_bytes;
}

int gva_step_is_fused(const gva_ctx* ctx, int B, int max_seq_len) {
  if (!ctx || B <= 0 || max_seq_len < 1) return -1;
  gva::Plan plan;
  if (!make_plan(ctx, B, max_seq_len, false, &plan)) return -1;
  return step_form(ctx, B, plan);
}

gva_status gva_decode_step_partial(gva_ctx* ctx, int B, const float* q_c, const float* q_r, const float* M,
                                   const void* v_new, const void* kr_new, void* v_pool, void* kr_pool,
                                   const int32_t* block_table, int max_blocks, int num_blocks,
                                   const int32_t* seq_lens, int max_seq_len, void* workspace, size_t ws_bytes,
                                   gva_stream_t stream) {
  if (!ctx || B < 0 || max_seq_len < 1) return GVA_ERR_INVALID_ARG;
  if (B == 0) return GVA_OK;
  if (!q_c || !M || !v_new || (ctx->dims.d_r > 0 && (!q_r || !kr_new))) return GVA_ERR_INVALID_ARG;
  if (!aligned16(q_c) || !aligned16(M) || !aligned16(v_new) || (q_r && !aligned16(q_r)) ||
      (kr_new && (reinterpret_cast<uintptr_t>(kr_new) & 3u)))
    return GVA_ERR_INVALID_ARG;
  if (!step_buffers_addressable(q_c, q_r, v_new, kr_new, nullptr)) return GVA_ERR_INVALID_ARG;
  const StepInputs in{q_c, q_r, M, v_new, kr_new, v_pool, kr_pool};
  return decode_common(ctx, false, kPhasePartial, B, nullptr, nullptr, nullptr, v_pool, kr_pool, block_table,
                       max_blocks, num_blocks, seq_lens, max_seq_len, nullptr, workspace, ws_bytes,
                       reinterpret_cast<cudaStream_t>(stream), 1, &in);
}

size_t gva_decode_step_workspace_size(const gva_ctx* ctx, int B, int max_seq_len) {
  if (!ctx || B <= 0 || max_seq_len < 1) return 0;
  gva::Plan plan;
  if (!make_plan(ctx, B, max_seq_len, false, &plan)) return 0;
  const gva_dims& d = ctx->dims;
  const size_t off = round_up(plan.ws_bytes, 256);
  // separate calls: the absorbed and rotated queries follow the decode workspace
  const size_t separate = sizeof(float) * static_cast<size_t>(B) * d.H * (d.d_v + d.d_r) + 16;
  const size_t fused = step_fusable(ctx, plan) ? step_stage_bytes(ctx, B, plan) : 0;
  return off + (fused > separate ? fused : separate);
}

gva_status gva_decode_step(gva_ctx* ctx, int B, const float* q_c, const float* q_r, const float* M,
                           const void* v_new, const void* kr_new, void* v_pool, void* kr_pool,
                           const int32_t* block_table, int max_blocks, int num_blocks,
                           const int32_t* seq_lens, int max_seq_len, float* out, void* workspace,
                           size_t ws_bytes, gva_stream_t stream_) {
  if (!ctx || B < 0 || max_seq_len < 1) return GVA_ERR_INVALID_ARG;
  if (B == 0) return GVA_OK;
  const gva_dims& d = ctx->dims;
  if (!q_c || !M || !v_new || !v_pool || !block_table || !seq_lens || !out) return GVA_ERR_INVALID_ARG;
  if (d.d_r > 0 && (!q_r || !kr_new || !kr_pool)) return GVA_ERR_INVALID_ARG;
  if (!aligned16(q_c) || !aligned16(M) || !aligned16(v_new) || (q_r && !aligned16(q_r)) ||
      (kr_new && (reinterpret_cast<uintptr_t>(kr_new) & 3u)))
    return GVA_ERR_INVALID_ARG;
  if (B > gva::kMaxBatch) return GVA_ERR_UNSUPPORTED;
  if (!on_ctx_device(ctx)) return GVA_ERR_INVALID_ARG;
  if (!step_buffers_addressable(q_c, q_r, v_new, kr_new, out)) return GVA_ERR_INVALID_ARG;
  gva::Plan plan;
  if (!make_plan(ctx, B, max_seq_len, false, &plan)) return GVA_ERR_UNSUPPORTED;
  const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int form = step_form(ctx, B, plan);
  if (form < 0) return GVA_ERR_UNSUPPORTED;
  if (form == 1) {
    const StepInputs in{q_c, q_r, M, v_new, kr_new, v_pool, kr_pool};
    return decode_common(ctx, false, kPhasePartial | kPhaseCombine, B, nullptr, nullptr, nullptr, v_pool,
                         kr_pool, block_table, max_blocks, num_blocks, seq_lens, max_seq_len, out,
                         workspace, ws_bytes, stream, 1, &in);
  }
  // Separate calls: append at position seq_lens[b] - 1, absorb at the same position, decode.
  const size_t off = round_up(plan.ws_bytes, 256);
  const size_t qbytes = sizeof(float) * static_cast<size_t>(B) * d.H * (d.d_v + d.d_r);
  if (!workspace || !aligned16(workspace) || ws_bytes < off + qbytes) return GVA_ERR_WORKSPACE;
  float* q_abs = reinterpret_cast<float*>(static_cast<char*>(workspace) + off);
  float* q_rot = d.d_r > 0 ? q_abs + static_cast<size_t>(B) * d.H * d.d_v : nullptr;
  if (gva::launch_append(ctx, B, 1, v_new, kr_new, nullptr, block_table, max_blocks, num_blocks, v_pool,
                         kr_pool, stream, seq_lens) != cudaSuccess ||
      gva::launch_absorb(ctx, B, q_c, q_r, nullptr, M, q_abs, q_rot, stream, seq_lens, true) != cudaSuccess)
    return GVA_ERR_CUDA;
  return decode_common(ctx, false, kPhasePartial | kPhaseCombine, B, q_abs, q_rot, nullptr, v_pool, kr_pool,
                       block_table, max_blocks, num_blocks, seq_lens, max_seq_len, out, workspace, off,
                       stream);
}

size_t gva_decode_step_workspace_size_multi(const gva_ctx* ctx, int B, int n_q, int max_seq_len) {
  if (!ctx || B <= 0 || n_q < 1 || max_seq_len < 1) return 0;
  if (n_q == 1) return gva_decode_step_workspace_size(ctx, B, max_seq_len);
  gva::Plan plan;
  if (!make_plan(ctx, B, max_seq_len, false, &plan, n_q)) return 0;
  const gva_dims& d = ctx->dims;
  return round_up(plan.ws_bytes, 256) + sizeof(float) * static_cast<size_t>(B) * n_q * d.H * (d.d_v + d.d_r) + 16;
}

gva_status gva_decode_step_multi(gva_ctx* ctx, int B, int n_q, const float* q_c, const float* q_r,
                                 const float* M, const void* v_new, const void* kr_new, void* v_pool,
                                 void* kr_pool, const int32_t* block_table, int max_blocks, int num_blocks,
                                 const int32_t* seq_lens, int max_seq_len, float* out, void* workspace,
                                 size_t ws_bytes, gva_stream_t stream_) {
  if (!ctx || B < 0 || n_q < 1 || max_seq_len < 1 || n_q > max_seq_len) return GVA_ERR_INVALID_ARG;
  if (n_q == 1)
    return gva_decode_step(ctx, B, q_c, q_r, M, v_new, kr_new, v_pool, kr_pool, block_table, max_blocks,
                           num_blocks, seq_lens, max_seq_len, out, workspace, ws_bytes, stream_);
  if (B == 0) return GVA_OK;
  const gva_dims& d = ctx->dims;
  if (!q_c || !M || !v_new || !v_pool || !block_table || !seq_lens || !out) return GVA_ERR_INVALID_ARG;
  if (d.d_r > 0 && (!q_r || !kr_new || !kr_pool)) return GVA_ERR_INVALID_ARG;
  if (!aligned16(q_c) || !aligned16(M) || !aligned16(v_new) || (q_r && !aligned16(q_r)) ||
      (kr_new && (reinterpret_cast<uintptr_t>(kr_new) & 3u)))
    return GVA_ERR_INVALID_ARG;
  if (B > gva::kMaxBatch || static_cast<long long>(B) * n_q > (1LL << 30)) return GVA_ERR_UNSUPPORTED;
  if (!on_ctx_device(ctx)) return GVA_ERR_INVALID_ARG;
  if (!step_buffers_addressable(q_c, q_r, v_new, kr_new, out)) return GVA_ERR_INVALID_ARG;
  gva::Plan plan;
  if (!make_plan(ctx, B, max_seq_len, false, &plan, n_q)) return GVA_ERR_UNSUPPORTED;
  const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // append the n_q tokens at the last n_q positions, absorb the B*n_q query rows at the same
  // positions (overlapping the append), decode
  const size_t off = round_up(plan.ws_bytes, 256);
  const size_t rows = static_cast<size_t>(B) * n_q;
  const size_t qbytes = sizeof(float) * rows * d.H * (d.d_v + d.d_r);
  if (!workspace || !aligned16(workspace) || ws_bytes < off + qbytes) return GVA_ERR_WORKSPACE;
  float* q_abs = reinterpret_cast<float*>(static_cast<char*>(workspace) + off);
  float* q_rot = d.d_r > 0 ? q_abs + rows * d.H * d.d_v : nullptr;
  if (gva::launch_append(ctx, B, n_q, v_new, kr_new, nullptr, block_table, max_blocks, num_blocks, v_pool,
                         kr_pool, stream, seq_lens) != cudaSuccess ||
      gva::launch_absorb(ctx, static_cast<int>(rows), q_c, q_r, nullptr, M, q_abs, q_rot, stream, seq_lens, true,
                         n_q) != cudaSuccess)
    return GVA_ERR_CUDA;
  return decode_common(ctx, false, kPhasePartial | kPhaseCombine, B, q_abs, q_rot, nullptr, v_pool, kr_pool,
                       block_table, max_blocks, num_blocks, seq_lens, max_seq_len, out, workspace, off, stream,
                       n_q);
}

gva_status gva_set_step_mode(gva_ctx* ctx, gva_step_mode mode) {
  if (!ctx || (mode != GVA_STEP_AUTO && mode != GVA_STEP_FUSED && mode != GVA_STEP_SEPARATE))
    return GVA_ERR_INVALID_ARG;
  ctx->step_mode = mode;
  return GVA_OK;
}

gva_status gqa_decode_attention(gva_ctx* ctx, int B, const float* q, const void* k_pool,
                                const void* v_pool, const int32_t* block_table, int max_blocks,
                                int num_blocks, const int32_t* seq_lens, int max_seq_len,
                                float* out, void* workspace, size_t ws_bytes,
                                gva_stream_t stream) {
  if (ctx && ctx->dims.d_r != 0) return GVA_ERR_INVALID_ARG;
  return decode_common(ctx, true, kPhasePartial | kPhaseCombine, B, q, nullptr, k_pool, v_pool,
                       nullptr, block_table, max_blocks, num_blocks, seq_lens, max_seq_len, out,
                       workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

gva_status gva_set_split_tokens(gva_ctx* ctx, int split_tokens) {
  if (!ctx || split_tokens < 0 || split_tokens % GVA_BLOCK_TOKENS != 0) return GVA_ERR_INVALID_ARG;
  ctx->split_tokens = split_tokens;
  return GVA_OK;
}

gva_status gva_set_decode_path(gva_ctx* ctx, gva_decode_path path) {
  if (!ctx || (path != GVA_PATH_AUTO && path != GVA_PATH_FMA && path != GVA_PATH_MMA))
    return GVA_ERR_INVALID_ARG;
  ctx->path = path;
  return GVA_OK;
}

gva_status gva_decode_plan(const gva_ctx* ctx, int B, int max_seq_len, int* split_tokens,
                           int* max_splits) {
  if (!ctx || B <= 0 || max_seq_len < 1) return GVA_ERR_INVALID_ARG;
  gva::Plan plan;
  // the GVA form when it applies, else the GQA form (d_r == 0 contexts)
  if (!make_plan(ctx, B, max_seq_len, false, &plan) && !make_plan(ctx, B, max_seq_len, true, &plan))
    return GVA_ERR_UNSUPPORTED;
  const long long units_max = static_cast<long long>(B) * ctx->dims.G *
                              ((max_seq_len + GVA_BLOCK_TOKENS - 1) / GVA_BLOCK_TOKENS);
  if (split_tokens)
    *split_tokens = static_cast<int>((units_max + plan.n_warps - 1) / plan.n_warps) * GVA_BLOCK_TOKENS;
  if (max_splits) *max_splits = plan.n_warps;
  return GVA_OK;
}

gva_status gva_get_device_error(gva_ctx* ctx, unsigned* bits) {
  if (!ctx || !bits) return GVA_ERR_INVALID_ARG;
  if (!on_ctx_device(ctx)) return GVA_ERR_INVALID_ARG;
  unsigned v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(&v, ctx->d_err, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(ctx->d_err, 0, sizeof(unsigned)) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess)
    return GVA_ERR_CUDA;
  *bits = v;
  return v ? GVA_ERR_DEVICE_INDEX : GVA_OK;
}

const char* gva_status_string(gva_status s) {
  switch (s) {
    case GVA_OK: return "ok";
    case GVA_ERR_INVALID_ARG: return "invalid argument";
    case GVA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case GVA_ERR_WORKSPACE: return "workspace missing or too small";
    case GVA_ERR_CUDA: return "CUDA runtime error";
    case GVA_ERR_DEVICE_INDEX: return "device reported an index error";
  }
  return "unknown status";
}

int gva_version(void) { return kVersion; }

}  // extern "C"
