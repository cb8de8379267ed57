// gva_append.cu -- writes new tokens into the compact GVA cache.
//
// Per token the cache gets the G grouped value rows (a bit copy) and ONE positional key,
// rotated to the token's own position (the cache holds grouped values plus a small,
// separately cached, rotated positional key: abstract "Grouped Value Attention: Efficient
// KV Caching via On-Demand Key Reconstruction"; review "[논문리뷰] Grouped Value Attention",
// section 3, Decoupled RoPE).  One warp per token: the value rows move as 16-byte vectors
// (loaded before the slot is known), lanes rotate the positional pairs (fp32 for bf16
// caches, fp64 for fp32 caches) and round once to the cache dtype.  The fp8 value cache
// quantises each value row instead of copying it (append_fp8_kernel).
#include <type_traits>

#include "gva_device.cuh"
#include "gva_internal.h"
#include "gva_sched.cuh"

namespace gva {
namespace {

struct AppendArgs {
  const void* v_new;
  const void* kr_new;
  const int32_t* pos;       // null: the n new tokens are the last n positions, seq_lens[b] - n + t
  const int32_t* seq_lens;
  const int32_t* block_table;
  void* v_pool;
  void* kr_pool;
  const double2* rope;   // fp64 RoPE digit table (fp32 caches)
  const float2* rope32;  // fp32 RoPE digit table (bf16 caches)
  unsigned* err;
  int B, n, G, d_v, d_r, max_blocks, num_blocks;
};

constexpr int kAppendThreads = 256;

constexpr int kAppendVecPerLane = 8;  // value-row 16-byte vectors held per lane

template <typename T>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendArgs a) {
  const long long warp_id =
      (static_cast<long long>(blockIdx.x) * kAppendThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  const long long ntok = static_cast<long long>(a.B) * a.n;
  if (warp_id >= ntok) return;
  const int b = static_cast<int>(warp_id / a.n);
  const int t = static_cast<int>(warp_id % a.n);
  const long long tok = static_cast<long long>(b) * a.n + t;

  // Loads that do not depend on the slot go out first.
  const int vec_per_row = a.d_v * static_cast<int>(sizeof(T)) / 16;
  const int nvec = a.G * vec_per_row;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(a.v_new) +
                                                    tok * a.G * a.d_v);
  uint4 vreg[kAppendVecPerLane];
#pragma unroll
  for (int c = 0; c < kAppendVecPerLane; ++c) {
    const int i = lane + 32 * c;
    if (i < nvec) vreg[c] = src[i];
  }
  const int pairs = a.d_r / 2;
  // bf16 keys are rotated in fp32: its error (a few units of 2^-24, relative) moves the bf16
  // result only for values that close to a rounding boundary, and then by one ulp.  fp32
  // keys are rotated in fp64 and rounded once.
  constexpr bool kF64 = sizeof(T) == 4;
  using R = typename std::conditional<kF64, double, float>::type;
  const T* x = static_cast<const T*>(a.kr_new) + tok * a.d_r;
  R x0 = 0, x1 = 0;
  if (lane < pairs) {
    x0 = static_cast<R>(CacheElem<T>::to_float(x[2 * lane]));
    x1 = static_cast<R>(CacheElem<T>::to_float(x[2 * lane + 1]));
  }
  const long long p =
      (a.pos ? static_cast<long long>(a.pos[b]) : static_cast<long long>(a.seq_lens[b]) - a.n) + t;

  // Resolve the slot; an unresolvable one skips the token and is reported.
  if (p < 0 || (p >> 6) >= a.max_blocks || p >= (1LL << 32)) {
    if (lane == 0) flag_error(a.err, GVA_DEVERR_POSITION);
    return;
  }
  const int blk = a.block_table[static_cast<long long>(b) * a.max_blocks + (p >> 6)];
  R c = 1, s = 0;
  if (lane < pairs) {
    if constexpr (kF64)
      rope_cos_sin(a.rope, pairs, p, lane, c, s);
    else
      rope_cos_sin_f32(a.rope32, pairs, p, lane, c, s);
  }
  if (blk < 0 || blk >= a.num_blocks) {
    if (lane == 0) flag_error(a.err, GVA_DEVERR_BLOCK_ID);
    return;
  }
  const int o = static_cast<int>(p & (kBlockTokens - 1));

  // Grouped value rows: G rows of d_v elements, copied bit for bit.
  auto dst_of = [&](int i) {
    const int g = i / vec_per_row, w = i - g * vec_per_row;
    return reinterpret_cast<uint4*>(static_cast<T*>(a.v_pool) +
                                    ((static_cast<long long>(blk) * a.G + g) * kBlockTokens + o) * a.d_v) +
           w;
  };
#pragma unroll
  for (int cc = 0; cc < kAppendVecPerLane; ++cc) {
    const int i = lane + 32 * cc;
    if (i < nvec) *dst_of(i) = vreg[cc];
  }
  for (int i = lane + 32 * kAppendVecPerLane; i < nvec; i += 32) *dst_of(i) = src[i];

  // Shared positional key, rotated to position p: pair (2i, 2i+1) turned by p*theta_i.
  T* y = static_cast<T*>(a.kr_pool) + (static_cast<long long>(blk) * kBlockTokens + o) * a.d_r;
  if (lane < pairs) {
    if constexpr (kF64) {
      // explicit roundings (no contraction) so each product is rounded on its own
      const double y0 = __dsub_rn(__dmul_rn(x0, c), __dmul_rn(x1, s));
      const double y1 = __dadd_rn(__dmul_rn(x0, s), __dmul_rn(x1, c));
      y[2 * lane] = CacheElem<T>::from_double(y0);
      y[2 * lane + 1] = CacheElem<T>::from_double(y1);
    } else {
      float y0, y1;
      rope_rotate_f32(x0, x1, c, s, y0, y1);
      y[2 * lane] = __float2bfloat16_rn(y0);
      y[2 * lane + 1] = __float2bfloat16_rn(y1);
    }
  }
}

// The fp8 value cache (E4M3 codes and a power-of-two scale per (token, group); bf16 new
// values and keys).  Same warp per token and slot resolution as above; each group's value
// row is quantised: e from the row's largest magnitude (fp8_row_exponent), every value
// times 2^-e (exact) rounded to E4M3 with saturation.  A lane holds 16-byte vectors of 8
// values; the vec_per_row lanes of a row (a power of two dividing 32) reduce its maximum by
// shuffles.  Codes go to the code region, the exponent after all codes.
__global__ void __launch_bounds__(kAppendThreads) append_fp8_kernel(const AppendArgs a) {
  const long long warp_id =
      (static_cast<long long>(blockIdx.x) * kAppendThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  const long long ntok = static_cast<long long>(a.B) * a.n;
  if (warp_id >= ntok) return;
  const int b = static_cast<int>(warp_id / a.n);
  const int t = static_cast<int>(warp_id % a.n);
  const long long tok = static_cast<long long>(b) * a.n + t;

  const int vec_per_row = a.d_v / 8;  // 8 or 16
  const int nvec = a.G * vec_per_row;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.v_new) + tok * a.G * a.d_v);
  uint4 vreg[kAppendVecPerLane];
#pragma unroll
  for (int c = 0; c < kAppendVecPerLane; ++c) {
    const int i = lane + 32 * c;
    if (i < nvec) vreg[c] = src[i];
  }
  const int pairs = a.d_r / 2;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.kr_new) + tok * a.d_r;
  float x0 = 0.f, x1 = 0.f;
  if (lane < pairs) {
    x0 = __bfloat162float(x[2 * lane]);
    x1 = __bfloat162float(x[2 * lane + 1]);
  }
  const long long p =
      (a.pos ? static_cast<long long>(a.pos[b]) : static_cast<long long>(a.seq_lens[b]) - a.n) + t;
  if (p < 0 || (p >> 6) >= a.max_blocks || p >= (1LL << 32)) {
    if (lane == 0) flag_error(a.err, GVA_DEVERR_POSITION);
    return;
  }
  const int blk = a.block_table[static_cast<long long>(b) * a.max_blocks + (p >> 6)];
  float c = 1.f, s = 0.f;
  if (lane < pairs) rope_cos_sin_f32(a.rope32, pairs, p, lane, c, s);
  if (blk < 0 || blk >= a.num_blocks) {
    if (lane == 0) flag_error(a.err, GVA_DEVERR_BLOCK_ID);
    return;
  }
  const int o = static_cast<int>(p & (kBlockTokens - 1));
  unsigned char* codes = static_cast<unsigned char*>(a.v_pool);
  signed char* exps = reinterpret_cast<signed char*>(codes) +
                      static_cast<long long>(a.num_blocks) * a.G * kBlockTokens * a.d_v;

  // vector i of the token (lane + 32 cc): row g = i / vec_per_row, 8 values from column 8w
  auto quantise = [&](const uint4& vv, int i) {
    float v[8];
    bf16x2_to_float2(vv.x, v[0], v[1]);
    bf16x2_to_float2(vv.y, v[2], v[3]);
    bf16x2_to_float2(vv.z, v[4], v[5]);
    bf16x2_to_float2(vv.w, v[6], v[7]);
    float amax = 0.f;
    if (i < nvec) {
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
    }
    for (int off = vec_per_row >> 1; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
    if (i < nvec) {
      const int g = i / vec_per_row, w = i - g * vec_per_row;
      const int e = fp8_row_exponent(amax);
      const float inv = exp2_int(-e);  // exact scaling: -e is in [-120, 126]
      uint2 q;
      q.x = f32x2_to_e4m3x2(v[0] * inv, v[1] * inv) | (f32x2_to_e4m3x2(v[2] * inv, v[3] * inv) << 16);
      q.y = f32x2_to_e4m3x2(v[4] * inv, v[5] * inv) | (f32x2_to_e4m3x2(v[6] * inv, v[7] * inv) << 16);
      const long long row = (static_cast<long long>(blk) * a.G + g) * kBlockTokens + o;
      reinterpret_cast<uint2*>(codes + row * a.d_v)[w] = q;
      if (w == 0) exps[row] = static_cast<signed char>(e);
    }
  };
#pragma unroll
  for (int cc = 0; cc < kAppendVecPerLane; ++cc)
    if (32 * cc < nvec) quantise(vreg[cc], lane + 32 * cc);  // warp-uniform condition
  for (int base = 32 * kAppendVecPerLane; base < nvec; base += 32) {
    const int i = lane + base;
    quantise(i < nvec ? src[i] : make_uint4(0, 0, 0, 0), i);
  }

  // Shared positional key (bf16), rotated to position p as in the bf16 cache.
  __nv_bfloat16* y = static_cast<__nv_bfloat16*>(a.kr_pool) + (static_cast<long long>(blk) * kBlockTokens + o) * a.d_r;
  if (lane < pairs) {
    float y0, y1;
    rope_rotate_f32(x0, x1, c, s, y0, y1);
    y[2 * lane] = __float2bfloat16_rn(y0);
    y[2 * lane + 1] = __float2bfloat16_rn(y1);
  }
}

}  // namespace

cudaError_t launch_append(const gva_ctx* ctx, int B, int n, const void* v_new,
                          const void* kr_new, const int32_t* pos, const int32_t* block_table,
                          int max_blocks, int num_blocks, void* v_pool, void* kr_pool,
                          cudaStream_t stream, const int32_t* seq_lens) {
  AppendArgs a;
  a.v_new = v_new;
  a.kr_new = kr_new;
  a.pos = pos;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.v_pool = v_pool;
  a.kr_pool = kr_pool;
  a.err = ctx->d_err;
  a.B = B;
  a.n = n;
  a.G = ctx->dims.G;
  a.d_v = ctx->dims.d_v;
  a.d_r = ctx->dims.d_r;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.rope = ctx->d_rope;
  a.rope32 = ctx->d_rope32;
  const long long threads = static_cast<long long>(B) * n * 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((threads + kAppendThreads - 1) / kAppendThreads));
  cfg.blockDim = dim3(kAppendThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (ctx->dims.cache_dtype == GVA_F32) return cudaLaunchKernelEx(&cfg, append_kernel<float>, a);
  if (ctx->dims.cache_dtype == GVA_FP8_E4M3) return cudaLaunchKernelEx(&cfg, append_fp8_kernel, a);
  return cudaLaunchKernelEx(&cfg, append_kernel<__nv_bfloat16>, a);
}

}  // namespace gva
