// gva_absorb.cu -- per-step query preparation for GVA decode.
//
// Absorption: the key map M_h (K_h = V_g(h) M_h) is folded into the query, q' = M_h q_c, so
// the content score becomes one inner product with the cached value and no content key is
// ever built (ai-feeds.com summary "Grouped Value Attention:通过按需 key 重建实现高效 KV
// 缓存", section 方法: Q' = Q M^T; m.szthrk.cn explainer, section "GVA 的正式方案").
// Decoupled RoPE: only the positional slice of the query is rotated, at the query's
// position (review "[논문리뷰] Grouped Value Attention", section 3).
//
// The work is tiny and latency-bound, so the kernel is laid out for few dependent memory
// round trips: one CTA per (head, 16 sequences); warps 0-3 stage M_h and the content
// queries in shared memory with bulk copies (one round trip), then compute the GEMV (fp32
// FMA in k order); warps 4-7 meanwhile rotate the positional queries (fp64, digit table).
#include "gva_device.cuh"
#include "gva_internal.h"
#include "gva_sched.cuh"

namespace gva {
namespace {

constexpr int kGemvThreads = 128;
constexpr int kAbsorbThreads = 256;
constexpr int kAbsorbSeqs = 16;

struct AbsorbArgs {
  const float* q_c;
  const float* q_r;
  const int32_t* pos_q;
  const float* M;
  float* q_abs;
  float* q_rot;
  const double2* rope;
  unsigned* err;
  int B, H, d_v, d_n, d_r;
};

__global__ void __launch_bounds__(kAbsorbThreads) absorb_kernel(const AbsorbArgs a) {
  extern __shared__ __align__(16) float sm[];
  __shared__ __align__(8) uint64_t bar;
  const int ldm = a.d_n + 4;     // padded row: conflict-free 16-byte reads by row
  float* Ms = sm;                // [d_v][d_n + 4]
  float* qs = sm + a.d_v * ldm;  // [kAbsorbSeqs][d_n]
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * kAbsorbSeqs;
  const int nb = min(kAbsorbSeqs, a.B - b0);
  griddep_wait();
  griddep_launch_dependents();

  if (threadIdx.x >= kGemvThreads) {
    // positional slice of the query, rotated at pos_q[b] in fp64
    const int pairs = a.d_r / 2;
    for (int idx = threadIdx.x - kGemvThreads; idx < nb * pairs; idx += kAbsorbThreads - kGemvThreads) {
      const int bt = idx / pairs, i = idx - bt * pairs;
      const long long row = (static_cast<long long>(b0 + bt) * a.H + h) * a.d_r;
      const float2 x = *reinterpret_cast<const float2*>(a.q_r + row + 2 * i);
      const long long p = a.pos_q[b0 + bt];
      double c = 1.0, s = 0.0;
      if (p >= 0)
        rope_cos_sin(a.rope, pairs, p, i, c, s);
      else if (i == 0)
        flag_error(a.err, GVA_DEVERR_POSITION);  // left unrotated
      const double x0 = x.x, x1 = x.y;
      float2 y;
      y.x = __double2float_rn(__dsub_rn(__dmul_rn(x0, c), __dmul_rn(x1, s)));
      y.y = __double2float_rn(__dadd_rn(__dmul_rn(x0, s), __dmul_rn(x1, c)));
      *reinterpret_cast<float2*>(a.q_rot + row + 2 * i) = y;
    }
    return;
  }

  // stage M_h (padded rows) and the content queries with bulk copies: one DRAM round trip
  const int t = threadIdx.x;
  if (t == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kGemvThreads) : "memory");
  const uint32_t row_bytes = static_cast<uint32_t>(a.d_n) * 4;
  if (t == 0) mbar_arrive_expect_tx(&bar, row_bytes * static_cast<uint32_t>(a.d_v + nb));
  asm volatile("bar.sync 1, %0;" ::"n"(kGemvThreads) : "memory");
  if (t < 32) {
    const float* Mh = a.M + static_cast<long long>(h) * a.d_v * a.d_n;
    for (int i = t; i < a.d_v; i += 32)
      bulk_g2s(Ms + i * ldm, Mh + static_cast<long long>(i) * a.d_n, row_bytes, &bar);
    for (int bt = t; bt < nb; bt += 32)
      bulk_g2s(qs + bt * a.d_n, a.q_c + (static_cast<long long>(b0 + bt) * a.H + h) * a.d_n, row_bytes, &bar);
  }
  if (!mbar_wait_bounded(&bar, 0)) {
    if (t == 0) flag_error(a.err, GVA_DEVERR_TIMEOUT);
    return;
  }

  // thread -> output row i (rows split over threads) and a set of sequences (when d_v is
  // smaller than the thread count, the sequences are split over `sets` threads per row)
  const int sets = a.d_v < kGemvThreads ? kGemvThreads / a.d_v : 1;
  const int rows_per_pass = kGemvThreads / sets;
  const int set = t / rows_per_pass;
  for (int i = t % rows_per_pass; i < a.d_v; i += rows_per_pass) {
    float acc[kAbsorbSeqs];
#pragma unroll
    for (int j = 0; j < kAbsorbSeqs; ++j) acc[j] = 0.f;
    const float* mrow = Ms + i * ldm;
    for (int k = 0; k < a.d_n; k += 4) {
      const float4 m4 = *reinterpret_cast<const float4*>(mrow + k);
#pragma unroll
      for (int j = 0; j < kAbsorbSeqs; ++j) {
        const int bt = set + j * sets;
        if (bt < nb) {
          const float4 q4 = *reinterpret_cast<const float4*>(qs + bt * a.d_n + k);
          acc[j] = fmaf(m4.x, q4.x, acc[j]);
          acc[j] = fmaf(m4.y, q4.y, acc[j]);
          acc[j] = fmaf(m4.z, q4.z, acc[j]);
          acc[j] = fmaf(m4.w, q4.w, acc[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kAbsorbSeqs; ++j) {
      const int bt = set + j * sets;
      if (bt < nb) a.q_abs[(static_cast<long long>(b0 + bt) * a.H + h) * a.d_v + i] = acc[j];
    }
  }
}

}  // namespace

cudaError_t launch_absorb(const gva_ctx* ctx, int B, const float* q_c, const float* q_r,
                          const int32_t* pos_q, const float* M, float* q_abs, float* q_rot,
                          cudaStream_t stream) {
  AbsorbArgs a;
  a.q_c = q_c;
  a.q_r = q_r;
  a.pos_q = pos_q;
  a.M = M;
  a.q_abs = q_abs;
  a.q_rot = q_rot;
  a.B = B;
  a.H = ctx->dims.H;
  a.d_v = ctx->dims.d_v;
  a.d_n = ctx->dims.d_n;
  a.d_r = ctx->dims.d_r;
  a.rope = ctx->d_rope;
  a.err = ctx->d_err;
  const size_t smem = sizeof(float) * (static_cast<size_t>(a.d_v) * (a.d_n + 4) + kAbsorbSeqs * a.d_n);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  static int configured[kMaxDevicesHost] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevicesHost || configured[dev] < static_cast<int>(smem)) {
    e = cudaFuncSetAttribute(absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevicesHost) configured[dev] = static_cast<int>(smem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.H, (B + kAbsorbSeqs - 1) / kAbsorbSeqs);
  cfg.blockDim = dim3(kAbsorbThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, absorb_kernel, a);
}

}  // namespace gva
