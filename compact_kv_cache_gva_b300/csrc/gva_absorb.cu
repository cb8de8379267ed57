// gva_absorb.cu -- per-step query preparation for GVA decode.
//
// Absorption: the key map M_h (K_h = V_g(h) M_h) is folded into the query, q' = M_h q_c, so
// the content score becomes one inner product with the cached value and no content key is
// ever built (ai-feeds.com summary "Grouped Value Attention:通过按需 key 重建实现高效 KV
// 缓存", section 方法: Q' = Q M^T; m.szthrk.cn explainer, section "GVA 的正式方案").
// Decoupled RoPE: only the positional slice of the query is rotated, at the query's
// position (review "[논문리뷰] Grouped Value Attention", section 3).
//
// One CTA per (head, 16 sequences): M_h rows are read through L1 as 16-byte vectors and the
// 16 content queries sit in shared memory (broadcast reads); fp32 FMA in k order.
#include "gva_device.cuh"
#include "gva_internal.h"

namespace gva {
namespace {

constexpr int kAbsorbThreads = 128;
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
  extern __shared__ __align__(16) float qs[];  // [kAbsorbSeqs][d_n]
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * kAbsorbSeqs;
  const int nb = min(kAbsorbSeqs, a.B - b0);

  for (int idx = threadIdx.x; idx < nb * a.d_n; idx += kAbsorbThreads) {
    const int bt = idx / a.d_n, k = idx - bt * a.d_n;
    qs[bt * a.d_n + k] = a.q_c[(static_cast<long long>(b0 + bt) * a.H + h) * a.d_n + k];
  }
  __syncthreads();

  for (int i = threadIdx.x; i < a.d_v; i += kAbsorbThreads) {
    float acc[kAbsorbSeqs];
#pragma unroll
    for (int bt = 0; bt < kAbsorbSeqs; ++bt) acc[bt] = 0.f;
    const float* row = a.M + (static_cast<long long>(h) * a.d_v + i) * a.d_n;
    for (int k = 0; k < a.d_n; k += 4) {
      const float4 m4 = *reinterpret_cast<const float4*>(row + k);
#pragma unroll
      for (int bt = 0; bt < kAbsorbSeqs; ++bt) {
        if (bt < nb) {
          const float4 q4 = *reinterpret_cast<const float4*>(qs + bt * a.d_n + k);
          acc[bt] = fmaf(m4.x, q4.x, acc[bt]);
          acc[bt] = fmaf(m4.y, q4.y, acc[bt]);
          acc[bt] = fmaf(m4.z, q4.z, acc[bt]);
          acc[bt] = fmaf(m4.w, q4.w, acc[bt]);
        }
      }
    }
#pragma unroll
    for (int bt = 0; bt < kAbsorbSeqs; ++bt)
      if (bt < nb) a.q_abs[(static_cast<long long>(b0 + bt) * a.H + h) * a.d_v + i] = acc[bt];
  }

  // Positional slice of the query, rotated at pos_q[b] in fp64 (digit-table rotation).
  const int pairs = a.d_r / 2;
  for (int idx = threadIdx.x; idx < nb * pairs; idx += kAbsorbThreads) {
    const int bt = idx / pairs, i = idx - bt * pairs;
    const long long row = (static_cast<long long>(b0 + bt) * a.H + h) * a.d_r;
    const double x0 = a.q_r[row + 2 * i], x1 = a.q_r[row + 2 * i + 1];
    const long long p = a.pos_q[b0 + bt];
    double c = 1.0, s = 0.0;
    if (p >= 0)
      rope_cos_sin(a.rope, pairs, p, i, c, s);
    else if (i == 0)
      flag_error(a.err, GVA_DEVERR_POSITION);  // left unrotated
    a.q_rot[row + 2 * i] = __double2float_rn(__dsub_rn(__dmul_rn(x0, c), __dmul_rn(x1, s)));
    a.q_rot[row + 2 * i + 1] = __double2float_rn(__dadd_rn(__dmul_rn(x0, s), __dmul_rn(x1, c)));
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
  const size_t smem = sizeof(float) * kAbsorbSeqs * a.d_n;
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid(a.H, (B + kAbsorbSeqs - 1) / kAbsorbSeqs);
  absorb_kernel<<<grid, kAbsorbThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gva
