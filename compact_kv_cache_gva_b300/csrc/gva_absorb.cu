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
// round trips: one CTA per (head, 16 sequences).  Every thread first issues its loads (the
// positional query and its position; a share of M_h and of the content queries as 16-byte
// vectors), then the threads that own a positional pair load the four RoPE table rows of
// its position at once and rotate it (fp32); M_h and the queries go to shared memory and
// the GEMV runs in fp32.  Two memory round trips in all.
//
// Summation order of q'_i = sum_k M_h[i][k] q_c[k] (shared with the fused decode step, which
// forms the same values in the decode kernel's prologue): k is cut into 4-element chunks; chunk
// c goes to partial sum c mod 4, each partial accumulating its chunks in increasing k with one
// fused multiply-add per element; q'_i = (p0 + p1) + (p2 + p3).
#include "gva_device.cuh"
#include "gva_internal.h"
#include "gva_sched.cuh"

namespace gva {
namespace {

constexpr int kAbsorbThreads = 256;
constexpr int kAbsorbSeqs = 16;
constexpr int kAbsorbVecs = 8;  // 16-byte vectors of M_h and q_c held per thread per pass
constexpr long long kMaxGridY = 65535;  // largest y extent of a grid

struct AbsorbArgs {
  const float* q_c;
  const float* q_r;
  const int32_t* pos_q;     // null: row b*n + i of n rows per sequence sits at seq_lens[b] - n + i
  const int32_t* seq_lens;
  int rows_per_seq;
  const float* M;
  float* q_abs;
  float* q_rot;
  const float2* rope;  // fp32 RoPE digit table
  unsigned* err;
  int B, H, d_v, d_n, d_r;
  // Set when the kernel directly follows the library's own append of the same step (which
  // waits for all earlier work before it lets this kernel start): the wait for it is moved to
  // the kernel's end, so the two overlap, and what follows still sees both done.
  int defer_wait;
};

// Rows b0 .. b0 + 15 (those below B) of head blockIdx.x.
__device__ __forceinline__ void absorb_rows(const AbsorbArgs& a, float* sm, int b0) {
  const int ldm = a.d_n + 4;     // padded rows: conflict-free 16-byte reads by row
  float* Ms = sm;                // [d_v][d_n + 4]
  float* qs = sm + a.d_v * ldm;  // [kAbsorbSeqs][d_n + 4]
  const int h = blockIdx.x;
  const int nb = min(kAbsorbSeqs, a.B - b0);
  const int t = threadIdx.x;

  // positional slice: thread t < nb * pairs owns pair (t % pairs) of sequence b0 + t / pairs
  const int pairs = a.d_r / 2;
  const bool rot = t < nb * pairs;
  long long p = 0;
  float2 x = make_float2(0.f, 0.f);
  long long qrow = 0;
  int pi = 0;
  if (rot) {
    const int bt = t / pairs;
    pi = t - bt * pairs;
    qrow = (static_cast<long long>(b0 + bt) * a.H + h) * a.d_r;
    const int row = b0 + bt;
    p = a.pos_q ? static_cast<long long>(a.pos_q[row])
                : static_cast<long long>(a.seq_lens[row / a.rows_per_seq]) - a.rows_per_seq + row % a.rows_per_seq;
    x = *reinterpret_cast<const float2*>(a.q_r + qrow + 2 * pi);
  }

  // M_h rows and the content queries into shared memory, 16-byte vectors
  const int v4 = a.d_n / 4;
  const int nm = a.d_v * v4, nq = nb * v4, ntot = nm + nq;
  const float4* Mg = reinterpret_cast<const float4*>(a.M + static_cast<long long>(h) * a.d_v * a.d_n);
  for (int base = 0; base < ntot; base += kAbsorbThreads * kAbsorbVecs) {
    float4 r[kAbsorbVecs];
#pragma unroll
    for (int j = 0; j < kAbsorbVecs; ++j) {
      const int i = base + t + j * kAbsorbThreads;
      if (i < nm) {
        r[j] = Mg[i];
      } else if (i < ntot) {
        const int bt = (i - nm) / v4, c = (i - nm) - bt * v4;
        r[j] = reinterpret_cast<const float4*>(a.q_c + (static_cast<long long>(b0 + bt) * a.H + h) * a.d_n)[c];
      }
    }
    if (base == 0 && rot) {  // the rotation overlaps the first pass's loads
      float c = 1.f, s = 0.f;
      if (p >= 0)
        rope_cos_sin_f32(a.rope, pairs, p, pi, c, s);
      else if (pi == 0)
        flag_error(a.err, GVA_DEVERR_POSITION);  // left unrotated
      float2 y;
      rope_rotate_f32(x.x, x.y, c, s, y.x, y.y);
      *reinterpret_cast<float2*>(a.q_rot + qrow + 2 * pi) = y;
    }
#pragma unroll
    for (int j = 0; j < kAbsorbVecs; ++j) {
      const int i = base + t + j * kAbsorbThreads;
      if (i < nm) {
        const int row = i / v4, c = i - row * v4;
        *reinterpret_cast<float4*>(Ms + row * ldm + 4 * c) = r[j];
      } else if (i < ntot) {
        const int bt = (i - nm) / v4, c = (i - nm) - bt * v4;
        *reinterpret_cast<float4*>(qs + bt * ldm + 4 * c) = r[j];
      }
    }
  }
  __syncthreads();

  // Register tiles of 2 rows x 4 sequences per thread: rows i and i + d_v/2 (the two rows'
  // 16-byte reads stay conflict-free across a warp), sequences 4s..4s+3 (the warp shares s,
  // so the query reads are broadcasts).  6 shared-memory reads feed 32 FMAs; each output
  // keeps its four partial sums (chunk c of k into partial c mod 4).
  const int half = a.d_v / 2;
  const int nsb = (nb + 3) / 4;
  const int nchunk = a.d_n / 4;
  for (int o = t; o < half * nsb; o += kAbsorbThreads) {
    const int i = o % half, sb = o / half;
    const float* m0 = Ms + i * ldm;
    const float* m1 = Ms + (i + half) * ldm;
    float acc[2][4][4];  // [row][sequence][partial]
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][j][e] = 0.f;
    auto chunk = [&](int c, int e) {  // chunk c (elements 4c..4c+3) into partial e
      const float4 ma = *reinterpret_cast<const float4*>(m0 + 4 * c);
      const float4 mb = *reinterpret_cast<const float4*>(m1 + 4 * c);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int bt = min(4 * sb + j, nb - 1);  // rows past nb repeat a valid one, unused
        const float4 q4 = *reinterpret_cast<const float4*>(qs + bt * ldm + 4 * c);
        acc[0][j][e] = fmaf(ma.x, q4.x, acc[0][j][e]);
        acc[0][j][e] = fmaf(ma.y, q4.y, acc[0][j][e]);
        acc[0][j][e] = fmaf(ma.z, q4.z, acc[0][j][e]);
        acc[0][j][e] = fmaf(ma.w, q4.w, acc[0][j][e]);
        acc[1][j][e] = fmaf(mb.x, q4.x, acc[1][j][e]);
        acc[1][j][e] = fmaf(mb.y, q4.y, acc[1][j][e]);
        acc[1][j][e] = fmaf(mb.z, q4.z, acc[1][j][e]);
        acc[1][j][e] = fmaf(mb.w, q4.w, acc[1][j][e]);
      }
    };
    int c = 0;
    for (; c + 4 <= nchunk; c += 4) {
#pragma unroll
      for (int e = 0; e < 4; ++e) chunk(c + e, e);
    }
    if (c < nchunk) chunk(c, 0);
    if (c + 1 < nchunk) chunk(c + 1, 1);
    if (c + 2 < nchunk) chunk(c + 2, 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int bt = 4 * sb + j;
      if (bt < nb) {
        float* dst = a.q_abs + (static_cast<long long>(b0 + bt) * a.H + h) * a.d_v;
        dst[i] = (acc[0][j][0] + acc[0][j][1]) + (acc[0][j][2] + acc[0][j][3]);
        dst[i + half] = (acc[1][j][0] + acc[1][j][1]) + (acc[1][j][2] + acc[1][j][3]);
      }
    }
  }
}

// One CTA per (head, block of 16 rows); a grid narrower than the row blocks (its y extent
// is capped at 65535) takes them in strides, so any row count runs.
__global__ void __launch_bounds__(kAbsorbThreads) absorb_kernel(const AbsorbArgs a) {
  extern __shared__ __align__(16) float sm[];
  if (!a.defer_wait) griddep_wait();
  griddep_launch_dependents();
  for (long long yb = blockIdx.y; yb * kAbsorbSeqs < a.B; yb += gridDim.y) {
    if (yb != blockIdx.y) __syncthreads();  // the previous rows' shared memory has been read
    absorb_rows(a, sm, static_cast<int>(yb * kAbsorbSeqs));
  }
  if (a.defer_wait) griddep_wait();
}

}  // namespace

cudaError_t launch_absorb(const gva_ctx* ctx, int B, const float* q_c, const float* q_r,
                          const int32_t* pos_q, const float* M, float* q_abs, float* q_rot,
                          cudaStream_t stream, const int32_t* seq_lens, bool after_own_append,
                          int rows_per_seq) {
  AbsorbArgs a;
  a.rows_per_seq = rows_per_seq;
  a.defer_wait = after_own_append ? 1 : 0;
  a.q_c = q_c;
  a.q_r = q_r;
  a.pos_q = pos_q;
  a.seq_lens = seq_lens;
  a.M = M;
  a.q_abs = q_abs;
  a.q_rot = q_rot;
  a.B = B;
  a.H = ctx->dims.H;
  a.d_v = ctx->dims.d_v;
  a.d_n = ctx->dims.d_n;
  a.d_r = ctx->dims.d_r;
  a.rope = ctx->d_rope32;
  a.err = ctx->d_err;
  const size_t smem = sizeof(float) * static_cast<size_t>(a.d_v + kAbsorbSeqs) * (a.d_n + 4);
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
  const long long row_blocks = (static_cast<long long>(B) + kAbsorbSeqs - 1) / kAbsorbSeqs;
  cfg.gridDim = dim3(a.H, static_cast<unsigned>(row_blocks < kMaxGridY ? row_blocks : kMaxGridY));
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
