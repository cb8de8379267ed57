// gva_decode_fma.cu -- split-T decode attention over the compact GVA cache on the CUDA
// cores (fp32 FMA), and the combine pass shared by every decode kernel.
//
// What is computed (ai-feeds.com summary "Grouped Value Attention:通过按需 key 重建实现高效
// KV 缓存", section 方法; review "[논문리뷰] Grouped Value Attention", section 3): for head h
// of value group g, s_j = scale * (q'_h . v_j + q~_r,h . k_r,j) over the cached tokens,
// softmax, o_h = sum_j p_j v_j.  The content key is never built: q'_h already holds M_h.
//
// Work split: a CTA owns (chunk of whole 64-token blocks, value group g, sequence b); each
// of its 4 warps takes every 4th block of the chunk through a private 2-stage ring filled
// by the bulk-copy engine (one copy for the group's [64][d_v] value tile, one for the
// shared [64][d_r] positional-key tile).  The tile is read once from HBM and used by all
// H/G heads of the group.  Lanes own d_v/32 consecutive value columns; scores of 8 tokens
// are finished with a transposing butterfly (9 shuffles for 8 tokens), softmax is online
// (running max and sum, log2 domain), and warps merge in shared memory at the end.  The
// partial (m, l, weighted sum) of each (b, chunk, h) goes to the workspace; the combine
// kernel merges the chunks of a sequence.
#include <math.h>

#include "gva_device.cuh"
#include "gva_internal.h"

namespace gva {
namespace {

constexpr int kFmaWarps = 4;
constexpr int kFmaThreads = 32 * kFmaWarps;
constexpr int kFmaStages = 2;
constexpr int kBarBytes = 128;  // mbarriers of all warps, ahead of the rings

template <typename T, int DV, bool SEPK>
struct FmaLayout {
  static constexpr int kTileBytes = kBlockTokens * DV * static_cast<int>(sizeof(T));
  static __host__ __device__ int kr_bytes(int d_r) {
    return kBlockTokens * d_r * static_cast<int>(sizeof(T));  // multiple of 256 for even d_r
  }
  static __host__ __device__ int stage_bytes(int d_r) {
    return kTileBytes * (SEPK ? 2 : 1) + (SEPK ? 0 : kr_bytes(d_r));
  }
  static __host__ __device__ int smem_bytes(int d_r) {
    return kBarBytes + kFmaWarps * kFmaStages * stage_bytes(d_r);
  }
};

// EPL consecutive elements of a row, converted to float.
template <typename T, int EPL>
__device__ __forceinline__ void load_row(const T* p, float (&x)[EPL]);

template <>
__device__ __forceinline__ void load_row<float, 1>(const float* p, float (&x)[1]) { x[0] = *p; }
template <>
__device__ __forceinline__ void load_row<float, 2>(const float* p, float (&x)[2]) {
  const float2 v = *reinterpret_cast<const float2*>(p);
  x[0] = v.x;
  x[1] = v.y;
}
template <>
__device__ __forceinline__ void load_row<float, 4>(const float* p, float (&x)[4]) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x;
  x[1] = v.y;
  x[2] = v.z;
  x[3] = v.w;
}
template <>
__device__ __forceinline__ void load_row<__nv_bfloat16, 1>(const __nv_bfloat16* p, float (&x)[1]) {
  x[0] = bf16_bits_to_float(*reinterpret_cast<const unsigned short*>(p));
}
template <>
__device__ __forceinline__ void load_row<__nv_bfloat16, 2>(const __nv_bfloat16* p, float (&x)[2]) {
  bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(p), x[0], x[1]);
}
template <>
__device__ __forceinline__ void load_row<__nv_bfloat16, 4>(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  bf16x2_to_float2(v.x, x[0], x[1]);
  bf16x2_to_float2(v.y, x[2], x[3]);
}

__device__ __forceinline__ float elem_to_float(float v) { return v; }
__device__ __forceinline__ float elem_to_float(__nv_bfloat16 v) { return __bfloat162float(v); }

// Transposing butterfly: lane holds partial dot products v[0..7] of tokens 0..7 (its own
// columns); returns the full 32-lane sum for token (lane >> 2) & 7.  Each step swaps half
// of the remaining values with the partner lane, so only 4 + 2 + 1 + 2 shuffles are spent.
__device__ __forceinline__ float transpose_reduce8(const float (&v)[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b4 ? v[i] : v[i + 4];
    const float keep = b4 ? v[i + 4] : v[i];
    a[i] = keep + __shfl_xor_sync(kFullMask, send, 16);
  }
  float c[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b3 ? a[i] : a[i + 2];
    const float keep = b3 ? a[i + 2] : a[i];
    c[i] = keep + __shfl_xor_sync(kFullMask, send, 8);
  }
  const float send = b2 ? c[0] : c[1];
  const float keep = b2 ? c[1] : c[0];
  float d = keep + __shfl_xor_sync(kFullMask, send, 4);
  d += __shfl_xor_sync(kFullMask, d, 2);
  d += __shfl_xor_sync(kFullMask, d, 1);
  return d;
}

template <typename T, int DV, int R, bool SEPK>
__global__ void __launch_bounds__(kFmaThreads) decode_fma_kernel(const DecodeArgs a) {
  using L = FmaLayout<T, DV, SEPK>;
  constexpr int EPL = DV / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;

  const int T_b = a.seq_lens[b];
  if (T_b <= 0 || T_b > a.max_seq_len) {
    if (c == 0 && g == 0 && threadIdx.x == 0) flag_error(a.err, GVA_DEVERR_SEQ_LEN);
    return;
  }
  const int nt = (T_b + kBlockTokens - 1) / kBlockTokens;
  const int t0 = c * a.chunk_tiles;
  if (t0 >= nt) return;
  const int t1 = min(nt, t0 + a.chunk_tiles);
  const int d_r = SEPK ? 0 : a.d_r;
  const int stage_bytes = L::stage_bytes(d_r);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + warp * kFmaStages;
  unsigned char* ring = smem + kBarBytes + warp * kFmaStages * stage_bytes;

  // Lane slice of the queries of the R heads of group g, pre-scaled by scale*log2(e).
  const int h0 = g * R;
  float qv[R][EPL], qk[R];
#pragma unroll
  for (int h = 0; h < R; ++h) {
    const long long row = static_cast<long long>(b) * a.H + h0 + h;
    load_row<float, EPL>(a.q_abs + row * DV + lane * EPL, qv[h]);
#pragma unroll
    for (int e = 0; e < EPL; ++e) qv[h][e] *= a.scale_log2;
    qk[h] = (lane < d_r) ? a.q_rot[row * d_r + lane] * a.scale_log2 : 0.f;
  }

  const int n_my = (t0 + warp < t1) ? (t1 - t0 - warp + kFmaWarps - 1) / kFmaWarps : 0;
  if (lane == 0) {
    for (int s = 0; s < kFmaStages; ++s) mbar_init(&bars[s], 1);
    mbar_init_fence();
  }
  __syncwarp();

  auto block_id = [&](int t) -> int {
    if (t >= a.max_blocks) return -1;
    const int blk = a.block_table[static_cast<long long>(b) * a.max_blocks + t];
    return (blk >= 0 && blk < a.num_blocks) ? blk : -1;
  };
  // Lane 0: start the copies of this warp's k-th tile into stage k % kFmaStages.
  auto issue = [&](int k) {
    const int s = k % kFmaStages;
    const int t = t0 + warp + k * kFmaWarps;
    const int blk = block_id(t);
    if (blk < 0) {
      flag_error(a.err, t >= a.max_blocks ? GVA_DEVERR_POSITION : GVA_DEVERR_BLOCK_ID);
      mbar_arrive(&bars[s]);  // completes the phase with no data; the tile is skipped
      return;
    }
    unsigned char* st = ring + s * stage_bytes;
    mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(stage_bytes));
    const size_t vofs = (static_cast<size_t>(blk) * a.G + g) * kBlockTokens * DV;
    bulk_g2s(st, static_cast<const T*>(a.v_pool) + vofs, L::kTileBytes, &bars[s]);
    if (SEPK) bulk_g2s(st + L::kTileBytes, static_cast<const T*>(a.k_pool) + vofs, L::kTileBytes, &bars[s]);
    if (!SEPK && d_r > 0)
      bulk_g2s(st + L::kTileBytes, static_cast<const T*>(a.kr_pool) + static_cast<size_t>(blk) * kBlockTokens * d_r,
               L::kr_bytes(d_r), &bars[s]);
  };

  if (lane == 0)
    for (int k = 0; k < min(kFmaStages, n_my); ++k) issue(k);

  float m[R], l[R], o[R][EPL];
#pragma unroll
  for (int h = 0; h < R; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[h][e] = 0.f;
  }
  const int tk = (lane >> 2) & 7;  // token of the 8-token group whose score this lane ends with

  int k = 0;
  bool ok = true;
  for (; k < n_my; ++k) {
    const int s = k % kFmaStages;
    const bool got = mbar_wait_bounded(&bars[s], (k / kFmaStages) & 1);
    if (!__all_sync(kFullMask, got)) {
      ok = false;
      break;
    }
    const int t = t0 + warp + k * kFmaWarps;
    if (block_id(t) >= 0) {
      const T* Vs = reinterpret_cast<const T*>(ring + s * stage_bytes);
      const T* Ks = SEPK ? Vs + kBlockTokens * DV : Vs;
      const T* KRs = Vs + kBlockTokens * DV;
      const int nv = min(kBlockTokens, T_b - t * kBlockTokens);
      for (int jb = 0; jb < nv; jb += 8) {
        const int nk = min(8, nv - jb);
        float part[R][8];
        float vk[SEPK ? 1 : 8][EPL];
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) {
          float kv[EPL];
          load_row<T, EPL>(Ks + (jb + k2) * DV + lane * EPL, kv);
          float kr = 0.f;
          if (!SEPK && lane < d_r) kr = elem_to_float(KRs[(jb + k2) * d_r + lane]);
#pragma unroll
          for (int h = 0; h < R; ++h) {
            float acc = qk[h] * kr;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc = fmaf(qv[h][e], kv[e], acc);
            part[h][k2] = acc;
          }
          if (!SEPK) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) vk[SEPK ? 0 : k2][e] = kv[e];
          }
        }
        float p[R];
#pragma unroll
        for (int h = 0; h < R; ++h) {
          float sc = transpose_reduce8(part[h], lane);
          sc = (tk < nk) ? sc : -INFINITY;
          float mx = fmaxf(sc, __shfl_xor_sync(kFullMask, sc, 4));
          mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 16));
          const float mn = fmaxf(m[h], mx);
          const float alpha = exp2f(m[h] - mn);
          p[h] = (tk < nk) ? exp2f(sc - mn) : 0.f;
          l[h] = fmaf(l[h], alpha, p[h]);
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[h][e] *= alpha;
          m[h] = mn;
        }
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) {
          if (k2 < nk) {
            float vv[EPL];
            if (SEPK) {
              load_row<T, EPL>(Vs + (jb + k2) * DV + lane * EPL, vv);
            } else {
#pragma unroll
              for (int e = 0; e < EPL; ++e) vv[e] = vk[SEPK ? 0 : k2][e];
            }
#pragma unroll
            for (int h = 0; h < R; ++h) {
              const float pk = __shfl_sync(kFullMask, p[h], k2 * 4);
#pragma unroll
              for (int e = 0; e < EPL; ++e) o[h][e] = fmaf(pk, vv[e], o[h][e]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && k + kFmaStages < n_my) {
      fence_proxy_async_smem();
      issue(k + kFmaStages);
    }
  }
  if (!ok) {
    // Report, then wait (bounded) for this warp's copies still in flight before the ring
    // memory is reused below.
    if (lane == 0) flag_error(a.err, GVA_DEVERR_TIMEOUT);
    for (int kk = k; kk < min(n_my, k + kFmaStages); ++kk)
      mbar_wait_bounded(&bars[kk % kFmaStages], (kk / kFmaStages) & 1);
    __syncwarp();
  }

  // Lanes sharing (lane >> 2) hold copies of one token slot's running sum.
#pragma unroll
  for (int h = 0; h < R; ++h) {
    l[h] += __shfl_xor_sync(kFullMask, l[h], 4);
    l[h] += __shfl_xor_sync(kFullMask, l[h], 8);
    l[h] += __shfl_xor_sync(kFullMask, l[h], 16);
  }

  // Merge the warps' states in shared memory (each warp writes into its own drained ring).
  constexpr int kRec = DV + 4;
  float* mine = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int h = 0; h < R; ++h) {
    if (lane == 0) {
      mine[h * kRec] = m[h];
      mine[h * kRec + 1] = l[h];
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) mine[h * kRec + 4 + lane * EPL + e] = o[h][e];
  }
  __syncthreads();
  const size_t rec_stride = partial_stride_floats(DV);
  for (int idx = threadIdx.x; idx < R * DV; idx += kFmaThreads) {
    const int h = idx / DV, d = idx - h * DV;
    float Mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kFmaWarps; ++w)
      Mx = fmaxf(Mx, reinterpret_cast<const float*>(smem + kBarBytes + w * kFmaStages * stage_bytes)[h * kRec]);
    float Ls = 0.f, Os = 0.f;
    if (Mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kFmaWarps; ++w) {
        const float* ws = reinterpret_cast<const float*>(smem + kBarBytes + w * kFmaStages * stage_bytes) + h * kRec;
        const float sc = exp2f(ws[0] - Mx);
        Ls = fmaf(sc, ws[1], Ls);
        Os = fmaf(sc, ws[4 + d], Os);
      }
    }
    float* rec = a.part + ((static_cast<size_t>(b) * a.n_chunks + c) * a.H + h0 + h) * rec_stride;
    if (d == 0) {
      rec[0] = Mx;
      rec[1] = Ls;
    }
    rec[4 + d] = Os;
  }
}

// Merges the chunk partials of one (b, h):  M = max m_c,  out = sum 2^(m_c-M) u_c / sum 2^(m_c-M) l_c.
__global__ void combine_kernel(const DecodeArgs a) {
  const int h = blockIdx.x, b = blockIdx.y;
  float* out = a.out + (static_cast<size_t>(b) * a.H + h) * a.d_v;
  const int T_b = a.seq_lens[b];
  if (T_b <= 0 || T_b > a.max_seq_len) {
    for (int d = threadIdx.x; d < a.d_v; d += blockDim.x) out[d] = 0.f;
    return;
  }
  const int nt = (T_b + kBlockTokens - 1) / kBlockTokens;
  const int nc = (nt + a.chunk_tiles - 1) / a.chunk_tiles;
  const size_t rs = partial_stride_floats(a.d_v);
  const float* rec0 = a.part + (static_cast<size_t>(b) * a.n_chunks * a.H + h) * rs;
  const size_t cs = static_cast<size_t>(a.H) * rs;
  float Mx = -INFINITY;
  for (int ci = 0; ci < nc; ++ci) Mx = fmaxf(Mx, rec0[ci * cs]);
  for (int d = threadIdx.x; d < a.d_v; d += blockDim.x) {
    float Ls = 0.f, Os = 0.f;
    if (Mx != -INFINITY) {
      for (int ci = 0; ci < nc; ++ci) {
        const float* r = rec0 + ci * cs;
        const float w = exp2f(r[0] - Mx);
        Ls = fmaf(w, r[1], Ls);
        Os = fmaf(w, r[4 + d], Os);
      }
    }
    out[d] = Ls > 0.f ? Os / Ls : 0.f;
  }
}

template <typename T, int DV, int R, bool SEPK>
cudaError_t launch_fma_t(const DecodeArgs& a, cudaStream_t stream) {
  using L = FmaLayout<T, DV, SEPK>;
  const int smem = L::smem_bytes(SEPK ? 0 : a.d_r);
  static int configured[kMaxDevices] = {};  // per instantiation and device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || configured[dev] < smem) {
    e = cudaFuncSetAttribute(decode_fma_kernel<T, DV, R, SEPK>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) configured[dev] = smem;
  }
  dim3 grid(a.n_chunks, a.G, a.B);
  decode_fma_kernel<T, DV, R, SEPK><<<grid, kFmaThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int DV, bool SEPK>
cudaError_t dispatch_r(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.H / a.G) {
    case 1: return launch_fma_t<T, DV, 1, SEPK>(a, stream);
    case 2: return launch_fma_t<T, DV, 2, SEPK>(a, stream);
    case 4: return launch_fma_t<T, DV, 4, SEPK>(a, stream);
    case 8: return launch_fma_t<T, DV, 8, SEPK>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, bool SEPK>
cudaError_t dispatch_dv(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.d_v) {
    case 32: return dispatch_r<T, 32, SEPK>(a, stream);
    case 64: return dispatch_r<T, 64, SEPK>(a, stream);
    case 128: return dispatch_r<T, 128, SEPK>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

int fma_smem_bytes(const gva_dims& d, bool sep_k) {
  const int es = d.cache_dtype == GVA_F32 ? 4 : 2;
  const int tile = kBlockTokens * d.d_v * es;
  const int stage = tile * (sep_k ? 2 : 1) + (sep_k ? 0 : kBlockTokens * d.d_r * es);
  return kBarBytes + kFmaWarps * kFmaStages * stage;
}

}  // namespace

bool fma_supported(const gva_dims& d, bool sep_k) {
  const int r = d.H / d.G;
  if (!(d.d_v == 32 || d.d_v == 64 || d.d_v == 128)) return false;
  if (!(r == 1 || r == 2 || r == 4 || r == 8)) return false;
  if (d.d_r < 0 || d.d_r > 32 || (d.d_r & 1)) return false;
  if (sep_k && d.d_r != 0) return false;
  return fma_smem_bytes(d, sep_k) <= 227 * 1024;
}

int fma_ctas_per_sm(const gva_dims& d, bool sep_k) {
  const int smem = fma_smem_bytes(d, sep_k);
  int per_sm = (228 * 1024) / (smem + 1024);  // 1 KB per CTA reserved by the hardware
  if (per_sm > 16) per_sm = 16;
  return per_sm < 1 ? 1 : per_sm;
}

cudaError_t launch_decode_fma(const DecodeArgs& a, int cache_dtype, bool sep_k,
                              cudaStream_t stream) {
  if (cache_dtype == GVA_F32)
    return sep_k ? dispatch_dv<float, true>(a, stream) : dispatch_dv<float, false>(a, stream);
  return sep_k ? dispatch_dv<__nv_bfloat16, true>(a, stream)
               : dispatch_dv<__nv_bfloat16, false>(a, stream);
}

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t stream) {
  int threads = ((a.d_v + 31) / 32) * 32;
  if (threads > 256) threads = 256;
  combine_kernel<<<dim3(a.H, a.B), threads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gva
