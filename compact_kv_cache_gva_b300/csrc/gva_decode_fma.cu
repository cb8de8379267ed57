// gva_decode_fma.cu -- split-T decode attention over the compact GVA cache on the CUDA
// cores (fp32 FMA): every cache dtype, and the fallback for shapes the tensor-core kernel
// does not cover.
//
// What is computed (ai-feeds.com summary "Grouped Value Attention:通过按需 key 重建实现高效
// KV 缓存", section 方法; review "[논문리뷰] Grouped Value Attention", section 3): for head h
// of value group g, s_j = scale * (q'_h . v_j + q~_r,h . k_r,j) over the cached tokens,
// softmax, o_h = sum_j p_j v_j.  The content key is never built: q'_h already holds M_h.
//
// Work split: each warp takes a balanced range of (sequence, group, 64-token tile) units
// (gva_sched.cuh) through a private 2-stage ring filled by the bulk-copy engine (one copy
// for the group's [64][d_v] value tile, one for the shared [64][d_r] positional-key tile).
// The tile is read once from HBM and used by all H/G heads of the group.  Lanes own d_v/32
// consecutive value columns; scores of 8 tokens are finished with a transposing butterfly
// (9 shuffles for 8 tokens), softmax is online (running max and sum, log2 domain), and the
// warp writes one partial record per (sequence, group) it touched; the combine kernel
// (gva_decode_combine.cu) merges them.
#include <math.h>

#include "gva_device.cuh"
#include "gva_internal.h"
#include "gva_sched.cuh"

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
  const int d_r = SEPK ? 0 : a.d_r;
  const int stage_bytes = L::stage_bytes(d_r);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + warp * kFmaStages;
  unsigned char* ring = smem + kBarBytes + warp * kFmaStages * stage_bytes;
  int* cum = reinterpret_cast<int*>(smem + L::smem_bytes(d_r));

  if (lane == 0) {
    for (int s = 0; s < kFmaStages; ++s) mbar_init(&bars[s], 1);
    mbar_init_fence();
  }
  griddep_wait();
  build_prefix<kFmaThreads>(a, cum);
  griddep_launch_dependents();

  // one range per warp (n_groups = warps, group_warps = 1): record index gw + f
  const long long U = static_cast<long long>(a.G) * cum[a.B];
  const long long gw = static_cast<long long>(blockIdx.x) * kFmaWarps + warp;
  const long long u0 = range_begin(gw, U, a.n_groups), u1 = range_begin(gw + 1, U, a.n_groups);
  const int n = static_cast<int>(u1 - u0);
  if (n <= 0) return;  // warp-uniform; no CTA-wide barrier follows
  float* recs = a.part + header_bytes(a.B) / 4;
  constexpr int kRec = DV + 4;

  UnitCursor ic = cursor_at(u0, cum, a.B, a.G);
  UnitCursor cc = ic;

  auto block_id = [&](int b, int t) -> int {
    if (t >= a.max_blocks) return -1;
    const int blk = a.block_table[static_cast<long long>(b) * a.max_blocks + t];
    return (blk >= 0 && blk < a.num_blocks) ? blk : -1;
  };
  auto issue = [&](int k) {  // lane 0: this warp's k-th unit into stage k % kFmaStages
    const int s = k % kFmaStages;
    const int blk = block_id(ic.b, ic.t);
    if (blk < 0) {
      flag_error(a.err, ic.t >= a.max_blocks ? GVA_DEVERR_POSITION : GVA_DEVERR_BLOCK_ID);
      mbar_arrive(&bars[s]);  // completes the phase with no data; the tile is skipped
    } else {
      unsigned char* st = ring + s * stage_bytes;
      mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(stage_bytes));
      const size_t vofs = (static_cast<size_t>(blk) * a.G + ic.g) * kBlockTokens * DV;
      bulk_g2s(st, static_cast<const T*>(a.v_pool) + vofs, L::kTileBytes, &bars[s]);
      if (SEPK) bulk_g2s(st + L::kTileBytes, static_cast<const T*>(a.k_pool) + vofs, L::kTileBytes, &bars[s]);
      if (!SEPK && d_r > 0)
        bulk_g2s(st + L::kTileBytes,
                 static_cast<const T*>(a.kr_pool) + static_cast<size_t>(blk) * kBlockTokens * d_r,
                 L::kr_bytes(d_r), &bars[s]);
    }
    cursor_next(ic, cum, a.B, a.G);
  };
  if (lane == 0)
    for (int k = 0; k < min(kFmaStages, n); ++k) issue(k);

  // Lane slice of the queries of the R heads of the current group, pre-scaled by
  // scale*log2(e).
  float qv[R][EPL], qk[R];
  auto load_q = [&](int b, int g) {
#pragma unroll
    for (int h = 0; h < R; ++h) {
      const long long row = static_cast<long long>(b) * a.H + g * R + h;
      load_row<float, EPL>(a.q_abs + row * DV + lane * EPL, qv[h]);
#pragma unroll
      for (int e = 0; e < EPL; ++e) qv[h][e] *= a.scale_log2;
      qk[h] = (lane < d_r) ? a.q_rot[row * d_r + lane] * a.scale_log2 : 0.f;
    }
  };
  float m[R], l[R], o[R][EPL];
  auto reset_state = [&]() {
#pragma unroll
    for (int h = 0; h < R; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[h][e] = 0.f;
    }
  };
  // Partial record of segment f: lanes sharing (lane >> 2) hold copies of one token slot's
  // running sum, so the sum runs over lanes 4 apart.
  auto flush = [&](long long f) {
    float* rec = recs + (gw + f) * R * kRec;
#pragma unroll
    for (int h = 0; h < R; ++h) {
      float lt = l[h];
      lt += __shfl_xor_sync(kFullMask, lt, 4);
      lt += __shfl_xor_sync(kFullMask, lt, 8);
      lt += __shfl_xor_sync(kFullMask, lt, 16);
      if (lane == 0) {
        rec[h * kRec] = m[h];
        rec[h * kRec + 1] = lt;
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) rec[h * kRec + 4 + lane * EPL + e] = o[h][e];
    }
  };

  const int tk = (lane >> 2) & 7;  // token of the 8-token group whose score this lane ends with
  reset_state();
  load_q(cc.b, cc.g);
  int k = 0;
  bool ok = true;
  for (; k < n; ++k) {
    const int s = k % kFmaStages;
    const bool got = mbar_wait_bounded(&bars[s], (k / kFmaStages) & 1);
    if (!__all_sync(kFullMask, got)) {
      ok = false;
      break;
    }
    if (block_id(cc.b, cc.t) >= 0) {
      const T* Vs = reinterpret_cast<const T*>(ring + s * stage_bytes);
      const T* Ks = SEPK ? Vs + kBlockTokens * DV : Vs;
      const T* KRs = Vs + kBlockTokens * DV;
      const int nv = min(kBlockTokens, a.seq_lens[cc.b] - cc.t * kBlockTokens);
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
    if (lane == 0 && k + kFmaStages < n) {
      fence_proxy_async_smem();
      issue(k + kFmaStages);
    }
    if (k + 1 < n) {
      const int pb = cc.b, pg = cc.g;
      cursor_next(cc, cum, a.B, a.G);
      if (cc.b != pb || cc.g != pg) {
        flush(segment_of(pg, pb, a.B));
        reset_state();
        load_q(cc.b, cc.g);
      }
    }
  }
  if (ok) {
    flush(segment_of(cc.g, cc.b, a.B));
    return;
  }
  // Report, wait (bounded) for this warp's copies still in flight, and leave empty records
  // for every segment still owed.
  if (lane == 0) flag_error(a.err, GVA_DEVERR_TIMEOUT);
  for (int kk = k; kk < min(n, k + kFmaStages); ++kk)
    mbar_wait_bounded(&bars[kk % kFmaStages], (kk / kFmaStages) & 1);
  __syncwarp();
  reset_state();
  flush(segment_of(cc.g, cc.b, a.B));
  for (int kk = k + 1; kk < n; ++kk) {
    const int pb = cc.b, pg = cc.g;
    cursor_next(cc, cum, a.B, a.G);
    if (cc.b != pb || cc.g != pg) flush(segment_of(cc.g, cc.b, a.B));
  }
}

inline int cum_bytes(int B) { return ((B + 1) * 4 + 15) / 16 * 16; }

template <typename T, int DV, int R, bool SEPK>
cudaError_t launch_fma_t(const DecodeArgs& a, int grid, cudaStream_t stream) {
  using L = FmaLayout<T, DV, SEPK>;
  const int smem = L::smem_bytes(SEPK ? 0 : a.d_r) + cum_bytes(a.B);
  auto kern = decode_fma_kernel<T, DV, R, SEPK>;
  static int configured[kMaxDevices] = {};  // per instantiation and device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || configured[dev] < smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) configured[dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int DV, bool SEPK>
cudaError_t dispatch_r(const DecodeArgs& a, int grid, cudaStream_t stream) {
  switch (a.H / a.G) {
    case 1: return launch_fma_t<T, DV, 1, SEPK>(a, grid, stream);
    case 2: return launch_fma_t<T, DV, 2, SEPK>(a, grid, stream);
    case 4: return launch_fma_t<T, DV, 4, SEPK>(a, grid, stream);
    case 8: return launch_fma_t<T, DV, 8, SEPK>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, bool SEPK>
cudaError_t dispatch_dv(const DecodeArgs& a, int grid, cudaStream_t stream) {
  switch (a.d_v) {
    case 32: return dispatch_r<T, 32, SEPK>(a, grid, stream);
    case 64: return dispatch_r<T, 64, SEPK>(a, grid, stream);
    case 128: return dispatch_r<T, 128, SEPK>(a, grid, stream);
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
  if (d.cache_dtype != GVA_F32 && d.cache_dtype != GVA_BF16) return false;  // fp8: tensor-core path only
  const int r = d.H / d.G;
  if (!(d.d_v == 32 || d.d_v == 64 || d.d_v == 128)) return false;
  if (!(r == 1 || r == 2 || r == 4 || r == 8)) return false;
  if (d.d_r < 0 || d.d_r > 32 || (d.d_r & 1)) return false;
  if (sep_k && d.d_r != 0) return false;
  return fma_smem_bytes(d, sep_k) + cum_bytes(kMaxBatch) <= 227 * 1024;
}

int fma_ctas_per_sm(const gva_dims& d, bool sep_k, int B) {
  const int smem = fma_smem_bytes(d, sep_k) + cum_bytes(B);
  int per_sm = (228 * 1024) / (smem + 1024);  // 1 KB per CTA reserved by the hardware
  if (per_sm > 4) per_sm = 4;
  return per_sm < 1 ? 1 : per_sm;
}

cudaError_t launch_decode_fma(const DecodeArgs& a, int cache_dtype, bool sep_k, int grid,
                              cudaStream_t stream) {
  if (cache_dtype == GVA_F32)
    return sep_k ? dispatch_dv<float, true>(a, grid, stream) : dispatch_dv<float, false>(a, grid, stream);
  return sep_k ? dispatch_dv<__nv_bfloat16, true>(a, grid, stream)
               : dispatch_dv<__nv_bfloat16, false>(a, grid, stream);
}

}  // namespace gva
