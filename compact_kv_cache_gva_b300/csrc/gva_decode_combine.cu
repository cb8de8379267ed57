// gva_decode_combine.cu -- merges the split-T partial records of each (sequence, group).
//
// For one head, partials (m_w, l_w, u_w) over disjoint token ranges (m in the log2 domain)
// combine exactly: M = max m_w, out = sum 2^(m_w - M) u_w / sum 2^(m_w - M) l_w.  The records
// of segment f = g*B + b were written by the warps of the unit ranges that meet the
// segment's units [g*cum[B] + cum[b], ... + nt_b) (range_of, gva_sched.cuh); record index =
// (range + f)*C + warp, so a segment's records are one contiguous block, and warp_touched
// says which records of the block hold data.  One CTA per (g, b) stages that block into
// shared memory with bulk copies (one round trip per 32 KB round, usually one), then merges
// it with online rescaling between rounds.  Launched as a programmatic dependent
// of the partial kernel, so its launch overlaps that kernel's run; it waits for the partial
// results before reading them.
#include <math.h>

#include "gva_device.cuh"
#include "gva_internal.h"
#include "gva_sched.cuh"

namespace gva {
namespace {

constexpr int kCombineWarps = 8;
constexpr int kCombineThreads = 32 * kCombineWarps;
constexpr int kStageBytes = 32 * 1024;  // records staged per round (7 CTAs fit on an SM)
// records staged per round when the grid has at most one CTA per SM (fewer rounds for segments
// with many records: many consumer warps per range, or several queries per pass)
constexpr int kBigStageBytes = 208 * 1024;
constexpr int kMaxRch = kCombineThreads;  // records per round: one thread tests each for data

template <int DV, int R>
struct CombineShape {
  static constexpr int kRs = DV + 4;  // floats per head record
  static constexpr int kRch = kStageBytes / (R * kRs * 4) < 64 ? kStageBytes / (R * kRs * 4) : 64;
  static constexpr int kRchBig =
      kBigStageBytes / (R * kRs * 4) < kMaxRch ? kBigStageBytes / (R * kRs * 4) : kMaxRch;
  static constexpr int kOut = (R * DV + kCombineThreads - 1) / kCombineThreads;  // outputs per thread
};

template <int DV, int R>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const DecodeArgs a) {
  using S = CombineShape<DV, R>;
  constexpr int rs = S::kRs;
  extern __shared__ __align__(16) float stage[];  // [kRch][R][rs] records of this round
  __shared__ __align__(8) uint64_t bar;
  __shared__ float wgt[S::kRchBig][R];            // 2^(m_j - M) of the round, 0 for unused
  __shared__ unsigned char valid[S::kRchBig];     // has_data of the round's records
  const int rch = a.combine_big ? S::kRchBig : S::kRch;  // records per round
  __shared__ float Mrun[R], Lrun[R], scale_old[R];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, b = blockIdx.y;
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  // cum[b], the tiles of sequence b and cum[B]: from the lengths before the wait when this
  // call's partial pass launched this kernel (the partial pass's rule: a length outside
  // [max(1, nq), max_seq_len] counts as no tile), else from the header that pass wrote.
  __shared__ int red[2][kCombineWarps];
  __shared__ int nt_b;
  int cb = 0, nt = 0, ctot = 0;
  if (a.combine_after_partial) {
    int before = 0, total = 0;
    for (int i = tid; i < a.B; i += kCombineThreads) {
      const int T = a.seq_lens[i];
      const int t = T >= a.nq && T >= 1 && T <= a.max_seq_len ? (T + kBlockTokens - 1) / kBlockTokens : 0;
      total += t;
      if (i < b) before += t;
      if (i == b) nt_b = t;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(kFullMask, before, o);
      total += __shfl_xor_sync(kFullMask, total, o);
    }
    if (lane == 0) {
      red[0][warp] = before;
      red[1][warp] = total;
    }
    __syncthreads();
    for (int w = 0; w < kCombineWarps; ++w) {
      cb += red[0][w];
      ctot += red[1][w];
    }
    nt = nt_b;
  }
  griddep_wait();
  griddep_launch_dependents();
  const float* recs = a.part + header_bytes(a.B) / 4;
  if (!a.combine_after_partial) {
    const int* hdr = reinterpret_cast<const int*>(a.part);
    cb = hdr[b];
    nt = hdr[b + 1] - cb;
    ctot = hdr[a.B];
  }
  // sub-record hh of a record: query q0 + hh / Rh of the pass, head hh % Rh of group g
  const int Rh = a.H / a.G;
  auto out_row = [&](int hh) {
    const int qi = hh / Rh, h = hh - qi * Rh;
    return a.out + ((static_cast<long long>(b) * a.nq + a.q0 + qi) * a.H + static_cast<long long>(g) * Rh + h) * DV;
  };
  if (nt == 0) {  // length outside [max(1, nq), max_seq_len]: reported by the partial kernel
    for (int i = tid; i < R * DV; i += kCombineThreads) out_row(i / DV)[i % DV] = 0.f;
    return;
  }
  const long long U = static_cast<long long>(a.G) * ctot;
  const long long NG = a.n_groups;
  const int C = a.group_warps;
  const long long s = static_cast<long long>(g) * ctot + cb;  // first unit of (g, b)
  const long long c0 = range_of(s, U, NG);
  const int nrec = static_cast<int>(range_of(s + nt - 1, U, NG) - c0 + 1) * C;
  const long long f = segment_of(g, b, a.B);
  const float* base = recs + (c0 + f) * C * R * rs;  // record j of this segment: base + j*R*rs
  // Record j belongs to warp j % C of range c0 + j / C; it holds data only if that warp
  // streamed a unit of this segment.
  auto has_data = [&](long long j) {
    const long long c = c0 + j / C;
    const long long rb = range_begin(c, U, NG), re = range_begin(c + 1, U, NG);
    const long long lo = (s > rb ? s : rb) - rb, hi = (s + nt < re ? s + nt : re) - rb;
    return warp_touched(lo, hi, static_cast<int>(j % C), C);
  };
  if (tid < R) {
    Mrun[tid] = -INFINITY;
    Lrun[tid] = 0.f;
  }
  float acc[S::kOut];
#pragma unroll
  for (int k = 0; k < S::kOut; ++k) acc[k] = 0.f;
  __syncthreads();

  uint32_t phase = 0;
  for (int j0 = 0; j0 < nrec; j0 += rch) {
    const int n = min(rch, nrec - j0);
    if (tid == 0) {
      fence_proxy_async_smem();  // earlier reads of the stage come before the copy's writes
      const uint32_t bytes = static_cast<uint32_t>(n) * R * rs * 4;
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_g2s(stage, base + static_cast<size_t>(j0) * R * rs, bytes, &bar);
    }
    // which of the round's records hold data, once per record (three 64-bit divisions each),
    // while the copy is in flight; the barrier below publishes them
    if (tid < n) valid[tid] = has_data(j0 + tid) ? 1 : 0;
    const bool got = mbar_wait_bounded(&bar, phase);
    phase ^= 1;
    if (!__syncthreads_and(got)) {
      if (tid == 0) flag_error(a.err, GVA_DEVERR_TIMEOUT);
      return;
    }
    // round maximum per head (warp hh), then weights and the rescale of the running sums
    for (int hh = warp; hh < R; hh += kCombineWarps) {
      float mx = -INFINITY;
      for (int j = lane; j < n; j += 32) {
        if (!valid[j]) continue;
        mx = fmaxf(mx, stage[(j * R + hh) * rs]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, o));
      const float mnew = fmaxf(Mrun[hh], mx);
      float ls = 0.f;
      for (int j = lane; j < n; j += 32) {
        const float mj = stage[(j * R + hh) * rs];
        const bool use = mnew != -INFINITY && valid[j] && mj != -INFINITY;
        const float wj = use ? exp2f(mj - mnew) : 0.f;
        wgt[j][hh] = wj;
        ls = fmaf(wj, use ? stage[(j * R + hh) * rs + 1] : 0.f, ls);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(kFullMask, ls, o);
      if (lane == 0) {
        const float sc = (mnew == -INFINITY) ? 1.f : exp2f(Mrun[hh] - mnew);
        scale_old[hh] = sc;
        Lrun[hh] = Lrun[hh] * sc + ls;
        Mrun[hh] = mnew;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < S::kOut; ++k) {
      const int i = tid + k * kCombineThreads;
      if (i < R * DV) {
        const int hh = i / DV, d = i - hh * DV;
        float v = acc[k] * scale_old[hh];
        for (int j = 0; j < n; ++j) {
          const float wj = wgt[j][hh];
          // records without data hold stale bytes (possibly NaN): skip rather than scale by 0
          if (wj != 0.f) v = fmaf(wj, stage[(j * R + hh) * rs + 4 + d], v);
        }
        acc[k] = v;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int k = 0; k < S::kOut; ++k) {
    const int i = tid + k * kCombineThreads;
    if (i < R * DV) {
      const int hh = i / DV;
      out_row(hh)[i - hh * DV] = Lrun[hh] > 0.f ? acc[k] / Lrun[hh] : 0.f;
    }
  }
}

template <int DV, int R>
cudaError_t launch_t(const DecodeArgs& a, cudaLaunchConfig_t& cfg) {
  using S = CombineShape<DV, R>;
  const int smem = (a.combine_big ? S::kRchBig : S::kRch) * R * S::kRs * 4;
  static int configured[kMaxDevicesHost] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevicesHost || !configured[dev]) {
    e = cudaFuncSetAttribute(combine_kernel<DV, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::kRchBig * R * S::kRs * 4);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevicesHost) configured[dev] = 1;
  }
  cfg.dynamicSmemBytes = smem;
  return cudaLaunchKernelEx(&cfg, combine_kernel<DV, R>, a);
}

// R here counts the sub-records of a record: (heads per group) x (queries per pass).
template <int DV>
cudaError_t launch_dv(const DecodeArgs& a, cudaLaunchConfig_t& cfg) {
  switch (a.H / a.G * a.nqp) {
    case 1: return launch_t<DV, 1>(a, cfg);
    case 2: return launch_t<DV, 2>(a, cfg);
    case 4: return launch_t<DV, 4>(a, cfg);
    case 8: return launch_t<DV, 8>(a, cfg);
    case 16:  // several queries per pass (d_v = 64 and 128)
      if constexpr (DV == 64 || DV == 128) return launch_t<DV, 16>(a, cfg);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.G, a.B);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (a.d_v) {
    case 32: return launch_dv<32>(a, cfg);
    case 64: return launch_dv<64>(a, cfg);
    case 128: return launch_dv<128>(a, cfg);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gva
