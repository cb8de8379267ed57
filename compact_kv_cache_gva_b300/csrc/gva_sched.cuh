// gva_sched.cuh -- balanced split-T work distribution shared by the decode kernels.
//
// The decode work of a batch is the list of units (g, b, t): value group g, sequence b,
// 64-token tile t < nt_b = ceil(T_b / 64), ordered by g, then b, then t.  With
// cum[b] = sum_{b' < b} nt_b' and TOT = cum[B] (tiles of the batch), unit (g, b, t) has
// index u = g*TOT + cum[b] + t and the batch has U = G*TOT units.  The units are cut into NG
// equal contiguous ranges, range c = [floor(c*U/NG), floor((c+1)*U/NG)), so every range
// holds the same number of tiles (give or take one) whatever the mix of context lengths.
// When NG = G*Q, range g*Q + q is exactly the q-th of Q equal slices of group g's tiles, so
// the G ranges with the same q stream the same cache blocks at the same time and the
// positional-key tile that all groups of a block read comes from L2 after its first read.
// The C warps of a range share it round-robin: unit k of the range (k counted from the
// range start) goes to warp k % C.  The CUDA-core kernel gives every warp a range of its
// own (NG = warps, C = 1); the tensor-core kernel gives every CTA one range that its
// consumer warps share.
//
// A warp emits one partial record (per head of its group: running max, running sum and the
// weighted value sum) for every (g, b) segment it touched.  Segments are numbered in unit
// order, f = g*B + b.  Record index = (c + f)*C + w: within one range the f's of its
// segments increase, and the first f of range c+1 is at least the last f of range c, so
// (c + f) is strictly increasing over the (range, segment) pairs and indices are unique and
// below (NG + B*G)*C.  The combine finds the ranges that meet segment f and the warps of
// each that touched it arithmetically (range_of, warp_touched below), so no record is ever
// read that was not written.
#pragma once

#include "gva_device.cuh"
#include "gva_internal.h"

namespace gva {

// Workspace: [header][records].  Header: cum[0..B] (int32), written by CTA 0 of the partial
// kernel and read by the combine; records start at a kHeaderAlign-aligned offset.
constexpr int kHeaderAlign = 256;
__host__ __device__ inline size_t header_bytes(int B) {
  return ((static_cast<size_t>(B + 1) * 4 + kHeaderAlign - 1) / kHeaderAlign) * kHeaderAlign;
}

// Range holding unit u (U units over NG ranges).
__host__ __device__ inline long long range_of(long long u, long long U, long long NG) {
  return ((u + 1) * NG - 1) / U;
}

// First unit of range c.
__host__ __device__ inline long long range_begin(long long c, long long U, long long NG) {
  return c * U / NG;
}

// Whether warp w of a range (C warps, round-robin) holds any of the range-local units
// [a, e).
__host__ __device__ inline bool warp_touched(long long a, long long e, int w, int C) {
  if (e <= a) return false;
  if (e - a >= C) return true;
  const long long first = a + ((w - a) % C + C) % C;  // first k >= a with k % C == w
  return first < e;
}

// Per-CTA prologue: cum[0..B] in shared memory from seq_lens; lengths outside
// [max(1, nq), max_seq_len] count as zero tiles (and are reported once by CTA 0).  Uses all
// blockDim.x threads of the CTA (a multiple of 32, at most MAXT); ends with __syncthreads().
// CTA 0 also publishes cum to the workspace header.  With `lens` (shared memory, B ints) the
// lengths are kept too, 0 for a length outside that range.
template <int MAXT>
__device__ void build_prefix(const DecodeArgs& a, int* cum, int* lens = nullptr) {
  __shared__ int warp_tot[MAXT / 32];
  __shared__ int carry;
  const int nthr = blockDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < a.B; base += nthr) {
    const int b = base + tid;
    int nt = 0;
    if (b < a.B) {
      const int T = a.seq_lens[b];
      const bool valid = T >= a.nq && T >= 1 && T <= a.max_seq_len;
      if (valid)
        nt = (T + kBlockTokens - 1) / kBlockTokens;
      else if (blockIdx.x == 0)
        flag_error(a.err, GVA_DEVERR_SEQ_LEN);
      if (lens) lens[b] = valid ? T : 0;
    }
    // inclusive warp scan, then across warps
    int v = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFullMask, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    int before = carry;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    if (b < a.B) cum[b] = before + v - nt;  // exclusive
    __syncthreads();
    if (tid == nthr - 1) carry = before + v;
    __syncthreads();
  }
  if (tid == 0) cum[a.B] = carry;
  __syncthreads();
  if (blockIdx.x == 0) {
    int* hdr = reinterpret_cast<int*>(a.part);
    for (int i = tid; i <= a.B; i += nthr) hdr[i] = cum[i];
  }
}

// Segment ordinal of (group g, sequence b): segments are numbered in unit order.
__host__ __device__ inline long long segment_of(int g, int b, int B) {
  return static_cast<long long>(g) * B + b;
}

// Position in the unit list: group g, sequence b, tile t of nt tiles.
struct UnitCursor {
  int b, g, t, nt;
};

// Cursor at unit u (0 <= u < U); cum in shared memory.
__device__ __forceinline__ UnitCursor cursor_at(long long u, const int* cum, int B, int G) {
  const long long tot = cum[B];
  UnitCursor c;
  c.g = static_cast<int>(u / tot);
  const int r = static_cast<int>(u - static_cast<long long>(c.g) * tot);
  int lo = 0, hi = B;  // cum[lo] <= r < cum[hi]: the last such lo has a non-empty sequence
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cum[mid] <= r)
      lo = mid;
    else
      hi = mid;
  }
  c.b = lo;
  c.nt = cum[lo + 1] - cum[lo];
  c.t = r - cum[lo];
  return c;
}

// First non-empty sequence at or after b (B if none).
__device__ __forceinline__ int next_nonempty(int b, const int* cum, int B) {
  while (b < B && cum[b + 1] == cum[b]) ++b;
  return b;
}

// Next unit (the caller never steps past the last unit of the batch).
__device__ __forceinline__ void cursor_next(UnitCursor& c, const int* cum, int B, int G) {
  if (++c.t < c.nt) return;
  c.t = 0;
  c.b = next_nonempty(c.b + 1, cum, B);
  if (c.b >= B) {
    if (++c.g >= G) return;
    c.b = next_nonempty(0, cum, B);
  }
  c.nt = cum[c.b + 1] - cum[c.b];
}

// Cursor moved forward by k >= 1 units (the caller never steps past the last unit).
__device__ __forceinline__ void cursor_advance(UnitCursor& c, int k, const int* cum, int B, int G) {
  while (true) {
    const int rem = c.nt - c.t;
    if (k < rem) {
      c.t += k;
      return;
    }
    k -= rem;
    c.t = 0;
    c.b = next_nonempty(c.b + 1, cum, B);
    if (c.b >= B) {
      if (++c.g >= G) return;
      c.b = next_nonempty(0, cum, B);
    }
    c.nt = cum[c.b + 1] - cum[c.b];
  }
}

// Programmatic dependent launch: wait for the grids this one depends on (their writes are
// then visible), and let the next grid in the stream start launching early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace gva
