// gva_sched.cuh -- balanced split-T work distribution shared by the decode kernels.
//
// The decode work of a batch is the list of units (b, g, t): sequence b, value group g,
// 64-token tile t < nt_b = ceil(T_b / 64), ordered by b, then g, then t.  With
// cum[b] = sum_{b' < b} nt_b', unit (b, g, t) has index u = G*cum[b] + g*nt_b + t and the
// batch has U = G*cum[B] units.  Each of the W warps of the grid takes the contiguous range
// [floor(w*U/W), floor((w+1)*U/W)), so every warp streams the same number of tiles (give or
// take one) whatever the mix of context lengths, and one wave of CTAs covers the batch.
//
// A warp emits one partial record (per head of its group: running max, running sum and the
// weighted value sum) for every (b, g) segment its range touches.  Record index = w + f with
// f = b*G + g: within one warp the f's of its segments are consecutive, and the first f of
// warp w+1 is at least the last f of warp w, so indices are unique and below W + B*G.  The
// combine finds the warps whose ranges meet segment f arithmetically (warp_of below).
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

// Warp whose range holds unit u (U units over W warps).
__host__ __device__ inline long long warp_of(long long u, long long U, long long W) {
  return ((u + 1) * W - 1) / U;
}

// Per-CTA prologue: cum[0..B] in shared memory from seq_lens; lengths outside
// [1, max_seq_len] count as zero tiles (and are reported once by CTA 0).  Uses all threads
// of the CTA; ends with __syncthreads().  CTA 0 also publishes cum to the workspace header.
template <int NTHREADS>
__device__ void build_prefix(const DecodeArgs& a, int* cum) {
  __shared__ int warp_tot[NTHREADS / 32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < a.B; base += NTHREADS) {
    const int b = base + tid;
    int nt = 0;
    if (b < a.B) {
      const int T = a.seq_lens[b];
      if (T >= 1 && T <= a.max_seq_len)
        nt = (T + kBlockTokens - 1) / kBlockTokens;
      else if (blockIdx.x == 0)
        flag_error(a.err, GVA_DEVERR_SEQ_LEN);
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
    if (tid == NTHREADS - 1) carry = before + v;
    __syncthreads();
  }
  if (tid == 0) cum[a.B] = carry;
  __syncthreads();
  if (blockIdx.x == 0) {
    int* hdr = reinterpret_cast<int*>(a.part);
    for (int i = tid; i <= a.B; i += NTHREADS) hdr[i] = cum[i];
  }
}

// Position in the unit list: sequence b, group g, tile t of nt tiles.
struct UnitCursor {
  int b, g, t, nt;
};

// Cursor at unit u (0 <= u < U); cum in shared memory.
__device__ __forceinline__ UnitCursor cursor_at(long long u, const int* cum, int B, int G) {
  int lo = 0, hi = B;  // G*cum[lo] <= u < G*cum[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<long long>(G) * cum[mid] <= u)
      lo = mid;
    else
      hi = mid;
  }
  UnitCursor c;
  c.b = lo;
  c.nt = cum[lo + 1] - cum[lo];
  const long long r = u - static_cast<long long>(G) * cum[lo];
  c.g = static_cast<int>(r / c.nt);
  c.t = static_cast<int>(r - static_cast<long long>(c.g) * c.nt);
  return c;
}

// Next unit (the caller never steps past the last unit of the batch).
__device__ __forceinline__ void cursor_next(UnitCursor& c, const int* cum, int B, int G) {
  if (++c.t < c.nt) return;
  c.t = 0;
  if (++c.g < G) return;
  c.g = 0;
  do {
    ++c.b;
  } while (c.b < B && cum[c.b + 1] == cum[c.b]);
  if (c.b < B) c.nt = cum[c.b + 1] - cum[c.b];
}

// Programmatic dependent launch: wait for the grids this one depends on (their writes are
// then visible), and let the next grid in the stream start launching early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace gva
