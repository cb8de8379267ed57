// gva_decode_mma.cuh -- split-T decode attention over the GVA cache on the tensor cores:
// the kernel template, its helpers and its launcher, instantiated by gva_decode_mma.cu (bf16
// caches) and gva_decode_mma_fp8.cu (fp8 value caches).
//
// Same contract and partial records as the CUDA-core kernel (gva_decode_fma.cu): for head h
// of value group g, s_j = scale * (q'_h . v_j + q~_r,h . k_r,j), online softmax, o_h =
// sum_j p_j v_j (ai-feeds.com summary "Grouped Value Attention:通过按需 key 重建实现高效 KV
// 缓存", section 方法; review "[논문리뷰] Grouped Value Attention", section 3).
//
// Per 64-token tile of group g, with the r = H/G heads of the group packed into the N=8
// columns of a warp-level bf16 MMA (m16n8k16 / m16n8k8, fp32 accumulate):
//   scores  S^T[64 tok x 8] = [V | k_r][64 x (d_v+d_r)] . [q'_hi | q'_lo]^T
//   output  O^T[d_v x 8]   += V^T[d_v x 64] . [p_hi | p_lo][64 x 8]
// Each head occupies two columns: its query (and later its probabilities) split into a
// bf16 high part and a bf16 remainder, so both products keep about 16 significant bits
// while using columns that the 4-head group would leave empty anyway.  The V tile arrives
// by TMA (tensor copy, 128-byte swizzle) so that ldmatrix reads it without bank conflicts,
// both as V (scores) and transposed as V^T (output); k_r arrives by a plain bulk copy.
// Probabilities never leave registers: movmatrix turns the score fragment (tokens on rows)
// into the B fragment of the output product (tokens on k).
//
// Multi-query passes of 16 (query, head) pairs take two other forms.  At d_v = 64 the queries
// go on M instead: S[pairs x 64 tok] = [q'_hi ; q'_lo] . V^T, both bf16 parts as A operands into
// one accumulator, whose fragment (pairs on rows) is the output product's B operand as it stands.
// At d_v = 128 the query operand stays in shared memory (ldmatrix per k-step), and each tile's
// pairs are split between two consumer warps that write their halves of one partial record.
//
// Work split (gva_sched.cuh): one CTA per SM streams a balanced range of (sequence, group,
// tile) units with a few consumer warps, each with a private ring of tiles that a copy warp
// keeps full (TMA) or, in the self-fed instances (multi-query passes and the fp8 cache at
// d_v = 64), that the consumer refills itself; the 16-pair passes at d_v = 128 give each ring
// two consumers.  The consumers take the range's tiles
// round-robin, each writing one partial record per (sequence, group) it touched.  The matching
// GQA form (a separate key cache, no positional slice) reuses the kernel with the key tile
// scored instead of the value tile.
//
// Fused decode step (FUSED instances): the absorption q' = M_h q_c and the rotation of the
// positional query (the neighbouring step of the decode path) run in the kernel's prologue
// instead of a kernel of their own.  The consumer warps, and the warps the launch has to spare
// beside them and their copy warps, compute them for every (group, sequence) segment of the
// CTA's range while the rings fill.  Each output is an fp32 dot product in the absorb kernel's
// summation order, so the results are bit-identical to it.  The new token of every sequence
// (the last position of its context) is appended between the copy engine and the consumer:
// the sequence's last tile lands on a barrier of its own, a patcher warp writes the value row
// and the rotated positional key into the staged tile and into the cache, and only then hands
// the tile to its consumer.
#pragma once

#include <cuda.h>

#include <algorithm>
#include <type_traits>
#include <math.h>

#include "gva_device.cuh"
#include "gva_internal.h"
#include "gva_sched.cuh"

namespace gva {
namespace {

constexpr int kMmaMaxThreads = 64 * kMmaMaxPairs;  // consumer warps + as many copy warps

// Threads a kernel instance is compiled for: twelve warps on the single-query d_v = 64 path,
// eight elsewhere.  A warp's registers come from its sub-partition's quarter of the register
// file, so the per-thread limit follows the warps a sub-partition hosts: up to 255 with eight
// warps (two each), 168 with nine to twelve.  Several queries per pass and d_v = 128 hold
// twice the accumulators and keep eight warps.
__host__ __device__ constexpr int mma_max_threads(int dv, int nq) { return dv == 64 && nq == 1 ? 384 : 256; }
// (query, head) column pairs a multi-query pass may hold: 16 (four n-tiles of hi/lo columns).
__host__ __device__ constexpr int mma_max_column_pairs(int) { return 16; }
// At d_v = 128 the query operand of a 16-pair pass (72 registers as B fragments) stays in shared
// memory, one copy per consumer, and each k-step's B fragments are loaded once per tile with
// ldmatrix, outside the loop over the tile's m-tiles.  Rows: column n = 2c + part (column pair c,
// bf16 part), its d_v content then d_r positional elements, the row stride an odd number of
// 16-byte units so that the eight rows of an ldmatrix fall in distinct banks.
__host__ __device__ constexpr bool mma_query_in_smem(int dv, int rq) { return dv == 128 && rq > 8; }
__host__ __device__ constexpr int mma_qop_stride(int dv, int dr) { return ((((dv + dr) * 2 + 15) / 16) | 1) * 16; }
__host__ __device__ constexpr int mma_qop_bytes(int dv, int dr, int rq) {
  return mma_query_in_smem(dv, rq) ? 8 * ((2 * rq + 7) / 8) * mma_qop_stride(dv, dr) : 0;
}
// Those passes also split each tile's 16 pairs between two consumer warps (eight each, with
// their halves of the operand): eight consumers, two per sub-partition, beside the four copy
// warps, so that one covers the other's dependent products.  Both write their halves of the
// ring's one partial record.
__host__ __device__ constexpr int mma_kernel_threads(int dv, int rq, int nq) {
  return mma_query_in_smem(dv, rq) ? 384 : mma_max_threads(dv, nq);
}
// Consumers a copy warp fills: one (warp pairs), or two where a CTA wants more consumers than
// pairs fit (a copy warp issues a tile in a small fraction of the time a consumer computes
// one): the bf16 cache at d_v = 64, d_r = 32 (6 consumers and 3 copy warps, which leaves the
// fused step a patcher and two helpers).  The fp8 instances at d_v = 64 are self-fed (below).
__host__ __device__ constexpr int mma_consumers_per_copy_warp(int dv, int dr, bool f8) {
  return dv == 64 && dr == 32 && !f8 ? 2 : 1;
}
// The passes of a multi-query call at d_v = 64 (and a call's single-query remainder pass, which
// shares their plan) have no copy warps: 8 consumers, two per sub-partition so that one
// computes while the other waits on its dependent products, each issuing the copies of its own
// ring.  A tile costs them over ten times longer to compute than its copies take to issue, and
// one copy warp for seven consumers left them waiting for tiles.
// The fp8 value cache at d_v = 64 does the same with twelve consumers: its small tiles make
// the consumers' instructions the limit, and the copy warps' issue slots serve them better as
// a third consumer per sub-partition.
__host__ __device__ constexpr bool mma_self_fed(int dv, bool multi, bool f8) { return dv == 64 && (multi || f8); }
constexpr int kSubTileBytes = kBlockTokens * 128;  // one [64 tokens][64 columns] bf16 swizzled box

// ---- PTX wrappers ------------------------------------------------------------------------

// The same copy with an L2 evict-first policy: for tiles read exactly once, so that the lines
// L2 should keep (positional-key tiles shared by a block's groups, the block table, the queries)
// are not pushed out by the stream.
__device__ __forceinline__ void tma_load_2d_evict_first(void* dst, const CUtensorMap* map, int x, int y,
                                                        uint64_t* bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
// A bulk copy with an L2 evict-last policy: for tiles several CTAs read at about the same time.
__device__ __forceinline__ void bulk_g2s_evict_last(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_16816_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t x, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(x), "r"(sel));
  return d;
}

__device__ __forceinline__ int ld_shared_s8(uint32_t addr) {
  int v;
  asm volatile("ld.shared.s8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void mma_1688(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// Asks L2 to fetch [p, p + bytes) (bytes <= kMaxWarmBytes), spread over every thread of the
// grid: one 128-byte line per request.
constexpr long long kMaxWarmBytes = 4ll << 20;
__device__ __forceinline__ void warm_l2(const void* p, long long bytes) {
  if (!p || bytes <= 0 || bytes > kMaxWarmBytes) return;
  const char* base = static_cast<const char*>(p);
  const long long lines = (bytes + 127) / 128;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < lines;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(base + i * 128));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Fused step: the new token (row o of block blk) into the staged tile of its group g -- its
// value row at the 128-byte-swizzled place the tensor copy gives it, its rotated positional
// key in the plain k_r tile -- and into the cache (the key from group 0 only: one per token).
// Lanes below d_v/8 move the value row (16 bytes each), lanes below d_r/2 a key pair.
template <int DV, int DR>
__device__ __forceinline__ void write_new_token(uint32_t vbase, uint32_t krbase, int o, uint4 vnew, uint32_t knew,
                                                long long blk, int g, int G, void* v_pool, void* kr_pool, int lane) {
  if (lane < DV / 8) {
    st_shared_v4(vbase + (lane >> 3) * kSubTileBytes + o * 128 + (((lane & 7) ^ (o & 7)) << 4), vnew);
    reinterpret_cast<uint4*>(v_pool)[((blk * G + g) * kBlockTokens + o) * (DV / 8) + lane] = vnew;
  }
  if (DR > 0 && lane < DR / 2) {
    st_shared_u32(krbase + o * (2 * DR) + 4 * lane, knew);
    if (g == 0) reinterpret_cast<uint32_t*>(kr_pool)[(blk * kBlockTokens + o) * (DR / 2) + lane] = knew;
  }
}

// fp8 value tile in shared memory: the tile's 64 x DV code bytes seen as rows of 128 bytes
// (DV = 64: two tokens per row), placed by the tensor copy with the 128-byte swizzle (16-byte
// chunk c of row r at chunk c ^ (r % 8)).  Address of the 16-byte chunk `chunk` of token tok.
template <int DV>
__device__ __forceinline__ uint32_t f8_addr(uint32_t base, int tok, int chunk) {
  const int L = tok * DV + chunk * 16;
  const int row = L >> 7, ch = (L >> 4) & 7;
  return base + row * 128 + ((ch ^ (row & 7)) << 4);
}

// The fp8 value cache's form: the new value row (8 bf16 per lane below DV/8) is quantised --
// its scale exponent from the row's largest magnitude, each value times 2^-e rounded to E4M3
// -- and its codes and exponent written to the staged tile and to the cache.  The whole warp
// calls it (the row maximum is a warp reduction).
template <int DV, int DR>
__device__ __forceinline__ void write_new_token_f8(uint32_t vbase, uint32_t krbase, uint32_t exbase, int o,
                                                   uint4 vnew, uint32_t knew, long long blk, int g, int G,
                                                   void* v_pool, signed char* v_exp, void* kr_pool, int lane) {
  float x[8];
  bf16x2_to_float2(vnew.x, x[0], x[1]);
  bf16x2_to_float2(vnew.y, x[2], x[3]);
  bf16x2_to_float2(vnew.z, x[4], x[5]);
  bf16x2_to_float2(vnew.w, x[6], x[7]);
  float amax = 0.f;
  if (lane < DV / 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
  const int e = fp8_row_exponent(amax);
  if (lane < DV / 8) {
    const float inv = exp2_int(-e);  // exact scaling: -e is in [-120, 126]
    uint2 c;
    c.x = f32x2_to_e4m3x2(x[0] * inv, x[1] * inv) | (f32x2_to_e4m3x2(x[2] * inv, x[3] * inv) << 16);
    c.y = f32x2_to_e4m3x2(x[4] * inv, x[5] * inv) | (f32x2_to_e4m3x2(x[6] * inv, x[7] * inv) << 16);
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(f8_addr<DV>(vbase, o, lane >> 1) + (lane & 1) * 8),
                 "r"(c.x), "r"(c.y)
                 : "memory");
    reinterpret_cast<uint2*>(v_pool)[((blk * G + g) * kBlockTokens + o) * (DV / 8) + lane] = c;
  }
  if (lane == 0) {
    asm volatile("st.shared.s8 [%0], %1;" ::"r"(exbase + o), "r"(e) : "memory");
    v_exp[(blk * G + g) * kBlockTokens + o] = static_cast<signed char>(e);
  }
  if (DR > 0 && lane < DR / 2) {
    st_shared_u32(krbase + o * (2 * DR) + 4 * lane, knew);
    if (g == 0) reinterpret_cast<uint32_t*>(kr_pool)[(blk * kBlockTokens + o) * (DR / 2) + lane] = knew;
  }
}

// 2^x by the special-function unit (relative error about 2^-22; results below 2^-126 flush to
// zero, 2^-inf = 0): softmax weights of the fp8 value cache.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Packs two floats as bf16 (first in the low half).
__device__ __forceinline__ uint32_t pack_bf16(float lo_half, float hi_half) {
  const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo_half));
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi_half));
  return a | (b << 16);
}

// Packs two floats as bf16 with one conversion (first in the low half).
__device__ __forceinline__ uint32_t pack2_bf16(float lo_half, float hi_half) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo_half, hi_half);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi); returns (hi, lo) packed.
__device__ __forceinline__ uint32_t split_pack(float x) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
  return static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
}

__device__ __forceinline__ float split_part(float x, int part) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  return part == 0 ? __bfloat162float(hi) : x - __bfloat162float(hi);
}

// The same splits with f16 parts (the operands of the fp8 value cache's f16 products).
__device__ __forceinline__ uint32_t pack_f16(float lo_half, float hi_half) {
  const uint32_t a = __half_as_ushort(__float2half_rn(lo_half));
  const uint32_t b = __half_as_ushort(__float2half_rn(hi_half));
  return a | (b << 16);
}

__device__ __forceinline__ float split_part_f16(float x, int part) {
  const __half hi = __float2half_rn(x);
  return part == 0 ? __half2float(hi) : x - __half2float(hi);
}

// Zeroes the bf16 halves of a fragment register whose token index is >= nv.
__device__ __forceinline__ uint32_t mask_pair(uint32_t v, int tok, int nv) {
  const uint32_t lo = tok < nv ? 0x0000ffffu : 0u;
  const uint32_t hi = tok + 1 < nv ? 0xffff0000u : 0u;
  return v & (lo | hi);
}

template <int DV, int DR, bool SEPK, bool F8 = false>
struct MmaLayout {
  static constexpr int kSub = F8 ? 1 : DV / 64;               // swizzled boxes per operand tile
  static constexpr int kVBytes = F8 ? kBlockTokens * DV : kSub * kSubTileBytes;  // one operand tile
  static constexpr int kOpBytes = kVBytes * (SEPK ? 2 : 1);   // operand tiles of a stage (1 KB multiple)
  static constexpr int kKrBytes = SEPK ? 0 : kBlockTokens * DR * 2;
  static constexpr int kExBytes = F8 ? kBlockTokens : 0;      // fp8 cache: the tile's 64 scale exponents
  static constexpr int kTx = kOpBytes + kKrBytes + kExBytes;  // bytes landing per stage
  static constexpr int kStageBytes = kOpBytes + kKrBytes + kExBytes;
};

// Shared memory: [alignment slack 1 KB][control 2 KB: full and empty mbarrier, valid length,
// block id and (fused step) landing mbarrier of every stage][P*D operand tiles, 1 KB aligned
// for the swizzled boxes][P*D k_r tiles][cum: B+1 ints].  Stage (c, slot) is index c*D + slot.
constexpr int kMaxStages = 40;
constexpr int kCtrlBytes = 2048;
static_assert(kMaxStages * (3 * 8 + 4 + 4) <= kCtrlBytes, "control block");
constexpr int kStepBatch = 16;  // fused step: segments whose absorbed queries a warp forms at once
constexpr int kStepBarrier = 1;  // fused step: named barrier that ends the prologue
constexpr int kLookupBarrier = 2;  // fused step: the copy warps' first block-table reads are out
// dynamic shared memory per CTA: the 227 KB opt-in limit less 1 KB for the kernel's static
// shared memory (the prefix scan's scratch, placed ahead of the 1 KB aligned dynamic block)
constexpr int kSmemLimit = 226 * 1024;
__host__ __device__ inline int cum_bytes(int B) { return ((B + 1) * 4 + 15) / 16 * 16; }
inline int ring_fixed_bytes(int B) { return 1024 + kCtrlBytes + cum_bytes(B); }

// One CTA streams one contiguous range of units (gva_sched.cuh) with P consumer warps and
// P/CPC copy warps (CPC = mma_consumers_per_copy_warp: 1, warp pairs, 2 or 7).  Consumer warp
// c (warps 0..P-1) takes units k = c, c + P, c + 2P, ... of the range; its d-th unit lands
// in its private ring slot d % D.  Copy warp c (warp P + c) serves the units k = c, c + P/CPC,
// ... in unit order (with CPC = 1, exactly consumer c's): its lanes look up the block ids of
// its next 32 units at once, one batch ahead, and lane 0 issues each unit's copies (TMA for
// the value (and key) tile, a bulk copy for the positional-key tile) as soon as the unit's
// consumer has released the slot.  Every barrier has one waiter that waits in order (the
// consumer on "full", the copy warp on "empty"), so phase parities are unambiguous, and about
// P*(D-1) tiles are in flight per SM while P are being computed.  The copy warps take the
// issue work (a few hundred cycles per tile) and the dependent block-table reads off the
// consumers' path.
//
// A FUSED launch adds E = (threads of the instance)/32 - P - P/CPC prologue warps that help
// form the queries; the first of them then stays as the patcher warp, the others exit.  (The
// fp8 instances at d_v = 64, twelve self-fed consumers, have none to spare: their consumers
// append themselves.)
//
// F8 instances read the fp8 value cache: the value tile is E4M3 codes (a tensor copy of
// 64 x DV bytes) plus its 64 scale exponents (a bulk copy), converted to f16 in registers for
// f16 products (every E4M3 value is an f16 value).  Scores: plain ldmatrix of the code rows
// gives each lane four consecutive columns 4tq..4tq+3 of a 16-column chunk, which serve as
// the k pairs (2tq, 2tq+1) and (2tq+8, 2tq+9) of the product: the query's B fragment is
// packed in the same column order, so the dot product is unchanged.  The content score of
// token j is then multiplied by its scale 2^e_j before the positional product adds to it.
// Output: transposed ldmatrix of the code rows gives each lane bytes (d, d+1) of tokens (t,
// t+1); one byte permutation makes them the token pairs of value rows d and d+1, which serve
// as rows gid and gid + 8 of the A fragment (the partial record writes them back in order).
// Probabilities enter as p_j 2^(e_j - E + 14) (E the largest exponent of the tile's tokens,
// in f16's normal range) into a per-tile accumulator that is added to o times 2^(E - 14).
template <int DV, int DR, int R, int NQ, bool CAUSAL, bool SEPK, bool FUSED, bool F8 = false>
__global__ void __launch_bounds__(mma_kernel_threads(DV, R * NQ, NQ), 1) decode_mma_kernel(const DecodeArgs a,
                                                                       const __grid_constant__ CUtensorMap tmv,
                                                                       const __grid_constant__ CUtensorMap tmk) {
  using L = MmaLayout<DV, DR, SEPK, F8>;
  constexpr int RQ = R * NQ;            // (query, head) column pairs of a group: c = i*R + h
  // 16-pair passes at d_v = 128: the query operand in shared memory, the pairs split between two
  // consumer warps per ring (mma_query_in_smem, mma_kernel_threads)
  constexpr bool kQS = mma_query_in_smem(DV, RQ) && !F8 && !SEPK;
  constexpr bool kSplit = kQS;
  constexpr int RQc = kSplit ? RQ / 2 : RQ;  // column pairs one consumer warp computes
  // 16-pair passes at d_v = 64 put the queries on M: S[pairs x 64 tok] = Q . V^T with the bf16
  // high parts and remainders of the query as two A operands into one accumulator, and the score
  // fragment (pairs on rows) serving as the output product's B operand as it stands: no
  // movmatrix, no adding of high and low score columns, two shuffle levels for a row maximum
  // (long-context four-query step 186.6 -> 180.3 us; with 8 pairs half of each M = 16 product
  // was empty and the two-query step went from 109.5 to 115.3 us, so those passes keep the
  // tokens on M).
  constexpr bool kQM = DV == 64 && CAUSAL && RQ > 8 && !F8 && !SEPK && !FUSED;
  constexpr int RH = RQ > 8 ? 2 : 1;  // queries on M: 8-pair row halves that hold pairs
  constexpr int NT = (2 * RQc + 7) / 8;      // its n-tiles of 8 columns (4 column pairs each)
  constexpr int KSV = DV / 16;          // k16 steps over the value (key) columns
  constexpr int KSR = DR / 16;          // k16 steps over the positional columns
  constexpr bool KR8 = (DR % 16) != 0;  // one trailing k8 step
  constexpr int MD = DV / 16;           // m16 tiles over d_v in the output product
  static_assert(DR % 8 == 0, "positional width must be a multiple of 8 on this path");
  static_assert(!SEPK || DR == 0, "the key-cache form has no positional slice");
  static_assert(!FUSED || (NQ == 1 && !CAUSAL && !SEPK), "the fused step is single-query GVA decode");
  static_assert(!F8 || (NQ == 1 && !CAUSAL && !SEPK), "the fp8 value cache is read by single-query GVA decode");
  constexpr int CPC = mma_consumers_per_copy_warp(DV, DR, F8);
  constexpr int QS = step_stage_floats(R, DV, DR);  // floats of one staged segment (fused step)
  constexpr int QST = mma_qop_stride(DV, DR);
  constexpr int kQopBytes = kQS ? 8 * NT * QST : 0;  // one consumer warp's query operand
  static_assert(!kQS || (NT == 2 && CAUSAL && !FUSED), "staged query operand: 16-pair multi-query passes");

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int P = a.group_warps;  // consumer warps
  constexpr bool kSelfFed = mma_self_fed(DV, CAUSAL, F8);
  const int PW = kSplit ? 2 * P : P;      // consumer warps (two per ring when the pairs are split)
  const int PC = kSelfFed ? 0 : P / CPC;  // copy warps; blockDim.x == 32 * (P + PC), plus the prologue warps of a fused launch
  const int D = a.n_stages;     // ring slots per pair
  const int N = P * D;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  int* nvs = reinterpret_cast<int*>(empty + kMaxStages);  // tokens from each stage's tile to the end (0 = skip)
  int* blks = nvs + kMaxStages;                            // block id of each stage's tile (fused step)
  // fused step: a sequence's last tile lands on landed[s] instead of full[s]; the patcher warp
  // writes the new token into it and then completes full[s]
  uint64_t* landed = reinterpret_cast<uint64_t*>(blks + kMaxStages);
  // Fused instances with a spare warp (all but the fp8 ones at d_v = 64) give the append to it: the
  // consumers' loop is then the plain kernel's.
  constexpr bool kPatcher = FUSED && !(DV == 64 && F8);
  unsigned char* tiles = smem + kCtrlBytes;
  unsigned char* krs = tiles + N * L::kOpBytes;
  unsigned char* exs = krs + N * L::kKrBytes;  // fp8 cache: the scale exponents of each stage's tile
  unsigned char* qops = exs + N * L::kExBytes;  // 16-pair passes at d_v = 128: each consumer's query operand
  int* cum = reinterpret_cast<int*>(qops + PW * kQopBytes);
  // fused step: the shared memory past the ring, [lengths: B ints][query stages]
  unsigned char* spare = reinterpret_cast<unsigned char*>(cum) + cum_bytes(a.B);
  int* lens_s = FUSED && a.spare_smem >= cum_bytes(a.B) ? reinterpret_cast<int*>(spare) : nullptr;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < N; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSplit ? 2 : 1);  // released by each consumer warp of the ring
      if (kPatcher) mbar_init(&landed[s], 1);
    }
    mbar_init_fence();
  }
  if (warp == (kSelfFed ? 0 : PW) && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    if (SEPK) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
  }
  // The lengths, the block table (and, for the fused step, the key maps) into L2 while this
  // kernel still waits for the earlier work in the stream: the scan and the first copies wait
  // on them, and the cache stream of the previous call has evicted them.  A prefetch returns no
  // data, and L2 keeps the lines coherent with any write that earlier work still makes, so it
  // may go out before the wait.  (All three are device memory; the step's own inputs may be
  // host memory.)
  warm_l2(a.seq_lens, static_cast<long long>(a.B) * 4);
  warm_l2(a.block_table, static_cast<long long>(a.B) * a.max_blocks * 4);
  if constexpr (FUSED) warm_l2(a.M, static_cast<long long>(a.H) * DV * DV * 4);
  // Everything below may read what earlier work in the stream wrote.
  griddep_wait();
  build_prefix<kMmaMaxThreads>(a, cum, lens_s);  // ends with __syncthreads: the barriers are set up
  griddep_launch_dependents();

  const long long U = static_cast<long long>(a.G) * cum[a.B];
  const long long u0 = range_begin(blockIdx.x, U, a.n_groups);
  const int n = static_cast<int>(range_begin(blockIdx.x + 1, U, a.n_groups) - u0);
  if (n <= 0) return;  // CTA-uniform; no CTA-wide barrier follows

  // ------------------------------------------------------------------ fused-step prologue
  // Absorbed and rotated queries of every segment f_lo + j of this range into stage j (in the
  // spare shared memory when they all fit, else stage c + f of the workspace), with the new
  // token's rotated positional key.  Work items: (32 rows of one head, up to kStepBatch
  // segments of one group); the item's M rows stay in registers while its segments' queries
  // stream past.  A thread's positional pairs are rotated while its first item's loads are in
  // flight, so the prologue costs about one memory round trip.
  long long f_lo = 0;       // first segment of the range
  int nseg = 0;             // segments of the range
  float* stage = nullptr;   // stage of segment f_lo
  if constexpr (FUSED) {
    const UnitCursor first = cursor_at(u0, cum, a.B, a.G);
    const UnitCursor last = cursor_at(u0 + n - 1, cum, a.B, a.G);
    f_lo = segment_of(first.g, first.b, a.B);
    nseg = static_cast<int>(segment_of(last.g, last.b, a.B) - f_lo) + 1;
    const long long stage_smem = lens_s ? a.spare_smem - cum_bytes(a.B) : 0;
    stage = static_cast<long long>(nseg) * QS * 4 <= stage_smem
                ? reinterpret_cast<float*>(spare + cum_bytes(a.B))
                : a.qstage + (static_cast<long long>(blockIdx.x) + f_lo) * QS;
  }
  auto absorb_segments = [&](int pw, int npw) {
    // The prologue's loads go out after the copy warps' first block-table reads, which the
    // first tile copies wait for (measured: 2.5 % of the long-context step; waiting until the
    // rings are primed, or not at all, was slower).
    named_barrier_sync(kLookupBarrier, static_cast<int>(blockDim.x));
    // positional pairs: R query pairs and the new key's pair per (segment, pair index)
    auto rotate_pairs = [&]() {
      if constexpr (DR > 0) {
        constexpr int PR = DR / 2;
        const int nrot = nseg * (R + 1) * PR;
        for (int it = pw * 32 + lane; it < nrot; it += npw * 32) {
          const int sg = it / ((R + 1) * PR);
          const int rem = it - sg * (R + 1) * PR;
          const int r = rem / PR, pi = rem - r * PR;
          const long long f = f_lo + sg;
          const int g = static_cast<int>(f / a.B);
          const int b = static_cast<int>(f - static_cast<long long>(g) * a.B);
          int T;
          if (lens_s) {
            T = lens_s[b];  // 0 when out of range
          } else {
            T = a.seq_lens[b];
            if (T > a.max_seq_len) T = 0;
          }
          if (T < 1) continue;  // no tile of this sequence is streamed
          const long long xoff = r < R ? (static_cast<long long>(b) * a.H + g * R + r) * DR + 2 * pi : 0;
          float2 x = make_float2(0.f, 0.f);
          uint32_t w = 0;
          if (r < R)
            x = *reinterpret_cast<const float2*>(a.q_r + xoff);
          else
            w = *reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.kr_new) +
                                                   static_cast<long long>(b) * DR + 2 * pi);
          float c, sn;
          rope_cos_sin_f32(a.rope32, PR, static_cast<long long>(T) - 1, pi, c, sn);
          float* slot = stage + static_cast<long long>(sg) * QS;
          if (r < R) {
            float2 y;
            rope_rotate_f32(x.x, x.y, c, sn, y.x, y.y);
            *reinterpret_cast<float2*>(slot + r * (DV + DR) + DV + 2 * pi) = y;
          } else {
            float x0, x1, y0, y1;
            bf16x2_to_float2(w, x0, x1);
            rope_rotate_f32(x0, x1, c, sn, y0, y1);
            reinterpret_cast<uint32_t*>(slot + R * (DV + DR))[pi] = pack_bf16(y0, y1);
          }
        }
      }
    };
    bool rotated = false;
    // q' rows: four lanes per row, lane e of the quad accumulating chunks c = e, e+4, ... (the
    // absorb kernel's summation order), so a warp's loads are 64 contiguous bytes per row
    constexpr int RB = R * DV / 32;  // 32-row blocks of the group's R*d_v query rows
    constexpr int XC = DV / 16;      // chunks per lane per row
    const int rq = lane >> 2, e = lane & 3;
    int item0 = 0;                   // item number of (this batch, block 0)
    for (int s0 = 0; s0 < nseg; item0 += RB) {
      const long long f0 = f_lo + s0;
      const int g = static_cast<int>(f0 / a.B);
      const int b0 = static_cast<int>(f0 - static_cast<long long>(g) * a.B);
      const int cnt = min(min(kStepBatch, nseg - s0), a.B - b0);  // segments of group g
      for (int rb = ((pw - item0) % npw + npw) % npw; rb < RB; rb += npw) {
        const int h = (rb * 32) / DV;
        const int head = g * R + h;
        // rows i0 + 8*rnd of head h, RP of the four rounds at a time (16 vectors of M in registers)
        const int i0 = rb * 32 - h * DV + rq;
        constexpr int RP = 256 / DV;
#pragma unroll 1
        for (int r0 = 0; r0 < 4; r0 += RP) {
        float4 m4[RP][XC];
#pragma unroll
        for (int rnd = 0; rnd < RP; ++rnd) {
          const float4* mrow =
              reinterpret_cast<const float4*>(a.M + (static_cast<long long>(head) * DV + i0 + 8 * (r0 + rnd)) * DV);
#pragma unroll
          for (int x = 0; x < XC; ++x) m4[rnd][x] = __ldg(mrow + 4 * x + e);
        }
        auto load_qc = [&](int j, float4 (&q4)[XC]) {
          const float4* qrow = reinterpret_cast<const float4*>(a.q_c + (static_cast<long long>(b0 + j) * a.H + head) * DV);
#pragma unroll
          for (int x = 0; x < XC; ++x) q4[x] = __ldg(qrow + 4 * x + e);
        };
        float4 qn[XC];  // the next segment's query chunks, loaded one segment ahead
        load_qc(0, qn);
        if (!rotated) {  // while the loads above are in flight
          rotate_pairs();
          rotated = true;
        }
        for (int j = 0; j < cnt; ++j) {
          float4 q4[XC];
#pragma unroll
          for (int x = 0; x < XC; ++x) q4[x] = qn[x];
          if (j + 1 < cnt) load_qc(j + 1, qn);
#pragma unroll
          for (int rnd = 0; rnd < RP; ++rnd) {
            float acc = 0.f;
#pragma unroll
            for (int x = 0; x < XC; ++x) {
              acc = fmaf(m4[rnd][x].x, q4[x].x, acc);
              acc = fmaf(m4[rnd][x].y, q4[x].y, acc);
              acc = fmaf(m4[rnd][x].z, q4[x].z, acc);
              acc = fmaf(m4[rnd][x].w, q4[x].w, acc);
            }
            acc += __shfl_xor_sync(kFullMask, acc, 1);  // p0 + p1, p2 + p3
            acc += __shfl_xor_sync(kFullMask, acc, 2);  // (p0 + p1) + (p2 + p3)
            if (e == 0) stage[static_cast<long long>(s0 + j) * QS + h * (DV + DR) + i0 + 8 * (r0 + rnd)] = acc;
          }
        }
        }
      }
      s0 += cnt;
    }
    if (!rotated) rotate_pairs();
  };
  if constexpr (FUSED) {
    const int E = static_cast<int>(blockDim.x / 32) - P - PC;  // prologue-only warps
    if (warp >= P + PC) {
      absorb_segments(P + (warp - P - PC), P + E);
      if (!kPatcher || warp != P + PC) {
        asm volatile("bar.arrive %0, %1;" ::"r"(kStepBarrier), "r"(32 * (P + E)) : "memory");
        return;
      }
      // ---------------------------------------------------------------- patcher warp
      // For every sequence whose last tile lies in this range (in unit order, which is each
      // copy warp's issue order): wait for the tile to land, write the new token's value row
      // and rotated positional key into it and into the cache, then hand it to its consumer.
      named_barrier_sync(kStepBarrier, 32 * (P + E));  // the rotated keys are staged
      const long long tot = cum[a.B];
      unsigned long long parity = 0;  // bit s: phase parity of landed[s]
      for (int j = 0; j < nseg; ++j) {
        const long long f = f_lo + j;
        const int g = static_cast<int>(f / a.B);
        const int b = static_cast<int>(f - static_cast<long long>(g) * a.B);
        if (cum[b + 1] == cum[b]) continue;  // no tile (or an out-of-range length)
        const long long kl = static_cast<long long>(g) * tot + cum[b + 1] - 1 - u0;  // its last unit
        if (kl < 0 || kl >= n) continue;  // in another range
        // the copy warp skips a tile whose block it cannot resolve (and completes full[s] itself)
        const int t_last = cum[b + 1] - cum[b] - 1;
        if (t_last >= a.max_blocks) continue;
        const int id = a.block_table[static_cast<long long>(b) * a.max_blocks + t_last];
        if (id < 0 || id >= a.num_blocks) continue;
        const int w = static_cast<int>(kl % P), d = static_cast<int>(kl / P);
        const int s = w * D + d % D;
        uint4 vnew = make_uint4(0, 0, 0, 0);
        uint32_t knew = 0;
        if (lane < DV / 8)
          vnew = __ldg(reinterpret_cast<const uint4*>(a.v_new) + (static_cast<long long>(b) * a.G + g) * (DV / 8) + lane);
        if (DR > 0 && lane < DR / 2) knew = reinterpret_cast<const uint32_t*>(stage + static_cast<long long>(j) * QS + R * (DV + DR))[lane];
        const bool got = mbar_wait_bounded(&landed[s], static_cast<uint32_t>((parity >> s) & 1));
        parity ^= 1ull << s;
        if (!__all_sync(kFullMask, got)) {
          if (lane == 0) flag_error(a.err, GVA_DEVERR_TIMEOUT);
        } else {
          const int nrem = nvs[s];
          if (nrem > 0) {
            if constexpr (F8)
              write_new_token_f8<DV, DR>(smem_addr(tiles + s * L::kOpBytes), smem_addr(krs + s * L::kKrBytes),
                                         smem_addr(exs + s * L::kExBytes), nrem - 1, vnew, knew, blks[s], g, a.G,
                                         a.v_pool_w, a.v_exp_w, a.kr_pool_w, lane);
            else
              write_new_token<DV, DR>(smem_addr(tiles + s * L::kOpBytes), smem_addr(krs + s * L::kKrBytes), nrem - 1,
                                      vnew, knew, blks[s], g, a.G, a.v_pool_w, a.kr_pool_w, lane);
          }
        }
        fence_proxy_async_smem();  // these writes come before the copy engine refills the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);  // the consumer may read the tile
      }
      return;
    }
  }

  // ------------------------------------------------------------------ copy warps
  // Lane i of a warp that issues the copies of the units base + stride*d (d < n_mine): block id
  // (or -1), group and valid tokens of unit d0 + i.
  auto lookup = [&](int base, int stride, int n_mine, int d0, int& blk, int& grp, int& nv) {
    blk = -1;
    grp = 0;
    nv = 0;
    const int d = d0 + lane;
    if (d < n_mine) {
      const UnitCursor cu = cursor_at(u0 + base + static_cast<long long>(stride) * d, cum, a.B, a.G);
      grp = cu.g;
      const int T = a.seq_lens[cu.b];  // issued beside the table read: one round trip
      if (cu.t >= a.max_blocks) {
        flag_error(a.err, GVA_DEVERR_POSITION);
      } else {
        const int id = a.block_table[static_cast<long long>(cu.b) * a.max_blocks + cu.t];
        if (id >= 0 && id < a.num_blocks) {
          blk = id;
          nv = T - cu.t * kBlockTokens;  // tokens from the tile's start to the end (>= 1)
        } else {
          flag_error(a.err, GVA_DEVERR_BLOCK_ID);
        }
      }
    }
  };
  // One thread: the copies of a unit (block bj, group gj, vj tokens to the end) into stage s,
  // completing full[s] (or, for a sequence's last tile in a fused step, landed[s]).
  // The value (or code) tile of a unit is read once: at d_v = 64 its copy carries an L2
  // evict-first policy (long-context step 97.4 -> 95.1 us, the fp8 step 91.9 -> 90.5 us), and
  // the positional-key tile, which the G CTAs of a slice read together, an evict-last one
  // (95.1 -> 94.5 us).  At d_v = 128 the ragged batch's step was 0.9 % slower with evict-first
  // values, so those copies keep the default policy.
  auto load_tile = [&](void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    if constexpr (DV == 64)
      tma_load_2d_evict_first(dst, map, x, y, bar);
    else
      tma_load_2d(dst, map, x, y, bar);
  };
  auto load_kr = [&](void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    if constexpr (DV == 64)
      bulk_g2s_evict_last(dst, src, bytes, bar);
    else
      bulk_g2s(dst, src, bytes, bar);
  };
  auto issue = [&](int s, int bj, int gj, int vj) {
    nvs[s] = bj >= 0 ? vj : 0;  // published by the arrive below (release)
    if (FUSED) blks[s] = bj;
    if (bj >= 0) {
      // fused step: a sequence's last tile goes to the patcher before the consumer
      uint64_t* bar = kPatcher && vj <= kBlockTokens ? &landed[s] : &full[s];
      mbar_arrive_expect_tx(bar, L::kTx);
      unsigned char* st = tiles + s * L::kOpBytes;
      if constexpr (F8) {
        // the tile's codes as DV/2 rows of 128 bytes, and its 64 exponents
        load_tile(st, &tmv, 0, (bj * a.G + gj) * (DV / 2), bar);
        bulk_g2s(exs + s * L::kExBytes, a.v_exp + (static_cast<long long>(bj) * a.G + gj) * kBlockTokens,
                 L::kExBytes, bar);
      } else {
        const int y = (bj * a.G + gj) * kBlockTokens;
#pragma unroll
        for (int sub = 0; sub < L::kSub; ++sub) {
          load_tile(st + sub * kSubTileBytes, &tmv, 64 * sub, y, bar);
          if (SEPK) load_tile(st + L::kVBytes + sub * kSubTileBytes, &tmk, 64 * sub, y, bar);
        }
      }
      if (!SEPK && DR > 0)
        load_kr(krs + s * L::kKrBytes,
                 static_cast<const __nv_bfloat16*>(a.kr_pool) + static_cast<size_t>(bj) * kBlockTokens * DR,
                 L::kKrBytes, bar);
    } else {
      mbar_arrive(&full[s]);  // completes the phase with no data; the tile is skipped
    }
  };
  if (!kSelfFed && warp >= PW) {
    // copy warp c serves the units k = c + PC*i of the range (i < n_mine): CPC consumers, unit
    // k going to consumer k % P as its (k / P)-th unit
    const int c = warp - PW;
    const int n_mine = n > c ? (n - c + PC - 1) / PC : 0;
    int blk, grp, nv;
    lookup(c, PC, n_mine, 0, blk, grp, nv);
    if constexpr (FUSED) asm volatile("bar.arrive %0, %1;" ::"r"(kLookupBarrier), "r"(static_cast<int>(blockDim.x)) : "memory");
    int issued = 0;
    bool ok = true;
    auto stage_of = [&](int i, int& dd) {  // ring stage of this warp's i-th unit; dd = its index at its consumer
      const int k = c + PC * i;
      dd = k / P;
      return (k - dd * P) * D + dd % D;
    };
    for (int d0 = 0; d0 < n_mine && ok; d0 += 32) {
      int nblk, ngrp, nnv;
      lookup(c, PC, n_mine, d0 + 32, nblk, ngrp, nnv);  // next batch: loads in flight while this one issues
      const int cnt = min(32, n_mine - d0);
      for (int j = 0; j < cnt; ++j) {
        const int bj = __shfl_sync(kFullMask, blk, j);
        const int gj = __shfl_sync(kFullMask, grp, j);
        const int vj = __shfl_sync(kFullMask, nv, j);
        if (lane == 0) {
          int dd;
          const int s = stage_of(d0 + j, dd);
          // the slot's previous unit must have been released by the consumer
          if (dd >= D && !mbar_wait_bounded(&empty[s], ((dd / D) & 1) ^ 1)) ok = false;
          if (ok) {
            issue(s, bj, gj, vj);
            ++issued;
          }
        }
        ok = __shfl_sync(kFullMask, ok, 0);
        if (!ok) break;
      }
      blk = nblk;
      grp = ngrp;
      nv = nnv;
    }
    if (lane == 0) {
      if (!ok) flag_error(a.err, GVA_DEVERR_TIMEOUT);
      // no copy may still be landing in shared memory when the CTA exits (the last D units of
      // each consumer served are the last CPC*D issued)
      for (int i = max(0, issued - CPC * D); i < issued; ++i) {
        int dd;
        const int s = stage_of(i, dd);
        if (!mbar_wait_bounded(&full[s], (dd / D) & 1)) flag_error(a.err, GVA_DEVERR_TIMEOUT);
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  // Self-fed consumer: its units are k = warp + P*i (i < n_own), unit i in slot i % D.  Lanes
  // hold the block ids of units [f0, f0 + 32) and of the next 32 (looked up a batch ahead); the
  // first D units' copies go out first (ahead of a fused launch's prologue), unit i + D's once
  // unit i is done.
  static_assert(!(kSelfFed && kPatcher), "self-fed consumers append the new token themselves");
  int n_own = 0, f0 = 0, i_own = 0;
  int fb = -1, fg = 0, fv = 0, xb = -1, xg = 0, xv = 0;
  if constexpr (kSelfFed) {
    n_own = n > warp ? (n - warp + P - 1) / P : 0;
    lookup(warp, P, n_own, 0, fb, fg, fv);
    lookup(warp, P, n_own, 32, xb, xg, xv);
    const int first = min(D, n_own);
    for (int j = 0; j < first; ++j) {
      const int bj = __shfl_sync(kFullMask, fb, j);
      const int gj = __shfl_sync(kFullMask, fg, j);
      const int vj = __shfl_sync(kFullMask, fv, j);
      if (lane == 0) issue(warp * D + j, bj, gj, vj);
    }
  }
  if constexpr (FUSED) {
    const int E = static_cast<int>(blockDim.x / 32) - P - PC;
    absorb_segments(warp, P + E);
    named_barrier_sync(kStepBarrier, 32 * (P + E));  // every stage of the range is written
  }
  const int NC = P;  // consumers (rings) sharing the range
  const int ring = kSplit ? warp % P : warp;  // this warp's ring and consumer (record) index
  const int cp0 = kSplit ? RQc * (warp / P) : 0;  // its first column pair
  int k = ring;
  if (k >= n) return;
  float* recs = a.part + header_bytes(a.B) / 4;
  constexpr int rec_floats = DV + 4;
  UnitCursor cc = cursor_at(u0 + k, cum, a.B, a.G);
  int slot = 0, ph = 0;  // ring slot and phase parity of this warp's next unit

  // query fragments (B operand of the score product) of the current (b, g), pre-scaled by
  // scale*log2(e); column n = 2*c + part for column pair c = i*R + h (query q0 + i of this
  // pass, head h of the group), part 0 = bf16(q), part 1 = bf16 remainder.
  uint32_t qb[kQS || kQM ? 1 : NT][kQS || kQM ? 1 : KSV + KSR][2];
  uint32_t qt[kQS || kQM ? 1 : NT];
  // queries on M: A fragments of the query (rows: column pairs; content then positional k16
  // steps, and the trailing k8 step), per bf16 part
  uint32_t qa[2][kQM ? KSV + KSR : 1][4];
  uint32_t qat[2][2];
  uint4 vnew = make_uint4(0, 0, 0, 0);  // fused step: a 16-byte piece of the new value row
  uint32_t knew = 0;                    // fused step: a pair of the new rotated positional key
  auto load_q = [&](int b, int g) {
    if constexpr (kQM) {
      const int lg = lane >> 2, lt4 = lane & 3;
      auto qv = [&](int c, int kk, int part) -> float {
        if (c >= RQ) return 0.f;
        const long long row = (static_cast<long long>(b) * a.nq + a.q0 + c / R) * a.H + g * R + c % R;
        const float x = kk < DV ? a.q_abs[row * DV + kk] : a.q_rot[row * DR + (kk - DV)];
        return split_part(x * a.scale_log2, part);
      };
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int ks = 0; ks < KSV + KSR; ++ks) {
          const int k0 = 16 * ks + 2 * lt4;
          qa[part][ks][0] = pack_bf16(qv(lg, k0, part), qv(lg, k0 + 1, part));
          qa[part][ks][1] = pack_bf16(qv(lg + 8, k0, part), qv(lg + 8, k0 + 1, part));
          qa[part][ks][2] = pack_bf16(qv(lg, k0 + 8, part), qv(lg, k0 + 9, part));
          qa[part][ks][3] = pack_bf16(qv(lg + 8, k0 + 8, part), qv(lg + 8, k0 + 9, part));
        }
        if constexpr (KR8) {
          const int k0 = 16 * (KSV + KSR) + 2 * lt4;
          qat[part][0] = pack_bf16(qv(lg, k0, part), qv(lg, k0 + 1, part));
          qat[part][1] = pack_bf16(qv(lg + 8, k0, part), qv(lg + 8, k0 + 1, part));
        }
      }
    } else if constexpr (kQS) {
      // operand rows n = 2c + part of this consumer's copy, element pairs (2kp, 2kp + 1)
      const uint32_t qb0 = smem_addr(qops + warp * kQopBytes);
      constexpr int KP = (DV + DR) / 2;
      static_assert(kSplit, "the staged operand holds a consumer's half of the pairs");
      __syncwarp();  // the previous segment's rows have been read
      for (int idx = lane; idx < 8 * NT * KP; idx += 32) {
        const int nr = idx / KP, kp = idx - nr * KP;
        const int c = (nr >> 1) + cp0, part = nr & 1;
        uint32_t w = 0;
        if (c < cp0 + RQc) {
          const long long row = (static_cast<long long>(b) * a.nq + a.q0 + c / R) * a.H + g * R + c % R;
          const int k = 2 * kp;
          const float* src = k < DV ? a.q_abs + row * DV + k : a.q_rot + row * DR + (k - DV);
          w = pack_bf16(split_part(src[0] * a.scale_log2, part), split_part(src[1] * a.scale_log2, part));
        }
        st_shared_u32(qb0 + nr * QST + 4 * kp, w);
      }
      __syncwarp();
    } else {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int cp = nt * 4 + ((lane >> 2) >> 1), part = (lane >> 2) & 1;
      const int tq = lane & 3;
      const bool valid = cp < RQc;
      const int qi = valid ? cp / R : 0, head = valid ? cp % R : 0;
      const long long row = (static_cast<long long>(b) * a.nq + a.q0 + qi) * a.H + g * R + head;
      const float* qa = FUSED ? stage + (segment_of(g, b, a.B) - f_lo) * QS + head * (DV + DR) : a.q_abs + row * DV;
      const float* qr = FUSED ? qa + DV : a.q_rot + row * DR;
      auto qv = [&](int kk) -> float {
        if (!valid) return 0.f;
        const float x = (kk < DV ? qa[kk] : qr[kk - DV]) * a.scale_log2;
        return split_part(x, part);
      };
      auto qv16 = [&](int kk) -> float {  // f16 parts (the fp8 cache's content product)
        if (!valid) return 0.f;
        return split_part_f16(qa[kk] * a.scale_log2, part);
      };
#pragma unroll
      for (int ks = 0; ks < KSV + KSR; ++ks) {
        if (F8 && ks < KSV) {  // columns 4tq..4tq+3 of chunk ks, the order the code rows arrive in
          const int k0 = 16 * ks + 4 * tq;
          qb[nt][ks][0] = pack_f16(qv16(k0), qv16(k0 + 1));
          qb[nt][ks][1] = pack_f16(qv16(k0 + 2), qv16(k0 + 3));
        } else {
          const int k0 = 16 * ks + 2 * tq;
          qb[nt][ks][0] = pack_bf16(qv(k0), qv(k0 + 1));
          qb[nt][ks][1] = pack_bf16(qv(k0 + 8), qv(k0 + 9));
        }
      }
      if (KR8) {
        const int k0 = 16 * (KSV + KSR) + 2 * tq;
        qt[nt] = pack_bf16(qv(k0), qv(k0 + 1));
      }
    }
    }
    if constexpr (FUSED && !kPatcher) {  // the new token's row, in case this warp meets the segment's last tile
      if (lane < DV / 8)
        vnew = __ldg(reinterpret_cast<const uint4*>(a.v_new) + (static_cast<long long>(b) * a.G + g) * (DV / 8) + lane);
      if (DR > 0 && lane < DR / 2)
        knew = reinterpret_cast<const uint32_t*>(stage + (segment_of(g, b, a.B) - f_lo) * QS + R * (DV + DR))[lane];
    }
  };

  // Wide instances (an even number of n-tiles: several queries per pass, or 8 heads a group)
  // give each accumulator column a column pair of its own: the probabilities' bf16 high parts
  // of n-tiles 2i and 2i+1 form one B operand and their remainders another, two products into
  // the same accumulator, whose column 2q + j then holds column pair (2i + j)*4 + q.  That
  // halves the output accumulators (the narrow form keeps a pair's high and low products in
  // two columns and adds them at the end).  They also take 2^x from the special-function
  // unit directly (relative error about 2^-22).
  constexpr bool kWide = !F8 && NT % 2 == 0;
  constexpr int NO = kWide ? NT / 2 : NT;  // accumulator n-tiles
  constexpr bool kFastExp = F8 || kWide;
  float m[NT], l[NT], o[NO][MD][4];
  float mq[RH], lq[RH], oq[RH][MD][4];  // queries on M: per row half (row gid, gid + 8 of it)
  auto reset_state = [&]() {
    if constexpr (kQM) {
#pragma unroll
      for (int rh = 0; rh < RH; ++rh) {
        mq[rh] = -INFINITY;
        lq[rh] = 0.f;
#pragma unroll
        for (int md = 0; md < MD; ++md)
#pragma unroll
          for (int e = 0; e < 4; ++e) oq[rh][md][e] = 0.f;
      }
      return;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt] = -INFINITY;
      l[nt] = 0.f;
    }
#pragma unroll
    for (int no = 0; no < NO; ++no)
#pragma unroll
      for (int md = 0; md < MD; ++md)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[no][md][e] = 0.f;
  };
  const int gid = lane >> 2, tq = lane & 3;
  // Partial record of segment f for this warp: per column pair (m, l, 0, 0, o[0..DV)).
  auto flush = [&](long long f) {
    float* rec = recs + ((static_cast<long long>(blockIdx.x) + f) * NC + ring) * RQ * rec_floats;
    if constexpr (kQM) {
      // pair c = 8 rh + gid: m and l (l summed over the row's four lanes); output column pairs
      // 8 rh + 2tq (+1), value rows 16 md + gid (+8)
#pragma unroll
      for (int rh = 0; rh < RH; ++rh) {
        float lt = lq[rh];
        lt += __shfl_xor_sync(kFullMask, lt, 1);
        lt += __shfl_xor_sync(kFullMask, lt, 2);
        const int c = 8 * rh + gid;
        if (tq == 0 && c < RQ) {
          rec[c * rec_floats] = mq[rh];
          rec[c * rec_floats + 1] = lt;
        }
#pragma unroll
        for (int md = 0; md < MD; ++md)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int cp = 8 * rh + 2 * tq + (e & 1);
            if (cp < RQ) rec[cp * rec_floats + 4 + 16 * md + gid + 8 * (e >> 1)] = oq[rh][md][e];
          }
      }
      return;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float lt = l[nt];
      lt += __shfl_xor_sync(kFullMask, lt, 4);
      lt += __shfl_xor_sync(kFullMask, lt, 8);
      lt += __shfl_xor_sync(kFullMask, lt, 16);
      const int cp = nt * 4 + tq;
      if (cp < RQc) {
        float* r = rec + (cp + cp0) * rec_floats;
        if (gid == 0) {
          r[0] = m[nt];
          r[1] = lt;
        }
#pragma unroll
        for (int md = 0; md < MD; ++md) {
          // fp8 cache: A-fragment rows gid and gid + 8 of chunk md are value rows 2gid, 2gid + 1
          if constexpr (kWide) {
            r[4 + 16 * md + gid] = o[nt / 2][md][nt % 2];
            r[4 + 16 * md + gid + 8] = o[nt / 2][md][2 + nt % 2];
          } else {
            r[4 + 16 * md + (F8 ? 2 * gid : gid)] = o[nt][md][0] + o[nt][md][1];
            r[4 + 16 * md + (F8 ? 2 * gid + 1 : gid + 8)] = o[nt][md][2] + o[nt][md][3];
          }
        }
      }
    }
  };

  // lane-dependent parts of the ldmatrix addresses
  const int ld_row = (lane & 7) + ((lane >> 3) & 1) * 8;  // non-transposed: row within m16
  const int ld_kc = lane >> 4;                             // non-transposed: 8-column chunk
  // fp8 cache: offset of this lane's row address in 16-column chunk pair cc of a code tile
  // (tokens ld_row of the first 16; the next 16 tokens are 16 DV bytes on, same swizzle)
  uint32_t f8_off[F8 ? DV / 32 : 1];
  if constexpr (F8) {
#pragma unroll
    for (int cc = 0; cc < DV / 32; ++cc) f8_off[cc] = f8_addr<DV>(0, ld_row, 2 * cc + ld_kc);
  }
  const int tr_tok = (lane & 7) + ((lane >> 4) & 1) * 8;   // transposed: token within k16
  const int tr_dc = (lane >> 3) & 1;                       // transposed: 8-column chunk

  reset_state();
  load_q(cc.b, cc.g);
  bool ok = true;
  while (true) {
    const int s = ring * D + slot;
    const bool got = mbar_wait_bounded(&full[s], ph);
    if (!__all_sync(kFullMask, got)) {
      ok = false;
      break;
    }
    const int nrem = nvs[s];
    bool patched = false;
    if (nrem > 0) {
      const int nv = min(nrem, kBlockTokens);  // valid tokens of the tile
      const uint32_t vbase = smem_addr(tiles + s * L::kOpBytes);
      const uint32_t kbase = SEPK ? vbase + L::kVBytes : vbase;  // tile that is scored
      const uint32_t krbase = smem_addr(krs + s * L::kKrBytes);
      const uint32_t exbase = smem_addr(exs + s * L::kExBytes);
      if constexpr (FUSED && !kPatcher) {
        if (nrem <= kBlockTokens) {  // the sequence's last tile: the new token is row nrem - 1
          if constexpr (F8)
            write_new_token_f8<DV, DR>(vbase, krbase, exbase, nrem - 1, vnew, knew, blks[s], cc.g, a.G, a.v_pool_w,
                                       a.v_exp_w, a.kr_pool_w, lane);
          else
            write_new_token<DV, DR>(vbase, krbase, nrem - 1, vnew, knew, blks[s], cc.g, a.G, a.v_pool_w,
                                    a.kr_pool_w, lane);
          patched = true;
          __syncwarp();
        }
      }
      if constexpr (kQM) {
        // scores S[pairs x 64 tokens]: thread holds rows gid, gid + 8 (e = 0, 1 and 2, 3) and
        // tokens 8 jb + 2tq (+1) of column block jb
        float sc[8][4];
#pragma unroll
        for (int jb = 0; jb < 8; ++jb)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[jb][e] = 0.f;
        // content: the value rows as B fragments (tokens on n), two column blocks per load:
        // matrices (tokens +0..7, chunk 2ks), (+0..7, 2ks + 1), (+8..15, 2ks), (+8..15, 2ks + 1)
#pragma unroll
        for (int ks = 0; ks < KSV; ++ks) {
#pragma unroll
          for (int jb = 0; jb < 8; jb += 2) {
            const int tok = 8 * jb + 8 * (lane >> 4) + (lane & 7);
            const int kc = 2 * ks + ((lane >> 3) & 1);
            uint32_t bf[4];
            ldsm_x4(kbase + (kc >> 3) * kSubTileBytes + tok * 128 + (((kc & 7) ^ (tok & 7)) << 4), bf);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              mma_16816(sc[jb], qa[part][ks], bf[0], bf[1]);
              mma_16816(sc[jb + 1], qa[part][ks], bf[2], bf[3]);
            }
          }
        }
        // positional: the k_r rows as B fragments, the same way (plain rows of 2 DR bytes)
#pragma unroll
        for (int ks = 0; ks < KSR; ++ks) {
#pragma unroll
          for (int jb = 0; jb < 8; jb += 2) {
            const int tok = 8 * jb + 8 * (lane >> 4) + (lane & 7);
            uint32_t bf[4];
            ldsm_x4(krbase + tok * (2 * DR) + (16 * ks + 8 * ((lane >> 3) & 1)) * 2, bf);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              mma_16816(sc[jb], qa[part][KSV + ks], bf[0], bf[1]);
              mma_16816(sc[jb + 1], qa[part][KSV + ks], bf[2], bf[3]);
            }
          }
        }
        if constexpr (KR8) {
#pragma unroll
          for (int jb = 0; jb < 8; jb += 4) {
            const int tok = 8 * jb + 8 * (lane >> 3) + (lane & 7);
            uint32_t bf[4];
            ldsm_x4(krbase + tok * (2 * DR) + 32 * KSR, bf);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int part = 0; part < 2; ++part) mma_1688(sc[jb + i], qat[part][0], qat[part][1], bf[i]);
          }
        }
        // online softmax along each row (column pair c = 8 rh + gid: query q0 + c/R, head c%R):
        // this thread's tokens, then the row's four lanes.  Query q of nq reads tokens
        // j < nrem - (nq - 1 - q) of this tile; most tiles are seen whole by every query.
        float al[RH];
        auto softmax_qm = [&](auto masked) {
          constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
          for (int rh = 0; rh < RH; ++rh) {
            const int c = 8 * rh + gid;
            const int lim = kMasked ? min(nv, nrem - (a.nq - 1 - (a.q0 + (c < RQ ? c / R : 0)))) : kBlockTokens;
            float mx = -INFINITY;
#pragma unroll
            for (int jb = 0; jb < 8; ++jb)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                if (kMasked && 8 * jb + 2 * tq + e >= lim) sc[jb][2 * rh + e] = -INFINITY;
                mx = fmaxf(mx, sc[jb][2 * rh + e]);
              }
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 2));
            const float mn = fmaxf(mq[rh], mx);
            const bool none = kMasked && mn == -INFINITY;
            al[rh] = none || mn == mq[rh] ? 1.f : fast_exp2(mq[rh] - mn);
            mq[rh] = mn;
            float ps = 0.f;
#pragma unroll
            for (int jb = 0; jb < 8; ++jb)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float pv = none ? 0.f : fast_exp2(sc[jb][2 * rh + e] - mn);
                sc[jb][2 * rh + e] = pv;
                ps += pv;
              }
            lq[rh] = fmaf(lq[rh], al[rh], ps);
          }
        };
        if (nrem - (a.nq - 1 - a.q0) >= kBlockTokens)
          softmax_qm(std::false_type{});
        else
          softmax_qm(std::true_type{});
        // rescale the accumulators (columns 2tq, 2tq + 1 of a row half: the factors of the rows
        // that lanes 8tq and 8tq + 4 hold), skipped by the whole warp when no maximum moved
        bool moved = false;
#pragma unroll
        for (int rh = 0; rh < RH; ++rh) moved |= al[rh] != 1.f;
        if (__any_sync(kFullMask, moved)) {
#pragma unroll
          for (int rh = 0; rh < RH; ++rh) {
            const float a0 = __shfl_sync(kFullMask, al[rh], 8 * tq);
            const float a1 = __shfl_sync(kFullMask, al[rh], 8 * tq + 4);
#pragma unroll
            for (int md = 0; md < MD; ++md) {
              oq[rh][md][0] *= a0;
              oq[rh][md][1] *= a1;
              oq[rh][md][2] *= a0;
              oq[rh][md][3] *= a1;
            }
          }
        }
        // output: O^T[d x pairs] += V^T[d x tok] P^T[tok x pairs], the probabilities' bf16 high
        // parts and remainders as two B operands taken straight from the score fragments
        // (tokens 2tq, 2tq + 1 of column blocks 2kt and 2kt + 1)
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          uint32_t bh[RH][2], bl[RH][2];
#pragma unroll
          for (int rh = 0; rh < RH; ++rh)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const float x0 = sc[2 * kt + h2][2 * rh], x1 = sc[2 * kt + h2][2 * rh + 1];
              const uint32_t hi = pack2_bf16(x0, x1);
              bh[rh][h2] = hi;
              bl[rh][h2] = pack2_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
            }
          const int tok = 16 * kt + tr_tok;
          const int jt = 16 * kt + 2 * tq;  // tokens of this thread's A-fragment halves
#pragma unroll
          for (int md = 0; md < MD; ++md) {
            const int dc = 2 * md + tr_dc;
            uint32_t af[4];
            ldsm_x4_trans(vbase + (dc >> 3) * kSubTileBytes + tok * 128 + (((dc & 7) ^ (tok & 7)) << 4), af);
            if (nv < kBlockTokens) {  // slots past the context may hold anything: zero them
              af[0] = mask_pair(af[0], jt, nv);
              af[1] = mask_pair(af[1], jt, nv);
              af[2] = mask_pair(af[2], jt + 8, nv);
              af[3] = mask_pair(af[3], jt + 8, nv);
            }
#pragma unroll
            for (int rh = 0; rh < RH; ++rh) {
              mma_16816(oq[rh][md], af, bh[rh][0], bh[rh][1]);
              mma_16816(oq[rh][md], af, bl[rh][0], bl[rh][1]);
            }
          }
        }
      } else {
      // fp8 cache: the scale 2^e of the tokens this thread's score rows hold (16mt + gid and
      // 16mt + gid + 8); E, the largest exponent among the tile's valid tokens, no lower than
      // -112 (so that 2^(14 - E) and 2^(E - 14) are normal floats); and each token's factor
      // 2^(e - E + 14) for its probability, 0 for slots past the context (they may hold any
      // byte: their exponent is clamped and left out of E)
      float fsc[4][2];
      float pfac[4][2];
      int emax = -112;
      if constexpr (F8) {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int tok = 16 * mt + gid + 8 * hh;
            const int e = max(ld_shared_s8(exbase + tok), -126);
            fsc[mt][hh] = exp2_int(e);
            if (tok < nv) emax = max(emax, e);
          }
        emax = max(emax, __shfl_xor_sync(kFullMask, emax, 4));
        emax = max(emax, __shfl_xor_sync(kFullMask, emax, 8));
        emax = max(emax, __shfl_xor_sync(kFullMask, emax, 16));
        const float pscale = exp2_int(14 - emax);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) pfac[mt][hh] = 16 * mt + gid + 8 * hh < nv ? fsc[mt][hh] * pscale : 0.f;
      }

      // scores
      float sc[NT][4][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][mt][e] = 0.f;
      if constexpr (kQS) {
        // each k-step's B fragments from the staged operand, once per tile: matrices (n +0..7,
        // k +0..7), (n +0..7, k +8..15), (n +8..15, k +0..7), (n +8..15, k +8..15)
        const uint32_t qb0 = smem_addr(qops + warp * kQopBytes);
        const uint32_t qlane = qb0 + (8 * (lane >> 4) + (lane & 7)) * QST + 16 * ((lane >> 3) & 1);
#pragma unroll
        for (int ks = 0; ks < KSV + KSR; ++ks) {
          uint32_t bq[NT][2];
#pragma unroll
          for (int np = 0; np < NT / 2; ++np) {
            uint32_t r4[4];
            ldsm_x4(qlane + 16 * np * QST + 32 * ks, r4);
            bq[2 * np][0] = r4[0];
            bq[2 * np][1] = r4[1];
            bq[2 * np + 1][0] = r4[2];
            bq[2 * np + 1][1] = r4[3];
          }
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            const int row = 16 * mt + ld_row;
            uint32_t af[4];
            if (ks < KSV) {
              const int kc = 2 * ks + ld_kc;
              ldsm_x4(kbase + (kc >> 3) * kSubTileBytes + row * 128 + (((kc & 7) ^ (row & 7)) << 4), af);
            } else {
              ldsm_x4(krbase + row * (2 * DR) + (2 * (ks - KSV) + ld_kc) * 16, af);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(sc[nt][mt], af, bq[nt][0], bq[nt][1]);
          }
        }
        if constexpr (KR8) {
          // the trailing k8 step: one matrix per n-tile (n +8i..+7, k 16(KSV + KSR) .. +7)
          uint32_t bt[2];
          ldsm_x2(qb0 + (8 * ((lane >> 3) & 1) + (lane & 7)) * QST + 32 * (KSV + KSR), bt[0], bt[1]);
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            const int row = 16 * mt + ld_row;
            uint32_t a0, a1;
            ldsm_x2(krbase + row * (2 * DR) + (2 * KSR) * 16, a0, a1);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_1688(sc[nt][mt], a0, a1, bt[nt]);
          }
        }
      } else {
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int row = 16 * mt + ld_row;
        if constexpr (F8) {
#pragma unroll
          for (int kp = 0; kp < KSV / 2; ++kp) {
            // matrices: (tokens +0..7, chunk 2kp), (+8..15, 2kp), (+0..7, 2kp+1), (+8..15, 2kp+1)
            uint32_t r4[4];
            ldsm_x4(kbase + 16 * DV * mt + f8_off[kp], r4);
            uint32_t af[4], ag[4];
            e4m3x4_to_f16x2x2(r4[0], af[0], af[2]);
            e4m3x4_to_f16x2x2(r4[1], af[1], af[3]);
            e4m3x4_to_f16x2x2(r4[2], ag[0], ag[2]);
            e4m3x4_to_f16x2x2(r4[3], ag[1], ag[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816_f16(sc[nt][mt], af, qb[nt][2 * kp][0], qb[nt][2 * kp][1]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_16816_f16(sc[nt][mt], ag, qb[nt][2 * kp + 1][0], qb[nt][2 * kp + 1][1]);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {  // content score times the token's scale
            sc[nt][mt][0] *= fsc[mt][0];
            sc[nt][mt][1] *= fsc[mt][0];
            sc[nt][mt][2] *= fsc[mt][1];
            sc[nt][mt][3] *= fsc[mt][1];
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < KSV; ++ks) {
            const int kc = 2 * ks + ld_kc;
            const uint32_t addr = kbase + (kc >> 3) * kSubTileBytes + row * 128 + (((kc & 7) ^ (row & 7)) << 4);
            uint32_t af[4];
            ldsm_x4(addr, af);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(sc[nt][mt], af, qb[nt][ks][0], qb[nt][ks][1]);
          }
        }
#pragma unroll
        for (int ks = 0; ks < KSR; ++ks) {
          uint32_t af[4];
          ldsm_x4(krbase + row * (2 * DR) + (2 * ks + ld_kc) * 16, af);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816(sc[nt][mt], af, qb[nt][KSV + ks][0], qb[nt][KSV + ks][1]);
        }
        if (KR8) {
          uint32_t a0, a1;
          ldsm_x2(krbase + row * (2 * DR) + (2 * KSR) * 16, a0, a1);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_1688(sc[nt][mt], a0, a1, qt[nt]);
        }
      }
      }

      // online softmax (log2 domain); thread holds column pair c = nt*4 + tq (query q0 + c/R,
      // head c%R) for tokens 16*mt + gid and 16*mt + gid + 8.  Query q of nq reads positions
      // up to T - nq + q: in this tile, tokens j < nrem - (nq - 1 - q).  Most tiles are seen
      // whole by every query of the pass (the earliest one is q0) and take the unmasked form;
      // the masked form also keeps the state of a query that sees no token of the tile (its
      // position precedes the tile) unchanged.
      uint32_t pb[NO][4][2];               // B operands: the probabilities (wide: their high parts)
      uint32_t pl[kWide ? NO : 1][4][2];   // wide: the remainders
      float pr[kWide ? NT : 1][4][2];      // wide: this tile's probabilities, packed below
      float al[NT];                        // wide: each column pair's rescale factor
      auto ex2 = [&](float x) {
        if constexpr (kFastExp)
          return fast_exp2(x);
        else
          return exp2f(x);
      };
      auto softmax = [&](auto masked) {
        constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float sv[4][2];
          float mx = -INFINITY;
          if constexpr (kMasked) {
            const int cp = nt * 4 + tq;
            const int lim = min(nv, nrem - (a.nq - 1 - (a.q0 + (cp < RQc ? (cp + cp0) / R : 0))));
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
              const int j0 = 16 * mt + gid;
              sv[mt][0] = j0 < lim ? sc[nt][mt][0] + sc[nt][mt][1] : -INFINITY;
              sv[mt][1] = j0 + 8 < lim ? sc[nt][mt][2] + sc[nt][mt][3] : -INFINITY;
              mx = fmaxf(mx, fmaxf(sv[mt][0], sv[mt][1]));
            }
          } else {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
              sv[mt][0] = sc[nt][mt][0] + sc[nt][mt][1];
              sv[mt][1] = sc[nt][mt][2] + sc[nt][mt][3];
              mx = fmaxf(mx, fmaxf(sv[mt][0], sv[mt][1]));
            }
          }
          mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 16));
          const float mn = fmaxf(m[nt], mx);
          const bool none = kMasked && mn == -INFINITY;
          const float alpha = none || (kWide && mn == m[nt]) ? 1.f : ex2(m[nt] - mn);
          m[nt] = mn;
          float ps = 0.f;
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            const float p0 = none ? 0.f : ex2(sv[mt][0] - mn);
            const float p1 = none ? 0.f : ex2(sv[mt][1] - mn);
            ps += p0 + p1;
            if constexpr (kWide) {
              pr[nt][mt][0] = p0;
              pr[nt][mt][1] = p1;
            } else {
              pb[nt][mt][0] = movmatrix_trans(split_pack(p0));
              pb[nt][mt][1] = movmatrix_trans(split_pack(p1));
            }
          }
          l[nt] = fmaf(l[nt], alpha, ps);
          if constexpr (kWide) {
            al[nt] = alpha;
          } else {
#pragma unroll
            for (int md = 0; md < MD; ++md)
#pragma unroll
              for (int e = 0; e < 4; ++e) o[nt][md][e] *= alpha;
          }
        }
      };
      if constexpr (!CAUSAL) {
        // one query per sequence at its last position: only the tokens past the end of the
        // context are masked
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float sv[4][2];
          float mx = -INFINITY;
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            const int j0 = 16 * mt + gid;
            sv[mt][0] = j0 < nv ? sc[nt][mt][0] + sc[nt][mt][1] : -INFINITY;
            sv[mt][1] = j0 + 8 < nv ? sc[nt][mt][2] + sc[nt][mt][3] : -INFINITY;
            mx = fmaxf(mx, fmaxf(sv[mt][0], sv[mt][1]));
          }
          mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 16));
          const float mn = fmaxf(m[nt], mx);
          const float alpha = kWide && mn == m[nt] ? 1.f : ex2(m[nt] - mn);
          m[nt] = mn;
          float ps = 0.f;
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            const float p0 = ex2(sv[mt][0] - mn);
            const float p1 = ex2(sv[mt][1] - mn);
            ps += p0 + p1;
            if constexpr (kWide) {
              pr[nt][mt][0] = p0;
              pr[nt][mt][1] = p1;
            } else if constexpr (F8) {
              // p_j 2^(e_j - E + 14) as one f16 (11 bits, far beyond the codes' 4; the second
              // column of the head stays 0)
              pb[nt][mt][0] = movmatrix_trans(__half_as_ushort(__float2half_rn(p0 * pfac[mt][0])));
              pb[nt][mt][1] = movmatrix_trans(__half_as_ushort(__float2half_rn(p1 * pfac[mt][1])));
            } else {
              pb[nt][mt][0] = movmatrix_trans(split_pack(p0));
              pb[nt][mt][1] = movmatrix_trans(split_pack(p1));
            }
          }
          l[nt] = fmaf(l[nt], alpha, ps);
          if constexpr (kWide) {
            al[nt] = alpha;
          } else {
#pragma unroll
            for (int md = 0; md < MD; ++md)
#pragma unroll
              for (int e = 0; e < 4; ++e) o[nt][md][e] *= alpha;
          }
        }
      } else if (nrem - (a.nq - 1 - a.q0) >= kBlockTokens) {
        softmax(std::false_type{});
      } else {
        softmax(std::true_type{});
      }
      if constexpr (kWide) {
        // rescale the accumulators, skipped by the whole warp when no running maximum moved
        bool moved = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) moved |= al[nt] != 1.f;
        if (__any_sync(kFullMask, moved)) {
#pragma unroll
          for (int no = 0; no < NO; ++no)
#pragma unroll
            for (int md = 0; md < MD; ++md) {
              o[no][md][0] *= al[2 * no];
              o[no][md][1] *= al[2 * no + 1];
              o[no][md][2] *= al[2 * no];
              o[no][md][3] *= al[2 * no + 1];
            }
        }
        // high parts and remainders of n-tiles 2no and 2no+1 (columns 2tq and 2tq+1 of the
        // 8x8 blocks that movmatrix turns into B fragments)
#pragma unroll
        for (int no = 0; no < NO; ++no)
#pragma unroll
          for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const float x0 = pr[2 * no][mt][hh], x1 = pr[2 * no + 1][mt][hh];
              const uint32_t hi = pack2_bf16(x0, x1);
              pb[no][mt][hh] = movmatrix_trans(hi);
              pl[no][mt][hh] = movmatrix_trans(pack2_bf16(x0 - __uint_as_float(hi << 16),
                                                          x1 - __uint_as_float(hi & 0xffff0000u)));
            }
      }

      // output: O^T[d x n] += V^T[d x tok] P[tok x n]
      if constexpr (F8) {
        float ot[NT][MD][4];  // this tile's product, in units of 2^(E - 14)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int md = 0; md < MD; ++md)
#pragma unroll
            for (int e = 0; e < 4; ++e) ot[nt][md][e] = 0.f;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          const int jt = 16 * kt + 2 * tq;
#pragma unroll
          for (int cp = 0; cp < MD / 2; ++cp) {
            // matrices (tokens +0..7, chunk 2cp), (+8..15, 2cp), (+0..7, 2cp+1), (+8..15, 2cp+1),
            // transposed: a lane gets bytes (d, d+1) of tokens (t, t+1), d = 2gid, t = 2tq; the
            // permutation makes the low half tokens (t, t+1) of row d and the high half of row d+1
            uint32_t x4[4];
            ldsm_x4_trans(vbase + 16 * DV * kt + f8_off[cp], x4);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t af[4];
              e4m3x4_to_f16x2x2(byte_perm(x4[2 * h2], 0x3120), af[0], af[1]);
              e4m3x4_to_f16x2x2(byte_perm(x4[2 * h2 + 1], 0x3120), af[2], af[3]);
              if (nv < kBlockTokens) {  // slots past the context may hold any byte: zero them
                af[0] = mask_pair(af[0], jt, nv);
                af[1] = mask_pair(af[1], jt, nv);
                af[2] = mask_pair(af[2], jt + 8, nv);
                af[3] = mask_pair(af[3], jt + 8, nv);
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) mma_16816_f16(ot[nt][2 * cp + h2], af, pb[nt][kt][0], pb[nt][kt][1]);
            }
          }
        }
        const float unit = exp2_int(emax - 14);  // exact: a power of two
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int md = 0; md < MD; ++md)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[nt][md][e] = fmaf(ot[nt][md][e], unit, o[nt][md][e]);
      } else {
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        const int tok = 16 * kt + tr_tok;
        const int jt = 16 * kt + 2 * tq;  // tokens of this thread's A-fragment halves
#pragma unroll
        for (int md = 0; md < MD; ++md) {
          const int dc = 2 * md + tr_dc;
          const uint32_t addr = vbase + (dc >> 3) * kSubTileBytes + tok * 128 + (((dc & 7) ^ (tok & 7)) << 4);
          uint32_t af[4];
          ldsm_x4_trans(addr, af);
          if (nv < kBlockTokens) {  // slots past the context may hold anything: zero them
            af[0] = mask_pair(af[0], jt, nv);
            af[1] = mask_pair(af[1], jt, nv);
            af[2] = mask_pair(af[2], jt + 8, nv);
            af[3] = mask_pair(af[3], jt + 8, nv);
          }
          if constexpr (kWide) {
#pragma unroll
            for (int no = 0; no < NO; ++no) {
              mma_16816(o[no][md], af, pb[no][kt][0], pb[no][kt][1]);
              mma_16816(o[no][md], af, pl[no][kt][0], pl[no][kt][1]);
            }
          } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(o[nt][md], af, pb[nt][kt][0], pb[nt][kt][1]);
          }
        }
      }
      }
      }
    }
    // the stage may be refilled (after this warp's own writes into it, if any, are ordered
    // before the copy engine's)
    if constexpr (kSelfFed) {
      const int inext = i_own + D;
      if (inext < n_own) {
        if (inext - f0 >= 32) {  // the next batch of block ids becomes current
          f0 += 32;
          fb = xb;
          fg = xg;
          fv = xv;
          lookup(warp, P, n_own, f0 + 32, xb, xg, xv);
        }
        const int bj = __shfl_sync(kFullMask, fb, inext - f0);
        const int gj = __shfl_sync(kFullMask, fg, inext - f0);
        const int vj = __shfl_sync(kFullMask, fv, inext - f0);
        fence_proxy_async_smem();  // this warp's reads of the stage come before the copy's writes
        __syncwarp();
        if (lane == 0) issue(s, bj, gj, vj);
      }
      ++i_own;
    } else {
      if (FUSED && !kPatcher && patched) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    k += NC;
    if (k >= n) break;
    const int pb_ = cc.b, pg = cc.g;
    cursor_advance(cc, NC, cum, a.B, a.G);
    if (cc.b != pb_ || cc.g != pg) {  // segment boundary: emit, start the next (b, g)
      flush(segment_of(pg, pb_, a.B));
      reset_state();
      load_q(cc.b, cc.g);
    }
    if (++slot == D) {
      slot = 0;
      ph ^= 1;
    }
  }
  if (ok) {
    flush(segment_of(cc.g, cc.b, a.B));
    return;
  }
  // A copy never arrived: report, and leave empty records for every segment still owed so
  // the combine reads defined values.  (The copy warp waits for its copies in flight; a
  // self-fed consumer waits for its own: units i_own .. i_own + D - 1.)
  if (lane == 0) {
    flag_error(a.err, GVA_DEVERR_TIMEOUT);
    if constexpr (kSelfFed)
      for (int j = i_own; j < min(i_own + D, n_own); ++j) (void)mbar_wait_bounded(&full[warp * D + j % D], (j / D) & 1);
  }
  reset_state();
  flush(segment_of(cc.g, cc.b, a.B));
  for (k += NC; k < n; k += NC) {
    const int pb_ = cc.b, pg = cc.g;
    cursor_advance(cc, NC, cum, a.B, a.G);
    if (cc.b != pb_ || cc.g != pg) flush(segment_of(cc.g, cc.b, a.B));
  }
}

template <int DV, int DR, int R, int NQ, bool CAUSAL, bool SEPK, bool FUSED, bool F8 = false>
cudaError_t launch_mma_t(const DecodeArgs& a, const CUtensorMap& mv, const CUtensorMap& mk, int grid,
                         cudaStream_t stream) {
  using L = MmaLayout<DV, DR, SEPK, F8>;
  const int P = a.group_warps, D = a.n_stages;
  constexpr int CPC = mma_consumers_per_copy_warp(DV, DR, F8);
  constexpr bool kSplit = mma_query_in_smem(DV, R * NQ) && !F8 && !SEPK;
  const int warps = (kSplit ? 2 * P : P) + (mma_self_fed(DV, CAUSAL, F8) ? 0 : P / CPC);
  if (P < 1 || P % CPC || 32 * warps > mma_kernel_threads(DV, R * NQ, NQ) || D < 1 || P * D > kMaxStages)
    return cudaErrorInvalidValue;
  if (a.nqp != NQ || (a.nq > 1) != CAUSAL || (a.fused != 0) != FUSED) return cudaErrorInvalidValue;
  const int smem = ring_fixed_bytes(a.B) + P * D * L::kStageBytes + P * (F8 || SEPK ? 0 : mma_qop_bytes(DV, DR, R * NQ));
  if (smem > kSmemLimit) return cudaErrorInvalidValue;
  // the fused step fills the instance's thread budget with prologue warps, and the shared
  // memory budget with query stages; its patcher warp is the first prologue warp
  const int threads = FUSED ? mma_max_threads(DV, NQ) : 32 * warps;
  if (FUSED && !(DV == 64 && F8) && threads <= 32 * warps) return cudaErrorInvalidValue;
  DecodeArgs args = a;
  args.spare_smem = FUSED ? kSmemLimit - smem : 0;
  const int dyn_smem = FUSED ? kSmemLimit : smem;
  auto kern = decode_mma_kernel<DV, DR, R, NQ, CAUSAL, SEPK, FUSED, F8>;
  static int configured[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= kMaxDevices || !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    if (dev < kMaxDevices) configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = dyn_smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args, mv, mk);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace
}  // namespace gva
