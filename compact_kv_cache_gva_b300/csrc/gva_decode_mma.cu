// gva_decode_mma.cu -- the tensor-core decode kernel's bf16 instances, its plan (warp pairs and
// ring depth) and the launch entry point; the kernel itself is in gva_decode_mma.cuh.
#include "gva_decode_mma.cuh"

namespace gva {
namespace {

template <int DV, int DR, int R, bool SEPK>
cudaError_t dispatch_nq(const DecodeArgs& a, const CUtensorMap& mv, const CUtensorMap& mk, int grid,
                        cudaStream_t stream) {
  if constexpr (!SEPK) {
    if (a.fused) {
      if (a.nqp == 1 && a.nq == 1 && a.d_v == DV) return launch_mma_t<DV, DR, R, 1, false, SEPK, true>(a, mv, mk, grid, stream);
      return cudaErrorInvalidValue;
    }
    constexpr int kCols = mma_max_column_pairs(DV);  // (query, head) column pairs of a pass
    if constexpr (R * 4 <= kCols)
      if (a.nqp == 4) return launch_mma_t<DV, DR, R, 4, true, SEPK, false>(a, mv, mk, grid, stream);
    if constexpr (R * 2 <= kCols)
      if (a.nqp == 2) return launch_mma_t<DV, DR, R, 2, true, SEPK, false>(a, mv, mk, grid, stream);
    if (a.nqp == 1 && a.nq > 1) return launch_mma_t<DV, DR, R, 1, true, SEPK, false>(a, mv, mk, grid, stream);
  }
  if (a.fused) return cudaErrorInvalidValue;
  if (a.nqp == 1 && a.nq == 1) return launch_mma_t<DV, DR, R, 1, false, SEPK, false>(a, mv, mk, grid, stream);
  return cudaErrorInvalidValue;
}

template <int DV, int DR, bool SEPK>
cudaError_t dispatch_r(const DecodeArgs& a, const CUtensorMap& mv, const CUtensorMap& mk, int grid,
                       cudaStream_t stream) {
  switch (a.H / a.G) {
    case 1: return dispatch_nq<DV, DR, 1, SEPK>(a, mv, mk, grid, stream);
    case 2: return dispatch_nq<DV, DR, 2, SEPK>(a, mv, mk, grid, stream);
    case 4: return dispatch_nq<DV, DR, 4, SEPK>(a, mv, mk, grid, stream);
    case 8: return dispatch_nq<DV, DR, 8, SEPK>(a, mv, mk, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int DV>
cudaError_t dispatch_dr(const DecodeArgs& a, const CUtensorMap& mv, const CUtensorMap& mk, bool sep_k,
                        int grid, cudaStream_t stream) {
  if (sep_k) return dispatch_r<DV, 0, true>(a, mv, mk, grid, stream);
  switch (a.d_r) {
    case 0: return dispatch_r<DV, 0, false>(a, mv, mk, grid, stream);
    case 8: return dispatch_r<DV, 8, false>(a, mv, mk, grid, stream);
    case 16: return dispatch_r<DV, 16, false>(a, mv, mk, grid, stream);
    case 24: return dispatch_r<DV, 24, false>(a, mv, mk, grid, stream);
    case 32: return dispatch_r<DV, 32, false>(a, mv, mk, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
// columns x 64 rows, swizzled in 128-byte rows.
bool make_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int G, int d_v) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_v),
                              static_cast<cuuint64_t>(num_blocks) * G * kBlockTokens};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d_v) * 2};
  const cuuint32_t box[2] = {64, kBlockTokens};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mma_supported(const gva_dims& d, bool sep_k) {
  if (d.cache_dtype != GVA_BF16 && !(d.cache_dtype == GVA_FP8_E4M3 && !sep_k)) return false;
  if (!(d.d_v == 64 || d.d_v == 128)) return false;
  if (sep_k) {
    if (d.d_r != 0) return false;
  } else if (!(d.d_r == 0 || d.d_r == 8 || d.d_r == 16 || d.d_r == 24 || d.d_r == 32)) {
    return false;
  }
  const int r = d.H / d.G;
  return r == 1 || r == 2 || r == 4 || r == 8;
}

// Consumer warps and ring depth, from measurements on B300 (the d_r sweep of the long-context
// workload, 0 <= d_r <= 32, and the ragged batch): fewer than four consumers lose throughput
// even with deeper rings; with d_v = 64, four pairs are best up to d_r = 24 (stages up to
// 11 KB; five or six were 2-8 % slower) and six consumers at d_r = 32 (12 KB stages, 12 %
// faster than four; three copy warps fill them, mma_consumers_per_copy_warp); the 19 KB stages
// of d_v = 128 use three pairs (four give the same time with half the depth).  D takes the
// rest of shared memory.
// Queries per pass: the largest power of two up to 4 whose (query, head) column pairs fit,
// 16 (four n-tiles of hi/lo columns, about 240 registers at 256 threads at d_v = 64; the
// long-context four-query decode in one pass instead of two; at d_v = 128 with the query
// operand in shared memory, mma_query_in_smem, since as registers the sixteen pairs
// spilled 508 bytes).
int mma_max_queries_per_pass(int R, int d_v) {
  const int cols = mma_max_column_pairs(d_v);
  int q = 1;
  while (2 * q <= 4 && 2 * q * R <= cols) q *= 2;
  return q;
}

bool mma_shape(const gva_dims& d, bool sep_k, int B, int nqp, int* pairs, int* stages) {
  const bool f8 = d.cache_dtype == GVA_FP8_E4M3;
  if (f8 && (sep_k || nqp > 1)) return false;
  const int op = f8 ? kBlockTokens * d.d_v : (d.d_v / 64) * kSubTileBytes * (sep_k ? 2 : 1);
  const int stage = op + (sep_k ? 0 : kBlockTokens * d.d_r * 2) + (f8 ? kBlockTokens : 0);
  int avail = kSmemLimit - ring_fixed_bytes(B);
  auto depth = [&](int p) { return std::min(avail / (p * stage), kMaxStages / p); };
  // Several queries per pass double the consumers' work per tile: at d_v = 64 eight self-fed
  // consumers with two-slot rings (mma_self_fed; the long-context two-query decode 110 us,
  // against 115 and 128 us with seven or six consumers and three slots, and 120 us with four
  // warp pairs); at d_v = 128 as many pairs as fit (four rather than three: the ragged batch's
  // two-query decode 690 us against 817 us).
  // The fp8 cache's consumers do more work per byte than the bf16 ones: at d_v = 64 twelve
  // self-fed consumers fill the 384 threads (mma_self_fed; the long-context partial pass: 4
  // pairs 120 us, 6 pairs 108.6 us, 8 consumers with 4 copy warps 84.0 us, 12 self-fed
  // 82.0 us, and the fused pass 90.4 -> 84.5 us); at d_v = 128 three pairs.
  const int P = nqp > 1 ? (d.d_v == 64 ? 8 : mma_max_threads(d.d_v, nqp) / 64)
                : f8    ? (d.d_v == 64 ? 12 : 3)
                        : std::min(stage <= 11 * 1024 ? 4 : stage <= 12 * 1024 ? 6 : 3,
                                   mma_max_threads(d.d_v, nqp) / 64);
  // 16-pair passes at d_v = 128 keep each consumer's query operand in shared memory
  if (!f8 && !sep_k) avail -= P * mma_qop_bytes(d.d_v, d.d_r, (d.H / d.G) * nqp);
  const int D = depth(P);
  if (D < 1) return false;
  *pairs = P;
  *stages = D;
  return true;
}

cudaError_t launch_decode_mma(const DecodeArgs& a, bool sep_k, int grid, cudaStream_t stream) {
  if (a.v_exp) return sep_k ? cudaErrorInvalidValue : launch_decode_mma_fp8(a, grid, stream);
  CUtensorMap mv, mk;
  if (!make_pool_map(&mv, a.v_pool, a.num_blocks, a.G, a.d_v)) return cudaErrorInvalidValue;
  if (sep_k) {
    if (!make_pool_map(&mk, a.k_pool, a.num_blocks, a.G, a.d_v)) return cudaErrorInvalidValue;
  } else {
    mk = mv;
  }
  switch (a.d_v) {
    case 64: return dispatch_dr<64>(a, mv, mk, sep_k, grid, stream);
    case 128: return dispatch_dr<128>(a, mv, mk, sep_k, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gva

