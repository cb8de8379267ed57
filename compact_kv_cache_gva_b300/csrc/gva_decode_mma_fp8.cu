// gva_decode_mma_fp8.cu -- the tensor-core decode kernel's instances over the fp8 value cache
// (E4M3 codes with a power-of-two scale per (token, group), bf16 positional keys): the plain
// split-T pass and the fused decode step, one query per sequence.  The kernel is in
// gva_decode_mma.cuh; the layout of the value pool is in include/gva.h.
#include "gva_decode_mma.cuh"

namespace gva {
namespace {

template <int DV, int DR, int R>
cudaError_t dispatch_fused(const DecodeArgs& a, const CUtensorMap& mv, int grid, cudaStream_t stream) {
  if (a.nq != 1 || a.nqp != 1) return cudaErrorInvalidValue;
  if (a.fused) return launch_mma_t<DV, DR, R, 1, false, false, true, true>(a, mv, mv, grid, stream);
  return launch_mma_t<DV, DR, R, 1, false, false, false, true>(a, mv, mv, grid, stream);
}

template <int DV, int DR>
cudaError_t dispatch_r(const DecodeArgs& a, const CUtensorMap& mv, int grid, cudaStream_t stream) {
  switch (a.H / a.G) {
    case 1: return dispatch_fused<DV, DR, 1>(a, mv, grid, stream);
    case 2: return dispatch_fused<DV, DR, 2>(a, mv, grid, stream);
    case 4: return dispatch_fused<DV, DR, 4>(a, mv, grid, stream);
    case 8: return dispatch_fused<DV, DR, 8>(a, mv, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int DV>
cudaError_t dispatch_dr(const DecodeArgs& a, const CUtensorMap& mv, int grid, cudaStream_t stream) {
  switch (a.d_r) {
    case 0: return dispatch_r<DV, 0>(a, mv, grid, stream);
    case 8: return dispatch_r<DV, 8>(a, mv, grid, stream);
    case 16: return dispatch_r<DV, 16>(a, mv, grid, stream);
    case 24: return dispatch_r<DV, 24>(a, mv, grid, stream);
    case 32: return dispatch_r<DV, 32>(a, mv, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

// The codes of an fp8 value pool seen as a 2-D byte tensor of 128-byte rows (NB*G*64*d_v/128
// rows); one box is one (block, group) tile, d_v/2 rows, swizzled in 128-byte rows.
bool make_code_map(CUtensorMap* map, const void* pool, int num_blocks, int G, int d_v) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(num_blocks) * G * kBlockTokens * d_v / 128};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(d_v / 2)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_decode_mma_fp8(const DecodeArgs& a, int grid, cudaStream_t stream) {
  CUtensorMap mv;
  if (!make_code_map(&mv, a.v_pool, a.num_blocks, a.G, a.d_v)) return cudaErrorInvalidValue;
  switch (a.d_v) {
    case 64: return dispatch_dr<64>(a, mv, grid, stream);
    case 128: return dispatch_dr<128>(a, mv, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gva
