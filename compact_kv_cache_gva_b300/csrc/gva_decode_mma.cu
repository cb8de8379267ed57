// gva_decode_mma.cu -- tensor-core decode path (bf16 cache).  Not built yet: every shape
// reports unsupported, so the CUDA-core path runs.
#include "gva_device.cuh"
#include "gva_internal.h"

namespace gva {

bool mma_supported(const gva_dims&, bool) { return false; }
int mma_ctas_per_sm(const gva_dims&, bool) { return 1; }
int mma_tiles_per_cta_unit(const gva_dims&) { return 4; }
cudaError_t launch_decode_mma(const DecodeArgs&, bool, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gva
