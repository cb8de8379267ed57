// gva_noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// gva_decode_attention needs scratch for its split-T partial results, and it expects the
// caller to pass that scratch in.  Some callers have no way to get it: an operator plugged
// into a host framework that hands over only its input and output buffers, an engine that
// has already given every byte of the GPU to its own pools, or a latency-critical loop where
// a call into the CUDA allocator (which may synchronise the device and takes an unbounded
// time) is not acceptable.  For them this file keeps the scratch in a fixed array that is
// part of the library's device image: the driver places it on every GPU that loads the
// library and it stays there until the process exits.  Nothing here allocates.
#include <mutex>

#include "gva_internal.h"

namespace {

// Scratch shared by every call of gva_decode_attention_noalloc on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GVA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up once per device.  In host code the
// array's name is only a host-side handle, never a device address, so it must not be
// handed to a kernel directly.
void* g_scratch_addr[gva::kMaxDevicesHost] = {};
std::mutex g_scratch_mutex;

gva_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GVA_ERR_CUDA;
  if (dev < 0 || dev >= gva::kMaxDevicesHost) return GVA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GVA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GVA_OK;
}

}  // namespace

extern "C" gva_status gva_decode_attention_noalloc(gva_ctx* ctx, int B, const float* q_abs,
                                                   const float* q_rot, const void* v_pool,
                                                   const void* kr_pool,
                                                   const int32_t* block_table, int max_blocks,
                                                   int num_blocks, const int32_t* seq_lens,
                                                   int max_seq_len, float* out,
                                                   gva_stream_t stream) {
  if (!ctx || B < 0 || max_seq_len < 1) return GVA_ERR_INVALID_ARG;
  if (B == 0) return GVA_OK;
  const size_t need = gva_decode_workspace_size(ctx, B, max_seq_len);
  if (need == 0) return GVA_ERR_UNSUPPORTED;
  if (need > GVA_NOALLOC_SCRATCH_BYTES) return GVA_ERR_WORKSPACE;  // batch too large for the fixed scratch
  void* scratch = nullptr;
  const gva_status st = scratch_address(&scratch);
  if (st != GVA_OK) return st;
  // The partial records are written in full before they are read, so the array needs no
  // clearing between calls.
  return gva_decode_attention(ctx, B, q_abs, q_rot, v_pool, kr_pool, block_table, max_blocks,
                              num_blocks, seq_lens, max_seq_len, out, scratch,
                              GVA_NOALLOC_SCRATCH_BYTES, stream);
}
