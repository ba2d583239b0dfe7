// mla_decode_noalloc: the mla_decode entry point for callers that cannot allocate.
//
// mla_decode splits each request's keys over many SMs and needs device scratch for the
// per-split partial results, which its caller normally allocates (see
// mla_decode_workspace_size).  Some callers cannot do that at decode time: a runtime
// whose memory is planned once at start-up and may not call cudaMalloc/cudaFree (or a
// caching allocator) on the decode path, a host program that links only this C library
// and owns no allocator, or a replayed sequence of launches that must not change the
// allocation state.  This entry point takes the scratch from one fixed array that the
// library declares in device memory instead; the caller passes only inputs and outputs.
//
// Limits:
//   * The array is kNoAllocScratchBytes (64 MiB) per device and every GPU that loads the
//     library keeps it until the process exits.  A call whose split-KV scratch would not
//     fit is rejected with MLA_ERR_UNSUPPORTED before anything is launched.
//   * All calls on a device share the array, which keeps the last call's contents.
//     Calls whose kernels overlap on the GPU (different streams, or different host
//     threads) race on it and must be serialised by the caller.  No part of the scratch
//     needs to start at zero: each call writes every word before reading it.
//   * The first call on a device looks up the array's device address with that device
//     current (cudaGetSymbolAddress, once per device); make that first call before any
//     stream capture.
//   * It calls no cudaMalloc, cudaFree or allocating library routine.
#include <cuda_runtime.h>

#include "internal.h"
#include "../../include/mla_decode.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;

// The scratch.  In host code this name is a host-side stand-in, not a device address:
// the device address comes from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

}  // namespace

extern "C" int mla_decode_noalloc(const void* q, const void* kv_cache, const int32_t* block_table,
                                  int64_t bt_stride, const int32_t* seq_lens,
                                  const int32_t* causal_seqlens_global, int B, int H, int q_len,
                                  int block_size, int num_blocks, int max_blocks, int cp_world,
                                  int cp_rank, float scale, void* out, float* lse,
                                  int lse_base_e, mla_stream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return mla::api_fail(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return mla::api_fail(MLA_ERR_UNSUPPORTED, "mla_decode_noalloc: device index %d", dev);
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess)
    return mla::api_fail(MLA_ERR_CUDA, "mla_decode_noalloc: %s", cudaGetErrorString(e));
  if (B > 0 && H > 0 && q_len > 0) {
    const size_t need = mla::decode_workspace_for(B, H, q_len, sms, block_size);
    if (need > kNoAllocScratchBytes)
      return mla::api_fail(MLA_ERR_UNSUPPORTED,
                           "mla_decode_noalloc: B=%d H=%d q_len=%d needs %zu bytes of split-KV "
                           "scratch, more than the library's fixed %zu; use mla_decode with a "
                           "caller workspace",
                           B, H, q_len, need, kNoAllocScratchBytes);
  }
  if (g_scratch_ptr[dev] == nullptr) {
    // once per device, with that device current: the array's device address
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess)
      return mla::api_fail(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetSymbolAddress: %s",
                           cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  return mla_decode(q, kv_cache, block_table, bt_stride, seq_lens, causal_seqlens_global, B, H,
                    q_len, block_size, num_blocks, max_blocks, cp_world, cp_rank, scale, out, lse,
                    lse_base_e, g_scratch_ptr[dev], kNoAllocScratchBytes, stream);
}
