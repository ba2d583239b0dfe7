// mla_decode_noalloc: the mla_decode entry point for callers that cannot allocate.
//
// mla_decode splits each request's keys over many SMs and needs device scratch for the
// per-split partial results, which its caller normally allocates (see
// mla_decode_workspace_size).  Some callers cannot do that at decode time: a runtime
// whose memory is planned once at start-up and may not call cudaMalloc/cudaFree (or a
// caching allocator) on the decode path, or a host program that links only this C library
// and owns no allocator.  This entry point takes the scratch from one fixed array that
// the library declares in device memory instead; the caller passes only inputs and
// outputs.
//
// Limits:
//   * The array is kNoAllocScratchBytes (64 MiB) per device and every GPU that loads the
//     library keeps it until the process exits.  A call whose split-KV scratch would not
//     fit is rejected with MLA_ERR_UNSUPPORTED before anything is launched (after the
//     same argument checks as mla_decode, so a bad argument gets mla_decode's error).
//   * All calls on a device share the array, which keeps the last call's contents.
//     Calls whose kernels overlap on the GPU (different streams, or different host
//     threads) race on it and must be serialised by the caller.  No part of the scratch
//     needs to start at zero: each call writes every word before reading it.
//   * The first call on a device looks up the array's device address with that device
//     current (cudaGetSymbolAddress, once per device); make that first call before any
//     stream capture.
//   * It calls no cudaMalloc, cudaFree or allocating library routine.
#include <atomic>
#include <functional>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "../../include/mla_decode.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;

// The scratch.  In host code this name is a host-side stand-in, not a device address:
// the device address comes from cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// The array's device address on each device, looked up once per device with that device
// current (std::call_once: safe when several host threads make their first call at once).
struct ScratchPtr {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  void* ptr = nullptr;
};
ScratchPtr g_scratch[kMaxDevices];

void resolve_scratch(ScratchPtr& s) { s.err = cudaGetSymbolAddress(&s.ptr, g_noalloc_scratch); }

}  // namespace

extern "C" int mla_decode_noalloc(const void* q, const void* kv_cache, const int32_t* block_table,
                                  int64_t bt_stride, const int32_t* seq_lens,
                                  const int32_t* causal_seqlens_global, int B, int H, int q_len,
                                  int causal, int block_size, int num_blocks, int max_blocks,
                                  int cp_world, int cp_rank, int interleave, float scale,
                                  void* out, float* lse, int lse_base_e, mla_stream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return mla::api_fail(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return mla::api_fail(MLA_ERR_UNSUPPORTED, "mla_decode_noalloc: device index %d", dev);
  ScratchPtr& sp = g_scratch[dev];
  std::call_once(sp.once, resolve_scratch, std::ref(sp));
  if (sp.err != cudaSuccess)
    return mla::api_fail(MLA_ERR_CUDA, "mla_decode_noalloc: cudaGetSymbolAddress: %s",
                         cudaGetErrorString(sp.err));
  // every argument is checked as mla_decode checks it; only then is the size of the
  // split-KV scratch compared with the array's
  return mla::decode_entry("mla_decode_noalloc", q, kv_cache, block_table, bt_stride, seq_lens,
                           causal_seqlens_global, B, H, q_len, causal, block_size, num_blocks,
                           max_blocks, cp_world, cp_rank, interleave, 1, scale, out, lse,
                           lse_base_e, sp.ptr, kNoAllocScratchBytes, true, stream);
}
