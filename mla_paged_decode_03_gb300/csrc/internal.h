// Internal launcher interface shared by the translation units of libmla_decode.so.
// Not part of the public ABI (include/mla_decode.h is).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mla {

// Arguments of one mla_decode call after host validation.
struct DecodeArgs {
  const uint16_t* q;             // bf16 [B*q_len*H, 576]
  const uint16_t* kv;            // bf16 [num_blocks*block_size, 576]
  const int32_t* block_table;    // [B, bt_stride]
  int64_t bt_stride;
  const int32_t* seq_lens;       // [B]
  const int32_t* gseq;           // [B] global lengths (seq_lens when cp_world == 1)
  int B, H, q_len, block_size, num_blocks, max_blocks, cp_world, cp_rank;
  // Requests per shard.  B == shard_B for one shard; a call over several shards has
  // B = n * shard_B, and its request b is request b % shard_B of q and gseq, in shard
  // cp_rank + b / shard_B (block_table, seq_lens, out and lse are shard-major).
  int shard_B;
  float scale;
  uint16_t* out;                 // bf16 [B*q_len*H, 512]
  float* lse;                    // [B*q_len*H] or null
  int lse_base_e;
  void* workspace;
  size_t workspace_bytes;
  int num_sms;
  unsigned int* status;          // device status word
};

// Split-KV decode: picks the tensor-core (tcgen05) kernel when the cache layout allows
// TMA tiles (block_size 16/32/64/128), else the warp-level MMA kernel.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
size_t decode_workspace_size(int B, int H, int q_len, int num_sms);

// tcgen05 / TMEM / TMA kernel (mla_decode_tc.cu)
bool tc_supported(const DecodeArgs& a);
size_t tc_workspace_size(int B, int H, int q_len, int num_sms);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream);

// warp-level mma.sync kernel (mla_decode_mma.cu)
size_t mma_workspace_size(int B, int H, int q_len, int num_sms);
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t stream);

// Split-KV scratch the kernel chosen for this block size uses at its preferred split.
size_t decode_workspace_for(int B, int H, int q_len, int num_sms, int block_size);

// Records a message for mla_last_error() and returns `code` (api.cu).
int api_fail(int code, const char* fmt, ...);

// Testing hook: 0 = automatic choice, 1 = force the warp-level kernel, 2 = force tcgen05.
void set_decode_kernel_choice(int choice);

// LSE combine of n partials per row.  in_log2: lses are base-2 (else base e).
// out_lse_mul: multiplier applied to the base-2 merged LSE before it is stored
// (1 for base 2, ln 2 for base e).  partial_row_stride: elements between rows of one
// shard (512 for dense), shard_stride: elements between shards.
cudaError_t launch_lse_combine(const void* partials, bool partials_fp32, const float* lses,
                               int n, long long rows, long long shard_stride_rows,
                               bool in_log2, float out_lse_mul, uint16_t* out,
                               float* out_lse, cudaStream_t stream);

cudaError_t launch_cp_local_slot(const int64_t* positions, const int32_t* block_table,
                                 int64_t bt_stride, int max_blocks, int B, int N,
                                 int block_size, int cp_size, int cp_rank, int interleave,
                                 int64_t* slots, unsigned int* status, cudaStream_t stream);

}  // namespace mla
