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
  int causal;                    // 0: every row reads the shard's whole local sequence
  int interleave;                // round-robin segment length of the KV sharding
  unsigned long long wait_ns;    // limit of every bounded on-chip wait
  int stall_test;                // tests only: one wait of each pair is never satisfied
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

// Which decode kernel a call runs: the tensor-core (tcgen05) kernel whenever the cache
// layout allows its TMA tiles; the warp-level MMA kernel only when a test selected it.
enum DecodeKernel { kDecodeTc, kDecodeMma, kDecodeNone };
DecodeKernel choose_decode_kernel(const DecodeArgs& a);

// Split-KV decode with the kernel choose_decode_kernel picks (not kDecodeNone).
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
size_t decode_workspace_size(int B, int H, int q_len, int num_sms);

// tcgen05 / TMEM / TMA kernel (mla_decode_tc.cu)
bool tc_block_size_ok(int block_size);
bool tc_supported(const DecodeArgs& a);
size_t tc_workspace_size(int B, int H, int q_len, int num_sms);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream);
// Rescale budget of the tcgen05 kernel: 0 = chosen per call, 1 = narrow, 2 = wide.
void set_rescale_budget_choice(int choice);

// warp-level mma.sync kernel (mla_decode_mma.cu)
size_t mma_workspace_size(int B, int H, int q_len, int num_sms);
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t stream);

// Split-KV scratch the kernel chosen for this block size uses at its preferred split.
size_t decode_workspace_for(int B, int H, int q_len, int num_sms, int block_size);

// Records a message for mla_last_error() and returns `code` (api.cu).
int api_fail(int code, const char* fmt, ...);

// Validation and launch behind mla_decode, mla_decode_shards and mla_decode_noalloc
// (api.cu); `stream` is a cudaStream_t.  With require_full_split the workspace must hold
// the scratch of the full split-KV schedule, else MLA_ERR_UNSUPPORTED (after every other
// check).
int decode_entry(const char* fn, const void* q, const void* kv_cache, const int32_t* block_table,
                 int64_t bt_stride, const int32_t* seq_lens, const int32_t* causal_seqlens_global,
                 int B, int H, int q_len, int causal, int block_size, int num_blocks,
                 int max_blocks, int cp_world, int cp_rank, int interleave, int n_shards,
                 float scale, void* out, float* lse, int lse_base_e, void* workspace,
                 size_t workspace_bytes, bool require_full_split, struct CUstream_st* stream);

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

// Fast division of 32-bit numerators by a fixed divisor d >= 1: q = mulhi64(m, n) with
// m = floor((2^64 - 1) / d) + 1 is exact for every n < 2^32 (Lemire, Kaser and Kurz,
// "Faster remainder by direct computation", 2019); d = 1 is kept apart (m would be 2^64).
// Launch configuration of a kernel that consumes the previous kernel's results in the same
// stream (programmatic dependent launch): the kernel may be scheduled while that kernel
// drains, and waits for its completion and memory with griddepcontrol.wait before it reads
// or writes global memory.  Without the attribute (or after a non-kernel operation) the
// wait returns at once.
struct DependentLaunch {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  DependentLaunch(dim3 grid, dim3 block, cudaStream_t stream) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};

struct FastDiv {
  unsigned long long m;
  unsigned int d;
};
inline FastDiv make_fastdiv(unsigned int d) {
  FastDiv f;
  f.d = d;
  f.m = d > 1 ? ~0ull / d + 1 : 0ull;
  return f;
}

cudaError_t launch_cp_local_slot(const int64_t* positions, const int32_t* block_table,
                                 int64_t bt_stride, int max_blocks, int B, int N,
                                 int block_size, int cp_size, int cp_rank, int interleave,
                                 int64_t* slots, unsigned int* status, cudaStream_t stream);

// Writes the KV rows of positions this rank owns into its pool (cp_local_slot.cu).
cudaError_t launch_cp_local_slot_scatter(const int64_t* positions, const uint16_t* kv_new,
                                         const int32_t* block_table, int64_t bt_stride,
                                         int max_blocks, int B, int N, int block_size,
                                         int cp_size, int cp_rank, int interleave,
                                         uint16_t* kv_cache, long long num_blocks,
                                         int64_t* slots, unsigned int* status,
                                         cudaStream_t stream);

}  // namespace mla
