// Kernel choice for mla_decode: the tcgen05 kernel wherever the KV layout allows its TMA
// tiles.  The warp-level kernel runs only when a test selects it (a second, independent
// GPU implementation to cross-check the first); other layouts are refused by the caller.
#include <atomic>

#include "internal.h"

namespace mla {
namespace {
std::atomic<int> g_choice{0};
}

void set_decode_kernel_choice(int choice) { g_choice.store(choice); }

size_t decode_workspace_size(int B, int H, int q_len, int num_sms) {
  const size_t a = tc_workspace_size(B, H, q_len, num_sms);
  const size_t b = mma_workspace_size(B, H, q_len, num_sms);
  return a > b ? a : b;
}

size_t decode_workspace_for(int B, int H, int q_len, int num_sms, int block_size) {
  if (g_choice != 1 && tc_block_size_ok(block_size)) return tc_workspace_size(B, H, q_len, num_sms);
  return mma_workspace_size(B, H, q_len, num_sms);
}

DecodeKernel choose_decode_kernel(const DecodeArgs& a) {
  if (g_choice == 1) return kDecodeMma;
  return tc_supported(a) ? kDecodeTc : kDecodeNone;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.B == 0 || a.H * a.q_len == 0) return cudaSuccess;
  const DecodeKernel k = choose_decode_kernel(a);
  if (k == kDecodeTc) return launch_decode_tc(a, stream);
  if (k != kDecodeMma) return cudaErrorNotSupported;
  if (a.shard_B == a.B) return launch_decode_mma(a, stream);
  // several shards in one call: the warp-level kernel takes them one launch each
  const long long rows = (long long)a.shard_B * a.q_len * a.H;
  for (int r = 0; r * a.shard_B < a.B; ++r) {
    DecodeArgs s = a;
    s.B = a.shard_B;
    s.cp_rank = a.cp_rank + r;
    s.block_table = a.block_table + (long long)r * a.shard_B * a.bt_stride;
    s.seq_lens = a.seq_lens + (long long)r * a.shard_B;
    s.out = a.out + rows * r * 512;
    s.lse = a.lse ? a.lse + rows * r : nullptr;
    const cudaError_t e = launch_decode_mma(s, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace mla
