// Kernel choice for mla_decode: the tcgen05 kernel wherever the KV layout allows TMA
// tiles, the warp-level kernel otherwise.
#include "internal.h"

namespace mla {
namespace {
int g_choice = 0;
}

void set_decode_kernel_choice(int choice) { g_choice = choice; }

size_t decode_workspace_size(int B, int H, int q_len, int num_sms) {
  const size_t a = tc_workspace_size(B, H, q_len, num_sms);
  const size_t b = mma_workspace_size(B, H, q_len, num_sms);
  return a > b ? a : b;
}

size_t decode_workspace_for(int B, int H, int q_len, int num_sms, int block_size) {
  const bool tc_bs = block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128;
  if (g_choice != 1 && tc_bs) return tc_workspace_size(B, H, q_len, num_sms);
  return mma_workspace_size(B, H, q_len, num_sms);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.B == 0 || a.H * a.q_len == 0) return cudaSuccess;
  const bool tc = g_choice == 2 || (g_choice == 0 && tc_supported(a));
  if (tc && tc_supported(a)) return launch_decode_tc(a, stream);
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
