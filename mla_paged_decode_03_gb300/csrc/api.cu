// C ABI of libmla_decode.so (declared in include/mla_decode.h): host-side argument
// validation, error reporting and kernel launches.  Nothing here allocates memory.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <functional>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "sm100.cuh"
#include "../../include/mla_decode.h"

namespace {

// One status word per device; kernels OR MLA_STATUS_* bits into it.
__device__ unsigned int g_mla_status = 0;

thread_local char t_err[512] = {0};

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  t_err[0] = 0;
  return MLA_OK;
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  const char* what = "";
  int num_sms = 0;
  unsigned int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

void device_setup(DeviceInfo& d, int dev) {
  int sms = 0;
  d.err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (d.err != cudaSuccess) {
    d.what = "cudaDeviceGetAttribute";
    return;
  }
  void* p = nullptr;
  d.err = cudaGetSymbolAddress(&p, g_mla_status);
  if (d.err != cudaSuccess) {
    d.what = "cudaGetSymbolAddress(status)";
    return;
  }
  d.num_sms = sms;
  d.status = static_cast<unsigned int*>(p);
}

// Resolves the current device's SM count and status-word address (once per device, also
// when several host threads make their first call at the same time).
int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MLA_ERR_UNSUPPORTED, "device index %d", dev);
  DeviceInfo& d = g_dev[dev];
  std::call_once(d.once, device_setup, std::ref(d), dev);
  if (d.err != cudaSuccess) return fail(MLA_ERR_CUDA, "%s: %s", d.what, cudaGetErrorString(d.err));
  *out = &d;
  return MLA_OK;
}

// Process-wide settings of the diagnostic entry points.
std::atomic<unsigned long long> g_wait_ns{0};   // 0: the default limit
std::atomic<int> g_stall_test{0};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace mla {
int api_fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return code;
}
}  // namespace mla

extern "C" {

int mla_abi_version(void) { return (2 << 16) | 0; }

int mla_set_decode_kernel(int choice) {
  static std::atomic<int> current{0};
  if (choice < 0 || choice > 2)
    return fail(MLA_ERR_INVALID_ARGUMENT, "mla_set_decode_kernel: choice %d not in 0..2", choice);
  mla::set_decode_kernel_choice(choice);
  return current.exchange(choice);
}

int mla_set_rescale_budget(int choice) {
  static std::atomic<int> current{0};
  if (choice < 0 || choice > 2)
    return fail(MLA_ERR_INVALID_ARGUMENT, "mla_set_rescale_budget: choice %d not in 0..2", choice);
  mla::set_rescale_budget_choice(choice);
  return current.exchange(choice);
}

int mla_set_test_stall(int on) {
  if (on != 0 && on != 1)
    return fail(MLA_ERR_INVALID_ARGUMENT, "mla_set_test_stall: %d is neither 0 nor 1", on);
  return g_stall_test.exchange(on);
}

int64_t mla_set_wait_limit_ns(int64_t ns) {
  if (ns < 0) return fail(MLA_ERR_INVALID_ARGUMENT, "mla_set_wait_limit_ns: ns=%lld < 0",
                          (long long)ns);
  return (int64_t)g_wait_ns.exchange((unsigned long long)ns);
}

const char* mla_last_error(void) { return t_err; }

size_t mla_decode_workspace_size(int B, int H, int q_len, int num_sms) {
  if (B <= 0 || H <= 0 || q_len <= 0 || num_sms <= 0) return 0;
  return mla::decode_workspace_size(B, H, q_len, num_sms);
}

}  // extern "C"

namespace mla {

// Shared by mla_decode (n_shards == 1, the given rank), mla_decode_shards (ranks
// 0 .. n_shards-1 of cp_world == n_shards, shard-major tables and outputs) and
// mla_decode_noalloc (require_full_split: the workspace must hold the scratch of the full
// split-KV schedule, else the call is refused after every other check).
int decode_entry(const char* fn, const void* q, const void* kv_cache, const int32_t* block_table,
                 int64_t bt_stride, const int32_t* seq_lens, const int32_t* causal_seqlens_global,
                 int B, int H, int q_len, int causal, int block_size, int num_blocks,
                 int max_blocks, int cp_world, int cp_rank, int interleave, int n_shards,
                 float scale, void* out, float* lse, int lse_base_e, void* workspace,
                 size_t workspace_bytes, bool require_full_split, mla_stream_t stream) {
  if (B < 0) return fail(MLA_ERR_INVALID_ARGUMENT, "%s: B=%d < 0", fn, B);
  if (H < 1) return fail(MLA_ERR_INVALID_ARGUMENT, "%s: H=%d < 1", fn, H);
  if (q_len < 1 || q_len > MLA_MAX_Q_LEN)
    return fail(q_len < 1 ? MLA_ERR_INVALID_ARGUMENT : MLA_ERR_UNSUPPORTED,
                "%s: q_len=%d outside [1, %d]", fn, q_len, MLA_MAX_Q_LEN);
  if (block_size < 1) return fail(MLA_ERR_INVALID_ARGUMENT, "%s: block_size < 1", fn);
  if (num_blocks < 1) return fail(MLA_ERR_INVALID_ARGUMENT, "%s: num_blocks < 1", fn);
  if (max_blocks < 1 || bt_stride < max_blocks)
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: need 1 <= max_blocks (%d) <= bt_stride (%lld)",
                fn, max_blocks, (long long)bt_stride);
  if ((long long)max_blocks * block_size > (1LL << 31) - 1)
    return fail(MLA_ERR_UNSUPPORTED, "%s: max_blocks*block_size exceeds 2^31-1", fn);
  if ((long long)num_blocks * block_size > (1LL << 40))
    return fail(MLA_ERR_UNSUPPORTED, "%s: cache too large", fn);
  if (cp_world < 1 || cp_rank < 0 || cp_rank >= cp_world)
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: need 0 <= cp_rank (%d) < cp_world (%d)", fn,
                cp_rank, cp_world);
  if (interleave < 1 || block_size % interleave != 0)
    return fail(MLA_ERR_INVALID_ARGUMENT,
                "%s: interleave (%d) must be >= 1 and divide block_size (%d)", fn, interleave,
                block_size);
  if ((long long)cp_world * interleave > (1LL << 31) - 1)
    return fail(MLA_ERR_UNSUPPORTED, "%s: cp_world*interleave exceeds 2^31-1", fn);
  if (!isfinite(scale) || !(scale > 0.f))
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: scale must be finite and > 0", fn);
  if (B == 0) return ok();
  if (!q || !kv_cache || !block_table || !seq_lens || !out)
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: null q/kv_cache/block_table/seq_lens/out", fn);
  if (causal_seqlens_global == nullptr && cp_world != 1 && causal)
    return fail(MLA_ERR_INVALID_ARGUMENT,
                "%s: causal_seqlens_global is required when cp_world > 1", fn);
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16))
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: q, kv_cache and out must be 16-byte aligned", fn);
  if (!aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      (causal_seqlens_global && !aligned(causal_seqlens_global, 4)) || (lse && !aligned(lse, 4)))
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: misaligned int32/float argument", fn);
  if (workspace && !aligned(workspace, 256))
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: workspace must be 256-byte aligned", fn);
  if ((long long)n_shards * B * q_len * H > (1LL << 31) - 1)
    return fail(MLA_ERR_UNSUPPORTED, "%s: too many query rows", fn);

  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != MLA_OK) return rc;

  mla::DecodeArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.kv = static_cast<const uint16_t*>(kv_cache);
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.gseq = causal_seqlens_global ? causal_seqlens_global : seq_lens;
  a.B = n_shards * B;
  a.shard_B = B;
  a.H = H;
  a.q_len = q_len;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks;
  a.cp_world = cp_world;
  a.cp_rank = cp_rank;
  a.causal = causal ? 1 : 0;
  a.interleave = interleave;
  const unsigned long long wait_ns = g_wait_ns.load();
  a.wait_ns = wait_ns ? wait_ns : mla::sm100::kDefaultWaitNs;
  a.stall_test = g_stall_test.load();
  a.scale = scale;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.lse_base_e = lse_base_e ? 1 : 0;
  a.workspace = workspace;
  a.workspace_bytes = workspace ? workspace_bytes : 0;
  a.num_sms = dev->num_sms;
  a.status = dev->status;
  const mla::DecodeKernel k = mla::choose_decode_kernel(a);
  if (k == mla::kDecodeNone)
    return fail(MLA_ERR_UNSUPPORTED,
                "%s: no decode kernel for this layout (block_size %d: the tcgen05 kernel takes "
                "16, 32 or a multiple of 64; q_len*H = %d rows need at most %d row tiles of 128)",
                fn, block_size, q_len * H, dev->num_sms / 2);
  if (require_full_split) {
    const size_t need = mla::decode_workspace_for(n_shards * B, H, q_len, dev->num_sms, block_size);
    if (need > workspace_bytes)
      return fail(MLA_ERR_UNSUPPORTED,
                  "%s: B=%d H=%d q_len=%d needs %zu bytes of split-KV scratch, more than the "
                  "library's fixed %zu; use mla_decode with a caller workspace",
                  fn, B, H, q_len, need, workspace_bytes);
  }
  cudaError_t e = mla::launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "%s launch: %s", fn, cudaGetErrorString(e));
  return ok();
}

}  // namespace mla

extern "C" {

int mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
               int64_t bt_stride, const int32_t* seq_lens,
               const int32_t* causal_seqlens_global, int B, int H, int q_len, int causal,
               int block_size, int num_blocks, int max_blocks, int cp_world, int cp_rank,
               int interleave, float scale, void* out, float* lse, int lse_base_e,
               void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  return mla::decode_entry("mla_decode", q, kv_cache, block_table, bt_stride, seq_lens,
                           causal_seqlens_global, B, H, q_len, causal, block_size, num_blocks,
                           max_blocks, cp_world, cp_rank, interleave, 1, scale, out, lse,
                           lse_base_e, workspace, workspace_bytes, false, stream);
}

int mla_decode_shards(const void* q, const void* kv_cache, const int32_t* block_table,
                      int64_t bt_stride, const int32_t* seq_lens,
                      const int32_t* causal_seqlens_global, int B, int H, int q_len,
                      int causal, int block_size, int num_blocks, int max_blocks, int n_shards,
                      int interleave, float scale, void* out, float* lse, int lse_base_e,
                      void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  if (n_shards < 1)
    return fail(MLA_ERR_INVALID_ARGUMENT, "mla_decode_shards: n_shards=%d < 1", n_shards);
  if (n_shards > 1 && B > 0 && (unsigned long long)n_shards * B * B >= (1ull << 32))
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode_shards: n_shards * B^2 must stay below 2^32");
  return mla::decode_entry("mla_decode_shards", q, kv_cache, block_table, bt_stride, seq_lens,
                           causal_seqlens_global, B, H, q_len, causal, block_size, num_blocks,
                           max_blocks, n_shards, 0, interleave, n_shards, scale, out, lse,
                           lse_base_e, workspace, workspace_bytes, false, stream);
}

int lse_merge(const void* partials, int partials_fp32, const float* lses, int n_shards,
              int T, int H, void* out, float* out_lse, int lse_base_e, mla_stream_t stream) {
  if (n_shards < 1) return fail(MLA_ERR_INVALID_ARGUMENT, "lse_merge: n_shards=%d < 1", n_shards);
  if (T < 0 || H < 1) return fail(MLA_ERR_INVALID_ARGUMENT, "lse_merge: need T >= 0, H >= 1");
  if (T == 0) return ok();
  if (!partials || !lses || !out)
    return fail(MLA_ERR_INVALID_ARGUMENT, "lse_merge: null partials/lses/out");
  if (!aligned(partials, 16) || !aligned(out, 16) || !aligned(lses, 4) ||
      (out_lse && !aligned(out_lse, 4)))
    return fail(MLA_ERR_INVALID_ARGUMENT, "lse_merge: partials/out need 16-byte alignment");
  const long long rows = (long long)T * H;
  cudaError_t e = mla::launch_lse_combine(partials, partials_fp32 != 0, lses, n_shards, rows,
                                          rows, !lse_base_e, lse_base_e ? 0.6931471805599453f : 1.f,
                                          static_cast<uint16_t*>(out), out_lse,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "lse_merge launch: %s", cudaGetErrorString(e));
  return ok();
}

static int slot_args_check(const char* fn, int B, int N, int block_size, int cp_size,
                           int cp_rank, int interleave, int max_blocks, int64_t bt_stride) {
  if (B < 0 || N < 0) return fail(MLA_ERR_INVALID_ARGUMENT, "%s: B, N must be >= 0", fn);
  if (block_size < 1 || cp_size < 1 || interleave < 1)
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: block_size, cp_size, interleave >= 1", fn);
  if (cp_rank < 0 || cp_rank >= cp_size)
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: need 0 <= cp_rank < cp_size", fn);
  if (block_size % interleave != 0)
    return fail(MLA_ERR_INVALID_ARGUMENT,
                "%s: block_size (%d) must be a multiple of interleave (%d)", fn, block_size,
                interleave);
  if (max_blocks < 1 || bt_stride < max_blocks)
    return fail(MLA_ERR_INVALID_ARGUMENT, "%s: need 1 <= max_blocks <= bt_stride", fn);
  if ((long long)block_size * cp_size > (1LL << 31) - 1)
    return fail(MLA_ERR_UNSUPPORTED, "%s: block_size*cp_size exceeds 2^31-1", fn);
  if ((long long)B * N > (1LL << 31) - 1)
    return fail(MLA_ERR_UNSUPPORTED, "%s: B*N exceeds 2^31-1 positions", fn);
  return MLA_OK;
}

int cp_local_slot(const int64_t* positions, const int32_t* block_table, int64_t bt_stride,
                  int max_blocks, int B, int N, int block_size, int cp_size, int cp_rank,
                  int interleave, int64_t* slots, mla_stream_t stream) {
  int rc = slot_args_check("cp_local_slot", B, N, block_size, cp_size, cp_rank, interleave,
                           max_blocks, bt_stride);
  if (rc != MLA_OK) return rc;
  if ((long long)B * N == 0) return ok();
  if (!positions || !block_table || !slots)
    return fail(MLA_ERR_INVALID_ARGUMENT, "cp_local_slot: null positions/block_table/slots");
  if (!aligned(positions, 8) || !aligned(slots, 8) || !aligned(block_table, 4))
    return fail(MLA_ERR_INVALID_ARGUMENT, "cp_local_slot: misaligned pointer");
  DeviceInfo* dev = nullptr;
  rc = device_info(&dev);
  if (rc != MLA_OK) return rc;
  cudaError_t e = mla::launch_cp_local_slot(positions, block_table, bt_stride, max_blocks, B, N,
                                            block_size, cp_size, cp_rank, interleave, slots,
                                            dev->status, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(MLA_ERR_CUDA, "cp_local_slot launch: %s", cudaGetErrorString(e));
  return ok();
}

int cp_local_slot_scatter(const int64_t* positions, const void* kv_new,
                          const int32_t* block_table, int64_t bt_stride, int max_blocks, int B,
                          int N, int block_size, int cp_size, int cp_rank, int interleave,
                          void* kv_cache, int num_blocks, int64_t* slots, mla_stream_t stream) {
  int rc = slot_args_check("cp_local_slot_scatter", B, N, block_size, cp_size, cp_rank,
                           interleave, max_blocks, bt_stride);
  if (rc != MLA_OK) return rc;
  if (num_blocks < 1)
    return fail(MLA_ERR_INVALID_ARGUMENT, "cp_local_slot_scatter: num_blocks < 1");
  if ((long long)B * N == 0) return ok();
  if (!positions || !kv_new || !block_table || !kv_cache)
    return fail(MLA_ERR_INVALID_ARGUMENT,
                "cp_local_slot_scatter: null positions/kv_new/block_table/kv_cache");
  if (!aligned(positions, 8) || (slots && !aligned(slots, 8)) || !aligned(block_table, 4) ||
      !aligned(kv_new, 16) || !aligned(kv_cache, 16))
    return fail(MLA_ERR_INVALID_ARGUMENT,
                "cp_local_slot_scatter: misaligned pointer (kv_new and kv_cache need 16 bytes)");
  DeviceInfo* dev = nullptr;
  rc = device_info(&dev);
  if (rc != MLA_OK) return rc;
  cudaError_t e = mla::launch_cp_local_slot_scatter(
      positions, static_cast<const uint16_t*>(kv_new), block_table, bt_stride, max_blocks, B, N,
      block_size, cp_size, cp_rank, interleave, static_cast<uint16_t*>(kv_cache), num_blocks,
      slots, dev->status, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(MLA_ERR_CUDA, "cp_local_slot_scatter launch: %s", cudaGetErrorString(e));
  return ok();
}

int mla_get_device_status(mla_stream_t stream, uint32_t* bits_out) {
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != MLA_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess)
    return fail(MLA_ERR_CUDA, "mla_get_device_status: %s", cudaGetErrorString(e));
  unsigned int bits = 0;
  e = cudaMemcpyFromSymbol(&bits, g_mla_status, sizeof(bits));
  if (e == cudaSuccess) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_mla_status, &zero, sizeof(zero));
  }
  if (e != cudaSuccess)
    return fail(MLA_ERR_CUDA, "mla_get_device_status: %s", cudaGetErrorString(e));
  if (bits_out) *bits_out = bits;
  if (bits == 0) return ok();
  return fail(MLA_ERR_DEVICE, "device status 0x%x:%s%s%s%s", bits,
              (bits & MLA_STATUS_BAD_PAGE) ? " bad block_table entry;" : "",
              (bits & MLA_STATUS_SEQ_TOO_LONG) ? " seq_len beyond max_blocks*block_size;" : "",
              (bits & MLA_STATUS_BAD_VBLOCK) ? " virtual block beyond max_blocks;" : "",
              (bits & MLA_STATUS_WAIT_TIMEOUT) ? " on-chip wait timed out;" : "");
}

}  // extern "C"
