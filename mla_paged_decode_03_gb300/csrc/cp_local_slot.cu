// cp_local_slot: DCP slot mapping (positions -> this rank's KV slot or PAD).
//
// Definition: "vLLM PR #52188 (DSpark + DCP)" page, section "关键源码片段"
// (cp_utils.py cp_local_slot) and section "实现拆解" step 4 (the page of a position is
// block_table[pos // (block_size * CP_SIZE)]).  Pure integer work, bit-exact.
//
// HBM-bound: 8 B of position in, 8 B of slot out per position, plus one 4-byte table
// entry per position (mostly L2 hits: consecutive positions share a virtual block).
// Each thread maps two consecutive positions with one 16-byte load and one 16-byte
// store when the row length and pointers allow it.
#include "internal.h"
#include "../../include/mla_decode.h"

namespace mla {
namespace {

struct SlotParams {
  const int32_t* block_table;
  int64_t bt_stride;
  int max_blocks, block_size, cp_size, cp_rank, interleave;
  unsigned int* status;
};

__device__ __forceinline__ long long map_one(long long pos, int b, const SlotParams& p,
                                             bool& bad) {
  if (pos < 0) return MLA_PAD_SLOT_ID;
  const long long vbs = (long long)p.block_size * p.cp_size;
  const long long vb = pos / vbs;
  if (vb >= p.max_blocks) {
    bad = true;
    return MLA_PAD_SLOT_ID;
  }
  const long long off = pos - vb * vbs;
  long long local;
  if (p.cp_size == 1) {
    local = off;
  } else {
    const long long seg = off / p.interleave;
    if ((int)(seg % p.cp_size) != p.cp_rank) return MLA_PAD_SLOT_ID;
    local = (off / ((long long)p.interleave * p.cp_size)) * p.interleave + off % p.interleave;
  }
  const long long page = __ldg(p.block_table + (long long)b * p.bt_stride + vb);
  return page * p.block_size + local;
}

// One thread per pair of positions; rows of even length and 16-byte aligned pointers.
__global__ void __launch_bounds__(256) cp_local_slot_vec2(const longlong2* __restrict__ pos,
                                                          longlong2* __restrict__ slots,
                                                          long long pairs, int pairs_per_row,
                                                          SlotParams p) {
  bool bad = false;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < pairs;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / pairs_per_row);
    const longlong2 v = __ldcs(pos + i);
    longlong2 r;
    r.x = map_one(v.x, b, p, bad);
    r.y = map_one(v.y, b, p, bad);
    __stcs(slots + i, r);
  }
  if (bad) atomicOr(p.status, MLA_STATUS_BAD_VBLOCK);
}

__global__ void __launch_bounds__(256) cp_local_slot_scalar(const long long* __restrict__ pos,
                                                            long long* __restrict__ slots,
                                                            long long total, int N,
                                                            SlotParams p) {
  bool bad = false;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / N);
    slots[i] = map_one(__ldcs(pos + i), b, p, bad);
  }
  if (bad) atomicOr(p.status, MLA_STATUS_BAD_VBLOCK);
}

}  // namespace

cudaError_t launch_cp_local_slot(const int64_t* positions, const int32_t* block_table,
                                 int64_t bt_stride, int max_blocks, int B, int N,
                                 int block_size, int cp_size, int cp_rank, int interleave,
                                 int64_t* slots, unsigned int* status, cudaStream_t stream) {
  const long long total = (long long)B * N;
  if (total == 0) return cudaSuccess;
  SlotParams p{block_table, bt_stride, max_blocks, block_size, cp_size, cp_rank, interleave,
               status};
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool vec = (N % 2 == 0) && ((uintptr_t)positions % 16 == 0) &&
                   ((uintptr_t)slots % 16 == 0);
  const long long work = vec ? total / 2 : total;
  long long blocks = (work + 255) / 256;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  if (vec) {
    cp_local_slot_vec2<<<(unsigned)blocks, 256, 0, stream>>>(
        reinterpret_cast<const longlong2*>(positions), reinterpret_cast<longlong2*>(slots),
        work, N / 2, p);
  } else {
    cp_local_slot_scalar<<<(unsigned)blocks, 256, 0, stream>>>(
        reinterpret_cast<const long long*>(positions), reinterpret_cast<long long*>(slots),
        total, N, p);
  }
  return cudaGetLastError();
}

}  // namespace mla
