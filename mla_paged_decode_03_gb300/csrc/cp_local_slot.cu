// cp_local_slot: DCP slot mapping (positions -> this rank's KV slot or PAD), and the scatter
// of new KV rows into the slots it gives.
//
// Definition: "vLLM PR #52188 (DSpark + DCP)" page, section "关键源码片段"
// (cp_utils.py cp_local_slot) and section "实现拆解" step 4 (the page of a position is
// block_table[pos // (block_size * CP_SIZE)]; the draft inputs apply cp_local_slot to
// the slots they write, so that a rank never writes a slot another rank owns).  Pure
// integer work, bit-exact.
//
// HBM-bound: 8 B of position in, 8 B of slot out per position, plus one 4-byte table
// entry per position (mostly L2 hits: consecutive positions share a virtual block).
// Each thread maps two consecutive positions with one 16-byte load and one 16-byte
// store when the row length and pointers allow it.  Divisions by the run's constants
// (block_size * cp_size, interleave, cp_size, positions per row) are multiply-high
// operations with host-computed multipliers: 64-bit integer division would make the
// kernel issue-bound (about 170 instructions per position).
//
// The scatter additionally copies each owned position's 1152-byte row (576 bf16) from
// the new rows to its slot (512 contiguous bytes per warp instruction); positions this rank
// does not own are neither read nor written.
#include "internal.h"
#include "../../include/mla_decode.h"

namespace mla {
namespace {

constexpr int kRowBytes = 576 * 2;
constexpr int kRowChunks = kRowBytes / 16;     // 72 16-byte pieces per KV row

struct SlotParams {
  const int32_t* block_table;
  int64_t bt_stride;
  int max_blocks, block_size, cp_size, cp_rank, interleave;
  unsigned int vbs;          // block_size * cp_size (checked < 2^31 on the host)
  FastDiv div_vbs, div_il, div_cp;
  unsigned int* status;
};

__device__ __forceinline__ unsigned int fdiv(unsigned int n, const FastDiv& f) {
  return f.d == 1u ? n : (unsigned int)__umul64hi(f.m, (unsigned long long)n);
}

// Slot of `pos` on this rank (>= 0), or MLA_PAD_SLOT_ID if the rank does not own it, the
// position is negative, or its virtual block lies past the table (then `bad` is set and
// the table is not read).
__device__ __forceinline__ long long map_one(long long pos, int b, const SlotParams& p,
                                             bool& bad) {
  if (pos < 0) return MLA_PAD_SLOT_ID;
  long long vb;
  unsigned int off;
  if (pos <= 0xffffffffLL) {
    const unsigned int q = fdiv((unsigned int)pos, p.div_vbs);
    vb = q;
    off = (unsigned int)pos - q * p.vbs;
  } else {
    vb = pos / p.vbs;
    off = (unsigned int)(pos - vb * p.vbs);
  }
  if (vb >= p.max_blocks) {
    bad = true;
    return MLA_PAD_SLOT_ID;
  }
  unsigned int local;
  if (p.cp_size == 1) {
    local = off;
  } else {
    // segment of `interleave` positions, its owner (segment mod cp) and its round
    const unsigned int seg = fdiv(off, p.div_il);
    const unsigned int rin = off - seg * (unsigned int)p.interleave;
    const unsigned int rnd = fdiv(seg, p.div_cp);
    if ((int)(seg - rnd * (unsigned int)p.cp_size) != p.cp_rank) return MLA_PAD_SLOT_ID;
    local = rnd * (unsigned int)p.interleave + rin;
  }
  const long long page = __ldg(p.block_table + (long long)b * p.bt_stride + vb);
  return page * p.block_size + local;
}

// One thread per pair of positions; rows of even length and 16-byte aligned pointers.
__global__ void __launch_bounds__(256) cp_local_slot_vec2(const longlong2* __restrict__ pos,
                                                          longlong2* __restrict__ slots,
                                                          long long pairs, FastDiv div_row,
                                                          SlotParams p) {
  bool bad = false;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < pairs;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)fdiv((unsigned int)i, div_row);
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
                                                            long long total, FastDiv div_row,
                                                            SlotParams p) {
  bool bad = false;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)fdiv((unsigned int)i, div_row);
    slots[i] = map_one(__ldcs(pos + i), b, p, bad);
  }
  if (bad) atomicOr(p.status, MLA_STATUS_BAD_VBLOCK);
}

// A warp takes 32 consecutive positions: each lane maps one (coalesced position loads and
// slot stores), then the warp copies the rows of the owned ones, four rows per round so that
// every lane has several 16-byte loads in flight before it stores.  `slots` (may be null)
// receives the mapping, as cp_local_slot gives it.
__global__ void __launch_bounds__(256) cp_local_slot_scatter_kernel(
    const long long* __restrict__ pos, const uint4* __restrict__ kv_new,
    uint4* __restrict__ kv_cache, long long* __restrict__ slots, long long total,
    long long cache_rows, FastDiv div_row, SlotParams p) {
  const int lane = threadIdx.x & 31;
  bool bad_vb = false, bad_page = false;
  const long long warps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long g = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; g * 32 < total;
       g += warps) {
    const long long i = g * 32 + lane;
    long long slot = MLA_PAD_SLOT_ID;
    if (i < total) {
      slot = map_one(__ldg(pos + i), (int)fdiv((unsigned int)i, div_row), p, bad_vb);
      if (slots != nullptr) slots[i] = slot;
      if (slot >= cache_rows) {
        bad_page = true;
        slot = MLA_PAD_SLOT_ID;
      }
    }
    unsigned int own = __ballot_sync(0xffffffffu, slot >= 0);
    while (own != 0u) {
      int src[4];
      long long dst[4];
      int nr = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        src[u] = 0;
        dst[u] = -1;
        if (own != 0u) {
          const int l = __ffs(own) - 1;
          own &= own - 1u;
          src[u] = l;
          dst[u] = __shfl_sync(0xffffffffu, slot, l);
          nr = u + 1;
        }
      }
      uint4 v[4][3];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const int ch = lane + 32 * c;
          if (u < nr && ch < kRowChunks) v[u][c] = __ldcs(kv_new + (g * 32 + src[u]) * kRowChunks + ch);
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const int ch = lane + 32 * c;
          if (u < nr && ch < kRowChunks) __stcs(kv_cache + dst[u] * kRowChunks + ch, v[u][c]);
        }
    }
  }
  if (__any_sync(0xffffffffu, bad_vb) && lane == 0) atomicOr(p.status, MLA_STATUS_BAD_VBLOCK);
  if (__any_sync(0xffffffffu, bad_page) && lane == 0) atomicOr(p.status, MLA_STATUS_BAD_PAGE);
}

SlotParams make_params(const int32_t* block_table, int64_t bt_stride, int max_blocks,
                       int block_size, int cp_size, int cp_rank, int interleave,
                       unsigned int* status) {
  SlotParams p;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.max_blocks = max_blocks;
  p.block_size = block_size;
  p.cp_size = cp_size;
  p.cp_rank = cp_rank;
  p.interleave = interleave;
  p.vbs = (unsigned int)block_size * (unsigned int)cp_size;
  p.div_vbs = make_fastdiv(p.vbs);
  p.div_il = make_fastdiv((unsigned int)interleave);
  p.div_cp = make_fastdiv((unsigned int)cp_size);
  p.status = status;
  return p;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0) {
    cudaGetLastError();
    return 148;
  }
  return sms;
}

}  // namespace

cudaError_t launch_cp_local_slot(const int64_t* positions, const int32_t* block_table,
                                 int64_t bt_stride, int max_blocks, int B, int N,
                                 int block_size, int cp_size, int cp_rank, int interleave,
                                 int64_t* slots, unsigned int* status, cudaStream_t stream) {
  const long long total = (long long)B * N;
  if (total == 0) return cudaSuccess;
  const SlotParams p = make_params(block_table, bt_stride, max_blocks, block_size, cp_size,
                                   cp_rank, interleave, status);
  const int sms = sm_count();
  const bool vec = (N % 2 == 0) && ((uintptr_t)positions % 16 == 0) &&
                   ((uintptr_t)slots % 16 == 0);
  const long long work = vec ? total / 2 : total;
  long long blocks = (work + 255) / 256;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  if (vec) {
    cp_local_slot_vec2<<<(unsigned)blocks, 256, 0, stream>>>(
        reinterpret_cast<const longlong2*>(positions), reinterpret_cast<longlong2*>(slots),
        work, make_fastdiv((unsigned int)(N / 2)), p);
  } else {
    cp_local_slot_scalar<<<(unsigned)blocks, 256, 0, stream>>>(
        reinterpret_cast<const long long*>(positions), reinterpret_cast<long long*>(slots),
        total, make_fastdiv((unsigned int)N), p);
  }
  return cudaGetLastError();
}

cudaError_t launch_cp_local_slot_scatter(const int64_t* positions, const uint16_t* kv_new,
                                         const int32_t* block_table, int64_t bt_stride,
                                         int max_blocks, int B, int N, int block_size,
                                         int cp_size, int cp_rank, int interleave,
                                         uint16_t* kv_cache, long long num_blocks,
                                         int64_t* slots, unsigned int* status,
                                         cudaStream_t stream) {
  const long long total = (long long)B * N;
  if (total == 0) return cudaSuccess;
  const SlotParams p = make_params(block_table, bt_stride, max_blocks, block_size, cp_size,
                                   cp_rank, interleave, status);
  const int sms = sm_count();
  long long blocks = (total + 255) / 256;        // 8 warps per block, 32 positions per warp
  const long long cap = (long long)sms * 16;
  if (blocks > cap) blocks = cap;
  cp_local_slot_scatter_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<const long long*>(positions), reinterpret_cast<const uint4*>(kv_new),
      reinterpret_cast<uint4*>(kv_cache), reinterpret_cast<long long*>(slots), total,
      num_blocks * block_size, make_fastdiv((unsigned int)N), p);
  return cudaGetLastError();
}

}  // namespace mla
