// LSE combine: merge n partial attention results of the same rows through their LSEs.
//
// Used for the public lse_merge (shard partials, "vLLM PR #54012 (FlashInfer native CP
// mask)" page, section "实现拆解" step 3: ranks are combined through LSEs in one common
// base) and for the split-KV reduction inside mla_decode (fp32 partials in workspace).
//
// One warp per (row, head): lane j owns dims [8j, 8j+8) and [256+8j, 256+8j+8) of the
// 512, so every load and store of a warp covers 512 contiguous bytes (bf16) or 1 KB
// (fp32).  The row max M of the n LSEs is reduced with warp shuffles; weights are
// 2^(lse*k - M*k) with k = 1 (base-2 LSEs) or log2(e) (natural LSEs).  HBM-bound:
// n * 1 KB (bf16) or n * 2 KB (fp32) read and 1 KB written per row.  Few rows of many
// bf16 shards take 2 or 4 warps per row instead (lse_combine_split_kernel), so that the
// n rounds of loads of a row are spread over more warps.
#include <math.h>

#include <cuda_bf16.h>

#include "internal.h"

namespace mla {
namespace {

constexpr int kDv = 512;
constexpr int kWarps = 8;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* v) {
  const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(h[k]);
    v[2 * k] = f.x;
    v[2 * k + 1] = f.y;
  }
}

__device__ __forceinline__ void load8(const float* p, float* v) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
lse_combine_kernel(const T* __restrict__ partials, const float* __restrict__ lses, int n,
                   long long rows, long long shard_stride_rows, float lse_to_log2,
                   float out_lse_mul, __nv_bfloat16* __restrict__ out,
                   float* __restrict__ out_lse) {
  // launched as a dependent of the kernel that wrote the partials
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;

  float m2 = -INFINITY;                       // max LSE, in log2 units
  for (int s = lane; s < n; s += 32)
    m2 = fmaxf(m2, __ldg(lses + s * shard_stride_rows + row) * lse_to_log2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));

  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float wsum = 0.f;
  if (m2 != -INFINITY) {
    for (int s = 0; s < n; ++s) {
      const float l2 = __ldg(lses + s * shard_stride_rows + row) * lse_to_log2;
      const float w = exp2f(l2 - m2);
      if (w == 0.f) continue;                 // empty shard: weight 0, partial unread
      wsum += w;
      const T* base = partials + (s * shard_stride_rows + row) * (long long)kDv;
      float v[8];
      load8(base + 8 * lane, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = fmaf(w, v[k], acc[k]);
      load8(base + 256 + 8 * lane, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[8 + k] = fmaf(w, v[k], acc[8 + k]);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* o = out + row * kDv;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint4 packed;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&packed);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      h[k] = __floats2bfloat162_rn(acc[8 * c + 2 * k] * inv, acc[8 * c + 2 * k + 1] * inv);
    *reinterpret_cast<uint4*>(o + 256 * c + 8 * lane) = packed;
  }
  if (out_lse != nullptr && lane == 0)
    out_lse[row] = wsum > 0.f ? (m2 + log2f(wsum)) * out_lse_mul : -INFINITY;
}

// The same merge for few rows of many shards: S warps per row, warp q of a row taking
// shards q, q + S, q + 2S, ...; the S weighted partial sums are added through shared
// memory by the row's first warp.  With one warp per row such a merge is latency-bound
// (n dependent rounds of loads per warp; 16 shards of 1,024 rows took 13.6 us for 8.4 MB).
template <typename T, int S>
__global__ void __launch_bounds__(kWarps * 32)
lse_combine_split_kernel(const T* __restrict__ partials, const float* __restrict__ lses, int n,
                         long long rows, long long shard_stride_rows, float lse_to_log2,
                         float out_lse_mul, __nv_bfloat16* __restrict__ out,
                         float* __restrict__ out_lse) {
  static_assert(kWarps % S == 0, "whole rows per block");
  __shared__ float s_acc[kWarps][kDv];
  __shared__ float s_w[kWarps];
  // launched as a dependent of the kernel that wrote the partials
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long row = (long long)blockIdx.x * (kWarps / S) + warp / S;
  const int part = warp % S;
  const bool valid = row < rows;

  float m2 = -INFINITY;                       // max LSE over all shards, in log2 units
  if (valid)
    for (int s = lane; s < n; s += 32)
      m2 = fmaxf(m2, __ldg(lses + s * shard_stride_rows + row) * lse_to_log2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));

  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float wsum = 0.f;
  if (valid && m2 != -INFINITY) {
    for (int s = part; s < n; s += S) {
      const float w = exp2f(__ldg(lses + s * shard_stride_rows + row) * lse_to_log2 - m2);
      if (w == 0.f) continue;                 // empty shard: weight 0, partial unread
      wsum += w;
      const T* base = partials + (s * shard_stride_rows + row) * (long long)kDv;
      float v[8];
      load8(base + 8 * lane, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = fmaf(w, v[k], acc[k]);
      load8(base + 256 + 8 * lane, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[8 + k] = fmaf(w, v[k], acc[8 + k]);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    s_acc[warp][8 * lane + k] = acc[k];
    s_acc[warp][256 + 8 * lane + k] = acc[8 + k];
  }
  if (lane == 0) s_w[warp] = wsum;
  __syncthreads();
  if (part != 0 || !valid) return;
  for (int q = 1; q < S; ++q) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc[k] += s_acc[warp + q][8 * lane + k];
      acc[8 + k] += s_acc[warp + q][256 + 8 * lane + k];
    }
    wsum += s_w[warp + q];
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* o = out + row * kDv;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint4 packed;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&packed);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      h[k] = __floats2bfloat162_rn(acc[8 * c + 2 * k] * inv, acc[8 * c + 2 * k + 1] * inv);
    *reinterpret_cast<uint4*>(o + 256 * c + 8 * lane) = packed;
  }
  if (out_lse != nullptr && lane == 0)
    out_lse[row] = wsum > 0.f ? (m2 + log2f(wsum)) * out_lse_mul : -INFINITY;
}

}  // namespace

cudaError_t launch_lse_combine(const void* partials, bool partials_fp32, const float* lses,
                               int n, long long rows, long long shard_stride_rows,
                               bool in_log2, float out_lse_mul, uint16_t* out,
                               float* out_lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const float k = in_log2 ? 1.0f : 1.4426950408889634f;
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
  // few rows of many bf16 shards: several warps per row (up to 4, at least 4 shards each,
  // at most 4 K warps).  From 2,048 rows on one warp per row has enough warps in flight
  // (2,048 rows of 8 shards: 10.2 us with one warp per row, 11.2 us with two; 1,024 rows
  // of 16 shards: 13.6 us with one, 9.2 us with four; GB300, ncu)
  int S = 1;
  if (rows < 2048)
    while (S < 4 && 2 * S * 4 <= n && rows * 2 * S <= 4096) S *= 2;
  if (!partials_fp32 && S > 1) {
    const long long rpb = kWarps / S;
    DependentLaunch dl(dim3((unsigned)((rows + rpb - 1) / rpb)), dim3(kWarps * 32), stream);
    const __nv_bfloat16* pb = static_cast<const __nv_bfloat16*>(partials);
    if (S == 2)
      return cudaLaunchKernelEx(&dl.cfg, lse_combine_split_kernel<__nv_bfloat16, 2>, pb, lses, n,
                                rows, shard_stride_rows, k, out_lse_mul, o, out_lse);
    return cudaLaunchKernelEx(&dl.cfg, lse_combine_split_kernel<__nv_bfloat16, 4>, pb, lses, n,
                              rows, shard_stride_rows, k, out_lse_mul, o, out_lse);
  }
  const long long blocks = (rows + kWarps - 1) / kWarps;
  DependentLaunch dl(dim3((unsigned)blocks), dim3(kWarps * 32), stream);
  if (partials_fp32)
    return cudaLaunchKernelEx(&dl.cfg, lse_combine_kernel<float>,
                              static_cast<const float*>(partials), lses, n, rows,
                              shard_stride_rows, k, out_lse_mul, o, out_lse);
  return cudaLaunchKernelEx(&dl.cfg, lse_combine_kernel<__nv_bfloat16>,
                            static_cast<const __nv_bfloat16*>(partials), lses, n, rows,
                            shard_stride_rows, k, out_lse_mul, o, out_lse);
}

}  // namespace mla
