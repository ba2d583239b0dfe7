// Split-KV paged MLA decode on the warp-level tensor-core path (mma.sync m16n8k16 bf16).
//
// What it computes (one shard): query row i of request b sees the global prefix
// G_i = max(0, G_b - (q_len-1-i)) ("vLLM PR #52188 (DSpark + DCP)" page, section
// "关键源码片段", _prepare_flattened_decode_metadata), of which this shard holds, under
// round-robin segments of I positions (span = cp * I),
// L_i = min(seq_lens[b], G_i / span * I + clamp(G_i % span - rank * I, 0, I)) keys (a
// non-causal block reads L_i = seq_lens[b] in every row, the snippet's other branch);
// keys are gathered page by page through the block table; out = softmax(scale * q K^T) V
// with V = K[:, :512] and lse in base e or 2 ("vLLM PR #54012" page, section "实现拆解"
// step 3; "vLLM PR #48180" page, section "实现拆解" step 1).
//
// This kernel is a cross-check of the tcgen05 kernel: calls run it only when a test
// selects it (mla_set_decode_kernel).
//
// Layout of the work: a CTA of 8 warps takes 64 query rows of one request (rows ordered
// (q-row i, head h), so a request's q_len*H rows share every key) and one contiguous
// range of that request's keys (split-KV).  Warp w owns rows 16*(w%4).. and the V/O
// half 256*(w/4)..; both halves recompute the same S = Q K^T tile (the warp-level path
// has no cross-warp S exchange).  Keys stream through a double-buffered shared-memory
// tile of 32 rows x 576 dims filled with 16-byte cp.async copies (zero-filled past the
// range, so poisoned cache slots are never read); Q stays in shared memory.  Online
// softmax runs in registers in base 2; P feeds the PV MMA straight from the S
// accumulators.  Splits write normalised fp32 partials + base-2 LSE to the workspace and
// the LSE combine kernel reduces them.
#include <math.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "internal.h"
#include "../../include/mla_decode.h"

namespace mla {
namespace {

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kRows = 64;
constexpr int kTok = 32;
constexpr int kStride = kD + 8;           // bf16 per smem row: 1168 B, conflict-free ldmatrix
constexpr int kThreads = 256;
constexpr int kSmemBytes = (kRows + 2 * kTok) * kStride * 2;
constexpr int kMaxSplits = 32;

struct Params {
  const uint16_t* q;
  const uint16_t* kv;
  const int32_t* bt;
  long long bt_stride;
  const int32_t* seq_lens;
  const int32_t* gseq;
  int B, H, q_len, bs, num_blocks, max_blocks, cp, rank;
  int causal, il;
  long long span;
  int rows;
  int splits;
  float scale_log2;
  float lse_mul;
  long long total_rows;
  uint16_t* out;
  float* lse;
  float* ws_o;
  float* ws_lse;
  unsigned int* status;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Keys visible to query row r (ordered (i, h)) of request b on this shard.
__device__ __forceinline__ int row_bound(const Params& p, int r, long long G, int cap) {
  if (!p.causal) return cap;
  const int i = r / p.H;
  long long Gi = G - (p.q_len - 1 - i);
  if (Gi < 0) Gi = 0;
  long long rem = Gi % p.span - (long long)p.rank * p.il;
  rem = rem < 0 ? 0 : (rem > p.il ? p.il : rem);
  const long long loc = Gi / p.span * p.il + rem;
  return (int)(loc < cap ? loc : cap);
}

__global__ void __launch_bounds__(kThreads, 1) mla_decode_mma_kernel(const Params p) {
  extern __shared__ __align__(128) uint16_t smem[];
  uint16_t* Qs = smem;                        // [64][kStride]
  uint16_t* Ks = smem + kRows * kStride;      // [2][32][kStride]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rg = warp & 3, dh = warp >> 2;
  const int split = blockIdx.x, rt = blockIdx.y, b = blockIdx.z;
  const int r0 = rt * kRows;

  // ---- bounds ---------------------------------------------------------------------
  int cap = __ldg(p.seq_lens + b);
  const int lim_all = p.max_blocks * p.bs;
  if (cap > lim_all) {
    if (tid == 0) atomicOr(p.status, MLA_STATUS_SEQ_TOO_LONG);
    cap = lim_all;
  }
  if (cap < 0) cap = 0;
  const long long G = __ldg(p.gseq + b);
  const int last_row = min(r0 + kRows, p.rows) - 1;
  const int Lmax = row_bound(p, last_row, G, cap);      // rows are ordered by i
  int chunk = (Lmax + p.splits - 1) / p.splits;
  chunk = (chunk + kTok - 1) / kTok * kTok;
  const int start = min(split * chunk, Lmax);
  const int end = min(start + chunk, Lmax);

  const int g = lane >> 2, c = lane & 3;
  const int rowA = r0 + rg * 16 + g, rowB = rowA + 8;
  const int limA = rowA < p.rows ? min(row_bound(p, rowA, G, cap), end) : 0;
  const int limB = rowB < p.rows ? min(row_bound(p, rowB, G, cap), end) : 0;

  // ---- Q -> smem (zero rows past the request's rows) -------------------------------
  const uint32_t qs_base = smem_u32(Qs);
  const uint32_t ks_base = smem_u32(Ks);
  for (int idx = tid; idx < kRows * (kD / 8); idx += kThreads) {
    const int rr = idx / (kD / 8), ch = idx % (kD / 8);
    const int row = r0 + rr;
    const bool ok = row < p.rows;
    const uint16_t* src = ok ? p.q + ((long long)b * p.rows + row) * kD + ch * 8 : p.q;
    cp_async16(qs_base + (rr * kStride + ch * 8) * 2, src, ok ? 16 : 0);
  }

  bool bad_page = false;
  const int ld_tok = tid >> 3, ld_c0 = tid & 7;
  auto load_tile = [&](int buf, int t0) {
    const int l = t0 + ld_tok;
    const uint16_t* src = nullptr;
    if (l < end) {
      const int page = __ldg(p.bt + (long long)b * p.bt_stride + l / p.bs);
      if (page < 0 || page >= p.num_blocks)
        bad_page = true;
      else
        src = p.kv + ((long long)page * p.bs + l % p.bs) * kD;
    }
    const uint32_t dst = ks_base + ((buf * kTok + ld_tok) * kStride) * 2;
#pragma unroll
    for (int k = 0; k < kD / 64; ++k) {
      const int ch = ld_c0 + 8 * k;
      cp_async16(dst + ch * 16, src ? src + ch * 8 : p.kv, src ? 16 : 0);
    }
  };

  const int ntiles = (end - start + kTok - 1) / kTok;
  if (ntiles > 0) load_tile(0, start);
  cp_async_commit();

  float acc[32][4];
#pragma unroll
  for (int n = 0; n < 32; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

  // ldmatrix lane addresses
  const int a_row = rg * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int a_col = (lane >> 4) * 8;
  const uint32_t a_addr0 = qs_base + (a_row * kStride + a_col) * 2;
  const int b_tok = (lane & 7) + (lane >> 4) * 8;
  const int b_col = ((lane >> 3) & 1) * 8;
  const int v_tok = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int v_col = dh * 256 + (lane >> 4) * 8;

  for (int it = 0; it < ntiles; ++it) {
    const int t0 = start + it * kTok;
    if (it + 1 < ntiles) {
      load_tile((it + 1) & 1, t0 + kTok);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t kbuf = ks_base + ((it & 1) * kTok * kStride) * 2;

    // ---- S = Q K^T over 576 dims: 16 rows x 32 keys per warp ----------------------
    float s[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < kD / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(a_addr0 + kk * 32, a0, a1, a2, a3);
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbuf + ((np * 16 + b_tok) * kStride + kk * 16 + b_col) * 2, b0, b1, b2, b3);
        mma_bf16(s[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }

    // ---- mask + online softmax (base 2) ------------------------------------------
    const int la = limA - t0, lb = limB - t0;
    float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = j * 8 + 2 * c + e;
        s[j][e] = tok < la ? s[j][e] * p.scale_log2 : -INFINITY;
        s[j][2 + e] = tok < lb ? s[j][2 + e] * p.scale_log2 : -INFINITY;
        mxA = fmaxf(mxA, s[j][e]);
        mxB = fmaxf(mxB, s[j][2 + e]);
      }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, o));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, o));
    }
    const float mnA = fmaxf(mA, mxA), mnB = fmaxf(mB, mxB);
    const float muA = mnA == -INFINITY ? 0.f : mnA;
    const float muB = mnB == -INFINITY ? 0.f : mnB;
    const float alA = exp2f(mA - muA), alB = exp2f(mB - muB);
    mA = mnA;
    mB = mnB;
    float sumA = 0.f, sumB = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s[j][0] = exp2f(s[j][0] - muA);
      s[j][1] = exp2f(s[j][1] - muA);
      s[j][2] = exp2f(s[j][2] - muB);
      s[j][3] = exp2f(s[j][3] - muB);
      sumA += s[j][0] + s[j][1];
      sumB += s[j][2] + s[j][3];
    }
    lA = lA * alA + sumA;
    lB = lB * alB + sumB;
#pragma unroll
    for (int n = 0; n < 32; ++n) {
      acc[n][0] *= alA;
      acc[n][1] *= alA;
      acc[n][2] *= alB;
      acc[n][3] *= alB;
    }

    // ---- O += P V over this warp's 256 V dims ------------------------------------
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t pa0 = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      const uint32_t pa1 = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      const uint32_t pa2 = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      const uint32_t pa3 = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      const uint32_t vrow = kbuf + ((kk * 16 + v_tok) * kStride + v_col) * 2;
#pragma unroll
      for (int np = 0; np < 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vrow + np * 32, b0, b1, b2, b3);
        mma_bf16(acc[2 * np], pa0, pa1, pa2, pa3, b0, b1);
        mma_bf16(acc[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  if (bad_page) atomicOr(p.status, MLA_STATUS_BAD_PAGE);

  // ---- epilogue ----------------------------------------------------------------------
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, o);
    lB += __shfl_xor_sync(0xffffffffu, lB, o);
  }
  const float invA = lA > 0.f ? 1.f / lA : 0.f, invB = lB > 0.f ? 1.f / lB : 0.f;
  const float lseA = lA > 0.f ? mA + log2f(lA) : -INFINITY;
  const float lseB = lB > 0.f ? mB + log2f(lB) : -INFINITY;
  const long long gA = (long long)b * p.rows + rowA, gB = (long long)b * p.rows + rowB;
  const int col0 = dh * 256 + 2 * c;
  if (p.splits == 1) {
    if (rowA < p.rows) {
      uint32_t* o = reinterpret_cast<uint32_t*>(p.out + gA * kDv + col0);
#pragma unroll
      for (int n = 0; n < 32; ++n) o[n * 4] = pack_bf16(acc[n][0] * invA, acc[n][1] * invA);
      if (p.lse != nullptr && dh == 0 && c == 0) p.lse[gA] = lseA * p.lse_mul;
    }
    if (rowB < p.rows) {
      uint32_t* o = reinterpret_cast<uint32_t*>(p.out + gB * kDv + col0);
#pragma unroll
      for (int n = 0; n < 32; ++n) o[n * 4] = pack_bf16(acc[n][2] * invB, acc[n][3] * invB);
      if (p.lse != nullptr && dh == 0 && c == 0) p.lse[gB] = lseB * p.lse_mul;
    }
  } else {
    const long long base = (long long)split * p.total_rows;
    if (rowA < p.rows) {
      float2* o = reinterpret_cast<float2*>(p.ws_o + (base + gA) * kDv + col0);
      if (lA > 0.f) {
#pragma unroll
        for (int n = 0; n < 32; ++n) o[n * 4] = make_float2(acc[n][0] * invA, acc[n][1] * invA);
      }
      if (dh == 0 && c == 0) p.ws_lse[base + gA] = lseA;
    }
    if (rowB < p.rows) {
      float2* o = reinterpret_cast<float2*>(p.ws_o + (base + gB) * kDv + col0);
      if (lB > 0.f) {
#pragma unroll
        for (int n = 0; n < 32; ++n) o[n * 4] = make_float2(acc[n][2] * invB, acc[n][3] * invB);
      }
      if (dh == 0 && c == 0) p.ws_lse[base + gB] = lseB;
    }
  }
}

int splits_for(int B, int H, int q_len, int num_sms) {
  const long long units = (long long)B * ((H * q_len + kRows - 1) / kRows);
  if (units <= 0) return 1;
  long long s = (2LL * num_sms + units - 1) / units;
  if (s < 1) s = 1;
  if (s > kMaxSplits) s = kMaxSplits;
  return (int)s;
}

size_t ws_bytes_for(int B, int H, int q_len, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = (size_t)B * H * q_len;
  const size_t o = (size_t)splits * rows * kDv * sizeof(float);
  const size_t l = (size_t)splits * rows * sizeof(float);
  return o + ((l + 255) / 256) * 256 + 256;
}

}  // namespace

size_t mma_workspace_size(int B, int H, int q_len, int num_sms) {
  return ws_bytes_for(B, H, q_len, splits_for(B, H, q_len, num_sms));
}

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t stream) {
  const int rows = a.H * a.q_len;
  if (a.B == 0 || rows == 0) return cudaSuccess;
  int splits = splits_for(a.B, a.H, a.q_len, a.num_sms);
  while (splits > 1 && ws_bytes_for(a.B, a.H, a.q_len, splits) > a.workspace_bytes) --splits;
  if (a.workspace == nullptr) splits = 1;

  Params p;
  p.q = a.q;
  p.kv = a.kv;
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.seq_lens = a.seq_lens;
  p.gseq = a.gseq;
  p.B = a.B;
  p.H = a.H;
  p.q_len = a.q_len;
  p.bs = a.block_size;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks;
  p.cp = a.cp_world;
  p.rank = a.cp_rank;
  p.causal = a.causal ? 1 : 0;
  p.il = a.interleave;
  p.span = (long long)a.cp_world * a.interleave;
  p.rows = rows;
  p.splits = splits;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.lse_mul = a.lse_base_e ? 0.6931471805599453f : 1.0f;
  p.total_rows = (long long)a.B * rows;
  p.out = a.out;
  p.lse = a.lse;
  p.status = a.status;
  if (splits > 1) {
    // partial O [splits][B*rows][512] fp32, then partial base-2 LSE [splits][B*rows]
    char* ws = static_cast<char*>(a.workspace);
    p.ws_o = reinterpret_cast<float*>(ws);
    p.ws_lse = reinterpret_cast<float*>(ws + (size_t)splits * p.total_rows * kDv * sizeof(float));
  } else {
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
  }

  // the shared-memory attribute is set on every call: this kernel runs only in tests,
  // and the call is cheap and safe from several host threads at once
  {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(splits, (rows + kRows - 1) / kRows, a.B);
  mla_decode_mma_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || splits == 1) return e;
  return launch_lse_combine(p.ws_o, true, p.ws_lse, splits, p.total_rows, p.total_rows, true,
                            p.lse_mul, a.out, a.lse, stream);
}

}  // namespace mla
