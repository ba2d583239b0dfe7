// Split-KV paged MLA decode on the Blackwell tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// What it computes is the same as the warp-level kernel (mla_decode_mma.cu): query row i
// of request b sees the global prefix G_i = max(0, G_b - (q_len-1-i)) ("vLLM PR #52188
// (DSpark + DCP)" page, section "关键源码片段"), of which this shard holds, under
// round-robin segments of I positions (span = cp * I),
// L_i = min(seq_lens[b], G_i / span * I + clamp(G_i % span - rank * I, 0, I)) keys; a
// non-causal block (the same snippet's other branch, a DSpark draft block) reads the
// shard's whole local sequence, L_i = seq_lens[b], in every row.
// out = softmax(scale q K^T) V with V = K[:, :512], lse in base e or 2 ("vLLM PR #54012"
// page, section "实现拆解" step 3; "vLLM PR #48180" page, section "实现拆解" step 1).
//
// Design.  A unit is 128 query rows of one request (rows ordered (q-row i, head h)); all
// of them share every key, so S = Q K^T and O = P V are dense 128-row contractions.  The
// fp32 accumulator O of 128 rows x 512 dims fills one SM's whole tensor memory, leaving
// no room for S.  So each unit runs on a CTA pair (a cluster of two SMs):
//
//   CTA 0 (the S-CTA) keeps Q in TMEM as the A operand (512 latent dims in 256 columns,
//     64 rope dims in 32) and two 64-column S buffers.  A TMA warp streams, for each unit,
//     Q (9 chunks of 128 rows x 64 dims) and then the keys (9 chunks of 64 keys x 64 dims
//     per tile, 128-byte swizzle, one 3-D box per 3 chunks) through a ring of 7 slots,
//     each freed as soon as the tcgen05.cp that moves a Q chunk into TMEM or the MMAs of
//     a key group complete; the MMA warp issues 36 MMAs (M=128, N=64, K=16) per tile into
//     S; eight softmax warps (two threads per query row, 32 keys each, swapping their row
//     maxima through shared memory) read S, apply the per-row causal bound,
//     keep the running max / sum (online softmax in base 2 against a per-row reference
//     max, set a headroom above a tile's max and moved only when a tile's max exceeds it
//     by more than a threshold, so that P <= 2^threshold and rescales of O are rare even
//     when a few keys score far above the rest; two budgets are compiled, see Budget),
//     and write P (bf16) with the per-row rescale factors into a
//     staging slot, which a copy warp bulk-copies into one of three receive slots of CTA 1.
//   CTA 1 (the O-CTA) holds O in all 512 TMEM columns.  A TMA warp streams the same keys'
//     first 512 dims (V) through five half-tile groups; the MMA warp issues 8 MMAs (M=128,
//     N=256, K=16) of P V per tile; eight warps rescale O in TMEM on the tiles where the
//     reference max moved, and at the end of a segment read O out, scale by 1/l and
//     store it.
//   Both MMA warps run their loops as whole converged warps and issue through elect.sync.
//
// Both CTAs compute every key exactly once for QK (576 dims) and once for PV (512 dims).
// Work is balanced statically: the 64-key tiles of all units are concatenated and cluster
// c takes tiles [c*T/C, (c+1)*T/C); a unit cut between clusters leaves bf16 partials
// (normalised out + base-2 LSE) in the workspace that the combine kernel merges.
//
// Safety: every wait is bounded (sm100.cuh); an abort word in each CTA (set on timeout,
// also written into the peer) makes all roles stop; TMA loads never point outside the
// cache (missing or invalid pages become out-of-range rows that TMA fills with zeros);
// V rows past a request's keys are zeroed in shared memory before the PV MMA, so that
// slots past seq_len (which may hold anything) never reach the accumulator.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <functional>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "sm100.cuh"
#include "../../include/mla_decode.h"

namespace mla {
namespace {

using namespace sm100;

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kM = 128;             // query rows per unit
constexpr int kTile = 64;           // keys per tile
constexpr int kChunkBytes = kTile * 128;      // 64 keys x 64 dims bf16 = 8 KB
constexpr int kKChunks = 9;         // 8 latent + 1 rope chunks per tile (S-CTA)
constexpr int kKGroup = 3;          // key chunks per TMA group (one 3-D box)
constexpr int kKGroups = 7;         // S-CTA key ring: 7 slots of 3 chunks (2.33 tiles)
constexpr int kVGroups = 5;         // O-CTA value ring: 5 half-tile groups of 4 chunks (2.5 tiles)
constexpr int kPBytes = kM * 128;   // P tile: 128 rows x 64 keys bf16 = 16 KB
constexpr int kSideBytes = 1024 + 16;         // alpha[128], inv_l[128], flags
constexpr int kPSlotBytes = 18432;  // P tile + sideband, 1 KB aligned
constexpr int kPRecv = 3;           // O-CTA P receive slots (the S-CTA stages in 2)
// Budget of the lazy rescale (log2 units).  A row's reference max is set kHeadroom above
// the tile max that moved it and moved again only when a tile's max exceeds it by more
// than kThreshold, so P <= 2^kThreshold and O is rescaled only when the running max has
// climbed by more than kThreshold + kHeadroom.  The narrow budget (32 / 64) keeps one
// rescale factor 2^-d normal for every move whose dropped sums could still matter
// (d <= 126 whenever they weigh more than 2^-30 of the new maximum).  The wide budget
// (64 / 80) rescales less often on long contexts with outlying keys; it sends the factor
// as a = 2^(-d/2) and every user multiplies by a twice, which stays normal up to d = 252,
// beyond which the dropped sums weigh less than 2^-108 of the new maximum.
template <bool kWide>
struct Budget {
  static constexpr float kThreshold = kWide ? 64.0f : 32.0f;
  static constexpr float kHeadroom = kWide ? 80.0f : 64.0f;
  static constexpr float kMaxTileSum = kWide ? 18446744073709551616.0f : 4294967296.0f;
  // exponent of the factor that is sent: (m_old - m_new) / 2 for the wide budget
  static constexpr float kFactorScale = kWide ? 0.5f : 1.0f;
};
constexpr int kThreads = 384;       // warps 0-3: roles; 4-11: softmax (S-CTA) / correction (O-CTA)
constexpr uint32_t kColRope = 384;  // TMEM columns: Q latent 0..255, S 256..383, Q rope 384..415
constexpr int kEvCorrect = 1;
constexpr int kEvFinal = 2;

// shared memory layout (identical offsets in both CTAs of a pair)
constexpr int kOffRing = 0;                                  // 7 x 24 KB (S) / 5 x 32 KB (O)
constexpr int kOffXchg = kOffRing + kKGroups * kKGroup * kChunkBytes;  // 172032: row max / sum
                                                             // exchange of the softmax warps
constexpr int kOffP = kOffXchg + kM * 128;                   // 188416
constexpr int kOffBar = kOffP + 2 * kPSlotBytes;             // 225280
constexpr int kOffPR = kVGroups * 4 * kChunkBytes;           // 163840: O-CTA receive slots
static_assert(kOffPR + kPRecv * kPSlotBytes <= kOffBar, "O-CTA receive slots");
constexpr int kOffFinInvL = kOffBar + 1024;                  // 128 floats (O-CTA)
constexpr int kOffMisc = kOffFinInvL + 512;                  // tmem base, abort, etc.
constexpr int kSmemBytes = kOffMisc + 64 + 1024;             // + alignment slack

// barrier indices (8 bytes each) inside [kOffBar, kOffBar + 1024)
enum Bar : int {
  // S-CTA
  B_KFULL = 0,            // [7] per key group slot
  B_KEMPTY = 7,           // [7]
  B_SFULL = 14,           // [2]
  B_SFREE = 16,           // [2]
  B_PFREE = 20,           // [3]  (arrived by the O-CTA's multicast commit)
  // O-CTA
  B_VFULL = 23,           // [5] per half-tile value group
  B_VEMPTY = 28,          // [5]
  B_PFULL = 33,           // [3]  (completed by the S-CTA's bulk copy)
  B_PVDONE = 36,
  B_EV = 37,              // MMA warp -> correction warps: one event (rescale or final)
  B_CORRDONE = 38,
  B_OFINAL = 39,
  B_OFREE = 40,
  // S-CTA: softmax warps <-> copy warp
  B_PSTAGED = 41,         // [2] P + sideband written into a staging slot (4 warps)
  B_STAGEFREE = 43,       // [2] the bulk copy has read the staging slot
  // both CTAs: the MMA warp's last tcgen05 operations have completed (abort path)
  B_DRAIN = 45,
  // S-CTA: never arrived at; the copy warp waits on it when a test asks for a stall
  B_NEVER = 46,
  B_COUNT = 47
};

struct Params {
  const uint16_t* q;
  const int32_t* bt;
  long long bt_stride;
  const int32_t* seq_lens;
  const int32_t* gseq;
  int B, H, q_len, bs, num_blocks, max_blocks, cp, rank;
  int causal;          // 0: every row of a block reads the shard's whole local sequence
  int il;              // interleave: round-robin segments of il positions
  long long span;      // cp * il
  unsigned long long wait_ns;   // limit of every bounded wait
  int stall_test;      // tests: the copy warp first waits for an arrival that never comes
  int seg_tiles;       // start-up share of a request on the split line, in tiles
  int shard_B;         // requests per shard (request b: q / gseq row b % shard_B, rank + b / shard_B)
  unsigned shard_mul;  // 0 for one shard, else ceil(2^32 / shard_B): b / shard_B = umulhi(b, shard_mul)
  int rows;            // H * q_len
  int row_tiles;       // ceil(rows / 128)
  int units;           // B * row_tiles
  int clusters;        // C
  int groups;          // G = clusters / row_tiles: clusters g*R .. g*R+R-1 form group g
  int whole_units;     // 1: no workspace, each group takes whole requests round-robin
  int box_rows;        // rows per TMA box = min(bs, 64)
  int kz, vz;          // chunks per K / V TMA box (3 and 4, or 1 when a page is < 64 rows)
  int out_v8;          // out is 32-byte aligned: output rows are written in 32-byte pieces
  float scale_log2;
  float lse_mul;
  uint16_t* out;
  float* lse;
  long long* hdr;      // workspace header: [0] = length T of this call's split line
  int2* meta;          // [units] first / last cluster of each unit
  float* ws_lse;       // [units + C][128]
  uint16_t* ws_o;      // [units + C][128][512] normalised partial outputs, bf16
  unsigned int* status;
};

// 32-byte global store (one full sector per thread); `dst` 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ uint32_t bar_addr(uint32_t smem_base, int i) {
  return smem_base + kOffBar + 8 * i;
}

// Keys visible to row r (0-based within the request's q_len*H rows): the shard's share of
// the row's global prefix under round-robin segments of il positions, at most cap.  Out of
// line: it is needed once per segment, and its 64-bit divisions inlined at every call
// site slowed the kernel's hot loops (code size; measured on GB300).
__device__ __noinline__ int row_bound(const Params& p, int r, long long G, int cap, int rank) {
  if (!p.causal) return cap;
  const int i = r / p.H;
  long long Gi = G - (p.q_len - 1 - i);
  if (Gi < 0) Gi = 0;
  long long rem = Gi % p.span - (long long)rank * p.il;
  rem = rem < 0 ? 0 : (rem > p.il ? p.il : rem);
  const long long loc = Gi / p.span * p.il + rem;
  return (int)(loc < cap ? loc : cap);
}

// Shard of request b and its row in q / gseq, without a division.
__device__ __forceinline__ int shard_of(const Params& p, int b) {
  return (int)__umulhi((unsigned)b, p.shard_mul);
}

__device__ __forceinline__ int seq_cap(const Params& p, int b) {
  int cap = __ldg(p.seq_lens + b);
  const int lim = p.max_blocks * p.bs;
  if (cap > lim) cap = lim;
  return cap < 0 ? 0 : cap;
}

// Largest visible length over the rows of unit u (rows are ordered by q-row).
__device__ __forceinline__ int unit_keys(const Params& p, int u) {
  const int b = u / p.row_tiles, rt = u % p.row_tiles;
  const int last_row = min((rt + 1) * kM, p.rows) - 1;
  const int sh = shard_of(p, b);
  return row_bound(p, last_row, __ldg(p.gseq + (b - sh * p.shard_B)), seq_cap(p, b), p.rank + sh);
}

__device__ __forceinline__ int unit_tiles(const Params& p, int u) {
  return (unit_keys(p, u) + kTile - 1) / kTile;
}

// Tiles of request b: those of its last row tile, which sees the most keys (rows are
// ordered by query position, and a later position sees one more key).
__device__ __forceinline__ int req_tiles(const Params& p, int b) {
  return unit_tiles(p, b * p.row_tiles + p.row_tiles - 1);
}

// Length of request b on the split line: its tiles plus the start-up share p.seg_tiles
// (none when it has no tile).
__device__ __forceinline__ long long req_span(const Params& p, int b) {
  const int nt = req_tiles(p, b);
  return nt > 0 ? (long long)nt + p.seg_tiles : 0;
}

// Work split.  The clusters form G groups of R = row_tiles clusters.  The requests' tiles
// are laid end to end, each request with a tile preceded by seg_tiles positions that stand
// for the cost of starting a segment; group g takes the positions [g*T/G, (g+1)*T/G) of
// that line (T = its length), and its cluster g*R + rt runs row tile rt of the tiles among
// them, so that the R units of a request read the same keys at the same time (from L2
// after the first).  A unit's range is clamped to its own tile count (at most one fewer
// than its request's).  SegIter walks the segments (unit, tile range) of one cluster in
// order; every role of both CTAs of the pair runs its own copy of it and sees the same
// sequence.
struct SegIter {
  int u;            // current unit = b * row_tiles + rt
  int b;            // its request
  int rt;           // this cluster's row tile
  int grp;          // this cluster's group
  int t_begin;      // first tile of the segment within the unit
  int t_end;        // one past the last tile
  long long g0;     // position of request b's first tile on the split line
  long long g_end;  // end of the group's range
  bool whole;
  bool single;      // the segment covers the whole unit
  int nt;           // the unit's tile count
  int slot;         // workspace slot of a partial: (b + grp) * R + rt
};

__device__ __forceinline__ long long range_start(long long T, int c, int C) {
  return T * c / C;
}

// Index of the group that owns request tile x.
__device__ __forceinline__ int owner_of(long long x, long long T, int C) {
  return (int)(((x + 1) * C - 1) / T);
}

// Sets the segment of request it.b from tile tb, clamped to the unit's tiles; false if
// that leaves nothing.
__device__ __forceinline__ bool seg_set(const Params& p, SegIter& it, int tb) {
  it.u = it.b * p.row_tiles + it.rt;
  const int nu = unit_tiles(p, it.u);
  int te = nu;
  if (!it.whole) te = (int)min((long long)te, it.g_end - it.g0);
  if (tb >= te) return false;
  it.t_begin = tb;
  it.t_end = te;
  it.single = (tb == 0 && te == nu);
  it.nt = nu;
  it.slot = (it.b + it.grp) * p.row_tiles + it.rt;
  return true;
}

__device__ bool seg_next(const Params& p, SegIter& it) {
  if (it.whole) {
    for (int b = it.b + p.groups; b < p.B; b += p.groups) {
      it.b = b;
      if (seg_set(p, it, 0)) return true;
    }
    return false;
  }
  for (;;) {
    // the next request's first tile, after its start-up share
    const long long g = it.g0 + req_tiles(p, it.b) + p.seg_tiles;
    if (g >= it.g_end) return false;
    int b = it.b + 1;
    while (b < p.B && req_tiles(p, b) == 0) ++b;
    if (b >= p.B) return false;
    it.b = b;
    it.g0 = g;
    if (seg_set(p, it, 0)) return true;
  }
}

// First segment of cluster c, or none.  s_scan holds the request whose span contains the
// group's first position and that request's first tile position (from the prologue's
// scan); a range that starts inside a start-up share starts at the request's first tile.
__device__ bool seg_first(const Params& p, int c, SegIter& it, long long T, int* s_scan) {
  it.grp = c / p.row_tiles;
  it.rt = c % p.row_tiles;
  it.whole = p.whole_units != 0;
  if (it.grp >= p.groups) return false;
  if (it.whole) {
    it.g0 = 0;
    it.g_end = 0;
    for (int b = it.grp; b < p.B; b += p.groups) {
      it.b = b;
      if (seg_set(p, it, 0)) return true;
    }
    return false;
  }
  const long long a = range_start(T, it.grp, p.groups), e = range_start(T, it.grp + 1, p.groups);
  if (a >= e || s_scan[0] < 0) return false;
  it.b = s_scan[0];
  it.g0 = ((long long)s_scan[2] << 32) | (unsigned)s_scan[1];
  it.g_end = e;
  return seg_set(p, it, a > it.g0 ? (int)(a - it.g0) : 0) || seg_next(p, it);
}

// Cache rows of a segment's TMA boxes for a producer warp: box i covers box_rows keys
// from token i * box_rows; a missing or invalid page becomes a row past the cache, which
// TMA fills with zeros.  Lane l holds box i0 + l of the current window of 32 boxes, and the
// page numbers of the next window are loaded one window ahead.
struct BoxWindow {
  const int32_t* btrow;
  int seg_keys, i0, cur, nxt, lane;
  bool bad;

  __device__ int row_of(const Params& p, int i) {
    const int tok = i * p.box_rows;
    int y = p.num_blocks * p.bs;
    if (tok < seg_keys) {
      const int page = __ldg(btrow + tok / p.bs);
      if (page >= 0 && page < p.num_blocks)
        y = page * p.bs + tok % p.bs;
      else
        bad = true;
    }
    return y;
  }
  __device__ void start(const Params& p, const SegIter& it) {
    btrow = p.bt + (long long)(it.u / p.row_tiles) * p.bt_stride;
    seg_keys = min(unit_keys(p, it.u), it.t_end * kTile);
    i0 = it.t_begin * (kTile / p.box_rows);
    cur = row_of(p, i0 + lane);
    nxt = row_of(p, i0 + 32 + lane);
  }
  // rows of the boxes of tile t; warp-collective.  A tile's boxes (1, 2 or 4 of them)
  // never straddle two windows.
  __device__ void tile_rows(const Params& p, int t, int (&ys)[4]) {
    const int nbox = kTile / p.box_rows;
    if (t * nbox >= i0 + 32) {
      i0 += 32;
      cur = nxt;
      nxt = row_of(p, i0 + 32 + lane);
    }
#pragma unroll
    for (int bx = 0; bx < 4; ++bx) ys[bx] = __shfl_sync(0xffffffffu, cur, (t * nbox + bx - i0) & 31);
  }
};

// ---------------------------------------------------------------------------------
// kernel
// ---------------------------------------------------------------------------------
struct SmemCtx {
  uint32_t base;          // shared address of the aligned base
  uint8_t* ptr;           // generic pointer of the aligned base
  volatile int* abort;
};

__device__ __forceinline__ void set_abort_both(const SmemCtx& s, uint32_t peer) {
  *s.abort = 1;
  st_cluster_u32(mapa(s.base + kOffMisc + 4, peer), 1u);
}

// Bounded wait; on failure the abort word of both CTAs of the pair is set.
__device__ __forceinline__ bool wait_bar(const SmemCtx& s, int i, uint32_t parity,
                                         const Params& p, bool cluster_scope = false) {
  if (mbar_wait(bar_addr(s.base, i), parity, s.abort, p.status, p.wait_ns, cluster_scope))
    return true;
  set_abort_both(s, cluster_ctarank() ^ 1u);
  return false;
}

// 2^x on the SFU (ex2.approx, flush-to-zero); arguments here are <= 32 or -inf.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 1/x and log2(x) on the SFU (rcp.approx / lg2.approx, relative error near 2^-23 and
// absolute error near 2^-22): a row's 1/l and LSE, taken once per segment.
__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (a single instruction on this architecture).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two fp32 lanes in one 64-bit register, and the paired fused multiply-add / add on them
// (each lane rounded exactly as the scalar fmaf / +).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Named barrier 1 over the 256 softmax threads that also ORs a flag across them.
__device__ __forceinline__ bool bar_or_256(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 256, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// A wait's outcome made uniform across the warp (every lane waited itself).
__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

// The same across the 256 threads of warps 4..11 (named barrier 2), so that no thread of
// the group leaves a loop that the others stay in (they meet again at named barriers).
__device__ __forceinline__ bool group_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.and.pred q, 2, 256, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}

template <bool kWide>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap,
                         const __grid_constant__ CUtensorMap qmap, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  SmemCtx s;
  s.ptr = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  s.base = smem_u32(s.ptr);
  uint32_t* misc = reinterpret_cast<uint32_t*>(s.ptr + kOffMisc);   // [0] tmem base, [1] abort
  s.abort = reinterpret_cast<volatile int*>(misc + 1);
  int* s_scan = reinterpret_cast<int*>(misc + 4);                     // [u, g0 lo, g0 hi]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t peer = crank ^ 1u;
  const int c = (int)cluster_id_x();
  const bool is_s = (crank == 0);

  // the tensor-map descriptors are fetched while the setup below runs
  if (tid == 96) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&vmap);
  }

  // ---- setup: barriers, TMEM, schedule scan -----------------------------------------
  if (tid == 0) {
    *s.abort = 0;
    for (int i = 0; i < kKGroups; ++i) {
      mbar_init(bar_addr(s.base, B_KFULL + i), 1);
      mbar_init(bar_addr(s.base, B_KEMPTY + i), 1);
    }
    for (int i = 0; i < kVGroups; ++i) {
      mbar_init(bar_addr(s.base, B_VFULL + i), 1);
      mbar_init(bar_addr(s.base, B_VEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_addr(s.base, B_SFULL + i), 1);
      mbar_init(bar_addr(s.base, B_SFREE + i), 8);
    }
    for (int i = 0; i < kPRecv; ++i) {
      mbar_init(bar_addr(s.base, B_PFREE + i), 1);
      mbar_init(bar_addr(s.base, B_PFULL + i), 1);
      // the O-CTA expects each receive slot's first P tile (and re-arms it after each use)
      if (crank == 1) mbar_arrive_expect_tx(bar_addr(s.base, B_PFULL + i), kPBytes + kSideBytes);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_addr(s.base, B_PSTAGED + i), 8);
      mbar_init(bar_addr(s.base, B_STAGEFREE + i), 1);
    }
    mbar_init(bar_addr(s.base, B_PVDONE), 1);
    mbar_init(bar_addr(s.base, B_EV), 1);
    mbar_init(bar_addr(s.base, B_CORRDONE), 8);
    mbar_init(bar_addr(s.base, B_OFINAL), 1);
    mbar_init(bar_addr(s.base, B_OFREE), 8);
    mbar_init(bar_addr(s.base, B_DRAIN), 1);
    mbar_init(bar_addr(s.base, B_NEVER), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(s.base + kOffMisc, 512);
    tmem_relinquish();
  }

  // schedule: the length T of the split line and the request holding this group's first
  // position
  long long T = 0;
  {
    __shared__ long long s_warp[kThreads / 32];
    if (tid == 0) s_scan[0] = -1;
    // pass 1: T, summed per warp (one shared 64-bit atomic per thread made this pass
    // ~10 us longer at 256 requests, measured on GB300)
    long long local = 0;
    for (int b = tid; b < p.B; b += kThreads) local += req_span(p, b);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if (lane == 0) s_warp[warp] = local;
    __syncthreads();
    for (int w = 0; w < kThreads / 32; ++w) T += s_warp[w];
    __syncthreads();
    if (!p.whole_units && T > 0 && c / p.row_tiles < p.groups) {
      const long long a = range_start(T, c / p.row_tiles, p.groups);
      // pass 2: chunked exclusive scan to find the request whose span contains position a
      long long running = 0;
      for (int base = 0; base < p.B; base += kThreads) {
        const int u = base + tid;          // a request index here
        const long long nt = u < p.B ? req_span(p, u) : 0;
        long long incl = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        long long wpre = 0, total = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
          if (w < warp) wpre += s_warp[w];
          total += s_warp[w];
        }
        const long long excl = running + wpre + incl - nt;
        if (u < p.B && nt > 0 && excl <= a && a < excl + nt) {
          const long long first = excl + p.seg_tiles;   // the request's first tile position
          s_scan[0] = u;
          s_scan[1] = (int)(first & 0xffffffffLL);
          s_scan[2] = (int)(first >> 32);
        }
        running += total;
        __syncthreads();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();          // barrier inits visible cluster-wide before any remote arrive
  tc_fence_after();
  const uint32_t tmem = misc[0];

  // meta for the combine: the owner of a unit's first tile records the range of groups that
  // hold it; cluster 0 records T so that the combine can skip groups with an empty range
  if (is_s && tid == 0 && c == 0 && !p.whole_units && p.hdr != nullptr) p.hdr[0] = T;

  const float kNegInf = -INFINITY;

  if (is_s) {
    // ============================== S-CTA ==========================================
    if (warp == 0) {
      // ---- K producer: per tile 3 groups of 3 chunks, each one 3-D TMA box per page
      // part (the whole warp runs the loop; one elected lane issues) --------------------
      SegIter it;
      BoxWindow win;
      win.lane = lane;
      win.bad = false;
      long long issued = 0; // key groups issued
      int slot = 0;
      uint32_t par = 1;     // a slot's first use passes at once
      bool okk = true;
      const int nbox = kTile / p.box_rows;
      if (seg_first(p, c, it, T, s_scan)) {
        do {
          // the unit's Q (128 rows x 576 dims) first: 9 chunks of 64 dims, one per ring
          // slot, which the MMA warp copies into TMEM; the unit's page rows are looked up
          // while the first seven are in flight
          const int qb = it.u / p.row_tiles;
          const int qy = (qb - shard_of(p, qb) * p.shard_B) * p.rows + (it.u % p.row_tiles) * kM;
          static_assert(kKChunks > kKGroups, "page window started inside the Q loop");
          for (int qc = 0; qc < kKChunks && okk; ++qc) {
            if (qc == kKGroups) win.start(p, it);
            okk = warp_all(wait_bar(s, B_KEMPTY + slot, par, p));
            if (!okk) break;
            const uint32_t fb = bar_addr(s.base, B_KFULL + slot);
            mbar_arrive_expect_tx_warp(fb, kM * 128);
            tma_load_2d_warp(s.base + kOffRing + slot * kKGroup * kChunkBytes, &qmap, qc * 64, qy, fb);
            ++issued;
            if (++slot == kKGroups) {
              slot = 0;
              par ^= 1u;
            }
          }
          // for the combine: the owner of a unit's first tile records the range of groups
          // that hold the unit (after the unit's Q is on its way)
          if (lane == 0 && okk && it.t_begin == 0 && !it.whole && p.meta != nullptr)
            p.meta[it.u] = make_int2(it.grp, owner_of(it.g0 + it.nt - 1, T, p.groups));
          for (int t = it.t_begin; t < it.t_end && okk; ++t) {
            int ys[4];
            win.tile_rows(p, t, ys);
            for (int g = 0; g < kKChunks / kKGroup; ++g) {
              okk = warp_all(wait_bar(s, B_KEMPTY + slot, par, p));
              if (!okk) break;
              const uint32_t fb = bar_addr(s.base, B_KFULL + slot);
              mbar_arrive_expect_tx_warp(fb, kKGroup * kChunkBytes);
              const uint32_t dst = s.base + kOffRing + slot * kKGroup * kChunkBytes;
              for (int cc = 0; cc < kKGroup; cc += p.kz)
#pragma unroll
                for (int bx = 0; bx < 4; ++bx)
                  if (bx < nbox)
                    tma_load_3d_warp(dst + cc * kChunkBytes + bx * p.box_rows * 128, &kmap, 0, ys[bx],
                                     kKGroup * g + cc, fb);
              ++issued;
              if (++slot == kKGroups) {
                slot = 0;
                par ^= 1u;
              }
            }
          }
        } while (okk && warp_all(*s.abort == 0) && seg_next(p, it));
      }
      if (__any_sync(0xffffffffu, win.bad) && lane == 0) atomicOr(p.status, MLA_STATUS_BAD_PAGE);
      if (*s.abort && lane == 0) {
        // let loads already issued land before the CTA exits
        for (long long m = (issued > kKGroups ? issued - kKGroups : 0); m < issued; ++m)
          mbar_wait_drain(bar_addr(s.base, B_KFULL + (int)(m % kKGroups)), (uint32_t)((m / kKGroups) & 1));
      }
    } else if (warp == 1) {
      // ---- QK MMA issuer (the whole warp runs the loop; one elected lane issues) --------
      SegIter it;
      long long n = 0;
      int nseg = 0;
      const uint32_t idesc = idesc_bf16(kM, kTile, false, false);
      int kslot = 0;          // key group slot of the next group, and its phase parity
      uint32_t kpar = 0;
      if (seg_first(p, c, it, T, s_scan)) {
        do {
          // the unit's Q: 9 chunks from the ring into TMEM (latent dims at columns 0..255,
          // rope dims at kColRope); in issue order after the previous unit's last QK
          bool ok = true;
          for (int qc = 0; qc < kKChunks && ok; ++qc) {
            ok = warp_all(wait_bar(s, B_KFULL + kslot, kpar, p));
            if (!ok) break;
            tc_fence_after();
            const uint32_t qb = s.base + kOffRing + kslot * kKGroup * kChunkBytes;
            const uint32_t tq = tmem + (qc < 8 ? (uint32_t)qc * 32 : kColRope);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tmem_cp_128x256b_warp(tq + 8 * k, smem_desc(qb + 32 * k, 16, 1024, kSwizzle128B));
            mma_commit_warp(bar_addr(s.base, B_KEMPTY + kslot));
            if (++kslot == kKGroups) {
              kslot = 0;
              kpar ^= 1u;
            }
          }
          if (!ok) break;
          for (int t = it.t_begin; t < it.t_end && ok; ++t, ++n) {
            const int g = (int)(n & 1);
            ok = warp_all(wait_bar(s, B_SFREE + g, (uint32_t)(((n >> 1) + 1) & 1), p));
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem + 256 + g * kTile;
            // the tile's chunks arrive in 3 groups (slots 3n .. 3n+2 mod 7); the 32 latent
            // MMAs take A from TMEM, the 4 rope MMAs from shared memory.  The loops are
            // unrolled so that the issue sequence has no branch between MMAs.
#pragma unroll
            for (int gi = 0; gi < kKChunks / kKGroup; ++gi) {
              ok = warp_all(wait_bar(s, B_KFULL + kslot, kpar, p));
              if (!ok) break;
              const uint32_t gb = s.base + kOffRing + kslot * kKGroup * kChunkBytes;
              {
                const int ch = kKGroup * gi;
                mma12_ts_warp(d, tmem + (uint32_t)ch * 32, tmem + (uint32_t)(ch + 1) * 32,
                              tmem + (ch + 2 < 8 ? (uint32_t)(ch + 2) * 32 : kColRope),
                              smem_desc(gb, 16, 1024, kSwizzle128B), idesc, gi != 0);
              }
              mma_commit_warp(bar_addr(s.base, B_KEMPTY + kslot));   // this group's slot is free
              if (++kslot == kKGroups) {
                kslot = 0;
                kpar ^= 1u;
              }
            }
            if (!ok) break;
            mma_commit_warp(bar_addr(s.base, B_SFULL + g));
          }
          if (!ok || !warp_all(*s.abort == 0)) break;
          ++nseg;
        } while (seg_next(p, it));
      }
      // every tcgen05 operation issued here completes before the CTA tears down (they read
      // the key ring and write TMEM); after an abort nothing else has waited for them
      mma_commit_warp(bar_addr(s.base, B_DRAIN));
      mbar_wait_drain(bar_addr(s.base, B_DRAIN), 0);
    } else if (warp == 2) {
      // ---- copy warp: each staged P tile (+ sideband) into the O-CTA's receive slot -----
      // n % 3 once its previous tile there has been multiplied (the O-CTA's commit arrives
      // on p_free), then the staging slot is handed back to the softmax warps.
      SegIter it;
      long long n = 0;
      bool ok = true;
      // a test of the timeout path: this wait runs out, and every role of the pair stops
      if (p.stall_test && lane == 0) ok = wait_bar(s, B_NEVER, 0, p);
      if (ok && lane == 0 && seg_first(p, c, it, T, s_scan)) {
        do {
          for (int t = it.t_begin; t < it.t_end && ok; ++t, ++n) {
            const int j = (int)(n & 1);
            const int jr = (int)(n % kPRecv);
            ok = wait_bar(s, B_PSTAGED + j, (uint32_t)((n >> 1) & 1), p) &&
                 wait_bar(s, B_PFREE + jr, (uint32_t)(((n / kPRecv) & 1) ^ 1), p, true);
            if (!ok) break;
            // the O-CTA has armed its receive barrier for these bytes
            const uint32_t rbar = mapa(bar_addr(s.base, B_PFULL + jr), peer);
            bulk_s2cluster(mapa(s.base + kOffPR + jr * kPSlotBytes, peer),
                           s.base + kOffP + j * kPSlotBytes, kPBytes + kSideBytes, rbar);
            bulk_commit();
            bulk_wait_read<0>();
            mbar_arrive(bar_addr(s.base, B_STAGEFREE + j));
          }
        } while (ok && *s.abort == 0 && seg_next(p, it));
        bulk_wait<0>();
        // the O-CTA's last PV commits arrive on this CTA's p_free barriers
        if (n > 0 && !*s.abort) {
          for (long long k = (n >= kPRecv ? n - kPRecv : 0); k < n; ++k)
            wait_bar(s, B_PFREE + (int)(k % kPRecv), (uint32_t)((k / kPRecv) & 1), p, true);
        }
      }
    } else if (warp >= 4) {
      // ---- softmax warps: two threads per query row (warps w and w+4 share a TMEM lane
      // quadrant), each owning 32 of a tile's 64 keys; the halves swap their row maxima
      // (and, on a unit's last tile, their sums) through shared memory, so that both take
      // the same decisions on the running max ---------------------------------------------
      const int q4 = warp & 3;
      const int hk = (warp - 4) >> 2;               // keys [32 hk, 32 hk + 32) of a tile
      const int r = q4 * 32 + lane;                 // row within the unit, = TMEM lane
      const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
      float* xmax = reinterpret_cast<float*>(s.ptr + kOffXchg);          // [2 tiles][2][128]
      float* xsum = xmax + 2 * 2 * kM;                                   // [2][128]
      SegIter it;
      long long n = 0;
      int nseg = 0;
      if (seg_first(p, c, it, T, s_scan)) {
        do {
          const int b = it.u / p.row_tiles, rt = it.u % p.row_tiles;
          const int row = rt * kM + r;
          const bool valid = row < p.rows;
          const int sh = shard_of(p, b);
          const long long G = __ldg(p.gseq + (b - sh * p.shard_B));
          const int cap = seq_cap(p, b);
          const int Lr = valid ? row_bound(p, row, G, cap, p.rank + sh) : 0;
          const int seg_end_tok = it.t_end * kTile;
          const int lim_row = min(Lr, seg_end_tok);

          float m_ref = kNegInf, l = 0.f;           // l: this half's share of the row sum
          bool aborted = false;
          for (int t = it.t_begin; t < it.t_end; ++t, ++n) {
            const int g = (int)(n & 1);
            const int j = (int)(n & 1);            // P staging slot
            // every exit from this loop is decided by all 256 threads together (they meet
            // at named barriers), so a thread that failed a wait of its own leaves here
            if (!group_all(!aborted && wait_bar(s, B_SFULL + g, (uint32_t)((n >> 1) & 1), p))) {
              aborted = true;
              break;
            }
            tc_fence_after();
            uint32_t sv[32];
            tmem_ld32(tmem + lane_off + 256 + g * kTile + 32 * hk, sv);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_addr(s.base, B_SFREE + g));

            const int t0 = t * kTile;
            const int lim = lim_row - t0 - 32 * hk;   // valid keys of this row in the half
            // keys of the half this row does not see score -inf: weight exactly 0, whatever
            // their cache slot holds, so one code path serves whole and partial halves
            if (lim < 32) {
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (k >= lim) sv[k] = 0xff800000u;
            }
            // Common case first: the running max already bounds this tile (no 2^x above
            // 2^threshold, checked through the sum).  All 256 threads then keep the running
            // max, and one barrier with an OR-reduction tells them whether any row needs the
            // full step below (a new max, or a unit's first tile), which all of them then
            // take.
            float alpha = 1.f;
            bool resc = false;
            uint32_t pk[16];
            float fsum = 0.f;
            bool fast = m_ref != kNegInf;
            if (fast) {
              const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2);
              const uint64_t nm2 = f32x2(-m_ref, -m_ref);
              uint64_t s2[4] = {0, 0, 0, 0};
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                float y0, y1;
                f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1])),
                                      sc2, nm2), y0, y1);
                const float e0 = fast_exp2(y0), e1 = fast_exp2(y1);
                s2[k & 3] = add_f32x2(s2[k & 3], f32x2(e0, e1));
                pk[k] = pack_bf16x2(e0, e1);
              }
              float t0, t1;
              f32x2_split(add_f32x2(add_f32x2(s2[0], s2[1]), add_f32x2(s2[2], s2[3])), t0, t1);
              fsum = t0 + t1;
              fast = fsum <= Budget<kWide>::kMaxTileSum;
            }
            const bool slow = bar_or_256(!fast);
            using Bd = Budget<kWide>;
            if (!slow) {
              l += fsum;
            } else {
              // running max on the raw scores (scale > 0 keeps the order), in log2 units,
              // with three-input maxima and paired fp32 arithmetic, so that these warps leave
              // issue slots to the MMA warp that shares their scheduler
              float m4[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
              for (int k = 0; k < 32; k += 8)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  m4[q] = fmax3(m4[q], __uint_as_float(sv[k + 2 * q]), __uint_as_float(sv[k + 2 * q + 1]));
              const float hmax = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
              float* xm = xmax + (n & 1) * 2 * kM;
              xm[hk * kM + r] = hmax;
              asm volatile("bar.sync 1, 256;" ::: "memory");
              const float smax = fmaxf(hmax, xm[(hk ^ 1) * kM + r]);
              const float tmax = smax * p.scale_log2;
              if (tmax > m_ref + Bd::kThreshold) {
                const float m_new = tmax + Bd::kHeadroom;
                if (m_ref != kNegInf) {
                  alpha = fast_exp2((m_ref - m_new) * Bd::kFactorScale);
                  resc = true;
                }
                l *= alpha;
                if (kWide) l *= alpha;
                m_ref = m_new;
              }
              const float neg_mu = (m_ref == kNegInf) ? 0.f : -m_ref;
              // e = 2^(s * scale_log2 - m) two keys per instruction (each lane rounds as fmaf)
              const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2);
              const uint64_t nm2 = f32x2(neg_mu, neg_mu);
              uint64_t s2[4] = {0, 0, 0, 0};
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                float y0, y1;
                f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1])),
                                      sc2, nm2), y0, y1);
                const float e0 = fast_exp2(y0), e1 = fast_exp2(y1);
                s2[k & 3] = add_f32x2(s2[k & 3], f32x2(e0, e1));
                pk[k] = pack_bf16x2(e0, e1);
              }
              float t0, t1;
              f32x2_split(add_f32x2(add_f32x2(s2[0], s2[1]), add_f32x2(s2[2], s2[3])), t0, t1);
              l += t0 + t1;
            }
            const bool last = (t + 1 == it.t_end);
            float l_row = 0.f;                     // the whole row's sum, on the last tile
            if (last) {
              xsum[hk * kM + r] = l;
              asm volatile("bar.sync 1, 256;" ::: "memory");
              l_row = l + xsum[(hk ^ 1) * kM + r];
            }
            const bool any_resc = __any_sync(0xffffffffu, resc);

            // staging slot j must no longer be read by the copy of tile n-2; a warp whose
            // wait failed writes nothing and leaves at the next group-wide decision
            if (!warp_all(wait_bar(s, B_STAGEFREE + j, (uint32_t)(((n >> 1) & 1) ^ 1), p))) {
              aborted = true;
              continue;
            }
            uint8_t* slot = s.ptr + kOffP + j * kPSlotBytes;
            uint8_t* prow = slot + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(prow + (((4 * hk + q) ^ (r & 7)) << 4)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            if (hk == 0) {
              float* side = reinterpret_cast<float*>(slot + kPBytes);
              // the O-CTA reads the factors only after a step that may rescale (taken by all
              // rows together), and 1 / l only on a unit's last tile
              if (slow) side[r] = alpha;
              if (last) side[128 + r] = l_row > 0.f ? fast_rcp(l_row) : 0.f;
              int* flags = reinterpret_cast<int*>(slot + kPBytes + 1024);
              if (lane == 0) flags[q4] = any_resc ? 1 : 0;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_addr(s.base, B_PSTAGED + j));
            if (last && valid && hk == 0) {
              const float lse2 = l_row > 0.f ? m_ref + fast_log2(l_row) : kNegInf;
              const long long grow = (long long)b * p.rows + row;
              if (it.single) {
                if (p.lse != nullptr) p.lse[grow] = lse2 * p.lse_mul;
              } else {
                p.ws_lse[(long long)it.slot * kM + r] = lse2;
              }
            }
          }
          if (!group_all(!aborted && *s.abort == 0)) break;
          ++nseg;
        } while (seg_next(p, it));
      }
    }
  } else {
    // ============================== O-CTA ==========================================
    if (warp == 0) {
      // ---- V producer: per half tile one group of 4 chunks, one 3-D TMA box per page
      // part (the whole warp runs the loop; one elected lane issues) --------------------
      SegIter it;
      BoxWindow win;
      win.lane = lane;
      win.bad = false;
      long long issued = 0;     // half-tile groups issued
      int grp = 0;
      uint32_t par = 1;
      bool okv = true;
      const int nbox = kTile / p.box_rows;
      if (seg_first(p, c, it, T, s_scan)) {
        do {
          win.start(p, it);
          for (int t = it.t_begin; t < it.t_end && okv; ++t) {
            int ys[4];
            win.tile_rows(p, t, ys);
            for (int h = 0; h < 2; ++h) {
              okv = warp_all(wait_bar(s, B_VEMPTY + grp, par, p));
              if (!okv) break;
              const uint32_t fb = bar_addr(s.base, B_VFULL + grp);
              mbar_arrive_expect_tx_warp(fb, 4 * kChunkBytes);
              const uint32_t dst = s.base + kOffRing + grp * 4 * kChunkBytes;
              for (int cc = 0; cc < 4; cc += p.vz)
#pragma unroll
                for (int bx = 0; bx < 4; ++bx)
                  if (bx < nbox)
                    tma_load_3d_warp(dst + cc * kChunkBytes + bx * p.box_rows * 128, &vmap, 0, ys[bx],
                                     4 * h + cc, fb);
              ++issued;
              if (++grp == kVGroups) {
                grp = 0;
                par ^= 1u;
              }
            }
          }
        } while (okv && warp_all(*s.abort == 0) && seg_next(p, it));
      }
      if (*s.abort && lane == 0) {
        for (long long q = (issued > kVGroups ? issued - kVGroups : 0); q < issued; ++q)
          mbar_wait_drain(bar_addr(s.base, B_VFULL + (int)(q % kVGroups)), (uint32_t)((q / kVGroups) & 1));
      }
    } else if (warp == 1) {
      // ---- PV MMA issuer (lane 0 issues; the warp zeroes V rows past the keys) ---------
      SegIter it;
      long long n = 0;
      long long pv_phase = 0;        // phases of B_PVDONE waited for (one per fresh commit)
      int nseg = 0;
      const uint32_t idesc = idesc_bf16(kM, 256, false, true);
      float* fin = reinterpret_cast<float*>(s.ptr + kOffFinInvL);
      volatile int* ev_word = reinterpret_cast<volatile int*>(misc + 8);
      int ncorr = 0;
      if (seg_first(p, c, it, T, s_scan)) {
        do {
          const int keys = unit_keys(p, it.u);
          const int seg_keys = min(keys, it.t_end * kTile);
          if (nseg > 0 && !warp_all(wait_bar(s, B_OFREE, (uint32_t)((nseg - 1) & 1), p))) break;
          tc_fence_after();
          bool ok = true;
          for (int t = it.t_begin; t < it.t_end && ok; ++t, ++n) {
            const int j = (int)(n % kPRecv);       // receive slot of this tile's P
            ok = warp_all(wait_bar(s, B_PFULL + j, (uint32_t)((n / kPRecv) & 1), p, true));
            if (!ok) break;
            // arm the slot for its next tile (the copy is issued only after this tile's PV)
            if (lane == 0) mbar_arrive_expect_tx(bar_addr(s.base, B_PFULL + j), kPBytes + kSideBytes);
            const uint8_t* slot = s.ptr + kOffPR + j * kPSlotBytes;
            const int* flags = reinterpret_cast<const int*>(slot + kPBytes + 1024);
            const bool first = (t == it.t_begin);
            const bool last = (t + 1 == it.t_end);
            const bool resc = !first && (flags[0] | flags[1] | flags[2] | flags[3]);
            if (last) {
              const float* side = reinterpret_cast<const float*>(slot + kPBytes);
              for (int k = lane; k < kM; k += 32) fin[k] = side[128 + k];
              __syncwarp();
            }
            if (resc) {
              // every PV issued so far must be complete before O is rescaled: one fresh
              // commit tracks all of them
              mma_commit_warp(bar_addr(s.base, B_PVDONE));
              ok = warp_all(wait_bar(s, B_PVDONE, (uint32_t)(pv_phase & 1), p));
              ++pv_phase;
              if (!ok) break;
              if (lane == 0) {
                *ev_word = kEvCorrect | (j << 8);
                mbar_arrive(bar_addr(s.base, B_EV));
              }
              ok = warp_all(wait_bar(s, B_CORRDONE, (uint32_t)(ncorr & 1), p));
              ++ncorr;
              if (!ok) break;
              tc_fence_after();
            }
            const int t0 = t * kTile;
            const int valid_keys = seg_keys - t0;
            const uint32_t pa = s.base + kOffPR + j * kPSlotBytes;
            for (int h = 0; h < 2 && ok; ++h) {
              const long long q = 2 * n + h;
              const int grp = (int)(q % kVGroups);
              ok = warp_all(wait_bar(s, B_VFULL + grp, (uint32_t)((q / kVGroups) & 1), p));
              if (!ok) break;
              if (valid_keys < kTile) {
                // zero V rows [valid_keys, 64) of the group's 4 chunks (whole 128-byte rows)
                const int r_lo = valid_keys < 0 ? 0 : valid_keys;
                for (int cc = 0; cc < 4; ++cc) {
                  uint8_t* base = s.ptr + kOffRing + (grp * 4 + cc) * kChunkBytes;
                  for (int idx = r_lo * 8 + lane; idx < kTile * 8; idx += 32) {
                    const int rr = idx >> 3, qq = idx & 7;
                    *reinterpret_cast<uint4*>(base + (rr >> 3) * 1024 + (rr & 7) * 128 + qq * 16) =
                        make_uint4(0, 0, 0, 0);
                  }
                }
                fence_proxy_async_smem();
              }
              __syncwarp();
              tc_fence_after();
              const uint32_t vb = s.base + kOffRing + grp * 4 * kChunkBytes;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t adesc = smem_desc(pa + 32 * k, 16, 1024, kSwizzle128B);
                const uint64_t bdesc = smem_desc(vb + k * 2048, kChunkBytes, 1024, kSwizzle128B);
                mma_ss_warp(tmem + h * 256, adesc, bdesc, idesc, (first && k == 0) ? 0u : 1u);
              }
              mma_commit_warp(bar_addr(s.base, B_VEMPTY + grp));     // this half's group is free
            }
            if (!ok) break;
            {
              mma_commit_multicast_warp(bar_addr(s.base, B_PFREE + j), (uint16_t)1);
              if (last) mma_commit_warp(bar_addr(s.base, B_OFINAL));
            }
            if (last && lane == 0) {
              *ev_word = kEvFinal;
              mbar_arrive(bar_addr(s.base, B_EV));
            }
            __syncwarp();
          }
          if (!ok || !warp_all(*s.abort == 0)) break;
          ++nseg;
        } while (seg_next(p, it));
      }
      // every PV complete before teardown
      if (n > 0 && warp_all(*s.abort == 0)) {
        mma_commit_warp(bar_addr(s.base, B_PVDONE));
        warp_all(wait_bar(s, B_PVDONE, (uint32_t)(pv_phase & 1), p));
        ++pv_phase;
      }
      mma_commit_warp(bar_addr(s.base, B_DRAIN));
      mbar_wait_drain(bar_addr(s.base, B_DRAIN), 0);
    } else if (warp >= 4) {
      // ---- correction / epilogue warps: thread = row; warps w and w+4 share a TMEM lane
      // quadrant and take O's columns [256 hc, 256 hc + 256) ------------------------------
      const int q4 = warp & 3;
      const int hc = (warp - 4) >> 2;
      const int r = q4 * 32 + lane;
      const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
      const float* fin = reinterpret_cast<const float*>(s.ptr + kOffFinInvL);
      volatile int* ev_word = reinterpret_cast<volatile int*>(misc + 8);
      SegIter it;
      int nseg = 0, nev = 0;
      if (seg_first(p, c, it, T, s_scan)) {
        do {
          const int b = it.u / p.row_tiles, rt = it.u % p.row_tiles;
          const int row = rt * kM + r;
          const bool valid = row < p.rows;
          bool ok = true;
          // events from the MMA warp: rescale requests, then the segment's final one
          for (;;) {
            ok = warp_all(wait_bar(s, B_EV, (uint32_t)(nev & 1), p));
            ++nev;
            if (!ok) break;
            const int ev = *ev_word;
            if ((ev & 0xff) == kEvFinal) break;
            const int j = (ev >> 8) & 3;
            const uint8_t* slot = s.ptr + kOffPR + j * kPSlotBytes;
            tc_fence_after();
            const float a = reinterpret_cast<const float*>(slot + kPBytes)[r];
            if (__any_sync(0xffffffffu, a != 1.f)) {
              for (int c32 = 8 * hc; c32 < 8 * hc + 8; ++c32) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + c32 * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                  float x = __uint_as_float(v[k]) * a;
                  if (kWide) x *= a;
                  v[k] = __float_as_uint(x);
                }
                tmem_st32(tmem + lane_off + c32 * 32, v);
              }
              tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_addr(s.base, B_CORRDONE));
          }
          if (!ok) break;
          // epilogue: O * (1/l) -> out (single segment) or a bf16 partial
          ok = warp_all(wait_bar(s, B_OFINAL, (uint32_t)(nseg & 1), p));
          if (!ok) break;
          tc_fence_after();
          const float inv = fin[r];
          for (int c32 = 8 * hc; c32 < 8 * hc + 8; ++c32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + c32 * 32, v);
            tmem_wait_ld();
            if (!valid) continue;
            // one row per thread: 32-byte stores write whole sectors (out only when it is
            // 32-byte aligned; the workspace always is)
            if (it.single) {
              uint16_t* dst = p.out + ((long long)b * p.rows + row) * kDv + c32 * 32;
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  w[e] = pack_bf16x2(__uint_as_float(v[16 * q + 2 * e]) * inv,
                                     __uint_as_float(v[16 * q + 2 * e + 1]) * inv);
                if (p.out_v8) {
                  st_global_v8(dst + 16 * q, w);
                } else {
                  reinterpret_cast<uint4*>(dst + 16 * q)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                  reinterpret_cast<uint4*>(dst + 16 * q)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                }
              }
            } else {
              uint16_t* dst = p.ws_o + ((long long)it.slot * kM + r) * kDv + c32 * 32;
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  w[e] = pack_bf16x2(__uint_as_float(v[16 * q + 2 * e]) * inv,
                                     __uint_as_float(v[16 * q + 2 * e + 1]) * inv);
                st_global_v8(dst + 16 * q, w);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_addr(s.base, B_OFREE));
          ++nseg;
        } while (warp_all(*s.abort == 0) && seg_next(p, it));
      }
    }
  }

  // ---- teardown ------------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge the partials of units that were cut between clusters; units with no visible key
// get out = 0 and lse = -inf.  A warp per (unit, row); the first thread of each block of
// 8 rows decides once for the block whether the unit needs anything (most units were
// finished by one cluster), instead of every warp working out the unit's tile count.
__device__ __forceinline__ void combine_row(const Params& p, int b, int rt, int r,
                                            int lane, int nt, int2 m) {
  const int row = rt * kM + r;
  const long long grow = (long long)b * p.rows + row;
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + grow * kDv;
  if (nt == 0) {
    *reinterpret_cast<uint4*>(o + 8 * lane) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(o + 256 + 8 * lane) = make_uint4(0, 0, 0, 0);
    if (p.lse != nullptr && lane == 0) p.lse[grow] = -INFINITY;
    return;
  }
  const long long T = p.hdr[0];
  auto holds = [&](int cc) {
    return range_start(T, cc, p.groups) < range_start(T, cc + 1, p.groups);
  };
  // lanes take one holder each (32 at a time): the LSEs in one round of loads, then every
  // holder's partial row loaded without waiting on its weight (a non-holder's slot is
  // read but not used), accumulated in holder order
  auto lse_at = [&](int cc) { return p.ws_lse[((long long)(b + cc) * p.row_tiles + rt) * kM + r]; };
  float mx = -INFINITY;
  for (int cb = m.x; cb <= m.y; cb += 32) {
    const int cc = cb + lane;
    if (cc <= m.y && holds(cc)) mx = fmaxf(mx, lse_at(cc));
  }
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int cb = m.x; cb <= m.y; cb += 32) {
      const int cc = cb + lane;
      const float wl = (cc <= m.y && holds(cc)) ? exp2f(lse_at(cc) - mx) : 0.f;
      const int nh = min(32, m.y - cb + 1);
#pragma unroll 4
      for (int k = 0; k < nh; ++k) {
        const float w = __shfl_sync(0xffffffffu, wl, k);
        const uint16_t* src = p.ws_o + (((long long)(b + cb + k) * p.row_tiles + rt) * kM + r) * kDv;
        const uint4 a0 = __ldcs(reinterpret_cast<const uint4*>(src + 8 * lane));
        const uint4 a1 = __ldcs(reinterpret_cast<const uint4*>(src + 256 + 8 * lane));
        if (w == 0.f) continue;
        wsum += w;
        const uint4 av[2] = {a0, a1};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 a = av[h];
          // bf16 -> fp32 is the upper half of the word
          acc[8 * h + 0] = fmaf(w, __uint_as_float(a.x << 16), acc[8 * h + 0]);
          acc[8 * h + 1] = fmaf(w, __uint_as_float(a.x & 0xffff0000u), acc[8 * h + 1]);
          acc[8 * h + 2] = fmaf(w, __uint_as_float(a.y << 16), acc[8 * h + 2]);
          acc[8 * h + 3] = fmaf(w, __uint_as_float(a.y & 0xffff0000u), acc[8 * h + 3]);
          acc[8 * h + 4] = fmaf(w, __uint_as_float(a.z << 16), acc[8 * h + 4]);
          acc[8 * h + 5] = fmaf(w, __uint_as_float(a.z & 0xffff0000u), acc[8 * h + 5]);
          acc[8 * h + 6] = fmaf(w, __uint_as_float(a.w << 16), acc[8 * h + 6]);
          acc[8 * h + 7] = fmaf(w, __uint_as_float(a.w & 0xffff0000u), acc[8 * h + 7]);
        }
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t w4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 hh = __floats2bfloat162_rn(acc[8 * h + 2 * e] * inv, acc[8 * h + 2 * e + 1] * inv);
      w4[e] = *reinterpret_cast<uint32_t*>(&hh);
    }
    *reinterpret_cast<uint4*>(o + 256 * h + 8 * lane) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
  if (p.lse != nullptr && lane == 0)
    p.lse[grow] = wsum > 0.f ? (mx + log2f(wsum)) * p.lse_mul : -INFINITY;
}

// unit_tiles in 32-bit arithmetic, for the combine's many blocks that only decide whether
// their unit needs them: equal to it because lengths (causal_seqlens_global, seq_lens)
// are below 2^31 and so is cp * interleave (both checked on the host).
__device__ __forceinline__ int unit_tiles32(const Params& p, int u) {
  const int b = u / p.row_tiles, rt = u % p.row_tiles;
  const int last_row = min((rt + 1) * kM, p.rows) - 1;
  const int sh = shard_of(p, b);
  const int cap = seq_cap(p, b);
  int keys = cap;
  if (p.causal) {
    const int g = __ldg(p.gseq + (b - sh * p.shard_B));
    const int i = last_row / p.H;
    const long long gi64 = (long long)g - (p.q_len - 1 - i);
    const unsigned int gi = gi64 < 0 ? 0u : (unsigned int)gi64;
    const unsigned int span = (unsigned int)p.span;
    const unsigned int q = gi / span;
    long long rem = (long long)(gi - q * span) - (long long)(p.rank + sh) * p.il;
    rem = rem < 0 ? 0 : (rem > p.il ? p.il : rem);
    const long long loc = (long long)q * p.il + rem;
    keys = (int)(loc < cap ? loc : cap);
  }
  return (keys + kTile - 1) / kTile;
}

__global__ void __launch_bounds__(256) mla_tc_combine_kernel(const Params p) {
  __shared__ int s_nt;
  __shared__ int2 s_m;
  // launched as a dependent of the decode kernel: every block waits for it here, before any
  // access to memory (so this grid also completes only after the decode kernel)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int u = blockIdx.x >> 4, rb = blockIdx.x & 15;      // 16 blocks of 8 rows per unit
  const int b = u / p.row_tiles, rt = u % p.row_tiles;
  if (threadIdx.x == 0) {
    if (rt == 0 && rb == 0 && __ldg(p.seq_lens + b) > p.max_blocks * p.bs)
      atomicOr(p.status, MLA_STATUS_SEQ_TOO_LONG);
    const int nt = unit_tiles32(p, u);
    int2 m = make_int2(0, 0);
    if (nt > 0 && !p.whole_units) {
      m = p.meta[u];                          // first and last group holding the unit
      // kept inside [0, groups) whatever the workspace holds (a decode that gave up early
      // may not have written it), so that every read stays inside the workspace
      m.x = min(max(m.x, 0), p.groups - 1);
      m.y = min(max(m.y, m.x), p.groups - 1);
    }
    s_nt = nt;
    s_m = m;
  }
  __syncthreads();
  const int nt = s_nt;
  const int2 m = s_m;
  // one cluster wrote the final result (or there is no workspace): nothing to do
  if (nt > 0 && (p.whole_units || m.x == m.y)) return;
  const int r = rb * 8 + (threadIdx.x >> 5);
  if (rt * kM + r >= p.rows) return;
  combine_row(p, b, rt, r, threadIdx.x & 31, nt, m);
}

PFN_cuTensorMapEncodeTiled_v12000 lookup_encoder() {
  cudaDriverEntryPointQueryResult q;
  void* f = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  return nullptr;
}

// Looked up once per process (a function-local static is initialised exactly once, also
// when several host threads make their first call at the same time).
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = lookup_encoder();
  return fn;
}

size_t tc_ws_bytes(int units, int clusters) {
  const size_t slots = (size_t)units + clusters;
  size_t b = 256;                                        // header
  b += ((size_t)units * sizeof(int2) + 255) / 256 * 256;
  b += (slots * kM * sizeof(float) + 255) / 256 * 256;
  b += slots * kM * kDv * sizeof(uint16_t);
  return b;
}

int tc_clusters(int num_sms) { return num_sms / 2 > 0 ? num_sms / 2 : 1; }

}  // namespace

bool tc_block_size_ok(int bs) {
  // a 64-key tile is 64 / bs whole pages (bs 16, 32) or part of one page (bs a multiple
  // of 64); one TMA box never crosses a page
  return bs == 16 || bs == 32 || (bs >= 64 && bs % 64 == 0);
}

bool tc_supported(const DecodeArgs& a) {
  const int bs = a.block_size;
  // every row tile of a request needs a cluster of its own (clusters = SMs / 2)
  if ((a.H * a.q_len + kM - 1) / kM > a.num_sms / 2) return false;
  if (!tc_block_size_ok(bs)) return false;
  if ((long long)a.num_blocks * bs + 64 >= (1LL << 31)) return false;
  if (reinterpret_cast<uintptr_t>(a.kv) % 16 != 0) return false;
  return get_encoder() != nullptr;
}

size_t tc_workspace_size(int B, int H, int q_len, int num_sms) {
  const int rt = (H * q_len + kM - 1) / kM;
  return tc_ws_bytes(B * rt, tc_clusters(num_sms));
}

namespace {

// Per-device set-up of the decode kernels, done once per device: the shared-memory
// attribute of both budget instantiations and the number of clusters that can be
// resident at once (the same for both: same block size and shared memory).
struct TcDevice {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  int active_clusters = 0;
};
constexpr int kMaxDevices = 64;
TcDevice g_tc_dev[kMaxDevices];

void tc_device_setup(TcDevice& d, int clusters_wanted) {
  d.err = cudaFuncSetAttribute(mla_decode_tc_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (d.err == cudaSuccess)
    d.err = cudaFuncSetAttribute(mla_decode_tc_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (d.err != cudaSuccess) return;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters_wanted);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, mla_decode_tc_kernel<false>, &cfg) == cudaSuccess &&
      active > 0)
    d.active_clusters = active;
  cudaGetLastError();
}

}  // namespace

namespace {
std::atomic<int> g_budget_choice{0};   // 0 automatic, 1 narrow, 2 wide
}

void set_rescale_budget_choice(int choice) { g_budget_choice.store(choice); }

bool tc_wide_budget(const DecodeArgs& a) {
  const int choice = g_budget_choice.load();
  if (choice != 0) return choice == 2;
  // the running max climbs past the narrow budget mostly over long contexts (the largest
  // of n scores keeps growing with n); the table spans max_blocks * block_size keys of
  // each shard, cp_world times that globally
  return (long long)a.max_blocks * a.block_size * a.cp_world >= (1LL << 18);
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  Params p;
  p.q = a.q;
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.seq_lens = a.seq_lens;
  p.gseq = a.gseq;
  p.B = a.B;
  p.shard_B = a.shard_B;
  // floor(b * ceil(2^32 / d) / 2^32) = floor(b / d) while b * d < 2^32, which the entry
  // point checks for several shards (b < n * d); one shard is shard 0 throughout
  p.shard_mul = a.shard_B == a.B
                    ? 0u
                    : (unsigned)((0x100000000ull + (unsigned long long)a.shard_B - 1) /
                                 (unsigned long long)a.shard_B);
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
  p.wait_ns = a.wait_ns;
  p.stall_test = a.stall_test;
  p.rows = a.H * a.q_len;
  p.row_tiles = (p.rows + kM - 1) / kM;
  p.units = a.B * p.row_tiles;
  p.box_rows = a.block_size < 64 ? a.block_size : 64;
  p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) % 32 == 0) ? 1 : 0;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.lse_mul = a.lse_base_e ? 0.6931471805599453f : 1.0f;
  p.out = a.out;
  p.lse = a.lse;
  p.status = a.status;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int C = tc_clusters(a.num_sms);
  TcDevice& td = g_tc_dev[dev];
  std::call_once(td.once, tc_device_setup, std::ref(td), C);
  if (td.err != cudaSuccess) return td.err;
  if (td.active_clusters > 0 && td.active_clusters < C) C = td.active_clusters;
  // whole groups of row_tiles clusters (row_tiles <= C is checked by tc_supported)
  p.groups = C / p.row_tiles;
  C = p.groups * p.row_tiles;
  p.clusters = C;
  // starting a segment (the output tile drained and written, the next unit's Q loaded, the
  // key ring refilled) takes about as long as 6 tiles: 4-7 us against ~1 us a tile (GB300)
  p.seg_tiles = 6;
  const size_t need = tc_ws_bytes(p.units, C);
  if (a.workspace != nullptr && a.workspace_bytes >= need) {
    char* ws = static_cast<char*>(a.workspace);
    const size_t slots = (size_t)p.units + C;
    p.hdr = reinterpret_cast<long long*>(ws);
    ws += 256;
    p.meta = reinterpret_cast<int2*>(ws);
    ws += ((size_t)p.units * sizeof(int2) + 255) / 256 * 256;
    p.ws_lse = reinterpret_cast<float*>(ws);
    ws += (slots * kM * sizeof(float) + 255) / 256 * 256;
    p.ws_o = reinterpret_cast<uint16_t*>(ws);
    p.whole_units = 0;
  } else {
    p.hdr = nullptr;
    p.meta = nullptr;
    p.ws_lse = nullptr;
    p.ws_o = nullptr;
    p.whole_units = 1;
    if (p.groups > p.B) p.groups = p.B;
    C = p.groups * p.row_tiles;
    p.clusters = C;
  }

  // The cache seen as [rows][9 chunks][64 dims]: dims 64 elements (contiguous), rows
  // (stride 1152 bytes), chunks (stride 128 bytes).  One box takes box_rows keys of
  // kz (vz) consecutive chunks and lands as [chunk][key][128 bytes], 128-byte swizzled,
  // which is the MMA operand layout of each chunk.
  CUtensorMap kmap, vmap;
  {
    p.kz = p.box_rows == 64 ? kKGroup : 1;
    p.vz = p.box_rows == 64 ? 4 : 1;
    cuuint64_t dims[3] = {64, (cuuint64_t)a.num_blocks * a.block_size, (cuuint64_t)kKChunks};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, 128};
    cuuint32_t es[3] = {1, 1, 1};
    cuuint32_t kbox[3] = {64, (cuuint32_t)p.box_rows, (cuuint32_t)p.kz};
    cuuint32_t vbox[3] = {64, (cuuint32_t)p.box_rows, (cuuint32_t)p.vz};
    CUresult r = get_encoder()(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                               const_cast<uint16_t*>(a.kv), dims, strides, kbox, es,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    r = get_encoder()(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.kv),
                      dims, strides, vbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // Q as [B * q_len * H rows][576]: a unit's 128 rows of one 64-dim chunk per box (rows
  // past the tensor read as zeros; rows of the next request in a partial unit are loaded
  // but belong to rows the unit never stores)
  CUtensorMap qmap;
  {
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)a.shard_B * p.rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kM};
    cuuint32_t es[2] = {1, 1};
    CUresult r = get_encoder()(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                               const_cast<uint16_t*>(a.q), dims, strides, box, es,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  if (tc_wide_budget(a))
    mla_decode_tc_kernel<true><<<2 * C, kThreads, kSmemBytes, stream>>>(kmap, vmap, qmap, p);
  else
    mla_decode_tc_kernel<false><<<2 * C, kThreads, kSmemBytes, stream>>>(kmap, vmap, qmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  DependentLaunch dl(dim3((unsigned)p.units * 16u), dim3(256), stream);
  return cudaLaunchKernelEx(&dl.cfg, mla_tc_combine_kernel, p);
}

}  // namespace mla
