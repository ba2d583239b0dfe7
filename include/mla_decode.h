/*
 * mla_decode.h -- C ABI of libmla_decode.so: paged multi-head-latent-attention (MLA)
 * decode with decode-context-parallel (DCP) shards, the LSE merge of shard partials,
 * and DCP slot mapping, for NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages summarising vLLM pull requests):
 *   [#52188] "支持 Kimi-K3 DSpark 推测解码与 DCP 并行组合" (vLLM PR 52188)
 *   [#54012] "带 DCP 的 MLA decode 改用 FlashInfer 原生 CP mask" (vLLM PR 54012)
 *   [#48180] "为 TokenSpeed MLA 后端添加 DCP 与 Eagle 支持" (vLLM PR 48180)
 *
 * Conventions shared by every call:
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless stated.
 *     The library allocates no memory when called.  Its device state is one status word
 *     per device (see mla_get_device_status) and the fixed scratch array that
 *     mla_decode_noalloc uses; its host state is per-device launch settings, filled on
 *     a device's first call.
 *   - Every call is asynchronous on `stream` (the legacy default stream when NULL) and
 *     returns one of the MLA_* codes.  Argument errors are found on the host before
 *     anything is launched; mla_last_error() then returns a message (thread-local).
 *   - Calls are stream-ordered: a call's kernels see every result issued before it on
 *     the stream.  The split-KV combine of mla_decode and the kernel of lse_merge are
 *     programmatic dependent launches: they may be scheduled while the kernel before
 *     them drains, but wait for its completion before they read or write memory.
 *   - bf16 means IEEE bfloat16 stored as 16-bit words; results are rounded to nearest
 *     even.  Tensors are dense and row-major unless a stride is given.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, without pulling in the CUDA headers. */
typedef struct CUstream_st* mla_stream_t;

#define MLA_OK 0
#define MLA_ERR_INVALID_ARGUMENT (-1) /* null pointer, bad size, range or alignment    */
#define MLA_ERR_UNSUPPORTED (-2)      /* valid request this build does not implement   */
#define MLA_ERR_CUDA (-3)             /* a CUDA runtime call or kernel launch failed    */
#define MLA_ERR_DEVICE (-4)           /* a kernel flagged bad data (see status word)    */

#define MLA_PAD_SLOT_ID (-1)   /* slot of a position this rank does not own            */
#define MLA_HEAD_DIM_QK 576    /* 512 latent (kv_lora_rank) + 64 rope dims            */
#define MLA_HEAD_DIM_V 512     /* V is the first 512 dims of each latent KV row        */
#define MLA_MAX_Q_LEN 16

/* Bits of the device status word. */
#define MLA_STATUS_BAD_PAGE 1u        /* block_table entry outside [0, num_blocks)      */
#define MLA_STATUS_SEQ_TOO_LONG 2u    /* seq_lens[b] > max_blocks * block_size          */
#define MLA_STATUS_BAD_VBLOCK 4u      /* cp_local_slot: virtual block >= max_blocks     */
#define MLA_STATUS_WAIT_TIMEOUT 8u    /* a bounded on-chip wait gave up                 */

/*
 * Bytes of workspace that mla_decode uses to split one request's KV range over several
 * thread blocks (split-KV) for a batch of B requests, H query heads, q_len query rows
 * and a device with num_sms SMs.  Passing less (or NULL) is allowed: the call then uses
 * fewer splits, down to none.  Pure function of its arguments; no CUDA call.
 */
size_t mla_decode_workspace_size(int B, int H, int q_len, int num_sms);

/*
 * mla_decode -- one shard's partial attention for a batch of multi-token decode blocks.
 *
 * Defines ([#54012] "关键源码片段", the native-DCP call; [#52188] "关键源码片段",
 * _prepare_flattened_decode_metadata; [#48180] "实现拆解" step 1):
 *   global position g lives on rank (g / interleave) % cp_world (round-robin segments of
 *   `interleave` positions); with span = cp_world * interleave a global prefix of G
 *   positions holds local_len(G) = G / span * interleave
 *                                  + clamp(G % span - cp_rank * interleave, 0, interleave)
 *   of this shard's keys.  causal != 0: query row i (0 <= i < q_len) of request b sees the
 *   global prefix G_i = max(0, causal_seqlens_global[b] - (q_len - 1 - i)), i.e.
 *       L_i = min(seq_lens[b], local_len(G_i))
 *   local keys; causal == 0 (a non-causal draft block, the snippet's other branch): every
 *   row reads the shard's whole local sequence, L_i = seq_lens[b].  The local key l < L_i
 *   is row kv_cache[block_table[b*bt_stride + l/block_size]][l % block_size].  With
 *   s_l = scale * <q_row, key_l> over all 576 dims,
 *       out = sum_l softmax(s)_l * key_l[0:512],   lse = log(sum_l exp(s_l)),
 *   lse in natural log when lse_base_e != 0, else in log2.  A row with L_i = 0 gets
 *   out = 0 and lse = -inf.
 *
 * Arguments:
 *   q            bf16 [B, q_len, H, 576], 16-byte aligned.
 *   kv_cache     bf16 [num_blocks, block_size, 576] (this shard's pool), 16-byte aligned;
 *                block_size 16, 32 or a multiple of 64.
 *   block_table  int32 [B, bt_stride]; only the first ceil(L/block_size) entries of a
 *                row are read.  An entry outside [0, num_blocks) is not dereferenced:
 *                its keys are read as zeros and MLA_STATUS_BAD_PAGE is set.
 *   seq_lens     int32 [B], this shard's token count of each request.  A value above
 *                max_blocks*block_size is clamped and MLA_STATUS_SEQ_TOO_LONG is set.
 *   causal_seqlens_global  int32 [B] global lengths; may be NULL when cp_world == 1 (then
 *                seq_lens is used) or causal == 0 (then it is not read).
 *   B >= 0, 1 <= H, 1 <= q_len <= MLA_MAX_Q_LEN, ceil(q_len*H/128) <= SMs/2,
 *   num_blocks >= 1, 1 <= max_blocks <= bt_stride, 1 <= cp_world, 0 <= cp_rank <
 *   cp_world, interleave >= 1 dividing block_size (the pool layout cp_local_slot gives),
 *   finite scale > 0.
 *   out          bf16 [B*q_len, H, 512], 16-byte aligned.
 *   lse          float [B*q_len, H] or NULL.
 *   workspace    device scratch of workspace_bytes (may be NULL / 0), 256-byte aligned.
 * Errors: MLA_ERR_INVALID_ARGUMENT for any violated condition above (nothing launched),
 *   MLA_ERR_UNSUPPORTED for a block size or row count the kernel does not take,
 *   MLA_ERR_CUDA if a launch fails.
 */
int mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
               int64_t bt_stride, const int32_t* seq_lens,
               const int32_t* causal_seqlens_global, int B, int H, int q_len, int causal,
               int block_size, int num_blocks, int max_blocks, int cp_world, int cp_rank,
               int interleave, float scale, void* out, float* lse, int lse_base_e,
               void* workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * mla_decode_shards -- every shard of one emulated context-parallel decode step in a
 * single launch (the ranks of the pages' native DCP decode, [#54012] "关键源码片段",
 * run side by side on one GPU instead of one per GPU).  The result is exactly that of
 *     for r in 0 .. n_shards-1:
 *         mla_decode(q, kv_cache, block_table + r*B*bt_stride, bt_stride, seq_lens + r*B,
 *                    causal_seqlens_global, B, H, q_len, causal, block_size, num_blocks,
 *                    max_blocks, n_shards, r, interleave, scale,
 *                    out + r*B*q_len*H*512, lse ? lse + r*B*q_len*H : NULL, lse_base_e, ...)
 * with all shards' pages in one cache.
 *
 * Arguments (as mla_decode unless stated):
 *   kv_cache     bf16 [num_blocks, block_size, 576]: the pages of every shard.
 *   block_table  int32 [n_shards*B, bt_stride], shard-major: row r*B + b holds shard r's
 *                page ids (into kv_cache) for request b.
 *   seq_lens     int32 [n_shards*B], shard-major token counts.
 *   causal_seqlens_global  int32 [B]; may be NULL only if n_shards == 1 or causal == 0.
 *   n_shards     >= 1; shard r is rank r of cp_world = n_shards.
 *   out          bf16 [n_shards, B*q_len, H, 512];  lse  float [n_shards, B*q_len, H] or NULL.
 *   workspace    sized by mla_decode_workspace_size(n_shards*B, H, q_len, num_sms).
 * Errors: as mla_decode; also MLA_ERR_INVALID_ARGUMENT for n_shards < 1 and
 *   MLA_ERR_UNSUPPORTED when n_shards > 1 and n_shards * B * B >= 2^32.
 */
int mla_decode_shards(const void* q, const void* kv_cache, const int32_t* block_table,
                      int64_t bt_stride, const int32_t* seq_lens,
                      const int32_t* causal_seqlens_global, int B, int H, int q_len,
                      int causal, int block_size, int num_blocks, int max_blocks, int n_shards,
                      int interleave, float scale, void* out, float* lse, int lse_base_e,
                      void* workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * lse_merge -- combine n_shards partial results of the same rows through their LSEs.
 *
 * Defines ([#54012] "实现拆解" step 3: shards are merged across ranks and must agree on
 * the LSE base; [#48180] "实现拆解" step 2: merge when DCP is on): per row (t, h),
 *   M = max_s lses[s,t,h],  w_s = base^(lses[s,t,h] - M),
 *   out[t,h,:] = sum_s w_s partials[s,t,h,:] / sum_s w_s,
 *   out_lse[t,h] = M + log_base(sum_s w_s),
 * base e when lse_base_e != 0, else 2.  A shard with lse = -inf has weight 0 and its
 * partial is not read; if every shard has -inf, out = 0 and out_lse = -inf.
 *
 * Arguments:
 *   partials        [n_shards, T, H, 512], bf16 when partials_fp32 == 0 else float,
 *                   16-byte aligned.
 *   lses            float [n_shards, T, H].
 *   n_shards >= 1, T >= 0, H >= 1.
 *   out             bf16 [T, H, 512], 16-byte aligned.
 *   out_lse         float [T, H] or NULL.
 * Errors: MLA_ERR_INVALID_ARGUMENT, MLA_ERR_CUDA.
 */
int lse_merge(const void* partials, int partials_fp32, const float* lses, int n_shards,
              int T, int H, void* out, float* out_lse, int lse_base_e,
              mla_stream_t stream);

/*
 * cp_local_slot -- this rank's KV slot of each position, MLA_PAD_SLOT_ID otherwise.
 *
 * Defines ([#52188] "关键源码片段", cp_utils.py cp_local_slot; "实现拆解" step 4): a
 * virtual block spans block_size*cp_size global positions and block_table[b, pos /
 * (block_size*cp_size)] names its page on every rank; with o = pos % (block_size*cp_size),
 * position pos is owned by rank (o / interleave) % cp_size, at local offset
 * (o / (interleave*cp_size)) * interleave + o % interleave, so
 *     slots[b,n] = page * block_size + local offset   if this rank owns it,
 *     slots[b,n] = MLA_PAD_SLOT_ID                     otherwise, or when pos < 0
 * (a negative position marks a rejected draft position).  cp_size == 1 gives
 * page * block_size + pos % block_size.
 *
 * Arguments:
 *   positions    int64 [B, N];  block_table int32 [B, bt_stride] with max_blocks valid
 *                columns;  slots int64 [B, N].
 *   B >= 0, N >= 0, block_size >= 1, cp_size >= 1, 0 <= cp_rank < cp_size,
 *   interleave >= 1 with block_size % interleave == 0, 1 <= max_blocks <= bt_stride.
 * A position whose virtual block is >= max_blocks gets MLA_PAD_SLOT_ID and sets
 * MLA_STATUS_BAD_VBLOCK; its table entry is not read.
 * Errors: MLA_ERR_INVALID_ARGUMENT, MLA_ERR_CUDA.
 */
int cp_local_slot(const int64_t* positions, const int32_t* block_table, int64_t bt_stride,
                  int max_blocks, int B, int N, int block_size, int cp_size, int cp_rank,
                  int interleave, int64_t* slots, mla_stream_t stream);

/*
 * cp_local_slot_scatter -- writes new KV rows into this rank's pool at the slots
 * cp_local_slot gives them.
 *
 * Defines ([#52188] "实现拆解" step 4: the draft inputs apply cp_local_slot to the slots
 * they write, with the page of a position taken from block_table[pos / (block_size *
 * cp_size)], so that a rank never writes a slot another rank is responsible for): for
 * every (b, n) with s = cp_local_slot(positions[b, n]) != MLA_PAD_SLOT_ID,
 *     kv_cache[s] = kv_new[b, n]          (576 bf16, copied bit for bit);
 * positions this rank does not own, and negative (rejected) positions, write nothing and
 * their rows are not read.
 *
 * Arguments (as cp_local_slot unless stated):
 *   kv_new       bf16 [B, N, 576], 16-byte aligned.
 *   kv_cache     bf16 [num_blocks, block_size, 576] (this rank's pool), 16-byte aligned.
 *   slots        int64 [B, N] or NULL: receives the slots, as cp_local_slot returns them.
 * A slot outside the cache (a table entry outside [0, num_blocks)) is not written and
 * sets MLA_STATUS_BAD_PAGE; a virtual block past the table sets MLA_STATUS_BAD_VBLOCK.
 * Two positions mapping to the same slot race (the pages' slot mapping never does that
 * for distinct positions of one request).
 * Errors: MLA_ERR_INVALID_ARGUMENT, MLA_ERR_UNSUPPORTED (B*N or block_size*cp_size beyond
 *   2^31-1), MLA_ERR_CUDA.
 */
int cp_local_slot_scatter(const int64_t* positions, const void* kv_new,
                          const int32_t* block_table, int64_t bt_stride, int max_blocks, int B,
                          int N, int block_size, int cp_size, int cp_rank, int interleave,
                          void* kv_cache, int num_blocks, int64_t* slots, mla_stream_t stream);

/*
 * mla_decode_noalloc -- mla_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call.  It computes exactly what mla_decode
 * computes, with the same arguments minus the workspace: some callers cannot call
 * cudaMalloc or any allocating routine on their decode path (a runtime whose memory is
 * planned once at start-up, a host program that links only this C library and owns no
 * allocator), yet split-KV needs scratch for its per-split partial results.  This call
 * takes that scratch from one fixed 64 MiB array that the library declares in device
 * memory; every GPU that loads the library holds the array until the process exits.
 *   - A problem whose split-KV scratch exceeds 64 MiB is rejected with
 *     MLA_ERR_UNSUPPORTED (message in mla_last_error) and nothing is launched; every
 *     other argument is checked first, exactly as mla_decode checks it.
 *   - All calls on a device share the array and it keeps the last call's contents;
 *     calls whose kernels overlap on the GPU (other streams or host threads) race on it
 *     and must be serialised.  Nothing in it needs to start at zero.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 * Errors: as mla_decode, plus MLA_ERR_UNSUPPORTED for the size limit.
 */
int mla_decode_noalloc(const void* q, const void* kv_cache, const int32_t* block_table,
                       int64_t bt_stride, const int32_t* seq_lens,
                       const int32_t* causal_seqlens_global, int B, int H, int q_len,
                       int causal, int block_size, int num_blocks, int max_blocks,
                       int cp_world, int cp_rank, int interleave, float scale, void* out,
                       float* lse, int lse_base_e, mla_stream_t stream);

/*
 * Waits for `stream`, then reads and clears the current device's status word.
 * Returns MLA_OK when no kernel flagged anything since the last call, MLA_ERR_DEVICE
 * when one did (mla_last_error() names the bits; *bits_out receives them if non-NULL),
 * MLA_ERR_CUDA if the read itself failed.
 */
int mla_get_device_status(mla_stream_t stream, uint32_t* bits_out);

/*
 * Selects the decode kernel for later mla_decode calls in this process (diagnostics and
 * tests): 0 = automatic (the tcgen05/TMEM/TMA kernel; a layout it does not take is
 * refused with MLA_ERR_UNSUPPORTED), 1 = the warp-level mma.sync kernel (any block size;
 * a second, independent implementation that tests compare with the first), 2 = the
 * tcgen05 kernel.  Returns the previous choice, or MLA_ERR_INVALID_ARGUMENT for any other
 * value.  Not to be changed while other threads call mla_decode.
 */
int mla_set_decode_kernel(int choice);

/*
 * Selects the lazy-rescale budget of the tcgen05 kernel's online softmax for later calls
 * (diagnostics and tests): 0 = chosen per call (the wide budget when max_blocks *
 * block_size * cp_world >= 2^18, i.e. for long contexts), 1 = narrow, 2 = wide.  Both
 * compute the same result; they differ in how often the accumulator is rescaled.
 * Returns the previous choice, or MLA_ERR_INVALID_ARGUMENT for any other value.
 */
int mla_set_rescale_budget(int choice);

/*
 * Sets the time limit of every bounded on-chip wait of later launches, in nanoseconds
 * (0 = the default, 2 s); returns the previous setting (0 = default), or
 * MLA_ERR_INVALID_ARGUMENT for ns < 0.  A wait that runs out makes the kernel stop every
 * role of its thread-block pair, let the copies in flight land, release its tensor
 * memory and return; mla_get_device_status then reports MLA_STATUS_WAIT_TIMEOUT and the
 * outputs of that call are undefined.  Tests use a tiny limit to exercise that path.
 */
int64_t mla_set_wait_limit_ns(int64_t ns);

/*
 * Tests of the timeout path only: with on = 1, later launches of the tcgen05 decode kernel
 * make one role of every thread-block pair first wait for an mbarrier arrival that never
 * comes, so that the wait runs out after the limit of mla_set_wait_limit_ns, the kernel
 * stops and returns (outputs undefined) and mla_get_device_status reports
 * MLA_STATUS_WAIT_TIMEOUT.  on = 0 (the default) turns it off.  Returns the previous
 * setting, or MLA_ERR_INVALID_ARGUMENT.
 */
int mla_set_test_stall(int on);

/* Message of the calling thread's last failed call (empty string if none). */
const char* mla_last_error(void);

/* ABI version of this library: (major << 16) | minor (2.0). */
int mla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
