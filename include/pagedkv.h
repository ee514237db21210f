/*
 * pagedkv.h -- C ABI of libpagedkv: chunk-wise paged self-attention over a
 * block-paged KV pool, for one NVIDIA GB300 (sm_103a).
 *
 * The operations follow the vllm-omni pages:
 *   - paged_attention.py (vllm_omni/experimental/ar_diffusion/kv_cache):
 *       _paged_write_attn_impl        -> paged_kv_write
 *       ar_diffusion_paged_attention  -> paged_attn_varlen (no segments)
 *       _reference_paged_attention    -> the block-table addressing
 *       video_block_table, build_block_table, max_video_blocks
 *                                     -> pkv_visible_window, pkv_block_table_row,
 *                                        pkv_table_width
 *   - piecewise_attn.py (vllm_omni/diffusion/attention/backends/utils):
 *       build_segments                -> build_segments
 *       piecewise_attn / module doc   -> the segment mask of paged_attn_varlen
 *       build_paged_piecewise_plan    -> span validation rules; one query offset per packed row
 *   - paged_attention_adapter.py (vllm_omni/diffusion/diffusion_kv):
 *       head divisibility and query-is-a-suffix rules.
 *
 * Conventions
 *   - Tensor pointers are DEVICE memory owned by the caller unless a comment
 *     says "host".  The library never allocates device memory: scratch space
 *     for split-KV comes from a caller-supplied workspace.
 *   - Every device call is asynchronous on the caller's stream (`stream` is a
 *     cudaStream_t passed as void*; NULL = the legacy default stream) and
 *     returns a pkv_status.  Host-checkable preconditions are validated before
 *     anything is launched; on failure nothing is launched.
 *   - pkv_last_error() returns a thread-local message for the last failure.
 *   - Device-resident metadata (slots, block table, query_start_loc,
 *     seq_lens, segments) is trusted unless PKV_CHECK_BOUNDS is set in
 *     `flags`: then kernels check every index they are about to use, skip the
 *     access when it is out of range, and raise a device error word that
 *     pkv_check() reads back.  Kernels never trap.
 *   - Layouts are row-major and contiguous:
 *       pool        [num_blocks * block_size, Hkv, D]  (== [num_blocks, block_size, Hkv, D])
 *       q, out      [Tq, Hq, D]   packed by query_start_loc
 *       k, v (new)  [T, Hkv, D]
 *       block_table [B, W] int32
 *   - Block size is 16 tokens.  Head dim D is 64 or 128.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,  /* bad pointer, size, layout or metadata seen on the host */
  PKV_ERR_UNSUPPORTED = 2,  /* dtype, head dim or block size the library does not handle */
  PKV_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  PKV_ERR_DEVICE_CHECK = 4, /* a kernel in PKV_CHECK_BOUNDS mode saw bad metadata */
  PKV_ERR_CAPACITY = 5      /* an output buffer or workspace is too small */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_F16 = 2 } pkv_dtype;

/* Flags for the device calls. */
#define PKV_CHECK_BOUNDS 0x1u  /* validate device metadata in the kernels */
#define PKV_FORCE_SIMT 0x2u    /* attention: use the CUDA-core kernel even for bf16/f16 */
#define PKV_NO_SPLIT 0x4u      /* attention: never split the key range */
/* attention: every row's block-table entries are consecutive (entry i = entry 0 + i), e.g. K/V staged by
 * paged_kv_gather; the tensor-core kernel then loads a whole 128-key tile per TMA box instead of one box per
 * 16-token block.  With PKV_CHECK_BOUNDS a row that breaks the promise is flagged (PKV_DEVERR_BLOCK) and
 * loaded block by block. */
#define PKV_CONTIGUOUS_KV 0x8u
/* attention: force n key-range splits (needs workspace); n > 16 is taken as 16; 0 = plan automatically */
#define PKV_SPLITS(n) ((((uint32_t)(n)) & 0xffu) << 8)

/* Segment modes. */
#define PKV_SEG_CAUSAL 0
#define PKV_SEG_FULL 1

/* Device error word bits reported by pkv_check(). */
#define PKV_DEVERR_SLOT 0x1u      /* a slot outside [0, num_slots) (negative slots are skips, not errors) */
#define PKV_DEVERR_BLOCK 0x2u     /* a block id outside [0, num_blocks) */
#define PKV_DEVERR_SEQLEN 0x4u    /* seq_lens[b] > W * block_size or > max_seq_len, or Sq > seq_len */
#define PKV_DEVERR_QUERY 0x8u     /* query_start_loc not monotone, or Sq > max_query_len */
#define PKV_DEVERR_SEGMENT 0x10u  /* a segment outside the row's query range, or a query row no segment covers */
#define PKV_DEVERR_TIMEOUT 0x20u  /* a pipeline wait inside a kernel gave up (the kernel unwound; results invalid) */

/*
 * One piece of a piecewise causal/full mask, in GLOBAL key coordinates
 * (piecewise_attn.py, Segment / build_segments):
 *   queries at global positions [q_start, q_end) attend keys [0, kv_end);
 *   mode PKV_SEG_FULL:   every one of those keys;
 *   mode PKV_SEG_CAUSAL: bottom-right aligned -- the query at position p sees
 *                        key j when j <= kv_end - (q_end - p).  With
 *                        kv_end == q_end (what build_segments emits) that is j <= p.
 */
typedef struct {
  int32_t q_start, q_end, kv_end, mode;
} pkv_segment;

/* Thread-local text of the last failure on this thread ("" if none). Never NULL. */
PKV_API const char* pkv_last_error(void);

/* Library version string. */
PKV_API const char* pkv_version(void);

/* ------------------------------------------------------------------------
 * Host metadata (run once per forward; shared by every layer)
 * ------------------------------------------------------------------------ */

/*
 * build_segments -- piecewise_attn.py, build_segments; validation as in
 * build_paged_piecewise_plan.
 *   spans        host, [n_spans][2] (start, end) half-open, global coordinates
 *   query_offset first global position of the query; query_len > 0 queries
 *   seq_len      key length of the row (spans must end at or before it)
 *   out          host, room for `capacity` segments (2 * n_spans + 1 always suffices)
 *   n_out        host, number written
 * Errors: PKV_ERR_INVALID_ARG for unsorted/overlapping spans, start >= end,
 * start < 0, end > seq_len, query_offset < 0, query_len <= 0,
 * query_offset + query_len > seq_len, or NULL pointers; PKV_ERR_CAPACITY if
 * `capacity` is too small.  Output is bit-exact with the definition.
 */
PKV_API pkv_status build_segments(const int32_t* spans, int n_spans, int32_t query_offset, int32_t query_len,
                          int32_t seq_len, pkv_segment* out, int capacity, int* n_out);

/*
 * pkv_slot_mapping -- the slot of each token: blocks[p / bs] * bs + p % bs
 * for p = first_position + t, t < n_tokens (the addressing of
 * paged_attention.py, _reference_paged_attention; the scratch chunk of
 * ensure_video_slots starts mid-block at first_position % bs).
 *   blocks        host, physical block of each logical block (index = p / bs)
 *   slots         host, out [n_tokens] int64
 * Errors: PKV_ERR_INVALID_ARG if a position's logical block is >= n_blocks,
 * or a block id is negative.
 */
PKV_API pkv_status pkv_slot_mapping(const int32_t* blocks, int64_t n_blocks, int64_t first_position, int64_t n_tokens,
                            int block_size, int64_t* slots);

/*
 * pkv_table_width -- fixed block-table width (paged_attention.py,
 * max_video_blocks docstring and build_block_table):
 *   ceil(sink / bs) + ceil((window + bs - gcd(chunk, bs)) / bs) + max(1, ceil(action_len / bs)).
 * Returns the width, or -1 on invalid input (see pkv_last_error()).
 */
PKV_API int64_t pkv_table_width(int64_t chunk_tokens, int64_t sink_tokens, int64_t window_tokens, int64_t action_len,
                        int block_size);

/*
 * pkv_visible_window -- blocks attention reads and how many of their slots hold
 * tokens (paged_attention.py, video_block_table): the sink [0, sink_tokens)
 * and the last window_tokens positions before end_tokens (current chunk
 * included), chosen by the positions each block holds; blocks lying wholly
 * between the two ranges are skipped, evicted blocks (id < 0) are skipped.
 *   row_blocks   host, physical block of logical block i (positions i*bs ..), or -1 if evicted;
 *                must cover ceil(end_tokens / bs) entries
 *   out_blocks   host, room for `capacity` ids; n_out and video_len are host outputs
 * Errors: PKV_ERR_INVALID_ARG (NULL, too few row_blocks, negative sizes),
 * PKV_ERR_CAPACITY, and PKV_ERR_INVALID_ARG if a partly written block would be
 * followed by another listed block.
 */
PKV_API pkv_status pkv_visible_window(const int32_t* row_blocks, int64_t n_row_blocks, int64_t end_tokens,
                              int64_t sink_tokens, int64_t window_tokens, int block_size, int32_t* out_blocks,
                              int64_t capacity, int64_t* n_out, int64_t* video_len);

/*
 * pkv_block_table_row -- one padded table row (paged_attention.py,
 * build_block_table): video blocks, then ceil(action_len / bs) action blocks,
 * then block 0 up to `width` entries.  *kv_len = video_len + action_len.
 * Errors: PKV_ERR_INVALID_ARG when action tokens would follow a partly
 * written video block (video_len % bs != 0) or nothing would be listed;
 * PKV_ERR_CAPACITY when the blocks do not fit `width`.
 */
PKV_API pkv_status pkv_block_table_row(const int32_t* video_blocks, int64_t n_video, int64_t video_len,
                               const int32_t* action_blocks, int64_t action_len, int block_size, int64_t width,
                               int32_t* out_row, int64_t* kv_len);

/* ------------------------------------------------------------------------
 * Device operations
 * ------------------------------------------------------------------------ */

/*
 * paged_kv_write -- key_pool[slot[t]] = k[t], value_pool[slot[t]] = v[t] for
 * t < T (paged_attention.py, _paged_write_attn_impl).  A bit copy: pools and
 * sources share `dt`.  K and V go in one launch.
 *   k, v          device [T, Hkv, D]
 *   slot_mapping  device [T] int64; slot < 0 skips the token; slots must be
 *                 distinct (duplicate slots race; the result is then one of the writes)
 *   key_pool, value_pool  device [num_slots, Hkv, D]
 * Rows must be 16-byte aligned (Hkv * D * sizeof(dt) a multiple of 16, base
 * pointers 16-byte aligned).  T == 0 is a no-op.
 */
PKV_API pkv_status paged_kv_write(const void* k, const void* v, const int64_t* slot_mapping, int64_t T, void* key_pool,
                          void* value_pool, int64_t num_slots, int Hkv, int D, pkv_dtype dt, uint32_t flags,
                          void* stream);

/*
 * paged_kv_write_attn -- paged_kv_write followed by paged_attn_varlen, in ONE launch
 * (paged_attention.py, _paged_write_attn_impl: write the chunk's K/V into the pools, then
 * attend through the block table).  The attention of the same launch reads the keys and
 * values at the queries' own positions -- row b's keys [base_b, base_b + Sq), see
 * paged_attn_varlen -- straight from k and v, while otherwise idle warps of the same CTAs
 * scatter k and v into the pools; no CTA waits for the write.  The result equals the two
 * calls in sequence when every token lands on the slot its key position implies:
 *   slot_mapping[t] = block_table[b*W + key/16] * 16 + key % 16,  key = base_b + (t - query_start_loc[b])
 * for the row b holding token t (what pkv_slot_mapping produces for the chunk).  Check mode
 * verifies it and flags PKV_DEVERR_SLOT for a token that breaks it (that token is not written).
 * A negative slot skips the token's write, as in paged_kv_write.
 *   k, v          device [Tq, Hkv, D], dtype dt: the query tokens' keys and values
 *   slot_mapping  device int64 [Tq]
 *   everything else as paged_attn_varlen; key_pool/value_pool are written (num_blocks*16 slots).
 * Tokens of different rows must not share pool blocks.  Splits add the combine launch.
 * Empty sizes (Tq, B or max_query_len == 0) return PKV_OK without a launch: no token is
 * written either.
 */
PKV_API pkv_status paged_kv_write_attn(const void* q, const void* k, const void* v, const int64_t* slot_mapping,
                                       int64_t Tq, int Hq, void* key_pool, void* value_pool, int64_t num_blocks,
                                       int block_size, int Hkv, int D, pkv_dtype dt, const int32_t* block_table,
                                       int B, int W, const int32_t* query_start_loc, const int32_t* seq_lens,
                                       int max_query_len, int max_seq_len, float softmax_scale,
                                       const pkv_segment* segs, const int32_t* seg_start, void* out, void* workspace,
                                       size_t ws_bytes, uint32_t flags, void* stream);

/*
 * paged_kv_gather -- copy blocks [first_block, first_block + n_blocks) of every row's block table into
 * contiguous staging buffers: stage[b][first_block*16 + t] = pool[table[b*W + first_block + t/16]*16 + t%16]
 * for t < n_blocks*16, for K and V (paged_attention.py, _stage_window / the contiguous gather branch of
 * ar_diffusion_paged_attention; first_block > 0 re-gathers only the current chunk's blocks when the
 * history is already staged, as stage_first_block does there).  A bit copy; one launch for K and V.
 *   key_pool, value_pool  device [num_blocks*16, Hkv, D]
 *   block_table           device [B, W] int32
 *   stage_k, stage_v      device [B, stage_rows, Hkv, D]; needs (first_block + n_blocks) * 16 <= stage_rows
 * Errors: PKV_ERR_INVALID_ARG (sizes, alignment, first_block + n_blocks > W); with PKV_CHECK_BOUNDS block
 * ids outside [0, num_blocks) are flagged (PKV_DEVERR_BLOCK) and their rows not copied.
 */
PKV_API pkv_status paged_kv_gather(const void* key_pool, const void* value_pool, int64_t num_blocks,
                                   const int32_t* block_table, int B, int W, int first_block, int n_blocks,
                                   void* stage_k, void* stage_v, int64_t stage_rows, int Hkv, int D, pkv_dtype dt,
                                   uint32_t flags, void* stream);

/*
 * paged_attn_workspace_size -- bytes of workspace paged_attn_varlen may use
 * for a call with these sizes (split-KV partial outputs and log-sum-exps):
 * the key-range splits the call would plan for these sizes on the current
 * device (up to 16; see below), and at least 8 so that PKV_SPLITS(n <= 8)
 * fits.  Tq = total query tokens; 0 for empty sizes.  A smaller workspace
 * makes a planned split count shrink to what fits.
 *
 * Planning: each kernel runs one CTA per item (256 queries of one row and
 * head for the tensor-core kernel, 128 for the CUDA-core one).  When the items
 * fill the SMs a whole number of times plus a partial last wave, the whole
 * waves run unsplit and only the last wave's items split their key range, into
 * the count that minimises that wave's estimated time; a second, combine launch
 * merges their partials.  With fewer items than SMs every item splits.  Forced
 * splits (PKV_SPLITS) split every item.  pkv_last_split_plan reports what the
 * last call chose.
 */
PKV_API size_t paged_attn_workspace_size(int64_t Tq, int Hq, int D, int B, int max_query_len, int max_seq_len);

/*
 * paged_attn_varlen -- varlen attention read through a block table, with an
 * optional piecewise causal/full mask per row (paged_attention.py,
 * ar_diffusion_paged_attention / _reference_paged_attention;
 * piecewise_attn.py, piecewise_attn).
 *
 * Row b has Sq = query_start_loc[b+1] - query_start_loc[b] queries and
 * L = seq_lens[b] keys; key j of row b is pool row
 * block_table[b*W + j/16] * 16 + j % 16.  Local query i sits at global position
 * base_b + i: base_b is the q_start of the row's first segment when the row has
 * segments (build_segments starts its cover at the query offset, so a packed row
 * whose write span starts at kv_start_pos -- DiffusionPagedAttentionRow, with
 * build_paged_piecewise_plan taking one query offset per row -- gets base_b =
 * kv_start_pos), else the suffix convention base_b = L - Sq.  base_b + Sq <= L;
 * check mode flags a row that breaks it (PKV_DEVERR_SEGMENT).
 * Query head h reads KV head h / (Hq / Hkv).
 *   segs, seg_start  device; segments of row b are segs[seg_start[b] .. seg_start[b+1]);
 *                    segs == NULL: every query sees all L keys (the pages' causal=False).
 *                    A row with an empty segment list also sees all L keys.
 *   out              device [Tq, Hq, D], dtype dt (fp32 results rounded to nearest even)
 *   workspace        device, ws_bytes >= paged_attn_workspace_size(...) when the
 *                    call may split the key range (NULL/0 disables splitting)
 *   max_query_len    >= every row's Sq;  max_seq_len >= every L, <= W * 16
 *   softmax_scale    multiplies Q.K (the pages pass D^-0.5).  For bf16/f16 it must be > 0: the
 *                    tensor-core kernel requires it, and any other value returns PKV_ERR_UNSUPPORTED
 *                    unless flags holds PKV_FORCE_SIMT, which runs the CUDA-core kernel (any finite
 *                    scale, about 50 times slower on bf16).  fp32 takes any finite scale.
 * A query that sees no key (only possible with ill-formed segments) gets 0.
 * Tq == 0, B == 0 or max_query_len == 0: nothing to compute; PKV_OK without a launch
 * (sizes and the dtype are still validated; out is not touched).
 * The softmax statistics and both products accumulate in fp32.
 * Supported: dt in {F32, BF16, F16}; D in {64, 128}; block_size 16; Hq % Hkv == 0.
 */
PKV_API pkv_status paged_attn_varlen(const void* q, int64_t Tq, int Hq, const void* key_pool, const void* value_pool,
                             int64_t num_blocks, int block_size, int Hkv, int D, pkv_dtype dt,
                             const int32_t* block_table, int B, int W, const int32_t* query_start_loc,
                             const int32_t* seq_lens, int max_query_len, int max_seq_len, float softmax_scale,
                             const pkv_segment* segs, const int32_t* seg_start, void* out, void* workspace,
                             size_t ws_bytes, uint32_t flags, void* stream);

/*
 * paged_attn_varlen_noalloc -- paged_attn_varlen for callers that cannot
 * allocate GPU memory.  (The pages have no counterpart: this is a calling
 * convention of this library.)
 *
 * Some callers may not call cudaMalloc or any allocating routine -- runtimes
 * that give all device memory to their own arena at start-up, real-time loops
 * where an allocation may synchronise the device or fail, plugin hosts that
 * hand a kernel library no allocator -- yet long windows still want the
 * key-range split, whose partial results need scratch space.  This call takes
 * the same arguments as paged_attn_varlen minus the workspace and uses instead
 * a fixed device array of PKV_NOALLOC_SCRATCH_BYTES inside the library, which
 * every GPU that loads the library's device code holds until the process exits.
 * Nothing is allocated at call time.
 *   - The array's device address is looked up once per device and CUDA
 *     context (a new context on the device, after cudaDeviceReset or a
 *     caller's own cuCtxCreate, looks it up again), inside the first call
 *     made with that device and context current; make that first call before
 *     any stream capture.
 *   - All calls share the array and it keeps the last call's contents (nothing
 *     in it has to start at zero).  Calls whose GPU work overlaps -- other
 *     streams, or unordered host threads -- race on it: do not issue them.
 *   - Splits forced with PKV_SPLITS(n) that would need more than the array
 *     holds (n * Tq * Hq * (D + 1) * 4 bytes) are refused with
 *     PKV_ERR_CAPACITY before anything is launched; automatic planning never
 *     asks for more than the array holds.
 * Everything else (arguments, layouts, errors, results) is as for paged_attn_varlen.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)
PKV_API pkv_status paged_attn_varlen_noalloc(const void* q, int64_t Tq, int Hq, const void* key_pool,
                                             const void* value_pool, int64_t num_blocks, int block_size, int Hkv,
                                             int D, pkv_dtype dt, const int32_t* block_table, int B, int W,
                                             const int32_t* query_start_loc, const int32_t* seq_lens,
                                             int max_query_len, int max_seq_len, float softmax_scale,
                                             const pkv_segment* segs, const int32_t* seg_start, void* out,
                                             uint32_t flags, void* stream);

/*
 * pkv_check -- synchronise `stream`, read and clear the device error word
 * raised by kernels run with PKV_CHECK_BOUNDS on the current device.
 *   bits   host, out: PKV_DEVERR_* bits seen since the last pkv_check (may be NULL)
 * Returns PKV_ERR_DEVICE_CHECK when any bit was set, PKV_ERR_CUDA if the
 * stream reports an error, else PKV_OK.
 */
PKV_API pkv_status pkv_check(void* stream, uint32_t* bits);

/*
 * pkv_last_launches -- number of kernels the last device call on this thread
 * (paged_kv_write, paged_kv_gather, paged_attn_varlen, paged_kv_write_attn,
 * paged_attn_varlen_noalloc, pkv_selftest_wait) launched: 0 when it launched nothing, 2 for an
 * attention call that split (the attention and its combine).
 */
PKV_API int pkv_last_launches(void);

/*
 * pkv_last_split_plan -- the key-range split of the last paged_attn_varlen /
 * paged_kv_write_attn call on this thread (each pointer may be NULL):
 *   splits       splits per split item (1: nothing was split)
 *   whole_items  items run unsplit before the split ones (tensor-core kernel; 0 when
 *                every item was split or nothing was)
 */
PKV_API void pkv_last_split_plan(int* splits, int64_t* whole_items);

/*
 * pkv_sm_count -- number of SMs of the current device (what the key-range
 * split planning counts waves in); -1 on error.
 */
PKV_API int pkv_sm_count(void);

/*
 * pkv_selftest_wait -- run the kernels' bounded pipeline wait on its own: one CTA waits on an
 * mbarrier that nothing completes, for limit_ns of wall time (0 < limit_ns <= 10 s), then sets
 * PKV_DEVERR_TIMEOUT in the device error word and exits.  A diagnostic (no counterpart on the
 * pages): it shows that an expired wait reports through pkv_check and leaves the context usable.
 * Asynchronous on `stream`.  Errors: PKV_ERR_INVALID_ARG (limit), PKV_ERR_CUDA (launch).
 */
PKV_API pkv_status pkv_selftest_wait(uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
