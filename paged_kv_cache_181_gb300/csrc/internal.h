// Declarations shared by the translation units of libpagedkv (not installed).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "pagedkv.h"

// Record a failure message for pkv_last_error() and return `code`.
pkv_status pkv_fail(pkv_status code, const char* fmt, ...);
void pkv_clear_error();
void pkv_set_launches(int n);
void pkv_set_split_plan(int splits, int64_t whole_items);

// Device error word of the current device (PKV_DEVERR_* bits); nullptr when unavailable.
unsigned int* pkv_device_error_word();

inline int pkv_dtype_size(pkv_dtype dt) { return dt == PKV_F32 ? 4 : 2; }

// Most key-range splits per item; larger PKV_SPLITS(n) requests are clamped to it.
constexpr int kPkvMaxSplits = 16;

// CUDA-core attention kernel: queries per CTA, keys per tile, CTAs resident per SM (its shared memory
// holds the fp32 Q, K, V and P tiles: one CTA per SM).  The split planner counts in these.
constexpr int kSimtItemRows = 128;
constexpr int kSimtKeyTile = 64;
constexpr int kSimtCtasPerSm = 1;

// Process-unique id of the CUDA context current on this thread (0: none, or the driver call is
// unavailable).  Per-device caches of device addresses and function attributes are keyed on it, so
// that a new context on the same device (after cudaDeviceReset, or a caller's own context) looks
// them up again instead of reusing the old context's values.
uint64_t pkv_context_id();

// Per-row work description shared by the attention kernels.
struct PkvAttnArgs {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  void* out;
  const int32_t* block_table;
  const int32_t* query_start_loc;
  const int32_t* seq_lens;
  const pkv_segment* segs;
  const int32_t* seg_start;
  float* part_o;    // [splits, Tq, Hq, D] fp32, when splitting
  float* part_lse;  // [splits, Tq, Hq] fp32 (natural log), when splitting
  unsigned int* err;
  int64_t num_blocks;
  int64_t Tq;
  int B, W, Hq, Hkv, D;
  int max_query_len, max_seq_len;
  int num_splits;
  // Split tail (num_splits > 1): items [0, split_direct) run one CTA each and write `out`;
  // every later item runs num_splits CTAs over parts of its key range and leaves partials for
  // the combine.  0: every item is split.
  int split_direct;
  // Which kernel's items the split tail counts: 0 the tensor-core kernel's (256 queries of one
  // row and head, pkv_tc_item order), 1 the CUDA-core kernel's (128 queries; the row's query
  // tiles fastest, then the rows, then the heads).
  int simt_items;
  int check;
  int contiguous;  // PKV_CONTIGUOUS_KV
  float scale;
  // Fused write (paged_kv_write_attn): the current tokens' K/V [Tq, Hkv, D] and their slots.
  // The same launch scatters them into the pools and its attention reads the keys of the
  // queries' own positions from here instead of the pools.  k_new == nullptr: no write.
  const void* k_new;
  const void* v_new;
  const int64_t* slots;
  int64_t num_slots;
};

// Launchers (each returns cudaGetLastError() as an int, 0 == success).
int pkv_launch_kv_write(const void* k, const void* v, const int64_t* slots, int64_t T, void* kp, void* vp,
                        int64_t num_slots, int row_bytes, unsigned int* err, int check, void* stream);
int pkv_launch_kv_gather(const void* kp, const void* vp, int64_t num_blocks, const int32_t* table, int B, int W,
                          int first_block, int n_blocks, void* sk, void* sv, int64_t stage_rows, int row_bytes,
                          unsigned int* err, int check, void* stream);
int pkv_launch_attn_simt(const PkvAttnArgs& a, pkv_dtype dt, void* stream);
int pkv_launch_attn_combine(const PkvAttnArgs& a, pkv_dtype dt, void* stream);
// tcgen05 path; returns -1 when the shape is not handled by it.
int pkv_launch_attn_tc(const PkvAttnArgs& a, pkv_dtype dt, void* stream);
bool pkv_attn_tc_supports(pkv_dtype dt, int D);
