// Host side of libpagedkv: error reporting and the once-per-forward metadata
// (segments, slot mapping, visible window, padded block-table row).
//
// Sources: piecewise_attn.py (build_segments, build_paged_piecewise_plan) and
// paged_attention.py (video_block_table, build_block_table, max_video_blocks,
// ensure_video_slots / _reference_paged_attention addressing).

#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "pagedkv.h"
#include "internal.h"

namespace {
thread_local char g_last_error[512] = "";
thread_local int g_last_launches = 0;
thread_local int g_last_splits = 1;
thread_local int64_t g_last_whole_items = 0;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t gcd64(int64_t a, int64_t b) {
  while (b) {
    int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}
}  // namespace

pkv_status pkv_fail(pkv_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

void pkv_clear_error() { g_last_error[0] = '\0'; }

void pkv_set_launches(int n) { g_last_launches = n; }

extern "C" int pkv_last_launches(void) { return g_last_launches; }

void pkv_set_split_plan(int splits, int64_t whole_items) {
  g_last_splits = splits;
  g_last_whole_items = whole_items;
}

extern "C" void pkv_last_split_plan(int* splits, int64_t* whole_items) {
  if (splits) *splits = g_last_splits;
  if (whole_items) *whole_items = g_last_whole_items;
}

extern "C" const char* pkv_last_error(void) { return g_last_error; }

extern "C" const char* pkv_version(void) { return "pagedkv 0.1 (sm_103a)"; }

extern "C" pkv_status build_segments(const int32_t* spans, int n_spans, int32_t query_offset, int32_t query_len,
                                     int32_t seq_len, pkv_segment* out, int capacity, int* n_out) {
  pkv_clear_error();
  if (n_out == nullptr || (n_spans > 0 && spans == nullptr) || n_spans < 0 || (capacity > 0 && out == nullptr))
    return pkv_fail(PKV_ERR_INVALID_ARG, "build_segments: NULL pointer or negative span count");
  // Validation (build_paged_piecewise_plan): sorted, non-overlapping, 0 <= start < end <= seq_len.
  int32_t previous_end = 0;
  for (int i = 0; i < n_spans; ++i) {
    const int32_t a = spans[2 * i], b = spans[2 * i + 1];
    if (a < previous_end || !(0 <= a && a < b && b <= seq_len))
      return pkv_fail(PKV_ERR_INVALID_ARG,
                      "build_segments: spans must be sorted, non-overlapping and within the sequence (span %d = "
                      "[%d, %d), seq_len %d)",
                      i, a, b, seq_len);
    previous_end = b;
  }
  if (query_offset < 0 || query_len <= 0 || (int64_t)query_offset + query_len > seq_len)
    return pkv_fail(PKV_ERR_INVALID_ARG, "build_segments: query range [%d, %d) must lie within [0, %d)",
                    query_offset, query_offset + query_len, seq_len);

  const int32_t q_lo = query_offset, q_hi = query_offset + query_len;
  int n = 0;
  auto emit = [&](int32_t s, int32_t e, int32_t kv_end, int32_t mode) -> bool {
    if (n >= capacity) return false;
    out[n++] = pkv_segment{s, e, kv_end, mode};
    return true;
  };
  int32_t cursor = q_lo;
  for (int i = 0; i < n_spans; ++i) {
    const int32_t a = spans[2 * i], b = spans[2 * i + 1];
    const int32_t lo = a > q_lo ? a : q_lo;
    const int32_t hi = b < q_hi ? b : q_hi;
    if (lo >= hi) continue;
    if (cursor < lo && !emit(cursor, lo, lo, PKV_SEG_CAUSAL)) goto full;
    if (!emit(lo, hi, b, PKV_SEG_FULL)) goto full;
    cursor = hi;
  }
  if (cursor < q_hi && !emit(cursor, q_hi, q_hi, PKV_SEG_CAUSAL)) goto full;
  *n_out = n;
  return PKV_OK;
full:
  return pkv_fail(PKV_ERR_CAPACITY, "build_segments: capacity %d is too small (2 * n_spans + 1 = %d suffices)",
                  capacity, 2 * n_spans + 1);
}

extern "C" pkv_status pkv_slot_mapping(const int32_t* blocks, int64_t n_blocks, int64_t first_position,
                                       int64_t n_tokens, int block_size, int64_t* slots) {
  pkv_clear_error();
  if (n_tokens < 0 || first_position < 0 || block_size <= 0 || n_blocks < 0)
    return pkv_fail(PKV_ERR_INVALID_ARG, "pkv_slot_mapping: negative size");
  if (n_tokens == 0) return PKV_OK;
  if (blocks == nullptr || slots == nullptr) return pkv_fail(PKV_ERR_INVALID_ARG, "pkv_slot_mapping: NULL pointer");
  const int64_t last_block = (first_position + n_tokens - 1) / block_size;
  if (last_block >= n_blocks)
    return pkv_fail(PKV_ERR_INVALID_ARG, "pkv_slot_mapping: position %lld needs logical block %lld of %lld",
                    (long long)(first_position + n_tokens - 1), (long long)last_block, (long long)n_blocks);
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int64_t p = first_position + t;
    const int32_t blk = blocks[p / block_size];
    if (blk < 0) return pkv_fail(PKV_ERR_INVALID_ARG, "pkv_slot_mapping: logical block %lld is not allocated",
                                 (long long)(p / block_size));
    slots[t] = (int64_t)blk * block_size + p % block_size;
  }
  return PKV_OK;
}

extern "C" int64_t pkv_table_width(int64_t chunk_tokens, int64_t sink_tokens, int64_t window_tokens,
                                   int64_t action_len, int block_size) {
  pkv_clear_error();
  if (chunk_tokens <= 0 || sink_tokens < 0 || window_tokens < 0 || action_len < 0 || block_size <= 0) {
    pkv_fail(PKV_ERR_INVALID_ARG, "pkv_table_width: sizes must be non-negative (chunk > 0)");
    return -1;
  }
  const int64_t sink_blocks = ceil_div(sink_tokens, block_size);
  const int64_t slack = block_size - gcd64(chunk_tokens, block_size);
  const int64_t recent_blocks = ceil_div(window_tokens + slack, block_size);
  const int64_t action_blocks = ceil_div(action_len, block_size);
  return sink_blocks + recent_blocks + (action_blocks > 1 ? action_blocks : 1);
}

extern "C" pkv_status pkv_visible_window(const int32_t* row_blocks, int64_t n_row_blocks, int64_t end_tokens,
                                         int64_t sink_tokens, int64_t window_tokens, int block_size,
                                         int32_t* out_blocks, int64_t capacity, int64_t* n_out,
                                         int64_t* video_len) {
  pkv_clear_error();
  if (n_out == nullptr || video_len == nullptr || block_size <= 0 || end_tokens < 0 || sink_tokens < 0 ||
      window_tokens < 0 || capacity < 0)
    return pkv_fail(PKV_ERR_INVALID_ARG, "pkv_visible_window: NULL output or negative size");
  const int64_t n_blocks = ceil_div(end_tokens, block_size);
  if (n_row_blocks < n_blocks || (n_blocks > 0 && row_blocks == nullptr))
    return pkv_fail(PKV_ERR_INVALID_ARG, "pkv_visible_window: %lld row blocks do not cover %lld positions",
                    (long long)n_row_blocks, (long long)end_tokens);
  const int64_t sink_end = sink_tokens;
  const int64_t recent_start = end_tokens - window_tokens;
  int64_t n = 0, len = 0;
  for (int64_t i = 0; i < n_blocks; ++i) {
    const int64_t first = i * block_size;
    const int32_t blk = row_blocks[i];
    if (blk < 0) continue;                                               // evicted
    if (first >= sink_end && first + block_size <= recent_start) continue;  // between sink and window
    if (len % block_size)
      return pkv_fail(PKV_ERR_INVALID_ARG,
                      "pkv_visible_window: would read past a partly written block (block %d followed by %d)",
                      out_blocks && n > 0 ? out_blocks[n - 1] : -1, blk);
    if (n >= capacity)
      return pkv_fail(PKV_ERR_CAPACITY, "pkv_visible_window: capacity %lld is too small", (long long)capacity);
    out_blocks[n++] = blk;
    const int64_t rest = end_tokens - first;
    len += rest < block_size ? rest : block_size;
  }
  *n_out = n;
  *video_len = len;
  return PKV_OK;
}

extern "C" pkv_status pkv_block_table_row(const int32_t* video_blocks, int64_t n_video, int64_t video_len,
                                          const int32_t* action_blocks, int64_t action_len, int block_size,
                                          int64_t width, int32_t* out_row, int64_t* kv_len) {
  pkv_clear_error();
  if (out_row == nullptr || kv_len == nullptr || block_size <= 0 || n_video < 0 || video_len < 0 ||
      action_len < 0 || width < 0 || (n_video > 0 && video_blocks == nullptr) ||
      (action_len > 0 && action_blocks == nullptr))
    return pkv_fail(PKV_ERR_INVALID_ARG, "pkv_block_table_row: NULL pointer or negative size");
  if (action_len > 0 && video_len % block_size)
    return pkv_fail(PKV_ERR_INVALID_ARG,
                    "pkv_block_table_row: cannot place action tokens after a partly written video block (the "
                    "video run ends %lld slots into its last block)",
                    (long long)(video_len % block_size));
  const int64_t n_action = ceil_div(action_len, block_size);
  const int64_t n = n_video + n_action;
  if (n == 0) return pkv_fail(PKV_ERR_INVALID_ARG, "pkv_block_table_row: needs at least one key block");
  if (n > width)
    return pkv_fail(PKV_ERR_CAPACITY, "pkv_block_table_row: %lld blocks do not fit width %lld", (long long)n,
                    (long long)width);
  int64_t w = 0;
  for (int64_t i = 0; i < n_video; ++i) out_row[w++] = video_blocks[i];
  for (int64_t i = 0; i < n_action; ++i) out_row[w++] = action_blocks[i];
  while (w < width) out_row[w++] = 0;
  *kv_len = video_len + action_len;
  return PKV_OK;
}
