// The slot-mapping scatter (paged_attention.py, _paged_write_attn_impl: pool[slots] = x), as a
// device routine shared by the write kernel and the fused write + attention kernels.
//
// Work item = one (token, K|V) row of Hkv*D*elem contiguous bytes; one warp copies it in 16-byte
// vectors (coalesced on both sides), up to kCopyUnroll loads in flight per lane.
#pragma once

#include "common.cuh"

constexpr int kCopyUnroll = 8;

PKV_DEVINLINE void pkv_copy_row(const uint4* __restrict__ src, uint4* __restrict__ dst, int vec_per_row, int lane) {
  int c = lane;
  for (; c + 32 * (kCopyUnroll - 1) < vec_per_row; c += 32 * kCopyUnroll) {
    uint4 x[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) x[u] = __ldg(src + c + 32 * u);
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) dst[c + 32 * u] = x[u];
  }
  for (; c < vec_per_row; c += 32) dst[c] = __ldg(src + c);
}

// Fused call only, check mode: token t must land on the slot its key position implies --
// row b with q0 = query_start_loc[b] <= t, key base_b + (t - q0), slot table[b][key/16]*16 + key%16 --
// since the attention of the same launch reads the token's K/V from the source, not the pool.
PKV_DEVINLINE bool pkv_slot_is_implied(const PkvAttnArgs& a, int64_t t, int64_t s) {
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.query_start_loc[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int b = lo;
  const int q0 = a.query_start_loc[b], q1 = a.query_start_loc[b + 1];
  if (t < q0 || t >= q1) return false;
  const int L = a.seq_lens[b];
  int s_begin = 0, s_end = 0;
  if (a.segs) {
    s_begin = a.seg_start[b];
    s_end = a.seg_start[b + 1];
  }
  const int64_t key = (int64_t)pkv_query_base(L, q1 - q0, a.segs, s_begin, s_end) + (t - q0);
  if (key < 0 || key >= L || key >= (int64_t)a.W * 16) return false;
  return s == (int64_t)a.block_table[(int64_t)b * a.W + key / 16] * 16 + key % 16;
}

// Rows w0, w0 + stride, ... of the 2T rows (row 2t = K of token t, 2t+1 = V); one warp calls it.
// A negative slot skips the token.  With `check`, slots >= num_slots are flagged and skipped, and
// with `fa` (the fused call) so are tokens that would not land on their implied slot.
PKV_DEVINLINE void pkv_scatter(const uint4* __restrict__ k, const uint4* __restrict__ v,
                               const int64_t* __restrict__ slots, int64_t T, uint4* __restrict__ kp,
                               uint4* __restrict__ vp, int64_t num_slots, int vec_per_row, unsigned int* err, int check,
                               int64_t w0, int64_t stride, int lane, const PkvAttnArgs* fa) {
  for (int64_t row = w0; row < 2 * T; row += stride) {
    const int64_t t = row >> 1;
    const bool is_v = row & 1;
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;
    if (check) {  // every lane evaluates the same row, so the decision is warp-uniform
      bool bad = s >= num_slots;
      if (!bad && fa && !is_v) bad = !pkv_slot_is_implied(*fa, t, s);
      if (bad) {
        if (lane == 0) pkv_raise(err, PKV_DEVERR_SLOT);
        continue;
      }
    }
    pkv_copy_row((is_v ? v : k) + t * vec_per_row, (is_v ? vp : kp) + s * vec_per_row, vec_per_row, lane);
  }
}
