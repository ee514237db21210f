// Device helpers shared by the CUDA translation units of libpagedkv.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

#define PKV_DEVINLINE __device__ __forceinline__

template <typename T>
PKV_DEVINLINE float pkv_to_f32(T x);
template <>
PKV_DEVINLINE float pkv_to_f32<float>(float x) { return x; }
template <>
PKV_DEVINLINE float pkv_to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
PKV_DEVINLINE float pkv_to_f32<__half>(__half x) { return __half2float(x); }

template <typename T>
PKV_DEVINLINE T pkv_from_f32(float x);
template <>
PKV_DEVINLINE float pkv_from_f32<float>(float x) { return x; }
template <>
PKV_DEVINLINE __nv_bfloat16 pkv_from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
PKV_DEVINLINE __half pkv_from_f32<__half>(float x) { return __float2half_rn(x); }

PKV_DEVINLINE void pkv_raise(unsigned int* err, unsigned int bits) {
  if (err) atomicOr(err, bits);
}

// Key limit of the query at global position p of a row with L keys: the query
// sees keys [0, limit).  Segments are the row's piecewise mask (global
// coordinates): full -> kv_end; causal (bottom-right) -> kv_end - (q_end - p) + 1.
// No segments -> L.  A row no segment covers sees nothing (and is flagged).
// Global key position of a row's first query: the first segment's q_start when the row has
// segments (build_segments starts its cover at the query offset, the row's kv_start_pos),
// else the suffix convention L - Sq.
PKV_DEVINLINE int pkv_query_base(int L, int Sq, const pkv_segment* segs, int s_begin, int s_end) {
  return (segs != nullptr && s_begin < s_end) ? segs[s_begin].q_start : L - Sq;
}

PKV_DEVINLINE int pkv_row_limit(int p, int L, const pkv_segment* segs, int s_begin, int s_end, bool* uncovered) {
  if (segs == nullptr || s_begin >= s_end) return L;
  for (int s = s_begin; s < s_end; ++s) {
    const pkv_segment g = segs[s];
    if (p >= g.q_start && p < g.q_end) {
      int lim = g.mode == PKV_SEG_FULL ? g.kv_end : g.kv_end - (g.q_end - p) + 1;
      lim = lim < 0 ? 0 : lim;
      return lim > L ? L : lim;
    }
  }
  *uncovered = true;
  return 0;
}

// Work items of the tensor-core kernel: 256 queries (two 128-query tiles) of one (row, head).
// Item u -> (group member gi, tile pair qp, kv head kvh, row b), gi fastest, so the items of one
// (row, kv head) are adjacent and run together.  The split-KV combine decodes the same order.
constexpr int kTcItemRows = 256;

struct PkvTcItem {
  int gi, qp, kvh, b;
};

PKV_DEVINLINE PkvTcItem pkv_tc_item(int u, int g, int n_qp, int Hkv) {
  PkvTcItem it;
  it.gi = u % g;
  u /= g;
  it.qp = u % n_qp;
  u /= n_qp;
  it.kvh = u % Hkv;
  it.b = u / Hkv;
  return it;
}
