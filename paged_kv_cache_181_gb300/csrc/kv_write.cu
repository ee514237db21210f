// Slot-mapping KV write: key_pool[slot[t]] = k[t], value_pool[slot[t]] = v[t]
// (paged_attention.py, _paged_write_attn_impl: ``pool[slots] = x`` for the
// video and the action tokens).
//
// HBM-bound copy.  One warp per (token, K|V) row: the row is Hkv*D*elem
// contiguous bytes both in the source and at its pool slot, so the lanes stride
// it in 16-byte vectors (fully coalesced on both sides), each lane keeping up to
// kUnroll loads in flight before it stores.  Indices are per row, so no
// per-vector division is needed.  K and V rows are interleaved in one launch;
// the grid is a multiple of the SM count.  (A vector-per-thread layout with a
// 64-bit division per vector measured 27.1 us per launch on the long-window
// workload; this one 24.8 us, 76 % of the measured copy bandwidth.)

#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kThreads) kv_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                            const int64_t* __restrict__ slots, int64_t T,
                                                            uint4* __restrict__ kp, uint4* __restrict__ vp,
                                                            int64_t num_slots, int vec_per_row, unsigned int* err,
                                                            int check) {
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = (int64_t)gridDim.x * kWarps;
  const int64_t rows = T * 2;
  for (int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); row < rows; row += n_warps) {
    const int64_t t = row >> 1;
    const bool is_v = row & 1;
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;  // negative slot: skip the token
    if (check && s >= num_slots) {
      if (lane == 0) pkv_raise(err, PKV_DEVERR_SLOT);
      continue;
    }
    const uint4* src = (is_v ? v : k) + t * vec_per_row;
    uint4* dst = (is_v ? vp : kp) + s * vec_per_row;
    int c = lane;
    for (; c + 32 * (kUnroll - 1) < vec_per_row; c += 32 * kUnroll) {
      uint4 x[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) x[u] = __ldg(src + c + 32 * u);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) dst[c + 32 * u] = x[u];
    }
    for (; c < vec_per_row; c += 32) dst[c] = __ldg(src + c);
  }
}

}  // namespace

int pkv_launch_kv_write(const void* k, const void* v, const int64_t* slots, int64_t T, void* kp, void* vp,
                        int64_t num_slots, int row_bytes, unsigned int* err, int check, void* stream) {
  const int vec_per_row = row_bytes / 16;
  int sms = pkv_sm_count();
  if (sms <= 0) sms = 152;
  int64_t grid = (T * 2 + kWarps - 1) / kWarps;  // one warp per row
  const int64_t cap = (int64_t)sms * 8;           // 8 resident 256-thread CTAs per SM
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  kv_write_kernel<<<(unsigned)grid, kThreads, 0, (cudaStream_t)stream>>>(
      (const uint4*)k, (const uint4*)v, slots, T, (uint4*)kp, (uint4*)vp, num_slots, vec_per_row, err, check);
  return (int)cudaGetLastError();
}
