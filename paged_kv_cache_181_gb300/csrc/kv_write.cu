// Slot-mapping KV write: key_pool[slot[t]] = k[t], value_pool[slot[t]] = v[t]
// (paged_attention.py, _paged_write_attn_impl: ``pool[slots] = x`` for the
// video and the action tokens).
//
// HBM-bound copy.  Every 16-byte vector of every token row is one work item;
// consecutive threads take consecutive vectors of a row, so both the read of
// the source row and the write into its pool slot are fully coalesced
// (each row is Hkv*D*elem contiguous bytes at both ends).  K and V rows are
// interleaved in one launch.  Each thread keeps UNROLL loads in flight before
// it stores, and the grid is a multiple of the SM count.

#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) kv_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                            const int64_t* __restrict__ slots, int64_t T,
                                                            uint4* __restrict__ kp, uint4* __restrict__ vp,
                                                            int64_t num_slots, int vec_per_row,
                                                            unsigned int* err, int check) {
  const int64_t total = T * 2 * (int64_t)vec_per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i < total; i += stride * kUnroll) {
    uint4 val[kUnroll];
    int64_t dst[kUnroll];
    uint4* pool[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t it = i + u * stride;
      dst[u] = -1;
      pool[u] = nullptr;
      if (it < total) {
        const int64_t row = it / vec_per_row;
        const int vec = (int)(it - row * vec_per_row);
        const int64_t t = row >> 1;
        const bool is_v = row & 1;
        const int64_t s = __ldg(slots + t);
        if (s >= 0 && (!check || s < num_slots)) {
          const uint4* src = (is_v ? v : k) + t * vec_per_row + vec;
          val[u] = __ldg(src);
          dst[u] = s * vec_per_row + vec;
          pool[u] = is_v ? vp : kp;
        } else if (check && s >= num_slots) {
          pkv_raise(err, PKV_DEVERR_SLOT);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (dst[u] >= 0) pool[u][dst[u]] = val[u];
  }
}

}  // namespace

int pkv_launch_kv_write(const void* k, const void* v, const int64_t* slots, int64_t T, void* kp, void* vp,
                        int64_t num_slots, int row_bytes, unsigned int* err, int check, void* stream) {
  const int vec_per_row = row_bytes / 16;
  const int64_t total = T * 2 * (int64_t)vec_per_row;
  int sms = pkv_sm_count();
  if (sms <= 0) sms = 152;
  const int64_t want = (total + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
  const int64_t cap = (int64_t)sms * 8;  // 8 resident 256-thread CTAs per SM
  int grid = (int)(want < cap ? want : cap);
  if (grid < 1) grid = 1;
  kv_write_kernel<<<grid, kThreads, 0, (cudaStream_t)stream>>>(
      (const uint4*)k, (const uint4*)v, slots, T, (uint4*)kp, (uint4*)vp, num_slots, vec_per_row, err, check);
  return (int)cudaGetLastError();
}
