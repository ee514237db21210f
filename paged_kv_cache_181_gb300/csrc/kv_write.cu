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

#include "kv_copy.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads) kv_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                            const int64_t* __restrict__ slots, int64_t T,
                                                            uint4* __restrict__ kp, uint4* __restrict__ vp,
                                                            int64_t num_slots, int vec_per_row, unsigned int* err,
                                                            int check) {
  pkv_scatter(k, v, slots, T, kp, vp, num_slots, vec_per_row, err, check,
              (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5), (int64_t)gridDim.x * kWarps, threadIdx.x & 31,
              nullptr);
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

// ---------------------------------------------------------------- block gather into staging
//
// stage[b][first*16 + t] = pool[table[b][first + t/16]*16 + t%16] for K and V (paged_attention.py,
// _stage_window).  Same shape as the write: one warp per (row b, token t, K|V) destination row.
namespace {

__global__ void __launch_bounds__(kThreads) kv_gather_kernel(const uint4* __restrict__ kp, const uint4* __restrict__ vp,
                                                             int64_t num_blocks, const int32_t* __restrict__ table,
                                                             int B, int W, int first_block, int n_blocks,
                                                             uint4* __restrict__ sk, uint4* __restrict__ sv,
                                                             int64_t stage_rows, int vec_per_row, unsigned int* err,
                                                             int check) {
  // The host keeps B * n_blocks * 32 below 2^31, so the row arithmetic stays in 32 bits.
  const int lane = threadIdx.x & 31;
  const int n_warps = gridDim.x * kWarps;
  const int per_row = n_blocks * 16;
  const int rows = B * per_row * 2;
  for (int w = blockIdx.x * kWarps + (threadIdx.x >> 5); w < rows; w += n_warps) {
    const bool is_v = w & 1;
    const int bt = w >> 1;
    const int b = bt / per_row;
    const int t = bt - b * per_row;
    int blk = __ldg(table + (int64_t)b * W + first_block + (int)(t >> 4));
    if (check && (blk < 0 || blk >= num_blocks)) {
      if (lane == 0) pkv_raise(err, PKV_DEVERR_BLOCK);
      continue;
    }
    const uint4* src = (is_v ? vp : kp) + ((int64_t)blk * 16 + (t & 15)) * vec_per_row;
    uint4* dst = (is_v ? sv : sk) + ((int64_t)b * stage_rows + (int64_t)first_block * 16 + t) * vec_per_row;
    pkv_copy_row(src, dst, vec_per_row, lane);
  }
}

}  // namespace

int pkv_launch_kv_gather(const void* kp, const void* vp, int64_t num_blocks, const int32_t* table, int B, int W,
                         int first_block, int n_blocks, void* sk, void* sv, int64_t stage_rows, int row_bytes,
                         unsigned int* err, int check, void* stream) {
  const int vec_per_row = row_bytes / 16;
  int sms = pkv_sm_count();
  if (sms <= 0) sms = 152;
  int64_t grid = ((int64_t)B * n_blocks * 32 + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sms * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  kv_gather_kernel<<<(unsigned)grid, kThreads, 0, (cudaStream_t)stream>>>(
      (const uint4*)kp, (const uint4*)vp, num_blocks, table, B, W, first_block, n_blocks, (uint4*)sk, (uint4*)sv,
      stage_rows, vec_per_row, err, check);
  return (int)cudaGetLastError();
}
