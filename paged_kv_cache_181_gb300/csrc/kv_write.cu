// Slot-mapping KV write: key_pool[slot[t]] = k[t], value_pool[slot[t]] = v[t]
// (paged_attention.py, _paged_write_attn_impl: ``pool[slots] = x`` for the
// video and the action tokens).
//
// HBM-bound copy of whole rows: a token's K (or V) row is Hkv*D*elem contiguous
// bytes both in the source and at its pool slot.  The rows are cut into chunks
// of kChunkVecs 16-byte vectors (2 KB); a warp copies one chunk per step, each
// lane loading its kU vectors before storing any, and the warps walk the flat
// list of (row, chunk) pairs with a grid stride, so every warp of a full wave
// has work even when the rows are few and wide (the long-window workload has
// 6240 rows of 10 KB for 152 x 64 warps).  Grid: one wave of resident CTAs.
// Measured per launch in bursts on distinct, cold buffers (% of the measured
// copy bandwidth): rows of 10 KB (128 MB) 22.4 us = 84 %; rows of 6 KB
// (201 MB) 35.8 us = 83 %; rows of 2 KB (52 MB) 10.3 us = 74 %; rows of 3 KB
// (38 MB) 8.2 us = 69 % (a launch pays a fixed few us of ramp-up and drain).
// One warp per whole row, all of it in registers, measured the same; TMA bulk
// copies staged through shared memory were slower (one issuing thread per CTA
// waits on each store's shared-memory read).

#include <atomic>

#include "kv_copy.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kU = 4;                       // vectors in flight per lane
constexpr int kChunkVecs = 32 * kU;         // 2 KB per warp step

// Rows are (token, K|V) pairs: row r is K (r even) or V (r odd) of token r/2; chunk c of the flat
// list is chunk c % cpr of row c / cpr.  A negative slot skips the token; with `check`, slots >=
// num_slots are flagged and skipped.  I is the index type: 32-bit when every chunk index fits.
template <typename I>
__global__ void __launch_bounds__(kThreads) kv_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                            const int64_t* __restrict__ slots, int64_t T,
                                                            uint4* __restrict__ kp, uint4* __restrict__ vp,
                                                            int64_t num_slots, int vec_per_row, int cpr,
                                                            unsigned int* err, int check) {
  const int lane = threadIdx.x & 31;
  const I n = (I)(2 * T) * (I)cpr;
  const I stride = (I)gridDim.x * kWarps;
  for (I c = (I)blockIdx.x * kWarps + (threadIdx.x >> 5); c < n; c += stride) {
    const I row = c / (I)cpr;
    const int ci = (int)(c - row * (I)cpr);
    const int64_t t = (int64_t)(row >> 1);
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;
    if (check && s >= num_slots) {
      if (lane == 0 && ci == 0) pkv_raise(err, PKV_DEVERR_SLOT);
      continue;
    }
    const uint4* src = ((row & 1) ? v : k) + t * vec_per_row;
    uint4* dst = ((row & 1) ? vp : kp) + s * vec_per_row;
    const int base = ci * kChunkVecs + lane;
    uint4 x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (base + 32 * u < vec_per_row) x[u] = __ldcs(src + base + 32 * u);
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (base + 32 * u < vec_per_row) dst[base + 32 * u] = x[u];
  }
}

// Resident CTAs per SM of one instantiation, per device (queried once; racing first calls from
// several host threads only store the same value).
template <typename I>
int resident_ctas() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kv_write_kernel<I>, kThreads, 0) != cudaSuccess || n <= 0) n = 4;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <typename I>
int launch_write(const void* k, const void* v, const int64_t* slots, int64_t T, void* kp, void* vp, int64_t num_slots,
                 int vec_per_row, int cpr, unsigned int* err, int check, int sms, void* stream) {
  const int64_t chunks = 2 * T * (int64_t)cpr;
  int64_t grid = (chunks + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sms * resident_ctas<I>();
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  kv_write_kernel<I><<<(unsigned)grid, kThreads, 0, (cudaStream_t)stream>>>(
      (const uint4*)k, (const uint4*)v, slots, T, (uint4*)kp, (uint4*)vp, num_slots, vec_per_row, cpr, err, check);
  return (int)cudaGetLastError();
}

}  // namespace

int pkv_launch_kv_write(const void* k, const void* v, const int64_t* slots, int64_t T, void* kp, void* vp,
                        int64_t num_slots, int row_bytes, unsigned int* err, int check, void* stream) {
  int sms = pkv_sm_count();
  if (sms <= 0) sms = 152;
  const int vec_per_row = row_bytes / 16;
  const int cpr = (vec_per_row + kChunkVecs - 1) / kChunkVecs;
  // 32-bit chunk indices while c + stride cannot wrap (the stride is at most a few hundred thousand).
  if (2 * T * (int64_t)cpr < ((int64_t)1 << 31))
    return launch_write<uint32_t>(k, v, slots, T, kp, vp, num_slots, vec_per_row, cpr, err, check, sms, stream);
  return launch_write<int64_t>(k, v, slots, T, kp, vp, num_slots, vec_per_row, cpr, err, check, sms, stream);
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
