// Slot-mapping KV write: key_pool[slot[t]] = k[t], value_pool[slot[t]] = v[t]
// (paged_attention.py, _paged_write_attn_impl: ``pool[slots] = x`` for the
// video and the action tokens).
//
// HBM-bound copy of whole rows: a token's K (or V) row is Hkv*D*elem contiguous
// bytes both in the source and at its pool slot.  The copy engine moves them:
// one warp per CTA, whose lane 0 takes batches of kStages rows, loads each row
// into shared memory with one bulk copy (completion counted on the row's
// mbarrier) and writes it to its slot with one bulk store; the next batch
// reuses the buffers once the stores have read them.  Grid: up to kCtasPerSm
// CTAs per SM.  Measured on the long-window workload (3120 tokens x 10 KB rows,
// K and V): 23.6 us per launch in 40-launch bursts (80 % of the measured copy
// bandwidth), against 25.3 us for one warp per row with 8 16-byte loads in
// flight per lane -- which stays as the kernel for rows too wide to stage.

#include <atomic>

#include "kv_copy.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 4;         // rows in flight per CTA
constexpr int kCtasPerSm = 4;
constexpr int kMaxStageBytes = 200 * 1024;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

PKV_DEVINLINE void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(ptx::smem_u32(bar))
               : "memory");
}

PKV_DEVINLINE void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes) : "memory");
}

// Rows are (token, K|V) pairs: row r is K (r even) or V (r odd) of token r/2.  A negative slot skips
// the token; with `check`, slots >= num_slots are flagged and skipped.  Every wait is bounded: on
// expiry the CTA records PKV_DEVERR_TIMEOUT, waits for its stores and exits.
__global__ void __launch_bounds__(32) kv_write_bulk_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                                                            const int64_t* __restrict__ slots, int64_t T,
                                                            uint8_t* __restrict__ kp, uint8_t* __restrict__ vp,
                                                            int64_t num_slots, int row_bytes, unsigned int* err,
                                                            int check) {
  extern __shared__ __align__(128) uint8_t stage[];
  __shared__ uint64_t bar[kStages];
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kStages; ++s) ptx::mbar_init(&bar[s], 1);
  ptx::fence_mbar_init();
  const uint32_t sbase = ptx::smem_u32(stage);
  const int64_t rows = 2 * T;
  int never = 0;
  uint32_t phase = 0;
  for (int64_t b0 = (int64_t)blockIdx.x * kStages; b0 < rows; b0 += (int64_t)gridDim.x * kStages, phase ^= 1) {
    int64_t dst[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      const int64_t r = b0 + s;
      dst[s] = -1;
      if (r < rows) {
        const int64_t sl = __ldg(slots + (r >> 1));
        if (sl >= 0 && check && sl >= num_slots) pkv_raise(err, PKV_DEVERR_SLOT);
        else dst[s] = sl;
      }
      // Each stage's barrier completes once per batch: on its row's bytes, or at once when it has none.
      if (dst[s] >= 0) {
        ptx::mbar_arrive_expect_tx(&bar[s], (uint32_t)row_bytes);
        bulk_load(sbase + s * row_bytes, ((r & 1) ? v : k) + (r >> 1) * row_bytes, (uint32_t)row_bytes, &bar[s]);
      } else {
        ptx::mbar_arrive(&bar[s]);
      }
    }
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      if (!ptx::mbar_wait(&bar[s], phase, &never, kWaitLimitNs)) {
        pkv_raise(err, PKV_DEVERR_TIMEOUT);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        return;
      }
      if (dst[s] >= 0) {
        const int64_t r = b0 + s;
        bulk_store(((r & 1) ? vp : kp) + dst[s] * row_bytes, sbase + s * row_bytes, (uint32_t)row_bytes);
      }
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // the buffers are free again
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Rows too wide to stage: one warp per row (pkv_scatter).
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
  int sms = pkv_sm_count();
  if (sms <= 0) sms = 152;
  const int64_t smem = (int64_t)kStages * row_bytes;
  if (smem <= kMaxStageBytes && err) {
    // Per device, once; racing first calls from several host threads only repeat the same setting.
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    const bool cached = dev >= 0 && dev < 64;
    if (!cached || !attr_set[dev].load(std::memory_order_acquire)) {
      const cudaError_t e = cudaFuncSetAttribute(kv_write_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kMaxStageBytes);
      if (e != cudaSuccess) return (int)e;
      if (cached) attr_set[dev].store(true, std::memory_order_release);
    }
    int64_t grid = (2 * T + kStages - 1) / kStages;
    const int64_t cap = (int64_t)sms * kCtasPerSm;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    kv_write_bulk_kernel<<<(unsigned)grid, 32, (size_t)smem, (cudaStream_t)stream>>>(
        (const uint8_t*)k, (const uint8_t*)v, slots, T, (uint8_t*)kp, (uint8_t*)vp, num_slots, row_bytes, err, check);
    return (int)cudaGetLastError();
  }
  const int vec_per_row = row_bytes / 16;
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
