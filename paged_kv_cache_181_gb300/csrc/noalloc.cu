// paged_attn_varlen_noalloc: the paged attention call for callers that cannot
// allocate GPU memory.
//
// Some callers of this library are not allowed to call cudaMalloc or any
// allocating routine: runtimes that hand every byte of device memory to their
// own fixed-size arena at start-up, real-time loops where an allocation (which
// may synchronise the device or fail under fragmentation) is not acceptable,
// and plugin hosts whose API gives a kernel library no allocator at all.  They
// still want the key-range split of long windows, whose partial outputs need
// scratch space.  This entry point gives them that scratch from a fixed array
// in the library itself, so it allocates nothing at call time.
//
// The scratch is a file-scope device array of PKV_NOALLOC_SCRATCH_BYTES bytes.
// Every GPU on which this library's device code is loaded holds it until the
// process exits.  In host code the array's name is only a host-side stand-in,
// not a device address, so its device address is looked up once per device
// (with that device current) through cudaGetSymbolAddress and cached, keyed
// on the current CUDA context, so a new context on the device (after
// cudaDeviceReset, or a caller's own context) looks it up again; that happens
// inside the first call made on each device (and in each new context), which
// should therefore come before any stream capture.  All calls share the one
// array and it keeps whatever the last call left in it; nothing in it needs to start at zero
// (every split writes its whole partial output and log-sum-exp before the
// combine reads them).  Calls whose work overlaps on the GPU -- on different
// streams, or from different host threads without ordering -- race on the
// array and must not be issued.

#include <mutex>

#include "common.cuh"

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
uint64_t g_scratch_ctx[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once per device and context).
pkv_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pkv_fail(PKV_ERR_CUDA, "paged_attn_varlen_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return pkv_fail(PKV_ERR_UNSUPPORTED, "paged_attn_varlen_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const uint64_t ctx = pkv_context_id();
  if (!g_scratch_addr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return pkv_fail(PKV_ERR_CUDA, "paged_attn_varlen_noalloc: cudaGetSymbolAddress of the scratch array failed: %s",
                      cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = pkv_context_id();
  }
  *out = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status paged_attn_varlen_noalloc(const void* q, int64_t Tq, int Hq, const void* key_pool,
                                                const void* value_pool, int64_t num_blocks, int block_size, int Hkv,
                                                int D, pkv_dtype dt, const int32_t* block_table, int B, int W,
                                                const int32_t* query_start_loc, const int32_t* seq_lens,
                                                int max_query_len, int max_seq_len, float softmax_scale,
                                                const pkv_segment* segs, const int32_t* seg_start, void* out,
                                                uint32_t flags, void* stream) {
  pkv_clear_error();
  pkv_set_launches(0);
  // A forced number of splits that the fixed scratch cannot hold is refused before anything runs.
  // (Clamped as paged_attn_varlen clamps it, so both calls accept the same requests.)
  int forced = (int)((flags >> 8) & 0xffu);
  if (forced > kPkvMaxSplits) forced = kPkvMaxSplits;
  if (forced > 1 && Tq > 0 && Hq > 0 && D > 0) {
    const unsigned long long need =
        (unsigned long long)forced * (unsigned long long)Tq * (unsigned long long)Hq * ((unsigned long long)D + 1) * 4ull;
    if (need > (unsigned long long)PKV_NOALLOC_SCRATCH_BYTES)
      return pkv_fail(PKV_ERR_CAPACITY,
                      "paged_attn_varlen_noalloc: %d key-range splits of %lld queries x %d heads x %d need %llu bytes "
                      "of scratch; the library's fixed scratch holds %llu",
                      forced, (long long)Tq, Hq, D, need, (unsigned long long)PKV_NOALLOC_SCRATCH_BYTES);
  }
  void* scratch = nullptr;
  const pkv_status st = scratch_address(&scratch);
  if (st != PKV_OK) return st;
  return paged_attn_varlen(q, Tq, Hq, key_pool, value_pool, num_blocks, block_size, Hkv, D, dt, block_table, B, W,
                           query_start_loc, seq_lens, max_query_len, max_seq_len, softmax_scale, segs, seg_start, out,
                           scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES, flags, stream);
}
