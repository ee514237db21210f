// Device entry points of libpagedkv: argument validation, key-range split
// planning, launches, and the device error word read back by pkv_check().

#include <cuda.h>
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace {

// One error word per device.  Kernels in PKV_CHECK_BOUNDS mode OR bits into it.
__device__ unsigned int g_pkv_error_word;

constexpr int kMaxDevices = 64;
unsigned int* g_err_ptr[kMaxDevices] = {};
uint64_t g_err_ctx[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::mutex g_mu;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

constexpr int kMaxSplits = kPkvMaxSplits;
constexpr int kWorkspaceSplits = 8;  // paged_attn_workspace_size covers at least this many (forced splits)

}  // namespace

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

uint64_t pkv_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = (CtxGetCurrentFn)p;
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = (CtxGetIdFn)p;
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return (uint64_t)id;
}

unsigned int* pkv_device_error_word() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  const uint64_t ctx = pkv_context_id();
  if (!g_err_ptr[dev] || ctx == 0 || g_err_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = (unsigned int*)p;
    g_err_ctx[dev] = pkv_context_id();  // the lookup makes the device's primary context current
  }
  return g_err_ptr[dev];
}

extern "C" int pkv_sm_count(void) {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sm_count[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

extern "C" pkv_status pkv_check(void* stream, uint32_t* bits) {
  pkv_clear_error();
  if (bits) *bits = 0;
  unsigned int* w = pkv_device_error_word();
  if (!w) return pkv_fail(PKV_ERR_CUDA, "pkv_check: no CUDA device");
  unsigned int host = 0;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&host, w, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(w, 0, sizeof(unsigned int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return pkv_fail(PKV_ERR_CUDA, "pkv_check: %s", cudaGetErrorString(e));
  if (bits) *bits = host;
  if (host) return pkv_fail(PKV_ERR_DEVICE_CHECK, "pkv_check: device metadata check failed (bits 0x%x)", host);
  return PKV_OK;
}

extern "C" pkv_status paged_kv_write(const void* k, const void* v, const int64_t* slot_mapping, int64_t T,
                                     void* key_pool, void* value_pool, int64_t num_slots, int Hkv, int D,
                                     pkv_dtype dt, uint32_t flags, void* stream) {
  pkv_clear_error();
  pkv_set_launches(0);
  if (T < 0 || num_slots < 0 || Hkv <= 0 || D <= 0)
    return pkv_fail(PKV_ERR_INVALID_ARG, "paged_kv_write: negative or zero size (T=%lld, Hkv=%d, D=%d)",
                    (long long)T, Hkv, D);
  if (dt != PKV_F32 && dt != PKV_BF16 && dt != PKV_F16)
    return pkv_fail(PKV_ERR_UNSUPPORTED, "paged_kv_write: unknown dtype %d", (int)dt);
  if (T == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !key_pool || !value_pool)
    return pkv_fail(PKV_ERR_INVALID_ARG, "paged_kv_write: NULL pointer");
  const int64_t row_bytes = (int64_t)Hkv * D * pkv_dtype_size(dt);
  if (row_bytes % 16 || !aligned16(k) || !aligned16(v) || !aligned16(key_pool) || !aligned16(value_pool))
    return pkv_fail(PKV_ERR_INVALID_ARG, "paged_kv_write: rows (%lld bytes) and base pointers must be 16-byte aligned",
                    (long long)row_bytes);
  if (row_bytes / 16 > (1 << 30)) return pkv_fail(PKV_ERR_UNSUPPORTED, "paged_kv_write: row too large");
  const int check = (flags & PKV_CHECK_BOUNDS) ? 1 : 0;
  unsigned int* err = check ? pkv_device_error_word() : nullptr;
  if (check && !err) return pkv_fail(PKV_ERR_CUDA, "paged_kv_write: device error word unavailable");
  const int rc = pkv_launch_kv_write(k, v, slot_mapping, T, key_pool, value_pool, num_slots, (int)row_bytes, err,
                                     check, stream);
  if (rc != 0) return pkv_fail(PKV_ERR_CUDA, "paged_kv_write: launch failed: %s", cudaGetErrorString((cudaError_t)rc));
  pkv_set_launches(1);
  return PKV_OK;
}

extern "C" pkv_status paged_kv_gather(const void* key_pool, const void* value_pool, int64_t num_blocks,
                                      const int32_t* block_table, int B, int W, int first_block, int n_blocks,
                                      void* stage_k, void* stage_v, int64_t stage_rows, int Hkv, int D, pkv_dtype dt,
                                      uint32_t flags, void* stream) {
  pkv_clear_error();
  pkv_set_launches(0);
  if (B < 0 || W < 0 || first_block < 0 || n_blocks < 0 || num_blocks < 0 || stage_rows < 0 || Hkv <= 0 || D <= 0)
    return pkv_fail(PKV_ERR_INVALID_ARG, "paged_kv_gather: negative or zero size");
  if (dt != PKV_F32 && dt != PKV_BF16 && dt != PKV_F16)
    return pkv_fail(PKV_ERR_UNSUPPORTED, "paged_kv_gather: unknown dtype %d", (int)dt);
  if ((int64_t)first_block + n_blocks > W)
    return pkv_fail(PKV_ERR_INVALID_ARG, "paged_kv_gather: blocks [%d, %d) run past the table width %d", first_block,
                    first_block + n_blocks, W);
  if (((int64_t)first_block + n_blocks) * 16 > stage_rows)
    return pkv_fail(PKV_ERR_INVALID_ARG, "paged_kv_gather: %d blocks do not fit %lld staging rows",
                    first_block + n_blocks, (long long)stage_rows);
  if ((int64_t)B * n_blocks * 32 >= ((int64_t)1 << 31))
    return pkv_fail(PKV_ERR_INVALID_ARG, "paged_kv_gather: %d rows x %d blocks is too many for one call", B, n_blocks);
  if (B == 0 || n_blocks == 0) return PKV_OK;
  if (!key_pool || !value_pool || !block_table || !stage_k || !stage_v)
    return pkv_fail(PKV_ERR_INVALID_ARG, "paged_kv_gather: NULL pointer");
  const int64_t row_bytes = (int64_t)Hkv * D * pkv_dtype_size(dt);
  if (row_bytes % 16 || !aligned16(key_pool) || !aligned16(value_pool) || !aligned16(stage_k) || !aligned16(stage_v))
    return pkv_fail(PKV_ERR_INVALID_ARG, "paged_kv_gather: rows and base pointers must be 16-byte aligned");
  const int check = (flags & PKV_CHECK_BOUNDS) ? 1 : 0;
  unsigned int* err = check ? pkv_device_error_word() : nullptr;
  if (check && !err) return pkv_fail(PKV_ERR_CUDA, "paged_kv_gather: device error word unavailable");
  const int rc = pkv_launch_kv_gather(key_pool, value_pool, num_blocks, block_table, B, W, first_block, n_blocks,
                                      stage_k, stage_v, stage_rows, (int)row_bytes, err, check, stream);
  if (rc != 0) return pkv_fail(PKV_ERR_CUDA, "paged_kv_gather: launch failed: %s", cudaGetErrorString((cudaError_t)rc));
  pkv_set_launches(1);
  return PKV_OK;
}

namespace {

struct SplitPlan {
  int splits;      // key-range splits of each split item (1: no split)
  int64_t direct;  // items run whole before the split ones
};

// Split the key range only where the grid would otherwise leave SMs idle: the items of the
// last, partly filled wave.  `items` = CTAs of the unsplit launch, `tiles` = key tiles per item,
// `sms` = CTAs that run at once.  The `full` whole waves run unsplit; the `tail` items after
// them split s ways, with s chosen to minimise the tail's time in key tiles: its waves, each
// taking one split's tiles plus a CTA's fixed cost (prologue, epilogue, partial store: about 8
// tiles' time), plus the combine at about 0.3 tiles per split.  Fit to one row x 8 heads x 256
// queries over 26520 keys: 354 / 193 / 113 / 73 / 61 us for 1 / 2 / 4 / 8 / 16 splits.  (Splitting
// every item of a full grid only adds fixed costs: 2 splits cost +8 % on the long-window workload.)
// The CUDA-core kernel uses the same estimate; its fixed cost is well under one of its slower
// 64-key tiles, so the estimate errs towards fewer splits there.
SplitPlan plan_splits(int64_t items, int64_t tiles, int sms, int max_splits) {
  const SplitPlan none{1, items};
  if (items <= 0 || tiles <= 1 || sms <= 0) return none;
  const int64_t full = items / sms;
  const int64_t tail = items - full * sms;
  if (tail == 0) return none;
  int best = 1;
  double best_cost = (double)(tiles + 8);
  for (int s = 2; s <= max_splits; ++s) {
    const int64_t per = (tiles + s - 1) / s;
    if (per < 4) break;  // too little work per split
    const int64_t waves = (tail * s + sms - 1) / sms;
    const double cost = (double)waves * (double)(per + 8) + 0.3 * s;
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best > 1 ? SplitPlan{best, full * sms} : none;
}

}  // namespace

// Key-range splits the call plans from host-visible sizes.  An item is what one CTA of the
// unsplit launch covers: 256 queries of one (row, head) for the tensor-core kernel, 128 for the
// CUDA-core one.  Both kernels split only the tail behind whole waves (every item when there
// are fewer items than CTA slots).  The CUDA-core kernel's tail runs as a one-dimensional grid,
// whose size must stay a valid grid dimension.
static SplitPlan planned_splits(int B, int Hq, int max_query_len, int max_seq_len, bool tc, int sms) {
  const int64_t q_unit = tc ? kTcItemRows : kSimtItemRows;
  const int64_t k_tile = tc ? 128 : kSimtKeyTile;
  const int64_t items = (int64_t)B * Hq * ((max_query_len + q_unit - 1) / q_unit);
  const int64_t tiles = ((int64_t)max_seq_len + k_tile - 1) / k_tile;
  SplitPlan p = plan_splits(items, tiles, tc ? sms : sms * kSimtCtasPerSm, kMaxSplits);
  if (!tc && p.direct > 0 && p.direct + (items - p.direct) * p.splits > 0x7fffffff) p = SplitPlan{1, items};
  return p;
}

extern "C" size_t paged_attn_workspace_size(int64_t Tq, int Hq, int D, int B, int max_query_len, int max_seq_len) {
  if (Tq <= 0 || Hq <= 0 || D <= 0) return 0;
  int sms = pkv_sm_count();
  if (sms <= 0) sms = 152;
  int splits = kWorkspaceSplits;
  for (int tc = 0; tc < 2; ++tc) {
    const int s = planned_splits(B, Hq, max_query_len, max_seq_len, tc == 1, sms).splits;
    splits = s > splits ? s : splits;
  }
  return (size_t)splits * (size_t)Tq * (size_t)Hq * ((size_t)D + 1) * sizeof(float);
}

namespace {

struct FusedWrite {
  const void* k;
  const void* v;
  const int64_t* slots;
};

pkv_status attn_impl(const char* fn, const void* q, int64_t Tq, int Hq, const void* key_pool, const void* value_pool,
                     int64_t num_blocks, int block_size, int Hkv, int D, pkv_dtype dt, const int32_t* block_table,
                     int B, int W, const int32_t* query_start_loc, const int32_t* seq_lens, int max_query_len,
                     int max_seq_len, float softmax_scale, const pkv_segment* segs, const int32_t* seg_start,
                     void* out, void* workspace, size_t ws_bytes, uint32_t flags, void* stream, const FusedWrite* fw) {
  pkv_clear_error();
  pkv_set_launches(0);
  pkv_set_split_plan(1, 0);
  if (Tq < 0 || B < 0 || W < 0 || max_query_len < 0 || max_seq_len < 0 || num_blocks < 0)
    return pkv_fail(PKV_ERR_INVALID_ARG, "%s: negative size", fn);
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv)
    return pkv_fail(PKV_ERR_INVALID_ARG,
                    "%s: num_heads must be a positive multiple of num_kv_heads (Hq=%d, Hkv=%d)", fn, Hq, Hkv);
  if (block_size != 16) return pkv_fail(PKV_ERR_UNSUPPORTED, "%s: block_size must be 16 (got %d)", fn, block_size);
  if (D != 64 && D != 128) return pkv_fail(PKV_ERR_UNSUPPORTED, "%s: head dim must be 64 or 128 (got %d)", fn, D);
  if (dt != PKV_F32 && dt != PKV_BF16 && dt != PKV_F16)
    return pkv_fail(PKV_ERR_UNSUPPORTED, "%s: unknown dtype %d", fn, (int)dt);
  if (!isfinite(softmax_scale)) return pkv_fail(PKV_ERR_INVALID_ARG, "%s: softmax_scale is not finite", fn);
  // The tensor-core kernel keeps its running maximum for a positive scale only; the CUDA-core kernel,
  // about 50 times slower on bf16, takes any scale, but only when asked for by name.
  if (dt != PKV_F32 && !(softmax_scale > 0.f) && !(flags & PKV_FORCE_SIMT))
    return pkv_fail(PKV_ERR_UNSUPPORTED,
                    "%s: a bf16/f16 call needs softmax_scale > 0 (got %g); pass PKV_FORCE_SIMT to run it on the "
                    "CUDA-core kernel", fn, (double)softmax_scale);
  if ((int64_t)max_seq_len > (int64_t)W * block_size)
    return pkv_fail(PKV_ERR_INVALID_ARG, "%s: max_seq_len %d exceeds the table's %d x %d slots", fn,
                    max_seq_len, W, block_size);
  if (Tq == 0 || B == 0 || max_query_len == 0) return PKV_OK;
  if (!q || !key_pool || !value_pool || !block_table || !query_start_loc || !seq_lens || !out)
    return pkv_fail(PKV_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (segs && !seg_start) return pkv_fail(PKV_ERR_INVALID_ARG, "%s: segs given without seg_start", fn);
  if (!aligned16(q) || !aligned16(key_pool) || !aligned16(value_pool) || !aligned16(out))
    return pkv_fail(PKV_ERR_INVALID_ARG, "%s: q, pools and out must be 16-byte aligned", fn);
  if (max_query_len > max_seq_len)
    return pkv_fail(PKV_ERR_INVALID_ARG, "%s: max_query_len %d > max_seq_len %d (the query is a "
                    "suffix of the key sequence)", fn, max_query_len, max_seq_len);

  PkvAttnArgs a{};
  a.q = q;
  a.k_pool = key_pool;
  a.v_pool = value_pool;
  a.out = out;
  a.block_table = block_table;
  a.query_start_loc = query_start_loc;
  a.seq_lens = seq_lens;
  a.segs = segs;
  a.seg_start = seg_start;
  a.num_blocks = num_blocks;
  a.Tq = Tq;
  a.B = B;
  a.W = W;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.max_query_len = max_query_len;
  a.max_seq_len = max_seq_len;
  a.scale = softmax_scale;
  a.check = (flags & PKV_CHECK_BOUNDS) ? 1 : 0;
  a.contiguous = (flags & PKV_CONTIGUOUS_KV) ? 1 : 0;
  // The error word is always passed: the tensor-core kernel reports pipeline timeouts through it.
  a.err = pkv_device_error_word();
  if (!a.err) return pkv_fail(PKV_ERR_CUDA, "%s: device error word unavailable", fn);

  // (The tensor-core launcher also declines a non-positive scale; plan for the kernel that runs.)
  const bool use_tc = !(flags & PKV_FORCE_SIMT) && pkv_attn_tc_supports(dt, D) && softmax_scale > 0.f;
  int sms = pkv_sm_count();
  if (sms <= 0) sms = 152;

  // Split planning from host-visible sizes only.
  int forced = (int)((flags >> 8) & 0xffu);
  int splits = 1;
  int64_t direct = 0;
  if (forced > 0) {
    splits = forced > kMaxSplits ? kMaxSplits : forced;
  } else if (!(flags & PKV_NO_SPLIT) && workspace && ws_bytes) {
    const SplitPlan plan = planned_splits(B, Hq, max_query_len, max_seq_len, use_tc, sms);
    splits = plan.splits;
    direct = plan.direct;
    // A planned split count the workspace cannot hold shrinks to what it can.
    const size_t per_split = (size_t)Tq * Hq * ((size_t)D + 1) * sizeof(float);
    const size_t fits = per_split ? ws_bytes / per_split : 0;
    if ((size_t)splits > fits) splits = fits > 1 ? (int)fits : 1;
  }
  if (splits > 1) {
    const size_t need = (size_t)splits * (size_t)Tq * Hq * ((size_t)D + 1) * sizeof(float);
    if (!workspace || ws_bytes < need) {
      if (forced > 0)
        return pkv_fail(PKV_ERR_CAPACITY, "%s: %d splits need %zu workspace bytes, got %zu", fn, splits,
                        need, ws_bytes);
      splits = 1;
    } else {
      if (!aligned16(workspace)) return pkv_fail(PKV_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", fn);
      a.part_o = (float*)workspace;
      a.part_lse = a.part_o + (size_t)splits * Tq * Hq * D;
    }
  }
  a.num_splits = splits;
  a.split_direct = splits > 1 ? (int)direct : 0;
  pkv_set_split_plan(splits, splits > 1 ? direct : (int64_t)0);
  if (fw) {
    if (!fw->k || !fw->v || !fw->slots) return pkv_fail(PKV_ERR_INVALID_ARG, "%s: NULL k, v or slot_mapping", fn);
    if (!aligned16(fw->k) || !aligned16(fw->v))
      return pkv_fail(PKV_ERR_INVALID_ARG, "%s: k and v must be 16-byte aligned", fn);
    a.k_new = fw->k;
    a.v_new = fw->v;
    a.slots = fw->slots;
    a.num_slots = num_blocks * block_size;
  }

  int rc = -1;
  if (use_tc) rc = pkv_launch_attn_tc(a, dt, stream);
  if (rc == -1) {
    // Planned for the tensor-core kernel, which declined: the CUDA-core kernel splits every item
    // instead (its combine then merges every row).  Planned for the CUDA-core kernel: its own tail.
    if (use_tc) {
      a.split_direct = 0;
      pkv_set_split_plan(splits, 0);
    }
    a.simt_items = 1;
    rc = pkv_launch_attn_simt(a, dt, stream);
  }
  if (rc != 0) return pkv_fail(PKV_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString((cudaError_t)rc));
  if (splits > 1) {
    rc = pkv_launch_attn_combine(a, dt, stream);
    if (rc != 0)
      return pkv_fail(PKV_ERR_CUDA, "%s: combine launch failed: %s", fn, cudaGetErrorString((cudaError_t)rc));
  }
  pkv_set_launches(splits > 1 ? 2 : 1);
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status paged_attn_varlen(const void* q, int64_t Tq, int Hq, const void* key_pool,
                                        const void* value_pool, int64_t num_blocks, int block_size, int Hkv, int D,
                                        pkv_dtype dt, const int32_t* block_table, int B, int W,
                                        const int32_t* query_start_loc, const int32_t* seq_lens, int max_query_len,
                                        int max_seq_len, float softmax_scale, const pkv_segment* segs,
                                        const int32_t* seg_start, void* out, void* workspace, size_t ws_bytes,
                                        uint32_t flags, void* stream) {
  return attn_impl("paged_attn_varlen", q, Tq, Hq, key_pool, value_pool, num_blocks, block_size, Hkv, D, dt,
                   block_table, B, W, query_start_loc, seq_lens, max_query_len, max_seq_len, softmax_scale, segs,
                   seg_start, out, workspace, ws_bytes, flags, stream, nullptr);
}

extern "C" pkv_status paged_kv_write_attn(const void* q, const void* k, const void* v, const int64_t* slot_mapping,
                                          int64_t Tq, int Hq, void* key_pool, void* value_pool, int64_t num_blocks,
                                          int block_size, int Hkv, int D, pkv_dtype dt, const int32_t* block_table,
                                          int B, int W, const int32_t* query_start_loc, const int32_t* seq_lens,
                                          int max_query_len, int max_seq_len, float softmax_scale,
                                          const pkv_segment* segs, const int32_t* seg_start, void* out,
                                          void* workspace, size_t ws_bytes, uint32_t flags, void* stream) {
  const FusedWrite fw{k, v, slot_mapping};
  return attn_impl("paged_kv_write_attn", q, Tq, Hq, key_pool, value_pool, num_blocks, block_size, Hkv, D, dt,
                   block_table, B, W, query_start_loc, seq_lens, max_query_len, max_seq_len, softmax_scale, segs,
                   seg_start, out, workspace, ws_bytes, flags, stream, &fw);
}
