// One layer's forward through the C ABI alone -- no Python, no torch types: host metadata from the
// library's own functions, device memory from cudaMalloc, the fused write + attention call, the
// device error word read back with pkv_check.  Then the same layer's attention again through
// paged_attn_varlen_noalloc (the pools now hold the chunk), as a caller without an allocator would
// run it: no workspace, the library's fixed scratch.
//
// usage: abi_forward <dir>
//   <dir>/params.txt   B Hq Hkv D pool_blocks chunk sink window action_len history query_tokens n_spans
//                      then n_spans pairs (span start, end), all whitespace-separated integers
//   <dir>/row_blocks.i32      B x ceil((history + query_tokens) / 16) physical blocks (video, per row)
//   <dir>/action_blocks.i32   B x ceil(action_len / 16) scratch blocks (per row), absent when action_len = 0
//   <dir>/q.bf16, k_hist.bf16, v_hist.bf16, k_cur.bf16, v_cur.bf16   raw bf16 (see the sizes below)
// writes <dir>/out.bf16 (fused call) and <dir>/out_noalloc.bf16: [B * (query_tokens + action_len), Hq, D]
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <fstream>
#include <string>
#include <vector>

#include "pagedkv.h"

namespace {

template <typename T>
std::vector<T> read_all(const std::string& path, size_t count) {
  std::vector<T> v(count);
  std::ifstream f(path, std::ios::binary);
  if (!f || !f.read(reinterpret_cast<char*>(v.data()), (std::streamsize)(count * sizeof(T)))) {
    std::fprintf(stderr, "cannot read %zu items from %s\n", count, path.c_str());
    std::exit(2);
  }
  return v;
}

#define CHECK_PKV(call)                                                                        \
  do {                                                                                         \
    const pkv_status st_ = (call);                                                             \
    if (st_ != PKV_OK) {                                                                       \
      std::fprintf(stderr, "%s failed (%d): %s\n", #call, (int)st_, pkv_last_error());        \
      std::exit(3);                                                                            \
    }                                                                                          \
  } while (0)

#define CHECK_CUDA(call)                                                                       \
  do {                                                                                         \
    const cudaError_t e_ = (call);                                                             \
    if (e_ != cudaSuccess) {                                                                   \
      std::fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));                  \
      std::exit(4);                                                                            \
    }                                                                                          \
  } while (0)

template <typename T>
T* to_device(const std::vector<T>& h) {
  T* d = nullptr;
  CHECK_CUDA(cudaMalloc(&d, h.size() * sizeof(T) + 16));
  if (!h.empty()) CHECK_CUDA(cudaMemcpy(d, h.data(), h.size() * sizeof(T), cudaMemcpyHostToDevice));
  return d;
}

}  // namespace

int main(int argc, char** argv) {
  if (argc != 2) {
    std::fprintf(stderr, "usage: %s <dir>\n", argv[0]);
    return 1;
  }
  const std::string dir = argv[1];
  std::ifstream pf(dir + "/params.txt");
  int64_t B, Hq, Hkv, D, pool_blocks, chunk, sink, window, action_len, history, query_tokens, n_spans;
  pf >> B >> Hq >> Hkv >> D >> pool_blocks >> chunk >> sink >> window >> action_len >> history >> query_tokens >> n_spans;
  std::vector<int32_t> spans(2 * n_spans);
  for (auto& x : spans) pf >> x;
  if (!pf) {
    std::fprintf(stderr, "bad params.txt\n");
    return 2;
  }
  const int bs = 16;
  const int64_t end_tokens = history + query_tokens;
  const int64_t n_video = (end_tokens + bs - 1) / bs, n_action = (action_len + bs - 1) / bs;
  const int64_t q_len = query_tokens + action_len, Tq = B * q_len;
  auto row_blocks = read_all<int32_t>(dir + "/row_blocks.i32", (size_t)(B * n_video));
  std::vector<int32_t> action_blocks;
  if (action_len) action_blocks = read_all<int32_t>(dir + "/action_blocks.i32", (size_t)(B * n_action));
  auto q = read_all<uint16_t>(dir + "/q.bf16", (size_t)(Tq * Hq * D));
  auto k_hist = read_all<uint16_t>(dir + "/k_hist.bf16", (size_t)(B * history * Hkv * D));
  auto v_hist = read_all<uint16_t>(dir + "/v_hist.bf16", (size_t)(B * history * Hkv * D));
  auto k_cur = read_all<uint16_t>(dir + "/k_cur.bf16", (size_t)(Tq * Hkv * D));
  auto v_cur = read_all<uint16_t>(dir + "/v_cur.bf16", (size_t)(Tq * Hkv * D));

  // Host metadata, all from the library: visible window -> padded table row, slots, segments.
  const int64_t W = pkv_table_width(chunk, sink, window, action_len, bs);
  if (W < 0) {
    std::fprintf(stderr, "pkv_table_width: %s\n", pkv_last_error());
    return 3;
  }
  std::vector<int32_t> table((size_t)(B * W)), seq_lens((size_t)B), qsl((size_t)B + 1, 0), seg_start(1, 0);
  std::vector<int64_t> slots((size_t)Tq), hist_slots((size_t)(B * history));
  std::vector<pkv_segment> segs;
  for (int64_t b = 0; b < B; ++b) {
    const int32_t* rb = row_blocks.data() + b * n_video;
    std::vector<int32_t> vis((size_t)n_video);
    int64_t n_vis = 0, video_len = 0;
    CHECK_PKV(pkv_visible_window(rb, n_video, end_tokens, sink, window, bs, vis.data(), n_video, &n_vis, &video_len));
    int64_t kv_len = 0;
    const int32_t* ab = action_len ? action_blocks.data() + b * n_action : nullptr;
    CHECK_PKV(pkv_block_table_row(vis.data(), n_vis, video_len, ab, action_len, bs, W, table.data() + b * W, &kv_len));
    seq_lens[(size_t)b] = (int32_t)kv_len;
    qsl[(size_t)b + 1] = qsl[(size_t)b] + (int32_t)q_len;
    CHECK_PKV(pkv_slot_mapping(rb, n_video, history, query_tokens, bs, slots.data() + b * q_len));
    if (action_len) CHECK_PKV(pkv_slot_mapping(ab, n_action, 0, action_len, bs, slots.data() + b * q_len + query_tokens));
    if (history) CHECK_PKV(pkv_slot_mapping(rb, n_video, 0, history, bs, hist_slots.data() + b * history));
    std::vector<pkv_segment> row(2 * (size_t)n_spans + 1);
    int n_out = 0;
    CHECK_PKV(build_segments(spans.data(), (int)n_spans, (int32_t)(kv_len - q_len), (int32_t)q_len, (int32_t)kv_len,
                             row.data(), (int)row.size(), &n_out));
    segs.insert(segs.end(), row.begin(), row.begin() + n_out);
    seg_start.push_back((int32_t)segs.size());
  }

  // Device memory from cudaMalloc; the library only reads and writes it.
  const int64_t num_slots = pool_blocks * bs;
  const size_t pool_bytes = (size_t)(num_slots * Hkv * D) * sizeof(uint16_t);
  void *kp = nullptr, *vp = nullptr, *out = nullptr;
  CHECK_CUDA(cudaMalloc(&kp, pool_bytes));
  CHECK_CUDA(cudaMalloc(&vp, pool_bytes));
  CHECK_CUDA(cudaMalloc(&out, (size_t)(Tq * Hq * D) * sizeof(uint16_t)));
  uint16_t *d_q = to_device(q), *d_kh = to_device(k_hist), *d_vh = to_device(v_hist), *d_kc = to_device(k_cur),
           *d_vc = to_device(v_cur);
  int32_t *d_table = to_device(table), *d_seq = to_device(seq_lens), *d_qsl = to_device(qsl),
          *d_seg_start = to_device(seg_start);
  int64_t *d_slots = to_device(slots), *d_hist_slots = to_device(hist_slots);
  pkv_segment* d_segs = to_device(segs);
  const size_t ws_bytes = paged_attn_workspace_size(Tq, (int)Hq, (int)D, (int)B, (int)q_len, (int)(W * bs));
  void* ws = nullptr;
  if (ws_bytes) CHECK_CUDA(cudaMalloc(&ws, ws_bytes));

  // Earlier forwards' history, then this forward's layer: write + attention in one launch.
  for (int64_t b = 0; b < B && history; ++b)
    CHECK_PKV(paged_kv_write(d_kh + b * history * Hkv * D, d_vh + b * history * Hkv * D, d_hist_slots + b * history,
                             history, kp, vp, num_slots, (int)Hkv, (int)D, PKV_BF16, PKV_CHECK_BOUNDS, nullptr));
  CHECK_PKV(paged_kv_write_attn(d_q, d_kc, d_vc, d_slots, Tq, (int)Hq, kp, vp, pool_blocks, bs, (int)Hkv, (int)D,
                                PKV_BF16, d_table, (int)B, (int)W, d_qsl, d_seq, (int)q_len, (int)(W * bs),
                                1.0f / std::sqrt((float)D), d_segs, d_seg_start, out, ws, ws_bytes, PKV_CHECK_BOUNDS,
                                nullptr));
  uint32_t bits = 0;
  CHECK_PKV(pkv_check(nullptr, &bits));
  std::vector<uint16_t> h_out((size_t)(Tq * Hq * D));
  CHECK_CUDA(cudaMemcpy(h_out.data(), out, h_out.size() * sizeof(uint16_t), cudaMemcpyDeviceToHost));
  std::ofstream of(dir + "/out.bf16", std::ios::binary);
  of.write(reinterpret_cast<const char*>(h_out.data()), (std::streamsize)(h_out.size() * sizeof(uint16_t)));
  const int launches = pkv_last_launches();

  // The attention alone, allocation-free: split partials (if any) in the library's fixed scratch.
  CHECK_CUDA(cudaMemset(out, 0, h_out.size() * sizeof(uint16_t)));
  CHECK_PKV(paged_attn_varlen_noalloc(d_q, Tq, (int)Hq, kp, vp, pool_blocks, bs, (int)Hkv, (int)D, PKV_BF16, d_table,
                                      (int)B, (int)W, d_qsl, d_seq, (int)q_len, (int)(W * bs),
                                      1.0f / std::sqrt((float)D), d_segs, d_seg_start, out, PKV_CHECK_BOUNDS,
                                      nullptr));
  const int launches_noalloc = pkv_last_launches();
  uint32_t bits_noalloc = 0;
  CHECK_PKV(pkv_check(nullptr, &bits_noalloc));
  CHECK_CUDA(cudaMemcpy(h_out.data(), out, h_out.size() * sizeof(uint16_t), cudaMemcpyDeviceToHost));
  std::ofstream of2(dir + "/out_noalloc.bf16", std::ios::binary);
  of2.write(reinterpret_cast<const char*>(h_out.data()), (std::streamsize)(h_out.size() * sizeof(uint16_t)));
  std::printf("abi_forward: %s, %lld tokens x %lld heads, launches %d, device bits 0x%x; noalloc launches %d, "
              "device bits 0x%x\n",
              pkv_version(), (long long)Tq, (long long)Hq, launches, bits, launches_noalloc, bits_noalloc);
  return 0;
}
