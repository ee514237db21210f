// CUDA-core paged attention (fp32 arithmetic throughout) and the split-KV combine.
//
// This is the kernel for fp32 inputs, where tensor-core tf32 would not meet a
// 1e-4 tolerance, and for shapes the tcgen05 kernel does not take.  It computes
// what _reference_paged_attention (paged_attention.py) computes -- gather each
// key through the block table, softmax(scale * q.k) over the visible keys,
// weighted sum of values -- with the piecewise causal/full mask of
// piecewise_attn.py expressed as a per-query key limit, and an online
// (running max / running sum) softmax so the key range can be streamed.
//
// CTA = 16 queries of one (row, head) and one key-range split; 4 warps, each
// owning 4 queries; keys staged 32 at a time in shared memory as fp32.

#include <math.h>

#include <type_traits>

#include "kv_copy.cuh"

namespace {

constexpr int kQT = 16;      // queries per CTA
constexpr int kKT = 32;      // keys per shared-memory tile
constexpr int kWarps = 4;
constexpr int kRowsPerWarp = kQT / kWarps;

template <typename T>
PKV_DEVINLINE void load_row_f32(const T* __restrict__ src, float* dst, int D, int lane_in_group, int group_size) {
  for (int d = lane_in_group; d < D; d += group_size) dst[d] = pkv_to_f32<T>(src[d]);
}

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) attn_simt_kernel(PkvAttnArgs a) {
  __shared__ float q_s[kQT][D];
  __shared__ float k_s[kKT][D + 1];
  __shared__ float v_s[kKT][D];
  __shared__ int lim_s[kQT];
  __shared__ int kv_hi_s;

  const int tiles_per_row = (a.max_query_len + kQT - 1) / kQT;
  const int b = blockIdx.x / tiles_per_row;
  const int tile = blockIdx.x % tiles_per_row;
  const int h = blockIdx.y;
  const int split = blockIdx.z;
  const int kvh = h / (a.Hq / a.Hkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int q0 = a.query_start_loc[b];
  const int q1 = a.query_start_loc[b + 1];
  int Sq = q1 - q0;
  int L = a.seq_lens[b];
  if (a.check) {
    int lmax = a.W * 16 < a.max_seq_len ? a.W * 16 : a.max_seq_len;
    if (Sq < 0 || Sq > a.max_query_len) {
      if (tid == 0 && tile == 0 && h == 0 && split == 0) pkv_raise(a.err, PKV_DEVERR_QUERY);
      Sq = Sq < 0 ? 0 : (Sq > a.max_query_len ? a.max_query_len : Sq);
    }
    if (L > lmax || L < Sq || L < 0) {
      if (tid == 0 && tile == 0 && h == 0 && split == 0) pkv_raise(a.err, PKV_DEVERR_SEQLEN);
      L = L > lmax ? lmax : (L < 0 ? 0 : L);
    }
  }
  // Fused call: this CTA's share of the slot-mapping scatter, before its attention work.  The
  // attention below reads the keys of the queries' own positions from the new tokens, so no CTA
  // depends on the write.
  if (a.k_new) {
    const int64_t cta = ((int64_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    pkv_scatter((const uint4*)a.k_new, (const uint4*)a.v_new, a.slots, a.Tq, (uint4*)a.k_pool, (uint4*)a.v_pool,
                a.num_slots, a.Hkv * D * (int)sizeof(T) / 16, a.err, a.check, cta * kWarps + warp,
                (int64_t)gridDim.x * gridDim.y * gridDim.z * kWarps, lane, &a);
  }
  const int i0 = tile * kQT;
  if (i0 >= Sq) return;

  // Per-query key limits from the row's segments.
  if (tid < kQT) {
    const int i = i0 + tid;
    int lim = 0;
    if (i < Sq) {
      bool uncovered = false;
      int s_begin = 0, s_end = 0;
      if (a.segs) {
        s_begin = a.seg_start[b];
        s_end = a.seg_start[b + 1];
      }
      const int base = pkv_query_base(L, Sq, a.segs, s_begin, s_end);
      lim = pkv_row_limit(base + i, L, a.segs, s_begin, s_end, &uncovered);
      if (a.check && (uncovered || base < 0 || base + Sq > L)) pkv_raise(a.err, PKV_DEVERR_SEGMENT);
    }
    lim_s[tid] = lim;
  }
  // Query tile, fp32 in shared memory.
  for (int e = tid; e < kQT * D; e += blockDim.x) {
    const int r = e / D, d = e % D;
    const int i = i0 + r;
    q_s[r][d] = i < Sq ? pkv_to_f32<T>(((const T*)a.q)[((int64_t)(q0 + i) * a.Hq + h) * D + d]) : 0.f;
  }
  __syncthreads();
  if (tid == 0) {
    int hi = 0;
    for (int r = 0; r < kQT; ++r) hi = lim_s[r] > hi ? lim_s[r] : hi;
    kv_hi_s = hi;
  }
  __syncthreads();
  const int kv_hi = kv_hi_s;

  // This split's range of key tiles.
  const int n_tiles = (kv_hi + kKT - 1) / kKT;
  const int per = (n_tiles + a.num_splits - 1) / a.num_splits;
  const int t_begin = split * per;
  const int t_end = min(n_tiles, t_begin + per);

  constexpr int kDL = D / 32;  // accumulator columns per lane
  float acc[kRowsPerWarp][kDL];
  float m[kRowsPerWarp], l[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < kDL; ++c) acc[r][c] = 0.f;
  }

  const T* kpool = (const T*)a.k_pool;
  const T* vpool = (const T*)a.v_pool;
  // Keys at the queries' own positions [cb, ce): read from the new tokens in a fused call.
  int cb = 0, ce = 0;
  if (a.k_new) {
    int s_begin = 0, s_end = 0;
    if (a.segs) {
      s_begin = a.seg_start[b];
      s_end = a.seg_start[b + 1];
    }
    cb = pkv_query_base(L, Sq, a.segs, s_begin, s_end);
    ce = cb + Sq;
  }
  for (int kt = t_begin; kt < t_end; ++kt) {
    const int j0 = kt * kKT;
    __syncthreads();
    // Gather 32 keys/values through the block table; 4 threads per key row.
    {
      const int jj = tid >> 2, part = tid & 3;
      const int j = j0 + jj;
      if (j < kv_hi && j >= cb && j < ce) {
        const int64_t tok = (int64_t)q0 + (j - cb);
        load_row_f32<T>((const T*)a.k_new + (tok * a.Hkv + kvh) * D, k_s[jj], D, part, 4);
        load_row_f32<T>((const T*)a.v_new + (tok * a.Hkv + kvh) * D, v_s[jj], D, part, 4);
      } else if (j < kv_hi) {
        int blk = a.block_table[(int64_t)b * a.W + (j >> 4)];
        if (a.check && (blk < 0 || blk >= a.num_blocks)) {
          pkv_raise(a.err, PKV_DEVERR_BLOCK);
          blk = 0;
        }
        const int64_t row = (int64_t)blk * 16 + (j & 15);
        const T* ksrc = kpool + (row * a.Hkv + kvh) * D;
        const T* vsrc = vpool + (row * a.Hkv + kvh) * D;
        load_row_f32<T>(ksrc, k_s[jj], D, part, 4);
        load_row_f32<T>(vsrc, v_s[jj], D, part, 4);
      } else {
        for (int d = part; d < D; d += 4) {
          k_s[jj][d] = 0.f;
          v_s[jj][d] = 0.f;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int qr = warp * kRowsPerWarp + r;
      const int lim = lim_s[qr];
      const int j = j0 + lane;
      float s = -INFINITY;
      if (j < lim) {
        float dot = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; ++d) dot = fmaf(q_s[qr][d], k_s[lane][d], dot);
        s = dot * a.scale;
      }
      float tmax = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_new = fmaxf(m[r], tmax);
      if (m_new == -INFINITY) continue;  // nothing visible yet for this query
      const float p = j < lim ? expf(s - m_new) : 0.f;
      const float alpha = expf(m[r] - m_new);  // exp(-inf) = 0 on the first visible tile
      float psum = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l[r] = l[r] * alpha + psum;
      m[r] = m_new;
#pragma unroll
      for (int c = 0; c < kDL; ++c) acc[r][c] *= alpha;
      for (int jj = 0; jj < kKT; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int c = 0; c < kDL; ++c) acc[r][c] = fmaf(pj, v_s[jj][lane + 32 * c], acc[r][c]);
      }
    }
  }

  // Epilogue: normalised output, or partial output + log-sum-exp per split.
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = i0 + warp * kRowsPerWarp + r;
    if (i >= Sq) continue;
    const int64_t tok = q0 + i;
    const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
    if (a.num_splits == 1) {
      T* o = (T*)a.out + (tok * a.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < kDL; ++c) o[lane + 32 * c] = pkv_from_f32<T>(acc[r][c] * inv);
    } else {
      float* o = a.part_o + (((int64_t)split * a.Tq + tok) * a.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < kDL; ++c) o[lane + 32 * c] = acc[r][c] * inv;
      if (lane == 0)
        a.part_lse[((int64_t)split * a.Tq + tok) * a.Hq + h] = l[r] > 0.f ? m[r] + logf(l[r]) : -INFINITY;
    }
  }
}

// NC consecutive output values of one lane, rounded to T (one 4-, 8- or 16-byte store).
template <typename T, int NC>
PKV_DEVINLINE void store_lane(T* dst, const float* v) {
  if constexpr (sizeof(T) == 4) {
    if constexpr (NC == 4)
      *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
    else
      *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
  } else {
    uint32_t p[NC / 2];
#pragma unroll
    for (int e = 0; e < NC / 2; ++e) {
      const T lo = pkv_from_f32<T>(v[2 * e]), hi = pkv_from_f32<T>(v[2 * e + 1]);
      p[e] = (uint32_t)(*reinterpret_cast<const uint16_t*>(&lo)) |
             ((uint32_t)(*reinterpret_cast<const uint16_t*>(&hi)) << 16);
    }
    if constexpr (NC == 4)
      *reinterpret_cast<uint2*>(dst) = make_uint2(p[0], p[1]);
    else
      *reinterpret_cast<uint32_t*>(dst) = p[0];
  }
}

// One (token, head) row by one warp: O = sum_s exp(lse_s - M) O_s / sum_s exp(lse_s - M).  Lane l
// holds columns [l NC, l NC + NC) (NC = D / 32) and reads them as one vector per split; lane s reads
// split s's log-sum-exp (at most 32 splits).  The first eight splits' rows are loaded together with
// the log-sum-exps, so a row with up to eight splits costs one round trip to memory.
template <typename T, int NC>
PKV_DEVINLINE void combine_row(const PkvAttnArgs& a, int64_t item, int lane) {
  using V = typename std::conditional<NC == 4, float4, float2>::type;
  const int S = a.num_splits;
  const int64_t stride = a.Tq * a.Hq;  // rows between splits
  const float* base = a.part_o + item * (32 * NC) + lane * NC;
  float x[8][NC];
  auto load = [&](int s0) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      V v;
      if (s0 + u < S)
        v = __ldg(reinterpret_cast<const V*>(base + (int64_t)(s0 + u) * stride * (32 * NC)));
      else
        memset(&v, 0, sizeof(v));
      const float* f = reinterpret_cast<const float*>(&v);
#pragma unroll
      for (int c = 0; c < NC; ++c) x[u][c] = f[c];
    }
  };
  const float lse = lane < S ? __ldg(a.part_lse + (int64_t)lane * stride + item) : -INFINITY;
  load(0);
  float M = lse;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  T* out = (T*)a.out + item * (32 * NC) + lane * NC;
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.f;
  if (M == -INFINITY) {  // no split saw a key: 0
    store_lane<T, NC>(out, acc);
    return;
  }
  const float w = lane < S ? expf(lse - M) : 0.f;  // 0 for an empty split (lse = -inf)
  float wsum = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  for (int s0 = 0;;) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float ws = __shfl_sync(0xffffffffu, w, (s0 + u) & 31);
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] = fmaf(s0 + u < S ? ws : 0.f, x[u][c], acc[c]);
    }
    s0 += 8;
    if (s0 >= S) break;
    load(s0);
  }
  const float inv = 1.f / wsum;
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] *= inv;
  store_lane<T, NC>(out, acc);
}

// One warp per combined (token, head) row.  With a split tail (split_direct > 0) only the split
// items' rows are combined: warp w takes row wi % rows of tensor-core item split_direct + wi / rows,
// decoded as the kernel decodes it.
template <typename T>
__global__ void __launch_bounds__(256) attn_combine_kernel(PkvAttnArgs a) {
  const int64_t wi = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  int64_t item = wi;  // token * Hq + head
  if (a.split_direct > 0) {
    const int rows = a.max_query_len < kTcItemRows ? a.max_query_len : kTcItemRows;
    const int g = a.Hq / a.Hkv;
    const int n_qp = (a.max_query_len + kTcItemRows - 1) / kTcItemRows;
    const int64_t items = (int64_t)a.B * a.Hq * n_qp;
    const int64_t u = a.split_direct + wi / rows;
    if (u >= items) return;
    const PkvTcItem it = pkv_tc_item((int)u, g, n_qp, a.Hkv);
    const int i = it.qp * kTcItemRows + (int)(wi % rows);
    const int q0 = a.query_start_loc[it.b];
    int Sq = a.query_start_loc[it.b + 1] - q0;
    Sq = Sq < 0 ? 0 : (Sq > a.max_query_len ? a.max_query_len : Sq);
    const int64_t tok = (int64_t)q0 + i;
    if (i >= Sq || tok < 0 || tok >= a.Tq) return;
    item = tok * a.Hq + it.kvh * g + it.gi;
  } else if (item >= a.Tq * a.Hq) {
    return;
  }
  if (a.D == 128)
    combine_row<T, 4>(a, item, lane);
  else
    combine_row<T, 2>(a, item, lane);
}

template <typename T>
int launch_simt_t(const PkvAttnArgs& a, cudaStream_t s) {
  const int tiles_per_row = (a.max_query_len + kQT - 1) / kQT;
  dim3 grid((unsigned)(a.B * tiles_per_row), (unsigned)a.Hq, (unsigned)a.num_splits);
  if (a.D == 64)
    attn_simt_kernel<T, 64><<<grid, kWarps * 32, 0, s>>>(a);
  else
    attn_simt_kernel<T, 128><<<grid, kWarps * 32, 0, s>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace

int pkv_launch_attn_simt(const PkvAttnArgs& a, pkv_dtype dt, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  switch (dt) {
    case PKV_F32: return launch_simt_t<float>(a, s);
    case PKV_BF16: return launch_simt_t<__nv_bfloat16>(a, s);
    case PKV_F16: return launch_simt_t<__half>(a, s);
  }
  return (int)cudaErrorInvalidValue;
}

int pkv_launch_attn_combine(const PkvAttnArgs& a, pkv_dtype dt, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  int64_t warps = a.Tq * a.Hq;
  if (a.split_direct > 0) {
    const int64_t n_qp = (a.max_query_len + kTcItemRows - 1) / kTcItemRows;
    const int64_t rows = a.max_query_len < kTcItemRows ? a.max_query_len : kTcItemRows;
    warps = ((int64_t)a.B * a.Hq * n_qp - a.split_direct) * rows;
  }
  if (warps <= 0) return 0;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  switch (dt) {
    case PKV_F32: attn_combine_kernel<float><<<grid, 256, 0, s>>>(a); break;
    case PKV_BF16: attn_combine_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a); break;
    case PKV_F16: attn_combine_kernel<__half><<<grid, 256, 0, s>>>(a); break;
  }
  return (int)cudaGetLastError();
}
