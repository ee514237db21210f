// CUDA-core paged attention (fp32 arithmetic throughout) and the split-KV combine.
//
// This is the kernel for fp32 inputs, where tensor-core tf32 would not meet a
// 1e-4 tolerance, and for calls that ask for it (PKV_FORCE_SIMT).  It computes
// what _reference_paged_attention (paged_attention.py) computes -- gather each
// key through the block table, softmax(scale * q.k) over the visible keys,
// weighted sum of values -- with the piecewise causal/full mask of
// piecewise_attn.py expressed as a per-query key limit, and an online
// (running max / running sum) softmax so the key range can be streamed.
//
// CTA = 128 queries of one (row, head) and one key-range split; 256 threads as a
// 16 x 16 grid (ty, tx).  Per 64-key tile, all in fp32 shared memory:
//   S = Q K^T  thread (ty, tx) owns rows ty + 16i (i < 8) and keys tx + 16j
//              (j < 4): per 4 dimensions it loads 8 query and 4 key float4s and
//              does 128 FMAs (rows and keys interleaved by 16, so a warp's key
//              loads hit distinct banks and its query loads are broadcasts);
//              the loop is unrolled, so the next dimensions' operands load while
//              these FMAs run (two warps per SM partition cannot hide shared-
//              memory latency otherwise);
//   softmax    each row's 64 scores sit in the 16 threads of one half-warp:
//              maxima and sums by shuffles; P goes to shared memory transposed;
//   O += P V   thread (ty, tx) owns rows 8ty..8ty+7 and columns 4tx + 64c:
//              per key two float4s of P and D/64 float4s of V for 32 D/64 FMAs,
//              the next key's operands loaded while these FMAs run.
// The keys come double-buffered (the next tile's arrive during this one), the
// values single-buffered (a tile's arrive during its scores and softmax): with
// 8 x 4 scores per thread instead of 4 x 4, the shared-memory wavefronts per FMA
// fall by a third, and Q, two key tiles, one value tile and P fit in 205 KB
// for D = 128.
// Like the tensor-core grid, the grid splits the key ranges of only its last,
// partly filled wave of items (every item when there are fewer than SMs).

#include <math.h>
#include <string.h>

#include <atomic>
#include <type_traits>

#include "kv_copy.cuh"

namespace {

constexpr int kSQ = kSimtItemRows;  // queries per item (the unit of the grid and the split planner)
constexpr int kSK = kSimtKeyTile;   // keys per tile
constexpr int kSThreads = 256;
constexpr int kSWarps = kSThreads / 32;

static_assert(kSQ == 128 && kSK == 64, "thread tiles assume 128-query items and 64-key tiles");

// Shared memory of a CTA over ROWS query rows (128; 64 when every row of the call has at most 64 queries).
template <int D, int ROWS>
struct SimtSmem {
  static constexpr int LD = D + 4;     // row stride (floats) of Q, K and V: 16-byte rows, staggered banks
  static constexpr int PL = ROWS + 4;  // row stride of P^T
  // Q, two key buffers (the next tile's keys load while this one is used), one value buffer (a tile's
  // values load during its scores and softmax), P^T, per-row state.
  static constexpr size_t floats = (size_t)ROWS * LD + (size_t)3 * kSK * LD + (size_t)kSK * PL + 3 * ROWS;
  static constexpr size_t bytes = floats * sizeof(float) + (ROWS + 1) * sizeof(int);
};

// 16-byte asynchronous copy global -> shared; `bytes` 0 zero-fills the destination without a read.
PKV_DEVINLINE void cp_async16(float* dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(bytes)
               : "memory");
}

// Four consecutive elements as fp32 (16-byte aligned for fp32, 8-byte for 16-bit types).
template <typename T>
PKV_DEVINLINE float4 load4(const T* __restrict__ p) {
  if constexpr (sizeof(T) == 4) {
    return __ldg(reinterpret_cast<const float4*>(p));
  } else {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    T t[4];
    memcpy(t, &u, sizeof(u));
    return make_float4(pkv_to_f32<T>(t[0]), pkv_to_f32<T>(t[1]), pkv_to_f32<T>(t[2]), pkv_to_f32<T>(t[3]));
  }
}

template <typename T>
PKV_DEVINLINE void store4(T* p, float x0, float x1, float x2, float x3) {
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(x0, x1, x2, x3);
  } else {
    T t[4] = {pkv_from_f32<T>(x0), pkv_from_f32<T>(x1), pkv_from_f32<T>(x2), pkv_from_f32<T>(x3)};
    uint2 u;
    memcpy(&u, t, sizeof(u));
    *reinterpret_cast<uint2*>(p) = u;
  }
}

// RI query rows per thread (scores: rows ty + 16i; output: rows RI*ty + i): 8 for a whole 128-query item,
// 4 when every row of the call has at most 64 queries (the CTA then covers its item's first 64 rows only).
template <typename T, int D, int RI>
__global__ void __launch_bounds__(kSThreads, 1) attn_simt_kernel(PkvAttnArgs a) {
  constexpr int ROWS = 16 * RI;
  using SM = SimtSmem<D, ROWS>;
  constexpr int LD = SM::LD, PL = SM::PL, NC = D / 64;
  extern __shared__ __align__(16) float sm[];
  float* q_s = sm;                          // [ROWS][LD]
  float* k_buf = q_s + ROWS * LD;           // two buffers of [kSK][LD] keys
  float* v_s = k_buf + 2 * kSK * LD;        // [kSK][LD] values
  float* p_s = v_s + kSK * LD;              // [kSK][PL], P transposed: p_s[key * PL + query]
  float* alpha_s = p_s + kSK * PL;  // [ROWS] per-tile rescale of each row's O
  float* l_s = alpha_s + ROWS;      // [ROWS]
  float* m_s = l_s + ROWS;          // [ROWS]
  int* lim_s = reinterpret_cast<int*>(m_s + ROWS);  // [ROWS], then the CTA's largest limit
  int* kv_hi_s = lim_s + ROWS;

  // CTA -> (row, query tile, head, key-range split).  Without a split tail the grid is (rows x
  // query tiles, heads, splits).  With one it is one-dimensional over the items in the same order
  // (query tiles fastest, then rows, then heads: the CTAs of one row and head run together and
  // share its keys in L2): items [0, split_direct) run whole, every later item takes num_splits
  // consecutive CTAs.
  const int tiles_per_row = (a.max_query_len + kSQ - 1) / kSQ;
  int x = blockIdx.x, h = blockIdx.y, split = blockIdx.z, nsplit = a.num_splits;
  if (a.split_direct > 0) {
    int u = blockIdx.x;
    split = 0;
    nsplit = 1;
    if (u >= a.split_direct) {
      const int p = u - a.split_direct;
      u = a.split_direct + p / a.num_splits;
      split = p % a.num_splits;
      nsplit = a.num_splits;
    }
    const int row_items = a.B * tiles_per_row;
    h = u / row_items;
    x = u % row_items;
  }
  const int b = x / tiles_per_row;
  const int tile = x % tiles_per_row;
  const int kvh = h / (a.Hq / a.Hkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ty = tid >> 4, tx = tid & 15;

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
                a.num_slots, a.Hkv * D * (int)sizeof(T) / 16, a.err, a.check, cta * kSWarps + warp,
                (int64_t)gridDim.x * gridDim.y * gridDim.z * kSWarps, lane, &a);
  }
  const int i0 = tile * kSQ;
  if (i0 >= Sq) return;

  int s_begin = 0, s_end = 0;
  if (a.segs) {
    s_begin = a.seg_start[b];
    s_end = a.seg_start[b + 1];
  }
  const int base = pkv_query_base(L, Sq, a.segs, s_begin, s_end);
  // Per-query key limits from the row's segments.
  if (tid < ROWS) {
    const int i = i0 + tid;
    int lim = 0;
    if (i < Sq) {
      bool uncovered = false;
      lim = pkv_row_limit(base + i, L, a.segs, s_begin, s_end, &uncovered);
      if (a.check && (uncovered || base < 0 || base + Sq > L)) pkv_raise(a.err, PKV_DEVERR_SEGMENT);
    }
    lim_s[tid] = lim;
  }
  // Query tile, fp32 in shared memory (rows past the row's queries are zero).
  for (int e = tid; e < ROWS * (D / 4); e += kSThreads) {
    const int r = e / (D / 4), c = (e % (D / 4)) * 4;
    const int i = i0 + r;
    const float4 x = i < Sq ? load4<T>((const T*)a.q + ((int64_t)(q0 + i) * a.Hq + h) * D + c)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(q_s + r * LD + c) = x;
  }
  __syncthreads();
  if (warp == 0) {
    int hi = 0;
#pragma unroll
    for (int r = lane; r < ROWS; r += 32) hi = lim_s[r] > hi ? lim_s[r] : hi;
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) *kv_hi_s = hi;
  }
  __syncthreads();
  const int kv_hi = *kv_hi_s;

  // This split's range of key tiles.
  const int n_tiles = (kv_hi + kSK - 1) / kSK;
  const int per = (n_tiles + nsplit - 1) / nsplit;
  const int t_begin = split * per;
  const int t_end = min(n_tiles, t_begin + per);

  // Keys at the queries' own positions [cb, ce): read from the new tokens in a fused call.
  const int cb = a.k_new ? base : 0, ce = a.k_new ? base + Sq : 0;

  int lim_r[RI];
#pragma unroll
  for (int i = 0; i < RI; ++i) lim_r[i] = lim_s[ty + 16 * i];
  float m[RI], l[RI];  // softmax state of rows ty + 16i (the same in all 16 threads of the half-warp)
#pragma unroll
  for (int i = 0; i < RI; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
  }
  float acc[RI][4 * NC];  // O rows RI*ty + i, columns 4tx + 64c + e
#pragma unroll
  for (int i = 0; i < RI; ++i)
#pragma unroll
    for (int c = 0; c < 4 * NC; ++c) acc[i][c] = 0.f;

  // Gather tile kt's 64 keys (is_v false) or values (true) through the block table into `dst`
  // (fp32); past kv_hi: zeros.  fp32 sources go by asynchronous 16-byte copies, one commit group per
  // call; 16-bit ones are loaded and converted.
  auto gather = [&](int kt, bool is_v, float* dst) {
    const T* pool = is_v ? (const T*)a.v_pool : (const T*)a.k_pool;
    const T* fresh = is_v ? (const T*)a.v_new : (const T*)a.k_new;
    const int j0 = kt * kSK;
    for (int e = tid; e < kSK * (D / 4); e += kSThreads) {
      const int jj = e / (D / 4), c = (e % (D / 4)) * 4;
      const int j = j0 + jj;
      const T* src = nullptr;
      if (j < kv_hi && j >= cb && j < ce) {
        src = fresh + (((int64_t)q0 + (j - cb)) * a.Hkv + kvh) * D + c;
      } else if (j < kv_hi) {
        int blk = a.block_table[(int64_t)b * a.W + (j >> 4)];
        if (a.check && (blk < 0 || blk >= a.num_blocks)) {
          pkv_raise(a.err, PKV_DEVERR_BLOCK);
          blk = -1;
        }
        if (blk >= 0) src = pool + (((int64_t)blk * 16 + (j & 15)) * a.Hkv + kvh) * D + c;
      }
      if constexpr (sizeof(T) == 4) {
        cp_async16(dst + jj * LD + c, src ? (const void*)src : (const void*)pool, src ? 16 : 0);
      } else {
        *reinterpret_cast<float4*>(dst + jj * LD + c) = src ? load4<T>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  // Per tile kt: its values and the next tile's keys are requested at the top (two commit groups), its
  // keys (requested one tile earlier) are waited for before the scores, its values before P.V.
  if (t_begin < t_end) gather(t_begin, false, k_buf);
  for (int kt = t_begin; kt < t_end; ++kt) {
    const int j0 = kt * kSK;
    const float* k_s = k_buf + ((kt - t_begin) & 1) * kSK * LD;
    __syncthreads();  // the previous tile's P.V no longer reads the values or P
    gather(kt, true, v_s);
    if (kt + 1 < t_end)
      gather(kt + 1, false, k_buf + ((kt + 1 - t_begin) & 1) * kSK * LD);
    else
      asm volatile("cp.async.commit_group;" ::: "memory");  // an empty group keeps the count
    asm volatile("cp.async.wait_group 2;" ::: "memory");  // this tile's keys have landed
    __syncthreads();

    // S = Q K^T for rows ty + 16i, keys tx + 16j.
    float s[RI][4];
#pragma unroll
    for (int i = 0; i < RI; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
    {
#pragma unroll
      for (int d = 0; d < D; d += 4) {
        float4 qv[RI], kv[4];
#pragma unroll
        for (int i = 0; i < RI; ++i) qv[i] = *reinterpret_cast<const float4*>(q_s + (ty + 16 * i) * LD + d);
#pragma unroll
        for (int j = 0; j < 4; ++j) kv[j] = *reinterpret_cast<const float4*>(k_s + (tx + 16 * j) * LD + d);
#pragma unroll
        for (int i = 0; i < RI; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qv[i].x, kv[j].x, s[i][j]);
#pragma unroll
        for (int i = 0; i < RI; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qv[i].y, kv[j].y, s[i][j]);
#pragma unroll
        for (int i = 0; i < RI; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qv[i].z, kv[j].z, s[i][j]);
#pragma unroll
        for (int i = 0; i < RI; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qv[i].w, kv[j].w, s[i][j]);
      }
    }
    // Online softmax per row: the row's 64 scores live in this half-warp (lanes with the same ty).
#pragma unroll
    for (int i = 0; i < RI; ++i) {
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        s[i][j] = j0 + tx + 16 * j < lim_r[i] ? s[i][j] * a.scale : -INFINITY;
        tmax = fmaxf(tmax, s[i][j]);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_new = fmaxf(m[i], tmax);
      float alpha = 1.f, psum = 0.f;
      if (m_new != -INFINITY) {  // else: nothing visible yet for this query; P = 0, O unchanged
        alpha = expf(m[i] - m_new);  // exp(-inf) = 0 on the first visible tile
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p = s[i][j] == -INFINITY ? 0.f : expf(s[i][j] - m_new);
          s[i][j] = p;
          psum += p;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      if (m_new != -INFINITY) {
        l[i] = l[i] * alpha + psum;
        m[i] = m_new;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) p_s[(tx + 16 * j) * PL + ty + 16 * i] = s[i][j];
      if (tx == 0) alpha_s[ty + 16 * i] = alpha;
    }
    asm volatile("cp.async.wait_group 1;" ::: "memory");  // this tile's values have landed
    __syncthreads();

    // O += P V for rows RI*ty + i, columns 4tx + 64c.
    {
#pragma unroll
      for (int q4 = 0; q4 < RI / 4; ++q4) {
        const float4 al = *reinterpret_cast<const float4*>(alpha_s + RI * ty + 4 * q4);
        const float alr[4] = {al.x, al.y, al.z, al.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int c = 0; c < 4 * NC; ++c) acc[4 * q4 + e][c] *= alr[e];
      }
      // Two keys per step: the next key's P and V are loaded while this key's FMAs run.
      float4 p0[RI / 4], p1[RI / 4], v0[NC], v1[NC];
#pragma unroll
      for (int q4 = 0; q4 < RI / 4; ++q4) p0[q4] = *reinterpret_cast<const float4*>(p_s + RI * ty + 4 * q4);
#pragma unroll
      for (int c = 0; c < NC; ++c) v0[c] = *reinterpret_cast<const float4*>(v_s + 4 * tx + 64 * c);
      auto pv_fma = [&](const float4 (&pv)[RI / 4], const float4 (&vv)[NC]) {
#pragma unroll
        for (int q4 = 0; q4 < RI / 4; ++q4) {
          const float pr[4] = {pv[q4].x, pv[q4].y, pv[q4].z, pv[q4].w};
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float* o = acc[4 * q4 + e] + 4 * c;
              o[0] = fmaf(pr[e], vv[c].x, o[0]);
              o[1] = fmaf(pr[e], vv[c].y, o[1]);
              o[2] = fmaf(pr[e], vv[c].z, o[2]);
              o[3] = fmaf(pr[e], vv[c].w, o[3]);
            }
        }
      };
#pragma unroll 4
      for (int k = 0; k < kSK; k += 2) {
#pragma unroll
        for (int q4 = 0; q4 < RI / 4; ++q4)
          p1[q4] = *reinterpret_cast<const float4*>(p_s + (k + 1) * PL + RI * ty + 4 * q4);
#pragma unroll
        for (int c = 0; c < NC; ++c) v1[c] = *reinterpret_cast<const float4*>(v_s + (k + 1) * LD + 4 * tx + 64 * c);
        pv_fma(p0, v0);
        if (k + 2 < kSK) {
#pragma unroll
          for (int q4 = 0; q4 < RI / 4; ++q4)
            p0[q4] = *reinterpret_cast<const float4*>(p_s + (k + 2) * PL + RI * ty + 4 * q4);
#pragma unroll
          for (int c = 0; c < NC; ++c) v0[c] = *reinterpret_cast<const float4*>(v_s + (k + 2) * LD + 4 * tx + 64 * c);
        }
        pv_fma(p1, v1);
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // nothing in flight into shared memory at exit

  // Epilogue: each row's softmax state to shared memory, then the normalised output (one split),
  // or the partial output and its natural-log log-sum-exp (a key-range split).
  if (tx == 0) {
#pragma unroll
    for (int i = 0; i < RI; ++i) {
      l_s[ty + 16 * i] = l[i];
      m_s[ty + 16 * i] = m[i];
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < RI; ++i) {
    const int r = RI * ty + i;
    const int qi = i0 + r;
    if (qi >= Sq) continue;
    const int64_t tok = (int64_t)q0 + qi;
    const float lr = l_s[r];
    const float inv = lr > 0.f ? 1.f / lr : 0.f;
    if (nsplit == 1) {
      T* o = (T*)a.out + (tok * a.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < NC; ++c)
        store4<T>(o + 4 * tx + 64 * c, acc[i][4 * c] * inv, acc[i][4 * c + 1] * inv, acc[i][4 * c + 2] * inv,
                  acc[i][4 * c + 3] * inv);
    } else {
      float* o = a.part_o + (((int64_t)split * a.Tq + tok) * a.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < NC; ++c)
        store4<float>(o + 4 * tx + 64 * c, acc[i][4 * c] * inv, acc[i][4 * c + 1] * inv, acc[i][4 * c + 2] * inv,
                      acc[i][4 * c + 3] * inv);
      if (tx == 0)
        a.part_lse[((int64_t)split * a.Tq + tok) * a.Hq + h] = lr > 0.f ? m_s[r] + logf(lr) : -INFINITY;
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
// split s's log-sum-exp (at most 32 splits).  The first kBatch splits' rows are loaded together with
// the log-sum-exps, so a row of up to kBatch splits costs one round trip to memory (the launch picks
// kBatch = 8 or 16 from the split count: the larger batch holds twice the registers).
template <typename T, int NC, int kBatch>
PKV_DEVINLINE void combine_row(const PkvAttnArgs& a, int64_t item, int lane) {
  using V = typename std::conditional<NC == 4, float4, float2>::type;
  const int S = a.num_splits;
  const int64_t stride = a.Tq * a.Hq;  // rows between splits
  const float* base = a.part_o + item * (32 * NC) + lane * NC;
  float x[kBatch][NC];
  auto load = [&](int s0) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
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
    for (int u = 0; u < kBatch; ++u) {
      const float ws = __shfl_sync(0xffffffffu, w, (s0 + u) & 31);
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[c] = fmaf(s0 + u < S ? ws : 0.f, x[u][c], acc[c]);
    }
    s0 += kBatch;
    if (s0 >= S) break;
    load(s0);
  }
  const float inv = 1.f / wsum;
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] *= inv;
  store_lane<T, NC>(out, acc);
}

// One warp per combined (token, head) row.  With a split tail (split_direct > 0) only the split
// items' rows are combined: warp w takes row wi % rows of item split_direct + wi / rows, decoded as
// the kernel that ran decodes it.
template <typename T, int kBatch>
__global__ void __launch_bounds__(256) attn_combine_kernel(PkvAttnArgs a) {
  // Launched as a programmatic dependent of the attention launch (it may be scheduled while the attention
  // drains): wait here until that grid has completed and its partial results are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t wi = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  int64_t item = wi;  // token * Hq + head
  if (a.split_direct > 0) {
    const int unit = a.simt_items ? kSimtItemRows : kTcItemRows;
    const int rows = a.max_query_len < unit ? a.max_query_len : unit;
    const int n_q = (a.max_query_len + unit - 1) / unit;
    const int64_t items = (int64_t)a.B * a.Hq * n_q;
    const int64_t u = a.split_direct + wi / rows;
    if (u >= items) return;
    int b, h, qt;
    if (a.simt_items) {
      const int64_t row_items = (int64_t)a.B * n_q;
      h = (int)(u / row_items);
      const int x = (int)(u % row_items);
      b = x / n_q;
      qt = x % n_q;
    } else {
      const int g = a.Hq / a.Hkv;
      const PkvTcItem it = pkv_tc_item((int)u, g, n_q, a.Hkv);
      b = it.b;
      h = it.kvh * g + it.gi;
      qt = it.qp;
    }
    const int i = qt * unit + (int)(wi % rows);
    const int q0 = a.query_start_loc[b];
    int Sq = a.query_start_loc[b + 1] - q0;
    Sq = Sq < 0 ? 0 : (Sq > a.max_query_len ? a.max_query_len : Sq);
    const int64_t tok = (int64_t)q0 + i;
    if (i >= Sq || tok < 0 || tok >= a.Tq) return;
    item = tok * a.Hq + h;
  } else if (item >= a.Tq * a.Hq) {
    return;
  }
  if (a.D == 128)
    combine_row<T, 4, kBatch>(a, item, lane);
  else
    combine_row<T, 2, kBatch>(a, item, lane);
}

template <typename T, int D, int RI>
int launch_simt_r(const PkvAttnArgs& a, cudaStream_t s) {
  const size_t smem = SimtSmem<D, 16 * RI>::bytes;
  // Keyed on the context: function attributes belong to the context they were set in.
  static std::atomic<uint64_t> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cached = dev >= 0 && dev < 64;
  const uint64_t ctx = pkv_context_id();
  if (!cached || ctx == 0 || attr_set[dev].load(std::memory_order_acquire) != ctx) {
    const cudaError_t e =
        cudaFuncSetAttribute(attn_simt_kernel<T, D, RI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    if (cached) attr_set[dev].store(ctx, std::memory_order_release);
  }
  const int tiles_per_row = (a.max_query_len + kSQ - 1) / kSQ;
  dim3 grid((unsigned)(a.B * tiles_per_row), (unsigned)a.Hq, (unsigned)a.num_splits);
  if (a.split_direct > 0) {
    const int64_t items = (int64_t)a.B * tiles_per_row * a.Hq;
    const int64_t ctas = a.split_direct + (items - a.split_direct) * a.num_splits;
    if (ctas > 0x7fffffff) return (int)cudaErrorInvalidConfiguration;  // the planner keeps it below
    grid = dim3((unsigned)ctas);
  }
  attn_simt_kernel<T, D, RI><<<grid, kSThreads, smem, s>>>(a);
  return (int)cudaGetLastError();
}

// Rows of at most 64 queries (every item then holds only those): the CTA covers 64 rows with 4 per thread,
// half the work of a 128-row CTA whose other rows would be padding.  The items are the same either way.
template <typename T, int D>
int launch_simt_d(const PkvAttnArgs& a, cudaStream_t s) {
  return a.max_query_len <= 64 ? launch_simt_r<T, D, 4>(a, s) : launch_simt_r<T, D, 8>(a, s);
}

template <typename T>
int launch_simt_t(const PkvAttnArgs& a, cudaStream_t s) {
  return a.D == 64 ? launch_simt_d<T, 64>(a, s) : launch_simt_d<T, 128>(a, s);
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
    const int64_t unit = a.simt_items ? kSimtItemRows : kTcItemRows;
    const int64_t n_q = (a.max_query_len + unit - 1) / unit;
    const int64_t rows = a.max_query_len < unit ? a.max_query_len : unit;
    warps = ((int64_t)a.B * a.Hq * n_q - a.split_direct) * rows;
  }
  if (warps <= 0) return 0;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  // Programmatic dependent launch: the combine's launch overlaps the attention's last CTAs; the kernel's
  // first instruction waits for the attention grid (griddepcontrol.wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaErrorInvalidValue;
  const bool wide = a.num_splits > 8;
  switch (dt) {
    case PKV_F32:
      e = wide ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<float, 16>, a)
               : cudaLaunchKernelEx(&cfg, attn_combine_kernel<float, 8>, a);
      break;
    case PKV_BF16:
      e = wide ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<__nv_bfloat16, 16>, a)
               : cudaLaunchKernelEx(&cfg, attn_combine_kernel<__nv_bfloat16, 8>, a);
      break;
    case PKV_F16:
      e = wide ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<__half, 16>, a)
               : cudaLaunchKernelEx(&cfg, attn_combine_kernel<__half, 8>, a);
      break;
  }
  return (int)e;
}
