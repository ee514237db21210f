// Tensor-core paged attention for bf16/f16 on sm_103a: TMA page gather,
// tcgen05 MMAs with TMEM accumulators, fp32 online softmax.
//
// What it computes is _reference_paged_attention (paged_attention.py): keys and
// values gathered through the block table, softmax(scale * q.k) over the
// visible keys, weighted sum of values -- with the piecewise causal/full mask
// of piecewise_attn.py expressed as a per-query key limit (every query sees a
// prefix [0, limit) of its row's keys).
//
// One CTA = 128 queries of one (row, query head) and one key-range split.
// Warp roles (192 threads):
//   warp 0     producer: gathers 128-key K and V tiles through the block table
//              with TMA, ONE box per 16-row pool block (4 KB for D=128): the
//              pool is viewed as a 5-D tensor (64 columns, 8 rows, D/64
//              column halves, row groups of 8, heads) so that a box lands as
//              [block][row group][column half][8 rows][128 B], 128-byte
//              swizzled.  Every 8-row x 128-byte atom then sits at a uniform
//              stride (GS = D/64 KB) in both the key and the value tile, which
//              is what the K-major (Q K^T) and MN-major (P V) shared-memory
//              descriptors need.  (Two 2 KB boxes per block -- one per column
//              half -- measured about half the load rate.)  3-stage ring per
//              operand; a partly written last block is loaded row by row;
//   warp 1     MMA issuer (one thread): S = Q K^T (Q from TMEM, K from shared
//              memory) into one of two TMEM score buffers, then O += P V (P from
//              TMEM, V from shared memory, MN-major) into the TMEM output;
//   warps 2-5  softmax: one query row per thread, matching TMEM lane = row.
//              Reads a score row from TMEM, masks, keeps a running maximum in
//              the exp2 domain, writes bf16/f16 probabilities back into the
//              score buffer's first columns for the P V MMA, and rescales its
//              O row only when the maximum grows by more than 2^8 (otherwise
//              the stale maximum is kept: probabilities stay <= 256).
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256,256+D), Q after O.
// Score buffers alternate, so QK^T of tile j+1 overlaps the softmax of tile j.
// Every mbarrier wait is bounded in time (1 s); on expiry the CTA records
// PKV_DEVERR_TIMEOUT, unwinds, waits for its own MMAs, frees TMEM and exits.

#include <cuda.h>

#include <mutex>

#include "tc_ptx.cuh"

namespace {

constexpr int BM = 128;      // queries per CTA
constexpr int BN = 128;      // keys per tile
constexpr int NST = 3;       // ring stages for K and for V
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait
constexpr float kRescaleThreshold = 8.0f;         // log2 units

template <int D>
struct alignas(1024) TcSmem {
  uint8_t k[NST][BN * D * 2];  // [D/64][BN rows][128 B], 128-byte swizzled
  uint8_t v[NST][BN * D * 2];
  uint64_t k_full[NST], k_empty[NST], v_full[NST], v_empty[NST];
  uint64_t s_full[2], p_full[2], o_done, q_ready, mma_done;
  uint32_t tmem_base;
  int lim_max;
  int abort;
};

struct TcMaps {
  CUtensorMap kb, vb;  // 5-D views, box = one whole pool block of one head
  CUtensorMap k1, v1;  // 3-D views (D, Hkv, slots), box = 64 columns of one row (partial blocks)
};

// Tile layout: byte offset of 128-byte row (tile row r, column half dh).
template <int D>
__host__ __device__ constexpr int tile_row_offset(int r, int dh) {
  return (r >> 4) * (2 * (D / 64) * 1024) + ((r >> 3) & 1) * ((D / 64) * 1024) + dh * 1024 + (r & 7) * 128;
}

template <int D>
PKV_DEVINLINE void note_abort(TcSmem<D>& sm, unsigned int* err) {
  sm.abort = 1;
  pkv_raise(err, PKV_DEVERR_TIMEOUT);
}

// Bounded wait by lane 0 of a warp, result broadcast so the warp stays converged.
PKV_DEVINLINE bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int lane) {
  bool ok = true;
  if (lane == 0) ok = ptx::mbar_wait(bar, parity, abort, kWaitLimitNs);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Producer: gather key rows [j0, j0 + rows) of one (row, kv head) into a stage.
template <int D>
PKV_DEVINLINE void load_tile(uint8_t* dst, const CUtensorMap* mb, const CUtensorMap* m1, uint64_t* full,
                             const PkvAttnArgs& a, int b, int kvh, int kt, int rows, int lane) {
  const int n_pages = (rows + 15) >> 4;
  const int rem = rows & 15;
  if (lane == 0) ptx::mbar_arrive_expect_tx(full, (uint32_t)(rows * D * 2));
  __syncwarp();
  if (lane < n_pages) {
    const int p = lane;
    int blk = a.block_table[(int64_t)b * a.W + kt * (BN / 16) + p];
    if (a.check && (blk < 0 || blk >= a.num_blocks)) {
      pkv_raise(a.err, PKV_DEVERR_BLOCK);
      blk = 0;
    }
    const bool partial = (p == n_pages - 1) && rem != 0;
    if (!partial) {
      ptx::tma_load_5d(dst + tile_row_offset<D>(p * 16, 0), mb, 0, 0, 0, blk * 2, kvh, full);
    } else {
      for (int r = 0; r < rem; ++r)
#pragma unroll
        for (int dh = 0; dh < D / 64; ++dh)
          ptx::tma_load_3d(dst + tile_row_offset<D>(p * 16 + r, dh), m1, dh * 64, kvh, blk * 16 + r, full);
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcMaps maps, const PkvAttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem<D>& sm = *reinterpret_cast<TcSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = a.Hq / a.Hkv;
  const int n_qt = (a.max_query_len + BM - 1) / BM;
  int u = blockIdx.x;
  const int gi = u % g;
  u /= g;
  const int qt = u % n_qt;
  u /= n_qt;
  const int kvh = u % a.Hkv;
  const int b = u / a.Hkv;
  const int h = kvh * g + gi;
  const int split = blockIdx.y;

  const int q0 = a.query_start_loc[b];
  int Sq = a.query_start_loc[b + 1] - q0;
  int L = a.seq_lens[b];
  if (a.check) {
    const int lmax = a.W * 16 < a.max_seq_len ? a.W * 16 : a.max_seq_len;
    const bool first = tid == 0 && qt == 0 && gi == 0 && split == 0;
    if (Sq < 0 || Sq > a.max_query_len) {
      if (first) pkv_raise(a.err, PKV_DEVERR_QUERY);
      Sq = Sq < 0 ? 0 : a.max_query_len;
    }
    if (L > lmax || L < Sq || L < 0) {
      if (first) pkv_raise(a.err, PKV_DEVERR_SEQLEN);
      L = L > lmax ? lmax : (L < 0 ? 0 : L);
    }
  }
  const int i0 = qt * BM;
  if (i0 >= Sq) return;  // whole CTA: no query rows here
  // A pipeline timeout earlier in this launch (or an unchecked earlier one) means
  // results are already invalid: fail fast instead of waiting again.
  if (*(volatile unsigned int*)a.err & PKV_DEVERR_TIMEOUT) return;

  // ---------------------------------------------------------------- setup
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      ptx::mbar_init(&sm.k_full[s], 1);
      ptx::mbar_init(&sm.k_empty[s], 1);
      ptx::mbar_init(&sm.v_full[s], 1);
      ptx::mbar_init(&sm.v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sm.s_full[s], 1);
      ptx::mbar_init(&sm.p_full[s], 128);
    }
    ptx::mbar_init(&sm.o_done, 1);
    ptx::mbar_init(&sm.q_ready, 128);
    ptx::mbar_init(&sm.mma_done, 1);
    sm.lim_max = 0;
    sm.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&maps.kb);
    ptx::prefetch_tmap(&maps.vb);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  __syncthreads();

  // Per-row key limit (softmax threads own rows).
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  int lim = 0;
  if (warp >= 2) {
    const int i = i0 + row;
    if (i < Sq) {
      bool uncovered = false;
      int s_begin = 0, s_end = 0;
      if (a.segs) {
        s_begin = a.seg_start[b];
        s_end = a.seg_start[b + 1];
      }
      lim = pkv_row_limit(L - Sq + i, L, a.segs, s_begin, s_end, &uncovered);
      if (a.check && uncovered) pkv_raise(a.err, PKV_DEVERR_SEGMENT);
    }
    atomicMax(&sm.lim_max, lim);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  const uint32_t tmem = sm.tmem_base;
  const int kv_hi = sm.lim_max;
  const int n_tiles = (kv_hi + BN - 1) / BN;
  const int per = (n_tiles + a.num_splits - 1) / a.num_splits;
  const int t_begin = split * per;
  const int t_end = min(n_tiles, t_begin + per);
  const int n = t_end > t_begin ? t_end - t_begin : 0;

  constexpr uint32_t S_COL[2] = {0, 128};
  constexpr uint32_t O_COL = 256;
  constexpr uint32_t Q_COL = 256 + D;
  constexpr uint32_t IDESC_QK = ptx::idesc_f16(BM, BN, BF16 ? 1 : 0, 0);
  constexpr uint32_t IDESC_PV = ptx::idesc_f16(BM, D, BF16 ? 1 : 0, 1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    for (int j = 0; j < n; ++j) {
      if (__any_sync(0xffffffffu, sm.abort != 0)) break;
      const int st = j % NST, use = j / NST;
      const int kt = t_begin + j;
      const int j0 = kt * BN;
      const int rows = min(BN, kv_hi - j0);
      if (j >= NST && !warp_wait(&sm.k_empty[st], (use - 1) & 1, &sm.abort, lane)) {
        if (lane == 0) note_abort(sm, a.err);
        break;
      }
      load_tile<D>(sm.k[st], &maps.kb, &maps.k1, &sm.k_full[st], a, b, kvh, kt, rows, lane);
      if (j >= NST && !warp_wait(&sm.v_empty[st], (use - 1) & 1, &sm.abort, lane)) {
        if (lane == 0) note_abort(sm, a.err);
        issued = j;  // K of tile j is in flight
        break;
      }
      if (rows < BN) {
        // Key rows past the last visible key are never loaded: zero them in V
        // (P is 0 there, but 0 * NaN would not be).  Zeroing whole 128-byte
        // rows is independent of the swizzle.
        const int nz = (BN - rows) * (D / 64) * 8;  // 16-byte chunks to clear
        for (int e = lane; e < nz; e += 32) {
          const int chunk = e & 7, rd = e >> 3;
          const int r = rows + rd / (D / 64), dh = rd % (D / 64);
          *reinterpret_cast<uint4*>(sm.v[st] + tile_row_offset<D>(r, dh) + chunk * 16) = make_uint4(0, 0, 0, 0);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
      }
      load_tile<D>(sm.v[st], &maps.vb, &maps.v1, &sm.v_full[st], a, b, kvh, kt, rows, lane);
      issued = j + 1;
    }
    if (sm.abort && lane == 0) {
      // Let the copies already issued land before the shared memory goes away.
      for (int j = (issued > NST ? issued - NST : 0); j < issued; ++j) {
        const int st = j % NST, use = j / NST;
        int dummy = 0;
        ptx::mbar_wait(&sm.k_full[st], use & 1, &dummy, kWaitLimitNs);
        ptx::mbar_wait(&sm.v_full[st], use & 1, &dummy, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      const uint32_t k_base = ptx::smem_u32(sm.k[0]);
      const uint32_t v_base = ptx::smem_u32(sm.v[0]);
      bool ok = ptx::mbar_wait(&sm.q_ready, 0, &sm.abort, kWaitLimitNs);
      ptx::tc_fence_after();
      auto issue_qk = [&](int j) -> bool {
        const int st = j % NST;
        if (!ptx::mbar_wait(&sm.k_full[st], (j / NST) & 1, &sm.abort, kWaitLimitNs)) return false;
        ptx::tc_fence_after();
        const uint32_t kst = k_base + st * (BN * D * 2);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          // K-major: 8-row atoms at stride GS, column half at +1024, 32 B per 16-column step.
          const uint64_t bdesc = ptx::smem_desc(kst + (ks >> 2) * 1024 + (ks & 3) * 32, 16, (D / 64) * 1024, 2);
          ptx::mma_ts(tmem + S_COL[j & 1], tmem + Q_COL + ks * 8, bdesc, IDESC_QK, ks > 0);
        }
        ptx::mma_commit(&sm.s_full[j & 1]);
        ptx::mma_commit(&sm.k_empty[st]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      if (ok && n > 1) ok = issue_qk(1);
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % NST;
        if (!ptx::mbar_wait(&sm.p_full[j & 1], (j >> 1) & 1, &sm.abort, kWaitLimitNs) ||
            !ptx::mbar_wait(&sm.v_full[st], (j / NST) & 1, &sm.abort, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t vst = v_base + st * (BN * D * 2);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          // MN-major: column halves at LBO = 1024, 8-row atoms at SBO = GS; one pool block per step.
          const uint64_t bdesc = ptx::smem_desc(vst + ks * tile_row_offset<D>(16, 0), 1024, (D / 64) * 1024, 2);
          ptx::mma_ts(tmem + O_COL, tmem + S_COL[j & 1] + ks * 8, bdesc, IDESC_PV, (j > 0 || ks > 0) ? 1u : 0u);
        }
        ptx::mma_commit(&sm.v_empty[st]);
        ptx::mma_commit(&sm.o_done);
        if (j + 2 < n) ok = issue_qk(j + 2);
      }
      if (!ok) note_abort(sm, a.err);
      // Everything issued must finish before TMEM is released.
      ptx::mma_commit(&sm.mma_done);
      int dummy = 0;
      ptx::mbar_wait(&sm.mma_done, 0, &dummy, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int i = i0 + row;
    const bool valid = i < Sq;
    const int64_t tok = (int64_t)q0 + i;
    // Q row -> TMEM (packed pairs of 16-bit values, column c holds elements 2c and 2c+1).
    {
      const uint4* src = reinterpret_cast<const uint4*>((const uint16_t*)a.q + (tok * a.Hq + h) * D);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4) {
          const uint4 x = valid ? src[c * 8 + v4] : make_uint4(0, 0, 0, 0);
          r[v4 * 4 + 0] = x.x;
          r[v4 * 4 + 1] = x.y;
          r[v4 * 4 + 2] = x.z;
          r[v4 * 4 + 3] = x.w;
        }
        ptx::tmem_st32(tmem + lane_base + Q_COL + c * 32, r);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&sm.q_ready);
    }
    const float sl2 = a.scale * 1.4426950408889634f;  // scale * log2(e)
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int sb = j & 1;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sm.s_full[sb], (j >> 1) & 1, &sm.abort, kWaitLimitNs))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      float s[BN];
      {
        uint32_t r[BN / 32][32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) ptx::tmem_ld32(tmem + lane_base + S_COL[sb] + c * 32, r[c]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          ptx::reg_fence32(r[c]);
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[c][e]);
        }
      }
      const int j0 = (t_begin + j) * BN;
      const int nvis = lim - j0;
      if (nvis < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = c < nvis ? s[c] : -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < BN; c += 4) {
        mx0 = fmaxf(mx0, s[c]);
        mx1 = fmaxf(mx1, s[c + 1]);
        mx2 = fmaxf(mx2, s[c + 2]);
        mx3 = fmaxf(mx3, s[c + 3]);
      }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
      // TMEM loads/stores are warp-collective: the warp rescales together when any
      // of its rows needs it (alpha = 1 for the others).
      const bool need = m_tile > m_ref + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ptx::ex2(m_ref - m_tile) : 1.f;  // 0 on a row's first visible tile
        l *= alpha;
        if (j > 0) {
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sm.o_done, (j - 1) & 1, &sm.abort, kWaitLimitNs))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            ptx::tmem_ld32(tmem + lane_base + O_COL + c * 32, r);
            ptx::tmem_wait_ld();
            ptx::reg_fence32(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            ptx::tmem_st32(tmem + lane_base + O_COL + c * 32, r);
          }
        }
        if (need) m_ref = m_tile;
      }
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      float l0 = 0.f, l1 = 0.f;
      // P occupies columns [0, BN/2) of the score buffer: 32 scores -> 16 packed columns.
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ptx::ex2(fmaf(s[c * 32 + 2 * e], sl2, -mu));
          const float p1 = ptx::ex2(fmaf(s[c * 32 + 2 * e + 1], sl2, -mu));
          l0 += p0;
          l1 += p1;
          r[e] = BF16 ? ptx::pack_bf16x2(p0, p1) : ptx::pack_f16x2(p0, p1);
        }
        ptx::tmem_st16(tmem + lane_base + S_COL[sb] + c * 16, r);
      }
      l += l0 + l1;
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&sm.p_full[sb]);
    }
    if (!ok) note_abort(sm, a.err);

    // ---------------------------------------------------------------- epilogue
    if (ok) {
      float o[D];
      if (n > 0) {
        // Not o_done: when the last tile is reached that barrier can still be two
        // phases behind (P.V of tile n-2 in flight), and a parity wait would then
        // pass at once.  mma_done completes exactly once, after every MMA.
        if (__all_sync(0xffffffffu, ptx::mbar_wait(&sm.mma_done, 0, &sm.abort, kWaitLimitNs))) {
          ptx::tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            ptx::tmem_ld32(tmem + lane_base + O_COL + c * 32, r);
            ptx::tmem_wait_ld();
            ptx::reg_fence32(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[c * 32 + e] = __uint_as_float(r[e]);
          }
        } else {
          note_abort(sm, a.err);
          l = 0.f;
        }
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (!valid) {
        // query row past the end of this row's queries: nothing to store
      } else if (a.num_splits == 1) {
        uint4* dst = reinterpret_cast<uint4*>((uint16_t*)a.out + (tok * a.Hq + h) * D);
#pragma unroll
        for (int v8 = 0; v8 < D / 8; ++v8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = n > 0 ? o[v8 * 8 + 2 * e] * inv : 0.f;
            const float x1 = n > 0 ? o[v8 * 8 + 2 * e + 1] * inv : 0.f;
            w[e] = BF16 ? ptx::pack_bf16x2(x0, x1) : ptx::pack_f16x2(x0, x1);
          }
          dst[v8] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        float4* dst = reinterpret_cast<float4*>(a.part_o + (((int64_t)split * a.Tq + tok) * a.Hq + h) * D);
#pragma unroll
        for (int v4 = 0; v4 < D / 4; ++v4) {
          dst[v4] = n > 0 ? make_float4(o[v4 * 4] * inv, o[v4 * 4 + 1] * inv, o[v4 * 4 + 2] * inv, o[v4 * 4 + 3] * inv)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // natural-log log-sum-exp of this split: ln 2 * (m_ref + log2 l)
        a.part_lse[((int64_t)split * a.Tq + tok) * a.Hq + h] =
            (n > 0 && l > 0.f) ? 0.6931471805599453f * (m_ref + __log2f(l)) : -INFINITY;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// Pool viewed as a 3-D tensor (D, Hkv, slots); box = 64 columns of one head in one slot, 128-byte swizzle.
bool encode_pool_rows(CUtensorMap* m, const void* pool, int64_t num_slots, int Hkv, int D, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)num_slots};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
  cuuint32_t box[3] = {64, 1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Pool viewed as a 5-D tensor: (64 columns, 8 rows, D/64 column halves, slot groups of 8, Hkv heads),
// strides (slot, 128 B, 8 slots, head).  Box = {64, 8, D/64, 2, 1} = one 16-row block of one head,
// landing as [row group][column half][8 rows][128 B].
bool encode_pool_blocks(CUtensorMap* m, const void* pool, int64_t num_slots, int Hkv, int D, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t slot = (cuuint64_t)Hkv * D * 2;
  cuuint64_t dims[5] = {64, 8, (cuuint64_t)(D / 64), (cuuint64_t)(num_slots / 8), (cuuint64_t)Hkv};
  cuuint64_t strides[4] = {slot, 128, 8 * slot, (cuuint64_t)D * 2};
  cuuint32_t box[5] = {64, 8, (cuuint32_t)(D / 64), 2, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
                  const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool BF16>
int launch_tc(const PkvAttnArgs& a, cudaStream_t s) {
  TcMaps maps;
  const int64_t num_slots = a.num_blocks * 16;
  if (!encode_pool_blocks(&maps.kb, a.k_pool, num_slots, a.Hkv, D, BF16) ||
      !encode_pool_blocks(&maps.vb, a.v_pool, num_slots, a.Hkv, D, BF16) ||
      !encode_pool_rows(&maps.k1, a.k_pool, num_slots, a.Hkv, D, BF16) ||
      !encode_pool_rows(&maps.v1, a.v_pool, num_slots, a.Hkv, D, BF16))
    return (int)cudaErrorInvalidValue;
  // At least ~116 KB so that two CTAs never share an SM: each allocates all 512 TMEM columns.
  const size_t smem = sizeof(TcSmem<D>) + 1024 > (size_t)(116 * 1024) ? sizeof(TcSmem<D>) + 1024 : (size_t)(116 * 1024);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    attr_set[dev] = true;
  }
  const int g = a.Hq / a.Hkv;
  const int n_qt = (a.max_query_len + BM - 1) / BM;
  const int64_t units = (int64_t)a.B * a.Hkv * n_qt * g;
  if (units > 0x7fffffff) return (int)cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)units, (unsigned)a.num_splits);
  attn_tc_kernel<D, BF16><<<grid, kThreads, smem, s>>>(maps, a);
  return (int)cudaGetLastError();
}

}  // namespace

bool pkv_attn_tc_supports(pkv_dtype dt, int D) { return (dt == PKV_BF16 || dt == PKV_F16) && (D == 64 || D == 128); }

int pkv_launch_attn_tc(const PkvAttnArgs& a, pkv_dtype dt, void* stream) {
  if (!pkv_attn_tc_supports(dt, a.D) || !(a.scale > 0.f) || !a.err) return -1;
  cudaStream_t s = (cudaStream_t)stream;
  if (a.D == 128) return dt == PKV_BF16 ? launch_tc<128, true>(a, s) : launch_tc<128, false>(a, s);
  return dt == PKV_BF16 ? launch_tc<64, true>(a, s) : launch_tc<64, false>(a, s);
}
