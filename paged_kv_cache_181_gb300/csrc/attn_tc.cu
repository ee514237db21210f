// Tensor-core paged attention for bf16/f16 on sm_103a: TMA page gather,
// tcgen05 MMAs with TMEM accumulators, fp32 online softmax.
//
// What it computes is _reference_paged_attention (paged_attention.py): keys and
// values gathered through the block table, softmax(scale * q.k) over the
// visible keys, weighted sum of values -- with the piecewise causal/full mask
// of piecewise_attn.py expressed as a per-query key limit (every query sees a
// prefix [0, limit) of its row's keys).
//
// One CTA = 256 queries of one (row, query head) -- two 128-query tiles that
// share every key/value tile -- or, for the items of a last, partly filled
// wave, one key-range split of them (the combine merges the splits).  Sharing halves the
// key/value bytes each SM has to take in per FLOP, which is what bounds this
// workload on this part (a one-tile CTA spent longer receiving its 64 KB per
// key tile than its tensor core spent on the MMAs).
//
// Warp roles (384 threads = 3 warpgroups):
//   warp 0     producer: TMA loads of both query tiles (once) and of the key
//              and value tiles through the block table, ONE box per 16-row pool
//              block: the pool is viewed as a 5-D tensor (64 columns, 8 rows,
//              D/64 column halves, row groups of 8, heads), so a box lands as
//              [row group][column half][8 rows][128 B], 128-byte swizzled, and
//              every 8-row atom sits at a uniform stride in the tile (what the
//              K-major and MN-major shared-memory descriptors need).  Key and
//              value tiles share one ring of slots (K_j, V_j, K_j+1, ...); a
//              partly written last block is loaded row by row; value rows past
//              the last visible key are zeroed.  Contiguous K/V (a consecutive
//              table): a whole 128-key tile is one box.  Fused write + attention:
//              the keys at the queries' own positions come from the new k/v
//              (one box per 16 tokens starting on an 8-token boundary);
//   warp 1     MMA issuer (one thread) and TMEM owner.  Per key tile j:
//                P0.V_j -> O0, Q0.K_j+1 -> S0, P1.V_j -> O1, Q1.K_j+1 -> S1
//              (A = Q from shared memory, or P from TMEM; B = K K-major or V
//              MN-major from shared memory), so while one softmax group works
//              on its scores the tensor core runs the other group's MMAs.  An
//              MMA issue returns when the pipe takes it, so the issue code is
//              kept lean (descriptors built once, offset per MMA);
//   warp 3     producer of the value tiles (warp 0 then loads Q and the key
//              tiles only): each producer warp shares an SM partition with two
//              softmax warps, and halving the per-tile instructions on one
//              partition shortened the softmax pass that is the critical path;
//   warp 2     fused write + attention only: the slot-mapping scatter of the
//              new k/v (this CTA's share of the rows);
//   warps 4-7  softmax of query tile 0, warps 8-11 of tile 1: one query row per
//              thread (TMEM lane = row).  Reads a score row from TMEM, masks,
//              keeps a running maximum in the exp2 domain, writes bf16/f16
//              probabilities over the first half of the score columns, and
//              rescales its O row only when the maximum grows by more than 2^8
//              (otherwise the stale maximum is kept: probabilities stay <= 256).
//              P.V of the previous tile is always complete by the time a score
//              tile is ready (the score MMA was issued after it), so the rescale
//              never waits.
// A row's ragged last tile of at most 64 queries (1560 = 6 x 256 + 24) runs alone in its CTA with
// M = 64 MMAs: half the tensor work (and energy) of M = 128 for the same rows; its accumulator rows
// sit in lanes 0-15 of each 32-lane TMEM quarter, so half of each softmax warp carries no row.
// Registers: the producer/MMA warpgroup (warps 0-3) gives up
// registers to the two softmax warpgroups (setmaxnreg 104 / 200; the launch
// provides 168 per thread and the host refuses to launch a build with another
// count, so the split always adds up).
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 after O0.
// Every mbarrier wait is bounded in time (1 s); on expiry the CTA records
// PKV_DEVERR_TIMEOUT, unwinds, waits for its own copies and MMAs, frees TMEM
// and exits.

#include <cuda.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "kv_copy.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int BM = 128;  // queries per tile; two tiles per CTA
constexpr int BN = 128;  // keys per tile
static_assert(2 * BM == kTcItemRows, "a work item is one tile pair");
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;  // registers per thread the kernel is compiled to (checked at launch)
constexpr int kRegsLow = 104;     // producer / MMA warpgroup
constexpr int kRegsHigh = 200;    // softmax warpgroups: 128*104 + 256*200 == 384*168
static_assert(128 * kRegsLow + 256 * kRegsHigh == kThreads * kLaunchRegs, "register split must add up");
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait
constexpr float kRescaleThreshold = 8.0f;         // log2 units

template <int D>
struct Cfg {
  static constexpr int TILE = BN * D * 2;          // one key or value tile
  static constexpr int NSLOT = D == 128 ? 5 : 10;  // ring slots (fits 227 KB with both query tiles)
  static constexpr int GS = (D / 64) * 1024;       // stride of 8-row atoms in a key/value tile
  static constexpr int PART_ROW = D * 4 + 16;      // staged fp32 partial row (padded: conflict-free)
};

template <int D>
struct alignas(1024) TcSmem {
  uint8_t q[2][BM * D * 2];                 // [D/64][128 rows][128 B] per query tile, 128-byte swizzled
  uint8_t kv[Cfg<D>::NSLOT][Cfg<D>::TILE];  // [block][row group][column half][8 rows][128 B]
  uint64_t full[Cfg<D>::NSLOT], empty[Cfg<D>::NSLOT];
  uint64_t q_full, s_full[2], p_full[2], mma_done;
  uint32_t tmem_base;
  int lim_max;
  int abort;
};

struct TcMaps {
  CUtensorMap q;       // (D, Hq, Tq), box = 64 columns x 128 tokens of one head
  CUtensorMap kb, vb;  // 5-D pool views, box = one whole 16-row pool block of one head
  CUtensorMap kc, vc;  // the same views, box = 8 consecutive blocks = one whole key tile (contiguous K/V)
  CUtensorMap k1, v1;  // 3-D pool views (D, Hkv, slots), box = 64 columns of one row (partial blocks)
  CUtensorMap kn5, vn5;  // fused call: new tokens in the pool's 5-D view, box = 16 tokens (8-aligned start)
  CUtensorMap kn8, vn8;  //   (D, Hkv, Tq), box = 64 columns x 8 tokens (one atom)
  CUtensorMap kn1, vn1;  //   the same, box = 64 columns of one token
  CUtensorMap o;         // output (D, Hq, Tq), box = 64 columns x 128 tokens of one head (one-split calls)
};

// The maps one operand (K or V) is loaded through.
struct OperandMaps {
  const CUtensorMap *blk, *tile, *row, *new5, *new8, *new1;
};

// Byte offset of 128-byte row (tile row r, column half dh) in a key/value tile.
template <int D>
__host__ __device__ constexpr int tile_row_offset(int r, int dh) {
  return (r >> 4) * (2 * Cfg<D>::GS) + ((r >> 3) & 1) * Cfg<D>::GS + dh * 1024 + (r & 7) * 128;
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

// Producer: gather key rows [kt*BN, kt*BN + rows) of one (row, kv head) into a slot.
// Contiguous K/V (the row's table entries are consecutive): a whole tile is one box of
// 8 blocks, which lands in the same [row group][column half][8 rows][128 B] layout.
// Fused call: keys [cb, ce) -- the queries' own positions -- come from the new tokens
// (token q0 + key - cb), whose write into the pool runs in the same launch.
template <int D>
PKV_DEVINLINE void load_tile(uint8_t* dst, const OperandMaps& m, uint64_t* full, const PkvAttnArgs& a, int b, int kvh,
                             int kt, int rows, int cb, int ce, int q0, int lane) {
  const int32_t* trow = a.block_table + (int64_t)b * a.W + kt * (BN / 16);
  const int t0 = kt * BN;
  const bool fused = a.k_new != nullptr;
  if (a.contiguous && rows == BN && !(fused && t0 < ce && t0 + BN > cb)) {
    int first = trow[0];
    bool ok = true;
    if (a.check) {
      const int e = lane < BN / 16 ? trow[lane] : first + lane;
      ok = __all_sync(0xffffffffu, e == first + lane) && first >= 0 && first <= a.num_blocks - BN / 16;
      if (!ok && lane == 0) pkv_raise(a.err, PKV_DEVERR_BLOCK);  // not consecutive: fall through to blocks
    }
    if (ok) {
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(full, (uint32_t)(BN * D * 2));
        ptx::tma_load_5d(dst, m.tile, 0, 0, 0, first * 2, kvh, full);
      }
      __syncwarp();
      return;
    }
  }
  const int n_pages = (rows + 15) >> 4;
  if (lane == 0) ptx::mbar_arrive_expect_tx(full, (uint32_t)(rows * D * 2));
  __syncwarp();
  if (lane < n_pages) {
    const int p = lane;
    const int k0 = t0 + 16 * p;                       // first key of this block
    const int nr = rows - 16 * p < 16 ? rows - 16 * p : 16;  // its rows inside the tile
    const bool all_new = fused && k0 >= cb && k0 + nr <= ce;
    const bool no_new = !fused || k0 + nr <= cb || k0 >= ce;
    int blk = 0;
    if (!all_new) {
      blk = trow[p];
      if (a.check && (blk < 0 || blk >= a.num_blocks)) {
        pkv_raise(a.err, PKV_DEVERR_BLOCK);
        blk = 0;
      }
    }
    if (nr == 16 && no_new) {
      ptx::tma_load_5d(dst + tile_row_offset<D>(p * 16, 0), m.blk, 0, 0, 0, blk * 2, kvh, full);
    } else if (nr == 16 && all_new && ((q0 + k0 - cb) & 7) == 0 && q0 + k0 - cb + 16 <= (int)(a.Tq & ~7ll)) {
      // 16 new tokens starting on an 8-token boundary: one box, as for a pool block.
      ptx::tma_load_5d(dst + tile_row_offset<D>(p * 16, 0), m.new5, 0, 0, 0, (q0 + k0 - cb) >> 3, kvh, full);
    } else if (nr == 16 && all_new) {
#pragma unroll
      for (int at = 0; at < 2; ++at)
#pragma unroll
        for (int dh = 0; dh < D / 64; ++dh)
          ptx::tma_load_3d(dst + tile_row_offset<D>(p * 16 + 8 * at, dh), m.new8, dh * 64, kvh,
                           q0 + (k0 + 8 * at - cb), full);
    } else {
      for (int r = 0; r < nr; ++r) {
        const int key = k0 + r;
        const bool from_new = fused && key >= cb && key < ce;
#pragma unroll
        for (int dh = 0; dh < D / 64; ++dh) {
          if (from_new)
            ptx::tma_load_3d(dst + tile_row_offset<D>(p * 16 + r, dh), m.new1, dh * 64, kvh, q0 + (key - cb), full);
          else
            ptx::tma_load_3d(dst + tile_row_offset<D>(p * 16 + r, dh), m.row, dh * 64, kvh, blk * 16 + r, full);
        }
      }
    }
  }
}

// Fused call: this CTA's share of the slot-mapping scatter, by warp 2 (idle otherwise).
PKV_DEVINLINE void fused_write_share(const PkvAttnArgs& a, int warp, int lane) {
  if (a.k_new == nullptr || warp != 2) return;
  const int64_t cta = (int64_t)blockIdx.y * gridDim.x + blockIdx.x;
  const int vec_per_row = a.Hkv * a.D * 2 / 16;
  pkv_scatter((const uint4*)a.k_new, (const uint4*)a.v_new, a.slots, a.Tq, (uint4*)a.k_pool, (uint4*)a.v_pool,
              a.num_slots, vec_per_row, a.err, a.check, cta, (int64_t)gridDim.x * gridDim.y, lane, &a);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcMaps maps, const PkvAttnArgs a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  TcSmem<D>& sm = *reinterpret_cast<TcSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = a.Hq / a.Hkv;
  // The split tail's combine (a programmatic dependent launch) may be scheduled once every CTA of this
  // grid is running; it waits for this grid's completion before it reads anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // CTA -> (group member gi, tile pair, kv head, row): the CTAs of one (row, kv head) are
  // adjacent in launch order, so they run together and share its keys and values in L2.
  // (Issuing the odd last tiles of every head after all pairs, to fill the last wave with
  // cheaper CTAs, gained 1 % and doubled the DRAM reads: those tiles re-read evicted keys.)
  // With a split tail, the CTAs past the first `split_direct` items take num_splits each per item:
  // only the items of the last, partly filled wave are split.
  // (`whole` and `split` are cheap to recompute from the launch parameters, so the epilogue
  // does that instead of keeping them live through the softmax loop.)
  const int n_qp = (a.max_query_len + 2 * BM - 1) / (2 * BM);
  const bool whole = a.num_splits == 1 || (int)blockIdx.x < a.split_direct;
  int u = blockIdx.x, split = 0;
  if (!whole) {
    const int p = u - a.split_direct;
    u = a.split_direct + p / a.num_splits;
    split = p % a.num_splits;
  }
  const int nsplit = whole ? 1 : a.num_splits;
  const PkvTcItem it = pkv_tc_item(u, g, n_qp, a.Hkv);
  const int gi = it.gi, t0 = 2 * it.qp, kvh = it.kvh, b = it.b;
  const int h = kvh * g + gi;

  const int q0 = a.query_start_loc[b];
  int Sq = a.query_start_loc[b + 1] - q0;
  int L = a.seq_lens[b];
  if (a.check) {
    const int lmax = a.W * 16 < a.max_seq_len ? a.W * 16 : a.max_seq_len;
    const bool first = tid == 0 && t0 == 0 && gi == 0 && split == 0;
    if (Sq < 0 || Sq > a.max_query_len) {
      if (first) pkv_raise(a.err, PKV_DEVERR_QUERY);
      Sq = Sq < 0 ? 0 : a.max_query_len;
    }
    if (L > lmax || L < Sq || L < 0) {
      if (first) pkv_raise(a.err, PKV_DEVERR_SEQLEN);
      L = L > lmax ? lmax : (L < 0 ? 0 : L);
    }
  }
  const int i0 = t0 * BM;
  if (i0 >= Sq) {  // whole CTA: no query rows here
    fused_write_share(a, warp, lane);
    return;
  }
  // A pipeline timeout earlier in this launch (or an unchecked earlier one) means
  // results are already invalid: fail fast instead of waiting again.
  if (*(volatile unsigned int*)a.err & PKV_DEVERR_TIMEOUT) {
    fused_write_share(a, warp, lane);
    return;
  }
  const int n_q = i0 + BM < Sq ? 2 : 1;  // query tiles with rows in them

  // Softmax groups: warps 4-7 own query tile 0, warps 8-11 tile 1; TMEM lane quarter = warp % 4.
  // Each row's key limit is read from the segments here, overlapping the set-up below.
  const int grp = warp >= 8 ? 1 : 0;
  const bool is_softmax = warp >= 4;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  // A lone tile of at most 64 rows (a row's ragged last tile) runs M = 64 MMAs, half the tensor work
  // of M = 128 for the same rows: their accumulator rows sit in lanes 0-15 of each 32-lane TMEM
  // quarter (row 16q + l at lane 32q + l), so thread (quarter q, lane l < 16) owns row 16q + l and
  // lanes 16-31 carry no row.
  const bool m64 = n_q == 1 && Sq - i0 <= 64;
  const bool row_lane = !m64 || lane < 16;
  const int i = row_lane ? i0 + grp * BM + (m64 ? quarter * 16 + lane : row) : Sq;  // local query index (Sq: none)
  int lim = 0;
  if (is_softmax && i < Sq) {
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

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      ptx::mbar_init(&sm.empty[s], 1);
    }
    ptx::mbar_init(&sm.q_full, 1);
    for (int w = 0; w < 2; ++w) {
      ptx::mbar_init(&sm.s_full[w], 1);
      ptx::mbar_init(&sm.p_full[w], 128);
    }
    ptx::mbar_init(&sm.mma_done, 1);
    sm.lim_max = 0;
    sm.abort = 0;
    ptx::fence_mbar_init();
    // Q does not depend on the key range: its load starts before the rows' key limits are reduced.
    ptx::mbar_arrive_expect_tx(&sm.q_full, (uint32_t)(n_q * BM * D * 2));
    for (int t = 0; t < n_q; ++t)
#pragma unroll
      for (int dh = 0; dh < D / 64; ++dh)  // rows past the last token read as zeros
        ptx::tma_load_3d(sm.q[t] + dh * (BM * 128), &maps.q, dh * 64, h, q0 + i0 + t * BM, &sm.q_full);
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&maps.kb);
    ptx::prefetch_tmap(&maps.vb);
    if (a.contiguous) {
      ptx::prefetch_tmap(&maps.kc);
      ptx::prefetch_tmap(&maps.vc);
    }
    if (a.k_new) {
      ptx::prefetch_tmap(&maps.kn8);
      ptx::prefetch_tmap(&maps.vn8);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  __syncthreads();

  if (is_softmax) {  // the CTA's largest key limit (warp maxima first)
    const int wmax = __reduce_max_sync(0xffffffffu, lim);
    if (lane == 0) atomicMax(&sm.lim_max, wmax);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  const uint32_t tmem = sm.tmem_base;
  const int kv_hi = sm.lim_max;
  const int n_tiles = (kv_hi + BN - 1) / BN;
  const int per = (n_tiles + nsplit - 1) / nsplit;
  const int t_begin = split * per;
  const int t_end = min(n_tiles, t_begin + per);
  const int n = t_end > t_begin ? t_end - t_begin : 0;

  constexpr uint32_t O_COL[2] = {256, 256 + D};
  const uint32_t IDESC_QK = ptx::idesc_f16(m64 ? 64 : BM, BN, BF16 ? 1 : 0, 0);
  const uint32_t IDESC_PV = ptx::idesc_f16(m64 ? 64 : BM, D, BF16 ? 1 : 0, 1);

  if (warp < 4) {
  ptx::regs_dec<kRegsLow>();
  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ producers: warp 0 key tiles, warp 3 value tiles
    // Keys at the queries' own positions [cb, ce) (fused call: read from the new tokens).
    int cb = 0, ce = 0;
    if (a.k_new) {
      int s_begin = 0, s_end = 0;
      if (a.segs) {
        s_begin = a.seg_start[b];
        s_end = a.seg_start[b + 1];
      }
      cb = pkv_query_base(L, Sq, a.segs, s_begin, s_end);
      ce = cb + Sq;
      cb = cb < 0 ? 0 : cb;
      ce = ce > L ? L : ce;
    }
    const OperandMaps km{&maps.kb, &maps.kc, &maps.k1, &maps.kn5, &maps.kn8, &maps.kn1};
    const OperandMaps vm{&maps.vb, &maps.vc, &maps.v1, &maps.vn5, &maps.vn8, &maps.vn1};
    if (warp == 0 && n == 0 && lane == 0) {
      // No key tile to process: nothing will wait for Q, but its copy must land before the CTA exits.
      int never = 0;
      ptx::mbar_wait(&sm.q_full, 0, &never, kWaitLimitNs);
    }
    for (int idx = warp == 0 ? 0 : 1; idx < 2 * n; idx += 2) {
      if (__any_sync(0xffffffffu, sm.abort != 0)) break;
      const int pos = idx % C::NSLOT, use = idx / C::NSLOT;
      const bool is_v = idx & 1;
      const int kt = t_begin + (idx >> 1);
      const int rows = min(BN, kv_hi - kt * BN);
      if (idx >= C::NSLOT && !warp_wait(&sm.empty[pos], (use - 1) & 1, &sm.abort, lane)) {
        if (lane == 0) note_abort(sm, a.err);
        break;
      }
      if (is_v && rows < BN) {
        // Value rows past the last visible key are never loaded: zero them (P is 0 there,
        // but 0 * NaN would not be).  Whole 128-byte rows: independent of the swizzle.
        const int nz = (BN - rows) * (D / 64) * 8;  // 16-byte chunks to clear
        for (int e = lane; e < nz; e += 32) {
          const int chunk = e & 7, rd = e >> 3;
          const int r = rows + rd / (D / 64), dh = rd % (D / 64);
          *reinterpret_cast<uint4*>(sm.kv[pos] + tile_row_offset<D>(r, dh) + chunk * 16) = make_uint4(0, 0, 0, 0);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
      }
      load_tile<D>(sm.kv[pos], is_v ? vm : km, &sm.full[pos], a, b, kvh, kt, rows, cb, ce, q0, lane);
    }
    if (warp == 0 && sm.abort && lane == 0) {
      // Let copies already issued land before the shared memory goes away.
      int dummy = 0;
      ptx::mbar_wait(&sm.q_full, 0, &dummy, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      const uint32_t q_base[2] = {ptx::smem_u32(sm.q[0]), ptx::smem_u32(sm.q[1])};
      const uint32_t kv_base = ptx::smem_u32(sm.kv[0]);
      bool ok = ptx::mbar_wait(&sm.q_full, 0, &sm.abort, kWaitLimitNs);
      ptx::tc_fence_after();
      auto slot_ready = [&](int idx) -> bool {
        const int pos = idx % C::NSLOT;
        if (!ptx::mbar_wait(&sm.full[pos], (idx / C::NSLOT) & 1, &sm.abort, kWaitLimitNs)) return false;
        ptx::tc_fence_after();
        return true;
      };
      // One issuing thread feeds the tensor core: an MMA (128x128x16) takes 64 cycles, so the
      // descriptors are built once and each MMA only offsets one (ptx::desc_add).  Rebuilding
      // them per MMA measured a third slower when Q.K^T and P.V alternate.
      // Q: [half][128 rows][128 B] -> 8-row atoms at 1024 B, column half at BM*128 B.
      const uint64_t q_desc[2] = {ptx::smem_desc(q_base[0], 16, 1024, 2), ptx::smem_desc(q_base[1], 16, 1024, 2)};
      // K: block-interleaved -> 8-row atoms at GS, column half at +1024 B.  V: MN-major.
      const uint64_t k_desc = ptx::smem_desc(kv_base, 16, C::GS, 2);
      const uint64_t v_desc = ptx::smem_desc(kv_base, 1024, C::GS, 2);
      // S_w = Q_w K_j^T (key tile j sits in slot (2j) % NSLOT)
      auto qk = [&](int w, int j) {
        const uint64_t kd = ptx::desc_add(k_desc, (uint32_t)(((2 * j) % C::NSLOT) * C::TILE) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_ss(tmem + 128 * w, ptx::desc_add(q_desc[w], ((ks >> 2) * (BM * 128) + (ks & 3) * 32) >> 4),
                      ptx::desc_add(kd, ((ks >> 2) * 1024 + (ks & 3) * 32) >> 4), IDESC_QK, ks > 0);
        ptx::mma_commit(&sm.s_full[w]);
      };
      // O_w (+)= P_w V_j (value tile j sits in slot (2j+1) % NSLOT; P_w over the first columns of S_w)
      auto pv = [&](int w, int j) {
        const uint64_t vd = ptx::desc_add(v_desc, (uint32_t)(((2 * j + 1) % C::NSLOT) * C::TILE) >> 4);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          ptx::mma_ts(tmem + O_COL[w], tmem + 128 * w + ks * 8, ptx::desc_add(vd, (ks * 2 * C::GS) >> 4), IDESC_PV,
                      (j > 0 || ks > 0) ? 1u : 0u);
      };
      if (ok) ok = slot_ready(0);
      if (ok)
        for (int w = 0; w < n_q; ++w) qk(w, 0);
      for (int j = 0; ok && j < n; ++j) {
        const bool next = j + 1 < n;
        if (!slot_ready(2 * j + 1)) {  // value tile j
          ok = false;
          break;
        }
        for (int w = 0; w < n_q && ok; ++w) {
          if (!ptx::mbar_wait(&sm.p_full[w], j & 1, &sm.abort, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          pv(w, j);
          if (next) {
            if (w == 0 && !slot_ready(2 * j + 2)) {  // key tile j+1
              ok = false;
              break;
            }
            qk(w, j + 1);
          }
        }
      }
      if (!ok) note_abort(sm, a.err);
      // Everything issued must finish before TMEM is released.
      ptx::mma_commit(&sm.mma_done);
      int dummy = 0;
      ptx::mbar_wait(&sm.mma_done, 0, &dummy, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ warp 2: fused write
    fused_write_share(a, warp, lane);
  }
  } else {
  ptx::regs_inc<kRegsHigh>();
  if (grp < n_q) {
    // ------------------------------------------------------------ softmax rows of query tile grp
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t S_COL = 128 * grp;
    const bool valid = i < Sq;
    const int64_t tok = (int64_t)q0 + i;
    const float sl2 = a.scale * 1.4426950408889634f;  // scale * log2(e)
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sm.s_full[grp], j & 1, &sm.abort, kWaitLimitNs))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      // Ring slots are released here rather than by MMA commits (each commit in the MMA stream
      // cost it ~150 cycles): the last group's scores of tile j are committed after every earlier
      // MMA, so key tile j and value tile j-1 are no longer read.
      if (grp == n_q - 1 && row == 0) {
        ptx::mbar_arrive(&sm.empty[(2 * j) % C::NSLOT]);
        if (j > 0) ptx::mbar_arrive(&sm.empty[(2 * j - 1) % C::NSLOT]);
      }
      float s[BN];
      {
        uint32_t r[BN / 32][32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) ptx::tmem_ld32(tmem + lane_base + S_COL + c * 32, r[c]);
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
      // Row maximum: four chains of three-input maxima.
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = fmaxf(s[2 * u], s[2 * u + 1]);
#pragma unroll
      for (int c = 16; c < BN; c += 16)
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = ptx::max3(mx[u], s[c + 2 * u], s[c + 2 * u + 1]);
      const float m_tile =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
      // TMEM loads/stores are warp-collective: the warp rescales together when any
      // of its rows needs it (alpha = 1 for the others).  P.V of tile j-1 is complete:
      // the score MMA of tile j, whose completion was just observed, was issued after it.
      const bool need = m_tile > m_ref + kRescaleThreshold;
      const bool rescale = __any_sync(0xffffffffu, need);
      const float alpha = need ? ptx::ex2(m_ref - m_tile) : 1.f;  // 0 on a row's first visible tile
      if (need) {
        l *= alpha;
        m_ref = m_tile;
      }
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
      // P occupies columns [0, BN/2) of the score buffer: 32 scores -> 16 packed columns.
      // Exponent arguments and partial sums run as packed fp32 pairs.
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x0, x1;
          ptx::fma2(x0, x1, s[c * 64 + 2 * e], s[c * 64 + 2 * e + 1], sl2, sl2, -mu, -mu);
          const float p0 = ptx::ex2(x0);
          const float p1 = ptx::ex2(x1);
          if (e & 1)
            ptx::add2(l2, l3, p0, p1);
          else
            ptx::add2(l0, l1, p0, p1);
          r[e] = BF16 ? ptx::pack_bf16x2(p0, p1) : ptx::pack_f16x2(p0, p1);
        }
        ptx::tmem_st32(tmem + lane_base + S_COL + c * 32, r);
      }
      l += (l0 + l1) + (l2 + l3);
      // O carries the previous maximum: rescale it before this tile's P.V accumulates into it
      // (the MMA warp issues that only after the arrive below).  Done once the scores are dead,
      // so the O chunk does not compete with them for registers.
      if (rescale && j > 0) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          ptx::tmem_ld32(tmem + lane_base + O_COL[grp] + c * 32, r);
          ptx::tmem_wait_ld();
          ptx::reg_fence32(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          ptx::tmem_st32(tmem + lane_base + O_COL[grp] + c * 32, r);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&sm.p_full[grp]);
    }
    if (!ok) note_abort(sm, a.err);

    // ---------------------------------------------------------------- epilogue
    // A full query tile of a one-split call leaves through shared memory (the Q buffer, free once
    // every MMA is done) and TMA stores: one head's rows are Hq*D apart in the output, so rows
    // stored thread by thread scatter.  A split's fp32 partials are staged too (below); a ragged
    // tile of a whole item stores per thread.  `staged` and `whole_out` are the same for every
    // thread of the warpgroup, which meets at a named barrier.
    const bool whole_out = a.num_splits == 1 || (int)blockIdx.x < a.split_direct;
    const bool staged = whole_out && n > 0 && i0 + grp * BM + BM <= Sq;
    float o[D];
    float inv = 0.f;
    if (ok) {
      if (n > 0) {
        // mma_done completes exactly once, after every MMA of the CTA.
        if (__all_sync(0xffffffffu, ptx::mbar_wait(&sm.mma_done, 0, &sm.abort, kWaitLimitNs))) {
          ptx::tc_fence_after();
          // All of the row's O columns in flight at once, one wait.
          uint32_t r[D / 32][32];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(tmem + lane_base + O_COL[grp] + c * 32, r[c]);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            ptx::reg_fence32(r[c]);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[c * 32 + e] = __uint_as_float(r[c][e]);
          }
        } else {
          note_abort(sm, a.err);
          l = 0.f;
        }
      }
      inv = l > 0.f ? 1.f / l : 0.f;
    }
    if (staged) {
      uint8_t* tile = sm.q[grp];  // [D/64][128 rows][128 B], 128-byte swizzled like the Q load
      if (ok) {
#pragma unroll
        for (int dh = 0; dh < D / 64; ++dh)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float x0 = o[dh * 64 + k * 8 + 2 * e] * inv;
              const float x1 = o[dh * 64 + k * 8 + 2 * e + 1] * inv;
              w[e] = BF16 ? ptx::pack_bf16x2(x0, x1) : ptx::pack_f16x2(x0, x1);
            }
            *reinterpret_cast<uint4*>(tile + dh * (BM * 128) + row * 128 + ((k ^ (row & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
      }
      ptx::fence_proxy_async_smem();
      asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(BM) : "memory");
      if (row == 0 && !sm.abort) {
#pragma unroll
        for (int dh = 0; dh < D / 64; ++dh)
          ptx::tma_store_3d(&maps.o, dh * 64, h, q0 + i0 + grp * BM, tile + dh * (BM * 128));
        ptx::bulk_commit();
        ptx::bulk_wait_read_all();  // shared memory read before the CTA (and its shared memory) goes away
      }
    } else if (!whole_out) {
      // A split's fp32 partial rows (D*4 bytes each, Hq*D*4 apart): stored thread by thread, each
      // warp instruction would touch 32 rows.  They go through shared memory instead -- the key/value
      // ring, which no copy or MMA uses once mma_done has completed -- and each warp then stores whole
      // rows, one per instruction.
      // Staged at the query's row of the tile (a lone M = 64 tile's rows sit in lanes 0-15).
      uint8_t* st = sm.kv[0] + grp * (BM * C::PART_ROW);
      if (ok && valid && !sm.abort) {
        uint8_t* srow = st + (i - (i0 + grp * BM)) * C::PART_ROW;
#pragma unroll
        for (int v4 = 0; v4 < D / 4; ++v4)
          *reinterpret_cast<float4*>(srow + v4 * 16) =
              n > 0 ? make_float4(o[v4 * 4] * inv, o[v4 * 4 + 1] * inv, o[v4 * 4 + 2] * inv, o[v4 * 4 + 3] * inv)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(BM) : "memory");
      const int sp = ((int)blockIdx.x - a.split_direct) % a.num_splits;
      if (ok && valid) {
        // natural-log log-sum-exp of this split: ln 2 * (m_ref + log2 l)
        a.part_lse[((int64_t)sp * a.Tq + tok) * a.Hq + h] =
            (n > 0 && l > 0.f) ? 0.6931471805599453f * (m_ref + __log2f(l)) : -INFINITY;
      }
      if (!sm.abort) {
        constexpr int V4 = D / 4;                           // 16-byte pieces per row
        const int row_lim = min(BM, Sq - (i0 + grp * BM));  // rows of this tile that are queries
        for (int e = quarter * 32 + lane; e < BM * V4; e += 128) {
          const int r = e / V4, v4 = e % V4;
          if (r >= row_lim) break;
          const int64_t t = (int64_t)q0 + i0 + grp * BM + r;
          reinterpret_cast<float4*>(a.part_o + (((int64_t)sp * a.Tq + t) * a.Hq + h) * D)[v4] =
              *reinterpret_cast<const float4*>(st + r * C::PART_ROW + v4 * 16);
        }
      }
    } else if (ok) {
      if (!valid) {
        // query row past the end of this row's queries: nothing to store
      } else {
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
      }
    }
  }

  }  // softmax warpgroups

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

bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool BF16>
int launch_tc(const PkvAttnArgs& a, cudaStream_t s) {
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  const int64_t num_slots = a.num_blocks * 16;
  const cuuint64_t slot = (cuuint64_t)a.Hkv * D * 2;
  // Pool as 5-D: (64 columns, 8 rows, D/64 column halves, slot groups of 8, heads),
  // strides (slot, 128 B, 8 slots, head); box = one 16-row block of one head.
  const cuuint64_t dims5[5] = {64, 8, (cuuint64_t)(D / 64), (cuuint64_t)(num_slots / 8), (cuuint64_t)a.Hkv};
  const cuuint64_t str5[4] = {slot, 128, 8 * slot, (cuuint64_t)D * 2};
  const cuuint32_t box5[5] = {64, 8, (cuuint32_t)(D / 64), 2, 1};
  const cuuint32_t box5c[5] = {64, 8, (cuuint32_t)(D / 64), 2 * (BN / 16), 1};
  const cuuint64_t dims3[3] = {(cuuint64_t)D, (cuuint64_t)a.Hkv, (cuuint64_t)num_slots};
  const cuuint64_t str3[2] = {(cuuint64_t)D * 2, slot};
  const cuuint32_t box1[3] = {64, 1, 1};
  const cuuint64_t dimsq[3] = {(cuuint64_t)D, (cuuint64_t)a.Hq, (cuuint64_t)a.Tq};
  const cuuint64_t strq[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hq * D * 2};
  const cuuint32_t boxq[3] = {64, 1, BM};
  if (!encode(&maps.kb, a.k_pool, 5, dims5, str5, box5, BF16) || !encode(&maps.vb, a.v_pool, 5, dims5, str5, box5, BF16) ||
      (a.contiguous && (!encode(&maps.kc, a.k_pool, 5, dims5, str5, box5c, BF16) ||
                        !encode(&maps.vc, a.v_pool, 5, dims5, str5, box5c, BF16))) ||
      !encode(&maps.k1, a.k_pool, 3, dims3, str3, box1, BF16) || !encode(&maps.v1, a.v_pool, 3, dims3, str3, box1, BF16) ||
      !encode(&maps.q, a.q, 3, dimsq, strq, boxq, BF16))
    return (int)cudaErrorInvalidValue;
  if ((a.num_splits == 1 || a.split_direct > 0) && !encode(&maps.o, a.out, 3, dimsq, strq, boxq, BF16)) return (int)cudaErrorInvalidValue;
  if (a.k_new) {
    // New tokens [Tq, Hkv, D]: (D, Hkv, Tq) with the pool's row stride.
    const cuuint64_t dimsn[3] = {(cuuint64_t)D, (cuuint64_t)a.Hkv, (cuuint64_t)a.Tq};
    const cuuint32_t boxn8[3] = {64, 1, 8};
    if (!encode(&maps.kn8, a.k_new, 3, dimsn, str3, boxn8, BF16) || !encode(&maps.vn8, a.v_new, 3, dimsn, str3, boxn8, BF16) ||
        !encode(&maps.kn1, a.k_new, 3, dimsn, str3, box1, BF16) || !encode(&maps.vn1, a.v_new, 3, dimsn, str3, box1, BF16))
      return (int)cudaErrorInvalidValue;
    if (a.Tq >= 16) {  // the kernel uses this view only for 16 tokens inside the first Tq & ~7
      const cuuint64_t dimsn5[5] = {64, 8, (cuuint64_t)(D / 64), (cuuint64_t)(a.Tq / 8), (cuuint64_t)a.Hkv};
      if (!encode(&maps.kn5, a.k_new, 5, dimsn5, str5, box5, BF16) || !encode(&maps.vn5, a.v_new, 5, dimsn5, str5, box5, BF16))
        return (int)cudaErrorInvalidValue;
    }
  }
  const size_t smem = sizeof(TcSmem<D>) + 1024;
  // Per device, once; racing first calls from several host threads only repeat the same settings.
  // Keyed on the context: function attributes belong to the context they were set in.
  static std::atomic<uint64_t> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cached = dev >= 0 && dev < 64;
  const uint64_t ctx = pkv_context_id();
  if (!cached || ctx == 0 || attr_set[dev].load(std::memory_order_acquire) != ctx) {
    // The warpgroup register split is only valid for the register count it was sized for.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_tc_kernel<D, BF16>);
    if (e != cudaSuccess) return (int)e;
    if (fa.numRegs != kLaunchRegs) return (int)cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(attn_tc_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    if (cached) attr_set[dev].store(ctx, std::memory_order_release);
  }
  const int g = a.Hq / a.Hkv;
  const int n_qp = (a.max_query_len + 2 * BM - 1) / (2 * BM);
  const int64_t items = (int64_t)a.B * a.Hkv * n_qp * g;
  if (a.split_direct < 0 || a.split_direct > items) return (int)cudaErrorInvalidValue;
  const int64_t ctas = a.num_splits > 1 ? a.split_direct + (items - a.split_direct) * a.num_splits : items;
  if (ctas > 0x7fffffff) return (int)cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)ctas);
  attn_tc_kernel<D, BF16><<<grid, kThreads, smem, s>>>(maps, a);
  return (int)cudaGetLastError();
}

}  // namespace

bool pkv_attn_tc_supports(pkv_dtype dt, int D) { return (dt == PKV_BF16 || dt == PKV_F16) && (D == 64 || D == 128); }

int pkv_launch_attn_tc(const PkvAttnArgs& a, pkv_dtype dt, void* stream) {
  if (!pkv_attn_tc_supports(dt, a.D) || !(a.scale > 0.f) || !a.err) return -1;
  if (a.Tq > 0x7fffffff) return -1;
  cudaStream_t s = (cudaStream_t)stream;
  if (a.D == 128) return dt == PKV_BF16 ? launch_tc<128, true>(a, s) : launch_tc<128, false>(a, s);
  return dt == PKV_BF16 ? launch_tc<64, true>(a, s) : launch_tc<64, false>(a, s);
}
